// k_gemm_f4.cu -- the NVFP4 instantiations of the tensor-core GEMM
// (k_gemm_tc.cuh): the fused gate/up GEMM with the FP4-to-FP4 gated
// activation and the down GEMM + residual of the NVFP4 encoder FFN
// (itsolotime FlashRT article, 7.2), in the weight-streaming role (<= 64
// tokens; BN = 16 / 32 / 64) and the tiled role (BN = 256, one accumulator;
// or 128, two).
#include "k_gemm_tc.cuh"

namespace frt {

cudaError_t launch_gemm_f4(const GemmLaunch &g, cudaStream_t s, bool pdl) {
    const bool gated = f4_gated(g.p.epi);
    // the gated epilogues run on whole tiles only (no split-K)
    if (gated && g.p.splits != 1)
        return cudaErrorInvalidValue;
    if (g.swap) {
        const int role = gated ? ROLE_GATED_TILE : g.p.cluster ? ROLE_CLUSTER_PLAIN : ROLE_ANY;
        switch (g.bn * 8 + role) {
        case 16 * 8 + ROLE_ANY: return run<16, true, false, ROLE_ANY, true>(g, s, pdl);
        case 16 * 8 + ROLE_GATED_TILE: return run<16, true, false, ROLE_GATED_TILE, true>(g, s, pdl);
        case 16 * 8 + ROLE_CLUSTER_PLAIN: return run<16, true, false, ROLE_CLUSTER_PLAIN, true>(g, s, pdl);
        case 32 * 8 + ROLE_ANY: return run<32, true, false, ROLE_ANY, true>(g, s, pdl);
        case 32 * 8 + ROLE_GATED_TILE: return run<32, true, false, ROLE_GATED_TILE, true>(g, s, pdl);
        case 32 * 8 + ROLE_CLUSTER_PLAIN: return run<32, true, false, ROLE_CLUSTER_PLAIN, true>(g, s, pdl);
        case 64 * 8 + ROLE_ANY: return run<64, true, false, ROLE_ANY, true>(g, s, pdl);
        case 64 * 8 + ROLE_GATED_TILE: return run<64, true, false, ROLE_GATED_TILE, true>(g, s, pdl);
        case 64 * 8 + ROLE_CLUSTER_PLAIN: return run<64, true, false, ROLE_CLUSTER_PLAIN, true>(g, s, pdl);
        default: return cudaErrorInvalidValue;
        }
    }
    if (g.bn == 128)
        return run<128, false, false, ROLE_ANY, true>(g, s, pdl);
    if (g.bn == 256)
        return run<256, false, false, ROLE_ANY, true>(g, s, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace frt
