// frt_noalloc.cu -- the FP8 GEMM entry point that allocates nothing.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured in global mode, allocator-free embedded or real-time hosts
// that forbid allocation after start-up, and hosts that hand every byte of
// device memory to their own pool.  frt_fp8_gemm_noalloc serves them: the
// caller passes the inputs and the output, and the only other device memory
// the kernel touches -- its split-K workspace and arrival counters -- lives
// in a file-scope __device__ array of fixed size that every GPU loading this
// library holds until the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <string>

#include "frt_ffn.h"
#include "frt_internal.h"

#define FRT_API extern "C" __attribute__((visibility("default")))

namespace {

// Maximum split-K workspace: 160 partial tiles of 128 x 64 fp32 values
// (5 MiB), enough for the weight-streaming path on every SM of a GB300, then
// the split-K arrival counters (2048 per split count, 136 KiB) and an error word.
constexpr size_t NOALLOC_WS_FLOATS = (size_t)160 * 128 * 64;
constexpr size_t NOALLOC_BYTES = NOALLOC_WS_FLOATS * 4 + (size_t)frt::SPLIT_COUNTERS * 4 + 4;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

constexpr int MAX_DEVICES = 64;
struct DevState {
    bool ready = false;
    unsigned char *base = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
};
DevState g_dev[MAX_DEVICES];

thread_local std::string g_err;

frt_status fail(frt_status st, const char *msg) {
    g_err = msg;
    return st;
}

}  // namespace

// Message of the last failed frt_fp8_gemm_noalloc call on this host thread.
FRT_API const char *frt_fp8_gemm_noalloc_last_error(void) { return g_err.c_str(); }

FRT_API frt_status frt_fp8_gemm_noalloc(const void *A, const void *B, void *C, int M, int N, int K, float alpha,
                                        frt_stream_t stream) {
    using namespace frt;
    if (!A || !B || !C || (reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
        (reinterpret_cast<uintptr_t>(C) & 15))
        return fail(FRT_ERR_INVALID_ARG, "A, B, C must be non-null, 16-byte aligned device pointers");
    if (M < 1 || M > 65536 || N < 128 || N % 128 || K < 16 || K % 16)
        return fail(FRT_ERR_INVALID_ARG, "need 1 <= M <= 65536, N % 128 == 0, K >= 16, K % 16 == 0");
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(FRT_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= MAX_DEVICES)
        return fail(FRT_ERR_UNSUPPORTED, "device index beyond the supported range");
    DevState &ds = g_dev[dev];
    if (!ds.ready) {
        // Once per device, with that device current: the device address of
        // the scratch array (the host-side symbol is only a stand-in).
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr)
            return fail(FRT_ERR_CUDA, "cudaGetSymbolAddress(g_noalloc_scratch) failed");
        e = cudaDeviceGetAttribute(&ds.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess || ds.num_sms <= 0)
            return fail(FRT_ERR_CUDA, "cudaDeviceGetAttribute(multiProcessorCount) failed");
        ds.base = static_cast<unsigned char *>(ptr);
        ds.ready = true;
    }
    GemmLaunch g;
    memset(&g.p, 0, sizeof g.p);
    const bool swap = M <= 64;
    plan_gemm(g, swap, M, N, K, ds.num_sms, 0);
    if (gemm_ws_floats(g) > NOALLOC_WS_FLOATS)
        return fail(FRT_ERR_UNSUPPORTED, "this shape needs more split-K workspace than the fixed 5 MiB scratch");
    if (g.p.splits > 1 && gemm_tiles(g) > MAX_SPLIT_TILES)
        return fail(FRT_ERR_UNSUPPORTED, "this shape has more split-K tiles than the fixed scratch counts");
    if (encode_tmap_u8(&g.tmP, swap ? B : A, swap ? N : M, K, 128) != cudaSuccess ||
        encode_tmap_u8(&g.tmQ, swap ? A : B, swap ? M : N, K, swap ? g.bn : g.bn / (g.p.pair ? 2 : 1)) != cudaSuccess)
        return fail(FRT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    float *ws = reinterpret_cast<float *>(ds.base);
    int *counters = reinterpret_cast<int *>(ds.base + NOALLOC_WS_FLOATS * 4);
    int *err = counters + SPLIT_COUNTERS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The counters must start at zero; a call that gave up a wait could have
    // left some set, so clear them on the stream before every launch.
    e = cudaMemsetAsync(counters, 0, (size_t)SPLIT_COUNTERS * 4 + 4, s);
    if (e != cudaSuccess)
        return fail(FRT_ERR_CUDA, cudaGetErrorString(e));
    g.p.epi = EPI_F32;
    g.p.alpha = alpha;
    g.p.out = C;
    g.p.ldo = N;
    g.p.ws = ws;
    g.p.counters = split_counters(counters, g.p.splits);
    g.p.err = err;
    e = launch_gemm(g, s, false);
    if (e != cudaSuccess)
        return fail(FRT_ERR_CUDA, cudaGetErrorString(e));
    return FRT_OK;
}
