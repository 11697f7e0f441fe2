// frt_noalloc.cu -- the FP8 GEMM entry point that allocates nothing.
//
// Some callers cannot call cudaMalloc: code that runs while a CUDA graph is
// being captured in global mode, allocator-free embedded or real-time hosts
// that forbid allocation after start-up, and hosts that hand every byte of
// device memory to their own pool.  frt_fp8_gemm_noalloc serves them: the
// caller passes the inputs and the output, and the only other device memory
// the kernel touches -- its split-K workspace, arrival counters and error
// word -- lives in a file-scope __device__ array of fixed size that every GPU
// loading this library holds until the process exits.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "frt_ffn.h"
#include "frt_internal.h"

#define FRT_API extern "C" __attribute__((visibility("default")))

namespace {

// Maximum split-K workspace: 160 partial tiles of 128 x 64 fp32 values
// (5 MiB), enough for the weight-streaming path on every SM of a GB300, then
// the split-K arrival counters (2048 per split count, 136 KiB) and an error word.
constexpr size_t NOALLOC_WS_FLOATS = (size_t)160 * 128 * 64;
constexpr size_t COUNTER_BYTES = (size_t)frt::SPLIT_COUNTERS * 4;
constexpr size_t NOALLOC_BYTES = NOALLOC_WS_FLOATS * 4 + COUNTER_BYTES + 4;

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_BYTES];

constexpr int MAX_DEVICES = 64;
struct DevState {
    std::atomic<bool> ready{false};
    unsigned char *base = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
};
DevState g_dev[MAX_DEVICES];
std::mutex g_init_mu;  // serialises the per-device set-up across host threads

thread_local std::string g_err;

frt_status fail(frt_status st, const char *msg) {
    g_err = msg;
    return st;
}

// The current device's state, set up on its first use: the device address of
// the scratch array (the host-side symbol is only a stand-in) and the SM
// count.  Double-checked under a mutex, so host threads making their first
// call on one device at once see one finished set-up.
frt_status dev_state(DevState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(FRT_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= MAX_DEVICES)
        return fail(FRT_ERR_UNSUPPORTED, "device index beyond the supported range");
    DevState &ds = g_dev[dev];
    if (!ds.ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(g_init_mu);
        if (!ds.ready.load(std::memory_order_relaxed)) {
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
            if (e != cudaSuccess || !ptr)
                return fail(FRT_ERR_CUDA, "cudaGetSymbolAddress(g_noalloc_scratch) failed");
            int sms = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess || sms <= 0)
                return fail(FRT_ERR_CUDA, "cudaDeviceGetAttribute(multiProcessorCount) failed");
            ds.base = static_cast<unsigned char *>(ptr);
            ds.num_sms = sms;
            ds.ready.store(true, std::memory_order_release);
        }
    }
    *out = &ds;
    return FRT_OK;
}

float *ws_of(const DevState &ds) { return reinterpret_cast<float *>(ds.base); }
int *counters_of(const DevState &ds) { return reinterpret_cast<int *>(ds.base + NOALLOC_WS_FLOATS * 4); }
int *err_of(const DevState &ds) { return counters_of(ds) + frt::SPLIT_COUNTERS; }

// Plan and launch one GEMM on the scratch array (stall: the test hook whose
// MMA thread waits for a phase nothing completes).
frt_status launch(const DevState &ds, const void *A, const void *B, void *C, int M, int N, int K, float alpha,
                  int stall, cudaStream_t s) {
    using namespace frt;
    GemmLaunch g;
    memset(&g.p, 0, sizeof g.p);
    const bool swap = M <= 64;
    plan_gemm(g, swap, M, N, K, ds.num_sms, stall ? 1 : 0);
    if (gemm_ws_floats(g) > NOALLOC_WS_FLOATS)
        return fail(FRT_ERR_UNSUPPORTED, "this shape needs more split-K workspace than the fixed 5 MiB scratch");
    if (g.p.splits > 1 && gemm_tiles(g) > MAX_SPLIT_TILES)
        return fail(FRT_ERR_UNSUPPORTED, "this shape has more split-K tiles than the fixed scratch counts");
    if (encode_tmap_u8(&g.tmP, swap ? B : A, swap ? N : M, K, 128) != cudaSuccess ||
        encode_tmap_u8(&g.tmQ, swap ? A : B, swap ? M : N, K, swap ? g.bn : g.bn / (g.p.pair ? 2 : 1)) != cudaSuccess)
        return fail(FRT_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    int *counters = counters_of(ds);
    // The split-K counters must start at zero; a call that gave up a wait can
    // leave some of them mid-count, so they are cleared on the stream before
    // every launch.  The error word is not: it keeps a timeout until
    // frt_fp8_gemm_noalloc_status reads it.
    cudaError_t e = cudaMemsetAsync(counters, 0, COUNTER_BYTES, s);
    if (e != cudaSuccess)
        return fail(FRT_ERR_CUDA, cudaGetErrorString(e));
    g.p.epi = EPI_F32;
    g.p.alpha = alpha;
    g.p.out = C;
    g.p.ldo = N;
    g.p.ws = ws_of(ds);
    g.p.counters = split_counters(counters, g.p.splits);
    g.p.err = err_of(ds);
    g.p.stall_test = stall;
    e = launch_gemm(g, s, false);
    if (e != cudaSuccess)
        return fail(FRT_ERR_CUDA, cudaGetErrorString(e));
    return FRT_OK;
}

}  // namespace

// Message of the last failed frt_fp8_gemm_noalloc* call on this host thread.
FRT_API const char *frt_fp8_gemm_noalloc_last_error(void) { return g_err.c_str(); }

FRT_API frt_status frt_fp8_gemm_noalloc(const void *A, const void *B, void *C, int M, int N, int K, float alpha,
                                        frt_stream_t stream) {
    if (!A || !B || !C || (reinterpret_cast<uintptr_t>(A) & 15) || (reinterpret_cast<uintptr_t>(B) & 15) ||
        (reinterpret_cast<uintptr_t>(C) & 15))
        return fail(FRT_ERR_INVALID_ARG, "A, B, C must be non-null, 16-byte aligned device pointers");
    if (M < 1 || M > 65536 || N < 128 || N % 128 || K < 16 || K % 16)
        return fail(FRT_ERR_INVALID_ARG, "need 1 <= M <= 65536, N % 128 == 0, K >= 16, K % 16 == 0");
    DevState *ds = nullptr;
    const frt_status st = dev_state(&ds);
    if (st != FRT_OK)
        return st;
    return launch(*ds, A, B, C, M, N, K, alpha, 0, static_cast<cudaStream_t>(stream));
}

FRT_API frt_status frt_fp8_gemm_noalloc_status(frt_stream_t stream) {
    DevState *ds = nullptr;
    frt_status st = dev_state(&ds);
    if (st != FRT_OK)
        return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return fail(FRT_ERR_CUDA, cudaGetErrorString(e));
    int h = 0;
    e = cudaMemcpy(&h, err_of(*ds), 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return fail(FRT_ERR_CUDA, cudaGetErrorString(e));
    if (h) {
        // a launch that gave up may have left split-K counters mid-count
        if ((e = cudaMemset(counters_of(*ds), 0, COUNTER_BYTES + 4)) != cudaSuccess ||
            (e = cudaDeviceSynchronize()) != cudaSuccess)
            return fail(FRT_ERR_CUDA, cudaGetErrorString(e));
        return fail(FRT_ERR_DEVICE_TIMEOUT, "an allocation-free GEMM gave up a bounded wait");
    }
    return FRT_OK;
}

FRT_API frt_status frt_fp8_gemm_noalloc_debug_stall(frt_stream_t stream) {
    DevState *ds = nullptr;
    frt_status st = dev_state(&ds);
    if (st != FRT_OK)
        return st;
    // a 64 x 256 x 128 weight-streaming GEMM whose operands and output are
    // regions of the scratch's workspace (whatever it holds): A at 0, B at
    // 64 KiB, C (64 KiB of fp32) at 1 MiB, all inside the 5 MiB workspace
    unsigned char *w = ds->base;
    st = launch(*ds, w, w + (64 << 10), w + (1 << 20), 64, 256, 128, 1.0f, 1, static_cast<cudaStream_t>(stream));
    if (st != FRT_OK)
        return st;
    return frt_fp8_gemm_noalloc_status(stream);
}
