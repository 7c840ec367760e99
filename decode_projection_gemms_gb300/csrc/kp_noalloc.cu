// skinny_gemm_noalloc: the CUDA-core split-K GEMM with its scratch in a fixed
// device array that the library carries, for callers that must not allocate.
//
// Who needs this: processes whose device memory is owned by a pooling/caching
// allocator that forbids the CUDA runtime from taking memory behind its back,
// and latency-critical paths that cannot afford cudaMalloc's implicit device
// synchronisation. skinny_gemm grows
// a workspace on demand; this entry point never does.
//
// The scratch is a file-scope __device__ array: every GPU that loads the
// library holds it (KP_NOALLOC_SCRATCH_FLOATS floats + KP_NOALLOC_TICKETS
// ints) until the process exits. Host code may not use the array's name as a
// device address, so the first call on each device looks the address up with
// cudaGetSymbolAddress (with that device current); later calls reuse the
// cached address. The tickets start at zero (a __device__ array is
// zero-initialised when the module loads) and every launch leaves them at
// zero, so nothing is cleared at set-up and no call synchronises.
#include <cstring>
#include <mutex>

#include "kp_internal.cuh"

// The fixed scratch (file scope; zero-initialised when the module loads).
static __device__ __align__(256) float g_noalloc_partials[KP_NOALLOC_SCRATCH_FLOATS];
static __device__ __align__(256) int g_noalloc_tickets[KP_NOALLOC_TICKETS];

namespace kp {
namespace {

struct NoAllocState {
    bool ready = false;
    float *partials = nullptr;
    int *tickets = nullptr;
    int sms = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
NoAllocState g_state[kMaxDevices];

int cuda_fail(cudaError_t e, const char *what) {
    return set_error(KP_ECUDA, "skinny_gemm_noalloc: %s: %s", what, cudaGetErrorString(e));
}

// Once per device, with that device current: resolve the arrays' device
// addresses. The tickets need no clearing: zero at module load, and the last
// CTA of every row tile resets its ticket before it exits.
int setup(NoAllocState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(KP_EINVAL, "skinny_gemm_noalloc: device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    NoAllocState &s = g_state[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major != 10 || minor != 3)
            return set_error(KP_ENODEV, "skinny_gemm_noalloc: device %d is sm_%d%d, not sm_103", dev,
                             major, minor);
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_partials)) != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(partials)");
        s.partials = static_cast<float *>(p);
        if ((e = cudaGetSymbolAddress(&p, g_noalloc_tickets)) != cudaSuccess)
            return cuda_fail(e, "cudaGetSymbolAddress(tickets)");
        s.tickets = static_cast<int *>(p);
        s.ready = true;
    }
    *out = &s;
    return KP_OK;
}

// Default CUDA-core configuration that fits the fixed scratch: about two CTAs
// per SM, fewer K slices when the partial sums would not fit (one slice needs
// no scratch at all). No programmatic dependent launch: the kernel would read
// W before waiting for the previous kernel on the stream, and a caller of
// this entry point may have just computed W there.
kp_cfg default_cfg(int M, int N, int K, int sms) {
    kp_cfg c;
    memset(&c, 0, sizeof c);
    c.kind = KP_KIND_CC;
    c.block = 256;
    c.rows = 4;
    c.k_unroll = 2;
    c.flags = 0;
    const int rows_cta = 8 * c.rows;
    const int tiles = (N + rows_cta - 1) / rows_cta;
    int S = (2 * sms + tiles - 1) / tiles;
    const int smax = K / 256 > 1 ? K / 256 : 1;
    if (S > smax) S = smax;
    if (S < 1) S = 1;
    for (;; --S) {
        c.split_k = S;
        const Scratch need = cc_scratch(M, N, K, c);
        if (S == 1 || (need.floats <= KP_NOALLOC_SCRATCH_FLOATS && need.counters <= KP_NOALLOC_TICKETS))
            break;
    }
    // the x slice must fit in shared memory: more slices if needed
    while (!cc_supported(M, K, c) && c.split_k < K / 8) ++c.split_k;
    return c;
}

}  // namespace
}  // namespace kp

using namespace kp;

extern "C" int skinny_gemm_noalloc(const void *x, const void *W, void *y, int M, int N, int K,
                                   const kp_cfg *cfg, kp_stream_t stream) {
    if (M < 0 || N < 1 || K < 8)
        return set_error(KP_EINVAL, "skinny_gemm_noalloc: bad sizes M=%d N=%d K=%d", M, N, K);
    if (K & 7) return set_error(KP_ESHAPE, "skinny_gemm_noalloc: K=%d is not a multiple of 8", K);
    if (M == 0) return KP_OK;
    if (M > 16)
        return set_error(KP_ECONFIG, "skinny_gemm_noalloc: runs the CUDA-core kernel, M <= 16 (got %d)", M);
    if (!x || !W || !y) return set_error(KP_EINVAL, "skinny_gemm_noalloc: NULL pointer");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(y)) & 15u)
        return set_error(KP_EALIGN, "skinny_gemm_noalloc: pointers must be 16-byte aligned");
    NoAllocState *s = nullptr;
    int rc = setup(&s);
    if (rc) return rc;
    kp_cfg c;
    if (cfg && cfg->kind != KP_KIND_AUTO) {
        c = *cfg;
        if (c.kind != KP_KIND_CC)
            return set_error(KP_ECONFIG, "skinny_gemm_noalloc: only the CUDA-core kernel (kind %d)",
                             KP_KIND_CC);
        if (!cc_supported(M, K, c))
            return set_error(KP_ECONFIG, "skinny_gemm_noalloc: config not valid for M=%d K=%d", M, K);
    } else {
        c = default_cfg(M, N, K, s->sms);
        if (cfg) c.flags = cfg->flags;
    }
    const Scratch need = cc_scratch(M, N, K, c);
    if (need.floats > KP_NOALLOC_SCRATCH_FLOATS || need.counters > KP_NOALLOC_TICKETS)
        return set_error(KP_ETOOBIG,
                         "skinny_gemm_noalloc: the config needs %zu partial floats and %zu tickets; the "
                         "fixed scratch holds %d and %d (use fewer K slices)",
                         need.floats, need.counters, KP_NOALLOC_SCRATCH_FLOATS, KP_NOALLOC_TICKETS);
    GemmArgs a;
    a.x = static_cast<const __nv_bfloat16 *>(x);
    a.ldx = K;
    a.W = static_cast<const __nv_bfloat16 *>(W);
    a.y = static_cast<__nv_bfloat16 *>(y);
    a.ldy = N;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ws = s->partials;
    a.counters = s->tickets;
    a.err = nullptr;
    cudaError_t e = cc_launch(a, c, stream);
    if (e != cudaSuccess) return cuda_fail(e, "launch");
    return KP_OK;
}
