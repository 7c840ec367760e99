// C ABI of the library (include/kdaproj.h): argument checks, configuration
// selection, scratch ownership and the two-stream projection sequence.
//
// The projection follows run_kda_projection_overlap of "[Kimi-K3] Overlap
// low-M TP8 KDA projections" (section "关键源码片段"): Q/K/V/G on the main
// stream; F_A/beta then F_B on an aux stream forked and joined with an event
// pair (maybe_execute_in_parallel); F_B reads the F_A half of the F_A/beta
// output in place (the page's split/view, no copy). The page's sequential
// fallback (KimiK3DeltaAttention.forward) is the same three GEMMs in order on
// one stream, which is what this library runs when overlap is off.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "kp_internal.cuh"

namespace kp {

// ---- errors ---------------------------------------------------------------------

static thread_local char t_err[512] = "";

int set_error(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof t_err, fmt, ap);
    va_end(ap);
    return code;
}

static int cuda_fail(cudaError_t e, const char *what) {
    return set_error(KP_ECUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

// A kernel wait on this device ran out earlier and nobody has read the code
// yet: refuse new work (the outputs of that call are undefined).
static int refuse_after_give_up(const int *err_host) {
    const int v = err_host ? __atomic_load_n(err_host, __ATOMIC_ACQUIRE) : 0;
    if (v == 0) return KP_OK;
    return set_error(KP_EDEVICE,
                     "a kernel wait on this device ran out earlier (code %d); the outputs of that "
                     "call are undefined. kp_device_error() reads and clears the code", v);
}

// ---- per-device state -------------------------------------------------------------

struct DevState {
    bool ok = false;
    int sms = 0;
    int major = 0, minor = 0;
    // Error word of this device's kernels, in mapped pinned host memory:
    // kernels write it with system-scope atomics (err), host code reads it
    // with plain atomics (err_host) and no CUDA call, so an entry point can
    // refuse new work after a give-up without synchronising.
    int *err = nullptr;
    int *err_host = nullptr;
    // skinny_gemm's scratch, grown on demand. A buffer that growth replaces is
    // kept (never freed while the process runs): work captured into a CUDA
    // graph before the growth still points at it.
    float *ws = nullptr;
    size_t ws_floats = 0;
    int *cnt = nullptr;
    size_t cnt_n = 0;
    std::vector<void *> retired;
};

static std::mutex g_dev_mu;
static std::map<int, DevState> g_dev;

static int device_state(DevState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DevState &d = g_dev[dev];
    if (!d.ok) {
        if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (d.major != 10 || d.minor != 3)
            return set_error(KP_ENODEV, "device %d is sm_%d%d; this library is built for sm_103a",
                             dev, d.major, d.minor);
        void *h = nullptr;
        if ((e = cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable)) != cudaSuccess)
            return cuda_fail(e, "cudaHostAlloc(error word)");
        memset(h, 0, 64);
        void *dp = nullptr;
        if ((e = cudaHostGetDevicePointer(&dp, h, 0)) != cudaSuccess) {
            cudaFreeHost(h);
            return cuda_fail(e, "cudaHostGetDevicePointer(error word)");
        }
        d.err_host = static_cast<int *>(h);
        d.err = static_cast<int *>(dp);
        d.ok = true;
    }
    *out = &d;
    return KP_OK;
}

// ---- autotune table ---------------------------------------------------------------

struct TableEntry {
    int M, N, K;
    kp_cfg cfg;
    int overlap;
};

static std::mutex g_tab_mu;
static std::vector<TableEntry> g_table;

static int parse_kind(const char *s) {
    if (!strcmp(s, "cc")) return KP_KIND_CC;
    if (!strcmp(s, "tc05")) return KP_KIND_TC05;
    if (!strcmp(s, "smallk")) return KP_KIND_SMALLK;
    char *end = nullptr;
    long v = strtol(s, &end, 10);
    if (end && *end == 0 && v >= 1 && v <= 3) return static_cast<int>(v);
    return -1;
}

static bool cfg_supported(int M, int N, int K, const kp_cfg &c) {
    switch (c.kind) {
    case KP_KIND_CC: return cc_supported(M, K, c);
    case KP_KIND_TC05: return tc05_supported(M < 256 ? M : 256, N, K, c);
    case KP_KIND_SMALLK: return smallk_supported(M, K, c);
    default: return false;
    }
}

// Built-in rule for shapes the table does not cover.
static kp_cfg builtin_config(int M, int N, int K, int sms) {
    kp_cfg c;
    memset(&c, 0, sizeof c);
    c.flags = KP_FLAG_PDL;
    if (K <= 256) {
        c.kind = KP_KIND_SMALLK;
        c.block = 256;
        c.rows = 16;
        return c;
    }
    if (M <= 4) {
        c.kind = KP_KIND_CC;
        c.block = 256;
        c.rows = 4;
        c.k_unroll = 2;
        const int rows_cta = 8 * c.rows;
        const int tiles = (N + rows_cta - 1) / rows_cta;
        int S = (4 * sms + tiles - 1) / tiles;
        int smax = K / 256;
        if (smax < 1) smax = 1;
        if (S > smax) S = smax;
        if (S < 1) S = 1;
        c.split_k = S;
        if (cc_supported(M, K, c)) return c;
    }
    return tc05_default(M, N, K, sms);
}

static kp_cfg select_config(int M, int N, int K, int sms, int *overlap) {
    {
        std::lock_guard<std::mutex> lk(g_tab_mu);
        const TableEntry *best = nullptr;
        for (const TableEntry &e : g_table) {
            if (e.N != N || e.K != K || e.M < M) continue;
            if (!best || e.M < best->M) best = &e;
        }
        if (best && cfg_supported(M, N, K, best->cfg)) {
            if (overlap) *overlap = best->overlap;
            return best->cfg;
        }
    }
    if (overlap) *overlap = 1;
    return builtin_config(M, N, K, sms);
}

static Scratch scratch_of(int M, int N, int K, const kp_cfg &c, int sms) {
    switch (c.kind) {
    case KP_KIND_CC: return cc_scratch(M, N, K, c);
    case KP_KIND_TC05: return tc05_scratch(M, N, K, c, sms);
    default: return Scratch();
    }
}

// Launch one GEMM with configuration c (TC05 covers any M in one launch:
// token tiles of 256 along the grid's y axis).
static cudaError_t launch_gemm(GemmArgs a, const kp_cfg &c, int sms, cudaStream_t s) {
    switch (c.kind) {
    case KP_KIND_CC: return cc_launch(a, c, s);
    case KP_KIND_SMALLK: return smallk_launch(a, c, s);
    case KP_KIND_TC05: return tc05_launch(a, c, sms, s);
    default: return cudaErrorInvalidValue;
    }
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_cfg(int M, int N, int K, const kp_cfg &c) {
    if (c.flags & KP_FLAG_FUSE_FB)
        return set_error(KP_ECONFIG, "KP_FLAG_FUSE_FB applies only to the F_A/beta branch of a plan");
    if (c.kind == KP_KIND_CC && M > 16)
        return set_error(KP_ECONFIG, "CUDA-core kernel supports M <= 16 (got M=%d)", M);
    if (!cfg_supported(M, N, K, c))
        return set_error(KP_ECONFIG,
                         "config kind=%d split_k=%d block=%d rows=%d k_unroll=%d producers=%d stages=%d "
                         "is not valid for M=%d N=%d K=%d",
                         c.kind, c.split_k, c.block, c.rows, c.k_unroll, c.producers, c.stages, M, N, K);
    return KP_OK;
}

// ---- plan -------------------------------------------------------------------------

}  // namespace kp

struct kda_plan {
    int K = 0, Nq = 0, Nfab = 0, Nfb = 0, max_M = 0;
    int dev = 0, sms = 0;
    int overlap_mode = -1;
    std::vector<kp_cfg> cfg[3];        // [branch][M], M in 1..max_M
    std::vector<uint8_t> overlap;      // [M]
    float *ws[3] = {nullptr, nullptr, nullptr};
    size_t ws_floats[3] = {0, 0, 0};
    int *cnt[3] = {nullptr, nullptr, nullptr};
    size_t cnt_n[3] = {0, 0, 0};
    int *err = nullptr;        // the device's error word (device view)
    int *err_host = nullptr;   // the same word, host view
};

namespace kp {

struct BranchShape {
    int N, K;
};

static BranchShape branch_shape(const kda_plan *p, int b);

// Whether the plan can run the whole projection as one launch at M with the
// Q/K/V/G configuration c: the tcgen05 kernel (F_A rows starting on a 128-row
// tile, room for the fused F_B operands, no M slicing), or the CUDA-core
// kernel with one K slice (M <= 8, F_A rows a whole cluster of CTAs).
static bool single_launch_ok(const kda_plan *p, int M, const kp_cfg &c) {
    if (c.kind == KP_KIND_CC)
        return p->Nfb >= 1 && cc_proj_supported(M, p->K, p->Nq + p->Nfab, c, p->Nq);
    return c.kind == KP_KIND_TC05 && M <= 256 && p->Nq % tc05_rows(c) == 0 &&
           tc05_supported(M, p->Nq + p->Nfab, p->K, c) && tc05_fusable(M, c);
}

// Validation of a configuration for one branch of a plan: the F_A/beta
// branch may carry KP_FLAG_FUSE_FB (tcgen05 kernel, F_A = its first 128 rows).
static int check_branch_cfg(int branch, int M, int N, int K, const kp_cfg &c) {
    if (!(c.flags & KP_FLAG_FUSE_FB)) return check_cfg(M, N, K, c);
    if (branch != KP_BRANCH_FAB)
        return set_error(KP_ECONFIG, "KP_FLAG_FUSE_FB applies only to the F_A/beta branch");
    kp_cfg plain = c;
    plain.flags &= ~KP_FLAG_FUSE_FB;
    int rc = check_cfg(M, N, K, plain);
    if (rc) return rc;
    if (c.kind != KP_KIND_TC05 || (M <= 256 && !tc05_fusable(M, c)))
        return set_error(KP_ECONFIG,
                         "KP_FLAG_FUSE_FB needs the tcgen05 kernel with room for the F_B operands");
    return KP_OK;
}

static BranchShape branch_shape(const kda_plan *p, int b) {
    if (b == KP_BRANCH_QKVG) return {p->Nq, p->K};
    if (b == KP_BRANCH_FAB) return {p->Nfab, p->K};
    return {p->Nfb, 128};
}

// Scratch a branch's configuration needs at M; the Q/K/V/G branch's also
// serves the single launch over the packed weight (N_qkvg + N_fab rows).
static Scratch branch_scratch(const kda_plan *p, int b, int M, const kp_cfg &c) {
    const BranchShape sh = branch_shape(p, b);
    const int N = b == KP_BRANCH_QKVG ? p->Nq + p->Nfab : sh.N;
    return scratch_of(M, N, sh.K, c, p->sms);
}

static void free_plan_memory(kda_plan *p) {
    for (int b = 0; b < 3; ++b) {
        if (p->ws[b]) cudaFree(p->ws[b]);
        if (p->cnt[b]) cudaFree(p->cnt[b]);
        p->ws[b] = nullptr;
        p->cnt[b] = nullptr;
    }
}

}  // namespace kp

using namespace kp;

// ---- exported functions ---------------------------------------------------------------

extern "C" {

const char *kp_last_error(void) { return t_err; }

int kp_version(void) { return KDAPROJ_VERSION; }

int kp_table_load(const char *path) {
    if (!path) return set_error(KP_EINVAL, "kp_table_load: NULL path");
    FILE *f = fopen(path, "r");
    if (!f) return set_error(KP_EIO, "kp_table_load: cannot open %s", path);
    std::vector<TableEntry> t;
    char line[512];
    int lineno = 0;
    while (fgets(line, sizeof line, f)) {
        ++lineno;
        char *h = strchr(line, '#');
        if (h) *h = 0;
        char kind[32];
        TableEntry e;
        memset(&e, 0, sizeof e);
        int n = sscanf(line, "%d %d %d %31s %d %d %d %d %d %d %d %d", &e.M, &e.N, &e.K, kind,
                       &e.cfg.split_k, &e.cfg.block, &e.cfg.rows, &e.cfg.k_unroll, &e.cfg.producers,
                       &e.cfg.stages, &e.cfg.flags, &e.overlap);
        if (n <= 0) continue;  // blank or comment
        if (n != 12 || (e.cfg.kind = parse_kind(kind)) < 0 || e.M < 1 || e.N < 1 || e.K < 8) {
            fclose(f);
            return set_error(KP_EIO, "kp_table_load: %s:%d: malformed entry", path, lineno);
        }
        t.push_back(e);
    }
    fclose(f);
    std::lock_guard<std::mutex> lk(g_tab_mu);
    g_table.swap(t);
    return KP_OK;
}

int kp_table_clear(void) {
    std::lock_guard<std::mutex> lk(g_tab_mu);
    g_table.clear();
    return KP_OK;
}

int kp_table_size(void) {
    std::lock_guard<std::mutex> lk(g_tab_mu);
    return static_cast<int>(g_table.size());
}

int kp_select_config(int M, int N, int K, int num_sms, kp_cfg *out) {
    if (!out || M < 1 || N < 1 || K < 8 || (K & 7))
        return set_error(KP_EINVAL, "kp_select_config: bad argument (M=%d N=%d K=%d)", M, N, K);
    if (num_sms <= 0) {
        DevState *d = nullptr;
        int rc = device_state(&d);
        if (rc) return rc;
        num_sms = d->sms;
    }
    *out = select_config(M, N, K, num_sms, nullptr);
    return KP_OK;
}

int kp_scratch_bytes(int M, int N, int K, const kp_cfg *cfg, int num_sms, size_t *bytes) {
    if (!cfg || !bytes || M < 1 || N < 1 || K < 8 || num_sms < 1)
        return set_error(KP_EINVAL, "kp_scratch_bytes: bad argument");
    int rc = check_cfg(M, N, K, *cfg);
    if (rc) return rc;
    Scratch s = scratch_of(M, N, K, *cfg, num_sms);
    *bytes = s.floats * sizeof(float) + s.counters * sizeof(int);
    return KP_OK;
}

// One CTA waits on a barrier that nothing completes; the bounded wait must
// give up after limit_ns, record DEV_SELFTEST and let the kernel exit.
__global__ void selftest_timeout_kernel(int *err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, err, DEV_SELFTEST, limit_ns);
}

int kp_selftest_timeout(int timeout_us, kp_stream_t stream) {
    if (timeout_us < 1 || timeout_us > 1000000)
        return set_error(KP_EINVAL, "kp_selftest_timeout: timeout_us=%d outside 1..1000000", timeout_us);
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        d->err, static_cast<unsigned long long>(timeout_us) * 1000ull);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "kp_selftest_timeout launch");
    return KP_OK;
}

// A dependent kernel (programmatic stream serialisation): lets its own
// dependents launch, waits for its predecessor, then adds the 16-bit patterns
// of n elements into *out, exactly.
__global__ void pdl_consumer_kernel(const uint16_t *buf, int64_t n, unsigned long long *out) {
    pdl_trigger();
    pdl_wait();
    unsigned long long s = 0;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        s += buf[i];
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if ((threadIdx.x & 31) == 0) atomicAdd(out, s);
}

int kp_pdl_consumer_checksum(const void *buf, int64_t n, unsigned long long *out, int pdl,
                             kp_stream_t stream) {
    if (!out || n < 0 || (n > 0 && !buf))
        return set_error(KP_EINVAL, "kp_pdl_consumer_checksum: bad arguments");
    if (reinterpret_cast<uintptr_t>(buf) & 1u)
        return set_error(KP_EALIGN, "kp_pdl_consumer_checksum: buffer must be 2-byte aligned");
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(d->sms), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, pdl_consumer_kernel, static_cast<const uint16_t *>(buf), n, out);
    if (e != cudaSuccess) return cuda_fail(e, "kp_pdl_consumer_checksum launch");
    return KP_OK;
}

int kp_device_error(int *code) {
    if (!code) return set_error(KP_EINVAL, "kp_device_error: NULL");
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    // one atomic read-and-clear: a code written meanwhile is never lost
    *code = __atomic_exchange_n(d->err_host, 0, __ATOMIC_ACQ_REL);
    return KP_OK;
}

int skinny_gemm(const void *x, const void *W, void *y, int M, int N, int K, const kp_cfg *cfg,
                kp_stream_t stream) {
    return skinny_gemm_ex(x, W, nullptr, y, M, N, K, KP_BF16, cfg, stream);
}

int skinny_gemm_ex(const void *x, const void *W, const void *residual, void *y, int M, int N,
                   int K, int dtype, const kp_cfg *cfg, kp_stream_t stream) {
    if (M < 0 || N < 1 || K < 8)
        return set_error(KP_EINVAL, "skinny_gemm: bad sizes M=%d N=%d K=%d", M, N, K);
    if (dtype != KP_BF16 && dtype != KP_FP16)
        return set_error(KP_EINVAL, "skinny_gemm: unknown element type %d", dtype);
    if (K & 7) return set_error(KP_ESHAPE, "skinny_gemm: K=%d is not a multiple of 8", K);
    if (M == 0) return KP_OK;
    if (!x || !W || !y) return set_error(KP_EINVAL, "skinny_gemm: NULL pointer");
    if (!aligned16(x) || !aligned16(W) || !aligned16(y))
        return set_error(KP_EALIGN, "skinny_gemm: pointers must be 16-byte aligned");
    if (residual && (reinterpret_cast<uintptr_t>(residual) & 1u))
        return set_error(KP_EALIGN, "skinny_gemm: the residual must be 2-byte aligned");
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    if ((rc = refuse_after_give_up(d->err_host))) return rc;
    kp_cfg c;
    if (cfg && cfg->kind != KP_KIND_AUTO) {
        c = *cfg;
        if ((rc = check_cfg(M, N, K, c))) return rc;
    } else {
        c = select_config(M, N, K, d->sms, nullptr);
        c.flags &= ~KP_FLAG_FUSE_FB;  // a plan-only flag in a table entry
        if (cfg) c.flags = cfg->flags | (c.flags & ~KP_FLAG_PDL);
        if ((rc = check_cfg(M, N, K, c))) return rc;
    }
    Scratch need = scratch_of(M, N, K, c, d->sms);
    {
        std::lock_guard<std::mutex> lk(g_dev_mu);
        if (need.floats > d->ws_floats || need.counters > d->cnt_n) {
            // Grow (rare; never during capture if the caller warmed up).
            cudaError_t e = cudaDeviceSynchronize();
            if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
            // At least double what is there, so that the replaced buffers
            // (kept, see DevState) add up to less than the final one.
            size_t nf = d->ws_floats, nc = d->cnt_n;
            if (need.floats > nf) nf = need.floats > 2 * nf ? need.floats : 2 * nf;
            if (need.counters > nc) nc = need.counters > 2 * nc ? need.counters : 2 * nc;
            if (nf > d->ws_floats) {
                if (d->ws) d->retired.push_back(d->ws);
                d->ws = nullptr;
                d->ws_floats = 0;
                if ((e = cudaMalloc(&d->ws, nf * sizeof(float))) != cudaSuccess)
                    return cuda_fail(e, "cudaMalloc(scratch)");
                d->ws_floats = nf;
            }
            if (nc > d->cnt_n) {
                if (d->cnt) d->retired.push_back(d->cnt);   // its tickets are all zero
                d->cnt = nullptr;
                d->cnt_n = 0;
                if ((e = cudaMalloc(&d->cnt, nc * sizeof(int))) != cudaSuccess)
                    return cuda_fail(e, "cudaMalloc(counters)");
                if ((e = cudaMemset(d->cnt, 0, nc * sizeof(int))) != cudaSuccess)
                    return cuda_fail(e, "cudaMemset(counters)");
                if ((e = cudaDeviceSynchronize()) != cudaSuccess)
                    return cuda_fail(e, "cudaDeviceSynchronize");
                d->cnt_n = nc;
            }
        }
    }
    GemmArgs a;
    a.x = static_cast<const __nv_bfloat16 *>(x);
    a.ldx = K;
    a.W = static_cast<const __nv_bfloat16 *>(W);
    a.y = static_cast<__nv_bfloat16 *>(y);
    a.ldy = N;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ws = d->ws;
    a.counters = d->cnt;
    a.err = d->err;
    a.dtype = dtype;
    a.res = static_cast<const uint16_t *>(residual);
    a.ldr = N;
    cudaError_t e = launch_gemm(a, c, d->sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "skinny_gemm launch");
    return KP_OK;
}

int kda_proj_plan(int K, int N_qkvg, int N_fab, int N_fb, int max_M, kda_plan **out) {
    if (!out) return set_error(KP_EINVAL, "kda_proj_plan: NULL out");
    *out = nullptr;
    if (K < 8 || N_qkvg < 1 || N_fb < 1 || max_M < 1 || max_M > 65536)
        return set_error(KP_EINVAL, "kda_proj_plan: bad sizes");
    if (K & 7) return set_error(KP_ESHAPE, "kda_proj_plan: K=%d is not a multiple of 8", K);
    if (N_fab < 128 || (N_fab & 7))
        return set_error(KP_ESHAPE, "kda_proj_plan: N_fab=%d must be >= 128 and a multiple of 8",
                         N_fab);
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc) return rc;
    kda_plan *p = new kda_plan();
    p->K = K;
    p->Nq = N_qkvg;
    p->Nfab = N_fab;
    p->Nfb = N_fb;
    p->max_M = max_M;
    cudaGetDevice(&p->dev);
    p->sms = d->sms;
    p->err = d->err;
    p->err_host = d->err_host;
    p->overlap.assign(max_M + 1, 1);
    Scratch need[3];
    for (int b = 0; b < 3; ++b) {
        const BranchShape sh = branch_shape(p, b);
        p->cfg[b].resize(max_M + 1);
        for (int M = 1; M <= max_M; ++M) {
            int ov = 1;
            kp_cfg c = select_config(M, sh.N, sh.K, p->sms, &ov);
            if (c.flags & KP_FLAG_FUSE_FB) {
                // a fused table entry that does not fit this branch: drop the fusion
                if (check_branch_cfg(b, M, sh.N, sh.K, c) != KP_OK) c.flags &= ~KP_FLAG_FUSE_FB;
            }
            if ((rc = check_branch_cfg(b, M, sh.N, sh.K, c))) {
                delete p;
                return rc;
            }
            p->cfg[b][M] = c;
            if (b == KP_BRANCH_QKVG) p->overlap[M] = static_cast<uint8_t>(ov < 0 ? 0 : ov > 2 ? 1 : ov);
            Scratch s = branch_scratch(p, b, M, c);
            if (s.floats > need[b].floats) need[b].floats = s.floats;
            if (s.counters > need[b].counters) need[b].counters = s.counters;
        }
        // Room for any tcgen05 configuration at up to 256 tokens (128 or 256
        // rows per CTA, clusters of up to 16 and at most one CTA per 64-element
        // K block), so kda_proj_set_config can swap them in: the split-K
        // partial tiles are C * Mpad * rows fp32 per tile.
        const int Mh = max_M < 256 ? max_M : 256;
        int Cmax = 16;
        while (Cmax > 1 && Cmax > (sh.K + 63) / 64) Cmax /= 2;
        for (int rows : {128, 256}) {
            if (Cmax < 2) break;
            kp_cfg c = {};
            c.kind = KP_KIND_TC05;
            c.split_k = Cmax;
            c.rows = rows;
            Scratch s = branch_scratch(p, b, Mh, c);
            if (s.floats > need[b].floats) need[b].floats = s.floats;
        }
        // and the CUDA-core kernel's combine tickets (one per CTA row tile, at
        // most one per output row), so a split-K CUDA-core configuration whose
        // partials fit the space above can be swapped in too
        const size_t rows_total = static_cast<size_t>(b == KP_BRANCH_QKVG ? p->Nq + p->Nfab : sh.N);
        if (rows_total > need[b].counters) need[b].counters = rows_total;
    }
    cudaError_t e = cudaSuccess;
    for (int b = 0; b < 3 && e == cudaSuccess; ++b) {
        if (need[b].floats) {
            e = cudaMalloc(&p->ws[b], need[b].floats * sizeof(float));
            if (e == cudaSuccess) p->ws_floats[b] = need[b].floats;
        }
        if (e == cudaSuccess && need[b].counters) {
            e = cudaMalloc(&p->cnt[b], need[b].counters * sizeof(int));
            if (e == cudaSuccess) e = cudaMemset(p->cnt[b], 0, need[b].counters * sizeof(int));
            if (e == cudaSuccess) p->cnt_n[b] = need[b].counters;
        }
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        free_plan_memory(p);
        delete p;
        return cuda_fail(e, "kda_proj_plan: scratch allocation");
    }
    *out = p;
    return KP_OK;
}

int kda_proj_set_overlap(kda_plan *plan, int mode) {
    if (!plan) return set_error(KP_ENOPLAN, "kda_proj_set_overlap: NULL plan");
    if (mode < -1 || mode > 2) return set_error(KP_EINVAL, "kda_proj_set_overlap: mode %d", mode);
    plan->overlap_mode = mode;
    return KP_OK;
}

int kda_proj_overlap_at(const kda_plan *plan, int M) {
    if (!plan || M < 1 || M > plan->max_M) return 0;
    if (plan->overlap_mode >= 0) return plan->overlap_mode;
    return plan->overlap[M];
}

int kda_proj_get_config(const kda_plan *plan, int branch, int M, kp_cfg *out) {
    if (!plan) return set_error(KP_ENOPLAN, "kda_proj_get_config: NULL plan");
    if (!out || branch < 0 || branch > 2 || M < 1 || M > plan->max_M)
        return set_error(KP_EINVAL, "kda_proj_get_config: bad argument");
    *out = plan->cfg[branch][M];
    return KP_OK;
}

int kda_proj_set_config(kda_plan *plan, int branch, int M, const kp_cfg *cfg) {
    if (!plan) return set_error(KP_ENOPLAN, "kda_proj_set_config: NULL plan");
    if (!cfg || branch < 0 || branch > 2 || M < 1 || M > plan->max_M)
        return set_error(KP_EINVAL, "kda_proj_set_config: bad argument");
    const BranchShape sh = branch_shape(plan, branch);
    int rc = check_branch_cfg(branch, M, sh.N, sh.K, *cfg);
    if (rc) return rc;
    Scratch s = branch_scratch(plan, branch, M, *cfg);
    if (s.floats > plan->ws_floats[branch] || s.counters > plan->cnt_n[branch])
        return set_error(KP_ETOOBIG, "kda_proj_set_config: config needs more scratch than the plan holds");
    plan->cfg[branch][M] = *cfg;
    return KP_OK;
}

int kda_proj_run(const kda_plan *plan, const void *x, const void *W_packed, const void *W_fb,
                 void *out_qkvg, void *out_fab, void *out_fb, int M, kp_stream_t main_stream,
                 kp_stream_t aux_stream, kp_event_t events[2]) {
    if (!plan) return set_error(KP_ENOPLAN, "kda_proj_run: NULL plan");
    if (M < 0) return set_error(KP_EINVAL, "kda_proj_run: M=%d", M);
    if (M > plan->max_M)
        return set_error(KP_ETOOBIG, "kda_proj_run: M=%d exceeds the plan's max_M=%d", M, plan->max_M);
    if (M == 0) return KP_OK;
    if (!x || !W_packed || !W_fb || !out_qkvg || !out_fab || !out_fb)
        return set_error(KP_EINVAL, "kda_proj_run: NULL pointer");
    if (!aligned16(x) || !aligned16(W_packed) || !aligned16(W_fb) || !aligned16(out_qkvg) ||
        !aligned16(out_fab) || !aligned16(out_fb))
        return set_error(KP_EALIGN, "kda_proj_run: pointers must be 16-byte aligned");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != plan->dev)
        return set_error(KP_EINVAL, "kda_proj_run: current device %d is not the plan's device %d",
                         dev, plan->dev);
    int rc = refuse_after_give_up(plan->err_host);
    if (rc) return rc;

    const int mode = kda_proj_overlap_at(plan, M);
    const bool overlap = mode == 1 && aux_stream && events && events[0] && events[1];
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
    const __nv_bfloat16 *wp = static_cast<const __nv_bfloat16 *>(W_packed);

    GemmArgs q;
    q.x = xb;
    q.ldx = plan->K;
    q.W = wp;
    q.y = static_cast<__nv_bfloat16 *>(out_qkvg);
    q.ldy = plan->Nq;
    q.M = M;
    q.N = plan->Nq;
    q.K = plan->K;
    q.ws = plan->ws[KP_BRANCH_QKVG];
    q.counters = plan->cnt[KP_BRANCH_QKVG];
    q.err = plan->err;

    GemmArgs f = q;
    f.W = wp + static_cast<int64_t>(plan->Nq) * plan->K;
    f.y = static_cast<__nv_bfloat16 *>(out_fab);
    f.ldy = plan->Nfab;
    f.N = plan->Nfab;
    f.ws = plan->ws[KP_BRANCH_FAB];
    f.counters = plan->cnt[KP_BRANCH_FAB];

    GemmArgs g = q;
    g.x = static_cast<const __nv_bfloat16 *>(out_fab);  // F_A = out_fab[:, 0:128]
    g.ldx = plan->Nfab;
    g.W = static_cast<const __nv_bfloat16 *>(W_fb);
    g.y = static_cast<__nv_bfloat16 *>(out_fb);
    g.ldy = plan->Nfb;
    g.N = plan->Nfb;
    g.K = 128;
    g.ws = plan->ws[KP_BRANCH_FB];
    g.counters = plan->cnt[KP_BRANCH_FB];

    const kp_cfg &cq = plan->cfg[KP_BRANCH_QKVG][M];
    const kp_cfg &cf = plan->cfg[KP_BRANCH_FAB][M];
    const kp_cfg &cb = plan->cfg[KP_BRANCH_FB][M];
    cudaStream_t ms = main_stream;
    cudaStream_t side = overlap ? static_cast<cudaStream_t>(aux_stream) : ms;

    if (mode == 2 && single_launch_ok(plan, M, cq)) {
        // One launch over the packed weight (tcgen05 or CUDA-core kernel, as
        // the Q/K/V/G configuration says): rows [0, N_qkvg) go to out_qkvg,
        // the rest to out_fab, and the cluster that owns the F_A rows computes
        // F_B. Q/K/V/G and F_A/beta tiles run side by side on the SMs.
        GemmArgs a = q;
        a.N = plan->Nq + plan->Nfab;
        SplitOut so;
        so.n_split = plan->Nq;
        so.y2 = f.y;
        so.ldy2 = f.ldy;
        FusedFB fb;
        fb.W = g.W;
        fb.N = g.N;
        fb.y = g.y;
        fb.ld = g.ldy;
        fb.row0 = plan->Nq;
        kp_cfg c = cq;
        c.flags &= ~KP_FLAG_FUSE_FB;
        e = c.kind == KP_KIND_CC ? cc_proj_launch(a, c, so, fb, ms)
                                 : tc05_launch(a, c, plan->sms, ms, &fb, &so);
        if (e != cudaSuccess) return cuda_fail(e, "single-launch projection");
        return KP_OK;
    }

    // F_A/beta, then F_B: one fused launch when the F_A/beta configuration
    // carries KP_FLAG_FUSE_FB (the F_A tile's cluster computes F_B), else two.
    const bool fuse = cf.kind == KP_KIND_TC05 && (cf.flags & KP_FLAG_FUSE_FB) && M <= 256;
    auto launch_aux = [&](cudaStream_t st) -> cudaError_t {
        kp_cfg c = cf;
        c.flags &= ~KP_FLAG_FUSE_FB;
        if (fuse) {
            FusedFB fb;
            fb.W = g.W;
            fb.N = g.N;
            fb.y = g.y;
            fb.ld = g.ldy;
            fb.row0 = 0;
            return tc05_launch(f, c, plan->sms, st, &fb);
        }
        cudaError_t e2 = launch_gemm(f, c, plan->sms, st);
        if (e2 != cudaSuccess) return e2;
        return launch_gemm(g, cb, plan->sms, st);
    };

    if (overlap) {
        if ((e = cudaEventRecord(events[0], ms)) != cudaSuccess) return cuda_fail(e, "fork: cudaEventRecord");
        if ((e = cudaStreamWaitEvent(side, events[0], 0)) != cudaSuccess)
            return cuda_fail(e, "fork: cudaStreamWaitEvent");
        // aux branch first, so its small grids are dispatched before the
        // main-stream kernel spreads over every SM
        if ((e = launch_aux(side)) != cudaSuccess) return cuda_fail(e, "F_A/beta -> F_B launch");
        if ((e = cudaEventRecord(events[1], side)) != cudaSuccess) return cuda_fail(e, "join: cudaEventRecord");
        if ((e = launch_gemm(q, cq, plan->sms, ms)) != cudaSuccess) return cuda_fail(e, "QKVG launch");
        if ((e = cudaStreamWaitEvent(ms, events[1], 0)) != cudaSuccess)
            return cuda_fail(e, "join: cudaStreamWaitEvent");
    } else {
        if ((e = launch_gemm(q, cq, plan->sms, ms)) != cudaSuccess) return cuda_fail(e, "QKVG launch");
        if ((e = launch_aux(ms)) != cudaSuccess) return cuda_fail(e, "F_A/beta -> F_B launch");
    }
    return KP_OK;
}

int kda_proj_destroy(kda_plan *plan) {
    if (!plan) return KP_OK;
    cudaDeviceSynchronize();
    free_plan_memory(plan);
    delete plan;
    return KP_OK;
}

}  // extern "C"
