// Host side of the CUDA-core split-K kernel: validation, scratch sizing and
// launch. The kernel itself is in kp_cc_kernel.cuh.
#include <mutex>
#include <set>
#include <utility>

#include "kp_cc_kernel.cuh"

namespace kp {

namespace {

constexpr int kMaxSmem = 200 * 1024;      // x slice
constexpr int kMaxDynSmem = 220 * 1024;   // x slice + weight ring (attribute raised to this; it
                                          // leaves room for the static shared memory)

int cc_variant(int R, int U) {
    for (int v = 0; v < kCCVariants; ++v)
        if (kCCR[v] == R && kCCU[v] == U) return v;
    return -1;
}

// stages: 0 = weights through registers, kCCRing = the shared-memory ring form.
CCKernelFn cc_kernel(int M, int R, int U, int dtype, int stages) {
    const int v = cc_variant(R, U);
    if (v < 0 || M < 1 || M > 16 || (dtype != KP_BF16 && dtype != KP_FP16)) return nullptr;
    if (stages == kCCRing) {
        if (dtype == KP_FP16) return M <= 8 ? cc_ring_lo_fp16[M - 1][v] : cc_ring_hi_fp16[M - 9][v];
        return M <= 8 ? cc_ring_lo_bf16[M - 1][v] : cc_ring_hi_bf16[M - 9][v];
    }
    if (stages != 0) return nullptr;
    if (dtype == KP_FP16) return M <= 8 ? cc_table_lo_fp16[M - 1][v] : cc_table_hi_fp16[M - 9][v];
    return M <= 8 ? cc_table_lo_bf16[M - 1][v] : cc_table_hi_bf16[M - 9][v];
}

// Dynamic shared memory of a launch: the x slice (16-bit), then the ring.
size_t cc_smem_bytes(int M, int Ks, const kp_cfg &c, int *ring_off) {
    const size_t xs = (static_cast<size_t>(M) * Ks * 2 + 15) & ~static_cast<size_t>(15);
    if (ring_off) *ring_off = static_cast<int>(xs);
    if (c.stages == 0) return xs;
    return xs + cc_ring_bytes(c.block / 32, c.stages, c.rows, c.k_unroll);
}

// K slice length: ceil(K / S) rounded up to 8 elements (16 bytes).
int cc_slice(int K, int S) {
    int ks = (K + S - 1) / S;
    return (ks + 7) & ~7;
}

std::mutex g_attr_mu;
std::set<std::pair<const void *, int>> g_attr_done;  // (kernel, device) raised to kMaxSmem

cudaError_t ensure_smem_attr(const void *fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (g_attr_done.count({fn, dev})) return cudaSuccess;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e == cudaSuccess) g_attr_done.insert({fn, dev});
    return e;
}

}  // namespace

bool cc_supported(int M, int K, const kp_cfg &c) {
    if (M < 1 || M > 16 || K < 8 || (K & 7)) return false;
    if (c.split_k < 1 || c.split_k > K / 8) return false;
    if (c.block < 32 || c.block > 512 || (c.block & 31)) return false;
    if (!cc_kernel(M, c.rows, c.k_unroll, KP_BF16, c.stages)) return false;  // same set for fp16
    const int ks = cc_slice(K, c.split_k);
    if (static_cast<long long>(M) * ks * 2 > kMaxSmem) return false;  // x slice (16-bit) fits in shared memory
    return cc_smem_bytes(M, ks, c, nullptr) <= static_cast<size_t>(kMaxDynSmem);   // and the ring beside it
}

Scratch cc_scratch(int M, int N, int K, const kp_cfg &c) {
    Scratch s;
    const int ks = cc_slice(K, c.split_k);
    const int S = (K + ks - 1) / ks;
    if (S > 1) {
        const int rows_cta = (c.block / 32) * c.rows;
        s.floats = static_cast<size_t>(S) * M * N;
        s.counters = static_cast<size_t>((N + rows_cta - 1) / rows_cta);
    }
    return s;
}

bool cc_proj_supported(int M, int K, int N, const kp_cfg &c, int n_split) {
    if (M < 1 || M > 8 || c.kind != KP_KIND_CC || c.split_k != 1 || c.stages != 0 || !cc_supported(M, K, c))
        return false;
    if (!cc_table_proj[M - 1][cc_variant(c.rows, c.k_unroll)]) return false;
    const int rows_cta = (c.block / 32) * c.rows;
    if (rows_cta > kFaWidth || kFaWidth % rows_cta) return false;   // F_A rows = whole CTAs
    if (kFaWidth / rows_cta > 8) return false;                        // portable cluster size
    return n_split > 0 && n_split % kFaWidth == 0 && N - n_split >= kFaWidth;
}

cudaError_t cc_proj_launch(const GemmArgs &a, const kp_cfg &c, const SplitOut &so, const FusedFB &fb,
                           cudaStream_t stream) {
    if (!cc_proj_supported(a.M, a.K, a.N, c, so.n_split) || fb.row0 != so.n_split ||
        a.dtype != KP_BF16 || a.res)
        return cudaErrorInvalidValue;
    CCKernelFn fn = cc_table_proj[a.M - 1][cc_variant(c.rows, c.k_unroll)];
    CCParams p;
    p.a = a;
    p.Ks = cc_slice(a.K, 1);
    p.S = 1;
    p.rows_cta = (c.block / 32) * c.rows;
    p.ring_off = 0;
    CCProj &q = p.proj;
    q.n_split = so.n_split;
    q.y2 = so.y2;
    q.ldy2 = so.ldy2;
    q.fa_ctas = kFaWidth / p.rows_cta;
    q.fa_tile0 = so.n_split / p.rows_cta;
    const int tiles = (a.N + p.rows_cta - 1) / p.rows_cta;
    q.n_tiles = (tiles + q.fa_ctas - 1) / q.fa_ctas * q.fa_ctas;
    q.Wfb = fb.W;
    q.N_fb = fb.N;
    q.yfb = fb.y;
    q.ldfb = fb.ld;
    const size_t smem = static_cast<size_t>(a.M) * p.Ks * 2;
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(fn));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(q.n_tiles, 1, 1);
    cfg.blockDim = dim3(c.block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = q.fa_ctas;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    if (c.flags & KP_FLAG_PDL) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

cudaError_t cc_launch(const GemmArgs &a, const kp_cfg &c, cudaStream_t stream) {
    if (!cc_supported(a.M, a.K, c)) return cudaErrorInvalidValue;
    CCKernelFn fn = cc_kernel(a.M, c.rows, c.k_unroll, a.dtype, c.stages);
    if (!fn) return cudaErrorInvalidValue;
    CCParams p;
    p.a = a;
    p.Ks = cc_slice(a.K, c.split_k);
    p.S = (a.K + p.Ks - 1) / p.Ks;
    p.rows_cta = (c.block / 32) * c.rows;
    const int tiles = (a.N + p.rows_cta - 1) / p.rows_cta;
    const size_t smem = cc_smem_bytes(a.M, p.Ks, c, &p.ring_off);   // x slice (16-bit) + ring
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void *>(fn));
    if (e != cudaSuccess) return e;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, p.S, 1);
    cfg.blockDim = dim3(c.block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (c.flags & KP_FLAG_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace kp
