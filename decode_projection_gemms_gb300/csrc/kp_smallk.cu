// CUDA-core small-K kernel: y = round(x * W^T (+ residual)) for K <= 256,
// bf16 or fp16 elements; the F_B shape
// (out_fb[M, 1024] = f_a[M, 128] * W_fb^T, f_a read in place from the F_A/beta
// output with row stride N_fab) of "[Kimi-K3] Overlap low-M TP8 KDA
// projections" (run_fab_fb; _KdaSkinnyKGemm is the page's kernel for it and
// its body is not shown).
//
// Design: a CTA owns `rows` output features. Their weight rows are copied to
// shared memory (fp32) BEFORE griddepcontrol.wait, so with programmatic
// dependent launch the weight fetch overlaps the tail of the F_A/beta kernel;
// only then are the x rows (which that kernel writes) read. Each thread
// computes whole K-length dot products from shared memory in ascending k.
#include <mutex>
#include <set>

#include "kp_internal.cuh"

namespace kp {

namespace {

constexpr int kMaxK = 256;
constexpr int kMB = 32;  // tokens per pass

// 8 elements of a 16-byte chunk, widened to fp32 into two float4.
__device__ __forceinline__ void widen8(const uint4 v, int dtype, float4 *d) {
    if (dtype == KP_FP16) {
        d[0] = make_float4(elem_lo<KP_FP16>(v.x), elem_hi<KP_FP16>(v.x), elem_lo<KP_FP16>(v.y),
                           elem_hi<KP_FP16>(v.y));
        d[1] = make_float4(elem_lo<KP_FP16>(v.z), elem_hi<KP_FP16>(v.z), elem_lo<KP_FP16>(v.w),
                           elem_hi<KP_FP16>(v.w));
    } else {
        d[0] = make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
        d[1] = make_float4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w));
    }
}

__global__ void __launch_bounds__(256) smallk_kernel(const GemmArgs a, int rows_cta) {
    extern __shared__ float4 sk_smem[];
    const int K = a.K;
    const int KP = K + 4;  // padded row stride (floats): conflict-free 16-byte reads
    float *wsm = reinterpret_cast<float *>(sk_smem);  // [rows_cta][KP]
    float *xsm = wsm + rows_cta * KP;                  // [kMB][KP]
    const int n0 = blockIdx.x * rows_cta;
    const int nrows = min(rows_cta, a.N - n0);
    const int kc = K >> 3;

    for (int i = threadIdx.x; i < nrows * kc; i += blockDim.x) {
        const int r = i / kc;
        const int c = i - r * kc;
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.W + static_cast<int64_t>(n0 + r) * K + 8 * c));
        widen8(v, a.dtype, reinterpret_cast<float4 *>(wsm + r * KP + 8 * c));
    }
    pdl_wait();
    pdl_trigger();

    for (int m0 = 0; m0 < a.M; m0 += kMB) {
        const int mb = min(kMB, a.M - m0);
        __syncthreads();  // weights staged / previous pass finished with xsm
        for (int i = threadIdx.x; i < mb * kc; i += blockDim.x) {
            const int mm = i / kc;
            const int c = i - mm * kc;
            const uint4 v = *reinterpret_cast<const uint4 *>(a.x + (m0 + mm) * a.ldx + 8 * c);
            widen8(v, a.dtype, reinterpret_cast<float4 *>(xsm + mm * KP + 8 * c));
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < rows_cta * mb; idx += blockDim.x) {
            const int r = idx % rows_cta;
            const int mm = idx / rows_cta;
            if (r >= nrows) continue;
            const float4 *wp = reinterpret_cast<const float4 *>(wsm + r * KP);
            const float4 *xp = reinterpret_cast<const float4 *>(xsm + mm * KP);
            float acc = 0.f;
            for (int k4 = 0; k4 < (K >> 2); ++k4) {
                const float4 wv = wp[k4];
                const float4 xv = xp[k4];
                acc = fmaf(wv.x, xv.x, acc);
                acc = fmaf(wv.y, xv.y, acc);
                acc = fmaf(wv.z, xv.z, acc);
                acc = fmaf(wv.w, xv.w, acc);
            }
            const int m = m0 + mm;
            if (a.res) acc += elem_widen(a.res[m * a.ldr + n0 + r], a.dtype);
            reinterpret_cast<uint16_t *>(a.y)[m * a.ldy + n0 + r] = elem_round(acc, a.dtype);
        }
    }
}

std::mutex g_mu;
std::set<int> g_attr_devices;

size_t smem_of(int K, int rows) { return static_cast<size_t>(rows + kMB) * (K + 4) * sizeof(float); }

}  // namespace

bool smallk_supported(int M, int K, const kp_cfg &c) {
    if (M < 1 || K < 8 || K > kMaxK || (K & 7)) return false;
    if (c.rows < 1 || c.rows > 64) return false;
    if (c.block < 32 || c.block > 256 || (c.block & 31)) return false;
    return true;
}

cudaError_t smallk_launch(const GemmArgs &a, const kp_cfg &c, cudaStream_t stream) {
    if (!smallk_supported(a.M, a.K, c)) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_attr_devices.count(dev)) {
            e = cudaFuncSetAttribute(smallk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem_of(kMaxK, 64)));
            if (e != cudaSuccess) return e;
            g_attr_devices.insert(dev);
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.N + c.rows - 1) / c.rows, 1, 1);
    cfg.blockDim = dim3(c.block, 1, 1);
    cfg.dynamicSmemBytes = smem_of(a.K, c.rows);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (c.flags & KP_FLAG_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, smallk_kernel, a, c.rows);
}

}  // namespace kp
