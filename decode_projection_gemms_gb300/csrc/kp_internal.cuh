// Internal declarations and sm_103a PTX helpers shared by the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kdaproj.h"

namespace kp {

// ---------------------------------------------------------------------------
// Launch descriptions handed from the API layer to the kernel launchers.

struct GemmArgs {
    const __nv_bfloat16 *x;  // [M, ldx]
    int64_t ldx;             // x row stride in elements
    const __nv_bfloat16 *W;  // [N, K], row stride K
    __nv_bfloat16 *y;        // [M, ldy]
    int64_t ldy;
    int M, N, K;
    float *ws;               // split-K partials (may be null if unused)
    int *counters;           // per-tile tickets, zero between launches
    int *err;                // error word (mapped host memory, device view)
    // Element type of x, W, y and the residual (KP_BF16 or KP_FP16; the
    // pointers above are raw 16-bit storage), and an optional residual
    // [M, ldr] added to the fp32 sum before the one rounding.
    int dtype = KP_BF16;
    const uint16_t *res = nullptr;
    int64_t ldr = 0;
};

// Scratch requirement of a configuration (floats and counters).
struct Scratch {
    size_t floats = 0;
    size_t counters = 0;
};

// CUDA-core split-K kernel (kp_cc.cu)
bool cc_supported(int M, int K, const kp_cfg &c);
Scratch cc_scratch(int M, int N, int K, const kp_cfg &c);
cudaError_t cc_launch(const GemmArgs &a, const kp_cfg &c, cudaStream_t s);

// F_B fused into the F_A/beta launch: rows [row0, row0 + 128) of that GEMM are
// F_A (row0 a multiple of the configuration's rows per CTA);
// y = bf16(bf16(F_A) * W^T) with W [N, 128].
struct FusedFB {
    const __nv_bfloat16 *W;
    int N;
    __nv_bfloat16 *y;
    int64_t ld;
    int row0;
};

// Rows n >= n_split of a GEMM's output go to a second matrix y2 (row
// n - n_split, row stride ldy2); n_split must be a multiple of 128.
struct SplitOut {
    int n_split;
    __nv_bfloat16 *y2;
    int64_t ldy2;
};

// CUDA-core single-launch projection (kp_cc.cu): one K slice over the packed
// weight, rows >= split.n_split to split.y2, F_B computed by the cluster of
// the F_A rows (fb.row0 == split.n_split); bf16, M <= 8.
bool cc_proj_supported(int M, int K, int N, const kp_cfg &c, int n_split);
cudaError_t cc_proj_launch(const GemmArgs &a, const kp_cfg &c, const SplitOut &split, const FusedFB &fb,
                           cudaStream_t s);

// tcgen05 cluster split-K kernel (kp_tc05.cu)
bool tc05_supported(int M, int N, int K, const kp_cfg &c);
bool tc05_fusable(int M, const kp_cfg &c);
Scratch tc05_scratch(int M, int N, int K, const kp_cfg &c, int num_sms);
cudaError_t tc05_launch(const GemmArgs &a, const kp_cfg &c, int num_sms, cudaStream_t s,
                        const FusedFB *fb = nullptr, const SplitOut *split = nullptr);
int tc05_max_stages(int M);
int tc05_rows(const kp_cfg &c);   // feature rows per CTA of a configuration (128 or 256)
kp_cfg tc05_default(int M, int N, int K, int num_sms);

// small-K kernel (kp_smallk.cu)
bool smallk_supported(int M, int K, const kp_cfg &c);
cudaError_t smallk_launch(const GemmArgs &a, const kp_cfg &c, cudaStream_t s);

// error reporting shared with the API layer (kp_api.cu)
int set_error(int code, const char *fmt, ...);

// Device error codes written to the error word.
enum DevErr {
    DEV_OK = 0,
    DEV_TIMEOUT_FULL = 1,     // MMA warp waited too long for a TMA stage
    DEV_TIMEOUT_EMPTY = 2,    // producer waited too long for a free stage
    DEV_TIMEOUT_ACC_FULL = 3, // epilogue waited too long for an accumulator
    DEV_TIMEOUT_ACC_EMPTY = 4, // MMA warp waited too long for a free accumulator
    DEV_SELFTEST = 5           // kp_selftest_timeout's wait ran out (as it must)
};

}  // namespace kp

// ---------------------------------------------------------------------------
// Device helpers (inline PTX). Only compiled for the device pass.
#if defined(__CUDACC__)

namespace kp {

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// The two 16-bit input types, as compile-time (T) or run-time (dtype)
// choices: KP_BF16 or KP_FP16. lo/hi widen the low/high element of a 32-bit
// word; round converts fp32 to the type's bits (round to nearest even).
template <int T>
__device__ __forceinline__ float elem_lo(uint32_t v) {
    if constexpr (T == KP_FP16)
        return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
    else
        return bf16lo(v);
}
template <int T>
__device__ __forceinline__ float elem_hi(uint32_t v) {
    if constexpr (T == KP_FP16)
        return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
    else
        return bf16hi(v);
}
template <int T>
__device__ __forceinline__ uint16_t elem_round(float f) {
    if constexpr (T == KP_FP16)
        return __half_as_ushort(__float2half_rn(f));
    else
        return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float elem_widen(uint16_t b, int dtype) {
    return dtype == KP_FP16 ? __half2float(__ushort_as_half(b)) : __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ uint16_t elem_round(float f, int dtype) {
    return dtype == KP_FP16 ? elem_round<KP_FP16>(f) : elem_round<KP_BF16>(f);
}

// acc + w.lo * x.lo, then + w.hi * x.hi, for two 16-bit elements (bf16 or fp16,
// T) packed in each 32-bit word. The mixed-precision FMA takes the 16-bit
// operands directly: their product is exact in fp32 (8- or 11-bit
// significands) and each step rounds once, exactly as widening both to fp32
// and calling fmaf would.
template <int T>
__device__ __forceinline__ float fma_pair(uint32_t w, uint32_t x, float acc) {
    if constexpr (T == KP_FP16)
        asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
            "mov.b32 {wl, wh}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
            "fma.rn.f32.f16 %0, wl, xl, %0;\n\tfma.rn.f32.f16 %0, wh, xh, %0;\n\t}"
            : "+f"(acc)
            : "r"(w), "r"(x));
    else
        asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
            "mov.b32 {wl, wh}, %1;\n\tmov.b32 {xl, xh}, %2;\n\t"
            "fma.rn.f32.bf16 %0, wl, xl, %0;\n\tfma.rn.f32.bf16 %0, wh, xh, %0;\n\t}"
            : "+f"(acc)
            : "r"(w), "r"(x));
    return acc;
}

// Programmatic dependent launch. Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 policies for the weight stream (read once) and reused operands.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 16-byte streaming load of weights: read-only path, no L1 allocation,
// evict-first in L2.
__device__ __forceinline__ uint4 ldg_stream(const void *p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ---------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: spins on the barrier phase; after `limit_ns` of wall time
// (~1 s by default; or once another wait in this CTA has given up) it records
// `code` in the error word, raises the CTA's abort flag and returns false. The
// caller then proceeds as if the phase had completed: every address it touches
// stays in bounds, so a broken pipeline yields wrong numbers and an error
// code, never a hang.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int *abort_flag, int *err,
                                                  int code, uint64_t limit_ns = 1000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            if (err) atomicCAS_system(err, 0, code);   // host-mapped word
            return false;
        }
    }
}

// ---- TMA --------------------------------------------------------------------
// Contiguous bulk copy global -> this CTA's shared memory, completing `bytes`
// of transaction on the mbarrier. Both addresses 16-byte aligned, bytes a
// multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const void *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Prefetch a 2-D tile of a tensor map into L2 (no shared-memory destination).
__device__ __forceinline__ void tma_prefetch_l2_2d(const void *map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *map, uint32_t bar, int c0,
                                            int c1, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *map, uint32_t bar, int c0,
                                            int c1, int c2, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
        : "memory");
}

// ---- tcgen05 ----------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on an mbarrier once all previously issued MMAs of this thread finish.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns; thread i gets lane (base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
          "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- thread-block clusters ----------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Hardware barrier over every thread of every CTA in the cluster, with
// release/acquire ordering of shared-memory writes (all threads must call it).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Named barrier among `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace kp

#endif  // __CUDACC__
