// CUDA-core split-K weight-streaming GEMV for M <= 16 tokens.
//
// y[m, n] = round( sum_k x[m, k] * W[n, k] (+ residual[m, n]) ), fp32
// accumulation, bf16 or fp16 elements (template T): the skinny
// GEMM of the Kimi K3 support page, part 1 (vllm PR #50089 digest, CuteSkinnyGemm, section
// "关键源码片段"), whose design is prior art here: CUDA-core FMAs over 16-byte
// vector loads, warp-shuffle row reductions, M unrolled at compile time.
// Differences from that design: the K range is split over blockIdx.y (split-K)
// so small-N shapes still fill all SMs, x's K slice is staged once per CTA in
// shared memory in its own 16-bit type (one bulk copy per token, issued by one
// thread, so staging costs one round trip), each warp owns `R` output rows,
// the products use the mixed-precision FMA on the 16-bit operands directly (no
// widening instructions), and the S partial sums of a row tile are combined
// deterministically by the last CTA to finish (ticket counter, sum in split
// order 0..S-1, plus the residual if any, one rounding to the element type).
//
// Grid: (row tiles, S). Block: `block` threads, warp w owns rows
// tile*rows_cta + w*R .. +R-1. Lane l reads the 16-byte chunks l, l+32, ... of
// the CTA's K slice for each of its rows, U chunks per row at a time (a
// batch). Two batches are in flight per lane in registers, or (NS > 0) NS - 1
// batches in a per-warp ring in shared memory filled by asynchronous copies, so
// the bytes in flight are not bounded by the registers.
#pragma once

#include "kp_internal.cuh"

namespace kp {

constexpr int kXPieces = 8;   // x slice staged in at most this many K ranges

// The whole projection in one launch over a packed weight (kProj kernels,
// one K slice): rows >= n_split of the output go to y2, and the CTAs that
// own the 128 F_A rows [n_split, n_split + 128) form one thread-block cluster
// that also computes F_B = bf16(F_A) * W_fb^T (K = 128).
struct CCProj {
    int n_split;             // first F_A/beta row; a multiple of 128
    __nv_bfloat16 *y2;       // F_A/beta output [M, ldy2]
    int64_t ldy2;
    int fa_tile0;            // first tile of the F_A rows
    int fa_ctas;             // CTAs over the F_A rows = the cluster size
    int n_tiles;             // tiles in the grid, a multiple of fa_ctas
    const __nv_bfloat16 *Wfb;  // [N_fb, 128]
    int N_fb;
    __nv_bfloat16 *yfb;      // [M, ldfb]
    int64_t ldfb;
};

struct CCParams {
    GemmArgs a;
    int Ks;       // K slice length (multiple of 8)
    int S;        // number of K slices (gridDim.y)
    int rows_cta; // output rows per CTA
    int ring_off; // NS > 0: byte offset of the weight ring in dynamic shared memory
    CCProj proj;  // kProj kernels only
};

// Number of 16-byte chunks per lane, row and batch slot of the ring: warp w's
// ring holds NS slots x R rows x U chunks x 32 lanes of 16 bytes.
constexpr uint32_t cc_ring_bytes(int warps, int NS, int R, int U) {
    return static_cast<uint32_t>(warps) * NS * R * U * 32 * 16;
}

// 16-byte asynchronous copy global -> shared (L2 policy hint), and the group
// bookkeeping of those copies.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

constexpr int kFaWidth = 128;   // F_A columns = F_B's K

// Store one output: the residual (if any) joins the fp32 sum, then one rounding.
template <int T>
__device__ __forceinline__ void cc_store(const GemmArgs &a, int m, int n, float v) {
    if (a.res) v += elem_widen(a.res[m * a.ldr + n], T);
    reinterpret_cast<uint16_t *>(a.y)[m * a.ldy + n] = elem_round<T>(v);
}

// CTAs per SM the kernel is compiled for. The single-launch form's F_B code
// needs registers the plain kernel does not. Where the main loop fits in 64
// registers, this form also asks for two 512-thread CTAs per SM (64 registers
// each, the F_B part may spill), as the plain kernel gets by itself. With one
// CTA per SM, a 16-row, 512-thread configuration at M = 1 took 20.7 instead of
// 11.8 us per call.
template <int M, int R, int U, int NS, bool kProj>
constexpr int cc_min_blocks() {
    return kProj && (NS > 0 ? 1 : 2) * R * U * 4 + R * M + 24 <= 60 ? 2 : 1;
}

// kProj: the single-launch projection (bf16, one K slice; CCProj above).
// NS: 0 = weights in registers (two batches); > 1 = NS-slot shared-memory ring.
template <int M, int R, int U, int T, bool kProj = false, int NS = 0>
// At most 128 registers per thread: two 256-thread CTAs or one 512-thread CTA
// per SM (64 and two 512-thread CTAs for the small single-launch forms).
__global__ void __launch_bounds__(512, (cc_min_blocks<M, R, U, NS, kProj>())) cc_gemv_kernel(const CCParams p) {
    extern __shared__ __align__(16) uint8_t cc_smem[];
    const uint16_t *xs = reinterpret_cast<const uint16_t *>(cc_smem);  // [M][Ks], 16-bit
    // x's slice lands in up to kXPieces K ranges, each on its own barrier, so
    // the first chunks can be used while the rest are still in flight.
    __shared__ __align__(8) uint64_t xbar[kXPieces];
    __shared__ int abort_flag;

    const GemmArgs &a = p.a;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    int tile = blockIdx.x;
    if constexpr (kProj) {
        // The F_A cluster is dispatched first (its F_B epilogue is the
        // longest); CTAs wholly past N (padding to whole clusters) leave.
        tile = (static_cast<int>(blockIdx.x) + p.proj.fa_tile0) % p.proj.n_tiles;
        if (tile * p.rows_cta >= p.a.N) return;
    }
    const bool fa_cta = kProj && tile >= p.proj.fa_tile0 && tile < p.proj.fa_tile0 + p.proj.fa_ctas;
    const int s = blockIdx.y;
    const int row0 = tile * p.rows_cta + warp * R;
    const int k0 = s * p.Ks;
    const int klen = min(p.Ks, a.K - k0);
    const int nchunk = klen >> 3;
    const uint64_t pol = policy_evict_first();
    // The warp covers 64*U chunks per loop iteration; a piece of x is a whole
    // number of iterations.
    constexpr int kStep = 64 * U;
    const int iters = (nchunk + kStep - 1) / kStep;
    const int ipp = iters > kXPieces ? (iters + kXPieces - 1) / kXPieces : 1;   // iterations per piece
    const int pieces = (iters + ipp - 1) / ipp;

    if (threadIdx.x == 0) {
        for (int i = 0; i < pieces; ++i) mbar_init(smem_u32(&xbar[i]), 1);
        abort_flag = 0;
        fence_mbar_init();
        if (fa_cta) {
            // W_fb does not depend on the previous kernel: pull this CTA's F_B
            // weight rows into L2 now, so the F_B loads after the main loop hit
            const int rows_fb = (p.proj.N_fb + p.proj.fa_ctas - 1) / p.proj.fa_ctas;
            const int fb0 = (tile - p.proj.fa_tile0) * rows_fb;
            const int nfb = min(rows_fb, p.proj.N_fb - fb0);
            if (nfb > 0)
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                                 p.proj.Wfb + static_cast<int64_t>(fb0) * kFaWidth),
                             "r"(static_cast<uint32_t>(nfb) * kFaWidth * 2)
                             : "memory");
        }
    }

    // Rows past N read row N-1 (always valid) and are never stored.
    const __nv_bfloat16 *wrow[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int n = min(row0 + r, a.N - 1);
        wrow[r] = a.W + static_cast<int64_t>(n) * a.K + k0;
    }

    // Two batches of U chunks per row in flight per warp (double buffering):
    // the next batch is requested before the current one is consumed.
    auto load_batch = [&](uint4 (&w)[R][U], int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + 32 * u;
#pragma unroll
            for (int r = 0; r < R; ++r)
                w[r][u] = (c < nchunk) ? ldg_stream(wrow[r] + 8 * c, pol) : make_uint4(0, 0, 0, 0);
        }
    };
    // Ring form: batch b (chunks lane + 32 * (b * U + u)) goes to slot b % NS
    // of this warp's ring; a lane reads back only the chunks it copied, so the
    // copies' own completion (wait_group) is the only synchronisation.
    const int nb = (nchunk + 32 * U - 1) / (32 * U);   // batches of this lane's warp
    const uint4 *ring = reinterpret_cast<const uint4 *>(cc_smem + p.ring_off) +
                        static_cast<size_t>(warp) * (NS > 0 ? NS : 1) * R * U * 32 + lane;
    auto slot = [&](int st, int r, int u) { return ((st * R + r) * U + u) * 32; };
    auto issue = [&](int b) {
        if constexpr (NS > 0) {
            if (b < nb) {
                const int st = b % NS;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = lane + 32 * (b * U + u);
                    if (c < nchunk)
#pragma unroll
                        for (int r = 0; r < R; ++r) cp_async16(smem_u32(ring + slot(st, r, u)), wrow[r] + 8 * c, pol);
                }
            }
            cp_async_commit();   // one group per batch index, empty past the end
        }
    };

    float acc[R][M];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

    // Chunk c holds elements 8c .. 8c+7 of the slice; each accumulator takes
    // them in ascending order.
    auto compute = [&](const uint4 (&w)[R][U], int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + 32 * u;
            if (c < nchunk) {
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const uint4 xv = *reinterpret_cast<const uint4 *>(xs + m * p.Ks + 8 * c);
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        float t = acc[r][m];
                        t = fma_pair<T>(w[r][u].x, xv.x, t);
                        t = fma_pair<T>(w[r][u].y, xv.y, t);
                        t = fma_pair<T>(w[r][u].z, xv.z, t);
                        t = fma_pair<T>(w[r][u].w, xv.w, t);
                        acc[r][m] = t;
                    }
                }
            }
        }
    };

    // Weights never depend on the previous kernel: start streaming them
    // before waiting for it.
    uint4 wa[R][U], wb[R][U];
    if constexpr (NS > 0) {
        for (int b = 0; b < NS - 1; ++b) issue(b);
    } else {
        load_batch(wa, lane);
    }
    __syncthreads();   // the barrier's initialisation is visible to every waiter
    pdl_wait();
    pdl_trigger();

    // Stage x[0:M, k0:k0+klen] (rows of klen 16-bit elements, 16-byte aligned
    // since K, ldx and the slice start are multiples of 8): per piece, one bulk
    // copy per token.
    if (threadIdx.x == 0) {
        for (int i = 0; i < pieces; ++i) {
            const int ca = i * ipp * kStep;
            const int cb = min(nchunk, (i + 1) * ipp * kStep);
            const uint32_t bytes = static_cast<uint32_t>(cb - ca) * 16;
            mbar_expect_tx(smem_u32(&xbar[i]), bytes * M);
#pragma unroll
            for (int m = 0; m < M; ++m)
                bulk_load(smem_u32(xs + m * p.Ks + 8 * ca), a.x + m * a.ldx + k0 + 8 * ca, bytes,
                          smem_u32(&xbar[i]));
        }
    }

    auto wait_x = [&](int j) {   // x piece of iteration j (kStep chunks) landed
        if (j % ipp == 0 &&
            !mbar_wait_bounded(smem_u32(&xbar[j / ipp]), 0, &abort_flag, a.err, DEV_TIMEOUT_FULL) &&
            threadIdx.x == 0) {
            // x never landed: let the copies finish (bounded) before the CTA's
            // shared memory is released; the outputs are undefined (error word set)
            const uint64_t t0 = globaltimer_ns();
            for (int i = 0; i < pieces; ++i)
                while (!mbar_try_wait(smem_u32(&xbar[i]), 0) && globaltimer_ns() - t0 < 1000000000ull) {
                }
        }
    };
    if constexpr (NS > 0) {
        for (int b = 0; b < nb; ++b) {
            if ((b & 1) == 0) wait_x(b >> 1);
            cp_async_wait<NS - 2>();   // this lane's batch b has landed
            issue(b + NS - 1);         // into the slot batch b - 1 used
            const int st = b % NS;
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < R; ++r) wa[r][u] = ring[slot(st, r, u)];
            compute(wa, lane + 32 * U * b);
        }
        cp_async_wait<0>();
    } else {
        for (int j = 0; j < iters; ++j) {
            wait_x(j);
            const int c0 = lane + j * kStep;
            const int c1 = c0 + 32 * U;
            const int c2 = c1 + 32 * U;
            if (c1 < nchunk) load_batch(wb, c1);
            compute(wa, c0);
            if (c2 < nchunk) load_batch(wa, c2);
            if (c1 < nchunk) compute(wb, c1);
        }
    }

    // Butterfly reduction over the 32 lanes: every lane ends with the sums.
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float v = acc[r][m];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            acc[r][m] = v;
        }

    if constexpr (kProj) {
        // One K slice; rows < n_split to y, the rest to y2. The F_A cluster
        // also hands each rounded F_A value to every CTA of the cluster.
        __shared__ __align__(16) uint16_t fa_s[M][kFaWidth];   // bf16 F_A, every token
        const int fa_row0 = p.proj.n_split;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const int n = row0 + r;
                if (lane == ((r * M + m) & 31) && n < a.N) {
                    const uint16_t b = elem_round<KP_BF16>(acc[r][m]);
                    if (n < p.proj.n_split)
                        reinterpret_cast<uint16_t *>(a.y)[m * a.ldy + n] = b;
                    else
                        reinterpret_cast<uint16_t *>(p.proj.y2)[m * p.proj.ldy2 + (n - p.proj.n_split)] = b;
                    if (fa_cta) {
                        const uint32_t off = smem_u32(&fa_s[m][n - fa_row0]);
                        for (int c = 0; c < p.proj.fa_ctas; ++c)
                            asm volatile("st.shared::cluster.b16 [%0], %1;" ::"r"(
                                             mapa_shared(off, static_cast<uint32_t>(c))),
                                         "h"(b)
                                         : "memory");
                    }
                }
            }
        if (!fa_cta) return;
        // F_B rows of this CTA: one thread per row, k = 0..127 in ascending
        // order, fp32 accumulation, one rounding. The first row's weights are
        // requested before the cluster barrier (they do not depend on F_A), so
        // their L2 round trip overlaps the wait for the slowest peer.
        const int rows_fb = (p.proj.N_fb + p.proj.fa_ctas - 1) / p.proj.fa_ctas;
        const int fb0 = (tile - p.proj.fa_tile0) * rows_fb;
        uint4 w[kFaWidth / 8];
        auto load_fb_row = [&](int n) {
            const uint4 *wr = reinterpret_cast<const uint4 *>(p.proj.Wfb + static_cast<int64_t>(n) * kFaWidth);
#pragma unroll
            for (int c = 0; c < kFaWidth / 8; ++c) w[c] = __ldg(wr + c);
        };
        if (static_cast<int>(threadIdx.x) < rows_fb && fb0 + static_cast<int>(threadIdx.x) < p.proj.N_fb)
            load_fb_row(fb0 + threadIdx.x);
        // Every CTA of the cluster holds the whole bf16 F_A after this barrier.
        cluster_sync_all();
        for (int t = threadIdx.x; t < rows_fb; t += blockDim.x) {
            const int n = fb0 + t;
            if (n >= p.proj.N_fb) break;
            if (t != static_cast<int>(threadIdx.x)) load_fb_row(n);
            float f[M];
#pragma unroll
            for (int m = 0; m < M; ++m) f[m] = 0.f;
#pragma unroll
            for (int c = 0; c < kFaWidth / 8; ++c)
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const uint4 xv = *reinterpret_cast<const uint4 *>(&fa_s[m][8 * c]);
                    f[m] = fma_pair<KP_BF16>(w[c].x, xv.x, f[m]);
                    f[m] = fma_pair<KP_BF16>(w[c].y, xv.y, f[m]);
                    f[m] = fma_pair<KP_BF16>(w[c].z, xv.z, f[m]);
                    f[m] = fma_pair<KP_BF16>(w[c].w, xv.w, f[m]);
                }
#pragma unroll
            for (int m = 0; m < M; ++m)
                reinterpret_cast<uint16_t *>(p.proj.yfb)[m * p.proj.ldfb + n] = elem_round<KP_BF16>(f[m]);
        }
        return;
    } else if (p.S == 1) {
        // One K slice: round and store directly; lane j stores value j.
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < M; ++m) {
                const int n = row0 + r;
                if (lane == ((r * M + m) & 31) && n < a.N) cc_store<T>(a, m, n, acc[r][m]);
            }
        return;
    }

    if constexpr (!kProj) {
        // Split-K: write this slice's partials to ws[s][m][n] ...
    #pragma unroll
        for (int r = 0; r < R; ++r)
    #pragma unroll
            for (int m = 0; m < M; ++m) {
                const int n = row0 + r;
                if (lane == ((r * M + m) & 31) && n < a.N)
                    a.ws[(static_cast<int64_t>(s) * M + m) * a.N + n] = acc[r][m];
            }
        // ... then take a ticket; the CTA that takes the last one sums the S
        // partials of the tile in slice order and stores bf16. It never waits.
        __shared__ int s_last;
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const int prev = atomicAdd(a.counters + tile, 1);
            s_last = (prev == p.S - 1);
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        const int tile_row0 = tile * p.rows_cta;
        for (int i = threadIdx.x; i < M * p.rows_cta; i += blockDim.x) {
            const int m = i / p.rows_cta;
            const int n = tile_row0 + (i - m * p.rows_cta);
            if (n >= a.N) continue;
            // partials summed in slice order 0..S-1; loads issued 8 at a time
            float t = 0.f;
            for (int q0 = 0; q0 < p.S; q0 += 8) {
                float v[8];
    #pragma unroll
                for (int j = 0; j < 8; ++j)
                    v[j] = (q0 + j < p.S)
                               ? __ldcg(a.ws + (static_cast<int64_t>(q0 + j) * M + m) * a.N + n)
                               : 0.f;
    #pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (q0 + j < p.S) t += v[j];
            }
            cc_store<T>(a, m, n, t);
        }
        if (threadIdx.x == 0) a.counters[tile] = 0;  // ready for the next launch
    }
}

using CCKernelFn = void (*)(const CCParams);

// (R, U) variants instantiated for every M in 1..16.
constexpr int kCCVariants = 6;
constexpr int kCCR[kCCVariants] = {1, 2, 2, 4, 4, 8};
constexpr int kCCU[kCCVariants] = {4, 2, 4, 1, 2, 1};

}  // namespace kp

namespace kp {

// Kernel pointer for (M, variant, element type), or nullptr where the R*M
// accumulators would not fit in the 128 registers a thread gets.
template <int M, int V, int T>
constexpr CCKernelFn cc_pick() {
    if constexpr (kCCR[V] * M <= 64 && (kCCR[V] < 8 || M <= 4))
        return cc_gemv_kernel<M, kCCR[V], kCCU[V], T>;
    else
        return nullptr;
}

// The ring form of the same kernel (a 4-slot shared-memory weight ring).
constexpr int kCCRing = 4;
template <int M, int V, int T>
constexpr CCKernelFn cc_pick_ring() {
    if constexpr (kCCR[V] * M <= 64 && (kCCR[V] < 8 || M <= 4))
        return cc_gemv_kernel<M, kCCR[V], kCCU[V], T, false, kCCRing>;
    else
        return nullptr;
}

// The single-launch projection kernel for (M, variant), bf16, M <= 8.
template <int M, int V>
constexpr CCKernelFn cc_pick_proj() {
    if constexpr (kCCR[V] * M <= 64 && (kCCR[V] < 8 || M <= 4))
        return cc_gemv_kernel<M, kCCR[V], kCCU[V], KP_BF16, true>;
    else
        return nullptr;
}

#define KP_CC_ROW(M, T)                                                                    \
    {                                                                                      \
        cc_pick<M, 0, T>(), cc_pick<M, 1, T>(), cc_pick<M, 2, T>(), cc_pick<M, 3, T>(),   \
            cc_pick<M, 4, T>(), cc_pick<M, 5, T>()                                         \
    }

#define KP_CC_RING_ROW(M, T)                                                                              \
    {                                                                                                     \
        cc_pick_ring<M, 0, T>(), cc_pick_ring<M, 1, T>(), cc_pick_ring<M, 2, T>(), cc_pick_ring<M, 3, T>(), \
            cc_pick_ring<M, 4, T>(), cc_pick_ring<M, 5, T>()                                              \
    }

// [M - 1 within the half][variant], one table per half and element type
extern const CCKernelFn cc_table_lo_bf16[8][kCCVariants];  // M = 1..8
extern const CCKernelFn cc_table_hi_bf16[8][kCCVariants];  // M = 9..16
extern const CCKernelFn cc_table_lo_fp16[8][kCCVariants];
extern const CCKernelFn cc_table_hi_fp16[8][kCCVariants];
extern const CCKernelFn cc_table_proj[8][kCCVariants];      // M = 1..8, bf16, kProj
extern const CCKernelFn cc_ring_lo_bf16[8][kCCVariants];    // ring form, M = 1..8
extern const CCKernelFn cc_ring_hi_bf16[8][kCCVariants];    // ring form, M = 9..16
extern const CCKernelFn cc_ring_lo_fp16[8][kCCVariants];
extern const CCKernelFn cc_ring_hi_fp16[8][kCCVariants];

}  // namespace kp
