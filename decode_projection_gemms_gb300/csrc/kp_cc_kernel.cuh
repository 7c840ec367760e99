// CUDA-core split-K weight-streaming GEMV for M <= 16 tokens.
//
// y[m, n] = round( sum_k x[m, k] * W[n, k] (+ residual[m, n]) ), fp32
// accumulation, bf16 or fp16 elements (template T): the skinny
// GEMM of the Kimi K3 support page, part 1 (vllm PR #50089 digest, CuteSkinnyGemm, section
// "关键源码片段"), whose design is prior art here: CUDA-core FMAs over 16-byte
// vector loads, warp-shuffle row reductions, M unrolled at compile time.
// Differences from that design: the K range is split over blockIdx.y (split-K)
// so small-N shapes still fill all SMs, x's K slice is staged once per CTA in
// shared memory as fp32, each warp owns `R` output rows, and the S partial
// sums of a row tile are combined deterministically by the last CTA to finish
// (ticket counter, sum in split order 0..S-1, plus the residual if any, one
// rounding to the element type).
//
// Grid: (row tiles, S). Block: `block` threads, warp w owns rows
// tile*rows_cta + w*R .. +R-1. Lane l reads the 16-byte chunks l, l+32, ... of
// the CTA's K slice for each of its rows; `U` chunks per row are in flight per
// lane.
#pragma once

#include "kp_internal.cuh"

namespace kp {

struct CCParams {
    GemmArgs a;
    int Ks;       // K slice length (multiple of 8)
    int S;        // number of K slices (gridDim.y)
    int rows_cta; // output rows per CTA
};

// Store one output: the residual (if any) joins the fp32 sum, then one rounding.
template <int T>
__device__ __forceinline__ void cc_store(const GemmArgs &a, int m, int n, float v) {
    if (a.res) v += elem_widen(a.res[m * a.ldr + n], T);
    reinterpret_cast<uint16_t *>(a.y)[m * a.ldy + n] = elem_round<T>(v);
}

template <int M, int R, int U, int T>
__global__ void __launch_bounds__(256, 2) cc_gemv_kernel(const CCParams p) {
    extern __shared__ float4 cc_smem[];
    float *xs = reinterpret_cast<float *>(cc_smem);  // [M][Ks] fp32

    const GemmArgs &a = p.a;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int tile = blockIdx.x;
    const int s = blockIdx.y;
    const int row0 = tile * p.rows_cta + warp * R;
    const int k0 = s * p.Ks;
    const int klen = min(p.Ks, a.K - k0);
    const int nchunk = klen >> 3;
    const uint64_t pol = policy_evict_first();

    // Rows past N read row N-1 (always valid) and are never stored.
    const __nv_bfloat16 *wrow[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int n = min(row0 + r, a.N - 1);
        wrow[r] = a.W + static_cast<int64_t>(n) * a.K + k0;
    }

    // Two batches of U chunks per row in flight per warp (double buffering):
    // the next batch is requested before the current one is consumed.
    uint4 wa[R][U], wb[R][U];
    auto load_batch = [&](uint4 (&w)[R][U], int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + 32 * u;
#pragma unroll
            for (int r = 0; r < R; ++r)
                w[r][u] = (c < nchunk) ? ldg_stream(wrow[r] + 8 * c, pol) : make_uint4(0, 0, 0, 0);
        }
    };

    float acc[R][M];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

    auto compute = [&](const uint4 (&w)[R][U], int c0) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + 32 * u;
            if (c < nchunk) {
                // two halves of 4 k-elements keep the converted weights in
                // 4*R registers
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float wf[R][4];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t w0 = h ? w[r][u].z : w[r][u].x;
                        const uint32_t w1 = h ? w[r][u].w : w[r][u].y;
                        wf[r][0] = elem_lo<T>(w0); wf[r][1] = elem_hi<T>(w0);
                        wf[r][2] = elem_lo<T>(w1); wf[r][3] = elem_hi<T>(w1);
                    }
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        const float4 xv =
                            reinterpret_cast<const float4 *>(xs + m * p.Ks + 8 * c)[h];
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            float t = acc[r][m];
                            t = fmaf(wf[r][0], xv.x, t);
                            t = fmaf(wf[r][1], xv.y, t);
                            t = fmaf(wf[r][2], xv.z, t);
                            t = fmaf(wf[r][3], xv.w, t);
                            acc[r][m] = t;
                        }
                    }
                }
            }
        }
    };

    // Weights never depend on the previous kernel: start streaming them
    // before waiting for it.
    load_batch(wa, lane);
    pdl_wait();
    pdl_trigger();

    // Stage x[0:M, k0:k0+klen] as fp32.
    for (int i = threadIdx.x; i < M * nchunk; i += blockDim.x) {
        const int m = i / nchunk;
        const int c = i - m * nchunk;
        const uint4 v = *reinterpret_cast<const uint4 *>(a.x + m * a.ldx + k0 + 8 * c);
        float4 *d = reinterpret_cast<float4 *>(xs + m * p.Ks + 8 * c);
        d[0] = make_float4(elem_lo<T>(v.x), elem_hi<T>(v.x), elem_lo<T>(v.y), elem_hi<T>(v.y));
        d[1] = make_float4(elem_lo<T>(v.z), elem_hi<T>(v.z), elem_lo<T>(v.w), elem_hi<T>(v.w));
    }
    __syncthreads();

    for (int c0 = lane; c0 < nchunk; c0 += 64 * U) {
        const int c1 = c0 + 32 * U;
        const int c2 = c1 + 32 * U;
        if (c1 < nchunk) load_batch(wb, c1);
        compute(wa, c0);
        if (c2 < nchunk) load_batch(wa, c2);
        if (c1 < nchunk) compute(wb, c1);
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

    if (p.S == 1) {
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

using CCKernelFn = void (*)(const CCParams);

// (R, U) variants instantiated for every M in 1..16.
constexpr int kCCVariants = 6;
constexpr int kCCR[kCCVariants] = {1, 2, 2, 4, 4, 8};
constexpr int kCCU[kCCVariants] = {4, 2, 4, 1, 2, 1};

}  // namespace kp

namespace kp {

// Kernel pointer for (M, variant, element type), or nullptr where the R*M
// accumulators would not fit in the 128 registers a thread gets at two CTAs
// per SM.
template <int M, int V, int T>
constexpr CCKernelFn cc_pick() {
    if constexpr (kCCR[V] * M <= 64 && (kCCR[V] < 8 || M <= 4))
        return cc_gemv_kernel<M, kCCR[V], kCCU[V], T>;
    else
        return nullptr;
}

#define KP_CC_ROW(M, T)                                                                    \
    {                                                                                      \
        cc_pick<M, 0, T>(), cc_pick<M, 1, T>(), cc_pick<M, 2, T>(), cc_pick<M, 3, T>(),   \
            cc_pick<M, 4, T>(), cc_pick<M, 5, T>()                                         \
    }

// [M - 1 within the half][variant], one table per half and element type
extern const CCKernelFn cc_table_lo_bf16[8][kCCVariants];  // M = 1..8
extern const CCKernelFn cc_table_hi_bf16[8][kCCVariants];  // M = 9..16
extern const CCKernelFn cc_table_lo_fp16[8][kCCVariants];
extern const CCKernelFn cc_table_hi_fp16[8][kCCVariants];

}  // namespace kp
