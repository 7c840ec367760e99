// TMA-fed tcgen05/TMEM cluster split-K kernel for y = round(x * W^T (+ residual)),
// bf16 or fp16 elements, any M: up to 256 tokens per CTA (the MMA's N), more
// tokens as further token tiles along the grid's y axis of the same launch.
//
// The contraction is the skinny GEMM of the Kimi K3 support page, part 1
// (vllm PR #50089 digest, CuteSkinnyGemm docstring: C = A * B^T, bf16 in,
// fp32 accumulate). The tile pipeline follows the Blackwell pattern of the
// fused GEMM + reduce-scatter page (vllm PR #52079 digest, section "实现拆解"
// item 1: TMA loads of A and B, tcgen05 BF16 MMA, mbarrier expect-tx stages),
// taken as prior art and re-designed for decode, where
// the whole cost is streaming W once from HBM:
//
//  * swap-AB: the MMA's M = 128 rows are output features (rows of W), its N
//    is the token count padded to 16 (UMMA N = 16..256), so one instruction
//    serves every token of a 128-feature tile;
//  * split-K over a thread-block cluster: the C CTAs of a cluster share one
//    feature tile and each streams 1/C of its K range. Each writes its fp32
//    partial tile from TMEM to a scratch area (L2-resident); after a cluster
//    barrier, CTA r sums rows [r*128/C, (r+1)*128/C) of all C partials in rank
//    order 0..C-1 and rounds once to bf16. Deterministic, no counters. The
//    launches that fuse F_B keep the partial tiles in shared memory and pull
//    them over distributed shared memory (then a second barrier keeps them
//    alive for their readers): there the fused cluster's tail sets the
//    launch's end, and the other CTAs leaving earlier (L2 path) let the next
//    launch's weight stream contend with it (measured slower);
//  * few, large TMA operations: on this part a TMA/bulk copy stream is
//    limited by operations per issuing warp rather than by DRAM locality, so
//    each 64-wide K block of W is one 128-row x 128-byte box (16 KB) and the
//    x operand of a whole stage (nkb K blocks) is one 3-D box; stages are kept
//    small enough for two CTAs per SM, whose producers stream concurrently;
//  * cta_group::1; every CTA loads its own operand tiles.
//
// Warp roles (192 threads): warp 1 = TMEM allocator + MMA issuer (one lane),
// warps 2..5 = epilogue (TMEM lane quarter = warp % 4). TMA copies are issued
// by lane 0 of P "producer" warps (warp 0, then warps 2, 3, 4, 5): producer
// p issues the W boxes of K blocks j with j % P == p of every stage, producer
// 0 also the x box; each arrives once per stage on the stage's barrier. The
// epilogue warps produce during the main loop and drain the accumulator after
// it. All 192 threads take part in the cluster reduction.
//
// Shared memory per stage: W [nkb][128 rows][128 B] then x [nkb][Mpad rows]
// [128 B], written by TMA with the 128-byte swizzle, i.e. the K-major
// SWIZZLE_128B canonical layout (8-row groups 1024 bytes apart). For K block j
// of a stage the MMA's A descriptor starts at W + j*16 KB, the B descriptor at
// x + j*Mpad*128.
// TMEM: one fp32 accumulator of Mpad columns, lane = feature row.
#include <cstring>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include "kp_internal.cuh"

namespace kp {

namespace {

constexpr int kThreads = 192;
constexpr int kTileN = 128;            // features per tile (UMMA M)
constexpr int kBlockK = 64;            // K elements per block (128 bytes)
constexpr uint32_t kWBlockBytes = kTileN * kBlockK * 2;  // 16 KB per K block
constexpr int kMaxSmem = 227 * 1024;
constexpr int kBarBytes = 512;
constexpr int kMaxFbBufs = 8;          // W_fb tile buffers (one per F_B tile of a CTA)

struct Tc05Params {
    __nv_bfloat16 *y;
    int64_t ldy;
    // Rows n >= n_split go to y2[m * ldy2 + (n - n_split)] (one launch over a
    // packed weight writing two outputs); n_split >= N: y only. Multiple of 128.
    int n_split;
    __nv_bfloat16 *y2;
    int64_t ldy2;
    int *err;
    // Split-K partial tiles (C > 1): the CTA of (token tile y, feature tile t,
    // rank r) owns [Mpad][RT] fp32 at ws + ((y * n_tiles + t) * C + r) * Mpad * RT.
    float *ws;
    int dtype;                 // KP_BF16 / KP_FP16: operands, output and residual
    const uint16_t *res;       // optional residual [M, ldr], added before the rounding
    int64_t ldr;
    int M, N, Mpad;
    int KB;            // K blocks in K
    int C;             // CTAs per cluster = K splits per tile
    int nkb;           // K blocks per stage
    int x3d;           // 1: x of a full stage is one 3-D box (K % 64 == 0)
    int producers;     // warps issuing TMA copies (1..5)
    int stages;
    int n_tiles;       // feature tiles in the grid
    int tile_rot;      // cluster i of the launch order computes tile (i + tile_rot) % n_tiles
    // Fused F_B: the CTAs of tile `fb_tile` (whose 128 rows are F_A) also
    // compute yfb = bf16(bf16(F_A) * W_fb^T); -1 = no fusion.
    int fb_tile;
    int fb_tiles;      // 128-row tiles of W_fb
    int N_fb;
    __nv_bfloat16 *yfb;
    int64_t ldfb;
    uint32_t off_bfa;  // shared-memory offset of the F_A operand [2][Mpad][128 B]
    uint32_t off_wfb;  // shared-memory offset of the W_fb tile buffers, each [2][128][128 B]
    int fb_bufs;       // W_fb tile buffers: all of a CTA's F_B tiles, or 1 (reused)
    int fb_accs;       // TMEM accumulators the F_B tiles alternate between (1 or 2)
    uint32_t tmem_cols_fb;  // TMEM columns of the fused tile's CTAs
    uint32_t idesc;
    uint32_t tmem_cols;
    uint32_t stage_bytes;
    uint32_t w_stage_bytes;
    int vec4;          // 1: y and y2 take 8-byte stores of four features
};

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, stride byte
// offset `sbo` between 8-row groups, leading byte offset unused (1).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t sbo) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void store_bits(const Tc05Params &p, int m, int n, uint16_t b) {
    if (n < p.n_split)
        reinterpret_cast<uint16_t *>(p.y)[m * p.ldy + n] = b;
    else
        reinterpret_cast<uint16_t *>(p.y2)[m * p.ldy2 + (n - p.n_split)] = b;
}

// Output (m, n), n < N, of the general instantiation: the residual (if any)
// joins the fp32 sum, one rounding to the element type, store; returns the
// stored bits.
__device__ __forceinline__ uint16_t finish(const Tc05Params &p, int m, int n, float v) {
    if (p.res) v += elem_widen(p.res[m * p.ldr + n], p.dtype);
    const uint16_t b = elem_round(v, p.dtype);
    store_bits(p, m, n, b);
    return b;
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// Byte offset of element (token m, feature k) of the fused F_B's B operand:
// K-major, 128-byte swizzle, two 64-wide K blocks of Mpad rows x 128 bytes.
__device__ __forceinline__ uint32_t bfa_offset(int m, int k, int Mpad) {
    return static_cast<uint32_t>((k >> 6) * Mpad * 128 + m * 128 +
                                 ((((k & 63) >> 3) ^ (m & 7)) << 4) + (k & 7) * 2);
}

// Wait (bounded by time only) for a barrier phase; used to drain copies.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > 1000000000ull) break;
}

// kGeneral = false: bf16 operands and output, no residual (the projections);
// true: the element type and the residual come from the parameters.
// kTiled = false: one token tile (M <= 256); true: token tiles along the
// grid's y axis.
// kWide = false: a CTA owns 128 feature rows; true: 256, as two 128-row MMAs
// on the same x operand into two TMEM accumulators (x per weight byte halves).
// kFB: the launch fuses F_B into one cluster (bf16, one token tile); the other
// instantiations carry none of that code.
template <bool kGeneral, bool kTiled, bool kWide, bool kFB = false>
__global__ void __launch_bounds__(kThreads, 1)
    tc05_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                const __grid_constant__ CUtensorMap tmx3, const __grid_constant__ CUtensorMap tmfb,
                const Tc05Params p) {
    extern __shared__ uint8_t tc_smem_raw[];
    const uint32_t raw = smem_u32(tc_smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = tc_smem_raw + (base - raw);
    const int S = p.stages;

    uint64_t *full = reinterpret_cast<uint64_t *>(gbase + static_cast<size_t>(S) * p.stage_bytes);
    uint64_t *empty = full + S;
    uint64_t *accf = empty + S;
    uint64_t *fbw = accf + 1;                // fused F_B: W_fb tile landed, per buffer
    uint64_t *fbacc = fbw + kMaxFbBufs;      // fused F_B: accumulator ready, per accumulator
    uint64_t *fbempty = fbacc + 2;           // fused F_B: accumulator drained, per accumulator
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fbempty + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int C = p.C;
    const int rank = C > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    // The fused F_B tile (if any) is dispatched first: its cluster has the
    // longest epilogue.
    const int tile = (static_cast<int>(blockIdx.x) / C + p.tile_rot) % p.n_tiles;
    const bool fused = kFB && p.fb_tile >= 0 && tile == p.fb_tile;
    // Token tile of this CTA: tokens [m0, m0 + Mloc), along the grid's y axis.
    const int m0 = kTiled ? static_cast<int>(blockIdx.y) * p.Mpad : 0;
    const int Mloc = kTiled ? min(p.M - m0, p.Mpad) : p.M;
    const int kb0 = static_cast<int>((static_cast<long long>(p.KB) * rank) / C);
    const int kb1 = static_cast<int>((static_cast<long long>(p.KB) * (rank + 1)) / C);
    const int n_st = (kb1 - kb0 + p.nkb - 1) / p.nkb;  // stages of work for this CTA
    // fused F_B tiles of this CTA: rank, rank + C, ...
    const int my_fb = fused && rank < p.fb_tiles ? (p.fb_tiles - rank + C - 1) / C : 0;
    // With one F_B tile, its W_fb (two 16 KB boxes) goes into the stage buffer
    // whose last main-loop use ends first (stage n_st - S; a buffer the main
    // loop never uses if n_st < S), provided that buffer lies past the region
    // the epilogue writes (partial tile, F_A operand). Its load then starts
    // while the last stages are still in the tensor cores, instead of after
    // the whole main loop: the fused cluster's epilogue is the launch's
    // longest, and its tail no longer waits for these loads.
    int fb_early = -1;
    if (my_fb == 1 && p.stage_bytes >= 2 * kWBlockBytes) {
        const int b = n_st < S ? n_st : (n_st - S) % S;
        if (b < S && static_cast<uint32_t>(b) * p.stage_bytes >= p.off_wfb) fb_early = b;
    }
    // producer index of this warp's lane 0 (-1: not a producer)
    const int pidx = (warp == 0) ? 0 : (warp >= 2 && warp - 1 < p.producers) ? warp - 1 : -1;
    const int P = p.producers;
    const uint32_t xblk = static_cast<uint32_t>(p.Mpad) * kBlockK * 2;
    constexpr int RT = kWide ? 2 * kTileN : kTileN;               // feature rows per CTA
    constexpr uint32_t kWBlk = static_cast<uint32_t>(RT) * kBlockK * 2;  // W bytes per K block
    const int row0 = tile * RT;
    const int pre = n_st < S ? n_st : S;
    // W boxes of stage s of this CTA's range, producer pidx's share; producer
    // 0 also accounts for the stage's x bytes.
    auto issue_w = [&](int s, int stage, uint64_t pol_w) {
        const int k0 = kb0 + s * p.nkb;
        const int kbs = min(p.nkb, kb1 - k0);
        const uint32_t st = base + stage * p.stage_bytes;
        const uint32_t bar = smem_u32(full + stage);
        int mine = 0;
        for (int j = pidx; j < kbs; j += P) ++mine;
        uint32_t bytes = static_cast<uint32_t>(mine) * kWBlk;
        if (pidx == 0) bytes += static_cast<uint32_t>(kbs) * xblk;
        mbar_expect_tx(bar, bytes);   // every producer arrives once per stage
        for (int j = pidx; j < kbs; j += P)
            for (int h = 0; h < RT / kTileN; ++h)   // 128-row boxes
                tma_load_2d(st + j * kWBlk + h * kWBlockBytes, &tmw, bar, (k0 + j) * kBlockK,
                            row0 + h * kTileN, pol_w);
    };
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(full + s), static_cast<uint32_t>(p.producers));
            mbar_init(smem_u32(empty + s), 1);
        }
        mbar_init(smem_u32(accf), 1);
        for (int i = 0; i < kMaxFbBufs; ++i) mbar_init(smem_u32(fbw + i), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(fbacc + i), 1);
            mbar_init(smem_u32(fbempty + i), 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
        // the weight stream starts before the TMEM allocation and the block barrier
        for (int s = 0; s < pre; ++s) issue_w(s, s, policy_evict_first());
        tma_prefetch_desc(&tmx);
        if (p.x3d) tma_prefetch_desc(&tmx3);
        if (fused) {
            tma_prefetch_desc(&tmfb);
            // W_fb does not depend on the previous kernel: pull this CTA's
            // F_B weight tiles into L2 now, so their loads after the main
            // loop hit it.
            for (int i = 0; i < my_fb; ++i)
                for (int j = 0; j < 2; ++j)
                    tma_prefetch_l2_2d(&tmfb, j * kBlockK, (rank + i * C) * kTileN);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), fused ? p.tmem_cols_fb : p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Dependents may launch only once every CTA of this grid holds its TMEM:
    // a dependent CTA that took the columns first would wait for this grid
    // while this grid's allocation waited for it.
    pdl_trigger();

    if (pidx >= 0 && lane == 0) {
        // ---------------- TMA producers ----------------
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        // A full stage's x is one 3-D box; a short last stage uses one 2-D box
        // per K block (so nothing past this CTA's range is read).
        auto x_full = [&](int kbs) { return p.x3d && kbs == p.nkb; };
        auto issue_x = [&](int s, int stage) {
            const int k0 = kb0 + s * p.nkb;
            const int kbs = min(p.nkb, kb1 - k0);
            const uint32_t st = base + stage * p.stage_bytes + p.w_stage_bytes;
            const uint32_t bar = smem_u32(full + stage);
            if (x_full(kbs)) {
                tma_load_3d(st, &tmx3, bar, 0, m0, k0, pol_x);
            } else {
                for (int j = 0; j < kbs; ++j)
                    tma_load_2d(st + j * xblk, &tmx, bar, (k0 + j) * kBlockK, m0, pol_x);
            }
        };
        // Weights never depend on the previous kernel: the first stages' W
        // tiles go out before waiting for it (producer 0's right after the
        // barriers are initialised); x (producer 0) follows after the wait.
        if (pidx != 0)
            for (int s = 0; s < pre; ++s) issue_w(s, s, pol_w);
        if (pidx == 0) {
            pdl_wait();
            for (int s = 0; s < pre; ++s) issue_x(s, s);
        }
        for (int s = pre; s < n_st; ++s) {
            const int stage = s % S;
            mbar_wait_bounded(smem_u32(empty + stage), static_cast<uint32_t>(((s / S) - 1) & 1),
                              abort_flag, p.err, DEV_TIMEOUT_EMPTY);
            issue_w(s, stage, pol_w);
            if (pidx == 0) issue_x(s, stage);
        }
        if (*abort_flag) {
            // Something gave up: let our own copies land before exiting.
            const int first = n_st > S ? n_st - S : 0;
            for (int s = first; s < n_st; ++s)
                drain_wait(smem_u32(full + (s % S)), static_cast<uint32_t>((s / S) & 1));
        }
        if (pidx == 0 && fb_early >= 0) {
            // the early W_fb buffer: free once stage n_st - S's MMAs are done
            if (n_st >= S)
                mbar_wait_bounded(smem_u32(empty + fb_early), static_cast<uint32_t>(((n_st - S) / S) & 1),
                                  abort_flag, p.err, DEV_TIMEOUT_EMPTY);
            const uint32_t dst = base + static_cast<uint32_t>(fb_early) * p.stage_bytes;
            mbar_expect_tx(smem_u32(fbw), 2 * kWBlockBytes);
            for (int j = 0; j < 2; ++j)
                tma_load_2d(dst + j * kWBlockBytes, &tmfb, smem_u32(fbw), j * kBlockK, rank * kTileN,
                            policy_evict_last());
        } else if (pidx == 0 && my_fb > 0) {
            // The pipeline memory is free once every main-loop MMA has
            // completed: fetch this CTA's W_fb tiles (as many as have a
            // buffer) while the epilogue and the cluster reduction run.
            mbar_wait_bounded(smem_u32(accf), 0, abort_flag, p.err, DEV_TIMEOUT_ACC_FULL);
            const int nb = my_fb < p.fb_bufs ? my_fb : p.fb_bufs;
            for (int i = 0; i < nb; ++i) {
                const uint32_t dst = base + p.off_wfb + static_cast<uint32_t>(i) * 2 * kWBlockBytes;
                mbar_expect_tx(smem_u32(fbw + i), 2 * kWBlockBytes);
                for (int j = 0; j < 2; ++j)
                    tma_load_2d(dst + j * kWBlockBytes, &tmfb, smem_u32(fbw + i), j * kBlockK,
                                (rank + i * C) * kTileN, policy_evict_last());
            }
        }
    }
    if (warp == 0) {
        // lanes 1..31 of warp 0 have nothing to do until the end
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            const uint32_t xblk = static_cast<uint32_t>(p.Mpad) * kBlockK * 2;
            for (int s = 0; s < n_st; ++s) {
                const int stage = s % S;
                const int kbs = min(p.nkb, kb1 - (kb0 + s * p.nkb));
                mbar_wait_bounded(smem_u32(full + stage), static_cast<uint32_t>((s / S) & 1),
                                  abort_flag, p.err, DEV_TIMEOUT_FULL);
                tc_fence_after();
                const uint32_t st = base + stage * p.stage_bytes;
                for (int j = 0; j < kbs; ++j) {
                    const uint64_t ad = smem_desc(st + j * kWBlk, 1024);
                    const uint64_t bd = smem_desc(st + p.w_stage_bytes + j * xblk, 1024);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk)
                        // +32 bytes per 16-element K step inside the swizzle atom
                        umma_bf16(tmem_base, ad + 2 * kk, bd + 2 * kk, p.idesc,
                                  (s > 0 || j > 0 || kk > 0) ? 1u : 0u);
                    if constexpr (kWide) {
                        // rows 128..255 of the box (16 KB on), same x, next accumulator
                        const uint64_t ad1 = smem_desc(st + j * kWBlk + kWBlockBytes, 1024);
#pragma unroll
                        for (int kk = 0; kk < kBlockK / 16; ++kk)
                            umma_bf16(tmem_base + static_cast<uint32_t>(p.Mpad), ad1 + 2 * kk, bd + 2 * kk,
                                      p.idesc, (s > 0 || j > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                umma_commit(smem_u32(empty + stage));
            }
            umma_commit(smem_u32(accf));
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;          // TMEM lane quarter this warp may read
        const int row = q * 32 + lane;   // feature row within a 128-row half of the tile
        __syncwarp();   // lane 0 may have been producing
        pdl_wait();
        if constexpr (kGeneral) {
            if (p.res) {
                // Pull the residual this CTA adds at the end (its rows of the
                // tile, every token) into L2 while the main loop runs.
                const int rows = C == 1 ? RT : RT / C;
                const int nr0 = tile * RT + (C == 1 ? 0 : rank * rows);
                const int segs = (rows + 31) / 32;   // 64-byte pieces per token
                for (int i = threadIdx.x - 64; i < Mloc * segs; i += kThreads - 64) {
                    const int m = i / segs;
                    const int n = nr0 + (i - m * segs) * 32;
                    if (n < p.N)
                        asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(p.res + (m0 + m) * p.ldr + n));
                }
            }
        }
        mbar_wait_bounded(smem_u32(accf), 0, abort_flag, p.err, DEV_TIMEOUT_ACC_FULL);
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        // This CTA's partial tile [Mpad][RT] fp32 (a warp writes 32 consecutive
        // rows, 128 bytes, per token): in the scratch area for the plain
        // kernels, in the (by now free) stage memory for the fused-F_B one.
        float *const red = !kFB ? p.ws + ((static_cast<size_t>(blockIdx.y) * p.n_tiles + tile) * C + rank) *
                                             static_cast<size_t>(p.Mpad) * RT
                                : reinterpret_cast<float *>(gbase);
        // half h of the tile: rows h*128 .. h*128+127, accumulator columns h*Mpad ..
        for (int h = 0; h < (kWide ? 2 : 1); ++h) {
            const int rt = h * kTileN + row;   // row within the tile
            const int n = tile * RT + rt;
            auto take = [&](int m, float f) {
                if (C == 1) {
                    uint16_t b;
                    if constexpr (kGeneral) {
                        b = n < p.N ? finish(p, m0 + m, n, f) : 0;
                    } else {
                        b = bf16_bits_rn(f);
                        if (n < p.N) store_bits(p, m0 + m, n, b);
                    }
                    if (fused && h == 0)   // F_A = the fused tile's first 128 rows
                        *reinterpret_cast<uint16_t *>(gbase + p.off_bfa + bfa_offset(m, row, p.Mpad)) = b;
                } else {
                    red[m * RT + rt] = f;
                }
            };
            const uint32_t tcol = taddr + static_cast<uint32_t>(h * p.Mpad);
            for (int c0 = 0; c0 < p.Mpad; c0 += 16) {
                uint32_t va[16];
                tmem_ld16(tcol + c0, va);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (c0 + i < Mloc) take(c0 + i, __uint_as_float(va[i]));
            }
        }
        tc_fence_before();
    }

    if (C > 1) {
        // Every partial tile of the cluster is written (and, by the barrier's
        // release/acquire at cluster scope, visible to every peer) after this.
        __syncwarp();
        cluster_sync_all();
        const float *const parts = !kFB ? p.ws + (static_cast<size_t>(blockIdx.y) * p.n_tiles + tile) * C *
                                                     static_cast<size_t>(p.Mpad) * RT
                                        : nullptr;
        const size_t part_stride = static_cast<size_t>(p.Mpad) * RT;   // one rank's tile
        // This CTA reduces rows r0 .. r0 + rpc - 1 of the tile for every
        // token. A thread owns four of those rows (rr .. rr + 3) and walks
        // the tokens m = t / groups, + mstep, ...: the rows and the output
        // row pointer are fixed per thread, so a token costs C remote loads,
        // the rank-order sums and one store.
        const int rpc = RT / C;                 // rows reduced by this CTA (>= 8)
        const int lg_groups = 29 - __clz(rpc);  // log2(rpc / 4): float4 groups per token
        const int g = threadIdx.x & ((1 << lg_groups) - 1);
        const int mstep = kThreads >> lg_groups;   // groups (<= 64) divides 192
        const int rr = rank * rpc + 4 * g;
        const int nb = tile * RT + rr;
        // output row for features nb .. nb + 3 (one side of n_split, a multiple of 128)
        const bool lo = nb < p.n_split;
        uint16_t *const yrow = reinterpret_cast<uint16_t *>(lo ? p.y : p.y2) + (lo ? nb : nb - p.n_split);
        const int64_t ldo = lo ? p.ldy : p.ldy2;
        const bool whole = p.vec4 && nb + 3 < p.N;
        // Round the sum of rows rr .. rr + 3 for token m, store it, and
        // (fused tile) hand it to the F_B operand.
        auto emit = [&](int m, const float4 &acc) {
            uint32_t w0, w1;   // bf16 bits of rows rr, rr+1 and rr+2, rr+3
            if constexpr (kGeneral) {
                uint32_t b[4];
                const float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) b[e] = nb + e < p.N ? finish(p, m0 + m, nb + e, v[e]) : 0;
                w0 = b[0] | (b[1] << 16);
                w1 = b[2] | (b[3] << 16);
            } else {
                const __nv_bfloat162 h0 = __floats2bfloat162_rn(acc.x, acc.y);
                const __nv_bfloat162 h1 = __floats2bfloat162_rn(acc.z, acc.w);
                w0 = *reinterpret_cast<const uint32_t *>(&h0);
                w1 = *reinterpret_cast<const uint32_t *>(&h1);
                uint16_t *const dst = yrow + (m0 + m) * ldo;
                if (whole) {
                    *reinterpret_cast<uint2 *>(dst) = make_uint2(w0, w1);
                } else {
                    if (nb + 0 < p.N) dst[0] = static_cast<uint16_t>(w0);
                    if (nb + 1 < p.N) dst[1] = static_cast<uint16_t>(w0 >> 16);
                    if (nb + 2 < p.N) dst[2] = static_cast<uint16_t>(w1);
                    if (nb + 3 < p.N) dst[3] = static_cast<uint16_t>(w1 >> 16);
                }
            }
            if (fused && rr < kTileN) {
                // this rank's features rr..rr+3 of the F_B operand (8 bytes),
                // written into its own copy and into every CTA of the cluster
                // that computes F_B tiles (the F_B operand region lies past
                // the partial tiles, so no reader is disturbed)
                const uint2 pk = make_uint2(w0, w1);
                const uint32_t off = base + p.off_bfa + bfa_offset(m, rr, p.Mpad);
                *reinterpret_cast<uint2 *>(gbase + p.off_bfa + bfa_offset(m, rr, p.Mpad)) = pk;
                for (int c = 0; c < C && c < p.fb_tiles; ++c)
                    if (c != rank)
                        asm volatile("st.shared::cluster.v2.b32 [%0], {%1, %2};" ::"r"(
                                         mapa_shared(off, static_cast<uint32_t>(c))),
                                     "r"(pk.x), "r"(pk.y)
                                     : "memory");
            }
        };
        auto add4 = [](float4 &a, const float4 &b) {
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        };
        const int mfirst = threadIdx.x >> lg_groups;
        // T tokens per pass with up to CM peers each: T * CM remote loads
        // in flight together before their sums (two tokens measured best
        // up to clusters of 8; four were slower at C = 4).
        auto passes = [&](auto t_c, auto cm_c) {
            constexpr int T = decltype(t_c)::value;
            constexpr int CM = decltype(cm_c)::value;
            for (int m = mfirst; m < Mloc; m += T * mstep) {
                float4 part[T][CM];
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const int mt = m + t * mstep;
                    if (mt < Mloc) {
                        if constexpr (!kFB) {
                            // the peers' partial tiles, through L2
                            const float *src = parts + mt * RT + rr;
#pragma unroll
                            for (int c = 0; c < CM; ++c)
                                if (c < C)
                                    part[t][c] = __ldcg(reinterpret_cast<const float4 *>(src + c * part_stride));
                        } else {
                            // the peers' partial tiles, over distributed shared memory
                            const uint32_t off = base + static_cast<uint32_t>((mt * RT + rr) * 4);
#pragma unroll
                            for (int c = 0; c < CM; ++c)
                                if (c < C) part[t][c] = ld_dsmem_f4(mapa_shared(off, static_cast<uint32_t>(c)));
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const int mt = m + t * mstep;
                    if (mt < Mloc) {
                        float4 acc = part[t][0];
#pragma unroll
                        for (int c = 1; c < CM; ++c)
                            if (c < C) add4(acc, part[t][c]);
                        emit(mt, acc);
                    }
                }
            }
        };
        if (C <= 4)
            passes(std::integral_constant<int, 2>(), std::integral_constant<int, 4>());
        else if (C <= 8)
            passes(std::integral_constant<int, 2>(), std::integral_constant<int, 8>());
        else
            passes(std::integral_constant<int, 1>(), std::integral_constant<int, 16>());
        if constexpr (kFB) {
            // Written F_B operand slices reach the tensor cores' (async) proxy
            // of whichever CTA reads them after the barrier.
            if (fused) asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
            // Peers may still be reading this CTA's partial tile; after this
            // barrier every F_B operand slice has landed everywhere.
            cluster_sync_all();
        }
    } else if (fused) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        tc_fence_before();
        __syncthreads();
    }

    if (my_fb > 0) {
        // ---------------- fused F_B: out_fb = bf16(F_A) * W_fb^T ----------------
        // Tile i uses W_fb buffer i % B and TMEM accumulator i % A. Either
        // every tile has its own buffer (B >= my_fb, loaded above), or B = 1
        // and A = 1 and the buffer is refilled once the previous tile's MMAs
        // are done.
        const int B = p.fb_bufs;
        const int A = p.fb_accs;
        const uint32_t b_base = base + p.off_bfa;
        auto a_base = [&](int i) {
            if (fb_early >= 0) return base + static_cast<uint32_t>(fb_early) * p.stage_bytes;   // i == 0
            return base + p.off_wfb + static_cast<uint32_t>(i % B) * 2 * kWBlockBytes;
        };
        if (warp == 0 && lane == 0) {
            for (int i = B; i < my_fb; ++i) {   // only with B = A = 1
                mbar_wait_bounded(smem_u32(fbacc), static_cast<uint32_t>((i - 1) & 1), abort_flag,
                                  p.err, DEV_TIMEOUT_ACC_FULL);
                mbar_expect_tx(smem_u32(fbw), 2 * kWBlockBytes);
                for (int j = 0; j < 2; ++j)
                    tma_load_2d(a_base(i) + j * kWBlockBytes, &tmfb, smem_u32(fbw), j * kBlockK,
                                (rank + i * C) * kTileN, policy_evict_last());
            }
        } else if (warp == 1 && lane == 0) {
            tc_fence_after();
            for (int i = 0; i < my_fb; ++i) {
                const int a = i % A;
                if (i >= A)
                    mbar_wait_bounded(smem_u32(fbempty + a), static_cast<uint32_t>(((i - A) / A) & 1),
                                      abort_flag, p.err, DEV_TIMEOUT_ACC_EMPTY);
                mbar_wait_bounded(smem_u32(fbw + i % B), static_cast<uint32_t>((i / B) & 1), abort_flag,
                                  p.err, DEV_TIMEOUT_FULL);
                tc_fence_after();
                for (int j = 0; j < 2; ++j) {
                    const uint64_t ad = smem_desc(a_base(i) + j * kWBlockBytes, 1024);
                    const uint64_t bd = smem_desc(b_base + j * p.Mpad * 128, 1024);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk)
                        umma_bf16(tmem_base + static_cast<uint32_t>(a * p.Mpad), ad + 2 * kk, bd + 2 * kk,
                                  p.idesc, (j > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(smem_u32(fbacc + a));
            }
        } else if (warp >= 2) {
            const int q = warp & 3;
            const int row = q * 32 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            for (int i = 0; i < my_fb; ++i) {
                const int a = i % A;
                mbar_wait_bounded(smem_u32(fbacc + a), static_cast<uint32_t>((i / A) & 1), abort_flag,
                                  p.err, DEV_TIMEOUT_ACC_FULL);
                tc_fence_after();
                const int n = (rank + i * C) * kTileN + row;
                const uint32_t tcol = taddr + static_cast<uint32_t>(a * p.Mpad);
                for (int c0 = 0; c0 < p.Mpad; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tcol + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int m = c0 + e;
                        if (m < Mloc && n < p.N_fb)
                            p.yfb[m * p.ldfb + n] = __float2bfloat16_rn(__uint_as_float(v[e]));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(fbempty + a));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, fused ? p.tmem_cols_fb : p.tmem_cols);
}

// ---- host helpers -------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
// Per device: kernel attributes raised, and the SM's shared memory and the
// per-block reserve (read once, used by every launch's TMEM-safety padding).
struct DevAttrs {
    int sm_smem = 0;
    int reserved = 0;
};
std::map<int, DevAttrs> g_attr_devices;

cudaError_t get_encode(EncodeTiledFn *out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = g_encode;
    return cudaSuccess;
}

// Encoded tensor maps, cached. A map is a pure function of (address, shape,
// row stride, box, element type), all of which form the key, so a cached copy
// is always the map the encoder would return: an address that is freed and
// reused for another tensor of the same shape gets the same, correct map.
// Direct-mapped, 1024 slots; a colliding key replaces the slot.
struct MapKey {
    const void *ptr;
    int64_t ld;
    int rows, cols, box_rows, nkb, dtype, rank;
    bool operator==(const MapKey &o) const {
        return ptr == o.ptr && ld == o.ld && rows == o.rows && cols == o.cols &&
               box_rows == o.box_rows && nkb == o.nkb && dtype == o.dtype && rank == o.rank;
    }
};
struct MapSlot {
    bool valid = false;
    MapKey key;
    CUtensorMap map;
};
constexpr int kMapSlots = 1024;
std::mutex g_map_mu;
MapSlot g_maps[kMapSlots];

int map_slot(const MapKey &k) {
    uint64_t h = reinterpret_cast<uint64_t>(k.ptr) * 0x9E3779B97F4A7C15ull;
    for (int64_t v : {k.ld, static_cast<int64_t>(k.rows), static_cast<int64_t>(k.cols),
                      static_cast<int64_t>(k.box_rows) * 64 + k.nkb * 4 + k.dtype * 2 + k.rank})
        h = (h ^ static_cast<uint64_t>(v)) * 0x100000001B3ull;
    return static_cast<int>((h >> 32) % kMapSlots);
}

bool map_lookup(const MapKey &k, CUtensorMap *out) {
    const int i = map_slot(k);
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (!g_maps[i].valid || !(g_maps[i].key == k)) return false;
    memcpy(out, &g_maps[i].map, sizeof(CUtensorMap));
    return true;
}

void map_store(const MapKey &k, const CUtensorMap &m) {
    const int i = map_slot(k);
    std::lock_guard<std::mutex> lk(g_map_mu);
    g_maps[i].valid = true;
    g_maps[i].key = k;
    memcpy(&g_maps[i].map, &m, sizeof(CUtensorMap));
}

// 2-D bf16 tensor map: `rows` x `cols` (cols contiguous, row stride `ld`
// elements), box = box_rows x 64 columns, 128-byte swizzle, zero fill.
CUtensorMapDataType map_type(int dtype) {
    return dtype == KP_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

cudaError_t make_map(CUtensorMap *map, const void *ptr, int rows, int cols, int64_t ld,
                     int box_rows, int dtype = KP_BF16) {
    const MapKey key{ptr, ld, rows, cols, box_rows, 0, dtype, 2};
    if (map_lookup(key, map)) return cudaSuccess;
    EncodeTiledFn enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, map_type(dtype), 2, const_cast<void *>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    map_store(key, *map);
    return cudaSuccess;
}

// 3-D bf16 view of a [rows, cols] row-major matrix as (64, rows, cols / 64):
// element (i, r, b) is at r * ld + b * 64 + i. Box = 64 x box_rows x nkb, so
// one copy lands nkb consecutive [box_rows][64] blocks. Needs cols % 64 == 0.
cudaError_t make_map3(CUtensorMap *map, const void *ptr, int rows, int cols, int64_t ld,
                      int box_rows, int nkb, int dtype) {
    const MapKey key{ptr, ld, rows, cols, box_rows, nkb, dtype, 3};
    if (map_lookup(key, map)) return cudaSuccess;
    EncodeTiledFn enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kBlockK), static_cast<cuuint64_t>(rows),
                          static_cast<cuuint64_t>(cols / kBlockK)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(kBlockK) * 2};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kBlockK), static_cast<cuuint32_t>(box_rows),
                         static_cast<cuuint32_t>(nkb)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, map_type(dtype), 3, const_cast<void *>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    map_store(key, *map);
    return cudaSuccess;
}

// Tokens per CTA (the MMA's N): M padded to 16, at most 256 (one token tile).
int mpad_of(int M) { return ((M < 256 ? M : 256) + 15) & ~15; }

// Feature rows per CTA: 256 when the configuration asks for it (rows = 256),
// else 128.
int rows_of(const kp_cfg &c) { return c.rows == 2 * kTileN ? 2 * kTileN : kTileN; }

uint32_t w_stage_bytes_of(int nkb, int rt) { return static_cast<uint32_t>(nkb) * rt * kBlockK * 2; }

uint32_t stage_bytes_of(int Mpad, int nkb, int rt) {
    return w_stage_bytes_of(nkb, rt) + static_cast<uint32_t>(nkb) * Mpad * kBlockK * 2;
}

size_t smem_of(int Mpad, int nkb, int stages, int rt) {
    return static_cast<size_t>(stages) * stage_bytes_of(Mpad, nkb, rt) + 1024 + kBarBytes;
}

uint32_t tmem_cols_of(int Mpad) {
    uint32_t c = 32;
    while (c < static_cast<uint32_t>(Mpad)) c <<= 1;
    return c;
}

int max_stages(int Mpad, int nkb, int rt) {
    int s = static_cast<int>((kMaxSmem - 1024 - kBarBytes) / stage_bytes_of(Mpad, nkb, rt));
    return s > 16 ? 16 : s;
}

int cluster_of(const kp_cfg &c) { return c.split_k < 1 ? 1 : c.split_k; }
int producers_of(const kp_cfg &c) { return c.producers < 1 ? 1 : c.producers; }
int nkb_of(const kp_cfg &c) { return c.k_unroll < 1 ? 1 : c.k_unroll; }

}  // namespace

int tc05_max_stages(int M) { return max_stages(mpad_of(M), 1, kTileN); }

kp_cfg tc05_default(int M, int N, int K, int num_sms) {
    kp_cfg c = {};
    c.kind = KP_KIND_TC05;
    c.flags = KP_FLAG_PDL;
    const int T = (N + kTileN - 1) / kTileN;
    const int KB = (K + kBlockK - 1) / kBlockK;
    const int mt = (M + 255) / 256;   // token tiles
    int C = 1;
    while (C < 16 && T * mt * C * 2 <= num_sms && C * 2 <= KB) C *= 2;
    const int Mpad = mpad_of(M);
    int nkb = 4;
    while (nkb > 1 && max_stages(Mpad, nkb, kTileN) < 3) nkb /= 2;
    c.split_k = C;
    c.k_unroll = nkb;
    c.producers = nkb;
    c.stages = 0;
    if (mt > 1) {
        // Prefill (measured on N=4096, K=7168): while the 128-row grid fits
        // on the SMs, deep stages of two K blocks (M=1024: 877 TFLOP/s);
        // beyond that, 256-row CTAs that share each x tile between two
        // accumulators (M=4096: 1125 TFLOP/s; 128 rows, max stages: 781).
        c.split_k = 1;
        c.producers = 1;
        if (T * mt <= num_sms) {
            c.k_unroll = 2;
        } else {
            c.rows = 2 * kTileN;
            c.k_unroll = 1;
        }
    }
    return c;
}

bool tc05_supported(int M, int N, int K, const kp_cfg &c) {
    if (M < 1 || N < 1 || K < 8 || (K & 7)) return false;
    if ((M + 255) / 256 > 65535) return false;   // token tiles along the grid's y axis
    const int C = cluster_of(c);
    if (C != 1 && C != 2 && C != 4 && C != 8 && C != 16) return false;
    const int KB = (K + kBlockK - 1) / kBlockK;
    if (C > KB) return false;
    const int nkb = nkb_of(c);
    if (nkb != 1 && nkb != 2 && nkb != 4) return false;
    if (c.producers < 0 || c.producers > 5) return false;
    const int Mpad = mpad_of(M);
    const int rt = rows_of(c);
    const int ms = max_stages(Mpad, nkb, rt);
    const int st = c.stages ? c.stages : ms;
    if (st < 1 || st > ms) return false;
    return true;
}

// Split-K partial tiles: C > 1 keeps C fp32 tiles of Mpad x rows per feature
// tile and token tile.
Scratch tc05_scratch(int M, int N, int K, const kp_cfg &c, int) {
    (void)K;
    Scratch s;
    const int C = cluster_of(c);
    if (C == 1 || M < 1 || N < 1) return s;
    const int rt = rows_of(c);
    const size_t tiles = static_cast<size_t>((N + rt - 1) / rt);
    const size_t mt = static_cast<size_t>((M + 255) / 256);
    s.floats = mt * tiles * C * static_cast<size_t>(mpad_of(M)) * rt;
    return s;
}

namespace {
// Shared-memory layout of the fused F_B after the main loop (offsets from the
// 1024-aligned base): [partial tile Mpad x rt fp32][F_A operand 2 x Mpad x
// 128 B][nbuf W_fb tiles of 2 x 16 KB]. It must fit in the pipeline memory.
void fb_layout(int Mpad, int rt, uint32_t *off_bfa, uint32_t *off_wfb, uint32_t *end, int nbuf = 1) {
    auto al = [](uint32_t v) { return (v + 1023u) & ~1023u; };
    *off_bfa = al(static_cast<uint32_t>(Mpad) * rt * 4);
    *off_wfb = al(*off_bfa + static_cast<uint32_t>(Mpad) * 256);
    *end = *off_wfb + static_cast<uint32_t>(nbuf) * 2 * kWBlockBytes;
}
}  // namespace

bool tc05_fusable(int M, const kp_cfg &c) {
    if (M < 1 || M > 256) return false;
    const int Mpad = mpad_of(M);
    const int nkb = nkb_of(c);
    const int rt = rows_of(c);
    const int st = c.stages ? c.stages : max_stages(Mpad, nkb, rt);
    uint32_t ob, ow, end;
    fb_layout(Mpad, rt, &ob, &ow, &end);
    return end <= static_cast<size_t>(st) * stage_bytes_of(Mpad, nkb, rt);
}

int tc05_rows(const kp_cfg &c) { return rows_of(c); }

cudaError_t tc05_launch(const GemmArgs &a, const kp_cfg &c, int num_sms, cudaStream_t stream,
                        const FusedFB *fb, const SplitOut *split) {
    (void)num_sms;
    if (!tc05_supported(a.M, a.N, a.K, c)) return cudaErrorInvalidValue;
    if (fb && !tc05_fusable(a.M, c)) return cudaErrorInvalidValue;
    // the fused F_B and the split output serve the bf16 projection only
    if ((fb || split) && (a.dtype != KP_BF16 || a.res || a.M > 256)) return cudaErrorInvalidValue;
    if (a.dtype != KP_BF16 && a.dtype != KP_FP16) return cudaErrorInvalidValue;
    const int Mpad = mpad_of(a.M);
    const int nkb = nkb_of(c);
    const int rt = rows_of(c);
    const int stages = c.stages ? c.stages : max_stages(Mpad, nkb, rt);
    Tc05Params p;
    p.y = a.y;
    p.ldy = a.ldy;
    p.n_split = a.N;
    p.y2 = nullptr;
    p.ldy2 = 0;
    if (split) {
        if (split->n_split % rt) return cudaErrorInvalidValue;
        p.n_split = split->n_split;
        p.y2 = split->y2;
        p.ldy2 = split->ldy2;
    }
    p.err = a.err;
    p.ws = a.ws;
    // the plain kernels' split-K partial tiles need scratch (the fused-F_B one
    // keeps them in shared memory)
    if (!fb && cluster_of(c) > 1 && !p.ws) return cudaErrorInvalidValue;
    p.dtype = a.dtype;
    p.res = a.res;
    p.ldr = a.ldr;
    p.M = a.M;
    p.N = a.N;
    p.Mpad = Mpad;
    p.KB = (a.K + kBlockK - 1) / kBlockK;
    p.C = cluster_of(c);
    p.nkb = nkb;
    p.producers = producers_of(c);
    p.stages = stages;
    p.n_tiles = (a.N + rt - 1) / rt;
    p.tile_rot = 0;
    // kind::f16 instruction descriptor: D fp32 (bit 4), A and B formats at
    // bits 7 and 10 (1 = bf16, 0 = fp16), both K-major, N >> 3 at bit 17,
    // M >> 4 at bit 24.
    const uint32_t ab = a.dtype == KP_FP16 ? 0u : (1u << 7) | (1u << 10);
    p.idesc = (1u << 4) | ab | (static_cast<uint32_t>(Mpad >> 3) << 17) |
              (static_cast<uint32_t>(kTileN >> 4) << 24);
    p.tmem_cols = tmem_cols_of(rt / kTileN * Mpad);   // one accumulator per 128-row half
    p.stage_bytes = stage_bytes_of(Mpad, nkb, rt);
    p.w_stage_bytes = w_stage_bytes_of(nkb, rt);
    p.vec4 = (p.ldy % 4 == 0 && (reinterpret_cast<uintptr_t>(p.y) & 7) == 0 &&
              (!p.y2 || (p.ldy2 % 4 == 0 && (reinterpret_cast<uintptr_t>(p.y2) & 7) == 0)))
                 ? 1 : 0;
    p.fb_tile = -1;
    p.fb_tiles = 0;
    p.N_fb = 0;
    p.yfb = nullptr;
    p.ldfb = 0;
    p.off_bfa = p.off_wfb = 0;
    p.fb_bufs = 1;
    p.fb_accs = 1;
    p.tmem_cols_fb = p.tmem_cols;
    CUtensorMap mfb;
    memset(&mfb, 0, sizeof mfb);
    if (fb) {
        uint32_t end;
        fb_layout(Mpad, rt, &p.off_bfa, &p.off_wfb, &end);
        if (fb->row0 % rt) return cudaErrorInvalidValue;   // F_A rows start a tile
        // a buffer per F_B tile of a CTA when they fit (else one, refilled),
        // and two TMEM accumulators when a CTA has several tiles
        const int tiles = (fb->N + kTileN - 1) / kTileN;
        const int per_cta = (tiles + p.C - 1) / p.C;
        const size_t pipe = static_cast<size_t>(stages) * stage_bytes_of(Mpad, nkb, rt);
        uint32_t ob, ow, end_all;
        fb_layout(Mpad, rt, &ob, &ow, &end_all, per_cta);
        p.fb_bufs = (per_cta <= kMaxFbBufs && end_all <= pipe) ? per_cta : 1;
        p.fb_accs = (p.fb_bufs >= per_cta && per_cta > 1 && 2 * Mpad <= 256) ? 2 : 1;
        p.tmem_cols_fb = tmem_cols_of(p.fb_accs * Mpad);
        if (p.tmem_cols_fb < p.tmem_cols) p.tmem_cols_fb = p.tmem_cols;
        p.fb_tile = fb->row0 / rt;
        p.tile_rot = p.fb_tile;
        p.N_fb = fb->N;
        p.fb_tiles = (fb->N + kTileN - 1) / kTileN;
        p.yfb = fb->y;
        p.ldfb = fb->ld;
        cudaError_t e2 = make_map(&mfb, fb->W, fb->N, kTileN, kTileN, kTileN);
        if (e2 != cudaSuccess) return e2;
    }

    CUtensorMap mw, mx, mx3;
    cudaError_t e = make_map(&mw, a.W, a.N, a.K, a.K, kTileN, a.dtype);
    if (e != cudaSuccess) return e;
    e = make_map(&mx, a.x, a.M, a.K, a.ldx, Mpad, a.dtype);
    if (e != cudaSuccess) return e;
    p.x3d = 0;
    memset(&mx3, 0, sizeof mx3);
    if (a.K % kBlockK == 0 && nkb > 1 && make_map3(&mx3, a.x, a.M, a.K, a.ldx, Mpad, nkb, a.dtype) == cudaSuccess)
        p.x3d = 1;

    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    DevAttrs da;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_attr_devices.find(dev);
        if (it != g_attr_devices.end()) {
            da = it->second;
        } else {
            for (auto fn : {tc05_kernel<false, false, false>, tc05_kernel<true, false, false>,
                            tc05_kernel<false, true, false>, tc05_kernel<true, true, false>,
                            tc05_kernel<false, false, true>, tc05_kernel<true, false, true>,
                            tc05_kernel<false, true, true>, tc05_kernel<true, true, true>,
                            tc05_kernel<false, false, false, true>, tc05_kernel<false, false, true, true>}) {
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
                if (e == cudaSuccess)
                    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            }
            if (e != cudaSuccess) return e;
            if (cudaDeviceGetAttribute(&da.sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&da.reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess)
                return cudaErrorInvalidValue;
            g_attr_devices[dev] = da;
        }
    }

    const int T = (a.N + rt - 1) / rt;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(T * p.C, (a.M + Mpad - 1) / Mpad, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    // TMEM is 512 columns per SM and an allocation that does not fit waits;
    // CTAs of a cluster wait for each other, so the CTAs that can share an SM
    // must never need more than 512 columns together. Shared memory bounds
    // what shares an SM: each CTA takes at least cols/512 of the SM's shared
    // memory (with its per-block reserve), so any mix of such CTAs fits.
    size_t smem = smem_of(Mpad, nkb, stages, rt);
    {
        const uint32_t cols = p.tmem_cols_fb > p.tmem_cols ? p.tmem_cols_fb : p.tmem_cols;
        const long long need =
            (static_cast<long long>(da.sm_smem) * cols + 511) / 512 - da.reserved;
        if (need > static_cast<long long>(smem)) smem = static_cast<size_t>(need);
        if (smem > static_cast<size_t>(kMaxSmem)) return cudaErrorInvalidValue;
    }
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = p.C;
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
    const bool general = a.dtype != KP_BF16 || a.res != nullptr;
    const bool tiled = cfg.gridDim.y > 1;
    using Fn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, Tc05Params);
    static const Fn kernels[2][2][2] = {
        {{tc05_kernel<false, false, false>, tc05_kernel<false, false, true>},
         {tc05_kernel<false, true, false>, tc05_kernel<false, true, true>}},
        {{tc05_kernel<true, false, false>, tc05_kernel<true, false, true>},
         {tc05_kernel<true, true, false>, tc05_kernel<true, true, true>}}};
    // the fused F_B has its own instantiations (bf16, one token tile: checked above)
    const Fn fn = fb ? (rt == 2 * kTileN ? tc05_kernel<false, false, true, true> : tc05_kernel<false, false, false, true>)
                     : kernels[general][tiled][rt == 2 * kTileN];
    return cudaLaunchKernelEx(&cfg, fn, mw, mx, mx3, mfb, p);
}

}  // namespace kp
