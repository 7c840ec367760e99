// TMA-fed tcgen05/TMEM stream-K kernel for y = bf16(x * W^T), any M <= 256.
//
// The contraction is the skinny GEMM of "[Model] Kimi K3 support part 1"
// (CuteSkinnyGemm docstring: C = A * B^T, bf16 in, fp32 accumulate). The
// tile pipeline follows the Blackwell pattern that "Kimi-K3 GEMM-RS" (vllm PR
// 52079, section "实现拆解" item 1: TMA loads of A and B, tcgen05 BF16 MMA,
// mbarrier expect-tx stages) uses as prior art, re-designed for decode:
//
//  * swap-AB: the MMA's M = 128 rows come from W (output features), its N is
//    the token count padded to 16 (UMMA N in 16..256), so one instruction
//    serves every token of a 128-feature tile;
//  * stream-K: the (feature tile, 64-wide K block) pairs are split evenly over
//    a persistent grid (one CTA per SM by default), so every SM streams the
//    same number of weight bytes whatever N and K are;
//  * tiles split between CTAs are combined by the last CTA to finish (ticket
//    counter, partials summed in CTA order, one bf16 rounding): deterministic
//    and wait-free;
//  * cta_group::1 only, no clusters, no multicast.
//
// Warp roles (192 threads): warp 0 = TMA producer (one lane), warp 1 = TMEM
// allocator + MMA issuer (one lane), warps 2..5 = epilogue (TMEM lane quarter
// = warp % 4).
//
// Shared memory per stage: W tile 128 x 64 bf16 (16 KB) then x tile Mpad x 64
// bf16, both written by TMA with the 128-byte swizzle, which is the K-major
// SWIZZLE_128B canonical layout the MMA's shared-memory descriptors name.
// TMEM: two accumulators of Mpad fp32 columns (lane = feature row).
#include <mutex>
#include <set>
#include <utility>

#include "kp_internal.cuh"

namespace kp {

namespace {

constexpr int kThreads = 192;
constexpr int kTileN = 128;          // features per tile (UMMA M)
constexpr int kBlockK = 64;          // K elements per stage (128 bytes)
constexpr uint32_t kWBytes = kTileN * kBlockK * 2;  // 16 KB
constexpr int kMaxSmem = 227 * 1024;
constexpr int kBarBytes = 512;

struct Tc05Params {
    __nv_bfloat16 *y;
    int64_t ldy;
    float *ws;         // [G][2][Mpad][128] partial tiles
    int *counters;     // [T] tickets
    int *err;
    int M, N, Mpad, KB, T, G, stages;
    long long total;   // T * KB
    uint32_t idesc;
    uint32_t tmem_cols;
    uint32_t stage_bytes;
};

__device__ __forceinline__ long long range_begin(long long total, int G, int c) {
    return (total * c) / G;
}
// The CTA whose range [begin(c), begin(c+1)) holds flat K-block index i.
__device__ __forceinline__ int range_owner(long long i, long long total, int G) {
    return static_cast<int>(((i + 1) * G + total - 1) / total) - 1;
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), leading byte offset unused (1).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Wait (bounded by time only, ignoring the abort flag) for a barrier phase.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > 1000000000ull) break;
}

__global__ void __launch_bounds__(kThreads, 1)
    tc05_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx,
                const Tc05Params p) {
    extern __shared__ uint8_t tc_smem_raw[];
    const uint32_t raw = smem_u32(tc_smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = tc_smem_raw + (base - raw);
    const int S = p.stages;

    uint64_t *full = reinterpret_cast<uint64_t *>(gbase + static_cast<size_t>(S) * p.stage_bytes);
    uint64_t *empty = full + S;
    uint64_t *accf = empty + S;
    uint64_t *acce = accf + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acce + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long kb_begin = range_begin(p.total, p.G, cta);
    const long long kb_end = range_begin(p.total, p.G, cta + 1);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(full + s), 1);
            mbar_init(smem_u32(empty + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(accf + b), 1);
            mbar_init(smem_u32(acce + b), 4);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmw);
        tma_prefetch_desc(&tmx);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            const uint32_t xbytes = static_cast<uint32_t>(p.Mpad) * kBlockK * 2;
            const long long n_kb = kb_end - kb_begin;
            const int pre = static_cast<int>(n_kb < S ? n_kb : S);
            // Weight tiles of the first stages go out before the wait on the
            // previous kernel (weights never depend on it); x follows after.
            for (int j = 0; j < pre; ++j) {
                const long long g = kb_begin + j;
                const int t = static_cast<int>(g / p.KB);
                const int kb = static_cast<int>(g - static_cast<long long>(t) * p.KB);
                const uint32_t st = base + j * p.stage_bytes;
                mbar_expect_tx(smem_u32(full + j), kWBytes + xbytes);
                tma_load_2d(st, &tmw, smem_u32(full + j), kb * kBlockK, t * kTileN, pol_w);
            }
            pdl_wait();
            for (int j = 0; j < pre; ++j) {
                const long long g = kb_begin + j;
                const int t = static_cast<int>(g / p.KB);
                const int kb = static_cast<int>(g - static_cast<long long>(t) * p.KB);
                const uint32_t st = base + j * p.stage_bytes;
                tma_load_2d(st + kWBytes, &tmx, smem_u32(full + j), kb * kBlockK, 0, pol_x);
            }
            int stage = pre % S;
            uint32_t phase = (pre == S) ? 1u : 0u;
            for (long long g = kb_begin + pre; g < kb_end; ++g) {
                mbar_wait_bounded(smem_u32(empty + stage), phase ^ 1u, abort_flag, p.err,
                                  DEV_TIMEOUT_EMPTY);
                const int t = static_cast<int>(g / p.KB);
                const int kb = static_cast<int>(g - static_cast<long long>(t) * p.KB);
                const uint32_t st = base + stage * p.stage_bytes;
                mbar_expect_tx(smem_u32(full + stage), kWBytes + xbytes);
                tma_load_2d(st, &tmw, smem_u32(full + stage), kb * kBlockK, t * kTileN, pol_w);
                tma_load_2d(st + kWBytes, &tmx, smem_u32(full + stage), kb * kBlockK, 0, pol_x);
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (*abort_flag) {
                // Something gave up: let our own copies land before exiting.
                const long long issued = n_kb;
                const long long first = issued > S ? issued - S : 0;
                for (long long u = first; u < issued; ++u)
                    drain_wait(smem_u32(full + (u % S)), static_cast<uint32_t>((u / S) & 1));
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int stage = 0;
            uint32_t phase = 0;
            int j = 0;
            for (long long g0 = kb_begin; g0 < kb_end; ++j) {
                const int t = static_cast<int>(g0 / p.KB);
                const long long tile_end = static_cast<long long>(t + 1) * p.KB;
                const long long seg_end = kb_end < tile_end ? kb_end : tile_end;
                const int buf = j & 1;
                const uint32_t aph = static_cast<uint32_t>((j >> 1) & 1);
                mbar_wait_bounded(smem_u32(acce + buf), aph ^ 1u, abort_flag, p.err,
                                  DEV_TIMEOUT_ACC_EMPTY);
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(buf * p.Mpad);
                for (long long g = g0; g < seg_end; ++g) {
                    mbar_wait_bounded(smem_u32(full + stage), phase, abort_flag, p.err,
                                      DEV_TIMEOUT_FULL);
                    tc_fence_after();
                    const uint32_t st = base + stage * p.stage_bytes;
                    const uint64_t ad = smem_desc(st);
                    const uint64_t bd = smem_desc(st + kWBytes);
#pragma unroll
                    for (int kk = 0; kk < kBlockK / 16; ++kk) {
                        // +32 bytes per 16-element K step inside the swizzle atom
                        umma_bf16(d, ad + 2 * kk, bd + 2 * kk, p.idesc,
                                  (g > g0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(smem_u32(empty + stage));
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                umma_commit(smem_u32(accf + buf));
                g0 = seg_end;
            }
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;              // TMEM lane quarter this warp may read
        const int row = q * 32 + lane;       // feature row within the tile
        const int et = threadIdx.x - 64;     // 0..127
        pdl_wait();
        int j = 0;
        for (long long g0 = kb_begin; g0 < kb_end; ++j) {
            const int t = static_cast<int>(g0 / p.KB);
            const long long tile_begin = static_cast<long long>(t) * p.KB;
            const long long tile_end = tile_begin + p.KB;
            const long long seg_end = kb_end < tile_end ? kb_end : tile_end;
            const int buf = j & 1;
            const uint32_t aph = static_cast<uint32_t>((j >> 1) & 1);
            mbar_wait_bounded(smem_u32(accf + buf), aph, abort_flag, p.err, DEV_TIMEOUT_ACC_FULL);
            tc_fence_after();
            const bool whole = (g0 == tile_begin) && (seg_end == tile_end);
            const int n = t * kTileN + row;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(buf * p.Mpad);
            float *part = nullptr;
            if (!whole) {
                const int slot = (kb_begin >= tile_begin) ? 0 : 1;
                part = p.ws + static_cast<size_t>(cta * 2 + slot) * p.Mpad * kTileN;
            }
            for (int c0 = 0; c0 < p.Mpad; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(taddr + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int m = c0 + i;
                    if (m < p.M) {
                        const float f = __uint_as_float(v[i]);
                        if (whole) {
                            if (n < p.N) p.y[m * p.ldy + n] = __float2bfloat16_rn(f);
                        } else {
                            part[m * kTileN + row] = f;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(acce + buf));

            if (!whole) {
                __threadfence();
                named_bar_sync(1, 128);
                const int c_first = range_owner(tile_begin, p.total, p.G);
                const int c_last = range_owner(tile_end - 1, p.total, p.G);
                if (et == 0) {
                    const int prev = atomicAdd(p.counters + t, 1);
                    *last_flag = (prev == c_last - c_first) ? 1 : 0;
                }
                named_bar_sync(1, 128);
                if (*last_flag) {
                    __threadfence();
                    if (n < p.N) {
                        for (int m = 0; m < p.M; ++m) {
                            float acc = 0.f;
                            for (int c = c_first; c <= c_last; ++c) {
                                const int slot = (range_begin(p.total, p.G, c) >= tile_begin) ? 0 : 1;
                                acc += __ldcg(p.ws + (static_cast<size_t>(c * 2 + slot) * p.Mpad + m) *
                                                         kTileN + row);
                            }
                            p.y[m * p.ldy + n] = __float2bfloat16_rn(acc);
                        }
                    }
                    if (et == 0) p.counters[t] = 0;  // ready for the next launch
                }
                named_bar_sync(1, 128);
            }
            g0 = seg_end;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

// ---- host helpers -------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
std::set<int> g_attr_devices;

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

// 2-D bf16 tensor map: `rows` x `cols` (cols contiguous, row stride `ld`
// elements), box = box_rows x 64 columns, 128-byte swizzle, zero fill.
cudaError_t make_map(CUtensorMap *map, const void *ptr, int rows, int cols, int64_t ld,
                     int box_rows) {
    EncodeTiledFn enc;
    cudaError_t e = get_encode(&enc);
    if (e != cudaSuccess) return e;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int mpad_of(int M) { return (M + 15) & ~15; }

uint32_t stage_bytes_of(int Mpad) { return kWBytes + static_cast<uint32_t>(Mpad) * kBlockK * 2; }

size_t smem_of(int Mpad, int stages) {
    return static_cast<size_t>(stages) * stage_bytes_of(Mpad) + 1024 + kBarBytes;
}

uint32_t tmem_cols_of(int Mpad) {
    uint32_t need = 2u * static_cast<uint32_t>(Mpad);
    uint32_t c = 32;
    while (c < need) c <<= 1;
    return c;
}

int grid_of(int N, int K, const kp_cfg &c, int num_sms) {
    const long long T = (N + kTileN - 1) / kTileN;
    const long long KB = (K + kBlockK - 1) / kBlockK;
    long long G = c.ctas > 0 ? c.ctas : num_sms;
    if (G > T * KB) G = T * KB;
    if (G < 1) G = 1;
    return static_cast<int>(G);
}

}  // namespace

int tc05_max_stages(int M) {
    const int Mpad = mpad_of(M);
    int s = static_cast<int>((kMaxSmem - 1024 - kBarBytes) / stage_bytes_of(Mpad));
    return s > 16 ? 16 : s;
}

bool tc05_supported(int M, int N, int K, const kp_cfg &c) {
    if (M < 1 || M > 256 || N < 1 || K < 8 || (K & 7)) return false;
    if (c.ctas < 0 || c.stages < 0) return false;
    const int st = c.stages ? c.stages : tc05_max_stages(M);
    return st >= 2 && st <= tc05_max_stages(M);
}

Scratch tc05_scratch(int M, int N, int K, const kp_cfg &c, int num_sms) {
    Scratch s;
    const int G = grid_of(N, K, c, num_sms);
    s.floats = static_cast<size_t>(G) * 2 * mpad_of(M) * kTileN;
    s.counters = static_cast<size_t>((N + kTileN - 1) / kTileN);
    return s;
}

cudaError_t tc05_launch(const GemmArgs &a, const kp_cfg &c, int num_sms, cudaStream_t stream) {
    if (!tc05_supported(a.M, a.N, a.K, c)) return cudaErrorInvalidValue;
    const int Mpad = mpad_of(a.M);
    const int stages = c.stages ? c.stages : tc05_max_stages(a.M);
    Tc05Params p;
    p.y = a.y;
    p.ldy = a.ldy;
    p.ws = a.ws;
    p.counters = a.counters;
    p.err = a.err;
    p.M = a.M;
    p.N = a.N;
    p.Mpad = Mpad;
    p.KB = (a.K + kBlockK - 1) / kBlockK;
    p.T = (a.N + kTileN - 1) / kTileN;
    p.G = grid_of(a.N, a.K, c, num_sms);
    p.stages = stages;
    p.total = static_cast<long long>(p.T) * p.KB;
    // kind::f16 instruction descriptor: D fp32 (bit 4), A and B bf16 (bits
    // 7, 10), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
    p.idesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(Mpad >> 3) << 17) |
              (static_cast<uint32_t>(kTileN >> 4) << 24);
    p.tmem_cols = tmem_cols_of(Mpad);
    p.stage_bytes = stage_bytes_of(Mpad);

    CUtensorMap mw, mx;
    cudaError_t e = make_map(&mw, a.W, a.N, a.K, a.K, kTileN);
    if (e != cudaSuccess) return e;
    e = make_map(&mx, a.x, a.M, a.K, a.ldx, Mpad);
    if (e != cudaSuccess) return e;

    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_attr_devices.count(dev)) {
            e = cudaFuncSetAttribute(tc05_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kMaxSmem);
            if (e != cudaSuccess) return e;
            g_attr_devices.insert(dev);
        }
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.G, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_of(Mpad, stages);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (c.flags & KP_FLAG_PDL) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, tc05_kernel, mw, mx, p);
}

}  // namespace kp
