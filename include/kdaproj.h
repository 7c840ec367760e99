/*
 * kdaproj.h -- C ABI of the GB300 (sm_103a) KDA decode-projection library.
 *
 * The operation is the low-M "skinny GEMM"
 *
 *     y[m, n] = bf16( sum_k x[m, k] * W[n, k] ),   fp32 accumulation,
 *
 * i.e. C[M,N] = A[M,K] * B[N,K]^T with bf16 inputs, fp32 accumulation and bf16
 * output (Kimi K3 support page, part 1: vllm PR #50089 digest, section
 * "关键源码片段", CuteSkinnyGemm docstring), applied to the Kimi-K3 KDA input
 * projections of one TP8 rank ("[Kimi-K3] Overlap low-M TP8 KDA projections",
 * vllm PR 54697, section "关键源码片段", run_kda_projection_overlap):
 *
 *   main stream:  out_qkvg = x * W_packed[0 : N_qkvg]^T            (Q/K/V/G)
 *   aux stream:   out_fab  = x * W_packed[N_qkvg : N_qkvg+N_fab]^T (F_A/beta)
 *                 out_fb   = out_fab[:, 0:128] * W_fb^T            (F_B, chained
 *                            with programmatic dependent launch)
 *   fork/join:    events[0] recorded on main, waited on by aux; events[1]
 *                 recorded on aux, waited on by main.
 *
 * Layout and ownership (every call):
 *   - All matrices are bf16, row-major, densely packed (row stride = number of
 *     columns) except F_B's input, which is the F_A half of out_fab read in
 *     place with row stride N_fab.
 *   - Every device pointer must be 16-byte aligned. K must be a multiple of 8
 *     (16-byte rows). Pointers are device (or managed) memory owned by the
 *     caller; the library never frees or retains them after the call returns.
 *   - Streams and events are the caller's CUDA handles (cudaStream_t /
 *     cudaEvent_t); the library only enqueues work on them. NULL stream = the
 *     legacy default stream.
 *   - Calls are asynchronous: they return once the work is enqueued. Outputs
 *     are valid when the stream's work completes.
 *
 * Errors: every function returns an int; 0 (KP_OK) on success, a negative
 * kp_status otherwise, and kp_last_error() (thread-local) then describes the
 * failure, including the CUDA runtime's message for KP_ECUDA. Argument errors
 * are detected before anything is enqueued. Nothing throws across this ABI.
 * Kernel-side waits are bounded: a wait that runs out (after about 1 s, e.g.
 * on a GPU that is pre-empted or time-sliced away) records a code in the
 * device's error word and the kernel finishes instead of hanging. The outputs
 * of that call are then undefined. The word lives in mapped host memory, so
 * skinny_gemm, skinny_gemm_ex and kda_proj_run check it on entry without any
 * CUDA call and return KP_EDEVICE while it is set; kp_device_error() reads
 * and clears it.
 *
 * Determinism: the configuration used for a call depends only on (M, N, K)
 * and the loaded table (never on stream state), and every split-K reduction
 * sums its partials in a fixed order, so repeated calls, the sequential and
 * the overlapped projection, and graph replays give bit-identical outputs.
 */
#ifndef KDAPROJ_H
#define KDAPROJ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same tags as cudaStream_t / cudaEvent_t, so those convert implicitly. */
typedef struct CUstream_st *kp_stream_t;
typedef struct CUevent_st *kp_event_t;

#define KDAPROJ_VERSION 1

#if defined(__GNUC__)
#define KP_API __attribute__((visibility("default")))
#else
#define KP_API
#endif

enum kp_status {
    KP_OK = 0,
    KP_EINVAL = -1,   /* NULL pointer or out-of-range argument */
    KP_EALIGN = -2,   /* a pointer is not 16-byte aligned */
    KP_ESHAPE = -3,   /* unsupported shape (K % 8 != 0, N < 1, N_fab < 128 ...) */
    KP_ENOPLAN = -4,  /* NULL plan handle */
    KP_ECUDA = -5,    /* a CUDA runtime call failed; see kp_last_error() */
    KP_ETOOBIG = -6,  /* M above the plan's max_M (its workspace would overflow) */
    KP_ENODEV = -7,   /* current device is not an sm_103 GPU */
    KP_ECONFIG = -8,  /* explicit kp_cfg invalid for this shape */
    KP_EIO = -9,      /* autotune table file unreadable or malformed */
    KP_EDEVICE = -10  /* an earlier kernel wait on this device ran out (its
                         outputs are undefined); nothing was enqueued.
                         kp_device_error() returns the code and clears it */
};

/* Kernel families. */
enum kp_kind {
    KP_KIND_AUTO = 0,  /* look the shape up in the table (or the built-in rule) */
    KP_KIND_CC = 1,    /* CUDA-core split-K weight-streaming GEMV, M <= 16 */
    KP_KIND_TC05 = 2,  /* TMA-fed tcgen05/TMEM cluster split-K tile kernel */
    KP_KIND_SMALLK = 3 /* CUDA-core small-K kernel (K <= 256), the F_B shape */
};

/* Element type of x, W, y and the residual in skinny_gemm_ex. */
enum kp_dtype {
    KP_BF16 = 0,
    KP_FP16 = 1
};

enum kp_flags {
    KP_FLAG_PDL = 1,    /* launch with programmatic stream serialisation: the
                           kernel may start (and stream its weights) while the
                           previous kernel on the stream finishes; it waits for
                           that kernel before touching x, y, the residual or
                           scratch. W (and the projection's W_fb) is read
                           BEFORE that wait, so W must not be written by the
                           kernel just before on the same stream (weights
                           never are; this library's kernels let their
                           dependents start before they store y, so feeding
                           one call's y as the next call's W needs a
                           configuration without this flag) */
    KP_FLAG_FUSE_FB = 2 /* F_A/beta branch of kda_proj_run only (TC05 kind,
                           M <= 256): the F_A/beta launch also computes F_B
                           from its bf16 F_A tile, so the F_B launch is skipped */
};

/* One kernel configuration. Fields a kind does not use are ignored. */
typedef struct kp_cfg {
    int32_t kind;     /* enum kp_kind */
    int32_t split_k;  /* CC: number of K slices S >= 1 (S > 1 uses scratch);
                         TC05: CTAs per thread-block cluster sharing one
                         128-feature tile, each streaming 1/split_k of K
                         (1, 2, 4, 8, 16; with split_k > 1 each CTA's fp32
                         partial tile goes to scratch and the cluster sums
                         them in rank order) */
    int32_t block;    /* CC, SMALLK: threads per CTA (multiple of 32; CC <= 512,
                         SMALLK <= 256) */
    int32_t rows;     /* CC: output rows per warp (1, 2, 4, 8);
                         SMALLK: output rows per CTA (1..64);
                         TC05: feature rows per CTA, 256 (two 128-row MMAs
                         sharing each x tile) or anything else for 128 */
    int32_t k_unroll; /* CC: 16-byte W chunks per row per lane in one batch
                         (1, 2, 4);
                         TC05: 64-wide K blocks per pipeline stage (1, 2, 4) */
    int32_t producers;/* TC05: warps issuing TMA copies per CTA (1..5; 0 = 1) */
    int32_t stages;   /* CC: 0 = two batches in flight per lane in registers;
                         4 = each warp streams its W through a 4-slot ring in
                         shared memory (asynchronous 16-byte copies, three
                         batches in flight; the x slice plus block/32 * 4 *
                         rows * k_unroll * 512 bytes of ring must fit in
                         220 KB). Same sums, bit for bit.
                         TC05: shared-memory pipeline stages (0 = as many as fit) */
    int32_t flags;    /* enum kp_flags */
} kp_cfg;

/* Opaque plan for the full KDA projection. */
typedef struct kda_plan kda_plan;

/* ---------------------------------------------------------------------------
 * skinny_gemm: y[M, N] = bf16(x[M, K] * W[N, K]^T), fp32 accumulation.
 *   x   device, [M, K] bf16, row-major
 *   W   device, [N, K] bf16, row-major (K contiguous)
 *   y   device, [M, N] bf16, row-major; written, never read
 *   cfg NULL or kind == KP_KIND_AUTO: the autotune table picks the kernel;
 *       otherwise the given configuration is validated and used.
 * M == 0 is a no-op. The tcgen05 kernel takes any M in one launch: token
 * tiles of up to 256 along the grid's second axis, which all read a weight
 * tile while it is in L2 (the CUDA-core kernel takes M <= 16).
 * Scratch: split-K partial sums and tile counters live in a per-device
 * workspace owned by the library. It grows on demand, so the first call of a
 * larger shape may allocate (cudaMalloc, with a device synchronisation); do
 * one call per shape before stream capture. A workspace that growth replaces
 * stays allocated until the process exits, so work captured into a CUDA graph
 * before a later growth keeps valid scratch; each growth at least doubles the
 * workspace, so the kept buffers add up to less than the current one. Calls that use this workspace
 * must not run concurrently on one device (use one stream, or kda_proj_*
 * whose plans own their scratch).
 * Returns KP_OK, KP_EINVAL, KP_EALIGN, KP_ESHAPE, KP_ECONFIG, KP_ENODEV,
 * KP_ECUDA. */
KP_API int skinny_gemm(const void *x, const void *W, void *y, int M, int N, int K,
                const kp_cfg *cfg, kp_stream_t stream);

/* ---------------------------------------------------------------------------
 * skinny_gemm_ex: y[M, N] = round(x[M, K] * W[N, K]^T + residual[M, N]), fp32
 * accumulation, the residual (if any) widened to fp32 and added to the sum
 * once after the K loop, then one rounding (to nearest even) to the element
 * type. This is the skinny GEMM of the Kimi K3 support page, part 1 (vllm PR
 * #50089 digest, CuteSkinnyGemm: C = A * B^T + residual with bf16 or fp16
 * inputs and fp32 accumulation, the residual optional).
 *   x, W, y   as for skinny_gemm, all of type dtype
 *   residual  NULL, or device [M, N] row-major of type dtype, 2-byte aligned;
 *             it may be y itself (each element is read before it is written,
 *             by the same thread) but must not otherwise overlap y
 *   dtype     KP_BF16 or KP_FP16
 * Kernels, configurations, table lookup and scratch as for skinny_gemm (the
 * table is keyed by shape only). skinny_gemm(x, W, y, ...) is
 * skinny_gemm_ex(x, W, NULL, y, ..., KP_BF16, ...).
 * Returns KP_OK, KP_EINVAL (also for an unknown dtype), KP_EALIGN, KP_ESHAPE,
 * KP_ECONFIG, KP_ENODEV, KP_ECUDA, KP_EDEVICE. */
KP_API int skinny_gemm_ex(const void *x, const void *W, const void *residual, void *y, int M,
                          int N, int K, int dtype, const kp_cfg *cfg, kp_stream_t stream);

/* Host-only: the configuration skinny_gemm would use for (M, N, K) on a
 * device with `num_sms` SMs (0 = query the current device). Lookup rounds M
 * up to the next measured bucket of an (N, K) entry; shapes missing from the
 * table use the built-in rule. Returns KP_OK or KP_EINVAL. */
KP_API int kp_select_config(int M, int N, int K, int num_sms, kp_cfg *out);

/* Host-only: load an autotune table (text, see the package's tune/ folder),
 * replacing the loaded one. Plans made earlier keep their configurations.
 * Returns KP_OK, KP_EINVAL or KP_EIO. kp_table_clear() drops it. */
KP_API int kp_table_load(const char *path);
KP_API int kp_table_clear(void);
KP_API int kp_table_size(void);

/* ---------------------------------------------------------------------------
 * skinny_gemm_noalloc: the same product as skinny_gemm, computed by the
 * CUDA-core split-K kernel, with its scratch in a fixed device array that the
 * library itself carries, so the call never allocates. (The pages have no
 * counterpart: this entry point exists for callers of this library.)
 *
 * Meant for callers that cannot call cudaMalloc: processes whose device
 * memory is managed by a pooling allocator, and latency-critical paths that
 * cannot take cudaMalloc's device synchronisation. The caller still passes x, W and y (same layout as
 * skinny_gemm); the call calls no cudaMalloc, cudaFree or allocating library
 * routine.
 *   - Limits: M <= 16 (CUDA-core kernel). The kernel stages x's K slice in
 *     shared memory (M * ceil(K / split_k) * 2 bytes, at most 200 KiB), so a
 *     shape needs split_k >= ceil(M * K * 2 / 204800); its split-K partial
 *     sums (split_k * M * N floats when split_k > 1) must fit in
 *     KP_NOALLOC_SCRATCH_FLOATS and its row tiles (ceil(N / 32) with the
 *     default configuration) in KP_NOALLOC_TICKETS. With cfg NULL (or kind
 *     AUTO) the entry point sizes split_k for about two CTAs per SM, lowers
 *     it until the partial sums fit, then raises it again if x's slice does
 *     not fit in shared memory; a shape whose smallest such split_k needs
 *     more partial sums than the array holds (e.g. M = 16, K = 16384,
 *     N = 16384: split_k >= 3, 786432 floats) returns KP_ETOOBIG. An explicit
 *     cfg must be kind KP_KIND_CC.
 *   - Ordering: with cfg NULL the kernel launches without programmatic
 *     dependent launch, so x and W may both come from the kernel just before
 *     it on the stream. A cfg (kind AUTO or CC) supplies the flags, and with
 *     KP_FLAG_PDL W is read before that wait (see KP_FLAG_PDL).
 *   - Memory: every GPU that loads the library holds the array
 *     (2 MiB + 32 KiB) until the process exits.
 *   - First call per device: looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); it allocates and
 *     synchronises nothing. Later calls only launch the kernel.
 *   - Sharing: all calls on a device use the same array and it keeps the last
 *     call's partial sums; calls that overlap on the GPU (for example on
 *     different streams) race and give wrong results. Serialise
 *     them.
 * Returns KP_OK, KP_EINVAL, KP_EALIGN, KP_ESHAPE, KP_ECONFIG, KP_ETOOBIG,
 * KP_ENODEV, KP_ECUDA. */
#define KP_NOALLOC_SCRATCH_FLOATS (1 << 19)
#define KP_NOALLOC_TICKETS 8192
KP_API int skinny_gemm_noalloc(const void *x, const void *W, void *y, int M, int N, int K,
                               const kp_cfg *cfg, kp_stream_t stream);

/* ---------------------------------------------------------------------------
 * kda_proj_plan: prepare the projection for hidden size K, N_qkvg Q/K/V/G
 * rows, N_fab F_A/beta rows (the first 128 are F_A) and N_fb F_B rows, for
 * token counts 1..max_M. Picks a configuration per (branch, M) from the table,
 * and allocates (cudaMalloc, on the current device) the scratch of each branch
 * separately so the two streams never share it: enough for the chosen
 * configurations and, in every branch, for any tcgen05 configuration at up to
 * 256 tokens (its split-K partial tiles: split_k * Mpad * rows fp32 per 128- or
 * 256-row tile; about 71 MB for the Q/K/V/G branch of the pages' shapes at
 * max_M >= 256) plus one CUDA-core combine ticket per output row (a split-K
 * CUDA-core configuration fits when its S * M * N fp32 partials fit the space
 * above). The plan is immutable after
 * creation except through kda_proj_set_*; it is not thread-safe to modify a
 * plan while another thread runs it.
 * Returns KP_OK, KP_EINVAL, KP_ESHAPE, KP_ENODEV or KP_ECUDA. */
KP_API int kda_proj_plan(int K, int N_qkvg, int N_fab, int N_fb, int max_M, kda_plan **out);

/* Execution mode: -1 = per-M choice from the table (default);
 * 0 = sequential: Q/K/V/G, F_A/beta, F_B in order on main_stream;
 * 1 = overlapped: F_A/beta -> F_B on aux_stream concurrently with Q/K/V/G on
 *     main_stream (needs aux_stream and events, else runs as 0);
 * 2 = single launch: one tcgen05 launch over the packed weight computes
 *     Q/K/V/G and F_A/beta side by side, and the F_A tile's CTAs compute F_B
 *     (needs a tcgen05 Q/K/V/G configuration, N_qkvg % 128 == 0, M <= 256 and
 *     room for the F_B operands, else runs as 1). out_qkvg is bit-identical in
 *     all modes; out_fab and out_fb are bit-identical between modes 0 and 1,
 *     and equal to them in mode 2 when the F_A/beta configuration has the same
 *     split-K factor as the Q/K/V/G one (otherwise within the tolerance).
 * Returns KP_OK, KP_ENOPLAN, KP_EINVAL. */
KP_API int kda_proj_set_overlap(kda_plan *plan, int mode);

/* Branch ids for kda_proj_get_config / kda_proj_set_config. */
enum kp_branch { KP_BRANCH_QKVG = 0, KP_BRANCH_FAB = 1, KP_BRANCH_FB = 2 };

/* Read or replace the configuration a plan uses for (branch, M). A replaced
 * configuration must fit the scratch the plan allocated (else KP_ETOOBIG).
 * Returns KP_OK, KP_ENOPLAN, KP_EINVAL, KP_ECONFIG, KP_ETOOBIG. */
KP_API int kda_proj_get_config(const kda_plan *plan, int branch, int M, kp_cfg *out);
KP_API int kda_proj_set_config(kda_plan *plan, int branch, int M, const kp_cfg *cfg);

/* The mode the plan uses at this M (0, 1 or 2; see kda_proj_set_overlap). */
KP_API int kda_proj_overlap_at(const kda_plan *plan, int M);

/* ---------------------------------------------------------------------------
 * kda_proj_run: the full projection for M tokens (0 <= M <= max_M).
 *   x         device [M, K] bf16
 *   W_packed  device [N_qkvg + N_fab, K] bf16, Q/K/V/G rows first
 *   W_fb      device [N_fb, 128] bf16
 *   out_qkvg  device [M, N_qkvg] bf16 (written)
 *   out_fab   device [M, N_fab] bf16 (written; columns 0..127 are F_A, the
 *             rest beta; F_B reads F_A from here)
 *   out_fb    device [M, N_fb] bf16 (written)
 *   main_stream, aux_stream, events[2]: caller-owned. The plan's mode at this
 *   M (kda_proj_set_overlap) decides the schedule: overlapped (F_A/beta -> F_B
 *   on aux_stream, forked from and joined back into main_stream with
 *   events[0] / events[1]; needs aux_stream and both events), sequential (all
 *   in order on main_stream) or a single launch on main_stream. Either way, on
 *   return main_stream is ordered after all outputs. The sequence allocates nothing and never synchronises, so it can
 *   be captured into a CUDA graph (capture main_stream; aux joins through
 *   events[0]).
 * Returns KP_OK, KP_ENOPLAN, KP_EINVAL, KP_EALIGN, KP_ETOOBIG, KP_ECUDA. */
KP_API int kda_proj_run(const kda_plan *plan, const void *x, const void *W_packed, const void *W_fb,
                 void *out_qkvg, void *out_fab, void *out_fb, int M,
                 kp_stream_t main_stream, kp_stream_t aux_stream, kp_event_t events[2]);

/* Free the plan's scratch (synchronises the device first). NULL is a no-op. */
KP_API int kda_proj_destroy(kda_plan *plan);

/* ---------------------------------------------------------------------------
 * Diagnostics. */
KP_API const char *kp_last_error(void);           /* thread-local, never NULL */
KP_API int kp_version(void);                       /* KDAPROJ_VERSION */
/* Reads and clears (one atomic exchange, no CUDA call) the error word of the
 * current device: 0 if no kernel wait has run out, else the code of the
 * first one since the last read: 1 a stage of operands never landed, 2 a
 * pipeline stage was never freed, 3 an accumulator was never ready, 4 an
 * accumulator was never drained, 5 the self-test below. It does not wait for
 * the device: a kernel still running may set the word later, so read it once
 * the work in question has completed (e.g. after cudaStreamSynchronize).
 * Returns KP_OK, KP_ENODEV or KP_ECUDA. */
KP_API int kp_device_error(int *code);
/* Self-test of the failure path: launches one CTA on `stream` that waits on a
 * barrier nothing completes, with the kernels' bounded wait cut to timeout_us
 * (1 .. 1000000). The wait gives up, records code 5 in the device error word
 * and the kernel exits; the context stays usable. Not part of the
 * projections. Returns KP_OK, KP_EINVAL, KP_ENODEV or KP_ECUDA. */
KP_API int kp_selftest_timeout(int timeout_us, kp_stream_t stream);
/* Hand-off check for downstream kernels: launches on `stream` (with
 * programmatic stream serialisation when pdl != 0) a kernel that executes
 * griddepcontrol.wait and then adds the 16-bit patterns of buf[0 .. n) into
 * *out (device, unsigned 64-bit, exact). This library's kernels let such
 * dependents launch as soon as their own resources are set up, so a consumer
 * of kda_proj_run's outputs starts its prologue during the projection's tail;
 * after the wait it sees the outputs complete. buf: device, 2-byte aligned.
 * Returns KP_OK, KP_EINVAL, KP_EALIGN, KP_ENODEV or KP_ECUDA. */
KP_API int kp_pdl_consumer_checksum(const void *buf, int64_t n, unsigned long long *out, int pdl,
                                    kp_stream_t stream);
/* Bytes of scratch a configuration needs for (M, N, K), for tests/tools. */
KP_API int kp_scratch_bytes(int M, int N, int K, const kp_cfg *cfg, int num_sms, size_t *bytes);

#ifdef __cplusplus
}
#endif

#endif /* KDAPROJ_H */
