/*
 * rlk — deterministic, batch-invariant BF16 contractions on GB300 (sm_103a).
 *
 * A C ABI over hand-written tcgen05 / TMEM / TMA kernels.  Every entry point
 * takes plain pointers, sizes and leading dimensions; no framework types cross
 * this boundary.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Memory.  Every operand, output and workspace pointer is DEVICE memory on
 *    the current CUDA device, owned by the caller.  The library allocates no
 *    device memory and keeps no per-call state; its only device-resident state
 *    is a small error word (see rlk_get_device_error).
 *  - Layout.  Matrices are row-major with an explicit leading dimension ld (in
 *    elements, ld >= number of columns).  BF16 is passed as its 16-bit pattern.
 *  - Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Work is enqueued asynchronously; outputs are valid once
 *    the stream reaches that point.
 *  - Concurrency.  Entry points may be called from several host threads at once,
 *    each call with its own stream and workspace: host-side caches are guarded,
 *    no kernel waits on another launch's blocks, and the results are the bits of
 *    serial calls.  The device error word is shared by all calls of a process.
 *  - Errors.  Arguments are validated on the host before anything is launched;
 *    on any error nothing is launched and no output is touched.  A launch that
 *    the CUDA runtime rejects returns RLK_ERR_CUDA.  A zero-row call (N == 0 in
 *    rlk_linear_logp, M == 0 in rlk_det_gemm_fwd / _da) is a no-op that
 *    returns RLK_OK.
 *  - Determinism.  For fixed inputs every output bit is identical run to run,
 *    across streams, across leading dimensions and pointer alignment, and -- for
 *    every product whose reduction does not run over the rows (all but dB and
 *    the weight gradients) -- across the number of rows in the call (row
 *    chunking).  Which kernel, tile width and launch shape run may depend on the
 *    extents and the GPU's SM count, but the arithmetic of each output element
 *    (its ascending K reduction, the vocabulary split and merge order) depends
 *    only on the reduction and vocabulary extents, so the bits do not.
 *    rlk_numerics_version() changes whenever that arithmetic changes.
 *  - Alignment.  An operand whose base address is not 16-byte aligned, or
 *    whose leading dimension is not a multiple of 8 elements, is first copied
 *    into the workspace with a padded leading dimension (bit-identical result;
 *    the padding is zeros, which add exactly nothing).  The *_workspace_size
 *    functions account for that copy.
 *
 * Sources (web pages of the RL-Kernel project):
 *  [P3] "feat(linear-logp): add batch-invariant fused SM90 operator":
 *       Walkthrough (operator: hidden, lm-head weight, target ids, optional
 *       bias -> log-probability and log-sum-exp, never materialising the
 *       [N, V] logits), author notes (the vocabulary split is chosen from V
 *       only: V -> split count -> contiguous ranges -> ordered merge; backward
 *       is outside the contract and fails closed), PR body (online-softmax
 *       partials per split and an ordered combine).
 *  [P1] "feat(musa): add native deterministic gemm kernel": Summary (fixed
 *       ascending K-order reduction with FP32 accumulation; forward,
 *       dA = dC B^T, dB = A^T dC; FP32-output forward variant), review comment
 *       (an FP32-output forward's grad_output is cast to BF16 before dA / dB).
 *  [P2] "Support musa": review comment (det_gemm must never fall back to a
 *       non-deterministic matmul; it fails explicitly instead).
 */
#ifndef RLK_H
#define RLK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define RLK_API __attribute__((visibility("default")))
#else
#define RLK_API
#endif

#define RLK_NUMERICS_VERSION 2

typedef enum rlk_status {
    RLK_OK = 0,
    RLK_ERR_NULL = 1,               /* a required pointer is NULL                       */
    RLK_ERR_SHAPE = 2,              /* a size or leading dimension is out of range      */
    RLK_ERR_DTYPE = 3,              /* an rlk_dtype argument is not a supported value   */
    RLK_ERR_ALIGN = 4,              /* a pointer is not aligned to its element size     */
    RLK_ERR_WORKSPACE = 5,          /* workspace NULL or smaller than required          */
    RLK_ERR_UNSUPPORTED_DEVICE = 6, /* no CUDA device, or the device is not sm_103      */
    RLK_ERR_CUDA = 7,               /* the CUDA runtime rejected a launch or query      */
    RLK_ERR_TIMEOUT = 8,            /* a kernel's bounded wait expired (device error)   */
    RLK_ERR_BOUNDS = 9,             /* debug build: a kernel skipped an out-of-bounds store */
    RLK_ERR_NOT_DEBUG_BUILD = 10    /* the call exists only in the debug build          */
} rlk_status;

typedef enum rlk_dtype {
    RLK_BF16 = 0,                   /* bfloat16, 2 bytes                                */
    RLK_FP32 = 1                    /* IEEE binary32, 4 bytes                           */
} rlk_dtype;

/* Device error-word bits reported by rlk_get_device_error. */
#define RLK_DEVERR_TIMEOUT 0x1u     /* an mbarrier wait gave up after its time limit   */
#define RLK_DEVERR_BOUNDS 0x2u      /* debug build (librlk_debug.so, compiled with
                                       -DRLK_DEBUG): a global store's index fell outside
                                       the buffer it writes; the store was skipped      */

/* Human-readable name of a status code (static storage, never NULL). */
RLK_API const char* rlk_status_string(int status);

/* Bumped whenever a tile shape, reduction order or split policy change would
 * change output bits.  Equal versions => bit-identical outputs. */
RLK_API int rlk_numerics_version(void);

/* RLK_OK when the current CUDA device is sm_103 and usable, else the reason. */
RLK_API rlk_status rlk_device_check(void);

/*
 * Reads and clears the device error word after synchronising `stream`.
 * *flags receives the OR of RLK_DEVERR_* bits raised by kernels since the last
 * call (0 when nothing went wrong).  Returns RLK_ERR_TIMEOUT when the timeout
 * bit was set, else RLK_ERR_BOUNDS when the bounds bit was set, else RLK_OK.
 */
RLK_API rlk_status rlk_get_device_error(void* stream, uint32_t* flags);

/*
 * Diagnostic for the kernels' bounded waits.  Launches one CTA whose thread
 * waits on a shared-memory mbarrier that nothing ever completes, through the
 * same bounded-wait routine every tensor-core kernel uses, with a limit of
 * timeout_us microseconds (1 .. 2,000,000).  The wait gives up, raises
 * RLK_DEVERR_TIMEOUT in the device error word and the kernel returns, leaving
 * the CUDA context usable; rlk_get_device_error then reports RLK_ERR_TIMEOUT.
 * Returns RLK_ERR_SHAPE for a limit out of range.
 */
RLK_API rlk_status rlk_selftest_bounded_wait(uint32_t timeout_us, void* stream);

/*
 * Debug build.  The library is also built as librlk_debug.so with -DRLK_DEBUG
 * (same ABI, same arithmetic and output bits): there every kernel tests each
 * global store's index against the extent of the buffer it writes; a store
 * outside is skipped and raises RLK_DEVERR_BOUNDS (nothing traps), and the
 * linear-logp kernels record per-CTA phase timestamps and role cycle counters
 * (rlk_debug_trace_read).
 * rlk_is_debug_build returns 1 in that build, 0 in librlk.so.
 */
RLK_API int rlk_is_debug_build(void);

/*
 * Debug build: launches one thread that declares a store outside its buffer
 * through the store check; the store is skipped (no memory is written) and
 * RLK_DEVERR_BOUNDS is raised, so rlk_get_device_error then returns
 * RLK_ERR_BOUNDS.  librlk.so returns RLK_ERR_NOT_DEBUG_BUILD and launches nothing.
 */
RLK_API rlk_status rlk_selftest_store_check(void* stream);

/*
 * Debug build: copies the phase timestamps (%globaltimer, ns) and role cycle
 * counters that the linear-logp partials kernels recorded since the last read,
 * then clears them.  out receives
 * max_ctas records of RLK_TRACE_FIELDS uint64 values, indexed by CTA (block)
 * index: [0] CTA entry, [1] set-up done (barriers, TMEM, wait for the previous
 * kernel), [2] first operand stage landed (seen by the MMA issuer), [3] last MMA of
 * the CTA complete (accumulator handed to the epilogue), [4] last partial
 * written (epilogue), [5] CTA exit; then the SM's cycle counter at [6] entry and
 * [7] exit (cycles, not ns); then per-role SM cycle counts, each written when
 * the role finishes: the MMA issuer's [8] cycles waiting for operand stages
 * (after the first), [9] cycles waiting for a free accumulator, [10] cycles from
 * its first unit to its last MMA issued and [11] accumulator tiles issued (the
 * issuing CTA of a pair only); the TMA producer's [12] cycles waiting for free
 * ring slots and [13] cycles from its first unit to its last copy issued; the
 * first epilogue thread's [14] cycles waiting for complete accumulators and [15]
 * cycles reading and folding them.  0 = not recorded.  *n_ctas receives the
 * number of records kept (at most RLK_TRACE_MAX_CTAS).  librlk.so returns
 * RLK_ERR_NOT_DEBUG_BUILD.
 */
#define RLK_TRACE_FIELDS 16
#define RLK_TRACE_MAX_CTAS 1024
RLK_API rlk_status rlk_debug_trace_read(uint64_t* out, int64_t max_ctas, int64_t* n_ctas);

/* ===================================================================== *
 *  Fused linear log-probability                                  [P3]  *
 * ===================================================================== */

/*
 * The vocabulary split used by rlk_linear_logp, a function of V alone [P3
 * author notes].  The vocabulary is cut into vtiles = ceil(V / 256) tiles of
 * 256 ids; tiles are grouped into S contiguous, non-empty splits of
 * vtiles_per_split tiles (the last split may be shorter), with S no larger
 * than 1024:
 *     vtiles_per_split = ceil(vtiles / 1024),  S = ceil(vtiles / vtiles_per_split).
 * Split j covers vocabulary ids [j * vps * 256, min((j + 1) * vps * 256, V)).
 * Host-only; needs no device.  Returns RLK_ERR_SHAPE for V < 1 or V >= 2^31 - 256.
 */
RLK_API rlk_status rlk_vocab_split_policy(int64_t V, int64_t* num_splits, int64_t* vtiles_per_split,
                                  int64_t* num_vtiles);

/*
 * Workspace bytes that rlk_linear_logp needs for exactly these operands:
 * N * S * 8 bytes of per-(row, split) online-softmax partials, N * 4 bytes for
 * the gathered target logits, 256 bytes for the kernel's work-unit counter
 * (zeroed by each call that deals more than 8 rounds of units), plus a padded copy of hidden and/or weight when that
 * operand is misaligned (see "Alignment").  Each region starts on a 256-byte
 * boundary.  Returns 0 for invalid arguments.
 */
RLK_API size_t rlk_linear_logp_workspace_size(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                                      const void* weight, int64_t V, int64_t ld_weight);

/*
 * logp[r] = z[r, target[r]] - lse[r],   lse[r] = log sum_v exp(z[r, v]),
 * z[r, v] = sum_h hidden[r, h] * weight[v, h] (+ bias[v])          [P3 Walkthrough]
 *
 *  hidden        BF16 [N, H], leading dimension ld_hidden (>= H)
 *  weight        BF16 [V, H] (the lm-head weight), leading dimension ld_weight (>= H)
 *  bias          FP32 [V] or NULL; added in FP32 after the full H reduction
 *  target        int64, row r reads target[r * target_stride]; stride 0 means one
 *                id shared by every row (an expanded target)
 *  logp, lse     FP32 [N] outputs
 *  target_logit  FP32 [N] output or NULL: the logit z[r, target[r]] exactly as it
 *                entered the log-sum-exp
 *  workspace     >= rlk_linear_logp_workspace_size(...) bytes, 16-byte aligned
 *
 * Shapes: 0 <= N < 2^31 - 256, 1 <= H < 2^20, 1 <= V < 2^31 - 256 (the kernels
 * index rows and ids in 32-bit ints).  A target outside
 * [0, V) yields logp = NaN (and target_logit = NaN) for that row; lse is
 * still valid; nothing is read out of bounds.
 *
 * Arithmetic (fixed; depends on V and H only): FP32 accumulation over H in
 * ascending blocks of 64 (tensor cores, K=16 per instruction: M=256 x N=256
 * over a pair of SMs, or M=128 x N=256 on one SM for calls of at most 128
 * rows, which give the same bits per element); per 256-id tile
 * and per row an online max / sum-of-exponentials in ascending vocabulary
 * order; S = rlk_vocab_split_policy(V) partials per row merged in a fixed
 * order (lane j%32 ascending, then a fixed xor-butterfly).  Each row's bits
 * are therefore independent of N, of the row's position and of its
 * neighbours.  Equivalent to rlk_linear_logp_partials followed by
 * rlk_linear_logp_combine on the same stream.
 */
RLK_API rlk_status rlk_linear_logp(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                           const void* weight, int64_t V, int64_t ld_weight,
                           const float* bias, const int64_t* target, int64_t target_stride,
                           float* logp, float* lse, float* target_logit,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Throughput-mode ablation (not batch invariant when num_splits depends on N).
 *
 * The RL-Kernel linear-logp page [P3 PR body, "Why this happens"] describes the
 * project's earlier throughput scheduler: it picks the vocabulary split from N,
 * V and the SM count, so one row may take a different FP32 merge path when the
 * batch around it changes.  These entry points exist only to measure what the
 * V-only policy costs against such a scheduler; rlk_linear_logp stays the
 * operator.
 *
 * rlk_throughput_split_count: an occupancy-driven split count (the pages give
 * no formula; this is the reading taken): enough splits that the (split,
 * 256-row block) units number at least 8 per pair of SMs,
 *     num_splits = min(ceil(V / 256), ceil(8 * floor(sm_count / 2) / ceil(N / 256))).
 * sm_count = 0 queries the current device.  Host arithmetic only otherwise.
 * Returns RLK_ERR_SHAPE for N < 1, V < 1, N or V >= 2^31 - 256 or sm_count < 0.
 */
RLK_API rlk_status rlk_throughput_split_count(int64_t N, int64_t V, int32_t sm_count,
                                              int64_t* num_splits);

/*
 * rlk_linear_logp with an explicit split count: the 256-id tiles are cut into
 * ceil(vtiles / vps) contiguous splits of vps = ceil(vtiles / num_splits) tiles
 * (num_splits clamped to [1, vtiles]); num_splits = 0 selects the V-only policy
 * and then equals rlk_linear_logp bit for bit.  Every other argument, the
 * arithmetic within a split, the merge order and the error behaviour are those
 * of rlk_linear_logp; the workspace must hold
 * rlk_linear_logp_splits_workspace_size(..., num_splits) bytes.  Results are
 * deterministic for a given num_splits; they are batch invariant only if the
 * caller keeps num_splits fixed across batches.  RLK_ERR_SHAPE for num_splits < 0.
 */
RLK_API size_t rlk_linear_logp_splits_workspace_size(const void* hidden, int64_t N, int64_t H,
                                                     int64_t ld_hidden, const void* weight,
                                                     int64_t V, int64_t ld_weight,
                                                     int64_t num_splits);
RLK_API rlk_status rlk_linear_logp_splits(const void* hidden, int64_t N, int64_t H,
                                          int64_t ld_hidden, const void* weight, int64_t V,
                                          int64_t ld_weight, const float* bias,
                                          const int64_t* target, int64_t target_stride,
                                          float* logp, float* lse, float* target_logit,
                                          int64_t num_splits, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * First stage of rlk_linear_logp: one fused tensor-core kernel (projection
 * tiles + online-softmax epilogue) that writes the per-(row, split) partials
 * and the target logits into `workspace`.  Arguments as for rlk_linear_logp.
 */
RLK_API rlk_status rlk_linear_logp_partials(const void* hidden, int64_t N, int64_t H, int64_t ld_hidden,
                                    const void* weight, int64_t V, int64_t ld_weight,
                                    const float* bias, const int64_t* target,
                                    int64_t target_stride, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * Second stage: merges the S partials of each row in the fixed order and
 * writes logp, lse and (optionally) target_logit.  `workspace` must hold the
 * partials written by rlk_linear_logp_partials with the same N, H, V, operand
 * pointers and leading dimensions (those fix where the partials sit).
 */
RLK_API rlk_status rlk_linear_logp_combine(int64_t N, int64_t V, const int64_t* target,
                                   int64_t target_stride, float* logp, float* lse,
                                   float* target_logit, const void* workspace,
                                   size_t workspace_bytes, void* stream);

/* ---- Vocabulary-parallel linear-logp ------------------------------------
 * The page's split policy [P3 author notes: V -> split count -> contiguous
 * ranges -> ordered merge] lets the vocabulary be divided between devices at
 * split boundaries: a shard is a contiguous run of whole splits
 * [split_begin, split_end) of rlk_vocab_split_policy(V), i.e. the weight rows of
 * vocabulary ids [v_begin, v_end) with v_begin = split_begin * vps * 256 and
 * v_end = min(split_end * vps * 256, V).  Each shard computes the (m, s)
 * partials of its splits (bit for bit those the whole-vocabulary call computes)
 * and the target logits of the rows whose target it holds; after the partials
 * are exchanged, rlk_linear_logp_combine_shards merges every row's S partials in
 * the same fixed order as rlk_linear_logp, so logp, lse and the target logit
 * equal the one-device results bit for bit.
 */

/*
 * A balanced partition into num_shards (1 .. 64) shards: shard q gets splits
 * [floor(q S / num_shards), floor((q + 1) S / num_shards)) (empty when
 * num_shards > S) and the vocabulary ids they cover.  Host-only.
 * RLK_ERR_SHAPE for V out of range, num_shards outside [1, 64] or shard outside
 * [0, num_shards).
 */
RLK_API rlk_status rlk_vocab_shard_range(int64_t V, int64_t num_shards, int64_t shard,
                                         int64_t* split_begin, int64_t* split_end,
                                         int64_t* v_begin, int64_t* v_end);

/*
 * Workspace bytes of rlk_linear_logp_shard_partials: 256 bytes for the kernel's
 * work-unit counter plus padded copies of a misaligned hidden / weight shard.
 * Returns 0 for invalid arguments.
 */
RLK_API size_t rlk_linear_logp_shard_workspace_size(const void* hidden, int64_t N, int64_t H,
                                                    int64_t ld_hidden, const void* weight_shard,
                                                    int64_t V, int64_t split_begin,
                                                    int64_t split_end, int64_t ld_weight);

/*
 * Partials of one vocabulary shard.
 *  hidden        BF16 [N, H] (ld_hidden), as for rlk_linear_logp
 *  weight_shard  BF16 [v_end - v_begin, H] (ld_weight): rows v_begin .. v_end - 1 of
 *                the lm-head weight
 *  V             the WHOLE vocabulary size (it fixes the split policy)
 *  split_begin, split_end   0 <= split_begin <= split_end <= S
 *  bias_shard    FP32 [v_end - v_begin] (bias[v_begin ..]) or NULL
 *  target        int64 global ids, target[r * target_stride]
 *  partials      FP32 output: for row r and local split i (0 <= i < split_end -
 *                split_begin) the pair (m, s) at partials[2 (r ld_partials + i)];
 *                ld_partials >= split_end - split_begin (in pairs), 8-byte aligned
 *  target_logit  FP32 [N] output: written for the rows whose target lies in
 *                [v_begin, v_end) (the logit exactly as it entered the partials);
 *                every other entry is left untouched
 * N == 0 or an empty shard is a no-op.  Errors as for rlk_linear_logp.
 */
RLK_API rlk_status rlk_linear_logp_shard_partials(const void* hidden, int64_t N, int64_t H,
                                                  int64_t ld_hidden, const void* weight_shard,
                                                  int64_t V, int64_t split_begin,
                                                  int64_t split_end, int64_t ld_weight,
                                                  const float* bias_shard, const int64_t* target,
                                                  int64_t target_stride, float* partials,
                                                  int64_t ld_partials, float* target_logit,
                                                  void* workspace, size_t workspace_bytes,
                                                  void* stream);

/*
 * The fixed-order merge over gathered shard partials.
 *  split_offsets  HOST array of num_shards + 1 (1 .. 64 shards) split indices:
 *                 0 = split_offsets[0] <= ... <= split_offsets[num_shards] = S;
 *                 shard q holds splits [split_offsets[q], split_offsets[q + 1])
 *  partials       shard q's pair for row r and local split i at
 *                 partials[2 (q shard_stride + r ld_partials + i)] (shard_stride and
 *                 ld_partials in pairs; shard_stride >= N ld_partials when
 *                 num_shards > 1), e.g. an all-gather of every shard's output
 *  target_logits  shard q's target logits at target_logits[q zt_stride + r]
 *                 (zt_stride >= N when num_shards > 1); row r's value is taken
 *                 from the shard that holds its target
 *  target, target_stride, logp, lse, target_logit  as for rlk_linear_logp_combine
 * Output bits equal rlk_linear_logp's for the same rows.
 */
RLK_API rlk_status rlk_linear_logp_combine_shards(int64_t N, int64_t V, const int64_t* target,
                                                  int64_t target_stride, int64_t num_shards,
                                                  const int64_t* split_offsets,
                                                  const float* partials, int64_t ld_partials,
                                                  int64_t shard_stride,
                                                  const float* target_logits, int64_t zt_stride,
                                                  float* logp, float* lse, float* target_logit,
                                                  void* stream);

/*
 * rlk_linear_logp without a workspace argument, for callers that cannot
 * allocate device memory where they call it: a plugin inside a host framework
 * that owns the device allocator and exposes no scratch-buffer hook, code that
 * runs under a device-memory budget fixed in advance, or a latency-critical loop
 * that must not call cudaMalloc / cudaFree (they can synchronise the device).
 * The pages have no counterpart to this entry point; it exists for those callers.
 *
 * Same arguments, arithmetic and output bits as rlk_linear_logp.  Scratch comes
 * from one fixed 32 MiB array in the library's own device image, which every GPU
 * that loads the library holds until the process exits.  Nothing is allocated:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *  - Limit: the call needs N * S * 8 + N * 4 bytes (each rounded up to 256; S from
 *    rlk_vocab_split_policy(V)) + 256, plus a padded copy of any misaligned operand;
 *    more than RLK_NOALLOC_SCRATCH_BYTES returns RLK_ERR_WORKSPACE and launches
 *    nothing.  (V = 151936: up to about 7,000 rows per call.)
 *  - The first call on each device looks up the array's device address (with that
 *    device current) and caches it for as long as the same CUDA context stays
 *    current (a new context, e.g. after cudaDeviceReset, repeats the lookup); make
 *    that first call, in each context, before any stream capture.
 *  - Every call on a device shares the array and leaves its contents behind; no
 *    part of it needs to start at zero.  Calls whose GPU work overlaps (two streams
 *    without ordering between them) race on it: order them.
 */
#define RLK_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
RLK_API rlk_status rlk_linear_logp_noalloc(const void* hidden, int64_t N, int64_t H,
                                           int64_t ld_hidden, const void* weight, int64_t V,
                                           int64_t ld_weight, const float* bias,
                                           const int64_t* target, int64_t target_stride,
                                           float* logp, float* lse, float* target_logit,
                                           void* stream);

/*
 * Backward of rlk_linear_logp for an upstream gradient g = dL/dlogp [N].
 * The page fails closed on backward ("outside the first contract", [P3] author
 * notes); this is that next step.  With z = hidden . W^T (+ bias):
 *   G[r, v]       = g[r] * ([v == target[r]] - exp(z[r, v] - lse[r]))   (= dL/dz)
 *   grad_hidden   = G . W             [N, H]   (ascending over V)
 *   grad_weight   = G^T . hidden      [V, H]   (ascending over the N rows)
 *   grad_bias[v]  = sum_r G[r, v]     [V]      (ascending over the N rows)
 * G is formed in FP32 from the recomputed logits and the forward's lse, then
 * rounded to BF16 (nearest even); the three reductions run on that BF16 G with
 * FP32 accumulation (the products are rlk_det_gemm_fwd and rlk_det_gemm_db).
 * A row whose target is outside [0, V) contributes zero gradient.
 *
 *  hidden, weight, bias, target, target_stride  as for rlk_linear_logp (a
 *                misaligned hidden or weight is copied into the workspace first,
 *                as in the forward; bit-identical results)
 *  lse           FP32 [N], the forward's lse for these inputs
 *  grad_logp     FP32 [N]
 *  grad_hidden   [N, H] in grad_hidden_dtype (RLK_BF16 / RLK_FP32), pitch
 *                ld_grad_hidden; NULL to skip
 *  grad_weight   [V, H] in grad_weight_dtype, pitch ld_grad_weight; NULL to skip
 *  grad_bias     FP32 [V] or NULL to skip
 *  workspace     >= rlk_linear_logp_backward_workspace_size_for(...) bytes
 *                (rlk_linear_logp_backward_workspace_size(N, V) suffices when hidden
 *                and weight are 16-byte aligned with a pitch that is a multiple of 8
 *                elements), 256-byte aligned.  After the call its first
 *                N * 8*ceil(V/8) * 2 bytes hold G as BF16 [N, 8*ceil(V/8)] (row pitch
 *                8*ceil(V/8)); the next 256 bytes hold the kernel's work-unit counter
 *                (zeroed by a call that deals more than 8 rounds of units), then the
 *                padded copies of a misaligned hidden / weight.
 * Errors: every argument, including the output pointers, pitches and dtypes that
 * the two products check, is validated before the first launch; on an error
 * nothing is launched and no output or workspace byte is touched.
 * Determinism: every output is bitwise reproducible; a grad_hidden row depends
 * only on its own row's inputs (batch invariant), while grad_weight and
 * grad_bias sum over the rows of the call.  N == 0 writes zeros to grad_weight
 * and grad_bias.
 */
RLK_API size_t rlk_linear_logp_backward_workspace_size(int64_t N, int64_t V);
RLK_API size_t rlk_linear_logp_backward_workspace_size_for(const void* hidden, int64_t N,
                                                           int64_t H, int64_t ld_hidden,
                                                           const void* weight, int64_t V,
                                                           int64_t ld_weight);
RLK_API rlk_status rlk_linear_logp_backward(const void* hidden, int64_t N, int64_t H,
                                            int64_t ld_hidden, const void* weight, int64_t V,
                                            int64_t ld_weight, const float* bias,
                                            const int64_t* target, int64_t target_stride,
                                            const float* lse, const float* grad_logp,
                                            void* grad_hidden, int grad_hidden_dtype,
                                            int64_t ld_grad_hidden, void* grad_weight,
                                            int grad_weight_dtype, int64_t ld_grad_weight,
                                            float* grad_bias, void* workspace,
                                            size_t workspace_bytes, void* stream);

/* ===================================================================== *
 *  Deterministic GEMM family                                      [P1]  *
 * ===================================================================== */
/*
 * All three products accumulate in FP32 over the reduction index in ascending
 * blocks of 64 (16 per tensor-core instruction) with no split of the
 * reduction, no atomics and no data-dependent order, so every output is
 * bitwise reproducible.  Output tiles are 256 x 256 (one per pair of SMs, M=256 x
 * N=256 x K=16 per tensor-core instruction), or 256 x 128 (N=128) when the
 * 256-wide tiles would leave at least half of the SM pairs idle; with a
 * reduction of 16384 or more, a last wave of 256-wide tiles that would fill at
 * most half the pairs runs as 128-wide halves in a second launch on the same
 * stream; dA and the linear forward use 256 x 224 tiles where those fill the
 * waves better (rlk_det_gemm_tile_plan reports the choice).  Each output element
 * is the same sum whatever its tile, so the tiling never changes a bit.
 * Outputs are BF16 (round to nearest even from the FP32 accumulator) or FP32.
 * A batched operand [b, M, K] is passed flattened as [b * M, K] (a leading
 * shape is a row count), so fwd and dA are bitwise equal per row whatever the
 * batching, and dB sums over all b * M rows in ascending order.
 * Shapes: 0 <= M < 2^31 - 256 and 1 <= K, N < 2^31 - 256 (M is the row count of A / dC,
 * K the column count of A and row count of B, N the column count of B / dC).
 * Leading dimensions >= the column count of their matrix.
 */

#define RLK_GEMM_FWD 0
#define RLK_GEMM_DA 1
#define RLK_GEMM_DB 2
#define RLK_GEMM_LINEAR_FWD 3
#define RLK_GEMM_LINEAR_DX 4
#define RLK_GEMM_LINEAR_DW 5
#define RLK_GEMM_FWD_ACCUM 6

/*
 * The output tiling a det_gemm product uses (host arithmetic only, no device
 * call), for op (RLK_GEMM_*) with an out_rows x out_cols output reduced over
 * `red` elements on a device of sm_count SMs:
 *  *tile_cols     256; 128 when all 256-wide tiles fit in half a wave of SM pairs
 *                 (2 x tiles <= sm_count / 2); 224 for dA and the linear forward
 *                 (right operand read K-major) where 224-wide tiles cost fewer
 *                 wave-times per pair;
 *  *split_blocks  the number of 256-wide blocks at the end of the unit order that
 *                 are computed as two 128-wide halves in a second launch: the last
 *                 partial wave, when it would fill at most half the pairs and red
 *                 >= 16384 (0: none);
 *  *launches      1 or 2.
 * The tiling never changes an output bit (each element runs the same MMAs in the
 * same order); this reports it for tests and measurements.  RLK_ERR_NULL for a
 * null output pointer, RLK_ERR_SHAPE for an unknown op, an extent outside
 * [1, 2^31 - 256) or sm_count < 2.  The two-product entries (rlk_det_gemm_backward,
 * rlk_det_linear_backward) follow it for each product when they run the products
 * as separate launches; their one-launch path keeps 256-wide tiles.
 */
RLK_API rlk_status rlk_det_gemm_tile_plan(int op, int64_t out_rows, int64_t out_cols, int64_t red,
                                          int32_t sm_count, int32_t* tile_cols,
                                          int64_t* split_blocks, int32_t* launches);

/*
 * Workspace bytes the given op needs for exactly these inputs: padded copies
 * of misaligned BF16 operands and, for an FP32 dC, its BF16 rounding.
 * (x, y) are the op's two inputs in argument order:
 *   RLK_GEMM_FWD: x = A [M, K] (BF16),       y = B [K, N] (BF16)
 *   RLK_GEMM_DA:  x = dC [M, N] (x_dtype),   y = B [K, N] (BF16)
 *   RLK_GEMM_DB:  x = A [M, K] (BF16),       y = dC [M, N] (y_dtype)
 *   RLK_GEMM_LINEAR_FWD: x = X [M, K] (BF16),  y = W [N, K] (BF16)
 *   RLK_GEMM_LINEAR_DX:  x = dY [M, N] (x_dtype), y = W [N, K] (BF16)
 *   RLK_GEMM_LINEAR_DW:  x = dY [M, N] (x_dtype), y = X [M, K] (BF16)
 *   RLK_GEMM_FWD_ACCUM:  as RLK_GEMM_FWD
 * Returns 0 when nothing needs staging or the arguments are invalid.
 */
RLK_API size_t rlk_det_gemm_workspace_size(int op,
                                   const void* x, int x_dtype, int64_t x_rows, int64_t x_cols,
                                   int64_t ldx,
                                   const void* y, int y_dtype, int64_t y_rows, int64_t y_cols,
                                   int64_t ldy);

/*
 * C[M, N] = A[M, K] . B[K, N]                               [P1 Summary: forward]
 *  A  BF16 [M, K] (ld lda);  B  BF16 [K, N] (ld ldb);  C  c_dtype [M, N] (ld ldc).
 */
RLK_API rlk_status rlk_det_gemm_fwd(const void* A, int64_t M, int64_t K, int64_t lda,
                            const void* B, int64_t N, int64_t ldb,
                            void* C, int c_dtype, int64_t ldc,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * dA[M, K] = dC[M, N] . B[K, N]^T                                  [P1 Summary: dA]
 *  dC dc_dtype [M, N] (ld lddc): an FP32 dC (the gradient of an FP32-output
 *     forward) is rounded to BF16 (nearest even) before the product, as the
 *     FP32-output backward requires [P1 review comment].
 *  B  BF16 [K, N] (ld ldb);  dA out_dtype [M, K] (ld ldda).
 */
RLK_API rlk_status rlk_det_gemm_da(const void* dC, int dc_dtype, int64_t M, int64_t N, int64_t lddc,
                           const void* B, int64_t K, int64_t ldb,
                           void* dA, int out_dtype, int64_t ldda,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * dB[K, N] = A[M, K]^T . dC[M, N]                                  [P1 Summary: dB]
 *  Reduction over all M rows in ascending order.  dC as for rlk_det_gemm_da.
 *  A  BF16 [M, K] (ld lda);  dB out_dtype [K, N] (ld lddb).
 *  M == 0 is a valid empty reduction: dB is written with zeros.
 */
RLK_API rlk_status rlk_det_gemm_db(const void* A, int64_t M, int64_t K, int64_t lda,
                           const void* dC, int dc_dtype, int64_t N, int64_t lddc,
                           void* dB, int out_dtype, int64_t lddb,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * Both gradients of C = A . B from one dC                  [P1 Summary; review comment]
 *   dA[M, K] = dC . B^T   and   dB[K, N] = A^T . dC
 * bitwise equal to rlk_det_gemm_da and rlk_det_gemm_db on the same arguments, but
 * an FP32 dC (the gradient of an FP32-output forward) is rounded to BF16 once, into
 * the workspace, and both products read that copy (likewise a misaligned dC is
 * copied once).  dA or dB may be NULL to skip it.  Every argument of both products
 * is validated before the first launch.  M == 0: dA is empty, dB is written with
 * zeros.  When both products are wanted, each fills at least one wave of the SM
 * pairs with 256 x 256 tiles and their reductions (N and M) are within a factor
 * of two, both run in one launch over both tile lists (the same bits).
 * workspace >= rlk_det_gemm_backward_workspace_size(...) bytes (the staged copies
 * plus a 256-byte unit counter), 16-byte aligned.
 */
RLK_API size_t rlk_det_gemm_backward_workspace_size(const void* dC, int dc_dtype, int64_t M,
                                                    int64_t N, int64_t lddc, const void* A,
                                                    int64_t K, int64_t lda, const void* B,
                                                    int64_t ldb);
RLK_API rlk_status rlk_det_gemm_backward(const void* dC, int dc_dtype, int64_t M, int64_t N,
                                         int64_t lddc, const void* A, int64_t K, int64_t lda,
                                         const void* B, int64_t ldb, void* dA, int da_dtype,
                                         int64_t ldda, void* dB, int db_dtype, int64_t lddb,
                                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * Fixed-order sum of per-device partial results: the cross-device step of a dB
 * whose rows are divided between devices, where each device's partial product is
 * gathered and the parts are added in a fixed device order (a ring all-reduce
 * would add them in an order that depends on the ring):
 *   out[r, c] = part_0[r, c] + part_1[r, c] + ... + part_{P-1}[r, c]
 * added in FP32 (round to nearest) in ascending part order and written as FP32
 * or BF16 (round to nearest even).  Part p starts at partials + p * part_stride
 * (elements, >= rows * ld_partial when P > 1), row pitch ld_partial; out has
 * pitch ld_out and must not overlap the partials.  The result is bitwise
 * reproducible and the same on every device that runs it on the same gathered
 * partials; it depends on how the rows were divided (the order of the sum), so
 * it may differ in the last bits from one rlk_det_gemm_db over all rows.
 * rows == 0 is a no-op.  P must be >= 1.
 */
RLK_API rlk_status rlk_sum_partials_ordered(const float* partials, int64_t num_parts,
                                            int64_t rows, int64_t cols, int64_t ld_partial,
                                            int64_t part_stride, void* out, int out_dtype,
                                            int64_t ld_out, void* stream);

/*
 * C[M, N] += A[M, K] . B[K, N] with C in FP32 — the accumulate-into-FP32 forward
 * [P1 Implementation: forward_accum_fp32].  Reading taken: the product is formed
 * exactly as by rlk_det_gemm_fwd (same tiles, same ascending K order) and the
 * existing C is added to it once, in FP32 round-to-nearest, after the full K sum;
 * so the result equals C + rlk_det_gemm_fwd(..., RLK_FP32) evaluated in FP32.
 * C must not alias A or B.  K == 0 leaves C unchanged.
 */
RLK_API rlk_status rlk_det_gemm_fwd_accum_fp32(const void* A, int64_t M, int64_t K, int64_t lda,
                                              const void* B, int64_t N, int64_t ldb, float* C,
                                              int64_t ldc, void* workspace, size_t workspace_bytes,
                                              void* stream);

/*
 * The linear layout, weight stored [N, K] as in a linear layer
 * [P1 Implementation: transposed-RHS forward, linear(A, weight[N, K]), canonical
 * transposed dB for [N, K] weight gradients]:
 *   rlk_det_linear_fwd:  Y[M, N]  = X[M, K] . W[N, K]^T     (W's transpose never formed)
 *   rlk_det_linear_dx:   dX[M, K] = dY[M, N] . W[N, K]
 *   rlk_det_linear_dw:   dW[N, K] = dY[M, N]^T . X[M, K]    (ascending over all M rows)
 * dY may be BF16 or FP32; an FP32 dY (the gradient of an FP32-output forward) is
 * rounded to BF16 first [P1 review comment].  Same tile shape, reduction order,
 * output dtypes, staging and error rules as the three products above; rows of Y
 * and dX are bitwise independent of the other rows in the call.
 */
RLK_API rlk_status rlk_det_linear_fwd(const void* X, int64_t M, int64_t K, int64_t ldx,
                                     const void* W, int64_t N, int64_t ldw, void* Y, int y_dtype,
                                     int64_t ldy, void* workspace, size_t workspace_bytes,
                                     void* stream);
RLK_API rlk_status rlk_det_linear_dx(const void* dY, int dy_dtype, int64_t M, int64_t N,
                                    int64_t lddy, const void* W, int64_t K, int64_t ldw, void* dX,
                                    int out_dtype, int64_t lddx, void* workspace,
                                    size_t workspace_bytes, void* stream);
RLK_API rlk_status rlk_det_linear_dw(const void* dY, int dy_dtype, int64_t M, int64_t N,
                                    int64_t lddy, const void* X, int64_t K, int64_t ldx, void* dW,
                                    int out_dtype, int64_t lddw, void* workspace,
                                    size_t workspace_bytes, void* stream);

/*
 * Both gradients of Y = X . W^T (W stored [N, K]) from one dY:
 *   dX[M, K] = dY . W   and   dW[N, K] = dY^T . X
 * bitwise equal to rlk_det_linear_dx and rlk_det_linear_dw, with an FP32 dY rounded
 * to BF16 once and shared; the rest as for rlk_det_gemm_backward.
 */
RLK_API size_t rlk_det_linear_backward_workspace_size(const void* dY, int dy_dtype, int64_t M,
                                                      int64_t N, int64_t lddy, const void* X,
                                                      int64_t K, int64_t ldx, const void* W,
                                                      int64_t ldw);
RLK_API rlk_status rlk_det_linear_backward(const void* dY, int dy_dtype, int64_t M, int64_t N,
                                           int64_t lddy, const void* X, int64_t K, int64_t ldx,
                                           const void* W, int64_t ldw, void* dX, int dx_dtype,
                                           int64_t lddx, void* dW, int dw_dtype, int64_t lddw,
                                           void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* RLK_H */
