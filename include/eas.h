/*
 * eas.h - C ABI of the GB300 (sm_103a) block-sparse fused LM-head.
 *
 * The operation is the one described on "perf(megatron): add block-sparse
 * fused LM-head backward" (SkyRL PR #2376) and the layers it builds on
 * (#2374 "fuse LM-head entropy for RL", #2375 "add block-sparse fused LM-head
 * forward"):
 *
 *   - a loss mask marks which tokens (rows of `hidden`) are active;
 *   - the mask is turned into ordered active spans, coalescing runs whose
 *     inactive gap is at most max_gap (128 on the page, Bugbot "Overview");
 *   - the forward returns, for every active token, the target-token log
 *     probability and the softmax entropy of logits = hidden . W^T, computed
 *     one vocabulary tile at a time with an online log-sum-exp, never
 *     materialising the [T, V] logits;
 *   - the backward builds d-logits only for active tiles ("What does this PR
 *     do?", "How it works"), and projects them to dHidden and dW through the
 *     ordered spans, one vocabulary chunk at a time, the final chunk sized to
 *     its live width ("How it works"; greptile "Wide-tail grid exceeds live
 *     split").
 *
 * Formulas (the page names them; these are their textbook definitions):
 *   z      = W h_t                         W is [V, H] (nn.Linear layout)
 *   lse_t  = log sum_v exp(z_v)
 *   logp_t = z_target - lse_t
 *   H_t    = lse_t - sum_v p_v z_v,        p = exp(z - lse_t)
 *   dZ_t   = g_lp,t (onehot(target) - p) - g_H,t p (z - lse_t + H_t)
 *   dHidden = dZ W,   dW = dZ^T hidden
 * with g_lp = dL/dlogp and g_H = dL/dH (autograd convention: the gradient of
 * L = sum_t g_lp,t logp_t + g_H,t H_t).  Rows whose mask byte is 0 have
 * logp = H = lse = 0 and a zero dHidden row, whatever g holds there.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major,
 *     16-byte aligned.  Nothing is allocated and the host is never
 *     synchronised: every call only enqueues kernels on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream).
 *   - Argument errors that the host can see are returned at once and nothing
 *     is launched.  Errors only the device can see (spans that do not cover
 *     the mask, a span buffer that is too small, a pipeline wait that ran out
 *     of time) are written to a status word inside the workspace; read it with
 *     eas_read_device_status().  The status word is cleared at the start of
 *     every call that takes the workspace.
 *   - A workspace belongs to one call at a time: two calls whose kernels may
 *     run at the same time on the GPU (different streams, or threads without
 *     ordering) need different workspaces.
 *   - eas_last_error() returns a thread-local message about the last error.
 */
#ifndef EAS_H_
#define EAS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EAS_OK = 0,
    EAS_ERR_INVALID_ARG = 1,    /* a host-visible argument is wrong            */
    EAS_ERR_INVALID_SPANS = 2,  /* spans unsorted, out of range, overlapping,
                                   or an active token lies outside every span */
    EAS_ERR_UNSUPPORTED = 3,    /* shape or alignment the library does not run */
    EAS_ERR_WORKSPACE = 4,      /* workspace missing or smaller than required */
    EAS_ERR_CUDA = 5,           /* a CUDA runtime/driver call failed           */
    EAS_ERR_TIMEOUT = 6,        /* a kernel pipeline wait ran out of time      */
    EAS_ERR_SPAN_CAPACITY = 7,  /* more spans than the caller's buffer holds   */
    EAS_ERR_INVALID_LAYOUT = 8  /* packed-segment offsets not a valid CP layout */
} eas_status;

typedef enum {
    EAS_BF16 = 0,   /* hidden, W, dhidden bf16; tensor cores, fp32 accumulate */
    EAS_FP32 = 1,   /* hidden, W, dhidden fp32; fp32 FMA throughout           */
    EAS_E4M3 = 2    /* hidden, W in e4m3 with per-row fp32 scales
                       (eas_lmhead_fwd_fp8, eas_lmhead_bwd_fp8), tensor cores */
} eas_dtype;

/* Row policy for the forward/backward (the `flags` argument). */
#define EAS_ROWS_ACTIVE 0u  /* tensor-core work on the active rows of the
                               spans only (gap rows inside a span skipped)   */
#define EAS_ROWS_SPAN   1u  /* every row of every span, gap rows included
                               (span-contiguous schedule; gap rows still get
                               zero outputs and gradients)                  */

/* Backward only: the workspace still holds what eas_lmhead_fwd left in it
 * for the same hidden, mask, spans and row policy, enqueued before on the same
 * stream with nothing else touching the workspace in between.  The backward
 * then reuses that call's row schedule and packed hidden rows instead of
 * rebuilding them, and keeps its status word instead of clearing it.  The
 * backward's vocab_chunk does not matter for this. */
#define EAS_REUSE_FWD_ROWS 2u

/* Default vocabulary chunk width of the backward (columns of d-logits held
 * in the staging buffer at once).  0 passed as vocab_chunk selects it. */
#define EAS_DEFAULT_VOCAB_CHUNK 16384

/* ------------------------------------------------------------------ spans */

/* Bytes of workspace eas_build_active_spans needs for T tokens. */
size_t eas_spans_workspace_size(int64_t T);

/*
 * Ordered active spans of a loss mask ("What does this PR do?": ordered
 * active spans; Bugbot "Overview": coalesced with gaps <= 128).
 *
 *   mask      [T] uint8, nonzero = active token.
 *   max_gap   >= 0; two maximal active runs merge into one span when the
 *             number of inactive tokens between them is <= max_gap.
 *   spans     [cap][2] int32, out: half-open [start, end) pairs, ascending;
 *             spans start and end on active tokens.  Only the first
 *             min(S, cap) pairs are written.
 *   num_spans [1] int32 device, out: S, the true span count (may exceed cap,
 *             in which case the status word reads EAS_ERR_SPAN_CAPACITY).
 *   ws        workspace of eas_spans_workspace_size(T) bytes (holds the
 *             status word).
 * An empty mask gives S = 0; an all-active mask gives one span [0, T).
 */
eas_status eas_build_active_spans(const uint8_t* mask, int64_t T, int32_t max_gap,
                                  int32_t* spans, int64_t cap, int32_t* num_spans,
                                  void* ws, size_t ws_bytes, void* stream);

/*
 * Context-parallel local layout ("How it works": forward mask and spans come
 * from a CP-aware packed layout; diagram: "CP-local ordered spans").  Packed
 * segments are [seg_offsets[k], seg_offsets[k+1]) for k < n_segs
 * (seg_offsets[0] = 0, seg_offsets[n_segs] = T, device int32), each a
 * multiple of 2*cp_size long.  Load-balanced split: every segment is cut into
 * 2*cp_size equal chunks and rank cp_rank holds chunk cp_rank followed by
 * chunk 2*cp_size-1-cp_rank, segments in order.  Writes, for each of the
 * rank's T/cp_size local tokens, its global index (local_to_global) and its
 * mask byte (local_mask).  Run eas_build_active_spans on local_mask to get
 * the rank's CP-local ordered spans.  Offsets that do not form such a layout
 * set EAS_ERR_INVALID_LAYOUT in the status word of ws (>= 16 bytes).
 */
eas_status eas_cp_local_layout(const uint8_t* mask, const int32_t* seg_offsets, int32_t n_segs,
                               int64_t T, int32_t cp_size, int32_t cp_rank,
                               uint8_t* local_mask, int32_t* local_to_global,
                               void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- LM head */

/*
 * Bytes of workspace eas_lmhead_fwd and eas_lmhead_bwd need (the larger of
 * the two, so one workspace serves both).  vocab_chunk = 0 selects
 * EAS_DEFAULT_VOCAB_CHUNK.
 */
size_t eas_lmhead_workspace_size(int64_t T, int64_t H, int64_t V, eas_dtype dtype,
                                 int64_t vocab_chunk);

/*
 * Forward: target log-probability, softmax entropy and log-sum-exp of the
 * active tokens (#2375 "add block-sparse fused LM-head forward", #2374 "fuse
 * LM-head entropy for RL", as summarised on the #2376 page).
 *
 *   hidden   [T, H]  bf16 or fp32 (dtype)
 *   weight   [V, H]  same dtype
 *   targets  [T] int32, read only on active rows, must be in [0, V); an
 *            active row whose target is outside sets EAS_ERR_INVALID_ARG in
 *            the status word (that row's outputs are then meaningless)
 *   mask     [T] uint8 loss mask
 *   spans, num_spans, cap : spans as produced by eas_build_active_spans (or
 *            by the caller); they must be sorted, disjoint, inside [0, T)
 *            and cover every active token, else the status word reads
 *            EAS_ERR_INVALID_SPANS and all outputs are zero.
 *   flags    EAS_ROWS_ACTIVE or EAS_ROWS_SPAN
 *   logprob, entropy, lse  [T] fp32 out, overwritten; 0 on inactive rows.
 *            lse may be NULL when no backward follows (forward-only scoring,
 *            e.g. rollout log-probabilities and entropies).
 * Requirements: H % 64 == 0 (bf16) or H % 4 == 0 (fp32); V >= 1; T >= 0.
 */
eas_status eas_lmhead_fwd(const void* hidden, const void* weight,
                          const int32_t* targets, const uint8_t* mask,
                          const int32_t* spans, const int32_t* num_spans, int64_t cap,
                          int64_t T, int64_t H, int64_t V, eas_dtype dtype, uint32_t flags,
                          float* logprob, float* entropy, float* lse,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * Backward: dHidden and dW of L = sum_active g_lp logp + g_H H ("What does
 * this PR do?": skip inactive d-logits tiles, hidden-state gradients through
 * ordered active spans; "How it works": final vocabulary split sized to its
 * live width).
 *
 *   g_logprob, g_entropy [T] fp32 upstream gradients (ignored, even if NaN,
 *            on inactive rows)
 *   hidden, weight, targets, mask, spans, num_spans, cap, flags : as in the
 *            forward (the same spans must be passed)
 *   lse, entropy [T] fp32 : the forward's outputs for the same inputs
 *   vocab_chunk : d-logits columns per chunk (0 = default); the last chunk
 *            covers only the V - (n-1)*vocab_chunk live columns
 *   dhidden  [T, H] out, hidden's dtype, overwritten; exactly 0 on rows whose
 *            mask byte is 0
 *   dweight  [V, H] fp32 out, overwritten (every row written)
 */
eas_status eas_lmhead_bwd(const float* g_logprob, const float* g_entropy,
                          const void* hidden, const void* weight,
                          const int32_t* targets, const uint8_t* mask,
                          const int32_t* spans, const int32_t* num_spans, int64_t cap,
                          const float* lse, const float* entropy,
                          int64_t T, int64_t H, int64_t V, eas_dtype dtype, uint32_t flags,
                          int64_t vocab_chunk,
                          void* dhidden, float* dweight,
                          void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------- e4m3 forward */

/*
 * Per-row e4m3 (FP8, 4 exponent bits, 3 mantissa bits, largest value 448)
 * quantisation of a [R, H] bf16 or fp32 matrix: for each row
 *   amax = max |x|, scale[r] = amax / 448, q = e4m3(x * (448 / amax))
 * rounded to nearest-even and saturated at 448 (an all-zero row gets scale 1).
 * The row's values are then approximately e4m3(q) * scale[r].
 * dst [R, H] uint8 codes, scale [R] fp32 (device).
 */
eas_status eas_quantize_rows_e4m3(const void* src, eas_dtype src_dtype, int64_t R, int64_t H,
                                  uint8_t* dst, float* scale, void* stream);

/*
 * Forward (logprob, entropy, lse) with e4m3 operands: the logit of token t
 * and vocabulary row v is
 *   z = hidden_scale[t] * weight_scale[v] * sum_h e4m3(hidden[t,h]) e4m3(W[v,h])
 * accumulated in fp32 on the tensor cores (tcgen05 kind::f8f6f4); the rest is
 * eas_lmhead_fwd.  Used for forward-only scoring, and before eas_lmhead_bwd_fp8
 * when training on e4m3 logits.
 * Requires H % 128 == 0.  Workspace: eas_lmhead_workspace_size(..., EAS_E4M3, 0).
 */
eas_status eas_lmhead_fwd_fp8(const uint8_t* hidden_e4m3, const float* hidden_scale,
                              const uint8_t* weight_e4m3, const float* weight_scale,
                              const int32_t* targets, const uint8_t* mask,
                              const int32_t* spans, const int32_t* num_spans, int64_t cap,
                              int64_t T, int64_t H, int64_t V, uint32_t flags,
                              float* logprob, float* entropy, float* lse,
                              void* ws, size_t ws_bytes, void* stream);

/*
 * Backward of the e4m3 forward (training with e4m3 logits).  The pages give
 * no FP8 backward; this is the reading implemented here:
 *   - the d-logits are those of the logits the e4m3 forward computes,
 *       z' = hidden_scale[t] * weight_scale[v] * sum_h e4m3(hidden[t,h]) e4m3(W[v,h]),
 *     recomputed on the tensor cores with the same e4m3 operands (kind::f8f6f4),
 *     so they agree with the lse and entropy eas_lmhead_fwd_fp8 returned:
 *       dZ' = g_lp (onehot - p') - g_H p' (z' - lse + H),  p' = exp(z' - lse);
 *   - they are staged in bf16 and projected with the unquantised bf16
 *     operands, as eas_lmhead_bwd does: dHidden = dZ' W, dW = dZ'^T hidden.
 * Each vocabulary chunk is two launches: the e4m3 d-logits, then dW and
 * dHidden.
 *
 *   hidden, weight [T, H] / [V, H] bf16 : the unquantised operands
 *   hidden_e4m3, hidden_scale, weight_e4m3, weight_scale : the same operands
 *            quantised by eas_quantize_rows_e4m3 (as passed to the forward)
 *   lse, entropy [T] fp32 : eas_lmhead_fwd_fp8's outputs for these operands
 * Other arguments and outputs are those of eas_lmhead_bwd (dtype bf16).  The
 * backward packs its own rows: EAS_REUSE_FWD_ROWS is rejected.  Requires
 * H % 128 == 0.  Workspace: eas_lmhead_bwd_fp8_workspace_size(T, H, V,
 * vocab_chunk) bytes.
 */
size_t eas_lmhead_bwd_fp8_workspace_size(int64_t T, int64_t H, int64_t V, int64_t vocab_chunk);

eas_status eas_lmhead_bwd_fp8(const float* g_logprob, const float* g_entropy,
                              const void* hidden, const void* weight,
                              const uint8_t* hidden_e4m3, const float* hidden_scale,
                              const uint8_t* weight_e4m3, const float* weight_scale,
                              const int32_t* targets, const uint8_t* mask,
                              const int32_t* spans, const int32_t* num_spans, int64_t cap,
                              const float* lse, const float* entropy,
                              int64_t T, int64_t H, int64_t V, uint32_t flags,
                              int64_t vocab_chunk, void* dhidden, float* dweight,
                              void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------ vocabulary-parallel path */

/*
 * Vocabulary-parallel (tensor-parallel) use, as in the page's TP4 matrix
 * ("Performance"): W is split by rows into shards [v_lo, v_lo + V_shard),
 * one per GPU, and every GPU holds the same hidden rows.
 *
 *   1. eas_lmhead_fwd_shard on each shard writes per-token statistics
 *      stats[t] = (M, S, U, z) (4 floats, 16-byte aligned, [T][4]) over its
 *      columns, in base-2 units (y = z log2 e):
 *        M = max y, S = sum 2^(y - M), U = sum 2^(y - M) (y - M);
 *      z is the target logit if the target lies in the shard, else 0;
 *      inactive tokens get (0, 0, 0, 0).
 *   2. The shards' statistics are gathered into [n_shards][T][4] (on several
 *      GPUs: an all-gather), and eas_lmhead_combine_shards merges them in
 *      shard order into logprob, entropy and lse (lse may be NULL).
 *   3. eas_lmhead_bwd_shard on each shard, given the global lse and
 *      entropy, writes that shard's dW rows [V_shard, H] and its partial
 *      dHidden, i.e. its columns' contribution; the partials sum to dHidden
 *      (on several GPUs: an all-reduce).
 * Targets are global vocabulary ids.  Other arguments, workspaces and errors
 * are those of eas_lmhead_fwd / eas_lmhead_bwd with V = V_shard.
 */
eas_status eas_lmhead_fwd_shard(const void* hidden, const void* weight_shard, int64_t v_lo,
                                const int32_t* targets, const uint8_t* mask,
                                const int32_t* spans, const int32_t* num_spans, int64_t cap,
                                int64_t T, int64_t H, int64_t V_shard, eas_dtype dtype,
                                uint32_t flags, float* stats, void* ws, size_t ws_bytes,
                                void* stream);

eas_status eas_lmhead_combine_shards(const float* stats, int32_t n_shards, int64_t T,
                                     const uint8_t* mask, float* logprob, float* entropy,
                                     float* lse, void* stream);

eas_status eas_lmhead_bwd_shard(const float* g_logprob, const float* g_entropy,
                                const void* hidden, const void* weight_shard, int64_t v_lo,
                                const int32_t* targets, const uint8_t* mask,
                                const int32_t* spans, const int32_t* num_spans, int64_t cap,
                                const float* lse, const float* entropy,
                                int64_t T, int64_t H, int64_t V_shard, eas_dtype dtype,
                                uint32_t flags, int64_t vocab_chunk,
                                void* dhidden_partial, float* dweight_shard,
                                void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------- allocation-free forward */

/*
 * eas_lmhead_fwd without a workspace argument.  This entry point has no
 * counterpart on the page; it exists for callers that cannot allocate device
 * memory when they run the forward: a host whose pool allocator owns all of
 * the GPU's memory and lends none to libraries, an embedded or real-time host
 * that forbids allocation after start-up, or a plugin interface that hands a
 * library only its input and output buffers.
 *
 * Its scratch is a static device array of EAS_STATIC_SCRATCH_BYTES (64 MiB)
 * compiled into the library; every GPU that loads the library reserves it
 * until the process exits.  Arguments, outputs and results are those of
 * eas_lmhead_fwd; the caller still passes every input and output buffer.
 *   - Problems whose forward needs more scratch than that are rejected with
 *     EAS_ERR_WORKSPACE before anything is launched, and eas_last_error()
 *     gives the bytes needed (eas_lmhead_fwd with a workspace has no limit).
 *     For bf16 the need is about T * (2H + 12 ceil(V/256) + 16) bytes.
 *   - Set-up: the first call in a context looks up the array's device
 *     address there (cudaGetSymbolAddress, with that context current) and
 *     caches it under the context's unique ID.  For most callers that is the
 *     first call on each device, in its primary context; it happens again in
 *     a context the host created and made current through the driver API, and
 *     after cudaDeviceReset (each context holds its own copy of the array).
 *     Make the first call in a context before any stream capture.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call
 *     (leave eas_trace_enable off, since tracing creates CUDA events).
 *   - All calls share the one array, and it keeps what the last call left
 *     there; each call clears what must start at zero.  Calls whose kernels
 *     overlap on the GPU (different streams, or different host threads
 *     without ordering) race on the array and give wrong results: order them.
 *   - The device status word lives in the shared array and cannot be read
 *     back through this entry point, so errors only the device can see go
 *     unreported here: spans that fail validation leave every output zero
 *     (as with eas_lmhead_fwd), and an active row whose target lies outside
 *     [0, V) gets meaningless outputs with no error.  Callers that cannot
 *     vouch for their spans and targets should use eas_lmhead_fwd and
 *     eas_read_device_status.
 */
#define EAS_STATIC_SCRATCH_BYTES (64ull << 20)

eas_status eas_lmhead_fwd_noalloc(const void* hidden, const void* weight,
                                  const int32_t* targets, const uint8_t* mask,
                                  const int32_t* spans, const int32_t* num_spans, int64_t cap,
                                  int64_t T, int64_t H, int64_t V, eas_dtype dtype,
                                  uint32_t flags, float* logprob, float* entropy, float* lse,
                                  void* stream);

/* ------------------------------------------------------------- utilities */

/*
 * Waits for `stream`, then returns the status word the device wrote into
 * workspace `ws` during the last call that used it (EAS_OK if none).  This is
 * the only entry point that synchronises the host (cudaStreamSynchronize on
 * `stream`); every other call only enqueues work.
 */
eas_status eas_read_device_status(const void* ws, void* stream);

/*
 * Failure-detection self-test.  Launches one warp that waits on a pipeline
 * barrier nothing will complete, with the same bounded waits the GEMM kernels
 * use, and lets each run out after budget_cycles SM clocks (1 .. 2^34).  Afterwards
 * eas_read_device_status(ws) must report EAS_ERR_TIMEOUT and the device stays
 * usable.  ws: at least 16 bytes (the status word).  The pipeline waits of the
 * library kernels take their budget from the EAS_WAIT_BUDGET_CYCLES
 * environment variable (default 2^31 clocks, about one second).
 */
eas_status eas_selftest_wait_timeout(int64_t budget_cycles, void* ws, size_t ws_bytes,
                                     void* stream);

/*
 * Per-kernel timing.  eas_trace_enable(1) clears earlier records and makes
 * every later kernel launch of this library record a pair of CUDA events
 * around itself on its stream; eas_trace_enable(0) stops recording.
 * eas_trace_read() waits for the recorded events and writes, for the first
 * min(n, cap) launches, the kernel kind (see eas_kernel_name) and its
 * duration in milliseconds; it returns n, the number of recorded launches.
 * For eager launches only (not inside a CUDA graph capture).  The trace is
 * process-wide: launches from every host thread and device are recorded
 * into the one list, in the order they were issued.
 */
void eas_trace_enable(int32_t on);
int32_t eas_trace_read(int32_t* kinds, float* ms, int32_t cap);
const char* eas_kernel_name(int32_t kind);

/* Thread-local description of the last error returned on this thread. */
const char* eas_last_error(void);

/* Short name of a status code. */
const char* eas_status_string(eas_status s);

/* Version of this library: major * 10000 + minor * 100 + patch. */
int32_t eas_version(void);

#ifdef __cplusplus
}
#endif

#endif  /* EAS_H_ */
