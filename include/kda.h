/*
 * kda.h -- C ABI of libkda.so: chunked prefill of Kimi Delta Attention (KDA)
 * on a GB300 (sm_103a) GPU.
 *
 * The operation is the one the vLLM PR report "[Perf][GLM-5.3-Flash] Use
 * FlashKDA for KDA chunked prefill" (PR #55737) describes for FlashKDA's
 * `get_workspace_size` / `fwd` pair (Implementation breakdown, items 2 and
 * 3, and the "FlashKDA prefill call wrapper" listing), with the bf16 / fp32
 * state of "[KDA] Update flashKDA to support bf16 checkpoint state"
 * (PR #56485, Implementation breakdown item 2) and the value-dimension
 * split of "[Kimi-K3][Perf] Update FlashKDA for automatic K2 V-split"
 * (PR #52458, Features & motivation).  Per (sequence n, head h), token by
 * token, with S the 128 x 128 state (row = key channel, column = value
 * channel):
 *
 *   qh = scale * q / |q|      kh = k / |k|          (l2norm, eps 1e-6)
 *   a  = lower_bound * sigmoid(exp(A_log[h]) * (g + dt_bias[h, :]))
 *   S  = diag(exp(a)) S;      b = sigmoid(beta)
 *   S  = S + kh * (b * (v - S^T kh))^T;   out = S^T qh
 *
 * computed chunk by chunk (64 tokens, WY/UT form) on tcgen05 tensor cores.
 *
 * Conventions for every call below:
 *   - All tensor pointers are DEVICE pointers of the current CUDA device,
 *     owned by the caller.  The library allocates no device memory, takes
 *     no ownership and never synchronises inside kda_chunk_prefill_fwd*:
 *     the work is enqueued on `stream` and returns.
 *   - The workspace must be zero-filled once before its first use (the
 *     device status word starts at 0; kda_last_device_status() leaves it
 *     zero again).
 *   - Dense row-major layouts; T = total_tokens, H = heads, N = num_seqs,
 *     D = 128 (the only supported head dim):
 *       q, k, v, g      bf16  [T, H, D]   (g: raw gate logits)
 *       beta            bf16  [T, H]      (raw beta logits)
 *       A_log           fp32  [H]         dt_bias  fp32 [H, D]
 *       initial_state   [N, H, D, D] in state_dtype, or NULL for zeros
 *       final_state     [N, H, D, D] in state_dtype (may equal
 *                       initial_state: the update is then in place)
 *       cu_seqlens      int32 [N + 1], 0 = cu[0] <= cu[1] <= ... <= cu[N] <= T
 *       out             bf16  [T, H, D]; rows of tokens past cu[N] are not
 *                       written.  out must not overlap any input.
 *   - q, k, v, g, out, initial_state, final_state and workspace must be
 *     16-byte aligned; beta 2-byte; A_log and dt_bias 16-byte.
 *   - lower_bound must lie in [KDA_MIN_LOWER_BOUND, 0] = [-5, 0]: the gate
 *     is a log decay in (lower_bound, 0].  The kernels split each decay
 *     factor of a 64-token chunk into a row and a column factor anchored
 *     inside 32-token blocks; at saturated gates these reach
 *     2^(+-16 |lower_bound| log2 e), and past -5 the column factors of the
 *     cross-block products would leave the fp32/bf16 normal range for the
 *     smaller q/k entries.
 *   - Return value: KDA_OK (0) or a negative KDA_ERR_* code; nothing is
 *     enqueued when an error is returned.  Errors found on the device
 *     (malformed cu_seqlens, a bounded wait that gave up) are recorded in
 *     the workspace and read back with kda_last_device_status().
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same handle as cudaStream_t (NULL = the legacy default stream). */
typedef struct CUstream_st* kda_stream_t;

#define KDA_HEAD_DIM 128
#define KDA_MIN_LOWER_BOUND (-5.0f)

/* state storage dtypes (PR #56485: fp32 or bf16 checkpoint state) */
#define KDA_STATE_F32 0
#define KDA_STATE_BF16 1

/* status codes */
#define KDA_OK 0
#define KDA_ERR_INVALID_ARG (-1)         /* null pointer, bad size or dtype   */
#define KDA_ERR_UNSUPPORTED_DEVICE (-2)  /* current device is not sm_103      */
#define KDA_ERR_WORKSPACE_TOO_SMALL (-3) /* workspace_bytes below the query   */
#define KDA_ERR_UNSAFE_LOWER_BOUND (-4)  /* lower_bound outside [-5, 0]       */
#define KDA_ERR_MISALIGNED (-5)          /* a pointer breaks its alignment    */
#define KDA_ERR_LAUNCH_FAILED (-6)       /* the kernel launch was rejected    */
#define KDA_ERR_DEVICE_TIMEOUT (-7)      /* (device) a bounded wait gave up   */
#define KDA_ERR_BAD_CU_SEQLENS (-8)      /* (device) cu_seqlens not monotone
                                            or past total_tokens            */
#define KDA_ERR_CUDA (-9)                /* a CUDA runtime call failed        */
#define KDA_ERR_BAD_OUT_INDEX (-10)      /* (device) an out_index entry lies
                                            outside [0, out_rows)            */

/* kernel selectors for kda_chunk_prefill_fwd_ex */
#define KDA_KERNEL_AUTO 0  /* SPLIT_STREAMED when N * heads * P <= SMs / 2 for
                              P = 8, 4 or 2, or N * heads <= 3 SMs / 8 for
                              P = 1, the sequences average 2048 tokens
                              or more and the workspace holds the records
                              and claim words; else SPLIT when the value
                              split triggers and the workspace holds its
                              records; else TC_HELPERS
                              when N * heads <= min(SMs - 8, 5 SMs / 8),
                              N <= 128, the sequences average 4 or more
                              chunks and the workspace holds the records;
                              else PIPE (TC when the caller fixed P > 1)     */
#define KDA_KERNEL_TC 1    /* fused tcgen05 + TMA chunk kernel, C = 64: one CTA
                              per (sequence, head[, value slice])            */
#define KDA_KERNEL_REF 2   /* plain-CUDA-core chunk kernel (GPU parity aid)    */
#define KDA_KERNEL_SPLIT 3 /* the K1/K2 structure of PR #52458: a chunk-parallel
                              k-side kernel writes per-(chunk, head) records to
                              the workspace, then one chain CTA per (sequence,
                              head, value slice of 128 / P columns); P = 1 and
                              P = 2 run the chain on tcgen05 with the state
                              (slice) in TMEM, P = 4 and 8 on warp-level
                              MMAs with the slice in registers             */
#define KDA_KERNEL_TC_HELPERS 4 /* TC (P = 1) plus k-side helper CTAs on the SMs
                              it leaves free: they write records for chunks
                              taken from the end of each sequence, which the
                              fused CTAs then read instead of computing them;
                              needs N * heads < SM count and the records'
                              workspace                                      */
#define KDA_KERNEL_PIPE 5  /* fused warp-specialised tcgen05 + TMA kernel, C = 64:
                              one CTA per (sequence, head) whose k-side warps
                              build chunk c+1's operands while its chain warps
                              run chunk c; no value split (vsplit -1 or 1),
                              needs only the 256-byte workspace               */
#define KDA_KERNEL_SPLIT_STREAMED 6 /* SPLIT (any P) with the chain kernel
                              launched beside the k-side kernel (programmatic
                              dependent launch): the chain CTAs take
                              N * heads * P SMs, the k-side CTAs the others,
                              and each chain CTA copies a record as soon as
                              its claim word says it is written (bounded
                              wait).  Needs 2 * N * heads * P <= SM count
                              (P > 1) or 8 * N * heads <= 3 SM count (P = 1),
                              N <= 128 and the workspace of TC_HELPERS        */

/*
 * Bytes of device workspace a call needs for up to `total_tokens` tokens,
 * `heads` heads and `max_seqs` sequences.  Counterpart of FlashKDA's
 * get_workspace_size(max_num_batched_tokens, local_num_heads,
 * max_num_seqs) (PR #55737, Implementation breakdown item 2), where the
 * caller sizes a uint8 buffer once and reuses it every step.
 *
 * The workspace starts with the device status word (256 bytes: all the
 * fused kernel needs).  When some batch of up to max_seqs sequences would
 * take the value split on the current device (2 * heads * N <= SM count;
 * 152 SMs are assumed when no device answers) or take k-side helpers
 * (heads * N <= min(SM count - 8, 5 SM count / 8)), it also holds the records of
 * those paths: a 1 KB header, then 66,560 bytes per (chunk slot, head),
 * with ceil(total_tokens / 64) + N slots for the largest such N -- about
 * 1 KB per token-head -- and, for the helpers and the streamed split path
 * (whose batches lie inside the helpers' band), one int32 claim word per
 * (chunk slot, head).  A smaller workspace (at least 256 bytes) is
 * accepted; KDA_KERNEL_AUTO then runs the fused kernel alone.  Always a
 * multiple of 16; 0 for negative arguments.  A zero-filled workspace can
 * serve any number of calls, of any path: the streamed split path leaves
 * its header counters and claim words at zero when a call ends (after a
 * device timeout too), the helpers reset theirs when a call starts, and
 * the other paths use neither.
 */
size_t kda_workspace_size(int64_t total_tokens, int32_t heads, int32_t max_seqs);

/*
 * Chunked KDA prefill over N packed sequences (PR #55737, Implementation
 * breakdown item 3; argument order of FlashKDA's fwd, with the sizes a C
 * caller must pass explicitly appended).  `scale` multiplies the
 * normalised q (callers pass head_dim ** -0.5).  `state_dtype` is
 * KDA_STATE_F32 or KDA_STATE_BF16 and applies to both states; a bf16 final
 * state is rounded to nearest even.  `workspace` must hold at least
 * kda_workspace_size(total_tokens, heads, num_seqs) bytes
 * (`workspace_bytes`) for the split path, else the fused kernel runs; below
 * 256 bytes the call returns KDA_ERR_WORKSPACE_TOO_SMALL.  Concurrent calls
 * on different streams need different workspaces.  The value dimension is
 * split across CTAs automatically when 2 * heads * num_seqs <= SM count
 * (PR #52458); the split does not change the result beyond rounding.
 */
int kda_chunk_prefill_fwd(const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const float* A_log, const float* dt_bias,
                          float lower_bound, float scale, const void* initial_state,
                          const int32_t* cu_seqlens, void* out, void* final_state,
                          int state_dtype, void* workspace, kda_stream_t stream,
                          int64_t total_tokens, int32_t num_seqs, int32_t heads,
                          size_t workspace_bytes);

/*
 * As kda_chunk_prefill_fwd, with two overrides for tests and sweeps:
 * `vsplit` -1 = automatic, or a forced split factor in {1, 2, 4, 8};
 * `kernel` one of KDA_KERNEL_*.  Other values give KDA_ERR_INVALID_ARG.
 * KDA_KERNEL_SPLIT needs room for its records: 1024 + 66,560 bytes per
 * (chunk slot, head) with ceil(total_tokens / 64) + num_seqs slots, else
 * KDA_ERR_WORKSPACE_TOO_SMALL.  KDA_KERNEL_TC_HELPERS needs the same plus
 * 4 bytes per (chunk slot, head), vsplit -1 or 1 (else
 * KDA_ERR_INVALID_ARG), num_seqs * heads below the SM count and num_seqs
 * <= 128 (else KDA_ERR_INVALID_ARG).  KDA_KERNEL_SPLIT_STREAMED needs that
 * workspace too, vsplit -1 (P = 8, else 4, else 2, else 1) or a fixed P,
 * 2 * num_seqs * heads * P at most the SM count (P > 1; for P = 1,
 * 8 * num_seqs * heads at most 3 SM count) and num_seqs <= 128 (else
 * KDA_ERR_INVALID_ARG).
 */
int kda_chunk_prefill_fwd_ex(const void* q, const void* k, const void* v, const void* g,
                             const void* beta, const float* A_log, const float* dt_bias,
                             float lower_bound, float scale, const void* initial_state,
                             const int32_t* cu_seqlens, void* out, void* final_state,
                             int state_dtype, void* workspace, kda_stream_t stream,
                             int64_t total_tokens, int32_t num_seqs, int32_t heads,
                             size_t workspace_bytes, int vsplit, int kernel);

/*
 * As kda_chunk_prefill_fwd_ex, for inputs that are views rather than dense
 * tensors -- for instance q, k, v and g as slices of one fused projection
 * output [T, 4 * H * 128], so that no copy to a dense layout is needed (the
 * vLLM PR report "[Perf][GLM-5.3-Flash] Use FlashKDA for KDA chunked
 * prefill", PR #55737, measures such copies at about 115 us per layer at
 * 16k tokens: Risks & impact and the "FlashKDA prefill call wrapper"
 * listing).  Each stride is the distance in elements between consecutive
 * tokens: q element (t, h, d) is read at q[t * q_stride + h * 128 + d] (the
 * same for k, v, g) and beta (t, h) at beta[t * beta_stride + h].  The head
 * and channel dimensions stay dense; out is dense as before.  q/k/v/g
 * strides must be at least heads * 128 and a multiple of 8 (16-byte rows for
 * the TMA loads), beta_stride at least heads; otherwise KDA_ERR_INVALID_ARG
 * or KDA_ERR_MISALIGNED.
 */
int kda_chunk_prefill_fwd_strided(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const float* A_log, const float* dt_bias,
                                  float lower_bound, float scale, const void* initial_state,
                                  const int32_t* cu_seqlens, void* out, void* final_state,
                                  int state_dtype, void* workspace, kda_stream_t stream,
                                  int64_t total_tokens, int32_t num_seqs, int32_t heads,
                                  size_t workspace_bytes, int64_t q_stride, int64_t k_stride,
                                  int64_t v_stride, int64_t g_stride, int64_t beta_stride,
                                  int vsplit, int kernel);

/*
 * As kda_chunk_prefill_fwd_strided, writing each token's output row through a
 * row map: the H x 128 outputs of token t (0 <= t < cu_seqlens[N]) go to
 * out[out_index[t]], `out` being bf16 [out_rows, H, 128].  This is the
 * mixed step of the vLLM PR report "[Perf][GLM-5.3-Flash] Use FlashKDA for
 * KDA chunked prefill" (PR #55737, Implementation breakdown item 4): there
 * the prefill of the non-speculative tokens writes a workspace buffer that
 * index_copy_ then scatters into the layer output by non_spec_token_indx;
 * with the map the kernels write the layer output directly.  out_index is
 * device int32 [total_tokens] (entries past cu_seqlens[N] are not read),
 * 4-byte aligned; rows not named by the map are left untouched; two tokens
 * mapped to one row leave one of them there.  An entry outside
 * [0, out_rows) is not written and is recorded as KDA_ERR_BAD_OUT_INDEX
 * (kda_last_device_status).  A NULL out_index or a negative out_rows gives
 * KDA_ERR_INVALID_ARG.
 */
int kda_chunk_prefill_fwd_scatter(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const float* A_log, const float* dt_bias,
                                  float lower_bound, float scale, const void* initial_state,
                                  const int32_t* cu_seqlens, void* out, void* final_state,
                                  int state_dtype, void* workspace, kda_stream_t stream,
                                  int64_t total_tokens, int32_t num_seqs, int32_t heads,
                                  size_t workspace_bytes, int64_t q_stride, int64_t k_stride,
                                  int64_t v_stride, int64_t g_stride, int64_t beta_stride,
                                  const int32_t* out_index, int64_t out_rows, int vsplit,
                                  int kernel);

/*
 * Token-by-token KDA for decode and speculative-verify steps, where each
 * sequence brings a few tokens (1..k): the recurrent form of the same
 * operation, on the same state layout and dtypes, so a sequence can switch
 * between prefill and decode calls freely.  The pages route speculative
 * tokens through this recurrent form so that a rejected draft can be rolled
 * back via num_accepted_tokens (PR #55737, Discussion and Features &
 * motivation).  Arguments are those of kda_chunk_prefill_fwd (dense
 * inputs), plus `token_states`: NULL, or [T, H, 128, 128] in state_dtype,
 * which receives the state after every token -- a caller that accepts the
 * first m draft tokens of a sequence continues from the entry of its m-th
 * token.  The workspace needs only the 256 bytes of status words.  One CTA
 * per (sequence, head, 32 value columns); the time is the state's read and
 * write (plus the token states, if asked for).
 */
int kda_recurrent_fwd(const void* q, const void* k, const void* v, const void* g,
                      const void* beta, const float* A_log, const float* dt_bias,
                      float lower_bound, float scale, const void* initial_state,
                      const int32_t* cu_seqlens, void* out, void* final_state, int state_dtype,
                      void* token_states, void* workspace, kda_stream_t stream,
                      int64_t total_tokens, int32_t num_seqs, int32_t heads,
                      size_t workspace_bytes);

/*
 * kda_recurrent_fwd writing token t's output row to out[out_index[t]] (out
 * being [out_rows, H, 128]), with the conventions of
 * kda_chunk_prefill_fwd_scatter: in a mixed step the speculative tokens
 * (spec_token_indx in the pages' layer) and the prefill tokens write
 * disjoint rows of one layer output.
 */
int kda_recurrent_fwd_scatter(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const float* A_log, const float* dt_bias,
                              float lower_bound, float scale, const void* initial_state,
                              const int32_t* cu_seqlens, void* out, void* final_state,
                              int state_dtype, void* token_states, void* workspace,
                              kda_stream_t stream, int64_t total_tokens, int32_t num_seqs,
                              int32_t heads, size_t workspace_bytes, const int32_t* out_index,
                              int64_t out_rows);

/*
 * The low-M projections in front of KDA, for decode and small prefill steps: two
 * "skinny" GEMMs with bf16 operands, fp32 accumulation and bf16 results,
 *     y = x w_ab^T                 x [m, k], w_ab [n_ab, k]   ->  y [m, n_ab]
 *     z = y[:, :r] w_b^T           w_b [n_b, r]               ->  z [m, n_b]
 * (the second reads y as the first wrote it, in bf16).  These are the shapes of the
 * Kimi-K3 low-M KDA projection overlap in the vLLM PR report "[Bugfix] Fix Kimi-K3 KDA
 * projection overlap compile on Hopper" (Implementation breakdown; its skinny-GEMM test
 * uses k = 7168, n_ab = 144, r = 128, n_b = 1536 and m = 2, 8, 14).  Row strides are in
 * elements: x[i, j] at x[i * ldx + j], likewise y and z; w_ab and w_b are dense.
 * Requirements (else KDA_ERR_INVALID_ARG): 1 <= m <= 16; k a positive multiple of 512;
 * n_ab and n_b positive multiples of 16; r a multiple of 16 in [16, min(n_ab, 512)];
 * ldx >= k, ldy >= n_ab and ldz >= n_b.  Alignment (else KDA_ERR_MISALIGNED): x, w_ab,
 * w_b, y 16 bytes, z 4 bytes, ldx and ldy multiples of 8, ldz even.  y and z must not
 * overlap x or the weights.  The workspace holds fp32 partial sums and arrival counters:
 * kda_skinny_proj_workspace_size(k, n_ab) bytes, zero-filled once before its first use
 * (the kernels leave the counters at zero).  Asynchronous on `stream`; the second GEMM is
 * launched as a programmatic dependent of the first.
 */
size_t kda_skinny_proj_workspace_size(int32_t k, int32_t n_ab);
int kda_skinny_proj(const void* x, int64_t ldx, const void* w_ab, const void* w_b, void* y,
                    int64_t ldy, void* z, int64_t ldz, int32_t m, int32_t k, int32_t n_ab,
                    int32_t r, int32_t n_b, void* workspace, size_t workspace_bytes,
                    kda_stream_t stream);

/*
 * The value-dimension split factor the automatic path uses for a batch of
 * `num_seqs` sequences and `heads` heads on a GPU with `sm_count` SMs.
 * The trigger is PR #52458's: split only when 2 * heads * num_seqs <=
 * sm_count (else 1).  When it triggers, the factor is the largest P in
 * {2, 4, 8} with P * heads * num_seqs <= sm_count (P > 2 extends the
 * pages' split).  Host logic only; returns 1 for non-positive arguments.
 */
int kda_choose_vsplit(int32_t num_seqs, int32_t heads, int32_t sm_count);

/* Static text for a status code (never NULL). */
const char* kda_status_string(int status);

/*
 * Reads and clears the device status word that kernels enqueued with this
 * `workspace` leave behind.  Synchronises `stream` first (the only call of
 * this library that does).  Returns KDA_OK, the recorded KDA_ERR_* code,
 * or KDA_ERR_CUDA if the copy failed.
 */
int kda_last_device_status(void* workspace, kda_stream_t stream);

/* KDA_OK when `device` is an sm_103 GPU this library can run on, else
 * KDA_ERR_UNSUPPORTED_DEVICE (or KDA_ERR_CUDA when no device answers). */
int kda_device_check(int device);

/*
 * The path a kda_chunk_prefill_fwd_ex call with these sizes, workspace size
 * and selectors would take on the current device, without enqueuing
 * anything: *kernel_out gets KDA_KERNEL_TC, KDA_KERNEL_TC_HELPERS,
 * KDA_KERNEL_SPLIT, KDA_KERNEL_SPLIT_STREAMED, KDA_KERNEL_PIPE or
 * KDA_KERNEL_REF (AUTO resolved), *vsplit_out the value split factor P and
 * *launches_out the number of kernels the call enqueues (0, 1 or 2); any
 * output pointer may be NULL.  Returns the code such a call would return
 * for its sizes, selectors and workspace size (pointer checks aside), or
 * KDA_ERR_UNSUPPORTED_DEVICE / KDA_ERR_CUDA.  The pages have no
 * counterpart of this query; it lets callers and benchmarks see which
 * kernels ran.
 */
int kda_plan(int64_t total_tokens, int32_t num_seqs, int32_t heads, size_t workspace_bytes,
             int vsplit, int kernel, int* kernel_out, int* vsplit_out, int* launches_out);

/*
 * kda_plan for a device with `sm_count` multiprocessors, without touching any
 * device: the same checks of sizes and selectors, the same resolution of
 * AUTO, value split and launch count.  For planning on a host that has no
 * GPU (and for testing the dispatch there).  sm_count <= 0 gives
 * KDA_ERR_INVALID_ARG.  Output pointers may be NULL.
 */
int kda_plan_for(int64_t total_tokens, int32_t num_seqs, int32_t heads, size_t workspace_bytes,
                 int vsplit, int kernel, int32_t sm_count, int* kernel_out, int* vsplit_out,
                 int* launches_out);

/*
 * Test hook, for the failure-detection test only: while `on` is nonzero,
 * calls that take KDA_KERNEL_TC_HELPERS have the helpers leave one claimed
 * record unpublished (the last chunk of the longest sequence's head 0), so
 * the bounded device wait of the fused CTA that needs it runs out and the
 * call records KDA_ERR_DEVICE_TIMEOUT; calls that take
 * KDA_KERNEL_SPLIT_STREAMED leave the record of that sequence's first chunk
 * of head 0 unpublished, with the same outcome for its chain CTAs.  Off at load.  Read once per call
 * from an atomic flag (no environment lookup).  The pages have no
 * counterpart.
 */
void kda_test_drop_one_record(int on);

/*
 * kda_chunk_prefill_fwd for callers that cannot allocate device memory and
 * so cannot pass a workspace: for instance a plugin inside a host framework
 * that owns all device memory, or a hot loop where a cudaMalloc (which may
 * synchronise the device) is not allowed.  The pages have no counterpart of
 * this entry point.
 *
 * Arguments, layouts and ownership are those of kda_chunk_prefill_fwd
 * without the workspace; the warp-specialised tcgen05 kernel runs
 * (KDA_KERNEL_PIPE, P = 1: AUTO's choice whenever the workspace holds no
 * per-chunk records; never the split path, whose records need a real
 * workspace).
 * The scratch it needs (the 16-byte device status word) lives in a 256-byte
 * file-scope device array of this library, which every GPU that loads the
 * library holds until exit.  The library allocates nothing: no cudaMalloc,
 * cudaFree or allocating library call on any path of this function.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *     The address is kept for the life of the process: after a
 *     cudaDeviceReset on that device, do not call this entry point again.
 *   - Every call shares the array.  Each call clears the status word on
 *     `stream` before its kernel (this clearing may be enqueued even when
 *     the call then returns an argument error).  Calls that overlap on the
 *     GPU race on the array.  Device-side errors land in the array and are
 *     not reported back here; use kda_chunk_prefill_fwd with a workspace to
 *     read them.
 *   - Returns the codes of kda_chunk_prefill_fwd (the kernel needs only
 *     the 256 bytes the array holds).
 */
int kda_chunk_prefill_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                  const void* beta, const float* A_log, const float* dt_bias,
                                  float lower_bound, float scale, const void* initial_state,
                                  const int32_t* cu_seqlens, void* out, void* final_state,
                                  int state_dtype, kda_stream_t stream, int64_t total_tokens,
                                  int32_t num_seqs, int32_t heads);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
