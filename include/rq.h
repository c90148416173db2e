/*
 * rq.h -- C ABI of the GB300 (sm_103a) per-frame decode step of a Moshi-style
 * RQ-Transformer.
 *
 * What one frame computes ("inferencelayer 0.2.4 -- src/moshi_lm.rs", module doc and
 * `MoshiLm::step_ext`): for each of B independent sessions,
 *   1. the 8 user-audio codes are written into the 17-stream, 3-slot delayed-token
 *      ring at (offset + delay) % 3;
 *   2. the 17 model inputs are gathered at offset % 3, INITIAL tokens (text_card for
 *      the text stream, audio_card for audio) while offset <= delay;
 *   3. their embeddings are summed (16 audio tables, then the text table; code -1
 *      adds nothing, any other code adds row max(code, 0));
 *   4. the temporal decoder runs at position `offset` (pre-norm RMSNorm, fused qkv,
 *      interleaved-pair rotary embedding, K/V window of `context` positions, SiLU-gated
 *      FFN), then out_norm;
 *   5. the text head's first-wins argmax picks the text token;
 *   6. the depformer runs its 8 codebook steps (fresh per-frame K/V, step-specific
 *      weights, shared norms, no rotary embedding), each ending in an argmax;
 *   7. offset advances and the 9 generated tokens are written at offset % 3;
 *   8. once offset > 1 the delay-realigned [text, audio0..7] is read at
 *      (offset - 1 + delay) % 3.
 * Streams: 0 text, 1..8 generated audio codebooks, 9..16 user codebooks; delays
 * [0 | 0,1,1,1,1,1,1,1 | 0,1,1,1,1,1,1,1]; the ring starts UNGENERATED (-2).
 *
 * Ownership: weights belong to the caller; they must stay valid and unchanged until
 * rq_destroy and are never copied or freed here.  The handle owns the ring, the
 * offsets, the K/V caches, all scratch, the captured CUDA graph and the status word.
 *
 * Streams: every call enqueues on the stream given to rq_create (NULL = the legacy
 * default stream).  Calls with host outputs synchronize that stream before return.
 *
 * Errors: argument and token validation happens before anything is enqueued, so a
 * validation error leaves every session unchanged.  A CUDA error or a device-side
 * timeout poisons the handle: later calls return RQ_ERR_POISONED until
 * rq_reset(h, -1) or rq_destroy.  rq_last_error gives a one-line reason.
 *
 * Thread safety: one handle must not be used from two threads at once.
 */
#ifndef RQ_H_
#define RQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RQ_ABI_VERSION 1
#define RQ_N_STREAMS 17
#define RQ_N_Q 8 /* generated audio codebooks per frame */

typedef enum {
  RQ_OK = 0,
  RQ_ERR_ARG = 1,         /* bad pointer, size, shape or alignment */
  RQ_ERR_TOKEN = 2,       /* a user or forced token outside its range */
  RQ_ERR_CUDA = 3,        /* a CUDA runtime error (handle poisoned) */
  RQ_ERR_OOM = 4,         /* device or pinned-host allocation failed */
  RQ_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up (handle poisoned) */
  RQ_ERR_UNSUPPORTED = 6, /* shape or dtype this library does not implement */
  RQ_ERR_POISONED = 7     /* an earlier CUDA error or timeout; rq_reset(h, -1) */
} rq_status;

typedef enum { RQ_F32 = 0, RQ_BF16 = 1, RQ_Q8 = 2, RQ_Q4 = 3 } rq_dtype;

/* Model shape.  Defaults of the Moshi-7B shape ("moshi_lm.rs", consts DIM..DHIDDEN,
 * CARD, TEXT_CARD, RMS_EPS) in brackets. */
typedef struct {
  int32_t batch;      /* B independent sessions [1] */
  int32_t dim;        /* temporal model width D [4096] = heads * head_dim */
  int32_t layers;     /* temporal layers L [32] */
  int32_t heads;      /* [32] */
  int32_t head_dim;   /* [128]; must be 32, 64 or 128 */
  int32_t hidden;     /* gated-FFN hidden F [11264] */
  int32_t context;    /* K/V window C [3000] */
  int32_t text_card;  /* V [32000]; text tables have V+1 rows, V = INITIAL */
  int32_t audio_card; /* A [2048]; audio input tables have A+1 rows, A = INITIAL */
  int32_t ddim;       /* depformer width DD [1024] = dheads * dhead_dim */
  int32_t dlayers;    /* DL [6] */
  int32_t dheads;     /* [16] */
  int32_t dhead_dim;  /* [64]; must be 32, 64 or 128 */
  int32_t dhidden;    /* DF [2816] */
  int32_t weight_dtype; /* rq_dtype of every matrix and table [RQ_BF16]; with RQ_Q8 or
                           RQ_Q4 the matrices are in that weight band (rq_quantize) and the
                           tables are bf16; bands run under RQ_SCHEDULE_GRAPH and need dim,
                           hidden, ddim, dhidden multiples of 128 */
  int32_t kv_dtype;     /* rq_dtype of the temporal K/V cache [RQ_BF16] */
  float rms_eps;        /* [1e-8], inside the mean */
  float rope_theta;     /* [10000] */
  int32_t schedule;     /* RQ_SCHEDULE_*: how a frame is launched [RQ_SCHEDULE_AUTO] */
} rq_config;

/* Frame schedules.
 *   PERSISTENT  batch 1; f32 or bf16 weights with K/V of the same type, or a weight band
 *               with bf16 K/V.  All linears and attentions of a frame run as cooperative
 *               kernels: two launches per frame, the temporal stack, text head and
 *               depformer input projections at two CTAs per SM with grid barriers between
 *               dependent ops, then the depformer at one CTA per SM, whose ops exchange
 *               tagged 64-bit words (value and producing op) instead of meeting at
 *               barriers.  While the window is longer
 *               than 1350 positions the handle replays the GRAPH frame instead (its
 *               attention kernel then streams K/V faster).
 *   GRAPH       one streaming-GEMV kernel per op inside a CUDA graph.
 *   TENSOR      batch <= 64, bf16 weights, dim, hidden, ddim and dhidden multiples of 64:
 *               every linear as one tcgen05 tensor-core GEMM over all sessions (padded to
 *               a multiple of 16), the normalised f32 activations split into two bf16
 *               operand parts (16 significant bits), inside a CUDA graph.
 * AUTO picks PERSISTENT at batch 1 when it applies (not for weight bands: GRAPH runs them
 * faster), TENSOR at batch >= 2 when it applies (it streams every weight once per frame,
 * where GRAPH streams it once per session), else GRAPH.  Results agree within the parity
 * tolerance. */
enum {
  RQ_SCHEDULE_AUTO = 0,
  RQ_SCHEDULE_GRAPH = 1,
  RQ_SCHEDULE_PERSISTENT = 2,
  RQ_SCHEDULE_TENSOR = 3
};

/* Device pointers to the weights, row-major, matrices [out][in] ("moshi_lm.rs",
 * structs TemporalLayer, DepLayer, MoshiLm and `load_band`).  Matrices and tables are
 * in weight_dtype; the RMSNorm alphas are always f32.  Every pointer must be 16-byte
 * aligned.  Stacked arrays hold one block per layer / step / table, in this order:
 *   emb          [16][A+1][D]      audio input tables, stream 1+k uses table k
 *   text_emb     [V+1][D]
 *   norm1, norm2 [L][D]            f32 alphas
 *   in_proj      [L][3D][D]        rows: q, then k, then v
 *   out_proj     [L][D][D]
 *   gate_in      [L][2F][D]        rows 0..F-1 the SiLU half, F..2F-1 the multiplier
 *   gate_out     [L][D][F]
 *   out_norm     [D]               f32
 *   text_linear  [V][D]
 *   dep_in       [8][DD][D]
 *   dep_text_emb [V+1][DD]         conditions depformer step 0 on the text token
 *   dep_emb      [7][A+1][DD]      step cb >= 1 on audio token cb-1
 *   dnorm1, dnorm2 [DL][DD]        f32 alphas, shared by the 8 steps
 *   d_in_proj    [DL][8][3DD][DD]
 *   d_out_proj   [DL][8][DD][DD]
 *   d_gate_in    [DL][8][2DF][DD]
 *   d_gate_out   [DL][8][DD][DF]
 *   linears      [8][A][DD]        per-codebook output heads */
typedef struct {
  const void *emb, *text_emb;
  const float *norm1;
  const void *in_proj, *out_proj;
  const float *norm2;
  const void *gate_in, *gate_out;
  const float *out_norm;
  const void *text_linear;
  const void *dep_in, *dep_text_emb, *dep_emb;
  const float *dnorm1, *dnorm2;
  const void *d_in_proj, *d_out_proj, *d_gate_in, *d_gate_out;
  const void *linears;
} rq_weights;

typedef struct rq_handle rq_handle;

/* Create a decoder for cfg->batch sessions on the current CUDA device, all sessions
 * fresh (ring UNGENERATED, offset 0, empty K/V), as "moshi_lm.rs", `MoshiLm::state`
 * makes one session.  `cuda_stream` is a cudaStream_t
 * (may be NULL).  Allocates every device buffer and captures the frame as a CUDA
 * graph.  On failure *out is NULL and nothing is leaked. */
rq_status rq_create(const rq_config *cfg, const rq_weights *w, void *cuda_stream,
                    rq_handle **out);

/* Free every resource of the handle (after synchronizing its stream).  NULL is a
 * no-op. */
void rq_destroy(rq_handle *h);

/* Return session `session` (or every session, -1) to the fresh state of
 * "moshi_lm.rs", `MoshiLm::state` (ring UNGENERATED, offset 0, empty K/V window).  K/V
 * memory is not cleared: positions past the offset are never read.  rq_reset(h, -1) also
 * clears a poisoned handle. */
rq_status rq_reset(rq_handle *h, int32_t session);

/* One frame for every session ("moshi_lm.rs", `MoshiLm::step`).
 *   user_tokens  host [B][8]  codes in [-1, audio_card]; -1 = no code (embeds to
 *                zero); anything else -> RQ_ERR_TOKEN before any state changes.
 *   out_tokens   host [B][9]  the delay-realigned [text, audio0..7] (meaningful only
 *                where has_output is 1).
 *   has_output   host [B]     0 until that session's offset exceeds 1, then 1.
 * Synchronizes the stream. */
rq_status rq_step(rq_handle *h, const int32_t *user_tokens, int32_t *out_tokens,
                  uint8_t *has_output);

/* Teacher-forced frame: computes exactly as rq_step but conditions the depformer on
 * `forced` and writes `forced` into the ring in place of its own tokens
 * ("moshi_lm.rs", `MoshiState::force_generated`; "rlx_lm.rs",
 * `depformer_forced_logits_rlx`).
 *   forced      host [B][9]  [text, audio0..7]: text in [0, text_card), audio in
 *               [0, audio_card).
 *   own_tokens  host [B][9]  the frame's own argmax tokens [text, audio0..7].
 *   out_tokens, has_output   as rq_step (realigned from the forced ring). */
rq_status rq_step_forced(rq_handle *h, const int32_t *user_tokens,
                         const int32_t *forced, int32_t *own_tokens,
                         int32_t *out_tokens, uint8_t *has_output);

/* Enqueue one frame whose inputs and outputs stay on the device; no host
 * synchronization and no validation of the token values (the caller guarantees
 * [-1, audio_card]).
 *   d_user        device [B][8]  int32
 *   d_out_tokens  device [B][9]  int32, realigned output
 *   d_has_output  device [B]     uint8
 * Either output pointer may be NULL.  Errors of the frame show up at the next
 * rq_sync. */
rq_status rq_step_device(rq_handle *h, const int32_t *d_user, int32_t *d_out_tokens,
                         uint8_t *d_has_output);

/* Synchronize the handle's stream and read the device status word. */
rq_status rq_sync(rq_handle *h);

/* Debug / parity reads of the last frame (synchronize the stream), the logits fields of
 * "moshi_lm.rs", `StepTrace`:
 *   text  host [B][V] text-head logits;  audio host [B][8][A] depformer logits.
 * Either pointer may be NULL. */
rq_status rq_get_logits(rq_handle *h, float *text, float *audio);

/* The last frame's embedding sum and post-out_norm hidden ("moshi_lm.rs",
 * `StepTrace.emb_sum`, `.transformer_out`), host [B][D] each; either may be NULL. */
rq_status rq_get_trace(rq_handle *h, float *emb_sum, float *transformer_out);

/* The delayed-token ring cache (host [B][17][3], stream-major, slot = step % 3) and the
 * offsets (host [B]) of "moshi_lm.rs", `MoshiState` (`cache`, `offset`); either may be
 * NULL. */
rq_status rq_get_ring(rq_handle *h, int32_t *ring, int32_t *offsets);

/* Pre-fill session `session`: temporal K/V positions 0..n_pos-1 of every layer take
 * k, v ([L][n_pos][D] in kv_dtype, keys already rotated; host or device memory),
 * the offset becomes n_pos and the ring is left as it is ("moshi_lm.rs",
 * `MoshiState::advance_clock`).  0 <= n_pos <= context. */
rq_status rq_set_kv(rq_handle *h, int32_t session, int32_t n_pos, const void *k,
                    const void *v);

/* Per-kernel timing hook: enqueue `count` launches of one operation of the frame with
 * the frame's own buffers and launch configuration, so a caller can time that kernel
 * alone with events on the handle's stream.  Repeating an operation repeats its side
 * effects on activations and caches: call rq_reset(h, -1) before decoding again.
 *   op     one of RQ_OP_*;  layer  temporal layer index.
 * Under RQ_SCHEDULE_TENSOR the linear ops launch the tensor-core GEMM alone, on the bf16
 * operands the last frame left (the normalisation kernel in front of it is not repeated).
 * *bytes_per_launch (may be NULL) receives the weight + K/V bytes one launch must
 * stream. */
enum {
  RQ_OP_QKV = 0,      /* RMSNorm + in_proj GEMV + rotary + K/V append */
  RQ_OP_ATTN = 1,     /* split-K decode attention */
  RQ_OP_OUT = 2,      /* out_proj GEMV + residual */
  RQ_OP_GATE_IN = 3,  /* RMSNorm + gate_in GEMV + SiLU gate */
  RQ_OP_GATE_OUT = 4, /* gate_out GEMV + residual */
  RQ_OP_HEAD = 5,     /* out_norm + text head GEMV + argmax */
  RQ_OP_FRAME = 6     /* the persistent schedule's whole-frame kernel: its two cooperative
                         launches (the temporal stack, text head and depformer input
                         projections; then the depformer), layer ignored;
                         *bytes_per_launch = every weight once + the live K/V window */
};
rq_status rq_launch_op(rq_handle *h, int32_t op, int32_t layer, int32_t count,
                       double *bytes_per_launch);

/* Standalone decode attention, the kernel the frame runs after each qkv projection
 * ("moshi_lm.rs", `attend`): for each of `batch` single queries and each head,
 * softmax((q . k_j) / sqrt(head_dim)) weighted sum of v_j over the window of the
 * last min(pos + 1, context) positions, position j stored in cache slot j % context.
 *   q          device [batch][heads*head_dim] f32
 *   k, v       device [batch][context][heads*head_dim] in kv_dtype (RQ_F32 / RQ_BF16),
 *              16-byte aligned (RQ_ERR_ARG otherwise)
 *   positions  device [batch] int32, the query's own position (>= 0)
 *   out        device [batch][heads*head_dim] f32
 *   workspace  device scratch of at least rq_attention_workspace_size(...) bytes,
 *              owned by the caller; its contents need no initialisation.
 * head_dim must be 32, 64 or 128.  Enqueued on `cuda_stream`; no synchronization. */
size_t rq_attention_workspace_size(int32_t batch, int32_t heads, int32_t head_dim,
                                   int32_t context);
rq_status rq_attention(int32_t batch, int32_t heads, int32_t head_dim, int32_t context,
                       int32_t kv_dtype, const float *q, const void *k, const void *v,
                       const int32_t *positions, float *out, void *workspace,
                       size_t workspace_bytes, void *cuda_stream);

/* rq_attention without a workspace argument, for callers that cannot allocate device
 * memory -- e.g. a real-time audio thread, where cudaMalloc may wait on device-wide
 * synchronization for an unbounded time, or a plug-in whose host grants a fixed memory
 * budget at start-up and forbids allocation later.  The pages have no counterpart; this
 * is an addition of this library.  Arguments and results are those of rq_attention.
 *   Scratch: a fixed 4 MiB array in the library's device image (present on every GPU
 *   that loads the library until the process exits).  Calls whose scratch need,
 *   rq_attention_workspace_size(batch, heads, head_dim, context), exceeds 4 MiB are
 *   refused with RQ_ERR_UNSUPPORTED before anything is enqueued.
 *   Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   The first call on a device looks up the array's device address there (again after
 *   the device's context changes, e.g. after cudaDeviceReset, so no stale address is
 *   used); make that first call before any stream capture.
 *   Every call shares the one array and leaves its contents behind; the call clears
 *   what must start at zero itself.  Calls that overlap on the GPU (other streams or
 *   threads) race on the array: serialize them. */
rq_status rq_attention_noalloc(int32_t batch, int32_t heads, int32_t head_dim,
                               int32_t context, int32_t kv_dtype, const float *q,
                               const void *k, const void *v, const int32_t *positions,
                               float *out, void *cuda_stream);

/* Token picks ("moshi_lm.rs", `Sampling`, `MoshiLm::set_sampling`, `pick`): every frame
 * picks the text token (temp_text, top_k_text) and then codebooks 0..7 (temp, top_k),
 * each session from its own xorshift64 state ("moshi_lm.rs", `xorshift_u01`):
 *   RQ_PICK_GREEDY  first-wins argmax (the default; the parity and benchmark mode);
 *   RQ_PICK_TOPK    `topk_sample`: the top_k largest logits (taken in descending order,
 *                   equal logits by ascending index), softmax((l - max) / temp) in f64,
 *                   one draw per pick; top_k in 1..256;
 *   RQ_PICK_GUMBEL  `gumbel_full_pick`: argmax of l / temp - ln(-ln u) over the whole
 *                   vocabulary, one draw per logit.
 * seeds: host [B], required unless mode is greedy; session b's state becomes
 * max(seeds[b], 1).  With mode greedy and seeds NULL the states are kept.  Frames
 * report the picked tokens as their own tokens and feed them back as the argmax would
 * be.  Waits for the handle's stream and re-captures the frame graph. */
enum { RQ_PICK_GREEDY = 0, RQ_PICK_TOPK = 1, RQ_PICK_GUMBEL = 2 };
rq_status rq_set_sampling(rq_handle *h, int32_t mode, float temp, float temp_text,
                          int32_t top_k, int32_t top_k_text, const uint64_t *seeds);

/* Each session's sampler state after the last frame (host [B]; synchronizes). */
rq_status rq_get_rng(rq_handle *h, uint64_t *states);

/* Prompt priming ("moshi_lm.rs", `MoshiLm::step_forced`, the prompt-priming primitive):
 * n teacher-forced steps of session `session`.  Step t writes user[t] ([8], codes in
 * [-1, A]) at the user streams' delays, gathers and embeds the 17 inputs (INITIAL while
 * the offset is <= a stream's delay), runs the temporal stack at the session's offset
 * (only its K/V rows are kept: no text head, no depformer), advances the offset, and the
 * ring records forced[t] = [text in [0, V), agent codes in [0, A) x 8].  The n positions
 * run in chunks of up to 64 as the columns of the tensor-core temporal layers (a chunk
 * never wraps the K/V window).  Needs bf16 weights and dim, hidden, ddim, dhidden
 * multiples of 64 (else RQ_ERR_UNSUPPORTED); tokens out of range give RQ_ERR_TOKEN
 * before any state changes.  forced, user: host memory.  Synchronizes the stream. */
rq_status rq_prime(rq_handle *h, int32_t session, int32_t n, const int32_t *forced,
                   const int32_t *user);

/* Embedding replay ("moshi_lm.rs", `MoshiState::advance_clock`): the temporal stack
 * consumes x[t] ([dim] f32, host or device memory) at the session's offset, the offset
 * advances, the ring is not touched.  Same chunking and requirements as rq_prime. */
rq_status rq_replay(rq_handle *h, int32_t session, int32_t n, const float *x);

/* Session snapshot ("moshi_lm.rs", `MoshiState::snapshot`): the ring, the offset and the
 * K/V window of one session (min(offset, context) cache slots per layer, in the K/V
 * dtype), into a caller buffer of at least rq_snapshot_size bytes (host or device
 * memory).  rq_restore puts a snapshot of the same model back into any session of the
 * handle (RQ_ERR_ARG if the layout does not match).  The sampler state is not part of a
 * session.  Both synchronize the stream. */
size_t rq_snapshot_size(const rq_handle *h, int32_t session);
rq_status rq_snapshot(rq_handle *h, int32_t session, void *dst, size_t capacity);
rq_status rq_restore(rq_handle *h, int32_t session, const void *src, size_t size);

/* Weight bands ("moshi_lm.rs", `qn_roundtrip`; Q4_0 as at `q4_roundtrip`): every 32
 * consecutive values of a matrix row share one f32 scale d = mx / -(2^(bits-1)), mx the
 * first value of the largest magnitude in the group; value i is stored as the integer
 * q_i = clamp(round(x_i / d)) in [-2^(bits-1), 2^(bits-1) - 1] (round halves away from
 * zero; q = 0 where d = 0) and stands for q_i * d.  A row of `cols` values is its codes
 * followed by its cols/32 scales: RQ_Q8 one two's-complement byte per value, RQ_Q4 16
 * bytes per group, byte i = (q_i + 8) | (q_(i+16) + 8) << 4.  Stacked weight arrays keep
 * their row order (rq_weights), each row in this layout.
 * rq_band_row_bytes: bytes of one stored row (0 if cols is not a positive multiple of
 * 32).  rq_quantize: rows x cols values (src_dtype RQ_F32 or RQ_BF16, device memory)
 * into dst (device, rows * rq_band_row_bytes bytes), enqueued on cuda_stream. */
size_t rq_band_row_bytes(int32_t dtype, int32_t cols);
rq_status rq_quantize(int32_t dtype, const void *src, int32_t src_dtype, int64_t rows,
                      int32_t cols, void *dst, void *cuda_stream);

/* Number of kernel launches in one frame (the captured graph's kernel nodes; for a
 * persistent handle, the frame that runs while the window is at most 1350 positions). */
int32_t rq_frame_kernel_count(const rq_handle *h);

/* The schedule the handle runs: RQ_SCHEDULE_GRAPH, _PERSISTENT or _TENSOR. */
int32_t rq_schedule(const rq_handle *h);

/* Per-op timeline of the last frame the persistent kernel ran (frames past the long-window
 * switch do not run it and leave the timeline as it was): us[i] = time from the
 * start of op i to the start of op i+1 (the last: to the end of all ops), in
 * microseconds, stamped on the device with %globaltimer (synchronizes the stream).  Ops
 * in frame order: per temporal layer [qkv, attention, out_proj, gate_in, gate_out], the
 * text head, the input projections of all 8 depformer steps (one op), then per depformer
 * step [per layer (qkv — the first adding the step's embedding row —,
 * attention+out_proj, gate_in, gate_out), head].  us == NULL returns the op count; returns the number
 * written, 0 under the graph schedule.  -1 marks an op that was not stamped. */
int32_t rq_get_op_times(rq_handle *h, float *us, int32_t max_ops);

/* Test hook of the failure path: the limit, in nanoseconds, of the device-side waits of
 * the batch-1 whole-frame kernel (its grid-barrier, tagged-word and weight-ring waits); 0
 * restores the default of 2 s.  stall_op >= 0 makes the waits in front of op `stall_op` of
 * the frame's op table (the order of rq_get_op_times; op >= 1, not the depformer input
 * projections beside the text head and not the first op of the depformer launch, which
 * wait for nothing) unsatisfiable: its grid barrier waits for one CTA more than the grid
 * holds, or its tagged words for a tag nothing writes, so every wait there runs out after
 * limit_ns: the frame then returns
 * RQ_ERR_TIMEOUT, later calls RQ_ERR_POISONED until rq_reset(h, -1).  -1 removes the
 * stall.  Nothing traps and no wait is unbounded.  Applies to frames run by the
 * persistent kernel (RQ_ERR_UNSUPPORTED under the other schedules); synchronizes the
 * stream.  A wait that runs out reports an error instead of hanging. */
rq_status rq_set_wait_limit(rq_handle *h, uint64_t limit_ns, int32_t stall_op);

const char *rq_last_error(const rq_handle *h);
const char *rq_status_string(rq_status s);
int32_t rq_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* RQ_H_ */
