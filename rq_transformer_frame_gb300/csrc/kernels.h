// kernels.h -- parameter blocks and host launchers of the decode-step kernels.
// Shared by the kernel translation units and the C-ABI engine (rq_api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rqk {

// bf16 parts of a tensor-core activation operand: 3 gives the exact f32 value
// (hi + mid + lo), 2 a 16-significant-bit value (hi + lo)
#ifndef RQ_OPND_PARTS
#define RQ_OPND_PARTS 2
#endif
constexpr int kOpndParts = RQ_OPND_PARTS;
static_assert(kOpndParts == 2 || kOpndParts == 3, "two or three bf16 parts");

// ---------------------------------------------------------------- weight bands
// "moshi_lm.rs", `qn_roundtrip` (Q4_0: d = max / -8): every 32 consecutive values of a
// matrix row share one f32 scale d; value i is q_i * d with q_i an integer in
// [-2^(bits-1), 2^(bits-1) - 1].  A row of K values is stored as its codes followed by
// its K/32 scales: q8 one two's-complement byte per value (K bytes); q4 16 bytes per
// group, byte i = (q_i + 8) | (q_(i+16) + 8) << 4 (the Q4_0 layout, K/2 bytes).
struct q8_t {};
struct q4_t {};
enum WeightBand : int { BAND_NONE = 0, BAND_Q8 = 8, BAND_Q4 = 4 };
// bytes of one stored row of K values (K a multiple of 32); es: 4 f32, 2 bf16
__host__ __device__ inline size_t band_row_bytes(int band, int es, long long K) {
  if (band == BAND_Q8) return (size_t)K + (size_t)K / 8;
  if (band == BAND_Q4) return (size_t)K / 2 + (size_t)K / 8;
  return (size_t)K * es;
}
// quantize f32 or bf16 rows [rows][cols] (cols a multiple of 32) into the band layout
cudaError_t launch_quantize_band(int band, const void* src, bool src_bf16, long long rows,
                                 int cols, void* dst, cudaStream_t s);

// ---------------------------------------------------------------- token picks
// "moshi_lm.rs", `Sampling` / `pick`: greedy argmax, top-k temperature sampling or
// full-vocabulary Gumbel-max, driven by one xorshift64 state per session.  Within a
// frame pick p (0 the text token, 1 + cb codebook cb) draws from a fixed position of the
// session's stream (Gumbel: one draw per logit, top-k: one draw), so every draw is the
// frame-start state advanced by a known count (xorshift64 is linear over GF(2): the
// advance by n is the matrix power M^n, applied from a table of M^(2^k)).
enum SampleMode : int { SAMPLE_GREEDY = 0, SAMPLE_TOPK = 1, SAMPLE_GUMBEL = 2 };
constexpr int kXsLevels = 32;  // M^(2^k), k < 32: advances up to 2^32 - 1 draws
constexpr int kTopKMax = 256;  // largest k of a top-k pick
struct SampleParams {
  int mode;              // SampleMode
  float temp, temp_text;
  int top_k, top_k_text;
  int V, A;              // logits of the text pick and of each codebook pick
  uint64_t* rng;         // [B] sampler state at the start of the frame
  const uint64_t* jump;  // [kXsLevels][64]: column b of M^(2^k)
};
// the table above, computed on the host from the generator's definition
void xorshift_jump_table(uint64_t* table /*[kXsLevels * 64]*/);
// one CTA per session: pick p's token from logits [B][n] (row stride ld) by top-k
// sampling; writes keys[b * 9 + p] (an argmax key of the chosen token)
cudaError_t launch_topk_pick(const SampleParams& sp, const float* logits, long long ld,
                             int n, int p, unsigned long long* keys, int B, cudaStream_t s,
                             bool pdl);
// the sampler draws one frame consumes
long long frame_draws(const SampleParams& sp);

// ---------------------------------------------------------------- streaming GEMV
// y = W x for one weight matrix W [rows][K] streamed once from HBM through a
// shared-memory ring filled by bulk copies, with a fused prologue (how x is formed)
// and epilogue (where y goes).
enum GemvPro : int {
  PRO_PLAIN = 0,  // x = in[b]
  PRO_RMS = 1,    // x = in[b] * alpha * 1/sqrt(eps + mean(in[b]^2))
  PRO_DATTN = 2,  // x = depformer attention of dq[b] over keys 0..n_keys-1
  PRO_RMS_EMB = 3  // persistent schedule: x = in + E[prev] (CTA 0 also stores this x to
                   // side_out), then as PRO_RMS; prev is pick key_index (or the forced token)
};
enum GemvEpi : int {
  EPI_STORE = 0,   // out[b][r] = y
  EPI_RESID = 1,   // out[b][r] += y
  EPI_SWIGLU = 2,  // out[b][j] = silu(y_j) * y_{F+j}
  EPI_QKV = 3,     // rotary on q, k; q -> out, k/v -> temporal cache slot pos % C
  EPI_DQKV = 4,    // q -> out, k/v -> depformer per-frame cache entry
  EPI_ARGMAX = 5,  // out[b][r] = y (logits) and first-wins argmax -> keys
  EPI_DEPIN = 6    // out[b][r] = y + E[prev][r]
};

struct GemvPlan {
  int n_out;       // output rows (EPI_SWIGLU: F)
  int K;           // reduction length
  int tile_rows;   // weight rows per pipeline stage (SWIGLU: half gate, half mult)
  int tiles;       // number of tiles
  int grid;        // CTAs per session
  int n_stages;    // pipeline depth
  int tpr;         // threads per row group (power of two, 32..256)
  int rg;          // rows per thread per tile (1 or 2)
  int nch;         // 16-byte chunks of x per thread (kernel template parameter)
  int kparts;      // persistent schedule: reduction split into parts of <= 2 chunks/thread
  int kp_width;    // columns of every part but the last
  int max_tiles;   // tiles of the busiest CTA
  int smem;        // dynamic shared memory bytes
  double bytes;    // weight bytes one launch streams
};

struct GemvParams {
  const void* W;
  long long w_half;  // SWIGLU: byte offset of the multiplier half
  GemvPlan pl;
  // prologue
  const float* in;
  long long in_bs;     // batch stride (elements)
  const float* alpha;
  float eps;
  float* side_out;     // PRO_RMS: CTA 0 also stores x here (nullable)
  long long side_bs;
  const float* dq;     // PRO_DATTN: query [B][DD]
  long long dq_bs;
  const float* dk;     // PRO_DATTN: keys [n][DD] at dk + b*dkv_bs
  const float* dv;
  long long dkv_bs;
  int n_keys, dheads, dhead_dim;
  // epilogue
  float* out;
  long long out_bs;
  void* kcache;        // EPI_QKV: cache of this layer, session stride kv_bs
  void* vcache;
  long long kv_bs;
  int kv_bf16;
  int head_dim;
  int context;
  float rope_theta;
  const int* offsets;  // [B] current positions
  float* dk_out;       // EPI_DQKV
  float* dv_out;
  unsigned long long* keys;  // EPI_ARGMAX / EPI_DEPIN: [B][9]
  int key_index;
  const void* emb;     // EPI_DEPIN: table [rows][n_out] in the weight dtype
  const int* d_in;     // per-step input block (forced tokens / flags)
  int batch;
  uint32_t* status;
  SampleParams samp;   // EPI_ARGMAX: Gumbel-max scores when samp.mode is SAMPLE_GUMBEL
};

GemvPlan plan_gemv(int n_out, int K, int elem_bytes, bool paired, bool even_rows,
                   int num_sms, int band = BAND_NONE);
int gemv_chunks_per_thread(const GemvPlan& pl, int elem_bytes);
cudaError_t gemv_configure_all();
constexpr int kGemvMaxChunks = 6;  // 16-byte chunks of x per thread
constexpr int kGemvConsumers = 256;  // consumer threads of a GEMV CTA (+1 producer warp)
// wtype: 0 f32, 1 bf16, BAND_Q8, BAND_Q4 (matrix storage)
cudaError_t launch_gemv(const GemvParams& p, int pro, int epi, int wtype, int batch,
                        cudaStream_t s, bool pdl);

// ---------------------------------------------------------------- decode attention
struct AttnParams {
  const float* q;       // [B][D]
  const void* kbase;    // K cache viewed as rows of D elements; session b, slot j of this
  const void* vbase;    // layer is row  row_bs * b + row0 + j  (V alike)
  long long rows;       // rows of that view (the tensor maps' extent)
  long long row0, row_bs;
  const int* offsets;   // [B]
  float* part;          // [B][H][nsplit][hd + 2]
  int* counters;        // [B][H], zero between uses
  float* out;           // [B][D]
  uint16_t* out_bf16;   // nullable: the same output as a bf16 operand [parts][nb][D]
  int nb;               // rows per bf16 part
  int D, H, hd, C, kps, nsplit;
  int batch;
  uint32_t* status;
};
cudaError_t launch_attn(const AttnParams& p, bool kv_bf16, cudaStream_t s, bool pdl);
// Standalone decode attention (rq_attention and rq_attention_noalloc): positions per
// split, and the bytes of the per-split partials that precede the merge tickets in the
// scratch (B x H x nsplit rows of hd + 2 floats, rounded up to 256 bytes).
#ifndef RQ_ATTN_KPS
#define RQ_ATTN_KPS 64
#endif
constexpr int kStandaloneAttnKps = RQ_ATTN_KPS;
inline size_t standalone_attn_partial_bytes(int B, int H, int hd, int C) {
  const size_t nsplit = (size_t)(C + kStandaloneAttnKps - 1) / kStandaloneAttnKps;
  return ((size_t)B * H * nsplit * (hd + 2) * sizeof(float) + 255) & ~(size_t)255;
}
// shared-memory attribute and occupancy of the attention kernel (call outside capture)
cudaError_t attn_configure(int hd, bool kv_bf16, int kps);
cudaError_t launch_dattn_batched(const float* dq, long long dq_bs, const float* dk,
                                 const float* dv, long long dkv_bs, int n_keys, int B,
                                 int heads, int hd, uint16_t* out, long long out_bs, int nb,
                                 cudaStream_t s, bool pdl);

// ---------------------------------------------------------------- tensor-core GEMM
// Y[b][n] = X[b][:] . W[n][:] for all sessions b at once (batch 2..64): a CTA computes a
// 128-row tile of W against NB (padded) sessions on the tcgen05 tensor cores, operands
// fed by TMA, accumulator in tensor memory; optional split-K merged in split order.
struct TcPlan {
  int n_out, K;       // output rows (paired: F), reduction length (multiple of 64)
  int NB;             // padded batch: multiple of 16, <= 64 (operand rows: 3 NB)
  int paired;         // SiLU-gated: tile rows 0-63 gate, 64-127 multiplier
  int tiles_m, splits, ksteps, ksteps_split;
  int cluster;        // 1: a tile's K splits form one thread-block cluster and merge
                      // through its shared memory; 0: through L2 (partials + ticket)
  int n_stages, smem;
  double bytes;       // weight bytes one launch streams
};

struct TcParams {
  TcPlan pl;
  int epi;            // GemvEpi
  int B;              // sessions (<= NB)
  float* out;         // f32 outputs [B][..] (stride out_bs)
  long long out_bs;
  uint16_t* out_bf16; // EPI_SWIGLU: bf16 operand [parts][NB][F] (row stride outb_bs)
  long long outb_bs;
  void* kcache;       // EPI_QKV
  void* vcache;
  long long kv_bs;
  int kv_bf16, head_dim, context;
  const float2* rope; // [B][head_dim/2] (cos, sin) at each session's position
  const int* offsets;
  float* dk_out;      // EPI_DQKV
  float* dv_out;
  long long dkv_bs;
  unsigned long long* keys;
  int key_index;
  const void* emb;    // EPI_DEPIN
  const int* d_in;
  float* partial;     // split-K scratch [tiles_m][splits][NB][128]
  int* tickets;       // [tiles_m], zero between uses
  uint32_t* status;
  // fused RMSNorm.  Producer (EPI_RESID / EPI_DEPIN): also write the next GEMM's operand
  // bf16 parts of (new value * alpha_next) [parts][NB][n_out] (alpha_next null: the value) and,
  // when ss_out is set, per-tile sums of squares ss_out[tile][NB] of the new values.
  // Consumer: scale every accumulator column b by 1 / sqrt(eps + sum_t ss_in[t][b] / rms_K).
  uint16_t* opnd;
  const float* alpha_next;
  float* ss_out;
  const float* ss_in;
  int ss_tiles, rms_K;
  float eps;
  SampleParams samp;  // EPI_ARGMAX
};

TcPlan plan_tc(int n_out, int K, int NB, bool paired, int num_sms);
cudaError_t launch_tc(const TcParams& p, const CUtensorMap& wmap, const CUtensorMap& xmap,
                      cudaStream_t s, bool pdl);
cudaError_t tc_configure();
// encode a 2-D tensor map over a row-major rows x cols array (bf16 or f32), box
// {box_cols, box_rows}, 128-byte swizzle or none
cudaError_t encode_tmap_2d(CUtensorMap* map, bool bf16, const void* base, long long rows,
                           long long cols, int box_cols, int box_rows, bool swizzle128);
// encode a 2-D bf16 tensor map: rows x cols (row-major), box {64 cols, box_rows}
cudaError_t make_tmap_bf16(CUtensorMap* map, const void* base, long long rows, long long cols,
                           int box_rows);

// prep: X bf16 parts [parts][NB][K] = in or RMSNorm(in, alpha) for sessions < B (rows >= B zero);
// side (nullable) receives the f32 normalized rows
cudaError_t launch_prep_bf16(const float* in, long long in_bs, const float* alpha, float eps,
                             int B, int NB, int K, uint16_t* xb, float* side, long long side_bs,
                             cudaStream_t s, bool pdl);

// ---------------------------------------------------------------- persistent frame
// The whole frame's linears and attentions as one cooperative launch: an op table
// executed in order by every CTA, a bounded grid barrier between dependent ops, and
// a per-CTA producer warp that streams the weight tiles of all ops ahead of the
// consumers through one shared-memory ring.
enum PersOpType : int { OPT_GEMV = 0, OPT_ATTN = 1, OPT_TOPK = 2 };  // OPT_TOPK: pick key_index from logits `in`

struct PersOp {
  int type;       // PersOpType
  int pro, epi;   // GEMV prologue / epilogue (GemvPro / GemvEpi)
  int plan;       // index into PersParams::plans
  const void* W;  // weights of this op
  long long w_half;  // SWIGLU: byte offset of the multiplier half
  const float* in;      // prologue input (PRO_DATTN: the query)
  const float* alpha;
  float* side_out;
  const float* dk;      // PRO_DATTN keys / values [n][DD]
  const float* dv;
  int n_keys;
  float* out;
  void* kcache;         // EPI_QKV / OPT_ATTN: this layer's cache [C][D]
  void* vcache;
  float* dk_out;        // EPI_DQKV
  float* dv_out;
  int key_index;
  const void* emb;      // EPI_DEPIN / PRO_RMS_EMB: table [rows][n_out or K]
  int nobar;            // 1: no grid barrier before this op (it reads nothing the previous
                        // op writes)
  // The one-CTA-per-SM launch (the depformer) has no grid barriers: every activation one
  // CTA writes and another reads is a tagged word (see frame_persistent.cuh), and these
  // are the frame op indices whose tags the op waits for (-1: a plain read of what an
  // earlier launch wrote).  Its `in`, `out`, `side_out`, `dk`, `dv`, `dk_out`, `dv_out`
  // then point at tagged-word arrays (uint64, same element indexing), except the logits
  // (`out` of EPI_ARGMAX, plain f32 for the host; `side_out` there: their tagged copy for
  // a top-k pick, or null) and `in` of PRO_RMS_EMB (the first launch's f32 dep_pre).
  int tag_in;           // writer of `in` (PRO_DATTN: of the query; OPT_TOPK: of the logits)
  int tag_res;          // EPI_RESID: last writer of the residual rows `out`
  int tag_kv;           // PRO_DATTN: writer of key / value 0; key j's is tag_kv + j * tag_kv_step
  int tag_kv_step;
  int tag_key;          // PRO_RMS_EMB: the op that chose pick key_index (-1: the first launch)
  int key_slots;        // PRO_RMS_EMB: that op's key slots (the grid's CTAs, or 1: a top-k pick)
  int no_keymax;        // EPI_ARGMAX: a top-k pick follows; it alone writes keys[key_index]
};

constexpr int kPersMaxPlans = 12;

struct PersParams {
  const PersOp* ops;    // this launch's ops (the frame's op table from op_base on)
  int n_ops;
  int op_base;          // frame op index of ops[0]: the trace and the test stall use frame indices
  GemvPlan plans[kPersMaxPlans];
  int slot_bytes;   // bytes of one ring slot (>= every op's tile)
  int n_slots;
  int part_floats;  // per-op partial-sum buffer (floats)
  float eps;
  int kv_bf16, head_dim, context;
  float rope_theta;
  int dheads, dhead_dim;
  const int* offsets;
  unsigned long long* keys;
  const int* d_in;
  // attention
  const float* attn_q;
  float* attn_out;
  float* part;
  int* counters;
  int D, H, kps, nsplit;
  unsigned int* grid_bar;  // zero at launch
  // wait control read once per launch: [0] limit of the grid-barrier and weight-ring
  // waits in ns (0: kWaitLimitNs); [1] test stall: k + 1 makes the barrier before op k
  // wait for one CTA more than the grid has, so every wait there runs out (0: none)
  const unsigned long long* wait_ctl;
  uint32_t* status;
  unsigned long long* trace;  // [n_ops + 1] op start times (ns), CTA 0 (nullable)
  SampleParams samp;
  // tagged-word exchange (the one-CTA-per-SM launch): tags are (*epoch << 10) | frame op
  // index; a launch with epoch_bump set advances *epoch once (the frame's first launch)
  unsigned int* epoch;
  int epoch_bump;
  unsigned long long* key_ll;  // [9][grid][2] tagged halves of each CTA's best key per pick
  float* topk_scratch;         // [A] a top-k pick's logits, gathered from their tagged copy
};

GemvPlan plan_persistent(int n_out, int K, int elem_bytes, bool paired, bool even_rows,
                         int grid, int band = BAND_NONE);
// ---------------------------------------------------------------- tensor-core frame
// Everything a batched frame needs between frame_begin and frame_end: the per-op plans,
// the bf16 operand buffers [kOpndParts][NB][K] (hi, mid[, lo] parts; rows >= B stay zero) and one
// TMA map per weight matrix and per operand buffer.
struct TcFrame {
  int B, NB, D, L, C, F, V, A, DD, DL, DF, H, hd, dH, dhd;
  float eps;
  int kv_bf16;
  // bf16 matrices, f32 alphas (layout of rq_weights)
  const void *in_proj, *out_proj, *gate_in, *gate_out, *text_linear, *dep_in, *dep_text_emb,
      *dep_emb, *d_in_proj, *d_out_proj, *d_gate_in, *d_gate_out, *linears;
  const float *norm1, *norm2, *out_norm, *dnorm1, *dnorm2;
  // f32 state and outputs
  float *x, *q, *attn, *tout, *text_logits, *audio_logits, *dx, *dq, *dkv;
  void *kcache, *vcache;
  int32_t* offsets;
  const int32_t* d_in;
  unsigned long long* keys;
  SampleParams samp;  // token picks (EPI_ARGMAX scores; top-k picks after the heads)
  float* attn_part;
  int* attn_counters;
  int kps, nsplit;
  uint32_t* status;
  float2* rope;  // [B][hd/2]
  // bf16 operands
  uint16_t *xb, *attn_b, *u_b, *tout_b, *dxb, *do_b, *du_b;
  float* part;   // split-K partial tiles
  int* tickets;  // per tile, zero between uses
  float *ss_x, *ss_dx;  // fused RMSNorm: per-tile sums of squares [D/128][NB], [DD/128][NB]
  TcPlan p_qkv, p_out, p_gin, p_gout, p_head, p_depin, p_dqkv, p_dout, p_dgin, p_dgout, p_lin;
  CUtensorMap* wm;  // per weight matrix, see tc_frame_wmap_index
  int n_wm;
  CUtensorMap xm_x, xm_attn, xm_u, xm_tout, xm_dx, xm_do, xm_du;
  // prefill: the B columns are consecutive positions of ONE session whose K/V region
  // kcache / vcache point at ([L][C][D]); offsets[b] is column b's position
  int one_session;
};
// plans for every op; returns the split-K scratch floats and ticket count needed
void tc_frame_plan(TcFrame& f, int num_sms, size_t* part_floats, int* n_tickets);
// encode every tensor map (buffers and weights set, f.wm holds f.n_wm entries)
cudaError_t tc_frame_maps(TcFrame& f);
int tc_frame_n_maps(const TcFrame& f);
// the frame's ops after frame_begin, each launched with a programmatic edge
cudaError_t tc_frame_enqueue(const TcFrame& f, cudaStream_t s);
// the temporal layers alone (layer-0 norm, then qkv, attention, out, gate_in, gate_out)
cudaError_t tc_frame_enqueue_temporal(const TcFrame& f, cudaStream_t s);

// ---------------------------------------------------------------- prompt prefill
// T <= 64 consecutive positions of one session as the columns of the tensor-core
// temporal layers ("moshi_lm.rs", `MoshiLm::step_forced` priming and the embedding
// replay of `MoshiState::advance_clock`).
struct PrefillParams {
  int session, T, B, D, V, A, head_dim;
  float rope_theta;
  int32_t* ring;          // [B][17][3]
  int32_t* offsets;       // [B]
  const int32_t* forced;  // [T][9] priming (the ring records them); null: replay
  const int32_t* user;    // [T][8] priming
  int32_t* tokens;        // [T][17] scratch: each step's gathered inputs
  int32_t* pos;           // [T] column positions (written)
  float2* rope;           // [T][head_dim / 2] (written)
  const void* emb;        // [16][A+1][D]
  const void* text_emb;   // [V+1][D]
  float* x;               // [T][D] priming: the embedding sums (written); replay: given
};
cudaError_t launch_prefill_begin(const PrefillParams& p, bool bf16, cudaStream_t s);
// one op of a temporal layer alone (0 qkv, 1 attention, 2 out_proj, 3 gate_in, 4 gate_out,
// 5 text head): the GEMM on the operands left by the last frame
cudaError_t tc_frame_launch_op(const TcFrame& f, int op, int layer, cudaStream_t s);

// minb: CTAs per SM of the launch (2: the temporal stack; 1: the depformer)
cudaError_t launch_persistent(const PersParams& p, int wtype, bool kv_bf16, int grid,
                              int smem, cudaStream_t s, bool pdl, int minb = 2);
// uint32 index, in the persistent schedule's barrier allocation, of the depformer launch's
// grid-barrier counter (its own 128-byte line); frame_begin zeroes it with the first one
constexpr int kPersDepBarWord = 64;
// uint32 index there of the frame epoch (never zeroed: tags of earlier frames must differ)
constexpr int kPersEpochWord = 96;
// frame op indices fit the low 10 bits of a tag
constexpr int kPersMaxTaggedOps = 1024;
// key slots a tagged reader polls, one consumer thread each
constexpr int kPersMaxKeySlots = 256;
cudaError_t persistent_configure(int wtype, bool kv_bf16, int smem, int head_dim, int minb);
int persistent_max_grid(int wtype, bool kv_bf16, int smem, int head_dim, int minb);

// ---------------------------------------------------------------- frame begin / end
struct FrameParams {
  int B, D, V, A;
  int32_t* ring;        // [B][17][3]
  int32_t* offsets;     // [B]
  const int32_t* d_in;  // per-step input block
  int32_t* d_out;       // per-step output block (int32 words)
  uint8_t* d_has;
  unsigned long long* keys;  // [B][9]
  const void* emb;      // [16][A+1][D]
  const void* text_emb; // [V+1][D]
  float* x;             // [B][D]
  float* emb_sum;       // [B][D]
  unsigned int* grid_bar;  // persistent schedule's barrier counter (nullable)
  float2* rope;         // [B][head_dim/2] (cos, sin) at each session's position (nullable)
  int head_dim;
  float rope_theta;
  SampleParams samp;    // frame_end advances each session's sampler state
};
cudaError_t launch_frame_begin(const FrameParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_frame_end(const FrameParams& p, cudaStream_t s, bool pdl);
cudaError_t launch_reset(int32_t* ring, int32_t* offsets, int B, int session,
                         cudaStream_t s);
cudaError_t launch_set_offset(int32_t* offsets, int session, int value, cudaStream_t s);

}  // namespace rqk
