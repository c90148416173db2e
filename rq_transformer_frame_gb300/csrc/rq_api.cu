// rq_api.cu -- the C ABI (include/rq.h): handle, device state, the per-frame kernel
// schedule captured once as a CUDA graph with programmatic-dependent-launch edges,
// and the host-side validation and error model.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <cmath>
#include <vector>

#include "../../include/rq.h"
#include "common.cuh"
#include "kernels.h"
#include "sampling.cuh"

using namespace rqk;

namespace {
thread_local std::string g_create_err;  // why the last rq_create failed
}  // namespace

struct rq_handle {
  rq_config cfg{};
  rq_weights w{};
  cudaStream_t stream = nullptr;  // caller's stream
  cudaStream_t cap = nullptr;     // private stream used for graph capture
  int device = 0, num_sms = 0;
  bool wbf = false, kvbf = false;
  int wes = 4, kves = 4;  // element bytes of the tables (and of f32 / bf16 matrices), of K/V
  int band = BAND_NONE;   // matrices in a weight band (their tables are then bf16)
  int wtype = 0;          // matrix storage for launch_gemv: 0 f32, 1 bf16, BAND_Q8, BAND_Q4
  IoLayout io{1};
  // device state
  int32_t* ring = nullptr;
  int32_t* offsets = nullptr;
  void* kcache = nullptr;
  void* vcache = nullptr;
  int32_t* d_in = nullptr;
  uint8_t* d_outb = nullptr;
  float *x = nullptr, *emb_sum = nullptr, *q = nullptr, *attn = nullptr, *u = nullptr;
  float *tout = nullptr, *text_logits = nullptr, *audio_logits = nullptr;
  unsigned long long* keys = nullptr;
  float *dx = nullptr, *dq = nullptr, *dkv = nullptr, *du = nullptr;
  float* dep_pre = nullptr;  // persistent schedule: dep_in[cb] . t of the 8 steps [8][DD]
  // the depformer launch's tagged-word copies (64-bit words, element indexing of dx, dq,
  // du, dkv and the audio logits) and its key slots / top-k scratch
  float *dx_ll = nullptr, *dq_ll = nullptr, *du_ll = nullptr, *dkv_ll = nullptr;
  float *alog_ll = nullptr, *topk_scratch = nullptr;
  unsigned long long* key_ll = nullptr;
  float* part = nullptr;
  int* counters = nullptr;
  // pinned host staging
  int32_t* h_in = nullptr;
  uint8_t* h_out = nullptr;
  // graph
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int n_kernels = 0;
  // persistent schedule only: the same frame as one kernel per op, replayed once the
  // window is longer than kLongWindow (see frame_exec)
  cudaGraph_t graph_long = nullptr;
  cudaGraphExec_t exec_long = nullptr;
  // plans
  GemvPlan p_qkv{}, p_out{}, p_gin{}, p_gout{}, p_head{};
  GemvPlan p_depin{}, p_dqkv{}, p_dout{}, p_dgin{}, p_dgout{}, p_lin{};
  int kps = 64, nsplit = 1;
  // persistent schedule
  int schedule = RQ_SCHEDULE_GRAPH;
  PersOp* d_ops = nullptr;
  std::vector<char> pers_nobar;  // host copy: op k has no grid barrier in front of it
  unsigned int* grid_bar = nullptr;
  unsigned long long* trace = nullptr;
  PersParams pers{};
  int pers_grid = 0, pers_smem = 0;
  // the depformer's ops run as a second cooperative launch at one CTA per SM (pers_split:
  // frame op index of its first op; == the op count when everything runs in the first)
  PersParams pers_dep{};
  int pers_dep_grid = 0, pers_dep_smem = 0, pers_split = 0;
  // prompt prefill: up to kPrefillCols positions of one session per tensor-core pass
  TcFrame pf{};
  bool pf_ready = false;
  std::vector<CUtensorMap> pf_maps;
  std::vector<void*> pf_bufs;  // freed with the handle
  int32_t *pf_tokens = nullptr, *pf_pos = nullptr, *pf_forced = nullptr, *pf_user = nullptr;
  // token picks: the sampler configuration and each session's xorshift64 state
  SampleParams samp{};
  uint64_t* rng = nullptr;      // [B]
  uint64_t* xs_jump = nullptr;  // [kXsLevels][64]
  // tensor-core schedule
  TcFrame tcf{};
  std::vector<CUtensorMap> tc_maps;
  float2* rope = nullptr;
  uint16_t *xb = nullptr, *attn_b = nullptr, *u_b = nullptr, *tout_b = nullptr;
  uint16_t *dxb = nullptr, *do_b = nullptr, *du_b = nullptr;
  float* tc_part = nullptr;
  int* tc_tickets = nullptr;
  float *ss_x = nullptr, *ss_dx = nullptr;
  std::vector<int> host_off;  // host mirror of the offsets (for byte accounting)
  bool poisoned = false;
  bool forcing_dirty = true;
  std::string err;

  int32_t* d_out_words() const { return reinterpret_cast<int32_t*>(d_outb); }
  uint8_t* d_has() const { return d_outb + io.has_off_bytes(); }
  uint32_t* d_status() const { return reinterpret_cast<uint32_t*>(d_outb + io.status_off_bytes()); }
};

namespace {

rq_status fail(rq_handle* h, rq_status s, const std::string& msg) {
  if (h) h->err = msg;
  return s;
}

rq_status cuda_fail(rq_handle* h, cudaError_t e, const char* where) {
  if (h) {
    h->poisoned = true;
    h->err = std::string(where) + ": " + cudaGetErrorString(e);
  }
  return RQ_ERR_CUDA;
}

#define RQ_CUDA(h, call)                               \
  do {                                                 \
    cudaError_t e_ = (call);                           \
    if (e_ != cudaSuccess) return cuda_fail(h, e_, #call); \
  } while (0)

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// elements -> byte offset into a weight array
// the matrix that follows `rows_before` rows of K values in a stacked weight array
const void* mat(const rq_handle* h, const void* base, size_t rows_before, long long K) {
  return static_cast<const char*>(base) + rows_before * band_row_bytes(h->band, h->wes, K);
}

const void* woff(const void* base, size_t elems, int es) {
  return static_cast<const char*>(base) + elems * (size_t)es;
}

bool hd_ok(int hd) { return hd == 32 || hd == 64 || hd == 128; }

rq_status validate_config(const rq_config* c, std::string* why) {
  auto bad = [&](const char* m) { *why = m; return RQ_ERR_ARG; };
  auto uns = [&](const char* m) { *why = m; return RQ_ERR_UNSUPPORTED; };
  if (c->batch < 1 || c->dim < 1 || c->layers < 1 || c->heads < 1 || c->hidden < 1 ||
      c->context < 1 || c->text_card < 1 || c->audio_card < 1 || c->ddim < 1 ||
      c->dlayers < 1 || c->dheads < 1 || c->dhidden < 1)
    return bad("every size must be positive");
  if (c->heads * c->head_dim != c->dim) return bad("dim != heads * head_dim");
  if (c->dheads * c->dhead_dim != c->ddim) return bad("ddim != dheads * dhead_dim");
  if (!hd_ok(c->head_dim) || !hd_ok(c->dhead_dim)) return uns("head dims must be 32, 64 or 128");
  if (c->dheads > 32) return uns("at most 32 depformer heads");
  if ((c->weight_dtype != RQ_F32 && c->weight_dtype != RQ_BF16 && c->weight_dtype != RQ_Q8 &&
       c->weight_dtype != RQ_Q4) ||
      (c->kv_dtype != RQ_F32 && c->kv_dtype != RQ_BF16))
    return bad("weight_dtype must be RQ_F32, RQ_BF16, RQ_Q8 or RQ_Q4; kv_dtype RQ_F32 or RQ_BF16");
  if ((c->weight_dtype == RQ_Q8 || c->weight_dtype == RQ_Q4) &&
      (c->dim % 128 || c->hidden % 128 || c->ddim % 128 || c->dhidden % 128))
    return uns("weight bands need dim, hidden, ddim and dhidden multiples of 128");
  if (c->dim % 8 || c->hidden % 8 || c->ddim % 8 || c->dhidden % 8)
    return uns("dim, hidden, ddim and dhidden must be multiples of 8");
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return bad("bad rms_eps / rope_theta");
  if (c->schedule < RQ_SCHEDULE_AUTO || c->schedule > RQ_SCHEDULE_TENSOR)
    return bad("unknown schedule");
  return RQ_OK;
}

}  // namespace

namespace {

GemvParams base_params(const rq_handle* h, const GemvPlan& pl, const void* W) {
  GemvParams p{};
  p.W = W;
  p.pl = pl;
  p.eps = h->cfg.rms_eps;
  p.kv_bf16 = h->kvbf ? 1 : 0;
  p.head_dim = h->cfg.head_dim;
  p.context = h->cfg.context;
  p.rope_theta = h->cfg.rope_theta;
  p.offsets = h->offsets;
  p.keys = h->keys;
  p.d_in = h->d_in;
  p.batch = h->cfg.batch;
  p.status = h->d_status();
  p.samp = h->samp;
  return p;
}

// ---- temporal layer l ("moshi_lm.rs", `temporal_step`)
cudaError_t op_qkv(const rq_handle* h, int l, cudaStream_t s, bool pdl) {
  const rq_config& c = h->cfg;
  const size_t D = c.dim, C = c.context, L = c.layers;
  GemvParams p = base_params(h, h->p_qkv, mat(h, h->w.in_proj, (size_t)l * 3 * D, D));
  p.in = h->x;
  p.in_bs = D;
  p.alpha = h->w.norm1 + (size_t)l * D;
  p.out = h->q;
  p.out_bs = D;
  p.kcache = static_cast<char*>(h->kcache) + (size_t)l * C * D * h->kves;
  p.vcache = static_cast<char*>(h->vcache) + (size_t)l * C * D * h->kves;
  p.kv_bs = (long long)(L * C * D);
  return launch_gemv(p, PRO_RMS, EPI_QKV, h->wtype, c.batch, s, pdl);
}

cudaError_t op_attn(const rq_handle* h, int l, cudaStream_t s, bool pdl) {
  const rq_config& c = h->cfg;
  const size_t C = c.context, L = c.layers;
  AttnParams a{};
  a.q = h->q;
  a.kbase = h->kcache;  // [B][L][C][D]: session b, layer l, slot j is row (b L + l) C + j
  a.vbase = h->vcache;
  a.rows = (long long)h->cfg.batch * L * C;
  a.row0 = (long long)l * C;
  a.row_bs = (long long)(L * C);
  a.offsets = h->offsets;
  a.part = h->part;
  a.counters = h->counters;
  a.out = h->attn;
  a.D = c.dim;
  a.H = c.heads;
  a.hd = c.head_dim;
  a.C = c.context;
  a.kps = h->kps;
  a.nsplit = h->nsplit;
  a.batch = c.batch;
  a.status = h->d_status();
  return launch_attn(a, h->kvbf, s, pdl);
}

cudaError_t op_out(const rq_handle* h, int l, cudaStream_t s, bool pdl) {
  const size_t D = h->cfg.dim;
  GemvParams p = base_params(h, h->p_out, mat(h, h->w.out_proj, (size_t)l * D, D));
  p.in = h->attn;
  p.in_bs = D;
  p.out = h->x;
  p.out_bs = D;
  return launch_gemv(p, PRO_PLAIN, EPI_RESID, h->wtype, h->cfg.batch, s, pdl);
}

cudaError_t op_gate_in(const rq_handle* h, int l, cudaStream_t s, bool pdl) {
  const size_t D = h->cfg.dim, F = h->cfg.hidden;
  GemvParams p = base_params(h, h->p_gin, mat(h, h->w.gate_in, (size_t)l * 2 * F, D));
  p.w_half = (long long)(F * band_row_bytes(h->band, h->wes, D));
  p.in = h->x;
  p.in_bs = D;
  p.alpha = h->w.norm2 + (size_t)l * D;
  p.out = h->u;
  p.out_bs = F;
  return launch_gemv(p, PRO_RMS, EPI_SWIGLU, h->wtype, h->cfg.batch, s, pdl);
}

cudaError_t op_gate_out(const rq_handle* h, int l, cudaStream_t s, bool pdl) {
  const size_t D = h->cfg.dim, F = h->cfg.hidden;
  GemvParams p = base_params(h, h->p_gout, mat(h, h->w.gate_out, (size_t)l * D, F));
  p.in = h->u;
  p.in_bs = F;
  p.out = h->x;
  p.out_bs = D;
  return launch_gemv(p, PRO_PLAIN, EPI_RESID, h->wtype, h->cfg.batch, s, pdl);
}

// out_norm + text head + first-wins argmax ("moshi_lm.rs", `step_ext` steps 4-5)
cudaError_t op_head(const rq_handle* h, cudaStream_t s, bool pdl) {
  const size_t D = h->cfg.dim, V = h->cfg.text_card;
  GemvParams p = base_params(h, h->p_head, h->w.text_linear);
  p.in = h->x;
  p.in_bs = D;
  p.alpha = h->w.out_norm;
  p.side_out = h->tout;
  p.side_bs = D;
  p.out = h->text_logits;
  p.out_bs = V;
  p.key_index = 0;
  return launch_gemv(p, PRO_RMS, EPI_ARGMAX, h->wtype, h->cfg.batch, s, pdl);
}

// ---- depformer step cb ("moshi_lm.rs", `depformer_cycle`)
// per-frame K/V layout [B][DL][2][8][DD]: K of (layer l, step j) at ((l*2+0)*8+j)*DD
size_t dkv_off(const rq_handle* h, int l, int kv, int j) {
  const size_t DD = h->cfg.ddim;
  return (((size_t)l * 2 + kv) * 8 + j) * DD;
}

cudaError_t op_dep_in(const rq_handle* h, int cb, cudaStream_t s, bool pdl) {
  const rq_config& c = h->cfg;
  const size_t D = c.dim, DD = c.ddim, A = c.audio_card;
  GemvParams p = base_params(h, h->p_depin, mat(h, h->w.dep_in, (size_t)cb * DD, D));
  p.in = h->tout;
  p.in_bs = D;
  p.out = h->dx;
  p.out_bs = DD;
  p.emb = cb == 0 ? h->w.dep_text_emb : woff(h->w.dep_emb, (size_t)(cb - 1) * (A + 1) * DD, h->wes);
  p.key_index = cb;  // text token for cb 0, else audio cb-1 (key 1 + (cb-1))
  return launch_gemv(p, PRO_PLAIN, EPI_DEPIN, h->wtype, c.batch, s, pdl);
}

cudaError_t op_dlayer(const rq_handle* h, int cb, int l, cudaStream_t s, bool pdl) {
  const rq_config& c = h->cfg;
  const size_t DD = c.ddim, DF = c.dhidden;
  const size_t ls = (size_t)l * 8 + cb;
  const long long dkv_bs = (long long)c.dlayers * 2 * 8 * DD;
  cudaError_t e;
  {  // rms_norm + in_projs[cb] -> q, per-frame K/V entry cb
    GemvParams p = base_params(h, h->p_dqkv, mat(h, h->w.d_in_proj, ls * 3 * DD, DD));
    p.in = h->dx;
    p.in_bs = DD;
    p.alpha = h->w.dnorm1 + (size_t)l * DD;
    p.out = h->dq;
    p.out_bs = DD;
    p.dk_out = h->dkv + dkv_off(h, l, 0, cb);
    p.dv_out = h->dkv + dkv_off(h, l, 1, cb);
    p.dkv_bs = dkv_bs;
    if ((e = launch_gemv(p, PRO_RMS, EPI_DQKV, h->wtype, c.batch, s, pdl)) != cudaSuccess) return e;
  }
  {  // attention over entries 0..cb fused as the prologue of out_projs[cb] + residual
    GemvParams p = base_params(h, h->p_dout, mat(h, h->w.d_out_proj, ls * DD, DD));
    p.dq = h->dq;
    p.dq_bs = DD;
    p.dk = h->dkv + dkv_off(h, l, 0, 0);
    p.dv = h->dkv + dkv_off(h, l, 1, 0);
    p.dkv_bs = dkv_bs;
    p.n_keys = cb + 1;
    p.dheads = c.dheads;
    p.dhead_dim = c.dhead_dim;
    p.in = h->dq;  // unused by this prologue
    p.out = h->dx;
    p.out_bs = DD;
    if ((e = launch_gemv(p, PRO_DATTN, EPI_RESID, h->wtype, c.batch, s, pdl)) != cudaSuccess) return e;
  }
  {  // rms_norm + gating[cb].linear_in + silu gate
    GemvParams p = base_params(h, h->p_dgin, mat(h, h->w.d_gate_in, ls * 2 * DF, DD));
    p.w_half = (long long)(DF * band_row_bytes(h->band, h->wes, DD));
    p.in = h->dx;
    p.in_bs = DD;
    p.alpha = h->w.dnorm2 + (size_t)l * DD;
    p.out = h->du;
    p.out_bs = DF;
    if ((e = launch_gemv(p, PRO_RMS, EPI_SWIGLU, h->wtype, c.batch, s, pdl)) != cudaSuccess) return e;
  }
  {  // gating[cb].linear_out + residual
    GemvParams p = base_params(h, h->p_dgout, mat(h, h->w.d_gate_out, ls * DD, DF));
    p.in = h->du;
    p.in_bs = DF;
    p.out = h->dx;
    p.out_bs = DD;
    if ((e = launch_gemv(p, PRO_PLAIN, EPI_RESID, h->wtype, c.batch, s, pdl)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t op_linear(const rq_handle* h, int cb, cudaStream_t s, bool pdl) {
  const rq_config& c = h->cfg;
  const size_t DD = c.ddim, A = c.audio_card;
  GemvParams p = base_params(h, h->p_lin, mat(h, h->w.linears, (size_t)cb * A, DD));
  p.in = h->dx;
  p.in_bs = DD;
  p.out = h->audio_logits + (size_t)cb * A;
  p.out_bs = 8 * A;
  p.key_index = 1 + cb;
  return launch_gemv(p, PRO_PLAIN, EPI_ARGMAX, h->wtype, c.batch, s, pdl);
}

FrameParams frame_params(const rq_handle* h) {
  FrameParams f{};
  f.B = h->cfg.batch;
  f.D = h->cfg.dim;
  f.V = h->cfg.text_card;
  f.A = h->cfg.audio_card;
  f.ring = h->ring;
  f.offsets = h->offsets;
  f.d_in = h->d_in;
  f.d_out = h->d_out_words();
  f.d_has = h->d_has();
  f.keys = h->keys;
  f.emb = h->w.emb;
  f.text_emb = h->w.text_emb;
  f.x = h->x;
  f.emb_sum = h->emb_sum;
  f.grid_bar = h->grid_bar;
  f.rope = h->rope;
  f.head_dim = h->cfg.head_dim;
  f.rope_theta = h->cfg.rope_theta;
  f.samp = h->samp;
  return f;
}

// One whole frame, in the page's order ("moshi_lm.rs", `step_ext` steps 1-8).
cudaError_t enqueue_frame(const rq_handle* h, cudaStream_t s, int sched) {
  cudaError_t e;
  const FrameParams f = frame_params(h);
  if ((e = launch_frame_begin(f, h->wes == 2, s)) != cudaSuccess) return e;
  if (sched == RQ_SCHEDULE_PERSISTENT) {
    if ((e = launch_persistent(h->pers, h->wtype, h->kvbf, h->pers_grid, h->pers_smem, s, true)) !=
        cudaSuccess)
      return e;
    if (h->pers_dep_grid > 0 && h->pers_dep.n_ops > 0 &&
        (e = launch_persistent(h->pers_dep, h->wtype, h->kvbf, h->pers_dep_grid,
                               h->pers_dep_smem, s, true, 1)) != cudaSuccess)
      return e;
    return launch_frame_end(f, s, true);
  }
  if (sched == RQ_SCHEDULE_TENSOR) {
    if ((e = tc_frame_enqueue(h->tcf, s)) != cudaSuccess) return e;
    return launch_frame_end(f, s, true);
  }
  for (int l = 0; l < h->cfg.layers; ++l) {
    if ((e = op_qkv(h, l, s, true)) != cudaSuccess) return e;
    if ((e = op_attn(h, l, s, true)) != cudaSuccess) return e;
    if ((e = op_out(h, l, s, true)) != cudaSuccess) return e;
    if ((e = op_gate_in(h, l, s, true)) != cudaSuccess) return e;
    if ((e = op_gate_out(h, l, s, true)) != cudaSuccess) return e;
  }
  const int B = h->cfg.batch, V = h->cfg.text_card, A = h->cfg.audio_card;
  const bool topk = h->samp.mode == SAMPLE_TOPK;
  if ((e = op_head(h, s, true)) != cudaSuccess) return e;
  if (topk && (e = launch_topk_pick(h->samp, h->text_logits, V, V, 0, h->keys, B, s, true)) !=
                  cudaSuccess)
    return e;
  for (int cb = 0; cb < 8; ++cb) {
    if ((e = op_dep_in(h, cb, s, true)) != cudaSuccess) return e;
    for (int l = 0; l < h->cfg.dlayers; ++l)
      if ((e = op_dlayer(h, cb, l, s, true)) != cudaSuccess) return e;
    if ((e = op_linear(h, cb, s, true)) != cudaSuccess) return e;
    if (topk && (e = launch_topk_pick(h->samp, h->audio_logits + (size_t)cb * A, 8ll * A, A,
                                      1 + cb, h->keys, B, s, true)) != cudaSuccess)
      return e;
  }
  return launch_frame_end(f, s, true);
}

}  // namespace

namespace {

void free_all(rq_handle* h) {
  if (h->exec) cudaGraphExecDestroy(h->exec);
  if (h->graph) cudaGraphDestroy(h->graph);
  if (h->exec_long) cudaGraphExecDestroy(h->exec_long);
  if (h->graph_long) cudaGraphDestroy(h->graph_long);
  void* dev[] = {h->ring, h->offsets, h->kcache, h->vcache, h->d_in, h->d_outb, h->x,
                 h->emb_sum, h->q, h->attn, h->u, h->tout, h->text_logits, h->audio_logits,
                 h->keys, h->dx, h->dq, h->dkv, h->du, h->part, h->counters, h->rng,
                 h->dep_pre,
                 h->xs_jump};
  for (void* p : dev)
    if (p) cudaFree(p);
  void* tcb[] = {h->rope, h->xb, h->attn_b, h->u_b, h->tout_b, h->dxb, h->do_b, h->du_b,
                 h->tc_part, h->tc_tickets, h->ss_x, h->ss_dx, h->dx_ll, h->dq_ll, h->du_ll,
                 h->dkv_ll, h->alog_ll, h->topk_scratch, h->key_ll};
  for (void* p : tcb)
    if (p) cudaFree(p);
  for (void* p : h->pf_bufs)
    if (p) cudaFree(p);
  if (h->d_ops) cudaFree(h->d_ops);
  if (h->grid_bar) cudaFree(h->grid_bar);
  if (h->trace) cudaFree(h->trace);
  if (h->h_in) cudaFreeHost(h->h_in);
  if (h->h_out) cudaFreeHost(h->h_out);
  if (h->cap) cudaStreamDestroy(h->cap);
}

template <typename T>
cudaError_t dalloc(T** p, size_t bytes) {
  return cudaMalloc(reinterpret_cast<void**>(p), bytes < 16 ? 16 : bytes);
}

rq_status plan_all(rq_handle* h, std::string* why) {
  const rq_config& c = h->cfg;
  const int es = h->wes, sms = h->num_sms, bd = h->band;
  h->p_qkv = plan_gemv(3 * c.dim, c.dim, es, false, true, sms, bd);
  h->p_out = plan_gemv(c.dim, c.dim, es, false, false, sms, bd);
  h->p_gin = plan_gemv(c.hidden, c.dim, es, true, false, sms, bd);
  h->p_gout = plan_gemv(c.dim, c.hidden, es, false, false, sms, bd);
  h->p_head = plan_gemv(c.text_card, c.dim, es, false, false, sms, bd);
  h->p_depin = plan_gemv(c.ddim, c.dim, es, false, false, sms, bd);
  h->p_dqkv = plan_gemv(3 * c.ddim, c.ddim, es, false, false, sms, bd);
  h->p_dout = plan_gemv(c.ddim, c.ddim, es, false, false, sms, bd);
  h->p_dgin = plan_gemv(c.dhidden, c.ddim, es, true, false, sms, bd);
  h->p_dgout = plan_gemv(c.ddim, c.dhidden, es, false, false, sms, bd);
  h->p_lin = plan_gemv(c.audio_card, c.ddim, es, false, false, sms, bd);
  const GemvPlan* all[] = {&h->p_qkv, &h->p_out, &h->p_gin, &h->p_gout, &h->p_head, &h->p_depin,
                           &h->p_dqkv, &h->p_dout, &h->p_dgin, &h->p_dgout, &h->p_lin};
  for (const GemvPlan* p : all) {
    if (gemv_chunks_per_thread(*p, es) > kGemvMaxChunks) {
      *why = "a reduction length is too long for the GEMV kernel";
      return RQ_ERR_UNSUPPORTED;
    }
    if (p->smem > 200 * 1024) {
      *why = "a GEMV tile does not fit in shared memory";
      return RQ_ERR_UNSUPPORTED;
    }
  }
  h->kps = 64;
  h->nsplit = (c.context + h->kps - 1) / h->kps;
  return RQ_OK;
}


// ---- persistent schedule: plans for one cooperative grid and the frame's op table
#ifndef RQ_PERS_SLOT_BUDGET
#define RQ_PERS_SLOT_BUDGET (96 * 1024)
#endif
constexpr int kPersSlotBudget = RQ_PERS_SLOT_BUDGET;
#ifndef RQ_PERS_DEP_SLOT_BUDGET
#define RQ_PERS_DEP_SLOT_BUDGET (192 * 1024)  // the depformer launch: one CTA per SM
#endif
constexpr int kPersDepSlotBudget = RQ_PERS_DEP_SLOT_BUDGET;
#ifndef RQ_PERS_DEP_FIT
#define RQ_PERS_DEP_FIT 1
#endif
constexpr bool kPersDepFit = RQ_PERS_DEP_FIT != 0;
// batch 1: windows longer than this run the one-kernel-per-op frame (see frame_exec)
constexpr int kLongWindow = 1350;
// 64-bit word index, inside the grid barriers' 512-byte allocation, of the persistent
// kernel's wait-control pair (see PersParams::wait_ctl)
constexpr int kWaitCtlWord = 16;

void pers_plans(const rq_handle* h, int G, GemvPlan* pl) {
  const rq_config& c = h->cfg;
  const int es = h->wes, bd = h->band;
  pl[0] = plan_persistent(3 * c.dim, c.dim, es, false, true, G, bd);
  pl[1] = plan_persistent(c.dim, c.dim, es, false, false, G, bd);
  pl[2] = plan_persistent(c.hidden, c.dim, es, true, false, G, bd);
  pl[3] = plan_persistent(c.dim, c.hidden, es, false, false, G, bd);
  pl[4] = plan_persistent(c.text_card, c.dim, es, false, false, G, bd);
  pl[5] = plan_persistent(c.ddim, c.dim, es, false, false, G, bd);
  pl[6] = plan_persistent(3 * c.ddim, c.ddim, es, false, false, G, bd);
  pl[7] = plan_persistent(c.ddim, c.ddim, es, false, false, G, bd);
  pl[8] = plan_persistent(c.dhidden, c.ddim, es, true, false, G, bd);
  pl[9] = plan_persistent(c.ddim, c.dhidden, es, false, false, G, bd);
  pl[10] = plan_persistent(c.audio_card, c.ddim, es, false, false, G, bd);
  pl[11] = plan_persistent(8 * c.ddim, c.dim, es, false, false, G, bd);
}
constexpr int kPersPlans = 12;

std::vector<PersOp> pers_ops(const rq_handle* h, int* dep_first) {
  const rq_config& c = h->cfg;
  const size_t D = c.dim, C = c.context, F = c.hidden, A = c.audio_card;
  const size_t DD = c.ddim, DF = c.dhidden;
  const int es = h->wes;
  std::vector<PersOp> ops;
  auto gemv = [](int pro, int epi, int plan, const void* W) {
    PersOp o{};
    o.type = OPT_GEMV;
    o.pro = pro;
    o.epi = epi;
    o.plan = plan;
    o.W = W;
    return o;
  };
  for (int l = 0; l < c.layers; ++l) {
    void* kc = static_cast<char*>(h->kcache) + (size_t)l * C * D * h->kves;
    void* vc = static_cast<char*>(h->vcache) + (size_t)l * C * D * h->kves;
    PersOp o = gemv(PRO_RMS, EPI_QKV, 0, mat(h, h->w.in_proj, (size_t)l * 3 * D, D));
    o.in = h->x;
    o.alpha = h->w.norm1 + (size_t)l * D;
    o.out = h->q;
    o.kcache = kc;
    o.vcache = vc;
    ops.push_back(o);
    PersOp a{};
    a.type = OPT_ATTN;
    a.kcache = kc;
    a.vcache = vc;
    ops.push_back(a);
    o = gemv(PRO_PLAIN, EPI_RESID, 1, mat(h, h->w.out_proj, (size_t)l * D, D));
    o.in = h->attn;
    o.out = h->x;
    ops.push_back(o);
    o = gemv(PRO_RMS, EPI_SWIGLU, 2, mat(h, h->w.gate_in, (size_t)l * 2 * F, D));
    o.w_half = (long long)(F * band_row_bytes(h->band, es, D));
    o.in = h->x;
    o.alpha = h->w.norm2 + (size_t)l * D;
    o.out = h->u;
    ops.push_back(o);
    o = gemv(PRO_PLAIN, EPI_RESID, 3, mat(h, h->w.gate_out, (size_t)l * D, F));
    o.in = h->u;
    o.out = h->x;
    ops.push_back(o);
  }
  PersOp hd = gemv(PRO_RMS, EPI_ARGMAX, 4, h->w.text_linear);
  hd.in = h->x;
  hd.alpha = h->w.out_norm;
  hd.side_out = h->tout;
  hd.out = h->text_logits;
  hd.key_index = 0;
  ops.push_back(hd);
  // the 8 steps' input projections dep_in[cb] . t at once, beside the text head: t is the
  // same out_norm(x), so this op needs no barrier after the head; each step's first
  // layer adds its embedding row E[prev] in its prologue
  PersOp da = gemv(PRO_RMS, EPI_STORE, 11, h->w.dep_in);
  da.in = h->x;
  da.alpha = h->w.out_norm;
  da.out = h->dep_pre;
  da.nobar = 1;
  ops.push_back(da);
  auto topk_op = [&](const float* logits, int p) {
    PersOp t{};
    t.type = OPT_TOPK;
    t.in = logits;
    t.key_index = p;
    ops.push_back(t);
  };
  const bool topk = h->samp.mode == SAMPLE_TOPK;
  if (topk) topk_op(h->text_logits, 0);
  if (dep_first) *dep_first = (int)ops.size();
  // The depformer launch exchanges tagged words (ll): its buffers are the tagged copies
  // and every op names the frame op indices whose tags it waits for.  Otherwise (one launch
  // for the whole frame) the plain buffers and grid barriers.
  const bool ll = h->pers_dep_grid > 0;
  auto L = [&](float* plain, float* tagged, size_t elem) -> float* {
    return ll ? reinterpret_cast<float*>(reinterpret_cast<unsigned long long*>(tagged) + elem)
              : plain + elem;
  };
  const int step_ops = 4 * c.dlayers + 1 + (topk ? 1 : 0);  // ops of one depformer step
  std::vector<int> dqkv0(c.dlayers, -1);  // frame op index of step 0's qkv, per layer
  int last_dx = -1, last_du = -1;        // last writer of dx / du
  int key_tag = -1, key_slots = 0;       // the op that chose the previous step's token
  for (int cb = 0; cb < 8; ++cb) {
    PersOp o{};
    for (int l = 0; l < c.dlayers; ++l) {
      const size_t ls = (size_t)l * 8 + cb;
      const int iq = (int)ops.size();
      if (cb == 0) dqkv0[l] = iq;
      o = gemv(l == 0 ? PRO_RMS_EMB : PRO_RMS, EPI_DQKV, 6,
               mat(h, h->w.d_in_proj, ls * 3 * DD, DD));
      o.in = L(h->dx, h->dx_ll, 0);
      o.tag_in = last_dx;
      if (l == 0) {  // x = dep_in[cb] . t + E[prev], kept in dx for the residuals
        o.in = h->dep_pre + (size_t)cb * DD;
        o.tag_in = -1;
        o.side_out = L(h->dx, h->dx_ll, 0);
        o.emb = cb == 0 ? h->w.dep_text_emb
                        : woff(h->w.dep_emb, (size_t)(cb - 1) * (A + 1) * DD, es);
        o.key_index = cb;
        o.tag_key = key_tag;
        o.key_slots = key_slots;
        last_dx = iq;
      }
      o.alpha = h->w.dnorm1 + (size_t)l * DD;
      o.out = L(h->dq, h->dq_ll, 0);
      o.dk_out = L(h->dkv, h->dkv_ll, dkv_off(h, l, 0, cb));
      o.dv_out = L(h->dkv, h->dkv_ll, dkv_off(h, l, 1, cb));
      ops.push_back(o);
      o = gemv(PRO_DATTN, EPI_RESID, 7, mat(h, h->w.d_out_proj, ls * DD, DD));
      o.in = L(h->dq, h->dq_ll, 0);
      o.tag_in = iq;
      o.dk = L(h->dkv, h->dkv_ll, dkv_off(h, l, 0, 0));
      o.dv = L(h->dkv, h->dkv_ll, dkv_off(h, l, 1, 0));
      o.tag_kv = dqkv0[l];
      o.tag_kv_step = step_ops;
      o.n_keys = cb + 1;
      o.out = L(h->dx, h->dx_ll, 0);
      o.tag_res = last_dx;
      last_dx = (int)ops.size();
      ops.push_back(o);
      o = gemv(PRO_RMS, EPI_SWIGLU, 8, mat(h, h->w.d_gate_in, ls * 2 * DF, DD));
      o.w_half = (long long)(DF * band_row_bytes(h->band, es, DD));
      o.in = L(h->dx, h->dx_ll, 0);
      o.tag_in = last_dx;
      o.alpha = h->w.dnorm2 + (size_t)l * DD;
      o.out = L(h->du, h->du_ll, 0);
      last_du = (int)ops.size();
      ops.push_back(o);
      o = gemv(PRO_PLAIN, EPI_RESID, 9, mat(h, h->w.d_gate_out, ls * DD, DF));
      o.in = L(h->du, h->du_ll, 0);
      o.tag_in = last_du;
      o.out = L(h->dx, h->dx_ll, 0);
      o.tag_res = last_dx;
      last_dx = (int)ops.size();
      ops.push_back(o);
    }
    o = gemv(PRO_PLAIN, EPI_ARGMAX, 10, mat(h, h->w.linears, (size_t)cb * A, DD));
    o.in = L(h->dx, h->dx_ll, 0);
    o.tag_in = last_dx;
    o.out = h->audio_logits + (size_t)cb * A;
    o.key_index = 1 + cb;
    if (ll && topk) {  // the pick reads the tagged copy and alone writes the key
      o.side_out = L(nullptr, h->alog_ll, (size_t)cb * A);
      o.no_keymax = 1;
    }
    key_tag = (int)ops.size();
    key_slots = h->pers_dep_grid;
    ops.push_back(o);
    if (topk) {
      topk_op(ll ? L(nullptr, h->alog_ll, (size_t)cb * A) : h->audio_logits + (size_t)cb * A,
              1 + cb);
      ops.back().tag_in = key_tag;
      key_tag = (int)ops.size() - 1;
      key_slots = 1;
    }
  }
  return ops;
}

// Decide the schedule; for the persistent one build plans, ring geometry and op table.
bool tensor_eligible(const rq_handle* h) {
  const rq_config& c = h->cfg;
  return h->wbf && c.batch >= 1 && c.batch <= 64 && c.dim % 64 == 0 && c.hidden % 64 == 0 &&
         c.ddim % 64 == 0 && c.dhidden % 64 == 0;
}

rq_status setup_tensor(rq_handle* h) {
  const rq_config& c = h->cfg;
  TcFrame& f = h->tcf;
  f = TcFrame{};
  f.B = c.batch;
  f.NB = (c.batch + 15) / 16 * 16;
  f.D = c.dim;
  f.L = c.layers;
  f.C = c.context;
  f.F = c.hidden;
  f.V = c.text_card;
  f.A = c.audio_card;
  f.DD = c.ddim;
  f.DL = c.dlayers;
  f.DF = c.dhidden;
  f.H = c.heads;
  f.hd = c.head_dim;
  f.dH = c.dheads;
  f.dhd = c.dhead_dim;
  f.eps = c.rms_eps;
  f.kv_bf16 = h->kvbf ? 1 : 0;
  const rq_weights& w = h->w;
  f.in_proj = w.in_proj;
  f.out_proj = w.out_proj;
  f.gate_in = w.gate_in;
  f.gate_out = w.gate_out;
  f.text_linear = w.text_linear;
  f.dep_in = w.dep_in;
  f.dep_text_emb = w.dep_text_emb;
  f.dep_emb = w.dep_emb;
  f.d_in_proj = w.d_in_proj;
  f.d_out_proj = w.d_out_proj;
  f.d_gate_in = w.d_gate_in;
  f.d_gate_out = w.d_gate_out;
  f.linears = w.linears;
  f.norm1 = w.norm1;
  f.norm2 = w.norm2;
  f.out_norm = w.out_norm;
  f.dnorm1 = w.dnorm1;
  f.dnorm2 = w.dnorm2;
  f.x = h->x;
  f.q = h->q;
  f.attn = h->attn;
  f.tout = h->tout;
  f.text_logits = h->text_logits;
  f.audio_logits = h->audio_logits;
  f.dx = h->dx;
  f.dq = h->dq;
  f.dkv = h->dkv;
  f.kcache = h->kcache;
  f.vcache = h->vcache;
  f.offsets = h->offsets;
  f.d_in = h->d_in;
  f.keys = h->keys;
  f.samp = h->samp;
  f.attn_part = h->part;
  f.attn_counters = h->counters;
  f.kps = h->kps;
  f.nsplit = h->nsplit;
  f.status = h->d_status();
  size_t part_floats = 0;
  int n_tickets = 0;
  tc_frame_plan(f, h->num_sms, &part_floats, &n_tickets);
  const size_t NB = f.NB;
  auto A_ = [&](void** p, size_t bytes, const char* what) -> rq_status {
    cudaError_t e = cudaMalloc(p, bytes < 16 ? 16 : bytes);
    if (e == cudaSuccess) e = cudaMemset(*p, 0, bytes < 16 ? 16 : bytes);
    if (e == cudaSuccess) return RQ_OK;
    h->err = std::string("allocation failed: ") + what + ": " + cudaGetErrorString(e);
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? RQ_ERR_OOM : RQ_ERR_CUDA;
  };
  rq_status st;
#define TC_ALLOC(ptr, bytes) \
  if ((st = A_(reinterpret_cast<void**>(&(ptr)), (bytes), #ptr)) != RQ_OK) return st;
  TC_ALLOC(h->rope, (size_t)c.batch * (c.head_dim / 2) * sizeof(float2));
  const size_t R = kOpndParts * NB;  // operands: [parts][NB][K]
  TC_ALLOC(h->xb, R * c.dim * 2);
  TC_ALLOC(h->attn_b, R * c.dim * 2);
  TC_ALLOC(h->u_b, R * c.hidden * 2);
  TC_ALLOC(h->tout_b, R * c.dim * 2);
  TC_ALLOC(h->dxb, R * c.ddim * 2);
  TC_ALLOC(h->do_b, R * c.ddim * 2);
  TC_ALLOC(h->du_b, R * c.dhidden * 2);
  TC_ALLOC(h->tc_part, part_floats * 4);
  TC_ALLOC(h->tc_tickets, (size_t)n_tickets * 4);
  TC_ALLOC(h->ss_x, (size_t)((c.dim + 127) / 128) * NB * 4);
  TC_ALLOC(h->ss_dx, (size_t)((c.ddim + 127) / 128) * NB * 4);
#undef TC_ALLOC
  f.rope = h->rope;
  f.xb = h->xb;
  f.attn_b = h->attn_b;
  f.u_b = h->u_b;
  f.tout_b = h->tout_b;
  f.dxb = h->dxb;
  f.do_b = h->do_b;
  f.du_b = h->du_b;
  f.part = h->tc_part;
  f.tickets = h->tc_tickets;
  f.ss_x = h->ss_x;
  f.ss_dx = h->ss_dx;
  f.n_wm = tc_frame_n_maps(f);
  h->tc_maps.assign((size_t)f.n_wm, CUtensorMap{});
  f.wm = h->tc_maps.data();
  cudaError_t e = tc_configure();
  if (e != cudaSuccess) return cuda_fail(h, e, "tc_configure");
  e = tc_frame_maps(f);
  if (e != cudaSuccess) return cuda_fail(h, e, "tensor map encoding");
  h->schedule = RQ_SCHEDULE_TENSOR;
  return RQ_OK;
}

constexpr int kPrefillCols = 64;

bool prefill_eligible(const rq_handle* h) {
  const rq_config& c = h->cfg;
  return h->wbf && c.dim % 64 == 0 && c.hidden % 64 == 0 && c.ddim % 64 == 0 &&
         c.dhidden % 64 == 0;
}

// the prefill frame: the tensor-core temporal layers over kPrefillCols columns, which
// are consecutive positions of one session (TcFrame::one_session); built on first use
rq_status setup_prefill(rq_handle* h) {
  if (h->pf_ready) return RQ_OK;
  const rq_config& c = h->cfg;
  TcFrame f{};
  f.B = kPrefillCols;
  f.NB = kPrefillCols;
  f.D = c.dim;
  f.L = c.layers;
  f.C = c.context;
  f.F = c.hidden;
  f.V = c.text_card;
  f.A = c.audio_card;
  f.DD = c.ddim;
  f.DL = c.dlayers;
  f.DF = c.dhidden;
  f.H = c.heads;
  f.hd = c.head_dim;
  f.dH = c.dheads;
  f.dhd = c.dhead_dim;
  f.eps = c.rms_eps;
  f.kv_bf16 = h->kvbf ? 1 : 0;
  const rq_weights& w = h->w;
  f.in_proj = w.in_proj;
  f.out_proj = w.out_proj;
  f.gate_in = w.gate_in;
  f.gate_out = w.gate_out;
  f.text_linear = w.text_linear;
  f.dep_in = w.dep_in;
  f.dep_text_emb = w.dep_text_emb;
  f.dep_emb = w.dep_emb;
  f.d_in_proj = w.d_in_proj;
  f.d_out_proj = w.d_out_proj;
  f.d_gate_in = w.d_gate_in;
  f.d_gate_out = w.d_gate_out;
  f.linears = w.linears;
  f.norm1 = w.norm1;
  f.norm2 = w.norm2;
  f.out_norm = w.out_norm;
  f.dnorm1 = w.dnorm1;
  f.dnorm2 = w.dnorm2;
  f.d_in = h->d_in;
  f.keys = h->keys;
  f.samp = h->samp;
  f.kps = h->kps;
  f.nsplit = h->nsplit;
  f.status = h->d_status();
  f.one_session = 1;
  size_t part_floats = 0;
  int n_tickets = 0;
  tc_frame_plan(f, h->num_sms, &part_floats, &n_tickets);
  const size_t NB = kPrefillCols, R = kOpndParts * NB;
  auto A_ = [&](void** p, size_t bytes, const char* what) -> rq_status {
    cudaError_t e = cudaMalloc(p, bytes < 16 ? 16 : bytes);
    if (e == cudaSuccess) e = cudaMemset(*p, 0, bytes < 16 ? 16 : bytes);
    if (e == cudaSuccess) {
      h->pf_bufs.push_back(*p);
      return RQ_OK;
    }
    h->err = std::string("allocation failed: ") + what + ": " + cudaGetErrorString(e);
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? RQ_ERR_OOM : RQ_ERR_CUDA;
  };
  rq_status st;
#define PF_ALLOC(ptr, bytes) \
  if ((st = A_(reinterpret_cast<void**>(&(ptr)), (bytes), #ptr)) != RQ_OK) return st;
  PF_ALLOC(f.x, NB * c.dim * 4);
  PF_ALLOC(f.q, NB * c.dim * 4);
  PF_ALLOC(f.attn, NB * c.dim * 4);
  PF_ALLOC(f.attn_part, NB * c.heads * (size_t)h->nsplit * (c.head_dim + 2) * 4);
  PF_ALLOC(f.attn_counters, NB * c.heads * 4);
  PF_ALLOC(f.rope, NB * (c.head_dim / 2) * sizeof(float2));
  PF_ALLOC(f.xb, R * c.dim * 2);
  PF_ALLOC(f.attn_b, R * c.dim * 2);
  PF_ALLOC(f.u_b, R * c.hidden * 2);
  PF_ALLOC(f.tout_b, R * c.dim * 2);
  PF_ALLOC(f.dxb, R * c.ddim * 2);
  PF_ALLOC(f.do_b, R * c.ddim * 2);
  PF_ALLOC(f.du_b, R * c.dhidden * 2);
  PF_ALLOC(f.part, part_floats * 4);
  PF_ALLOC(f.tickets, (size_t)n_tickets * 4);
  PF_ALLOC(f.ss_x, (size_t)((c.dim + 127) / 128) * NB * 4);
  PF_ALLOC(f.ss_dx, (size_t)((c.ddim + 127) / 128) * NB * 4);
  PF_ALLOC(h->pf_tokens, NB * kStreams * 4);
  PF_ALLOC(h->pf_pos, NB * 4);
  PF_ALLOC(h->pf_forced, NB * 9 * 4);
  PF_ALLOC(h->pf_user, NB * 8 * 4);
#undef PF_ALLOC
  f.offsets = h->pf_pos;
  f.n_wm = tc_frame_n_maps(f);
  h->pf_maps.assign((size_t)f.n_wm, CUtensorMap{});
  f.wm = h->pf_maps.data();
  cudaError_t e = tc_configure();
  if (e != cudaSuccess) return cuda_fail(h, e, "tc_configure");
  e = tc_frame_maps(f);
  if (e != cudaSuccess) return cuda_fail(h, e, "tensor map encoding");
  h->pf = f;
  h->pf_ready = true;
  return RQ_OK;
}

// T prompt steps of one session from the prefill frame's x (replay) or from forced and
// user codes already in the staging buffers (priming)
rq_status enqueue_prefill_chunk(rq_handle* h, int session, int T, bool priming) {
  const rq_config& c = h->cfg;
  PrefillParams pp{};
  pp.session = session;
  pp.T = T;
  pp.B = c.batch;
  pp.D = c.dim;
  pp.V = c.text_card;
  pp.A = c.audio_card;
  pp.head_dim = c.head_dim;
  pp.rope_theta = c.rope_theta;
  pp.ring = h->ring;
  pp.offsets = h->offsets;
  pp.forced = priming ? h->pf_forced : nullptr;
  pp.user = h->pf_user;
  pp.tokens = h->pf_tokens;
  pp.pos = h->pf_pos;
  pp.rope = h->pf.rope;
  pp.emb = h->w.emb;
  pp.text_emb = h->w.text_emb;
  pp.x = h->pf.x;
  RQ_CUDA(h, launch_prefill_begin(pp, h->wbf, h->stream));
  TcFrame f = h->pf;
  f.B = T;
  const size_t sess = (size_t)session * c.layers * c.context * c.dim * h->kves;
  f.kcache = static_cast<char*>(h->kcache) + sess;
  f.vcache = static_cast<char*>(h->vcache) + sess;
  RQ_CUDA(h, tc_frame_enqueue_temporal(f, h->stream));
  h->host_off[session] += T;
  return RQ_OK;
}

// positions of the next chunk: up to kPrefillCols, but a chunk of more than one column
// must not wrap the window (a later column would overwrite a slot an earlier one reads)
int prefill_chunk(const rq_handle* h, int session, int left) {
  const int C = h->cfg.context, off = h->host_off[session];
  int T = left < kPrefillCols ? left : kPrefillCols;
  if (T > 1 && off + T > C) T = C - off > 1 ? C - off : 1;
  return T;
}

// the persistent kernel's op table for the current sampler (top-k adds a pick after the
// text head and after each linears[cb]); the op timeline has room for both tables
rq_status upload_pers_ops(rq_handle* h) {
  int dep_first = 0;
  std::vector<PersOp> ops = pers_ops(h, &dep_first);
  if (h->dx_ll) {
    // a new op table renumbers the ops: clear every tagged word, so that no word written
    // under the old numbering can carry a tag the new one waits for (words of the current
    // numbering are rewritten every frame, and a tag's 22-bit epoch only repeats after
    // 4 M frames)
    const rq_config& c = h->cfg;
    const size_t DD = c.ddim, DF = c.dhidden, A = c.audio_card, DL = c.dlayers;
    RQ_CUDA(h, cudaMemsetAsync(h->dx_ll, 0, DD * 8, h->stream));
    RQ_CUDA(h, cudaMemsetAsync(h->dq_ll, 0, DD * 8, h->stream));
    RQ_CUDA(h, cudaMemsetAsync(h->du_ll, 0, DF * 8, h->stream));
    RQ_CUDA(h, cudaMemsetAsync(h->dkv_ll, 0, DL * 2 * 8 * DD * 8, h->stream));
    RQ_CUDA(h, cudaMemsetAsync(h->alog_ll, 0, 8 * A * 8, h->stream));
    RQ_CUDA(h, cudaMemsetAsync(h->key_ll, 0, (size_t)9 * h->pers_dep_grid * 16, h->stream));
    RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  }
  if (h->d_ops) {
    cudaFree(h->d_ops);
    h->d_ops = nullptr;
  }
  RQ_CUDA(h, cudaMalloc(reinterpret_cast<void**>(&h->d_ops), ops.size() * sizeof(PersOp)));
  RQ_CUDA(h, cudaMemcpy(h->d_ops, ops.data(), ops.size() * sizeof(PersOp), cudaMemcpyHostToDevice));
  if (!h->trace) {
    const size_t n = ops.size() + (h->samp.mode == SAMPLE_TOPK ? 1 : 10);
    RQ_CUDA(h, cudaMalloc(reinterpret_cast<void**>(&h->trace), n * 8));
    RQ_CUDA(h, cudaMemset(h->trace, 0, n * 8));
  }
  const int n = (int)ops.size();
  h->pers_split = h->pers_dep_grid > 0 ? dep_first : n;
  h->pers.ops = h->d_ops;
  h->pers.n_ops = h->pers_split;
  h->pers.op_base = 0;
  h->pers_dep.ops = h->d_ops + h->pers_split;
  h->pers_dep.n_ops = n - h->pers_split;
  h->pers_dep.op_base = h->pers_split;
  h->pers_dep.trace = h->trace;
  h->pers_dep.samp = h->samp;
  h->pers_nobar.assign(ops.size(), 0);
  for (size_t k = 0; k < ops.size(); ++k) h->pers_nobar[k] = ops[k].nobar ? 1 : 0;
  // the depformer launch's first op waits for nothing (the first launch has finished)
  if (h->pers_split < n) h->pers_nobar[h->pers_split] = 1;
  h->pers.trace = h->trace;
  h->pers.samp = h->samp;
  return RQ_OK;
}

rq_status setup_schedule(rq_handle* h) {
  const rq_config& c = h->cfg;
  if (c.schedule == RQ_SCHEDULE_TENSOR ||
      (c.schedule == RQ_SCHEDULE_AUTO && c.batch >= 2 && tensor_eligible(h))) {
    if (!tensor_eligible(h))
      return fail(h, RQ_ERR_UNSUPPORTED,
                  "the tensor schedule needs batch <= 64, bf16 weights and dim, hidden, ddim, "
                  "dhidden multiples of 64");
    return setup_tensor(h);
  }
  // batch 1; f32 or bf16 weights with K/V of the same type, or a weight band (bf16 K/V,
  // head_dim 64 or 128)
  const bool can = c.batch == 1 &&
                   (h->band == BAND_NONE ? h->wbf == h->kvbf
                                         : h->kvbf && (c.head_dim == 64 || c.head_dim == 128));
  // weight bands run on the persistent kernel only when asked for: on Moshi-7B at batch 1
  // its band tiles take 4.85 (q8) / 7.16 ms (q4) per frame, the graph schedule 4.08 / 4.07
  if (c.schedule == RQ_SCHEDULE_AUTO && h->band != BAND_NONE) {
    h->schedule = RQ_SCHEDULE_GRAPH;
    return RQ_OK;
  }
  if (c.schedule == RQ_SCHEDULE_GRAPH || (c.schedule == RQ_SCHEDULE_AUTO && !can)) {
    h->schedule = RQ_SCHEDULE_GRAPH;
    return RQ_OK;
  }
  if (!can)
    return fail(h, RQ_ERR_UNSUPPORTED,
                "the persistent schedule needs batch 1 and f32 or bf16 weights of the K/V "
                "dtype, or a weight band with bf16 K/V and head_dim 64 or 128");
  GemvPlan pl[kPersMaxPlans];
  int G = 2 * h->num_sms, slot = 0, part = 0, ns = 0, smem = 0;
  // plans for a grid of G CTAs and the ring geometry of a shared-memory budget
  // (dep: the depformer launch, whose ops use plans 6..10 -- its slots are sized by its
  // own tiles, not the temporal ones)
  auto geometry = [&](int grid, int budget, GemvPlan* p, int& sl, int& pa, int& n, int& sm,
                      bool dep) -> bool {
    pers_plans(h, grid, p);
    sl = 0;
    pa = 0;
    for (int i = 0; i < kPersPlans; ++i) {
      if (p[i].nch == 0) return false;
      if (kPersDepFit && dep && (i < 6 || i > 10)) continue;
      const int tb = p[i].tile_rows * (int)band_row_bytes(h->band, h->wes, p[i].kp_width);
      sl = tb > sl ? tb : sl;
      const int pf = (p[i].max_tiles * p[i].tile_rows * (p[i].tpr / 32) + 3) & ~3;
      pa = pf > pa ? pf : pa;
    }
    // the partial-sum buffer also holds a top-k pick's scratch
    const int topk_floats = (int)((sizeof(TopkShared) + 15) / 16 * 4);
    pa = pa > topk_floats ? pa : topk_floats;
    sl = (sl + 127) & ~127;
    n = budget / sl;
    if (n < 2) n = 2;
    sm = n * sl + pa * 4 + 2 * n * 8;
    return true;
  };
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (!geometry(G, kPersSlotBudget, pl, slot, part, ns, smem, false))
      return fail(h, RQ_ERR_UNSUPPORTED, "GEMV shape unsupported");
    cudaError_t e = persistent_configure(h->wtype, h->kvbf, smem, c.head_dim, 2);
    if (e != cudaSuccess) return cuda_fail(h, e, "persistent_configure");
    const int maxg = persistent_max_grid(h->wtype, h->kvbf, smem, c.head_dim, 2);
    if (maxg >= G) break;
    if (attempt == 1 || maxg < h->num_sms) {
      if (c.schedule == RQ_SCHEDULE_PERSISTENT)
        return fail(h, RQ_ERR_UNSUPPORTED, "the persistent grid does not fit on this device");
      h->schedule = RQ_SCHEDULE_GRAPH;
      return RQ_OK;
    }
    G = h->num_sms;
  }
  RQ_CUDA(h, cudaMalloc(reinterpret_cast<void**>(&h->grid_bar), 512));
  RQ_CUDA(h, cudaMemset(h->grid_bar, 0, 512));
  PersParams& P = h->pers;
  P = PersParams{};
  for (int i = 0; i < kPersPlans; ++i) P.plans[i] = pl[i];
  P.slot_bytes = slot;
  P.n_slots = ns;
  P.part_floats = part;
  P.eps = c.rms_eps;
  P.kv_bf16 = h->kvbf ? 1 : 0;
  P.head_dim = c.head_dim;
  P.context = c.context;
  P.rope_theta = c.rope_theta;
  P.dheads = c.dheads;
  P.dhead_dim = c.dhead_dim;
  P.offsets = h->offsets;
  P.keys = h->keys;
  P.d_in = h->d_in;
  P.attn_q = h->q;
  P.attn_out = h->attn;
  P.part = h->part;
  P.counters = h->counters;
  P.D = c.dim;
  P.H = c.heads;
  P.kps = 16;  // shortest split; the kernel sizes splits from the window (16..64)
  P.nsplit = (c.context + 15) / 16;
  P.grid_bar = h->grid_bar;
  // the wait-control words live in the same 512-byte allocation, zero = defaults
  P.wait_ctl = reinterpret_cast<const unsigned long long*>(h->grid_bar) + kWaitCtlWord;
  P.status = h->d_status();
  h->pers_grid = G;
  h->pers_smem = smem;
  // The depformer's ops as a second cooperative launch at one CTA per SM: its small ops
  // are latency-bound, and a 152-CTA grid barrier, a register budget without spills and a
  // ring twice as deep run them faster (Moshi-7B: 1.29 -> 1.12 ms per frame), while the
  // temporal stack keeps two CTAs per SM to stream its weights.  Its ops wait for tagged
  // words instead of grid barriers (frame op indices must fit a tag's 10 bits: at most
  // 5 L + 3 + 8 (4 DL + 2) ops).  If that launch does not fit, the frame runs on the graph
  // schedule (the two-CTA kernel carries no depformer op).
  h->pers_dep_grid = 0;
  {
    GemvPlan pl2[kPersMaxPlans];
    int slot2 = 0, part2 = 0, ns2 = 0, smem2 = 0;
    const int G2 = h->num_sms;
    const int max_ops = 5 * c.layers + 3 + 8 * (4 * c.dlayers + 2);
    if (G == 2 * h->num_sms && max_ops < kPersMaxTaggedOps && G2 <= kPersMaxKeySlots &&
        geometry(G2, kPersDepSlotBudget, pl2, slot2, part2, ns2, smem2, true) &&
        persistent_configure(h->wtype, h->kvbf, smem2, c.head_dim, 1) == cudaSuccess &&
        persistent_max_grid(h->wtype, h->kvbf, smem2, c.head_dim, 1) >= G2) {
      PersParams& Q = h->pers_dep;
      Q = P;
      for (int i = 0; i < kPersPlans; ++i) Q.plans[i] = pl2[i];
      Q.slot_bytes = slot2;
      Q.n_slots = ns2;
      Q.part_floats = part2;
      Q.grid_bar = h->grid_bar + kPersDepBarWord;
      h->pers_dep_grid = G2;
      h->pers_dep_smem = smem2;
    }
    cudaGetLastError();  // a refused configuration leaves no sticky error
  }
  if (h->pers_dep_grid == 0) {
    // the two-CTA launch runs no depformer op: without the depformer's launch the frame
    // runs on the graph schedule
    if (c.schedule == RQ_SCHEDULE_PERSISTENT)
      return fail(h, RQ_ERR_UNSUPPORTED, "the persistent depformer launch does not fit on this device");
    h->schedule = RQ_SCHEDULE_GRAPH;
    return RQ_OK;
  }
  {
    const size_t DD = c.ddim, DF = c.dhidden, A = c.audio_card, DL = c.dlayers;
    RQ_CUDA(h, dalloc(&h->dx_ll, DD * 8));
    RQ_CUDA(h, dalloc(&h->dq_ll, DD * 8));
    RQ_CUDA(h, dalloc(&h->du_ll, DF * 8));
    RQ_CUDA(h, dalloc(&h->dkv_ll, DL * 2 * 8 * DD * 8));
    RQ_CUDA(h, dalloc(&h->alog_ll, 8 * A * 8));
    RQ_CUDA(h, dalloc(&h->topk_scratch, A * 4));
    RQ_CUDA(h, dalloc(&h->key_ll, (size_t)9 * h->pers_dep_grid * 16));
    // (upload_pers_ops zeroes them: tag 0 is never a frame's, the first frame advances
    // the epoch to 1)
    P.epoch = h->grid_bar + kPersEpochWord;
    P.epoch_bump = 1;
    PersParams& Q = h->pers_dep;
    Q.epoch = P.epoch;
    Q.epoch_bump = 0;
    Q.key_ll = h->key_ll;
    Q.topk_scratch = h->topk_scratch;
  }
  h->schedule = RQ_SCHEDULE_PERSISTENT;
  return upload_pers_ops(h);
}

rq_status capture_frame(rq_handle* h);

rq_status create_impl(rq_handle* h) {
  const rq_config& c = h->cfg;
  const size_t B = c.batch, D = c.dim, L = c.layers, C = c.context, F = c.hidden;
  const size_t V = c.text_card, A = c.audio_card, DD = c.ddim, DL = c.dlayers, DF = c.dhidden;
  RQ_CUDA(h, cudaGetDevice(&h->device));
  RQ_CUDA(h, cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device));
  std::string why;
  rq_status st = plan_all(h, &why);
  if (st != RQ_OK) return fail(h, st, why);
  RQ_CUDA(h, gemv_configure_all());
  RQ_CUDA(h, attn_configure(c.head_dim, h->kvbf, h->kps));
  RQ_CUDA(h, cudaStreamCreateWithFlags(&h->cap, cudaStreamNonBlocking));
  auto A_ = [&](cudaError_t e, const char* what) -> rq_status {
    if (e == cudaSuccess) return RQ_OK;
    h->err = std::string("allocation failed: ") + what + ": " + cudaGetErrorString(e);
    cudaGetLastError();
    return e == cudaErrorMemoryAllocation ? RQ_ERR_OOM : RQ_ERR_CUDA;
  };
#define RQ_ALLOC(ptr, bytes)                                   \
  if ((st = A_(dalloc(&(ptr), (bytes)), #ptr)) != RQ_OK) return st;
  RQ_ALLOC(h->ring, B * kStreams * kRing * 4);
  RQ_ALLOC(h->offsets, B * 4);
  RQ_ALLOC(h->kcache, B * L * C * D * h->kves);
  RQ_ALLOC(h->vcache, B * L * C * D * h->kves);
  RQ_ALLOC(h->d_in, h->io.in_words() * 4);
  RQ_ALLOC(h->d_outb, h->io.out_bytes());
  RQ_ALLOC(h->x, B * D * 4);
  RQ_ALLOC(h->emb_sum, B * D * 4);
  RQ_ALLOC(h->q, B * D * 4);
  RQ_ALLOC(h->attn, B * D * 4);
  RQ_ALLOC(h->u, B * F * 4);
  RQ_ALLOC(h->tout, B * D * 4);
  RQ_ALLOC(h->text_logits, B * V * 4);
  RQ_ALLOC(h->audio_logits, B * 8 * A * 4);
  RQ_ALLOC(h->keys, B * 9 * 8);
  RQ_ALLOC(h->rng, B * 8);
  RQ_ALLOC(h->xs_jump, (size_t)kXsLevels * 64 * 8);
  {  // greedy until rq_set_sampling; the page's `Sampling` defaults otherwise
    std::vector<uint64_t> table((size_t)kXsLevels * 64), ones(B, 1ull);
    xorshift_jump_table(table.data());
    RQ_CUDA(h, cudaMemcpy(h->xs_jump, table.data(), table.size() * 8, cudaMemcpyHostToDevice));
    RQ_CUDA(h, cudaMemcpy(h->rng, ones.data(), B * 8, cudaMemcpyHostToDevice));
    h->samp = SampleParams{};
    h->samp.mode = SAMPLE_GREEDY;
    h->samp.temp = 0.8f;
    h->samp.temp_text = 0.7f;
    h->samp.top_k = 250;
    h->samp.top_k_text = 25;
    h->samp.V = (int)V;
    h->samp.A = (int)A;
    h->samp.rng = h->rng;
    h->samp.jump = h->xs_jump;
  }
  RQ_ALLOC(h->dx, B * DD * 4);
  RQ_ALLOC(h->dep_pre, B * 8 * DD * 4);
  RQ_ALLOC(h->dq, B * DD * 4);
  RQ_ALLOC(h->dkv, B * DL * 2 * 8 * DD * 4);
  RQ_ALLOC(h->du, B * DF * 4);
  {  // attention partials: [B][H][nsplit] at 64 positions per split, or one session's
     // [H][ceil(C / 16)] for the persistent schedule's shorter splits
    const size_t n64 = B * (size_t)c.heads * h->nsplit, n16 = (size_t)c.heads * ((C + 15) / 16);
    RQ_ALLOC(h->part, (n64 > n16 ? n64 : n16) * (c.head_dim + 2) * 4);
  }
  RQ_ALLOC(h->counters, B * (size_t)c.heads * 4);
#undef RQ_ALLOC
  if ((st = A_(cudaMallocHost(reinterpret_cast<void**>(&h->h_in), h->io.in_words() * 4), "h_in")) != RQ_OK)
    return st;
  if ((st = A_(cudaMallocHost(reinterpret_cast<void**>(&h->h_out), h->io.out_bytes()), "h_out")) != RQ_OK)
    return st;
  std::memset(h->h_in, 0, h->io.in_words() * 4);
  // fresh sessions, zeroed scratch, cleared status
  RQ_CUDA(h, cudaMemsetAsync(h->counters, 0, B * (size_t)c.heads * 4, h->cap));
  RQ_CUDA(h, cudaMemsetAsync(h->d_outb, 0, h->io.out_bytes(), h->cap));
  RQ_CUDA(h, cudaMemsetAsync(h->d_in, 0, h->io.in_words() * 4, h->cap));
  RQ_CUDA(h, cudaMemsetAsync(h->keys, 0, B * 9 * 8, h->cap));
  RQ_CUDA(h, launch_reset(h->ring, h->offsets, (int)B, -1, h->cap));
  RQ_CUDA(h, cudaStreamSynchronize(h->cap));
  h->host_off.assign(B, 0);
  if ((st = setup_schedule(h)) != RQ_OK) return st;
  return capture_frame(h);
}

// capture one frame as a graph (programmatic edges between consecutive kernels),
// replacing the previous one
// Capture one frame of schedule `sched` into (graph, exec), replacing what was there.
rq_status capture_one(rq_handle* h, int sched, cudaGraph_t* graph, cudaGraphExec_t* exec) {
  if (*exec) {
    cudaGraphExecDestroy(*exec);
    *exec = nullptr;
  }
  if (*graph) {
    cudaGraphDestroy(*graph);
    *graph = nullptr;
  }
  RQ_CUDA(h, cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeThreadLocal));
  cudaError_t e = enqueue_frame(h, h->cap, sched);
  cudaGraph_t g = nullptr;
  cudaError_t e2 = cudaStreamEndCapture(h->cap, &g);
  if (e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return cuda_fail(h, e, "frame capture");
  }
  if (e2 != cudaSuccess) return cuda_fail(h, e2, "cudaStreamEndCapture");
  *graph = g;
  RQ_CUDA(h, cudaGraphInstantiate(exec, *graph, 0));
  RQ_CUDA(h, cudaGraphUpload(*exec, h->stream));
  return RQ_OK;
}

rq_status capture_frame(rq_handle* h) {
  rq_status st = capture_one(h, h->schedule, &h->graph, &h->exec);
  if (st != RQ_OK) return st;
  size_t n = 0;
  RQ_CUDA(h, cudaGraphGetNodes(h->graph, nullptr, &n));
  std::vector<cudaGraphNode_t> nodes(n);
  RQ_CUDA(h, cudaGraphGetNodes(h->graph, nodes.data(), &n));
  int k = 0;
  for (size_t i = 0; i < n; ++i) {
    cudaGraphNodeType t;
    RQ_CUDA(h, cudaGraphNodeGetType(nodes[i], &t));
    if (t == cudaGraphNodeTypeKernel) ++k;
  }
  h->n_kernels = k;
  if (h->schedule == RQ_SCHEDULE_PERSISTENT && h->cfg.context > kLongWindow)
    return capture_one(h, RQ_SCHEDULE_GRAPH, &h->graph_long, &h->exec_long);
  return RQ_OK;
}

// The graph of the next frame.  At batch 1 the persistent kernel's attention keeps one
// key per warp in flight, so its cost grows with the window faster than the split-K
// attention kernel of the one-kernel-per-op frame, which streams K/V at the HBM rate.
// Measured at the Moshi-7B shape: 4.39 / 4.61 ms per frame (persistent / per op) at a
// 1000-position window, 4.78 / 4.69 ms at 1500, 5.26 / 4.99 ms at 2900.  Both frames
// compute the same step on the same buffers.
cudaGraphExec_t frame_exec(const rq_handle* h) {
  if (h->exec_long) {
    const int len = std::min(h->host_off[0] + 1, h->cfg.context);
    if (len > kLongWindow) return h->exec_long;
  }
  return h->exec;
}

}  // namespace

extern "C" {

rq_status rq_create(const rq_config* cfg, const rq_weights* w, void* cuda_stream,
                    rq_handle** out) {
  if (!out) return RQ_ERR_ARG;
  *out = nullptr;
  if (!cfg || !w) return RQ_ERR_ARG;
  std::string why;
  rq_status st = validate_config(cfg, &why);
  if (st != RQ_OK) {
    g_create_err = why;
    return st;
  }
  const void* ptrs[] = {w->emb, w->text_emb, w->norm1, w->in_proj, w->out_proj, w->norm2,
                        w->gate_in, w->gate_out, w->out_norm, w->text_linear, w->dep_in,
                        w->dep_text_emb, w->dep_emb, w->dnorm1, w->dnorm2, w->d_in_proj,
                        w->d_out_proj, w->d_gate_in, w->d_gate_out, w->linears};
  for (const void* p : ptrs)
    if (!aligned16(p)) {
      g_create_err = "a weight pointer is NULL or not 16-byte aligned";
      return RQ_ERR_ARG;
    }
  rq_handle* h = new (std::nothrow) rq_handle();
  if (!h) return RQ_ERR_OOM;
  h->cfg = *cfg;
  h->w = *w;
  h->stream = static_cast<cudaStream_t>(cuda_stream);
  h->wbf = cfg->weight_dtype == RQ_BF16;
  h->kvbf = cfg->kv_dtype == RQ_BF16;
  h->band = cfg->weight_dtype == RQ_Q8 ? BAND_Q8 : (cfg->weight_dtype == RQ_Q4 ? BAND_Q4 : BAND_NONE);
  h->wtype = h->band != BAND_NONE ? h->band : (h->wbf ? 1 : 0);
  h->wes = (h->wbf || h->band != BAND_NONE) ? 2 : 4;
  h->kves = h->kvbf ? 2 : 4;
  h->io = IoLayout{cfg->batch};
  st = create_impl(h);
  if (st != RQ_OK) {
    g_create_err = h->err;
    free_all(h);
    delete h;
    return st;
  }
  *out = h;
  return RQ_OK;
}

void rq_destroy(rq_handle* h) {
  if (!h) return;
  cudaStreamSynchronize(h->stream);
  free_all(h);
  delete h;
}

}  // extern "C"

namespace {

rq_status check_usable(rq_handle* h) {
  if (!h) return RQ_ERR_ARG;
  if (h->poisoned) return RQ_ERR_POISONED;
  return RQ_OK;
}

// read the status word of the last frame (already copied to h_out) and poison on error
rq_status absorb_status(rq_handle* h, uint32_t status) {
  if (status == 0) return RQ_OK;
  h->poisoned = true;
  if (status & kDevTimeout) {
    h->err = "a bounded device-side wait timed out";
    return RQ_ERR_TIMEOUT;
  }
  h->err = "device reported bad input";
  return RQ_ERR_CUDA;
}

rq_status run_frame_host(rq_handle* h, const int32_t* user, const int32_t* forced,
                         int32_t* own, int32_t* out_tokens, uint8_t* has_output) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  const rq_config& c = h->cfg;
  const int B = c.batch;
  if (!user) return fail(h, RQ_ERR_ARG, "user_tokens is NULL");
  for (int i = 0; i < B * 8; ++i)
    if (user[i] < -1 || user[i] > c.audio_card)
      return fail(h, RQ_ERR_TOKEN, "user token outside [-1, audio_card]");
  if (forced) {
    for (int b = 0; b < B; ++b) {
      if (forced[b * 9] < 0 || forced[b * 9] >= c.text_card)
        return fail(h, RQ_ERR_TOKEN, "forced text token outside [0, text_card)");
      for (int k = 1; k < 9; ++k)
        if (forced[b * 9 + k] < 0 || forced[b * 9 + k] >= c.audio_card)
          return fail(h, RQ_ERR_TOKEN, "forced audio token outside [0, audio_card)");
    }
  }
  const IoLayout& io = h->io;
  std::memcpy(h->h_in + io.user_off(), user, (size_t)B * 8 * 4);
  if (forced) {
    std::memcpy(h->h_in + io.forced_off(), forced, (size_t)B * 9 * 4);
    for (int b = 0; b < B; ++b) h->h_in[io.flag_off() + b] = 1;
  } else {
    for (int b = 0; b < B; ++b) h->h_in[io.flag_off() + b] = 0;
  }
  RQ_CUDA(h, cudaMemcpyAsync(h->d_in, h->h_in, io.in_words() * 4, cudaMemcpyHostToDevice, h->stream));
  h->forcing_dirty = forced != nullptr;
  RQ_CUDA(h, cudaGraphLaunch(frame_exec(h), h->stream));
  RQ_CUDA(h, cudaMemcpyAsync(h->h_out, h->d_outb, io.out_bytes(), cudaMemcpyDeviceToHost, h->stream));
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  for (int b = 0; b < B; ++b) h->host_off[b] += 1;
  uint32_t status;
  std::memcpy(&status, h->h_out + io.status_off_bytes(), 4);
  if ((st = absorb_status(h, status)) != RQ_OK) return st;
  const int32_t* words = reinterpret_cast<const int32_t*>(h->h_out);
  if (own) std::memcpy(own, words + io.own_off(), (size_t)B * 9 * 4);
  if (out_tokens) std::memcpy(out_tokens, words + io.out_off(), (size_t)B * 9 * 4);
  if (has_output) std::memcpy(has_output, h->h_out + io.has_off_bytes(), (size_t)B);
  return RQ_OK;
}

}  // namespace

extern "C" {

rq_status rq_step(rq_handle* h, const int32_t* user_tokens, int32_t* out_tokens,
                  uint8_t* has_output) {
  return run_frame_host(h, user_tokens, nullptr, nullptr, out_tokens, has_output);
}

rq_status rq_step_forced(rq_handle* h, const int32_t* user_tokens, const int32_t* forced,
                         int32_t* own_tokens, int32_t* out_tokens, uint8_t* has_output) {
  if (!forced) return fail(h, RQ_ERR_ARG, "forced is NULL");
  return run_frame_host(h, user_tokens, forced, own_tokens, out_tokens, has_output);
}

rq_status rq_step_device(rq_handle* h, const int32_t* d_user, int32_t* d_out_tokens,
                         uint8_t* d_has_output) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  if (!d_user) return fail(h, RQ_ERR_ARG, "d_user is NULL");
  const IoLayout& io = h->io;
  const int B = h->cfg.batch;
  RQ_CUDA(h, cudaMemcpyAsync(h->d_in + io.user_off(), d_user, (size_t)B * 8 * 4,
                             cudaMemcpyDeviceToDevice, h->stream));
  if (h->forcing_dirty) {
    RQ_CUDA(h, cudaMemsetAsync(h->d_in + io.flag_off(), 0, (size_t)B * 4, h->stream));
    h->forcing_dirty = false;
  }
  RQ_CUDA(h, cudaGraphLaunch(frame_exec(h), h->stream));
  if (d_out_tokens)
    RQ_CUDA(h, cudaMemcpyAsync(d_out_tokens, h->d_out_words() + io.out_off(), (size_t)B * 9 * 4,
                               cudaMemcpyDeviceToDevice, h->stream));
  if (d_has_output)
    RQ_CUDA(h, cudaMemcpyAsync(d_has_output, h->d_has(), (size_t)B, cudaMemcpyDeviceToDevice,
                               h->stream));
  for (int b = 0; b < B; ++b) h->host_off[b] += 1;
  return RQ_OK;
}

rq_status rq_sync(rq_handle* h) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  uint32_t status = 0;
  RQ_CUDA(h, cudaMemcpy(&status, h->d_status(), 4, cudaMemcpyDeviceToHost));
  return absorb_status(h, status);
}

rq_status rq_get_logits(rq_handle* h, float* text, float* audio) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  const rq_config& c = h->cfg;
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  if (text)
    RQ_CUDA(h, cudaMemcpy(text, h->text_logits, (size_t)c.batch * c.text_card * 4, cudaMemcpyDeviceToHost));
  if (audio)
    RQ_CUDA(h, cudaMemcpy(audio, h->audio_logits, (size_t)c.batch * 8 * c.audio_card * 4,
                          cudaMemcpyDeviceToHost));
  return RQ_OK;
}

rq_status rq_get_trace(rq_handle* h, float* emb_sum, float* transformer_out) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  const size_t n = (size_t)h->cfg.batch * h->cfg.dim * 4;
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  if (emb_sum) RQ_CUDA(h, cudaMemcpy(emb_sum, h->emb_sum, n, cudaMemcpyDeviceToHost));
  if (transformer_out) RQ_CUDA(h, cudaMemcpy(transformer_out, h->tout, n, cudaMemcpyDeviceToHost));
  return RQ_OK;
}

rq_status rq_get_ring(rq_handle* h, int32_t* ring, int32_t* offsets) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  const int B = h->cfg.batch;
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  if (ring) RQ_CUDA(h, cudaMemcpy(ring, h->ring, (size_t)B * kStreams * kRing * 4, cudaMemcpyDeviceToHost));
  if (offsets) RQ_CUDA(h, cudaMemcpy(offsets, h->offsets, (size_t)B * 4, cudaMemcpyDeviceToHost));
  return RQ_OK;
}

rq_status rq_reset(rq_handle* h, int32_t session) {
  if (!h) return RQ_ERR_ARG;
  const int B = h->cfg.batch;
  if (session < -1 || session >= B) return fail(h, RQ_ERR_ARG, "session out of range");
  if (h->poisoned && session != -1) return RQ_ERR_POISONED;
  if (session == -1) {
    // clear the sticky CUDA error state of this thread, then every scratch word
    cudaGetLastError();
    RQ_CUDA(h, cudaStreamSynchronize(h->stream));
    RQ_CUDA(h, cudaMemsetAsync(h->d_outb, 0, h->io.out_bytes(), h->stream));
    RQ_CUDA(h, cudaMemsetAsync(h->counters, 0, (size_t)B * h->cfg.heads * 4, h->stream));
    RQ_CUDA(h, cudaMemsetAsync(h->keys, 0, (size_t)B * 9 * 8, h->stream));
  }
  RQ_CUDA(h, launch_reset(h->ring, h->offsets, B, session, h->stream));
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  for (int b = 0; b < B; ++b)
    if (session == -1 || b == session) h->host_off[b] = 0;
  if (session == -1) {
    h->poisoned = false;
    h->err.clear();
  }
  return RQ_OK;
}

rq_status rq_set_kv(rq_handle* h, int32_t session, int32_t n_pos, const void* k, const void* v) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  const rq_config& c = h->cfg;
  if (session < 0 || session >= c.batch) return fail(h, RQ_ERR_ARG, "session out of range");
  if (n_pos < 0 || n_pos > c.context) return fail(h, RQ_ERR_ARG, "n_pos outside [0, context]");
  if (n_pos > 0 && (!k || !v)) return fail(h, RQ_ERR_ARG, "k or v is NULL");
  const size_t D = c.dim, C = c.context, L = c.layers, es = h->kves;
  if (n_pos > 0) {
    const size_t dst0 = (size_t)session * L * C * D * es;
    RQ_CUDA(h, cudaMemcpy2DAsync(static_cast<char*>(h->kcache) + dst0, C * D * es, k,
                                 (size_t)n_pos * D * es, (size_t)n_pos * D * es, L,
                                 cudaMemcpyDefault, h->stream));
    RQ_CUDA(h, cudaMemcpy2DAsync(static_cast<char*>(h->vcache) + dst0, C * D * es, v,
                                 (size_t)n_pos * D * es, (size_t)n_pos * D * es, L,
                                 cudaMemcpyDefault, h->stream));
  }
  RQ_CUDA(h, launch_set_offset(h->offsets, session, n_pos, h->stream));
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  h->host_off[session] = n_pos;
  return RQ_OK;
}

rq_status rq_launch_op(rq_handle* h, int32_t op, int32_t layer, int32_t count,
                       double* bytes_per_launch) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  const rq_config& c = h->cfg;
  if (layer < 0 || layer >= c.layers || count < 0) return fail(h, RQ_ERR_ARG, "bad layer or count");
  double bytes = 0;
  if (op == RQ_OP_FRAME) {
    if (h->schedule != RQ_SCHEDULE_PERSISTENT)
      return fail(h, RQ_ERR_UNSUPPORTED, "RQ_OP_FRAME needs the persistent schedule");
    const double D = c.dim, F = c.hidden, DD = c.ddim, DF = c.dhidden;
    // bytes of one stored row of K values (weight bands: codes and scales)
    auto rb = [&](long long K) { return (double)band_row_bytes(h->band, h->wes, K); };
    bytes = c.layers * ((3 * D + D + 2 * F) * rb(c.dim) + D * rb(c.hidden)) +
            (double)c.text_card * rb(c.dim) +
            8.0 * c.dlayers * ((3 * DD + DD + 2 * DF) * rb(c.ddim) + DD * rb(c.dhidden)) +
            8.0 * DD * rb(c.dim) + 8.0 * c.audio_card * rb(c.ddim);
    const int len = h->host_off[0] + 1 < c.context ? h->host_off[0] + 1 : c.context;
    bytes += 2.0 * len * c.dim * h->kves * c.layers;
    if (bytes_per_launch) *bytes_per_launch = bytes;
    for (int i = 0; i < count; ++i) {
      RQ_CUDA(h, cudaMemsetAsync(h->grid_bar, 0, 4, h->stream));
      RQ_CUDA(h, cudaMemsetAsync(h->grid_bar + kPersDepBarWord, 0, 4, h->stream));
      RQ_CUDA(h, launch_persistent(h->pers, h->wtype, h->kvbf, h->pers_grid, h->pers_smem,
                                   h->stream, false));
      if (h->pers_dep_grid > 0 && h->pers_dep.n_ops > 0)
        RQ_CUDA(h, launch_persistent(h->pers_dep, h->wtype, h->kvbf, h->pers_dep_grid,
                                     h->pers_dep_smem, h->stream, false, 1));
    }
    return RQ_OK;
  }
  switch (op) {
    case RQ_OP_QKV: bytes = h->p_qkv.bytes; break;
    case RQ_OP_OUT: bytes = h->p_out.bytes; break;
    case RQ_OP_GATE_IN: bytes = h->p_gin.bytes; break;
    case RQ_OP_GATE_OUT: bytes = h->p_gout.bytes; break;
    case RQ_OP_HEAD: bytes = h->p_head.bytes; break;
    case RQ_OP_ATTN:
      for (int b = 0; b < c.batch; ++b) {
        const int len = h->host_off[b] + 1 < c.context ? h->host_off[b] + 1 : c.context;
        bytes += 2.0 * len * c.dim * h->kves;
      }
      break;
    default: return fail(h, RQ_ERR_ARG, "unknown op");
  }
  if (bytes_per_launch) *bytes_per_launch = bytes;
  if (h->schedule == RQ_SCHEDULE_TENSOR) {
    if (op == RQ_OP_QKV) bytes = h->tcf.p_qkv.bytes;
    if (op == RQ_OP_OUT) bytes = h->tcf.p_out.bytes;
    if (op == RQ_OP_GATE_IN) bytes = h->tcf.p_gin.bytes;
    if (op == RQ_OP_GATE_OUT) bytes = h->tcf.p_gout.bytes;
    if (op == RQ_OP_HEAD) bytes = h->tcf.p_head.bytes;
    if (bytes_per_launch) *bytes_per_launch = bytes;
    for (int i = 0; i < count; ++i) {
      cudaError_t e = tc_frame_launch_op(h->tcf, op, layer, h->stream);
      if (e != cudaSuccess) return cuda_fail(h, e, "rq_launch_op");
    }
    return RQ_OK;
  }
  for (int i = 0; i < count; ++i) {
    cudaError_t e = cudaSuccess;
    switch (op) {
      case RQ_OP_QKV: e = op_qkv(h, layer, h->stream, true); break;
      case RQ_OP_ATTN: e = op_attn(h, layer, h->stream, true); break;
      case RQ_OP_OUT: e = op_out(h, layer, h->stream, true); break;
      case RQ_OP_GATE_IN: e = op_gate_in(h, layer, h->stream, true); break;
      case RQ_OP_GATE_OUT: e = op_gate_out(h, layer, h->stream, true); break;
      case RQ_OP_HEAD: e = op_head(h, h->stream, true); break;
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "rq_launch_op");
  }
  return RQ_OK;
}

rq_status rq_set_sampling(rq_handle* h, int32_t mode, float temp, float temp_text,
                          int32_t top_k, int32_t top_k_text, const uint64_t* seeds) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  if (mode < RQ_PICK_GREEDY || mode > RQ_PICK_GUMBEL)
    return fail(h, RQ_ERR_ARG, "unknown pick mode");
  if (mode != RQ_PICK_GREEDY) {
    if (!(temp > 0.f) || !(temp_text > 0.f) || !std::isfinite(temp) || !std::isfinite(temp_text))
      return fail(h, RQ_ERR_ARG, "temperatures must be finite and > 0");
    if (mode == RQ_PICK_TOPK && (top_k < 1 || top_k > kTopKMax || top_k_text < 1 ||
                                 top_k_text > kTopKMax))
      return fail(h, RQ_ERR_ARG, "top-k must be in 1..256");
    if (!seeds) return fail(h, RQ_ERR_ARG, "seeds required");
  }
  const int B = h->cfg.batch;
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));  // no frame of the old graph in flight
  if (seeds) {
    std::vector<uint64_t> s0(seeds, seeds + B);
    for (uint64_t& v : s0) v = v > 1 ? v : 1;  // "moshi_lm.rs", `set_sampling`: seed.max(1)
    RQ_CUDA(h, cudaMemcpy(h->rng, s0.data(), (size_t)B * 8, cudaMemcpyHostToDevice));
  }
  h->samp.mode = mode;
  if (mode != RQ_PICK_GREEDY) {
    h->samp.temp = temp;
    h->samp.temp_text = temp_text;
    h->samp.top_k = top_k;
    h->samp.top_k_text = top_k_text;
  }
  h->tcf.samp = h->samp;
  if (h->schedule == RQ_SCHEDULE_PERSISTENT && (st = upload_pers_ops(h)) != RQ_OK) return st;
  return capture_frame(h);
}

rq_status rq_get_rng(rq_handle* h, uint64_t* states) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  if (!states) return fail(h, RQ_ERR_ARG, "null states");
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  RQ_CUDA(h, cudaMemcpy(states, h->rng, (size_t)h->cfg.batch * 8, cudaMemcpyDeviceToHost));
  return RQ_OK;
}

size_t rq_band_row_bytes(int32_t dtype, int32_t cols) {
  if (cols <= 0 || cols % 32 != 0) return 0;
  if (dtype == RQ_Q8) return band_row_bytes(BAND_Q8, 1, cols);
  if (dtype == RQ_Q4) return band_row_bytes(BAND_Q4, 1, cols);
  if (dtype == RQ_BF16) return (size_t)cols * 2;
  if (dtype == RQ_F32) return (size_t)cols * 4;
  return 0;
}

rq_status rq_quantize(int32_t dtype, const void* src, int32_t src_dtype, int64_t rows,
                      int32_t cols, void* dst, void* cuda_stream) {
  if ((dtype != RQ_Q8 && dtype != RQ_Q4) || (src_dtype != RQ_F32 && src_dtype != RQ_BF16) ||
      rows < 0 || cols <= 0 || cols % 32 != 0 || (rows > 0 && (!src || !dst)))
    return RQ_ERR_ARG;
  const cudaError_t e =
      launch_quantize_band(dtype == RQ_Q8 ? BAND_Q8 : BAND_Q4, src, src_dtype == RQ_BF16, rows,
                           cols, dst, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return RQ_ERR_CUDA;
  }
  return RQ_OK;
}

rq_status rq_prime(rq_handle* h, int32_t session, int32_t n, const int32_t* forced,
                   const int32_t* user) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  const rq_config& c = h->cfg;
  if (session < 0 || session >= c.batch || n < 0) return fail(h, RQ_ERR_ARG, "bad session or n");
  if (n == 0) return RQ_OK;
  if (!forced || !user) return fail(h, RQ_ERR_ARG, "null forced or user codes");
  if (!prefill_eligible(h))
    return fail(h, RQ_ERR_UNSUPPORTED, "prefill needs bf16 weights and dim, hidden, ddim, "
                                       "dhidden multiples of 64");
  for (int64_t i = 0; i < (int64_t)n * 9; ++i) {  // tokens a frame could have generated
    const int lim = i % 9 == 0 ? c.text_card : c.audio_card;
    if (forced[i] < 0 || forced[i] >= lim) return fail(h, RQ_ERR_TOKEN, "forced token out of range");
  }
  for (int64_t i = 0; i < (int64_t)n * 8; ++i)
    if (user[i] < -1 || user[i] > c.audio_card) return fail(h, RQ_ERR_TOKEN, "user code out of range");
  if ((st = setup_prefill(h)) != RQ_OK) return st;
  for (int done = 0; done < n;) {
    const int T = prefill_chunk(h, session, n - done);
    RQ_CUDA(h, cudaMemcpyAsync(h->pf_forced, forced + (size_t)done * 9, (size_t)T * 9 * 4,
                               cudaMemcpyHostToDevice, h->stream));
    RQ_CUDA(h, cudaMemcpyAsync(h->pf_user, user + (size_t)done * 8, (size_t)T * 8 * 4,
                               cudaMemcpyHostToDevice, h->stream));
    if ((st = enqueue_prefill_chunk(h, session, T, true)) != RQ_OK) return st;
    done += T;
  }
  return rq_sync(h);
}

rq_status rq_replay(rq_handle* h, int32_t session, int32_t n, const float* x) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  const rq_config& c = h->cfg;
  if (session < 0 || session >= c.batch || n < 0) return fail(h, RQ_ERR_ARG, "bad session or n");
  if (n == 0) return RQ_OK;
  if (!x) return fail(h, RQ_ERR_ARG, "null embedding rows");
  if (!prefill_eligible(h))
    return fail(h, RQ_ERR_UNSUPPORTED, "prefill needs bf16 weights and dim, hidden, ddim, "
                                       "dhidden multiples of 64");
  if ((st = setup_prefill(h)) != RQ_OK) return st;
  for (int done = 0; done < n;) {
    const int T = prefill_chunk(h, session, n - done);
    RQ_CUDA(h, cudaMemcpyAsync(h->pf.x, x + (size_t)done * c.dim, (size_t)T * c.dim * 4,
                               cudaMemcpyDefault, h->stream));
    if ((st = enqueue_prefill_chunk(h, session, T, false)) != RQ_OK) return st;
    done += T;
  }
  return rq_sync(h);
}

namespace {
// snapshot layout: this header, then K [L][n][D] and V [L][n][D] in the K/V dtype, where
// n = min(offset, context) cache slots 0..n-1 (slot p % C holds position p)
struct SnapHeader {
  char magic[8];
  int32_t layers, context, dim, kv_bytes, offset, n;
  int32_t ring[kStreams * kRing];
};
const char kSnapMagic[8] = {'R', 'Q', 'S', 'N', 'A', 'P', '0', '1'};

size_t snap_bytes(const rq_handle* h, int n) {
  const rq_config& c = h->cfg;
  return sizeof(SnapHeader) + 2 * (size_t)c.layers * n * c.dim * h->kves;
}
}  // namespace

size_t rq_snapshot_size(const rq_handle* h, int32_t session) {
  if (!h || session < 0 || session >= h->cfg.batch) return 0;
  const int off = h->host_off[session];
  return snap_bytes(h, off < h->cfg.context ? off : h->cfg.context);
}

rq_status rq_snapshot(rq_handle* h, int32_t session, void* dst, size_t capacity) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  const rq_config& c = h->cfg;
  if (session < 0 || session >= c.batch || !dst) return fail(h, RQ_ERR_ARG, "bad session or dst");
  const int off = h->host_off[session], n = off < c.context ? off : c.context;
  if (capacity < snap_bytes(h, n)) return fail(h, RQ_ERR_ARG, "snapshot buffer too small");
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  SnapHeader hd{};
  std::memcpy(hd.magic, kSnapMagic, 8);
  hd.layers = c.layers;
  hd.context = c.context;
  hd.dim = c.dim;
  hd.kv_bytes = h->kves;
  hd.offset = off;
  hd.n = n;
  RQ_CUDA(h, cudaMemcpy(hd.ring, h->ring + (size_t)session * kStreams * kRing, sizeof(hd.ring),
                        cudaMemcpyDeviceToHost));
  RQ_CUDA(h, cudaMemcpy(dst, &hd, sizeof(hd), cudaMemcpyDefault));
  const size_t rowb = (size_t)c.dim * h->kves, layer = (size_t)c.context * rowb;
  const size_t sess = (size_t)session * c.layers * layer;
  char* out = static_cast<char*>(dst) + sizeof(SnapHeader);
  for (int kv = 0; kv < 2; ++kv) {
    const char* cache = static_cast<const char*>(kv ? h->vcache : h->kcache) + sess;
    for (int l = 0; l < c.layers; ++l, out += (size_t)n * rowb)
      if (n > 0)
        RQ_CUDA(h, cudaMemcpyAsync(out, cache + (size_t)l * layer, (size_t)n * rowb,
                                   cudaMemcpyDefault, h->stream));
  }
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  return RQ_OK;
}

rq_status rq_restore(rq_handle* h, int32_t session, const void* src, size_t size) {
  rq_status st = check_usable(h);
  if (st != RQ_OK) return st;
  const rq_config& c = h->cfg;
  if (session < 0 || session >= c.batch || !src || size < sizeof(SnapHeader))
    return fail(h, RQ_ERR_ARG, "bad session or snapshot");
  SnapHeader hd{};
  RQ_CUDA(h, cudaMemcpy(&hd, src, sizeof(hd), cudaMemcpyDefault));
  if (std::memcmp(hd.magic, kSnapMagic, 8) != 0 || hd.layers != c.layers ||
      hd.context != c.context || hd.dim != c.dim || hd.kv_bytes != h->kves || hd.offset < 0 ||
      hd.n != (hd.offset < c.context ? hd.offset : c.context) || size < snap_bytes(h, hd.n))
    return fail(h, RQ_ERR_ARG, "snapshot does not match this model");
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  const int n = hd.n;
  const size_t rowb = (size_t)c.dim * h->kves, layer = (size_t)c.context * rowb;
  const size_t sess = (size_t)session * c.layers * layer;
  const char* in = static_cast<const char*>(src) + sizeof(SnapHeader);
  for (int kv = 0; kv < 2; ++kv) {
    char* cache = static_cast<char*>(kv ? h->vcache : h->kcache) + sess;
    for (int l = 0; l < c.layers; ++l, in += (size_t)n * rowb)
      if (n > 0)
        RQ_CUDA(h, cudaMemcpyAsync(cache + (size_t)l * layer, in, (size_t)n * rowb,
                                   cudaMemcpyDefault, h->stream));
  }
  RQ_CUDA(h, cudaMemcpyAsync(h->ring + (size_t)session * kStreams * kRing, hd.ring,
                             sizeof(hd.ring), cudaMemcpyHostToDevice, h->stream));
  RQ_CUDA(h, launch_set_offset(h->offsets, session, hd.offset, h->stream));
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  h->host_off[session] = hd.offset;
  return RQ_OK;
}

int32_t rq_frame_kernel_count(const rq_handle* h) { return h ? h->n_kernels : 0; }

int32_t rq_schedule(const rq_handle* h) { return h ? h->schedule : 0; }

rq_status rq_set_wait_limit(rq_handle* h, uint64_t limit_ns, int32_t stall_op) {
  if (!h) return RQ_ERR_ARG;
  if (h->schedule != RQ_SCHEDULE_PERSISTENT || !h->grid_bar)
    return fail(h, RQ_ERR_UNSUPPORTED, "the wait limit applies to the persistent schedule");
  if (stall_op < -1 || stall_op == 0 || stall_op >= h->pers.n_ops + h->pers_dep.n_ops ||
      (stall_op > 0 && h->pers_nobar[stall_op]))
    return fail(h, RQ_ERR_ARG, "stall_op is not an op with a grid barrier in front (or -1)");
  const unsigned long long ctl[2] = {(unsigned long long)limit_ns,
                                     (unsigned long long)(stall_op + 1)};
  RQ_CUDA(h, cudaStreamSynchronize(h->stream));
  RQ_CUDA(h, cudaMemcpy(reinterpret_cast<unsigned long long*>(h->grid_bar) + kWaitCtlWord, ctl,
                        sizeof(ctl), cudaMemcpyHostToDevice));
  return RQ_OK;
}

int32_t rq_get_op_times(rq_handle* h, float* us, int32_t max_ops) {
  if (!h || h->schedule != RQ_SCHEDULE_PERSISTENT || !h->trace) return 0;
  const int n = h->pers.n_ops + h->pers_dep.n_ops;
  if (!us) return n;
  if (cudaStreamSynchronize(h->stream) != cudaSuccess) return 0;
  std::vector<unsigned long long> t((size_t)n + 1);
  if (cudaMemcpy(t.data(), h->trace, t.size() * 8, cudaMemcpyDeviceToHost) != cudaSuccess)
    return 0;
  const int m = n < max_ops ? n : max_ops;
  for (int i = 0; i < m; ++i)
    us[i] = (t[i + 1] >= t[i] && t[i] != 0) ? (float)((t[i + 1] - t[i]) * 1e-3) : -1.f;
  return m;
}

const char* rq_last_error(const rq_handle* h) {
  if (!h) return g_create_err.c_str();
  return h->err.c_str();
}

const char* rq_status_string(rq_status s) {
  switch (s) {
    case RQ_OK: return "ok";
    case RQ_ERR_ARG: return "invalid argument";
    case RQ_ERR_TOKEN: return "token out of range";
    case RQ_ERR_CUDA: return "CUDA error";
    case RQ_ERR_OOM: return "out of memory";
    case RQ_ERR_TIMEOUT: return "device-side wait timed out";
    case RQ_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case RQ_ERR_POISONED: return "handle poisoned by an earlier error";
  }
  return "unknown status";
}

int32_t rq_abi_version(void) { return RQ_ABI_VERSION; }

}  // extern "C"
