// tc_frame.cu -- a whole frame at batch 2..64 on the tensor cores: per linear, one
// tcgen05 GEMM over all sessions (weights read once per frame), bf16 operands prepared
// by a small normalisation kernel, the fused epilogues of the streaming path.
//
// "inferencelayer 0.2.4 -- src/moshi_lm.rs", `step_ext` steps 3-6: `temporal_step` per
// layer, out_norm + text head, `depformer_cycle` per codebook step.
#include "kernels.h"

namespace rqk {

namespace {

// element offset -> byte pointer of a bf16 array
const void* bf(const void* base, size_t elems) {
  return static_cast<const char*>(base) + elems * 2;
}

// weight map slots: temporal [L][4] (qkv, out, gate_in, gate_out), text head,
// dep_in [8], depformer [8][DL][4], linears [8]
int wi_layer(int l, int k) { return 4 * l + k; }
int wi_head(const TcFrame& f) { return 4 * f.L; }
int wi_depin(const TcFrame& f, int cb) { return 4 * f.L + 1 + cb; }
int wi_dep(const TcFrame& f, int cb, int l, int k) {
  return 4 * f.L + 9 + (cb * f.DL + l) * 4 + k;
}
int wi_lin(const TcFrame& f, int cb) { return 4 * f.L + 9 + 32 * f.DL + cb; }

TcParams base(const TcFrame& f, const TcPlan& pl, int epi) {
  TcParams p{};
  p.eps = f.eps;
  p.pl = pl;
  p.epi = epi;
  p.B = f.B;
  p.offsets = f.offsets;
  p.keys = f.keys;
  p.samp = f.samp;
  p.d_in = f.d_in;
  p.partial = f.part;
  p.tickets = f.tickets;
  p.status = f.status;
  p.head_dim = f.hd;
  p.context = f.C;
  p.kv_bf16 = f.kv_bf16;
  p.rope = f.rope;
  return p;
}

cudaError_t prep(const TcFrame& f, const float* in, int K, const float* alpha, uint16_t* xb,
                 float* side, cudaStream_t s) {
  return launch_prep_bf16(in, K, alpha, f.eps, f.B, f.NB, K, xb, side, K, s, true);
}

// fused RMSNorm: the consumer scales by 1 / rms from the producer's tile sums
void rms_in(const TcFrame& f, TcParams& p, bool depformer) {
  p.ss_in = depformer ? f.ss_dx : f.ss_x;
  p.rms_K = depformer ? f.DD : f.D;
  p.ss_tiles = (p.rms_K + 127) / 128;
}

// the producer writes the next GEMM's operand (value * alpha, or the value) and,
// when that GEMM normalises, the tile sums of squares
void feed(const TcFrame& f, TcParams& p, bool depformer, const float* alpha, bool rms) {
  p.opnd = depformer ? f.dxb : f.xb;
  p.alpha_next = alpha;
  p.ss_out = rms ? (depformer ? f.ss_dx : f.ss_x) : nullptr;
}

}  // namespace

int tc_frame_n_maps(const TcFrame& f) { return wi_lin(f, 8); }

void tc_frame_plan(TcFrame& f, int sms, size_t* part_floats, int* n_tickets) {
  f.p_qkv = plan_tc(3 * f.D, f.D, f.NB, false, sms);
  f.p_out = plan_tc(f.D, f.D, f.NB, false, sms);
  f.p_gin = plan_tc(f.F, f.D, f.NB, true, sms);
  f.p_gout = plan_tc(f.D, f.F, f.NB, false, sms);
  f.p_head = plan_tc(f.V, f.D, f.NB, false, sms);
  f.p_depin = plan_tc(f.DD, f.D, f.NB, false, sms);
  f.p_dqkv = plan_tc(3 * f.DD, f.DD, f.NB, false, sms);
  f.p_dout = plan_tc(f.DD, f.DD, f.NB, false, sms);
  f.p_dgin = plan_tc(f.DF, f.DD, f.NB, true, sms);
  f.p_dgout = plan_tc(f.DD, f.DF, f.NB, false, sms);
  f.p_lin = plan_tc(f.A, f.DD, f.NB, false, sms);
  const TcPlan* all[] = {&f.p_qkv, &f.p_out, &f.p_gin, &f.p_gout, &f.p_head, &f.p_depin,
                         &f.p_dqkv, &f.p_dout, &f.p_dgin, &f.p_dgout, &f.p_lin};
  size_t pf = 0;
  int nt = 0;
  for (const TcPlan* p : all) {
    if (p->splits > 1) {
      const size_t need = (size_t)p->tiles_m * p->splits * p->NB * 128;
      pf = need > pf ? need : pf;
    }
    nt = p->tiles_m > nt ? p->tiles_m : nt;
  }
  *part_floats = pf;
  *n_tickets = nt;
}

cudaError_t tc_frame_maps(TcFrame& f) {
  const size_t D = f.D, F = f.F, V = f.V, DD = f.DD, DF = f.DF, A = f.A;
  cudaError_t e;
#define MAP(slot, base, rows, cols, box) \
  if ((e = make_tmap_bf16(&(slot), (base), (rows), (cols), (box))) != cudaSuccess) return e;
  const int R = kOpndParts * f.NB;  // operand rows: the bf16 parts of each session
  MAP(f.xm_x, f.xb, R, D, R);
  MAP(f.xm_attn, f.attn_b, R, D, R);
  MAP(f.xm_u, f.u_b, R, F, R);
  MAP(f.xm_tout, f.tout_b, R, D, R);
  MAP(f.xm_dx, f.dxb, R, DD, R);
  MAP(f.xm_do, f.do_b, R, DD, R);
  MAP(f.xm_du, f.du_b, R, DF, R);
  for (int l = 0; l < f.L; ++l) {
    MAP(f.wm[wi_layer(l, 0)], bf(f.in_proj, (size_t)l * 3 * D * D), 3 * D, D, 128);
    MAP(f.wm[wi_layer(l, 1)], bf(f.out_proj, (size_t)l * D * D), D, D, 128);
    MAP(f.wm[wi_layer(l, 2)], bf(f.gate_in, (size_t)l * 2 * F * D), 2 * F, D, 64);
    MAP(f.wm[wi_layer(l, 3)], bf(f.gate_out, (size_t)l * D * F), D, F, 128);
  }
  MAP(f.wm[wi_head(f)], f.text_linear, V, D, 128);
  for (int cb = 0; cb < 8; ++cb) {
    MAP(f.wm[wi_depin(f, cb)], bf(f.dep_in, (size_t)cb * DD * D), DD, D, 128);
    MAP(f.wm[wi_lin(f, cb)], bf(f.linears, (size_t)cb * A * DD), A, DD, 128);
    for (int l = 0; l < f.DL; ++l) {
      const size_t ls = (size_t)l * 8 + cb;
      MAP(f.wm[wi_dep(f, cb, l, 0)], bf(f.d_in_proj, ls * 3 * DD * DD), 3 * DD, DD, 128);
      MAP(f.wm[wi_dep(f, cb, l, 1)], bf(f.d_out_proj, ls * DD * DD), DD, DD, 128);
      MAP(f.wm[wi_dep(f, cb, l, 2)], bf(f.d_gate_in, ls * 2 * DF * DD), 2 * DF, DD, 64);
      MAP(f.wm[wi_dep(f, cb, l, 3)], bf(f.d_gate_out, ls * DD * DF), DD, DF, 128);
    }
  }
#undef MAP
  return cudaSuccess;
}

namespace {

void* layer_cache(const TcFrame& f, void* base, int l) {
  const size_t kves = f.kv_bf16 ? 2 : 4;
  return static_cast<char*>(base) + (size_t)l * f.C * f.D * kves;
}

cudaError_t tc_qkv(const TcFrame& f, int l, cudaStream_t s) {
  TcParams p = base(f, f.p_qkv, EPI_QKV);
  if (l > 0) rms_in(f, p, false);  // layer 0's operand is normalised by the prep kernel
  p.out = f.q;
  p.out_bs = f.D;
  p.kcache = layer_cache(f, f.kcache, l);
  p.vcache = layer_cache(f, f.vcache, l);
  p.kv_bs = f.one_session ? 0 : (long long)f.L * f.C * f.D;  // columns: sessions or positions
  return launch_tc(p, f.wm[wi_layer(l, 0)], f.xm_x, s, true);
}

// split-K attention over the context, with a bf16 copy of the output for the next GEMM
cudaError_t tc_attn(const TcFrame& f, int l, cudaStream_t s) {
  AttnParams a{};
  a.q = f.q;
  a.kbase = f.kcache;  // [B][L][C][D]: session b, layer l, slot j is row (b L + l) C + j
  a.vbase = f.vcache;
  a.rows = (long long)(f.one_session ? 1 : f.B) * f.L * f.C;
  a.row0 = (long long)l * f.C;
  a.row_bs = f.one_session ? 0 : (long long)f.L * f.C;
  a.offsets = f.offsets;
  a.part = f.attn_part;
  a.counters = f.attn_counters;
  a.out = f.attn;
  a.out_bf16 = f.attn_b;
  a.nb = f.NB;
  a.D = f.D;
  a.H = f.H;
  a.hd = f.hd;
  a.C = f.C;
  a.kps = f.kps;
  a.nsplit = f.nsplit;
  a.batch = f.B;
  a.status = f.status;
  return launch_attn(a, f.kv_bf16 != 0, s, true);
}

cudaError_t tc_out(const TcFrame& f, int l, cudaStream_t s) {
  TcParams p = base(f, f.p_out, EPI_RESID);
  p.out = f.x;
  p.out_bs = f.D;
  feed(f, p, false, f.norm2 + (size_t)l * f.D, true);  // gate_in's rms_norm
  return launch_tc(p, f.wm[wi_layer(l, 1)], f.xm_attn, s, true);
}

cudaError_t tc_gin(const TcFrame& f, int l, cudaStream_t s) {
  TcParams p = base(f, f.p_gin, EPI_SWIGLU);
  rms_in(f, p, false);
  p.out_bf16 = f.u_b;
  p.outb_bs = f.F;
  return launch_tc(p, f.wm[wi_layer(l, 2)], f.xm_x, s, true);
}

cudaError_t tc_gout(const TcFrame& f, int l, cudaStream_t s) {
  TcParams p = base(f, f.p_gout, EPI_RESID);
  p.out = f.x;
  p.out_bs = f.D;
  if (l + 1 < f.L) feed(f, p, false, f.norm1 + (size_t)(l + 1) * f.D, true);  // next qkv
  return launch_tc(p, f.wm[wi_layer(l, 3)], f.xm_u, s, true);
}

cudaError_t tc_head(const TcFrame& f, cudaStream_t s) {
  TcParams p = base(f, f.p_head, EPI_ARGMAX);
  p.out = f.text_logits;
  p.out_bs = f.V;
  p.key_index = 0;
  return launch_tc(p, f.wm[wi_head(f)], f.xm_tout, s, true);
}

}  // namespace

cudaError_t tc_frame_launch_op(const TcFrame& f, int op, int layer, cudaStream_t s) {
  switch (op) {
    case 0: return tc_qkv(f, layer, s);
    case 1: return tc_attn(f, layer, s);
    case 2: return tc_out(f, layer, s);
    case 3: return tc_gin(f, layer, s);
    case 4: return tc_gout(f, layer, s);
    case 5: return tc_head(f, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t tc_frame_enqueue_temporal(const TcFrame& f, cudaStream_t s) {
  cudaError_t e;
#define CK(call) \
  if ((e = (call)) != cudaSuccess) return e;
  // rms_norm of layer 0's input; later norms are fused (producer epilogue + consumer scale)
  CK(prep(f, f.x, f.D, f.norm1, f.xb, nullptr, s));
  for (int l = 0; l < f.L; ++l) {
    CK(tc_qkv(f, l, s));
    CK(tc_attn(f, l, s));
    CK(tc_out(f, l, s));
    CK(tc_gin(f, l, s));
    CK(tc_gout(f, l, s));
  }
#undef CK
  return cudaSuccess;
}

cudaError_t tc_frame_enqueue(const TcFrame& f, cudaStream_t s) {
  const size_t D = f.D, A = f.A, DD = f.DD, DF = f.DF;
  const long long dkv_bs = (long long)f.DL * 2 * 8 * DD;
  auto dkv_off = [&](int l, int kv, int j) { return (((size_t)l * 2 + kv) * 8 + j) * DD; };
  cudaError_t e;
#define CK(call) \
  if ((e = (call)) != cudaSuccess) return e;
  CK(tc_frame_enqueue_temporal(f, s));
  // out_norm (kept as the depformer's input) + text head + first-wins argmax
  CK(prep(f, f.x, f.D, f.out_norm, f.tout_b, f.tout, s));
  CK(tc_head(f, s));
  if (f.samp.mode == SAMPLE_TOPK)
    CK(launch_topk_pick(f.samp, f.text_logits, f.V, f.V, 0, f.keys, f.B, s, true));
  for (int cb = 0; cb < 8; ++cb) {
    {  // depformer_in[cb](tout) + embedding of the previous token; feeds layer 0's norm
      TcParams p = base(f, f.p_depin, EPI_DEPIN);
      p.out = f.dx;
      p.out_bs = DD;
      p.emb = cb == 0 ? f.dep_text_emb : bf(f.dep_emb, (size_t)(cb - 1) * (A + 1) * DD);
      p.key_index = cb;
      feed(f, p, true, f.dnorm1, true);
      CK(launch_tc(p, f.wm[wi_depin(f, cb)], f.xm_tout, s, true));
    }
    for (int l = 0; l < f.DL; ++l) {
      {
        TcParams p = base(f, f.p_dqkv, EPI_DQKV);
        rms_in(f, p, true);
        p.out = f.dq;
        p.out_bs = DD;
        p.dk_out = f.dkv + dkv_off(l, 0, cb);
        p.dv_out = f.dkv + dkv_off(l, 1, cb);
        p.dkv_bs = dkv_bs;
        CK(launch_tc(p, f.wm[wi_dep(f, cb, l, 0)], f.xm_dx, s, true));
      }
      CK(launch_dattn_batched(f.dq, (long long)DD, f.dkv + dkv_off(l, 0, 0),
                              f.dkv + dkv_off(l, 1, 0), dkv_bs, cb + 1, f.B, f.dH, f.dhd,
                              f.do_b, (long long)DD, f.NB, s, true));
      {
        TcParams p = base(f, f.p_dout, EPI_RESID);
        p.out = f.dx;
        p.out_bs = DD;
        feed(f, p, true, f.dnorm2 + (size_t)l * DD, true);  // gate_in's rms_norm
        CK(launch_tc(p, f.wm[wi_dep(f, cb, l, 1)], f.xm_do, s, true));
      }
      {
        TcParams p = base(f, f.p_dgin, EPI_SWIGLU);
        rms_in(f, p, true);
        p.out_bf16 = f.du_b;
        p.outb_bs = DF;
        CK(launch_tc(p, f.wm[wi_dep(f, cb, l, 2)], f.xm_dx, s, true));
      }
      {
        // next layer's rms_norm, or the head's plain operand (no norm before linears)
        TcParams p = base(f, f.p_dgout, EPI_RESID);
        p.out = f.dx;
        p.out_bs = DD;
        if (l + 1 < f.DL)
          feed(f, p, true, f.dnorm1 + (size_t)(l + 1) * DD, true);
        else
          feed(f, p, true, nullptr, false);
        CK(launch_tc(p, f.wm[wi_dep(f, cb, l, 3)], f.xm_du, s, true));
      }
    }
    {
      TcParams p = base(f, f.p_lin, EPI_ARGMAX);
      p.out = f.audio_logits + (size_t)cb * A;
      p.out_bs = (long long)(8 * A);
      p.key_index = 1 + cb;
      CK(launch_tc(p, f.wm[wi_lin(f, cb)], f.xm_dx, s, true));
    }
    if (f.samp.mode == SAMPLE_TOPK)
      CK(launch_topk_pick(f.samp, f.audio_logits + (size_t)cb * A, 8ll * A, A, 1 + cb, f.keys,
                          f.B, s, true));
  }
#undef CK
  return cudaSuccess;
}

}  // namespace rqk
