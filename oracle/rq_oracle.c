/*
 * rq_oracle.c -- TEST INFRASTRUCTURE, not part of the product.
 *
 * A plain, slow, scalar CPU restatement (f32, as the page fixes) of the per-frame
 * decode step of a Moshi-style RQ-Transformer, written from the docs.rs page
 * "inferencelayer 0.2.4 -- src/moshi_lm.rs" (module doc comment, `rms_norm`,
 * `silu`, `argmax`, `xorshift_u01`, `topk_sample`, `gumbel_full_pick`, `pick`,
 * `rope_row`, `attend`, `embed`, `temporal_step`, `depformer_cycle`, `step_ext`,
 * `MoshiState::force_generated`, `Sampling`, `set_sampling`), plus the forced
 * depformer conditioning of "rlx-moshi -- src/rlx_lm.rs" (`depformer_sample_rlx`,
 * `depformer_forced_logits_rlx`).
 *
 * Rules this file keeps:
 *   - one function per definition on the page, in the page's order of operations;
 *     every dot product is a strictly sequential f32 sum over k = 0..K-1; compiled
 *     with -ffp-contract=off so no multiply-add is fused behind the reader's back;
 *   - OpenMP, when present, only splits independent output rows or heads, so each
 *     row's summation order is untouched and results are bitwise identical for any
 *     thread count;
 *   - it shares no code, header, table or helper with the CUDA library; only
 *     tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference arm
 *     load it.
 *
 * Readings where the pages leave a step open (each is also listed in the design
 * notes):
 *   - bf16 configurations hold every matrix and table as bf16 bit patterns; each
 *     element is widened exactly to f32 before use;
 *   - bf16 configurations round the temporal K and V rows to bf16 (round to
 *     nearest even) when they are appended to the window, as the GPU cache stores
 *     them; the depformer's per-frame K/V stay f32;
 *   - forcing: `forced` = [text, audio0..7] conditions the depformer chain and is
 *     what the ring records, while the step still reports its own picked tokens;
 *   - `topk_sample` walks the k selected logits in descending order, equal logits by
 *     ascending index (the page's partial selection leaves that order open);
 *   - each session owns its sampler state (the page has one session per model).
 *
 * Parity pins (tests/test_oracle_pins.py): RMSNorm closed forms, RoPE hand vectors,
 * argmax tie/NaN cases, the published xorshift64 sequence, the Gumbel-max and top-k
 * pick frequencies against the softmax they sample, one-key attention, attention and
 * GEMV against independent
 * f64 routines, the hand-traced ring schedule, -1 zero embedding, depformer reset
 * versus a from-scratch causal recompute, and an independent NumPy f64
 * restatement of whole frames.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_STREAMS 17 /* 1 text + 8 generated audio + 8 user audio */
#define ORC_DEP_Q 8    /* generated audio codebooks per frame */
#define ORC_MAX_DELAY 1
#define ORC_CT (ORC_MAX_DELAY + 2) /* ring length */
#define ORC_UNGENERATED (-2)

/* moshi_lm.rs, module doc "streams and delays" / const DELAYS */
static const int ORC_DELAYS[ORC_STREAMS] = {0, 0, 1, 1, 1, 1, 1, 1, 1,
                                            0, 1, 1, 1, 1, 1, 1, 1};

typedef struct {
  int32_t dim, layers, heads, head_dim, hidden, context;
  int32_t text_card, audio_card;
  int32_t ddim, dlayers, dheads, dhead_dim, dhidden;
  int32_t w_bf16;  /* 1: matrices and embedding tables are bf16 bit patterns */
  int32_t kv_bf16; /* 1: temporal K/V rows are rounded to bf16 when appended */
  float eps;       /* RMSNorm epsilon (1e-8) */
  float rope_theta;/* 10000 */
} orc_cfg;

typedef struct {
  const void *emb;          /* [16][A+1][D]   audio input tables */
  const void *text_emb;     /* [V+1][D] */
  const float *norm1;       /* [L][D] */
  const void *in_proj;      /* [L][3D][D] */
  const void *out_proj;     /* [L][D][D] */
  const float *norm2;       /* [L][D] */
  const void *gate_in;      /* [L][2F][D]  rows 0..F-1 gate, F..2F-1 mult */
  const void *gate_out;     /* [L][D][F] */
  const float *out_norm;    /* [D] */
  const void *text_linear;  /* [V][D] */
  const void *dep_in;       /* [8][DD][D] */
  const void *dep_text_emb; /* [V+1][DD] */
  const void *dep_emb;      /* [7][A+1][DD] */
  const float *dnorm1;      /* [DL][DD] shared by the 8 steps */
  const float *dnorm2;      /* [DL][DD] */
  const void *d_in_proj;    /* [DL][8][3DD][DD] */
  const void *d_out_proj;   /* [DL][8][DD][DD] */
  const void *d_gate_in;    /* [DL][8][2DF][DD] */
  const void *d_gate_out;   /* [DL][8][DD][DF] */
  const void *linears;      /* [8][A][DD] */
} orc_weights;

/* moshi_lm.rs, struct MoshiState: ring cache, offset, temporal K/V window
 * ([layer][step][dim], oldest first). */
/* moshi_lm.rs, struct `Sampling` and `MoshiLm::set_sampling`: how `pick` chooses a
 * token.  mode 0 = greedy argmax (no sampler set), 1 = `topk_sample`, 2 =
 * `gumbel_full_pick`; text picks use temp_text / top_k_text. */
typedef struct {
  int32_t mode;
  float temp, temp_text;
  int32_t top_k, top_k_text;
} orc_sampling;

typedef struct {
  int64_t ring[ORC_STREAMS][ORC_CT];
  int64_t offset;
  orc_sampling smp; /* greedy unless orc_state_set_sampling was called */
  uint64_t rng;     /* xorshift64 state of this session's sampler */
  int32_t layers, context, dim;
  int32_t *kv_len; /* [L] entries currently in the window */
  float *k;        /* [L][C][D] */
  float *v;        /* [L][C][D] */
} orc_state;

/* ---------------------------------------------------------------- elements */

static float bf16_bits_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* round an f32 to the nearest bf16 (ties to even) and widen it back */
static float round_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) { /* inf / nan: keep, quiet the nan */
    if (u & 0x007fffffu) u |= 0x00400000u;
    u &= 0xffff0000u;
  } else {
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    u &= 0xffff0000u;
  }
  float r;
  memcpy(&r, &u, 4);
  return r;
}

/* element i of a weight array stored as bf16 bits or f32 */
static float wat(const void *base, int bf16, size_t i) {
  if (bf16) return bf16_bits_to_f32(((const uint16_t *)base)[i]);
  return ((const float *)base)[i];
}

static const void *woff(const void *base, int bf16, size_t elems) {
  return (const char *)base + elems * (bf16 ? 2u : 4u);
}

/* ---------------------------------------------------------------- primitives */

/* moshi_lm.rs, `Band::mv`: out = W x, W row-major [rows][k]; each row is a
 * sequential f32 dot product. */
void orc_gemv(const void *w, int32_t bf16, int32_t rows, int32_t k,
              const float *x, float *out) {
  int r;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) if ((long)rows * k > 65536)
#endif
  for (r = 0; r < rows; r++) {
    float acc = 0.0f;
    size_t base = (size_t)r * (size_t)k;
    for (int c = 0; c < k; c++) acc += wat(w, bf16, base + c) * x[c];
    out[r] = acc;
  }
}

/* moshi_lm.rs, `rms_norm`: y = x * alpha * (1 / sqrt(eps + sum(x^2)/n)) --
 * eps inside the mean, no re-centering. */
void orc_rms_norm(const float *x, const float *alpha, int32_t n, float eps,
                  float *out) {
  float ss = 0.0f;
  for (int i = 0; i < n; i++) ss += x[i] * x[i];
  float var = eps + ss / (float)n;
  float inv = 1.0f / sqrtf(var);
  for (int i = 0; i < n; i++) out[i] = x[i] * alpha[i] * inv;
}

/* moshi_lm.rs, `silu`: x / (1 + exp(-x)) */
float orc_silu(float x) { return x / (1.0f + expf(-x)); }

/* moshi_lm.rs, `argmax`: strict `>` scan from (-inf, 0): the first index wins a
 * tie, NaN never wins, an all -inf (or all NaN) row gives 0. */
uint32_t orc_argmax(const float *v, int32_t n) {
  float best = -INFINITY;
  uint32_t bi = 0;
  for (int i = 0; i < n; i++) {
    if (v[i] > best) {
      best = v[i];
      bi = (uint32_t)i;
    }
  }
  return bi;
}

/* moshi_lm.rs, `xorshift_u01`: one xorshift64 step (shifts 13, 7, 17, as in
 * G. Marsaglia, "Xorshift RNGs", J. Stat. Soft. 8(14), 2003) of the state, returned
 * raw; orc_xorshift_u01 maps its top 53 bits to [0, 1). */
uint64_t orc_xorshift_next(uint64_t *st) {
  uint64_t x = *st;
  x ^= x << 13;
  x ^= x >> 7;
  x ^= x << 17;
  *st = x;
  return x;
}

double orc_xorshift_u01(uint64_t *st) {
  uint64_t x = orc_xorshift_next(st);
  return (double)(x >> 11) / (double)(1ull << 53);
}

/* moshi_lm.rs, `qn_roundtrip` (the symmetric weight bands): every group of `group`
 * consecutive values of a row, with mx the first value of the largest magnitude,
 * d = mx / -(2^(bits-1)), id = 1/d (0 when d == 0), is replaced by
 * clamp(round(x * id), -(2^(bits-1)), 2^(bits-1) - 1) * d; `round` halves away from zero
 * as Rust's f32::round.  bits 4 with group 32 is the Q4_0 band (d = max / -8), bits 8 the
 * q8_0-style band.  In place on an f32 [rows][cols] array. */
void orc_qn_roundtrip(float *v, int32_t rows, int32_t cols, int32_t bits, int32_t group) {
  const int32_t qmin = -(1 << (bits - 1)), qmax = (1 << (bits - 1)) - 1;
  for (int32_t r = 0; r < rows; r++) {
    for (int32_t b = 0; b < cols / group; b++) {
      float *blk = v + (size_t)r * cols + (size_t)b * group;
      float amax = 0.0f, mx = 0.0f;
      for (int32_t i = 0; i < group; i++) {
        if (fabsf(blk[i]) > amax) {
          amax = fabsf(blk[i]);
          mx = blk[i];
        }
      }
      float d = mx / (float)qmin;
      float id = d != 0.0f ? 1.0f / d : 0.0f;
      for (int32_t i = 0; i < group; i++) {
        float q = roundf(blk[i] * id);
        int32_t qi = (int32_t)q;
        if (qi < qmin) qi = qmin;
        if (qi > qmax) qi = qmax;
        blk[i] = (float)qi * d;
      }
    }
  }
}

/* moshi_lm.rs, `gumbel_full_pick`: argmax over i of logits[i] / temp + g_i with
 * g_i = -ln(-ln(u_i)) in f64 (u_i the i-th draw, at least 1e-300) rounded to f32;
 * the first strictly greater score wins.  Consumes n draws. */
uint32_t orc_gumbel_pick(const float *logits, int32_t n, float temp, uint64_t *st) {
  float best = -INFINITY;
  uint32_t bi = 0;
  for (int32_t i = 0; i < n; i++) {
    double u = orc_xorshift_u01(st);
    if (u < 1e-300) u = 1e-300;
    float g = (float)(-log(-log(u)));
    float sc = logits[i] / temp + g;
    if (sc > best) {
      best = sc;
      bi = (uint32_t)i;
    }
  }
  return bi;
}

/* the total order of f32 values (-NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN) as
 * an unsigned key */
static uint32_t total_order_key(float v) {
  uint32_t u;
  memcpy(&u, &v, 4);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

static const float *g_sort_logits;
/* descending total order of the logit; equal logits by ascending index */
static int topk_cmp(const void *a, const void *b) {
  uint32_t ia = *(const uint32_t *)a, ib = *(const uint32_t *)b;
  uint32_t ka = total_order_key(g_sort_logits[ia]), kb = total_order_key(g_sort_logits[ib]);
  if (ka != kb) return ka > kb ? -1 : 1;
  return ia < ib ? -1 : (ia > ib);
}

/* moshi_lm.rs, `topk_sample`: the k largest logits (reading: taken in descending order,
 * equal logits by ascending index -- the page leaves the order of the selected k
 * open), p_i = exp(((l_i - max) / temp) in f32, widened to f64), normalised by their
 * sequential f64 sum; one draw u, and the first i at which u - p_0 - ... - p_i <= 0 is
 * the token (the last candidate if none).  Consumes one draw. */
uint32_t orc_topk_pick(const float *logits, int32_t n, float temp, int32_t k, uint64_t *st) {
  if (k > n) k = n;
  if (k < 1) k = 1;
  uint32_t *idx = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)n);
  for (int32_t i = 0; i < n; i++) idx[i] = (uint32_t)i;
  g_sort_logits = logits;
  qsort(idx, (size_t)n, sizeof(uint32_t), topk_cmp);
  float mx = -INFINITY;
  for (int32_t i = 0; i < k; i++) mx = fmaxf(mx, logits[idx[i]]);
  double *p = (double *)malloc(sizeof(double) * (size_t)k);
  double sum = 0.0;
  for (int32_t i = 0; i < k; i++) {
    p[i] = exp((double)((logits[idx[i]] - mx) / temp));
    sum += p[i];
  }
  for (int32_t i = 0; i < k; i++) p[i] /= sum;
  double u = orc_xorshift_u01(st);
  uint32_t tok = idx[k - 1];
  for (int32_t i = 0; i < k; i++) {
    u -= p[i];
    if (u <= 0.0) {
      tok = idx[i];
      break;
    }
  }
  free(p);
  free(idx);
  return tok;
}

/* moshi_lm.rs, `pick`: greedy argmax without a sampler, else the configured sampler
 * with the text or the audio temperature and k. */
static uint32_t pick(const orc_sampling *smp, uint64_t *rng, const float *logits,
                     int32_t n, int text) {
  if (smp == NULL || smp->mode == 0) return orc_argmax(logits, n);
  float temp = text ? smp->temp_text : smp->temp;
  if (smp->mode == 2) return orc_gumbel_pick(logits, n, temp, rng);
  return orc_topk_pick(logits, n, temp, text ? smp->top_k_text : smp->top_k, rng);
}

/* moshi_lm.rs, `rope_row`: interleaved pairs (2i, 2i+1) of every head rotated by
 * freq_i * pos, freq_i = exp(-ln(theta) * 2i / head_dim), all in f32. */
void orc_rope_row(float *row, int32_t n, int64_t pos, int32_t head_dim,
                  float theta) {
  float ts = (float)pos;
  for (int h = 0; h < n / head_dim; h++) {
    float *head = row + (size_t)h * head_dim;
    for (int i = 0; i < head_dim / 2; i++) {
      float freq = expf(-logf(theta) * 2.0f * (float)i / (float)head_dim);
      float ang = freq * ts;
      float s = sinf(ang), c = cosf(ang);
      float r = head[2 * i], im = head[2 * i + 1];
      head[2 * i] = r * c - im * s;
      head[2 * i + 1] = r * s + im * c;
    }
  }
}

/* moshi_lm.rs, `attend`: single-query multi-head attention over n_keys cached rows
 * (row j of ks / vs has `heads * head_dim` values, j = 0 is the oldest);
 * scores scaled by 1/sqrt(head_dim), softmax with the maximum subtracted, f32. */
void orc_attend(const float *q, const float *ks, const float *vs, int32_t n_keys,
                int32_t heads, int32_t head_dim, float *out) {
  int dim = heads * head_dim;
  float scale = 1.0f / sqrtf((float)head_dim);
  for (int i = 0; i < dim; i++) out[i] = 0.0f;
  int h;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) if ((long)n_keys * dim > 262144)
#endif
  for (h = 0; h < heads; h++) {
    const float *qh = q + (size_t)h * head_dim;
    float *scores = (float *)malloc(sizeof(float) * (size_t)(n_keys > 0 ? n_keys : 1));
    for (int j = 0; j < n_keys; j++) {
      const float *kh = ks + (size_t)j * dim + (size_t)h * head_dim;
      float dot = 0.0f;
      for (int d = 0; d < head_dim; d++) dot += qh[d] * kh[d];
      scores[j] = dot * scale;
    }
    float mx = -INFINITY;
    for (int j = 0; j < n_keys; j++) mx = fmaxf(mx, scores[j]);
    float den = 0.0f;
    for (int j = 0; j < n_keys; j++) {
      scores[j] = expf(scores[j] - mx);
      den += scores[j];
    }
    float *oh = out + (size_t)h * head_dim;
    for (int j = 0; j < n_keys; j++) {
      float wgt = scores[j] / den;
      const float *vh = vs + (size_t)j * dim + (size_t)h * head_dim;
      for (int d = 0; d < head_dim; d++) oh[d] += wgt * vh[d];
    }
    free(scores);
  }
}

/* moshi_lm.rs, `embed` (ScaledEmbedding): token -1 adds nothing (an exact zero
 * contribution); any other token adds row max(tok, 0). */
void orc_embed(const void *table, int32_t bf16, int32_t dim, int64_t tok,
               float *acc) {
  if (tok == -1) return;
  size_t row = (size_t)(tok > 0 ? tok : 0);
  for (int i = 0; i < dim; i++) acc[i] += wat(table, bf16, row * dim + i);
}

/* ---------------------------------------------------------------- state */

orc_state *orc_state_new(const orc_cfg *c) {
  orc_state *st = (orc_state *)calloc(1, sizeof(orc_state));
  if (!st) return NULL;
  st->layers = c->layers;
  st->context = c->context;
  st->dim = c->dim;
  st->kv_len = (int32_t *)calloc((size_t)c->layers, sizeof(int32_t));
  size_t n = (size_t)c->layers * c->context * c->dim;
  st->k = (float *)calloc(n, sizeof(float));
  st->v = (float *)calloc(n, sizeof(float));
  if (!st->kv_len || !st->k || !st->v) {
    free(st->kv_len); free(st->k); free(st->v); free(st);
    return NULL;
  }
  /* moshi_lm.rs, `MoshiLm::state`: ring all UNGENERATED, offset 0, empty KV */
  for (int s = 0; s < ORC_STREAMS; s++)
    for (int j = 0; j < ORC_CT; j++) st->ring[s][j] = ORC_UNGENERATED;
  st->offset = 0;
  st->rng = 1;
  return st;
}

/* moshi_lm.rs, `MoshiLm::set_sampling`: the sampler and its seed (at least 1) */
void orc_state_set_sampling(orc_state *st, int32_t mode, float temp, float temp_text,
                            int32_t top_k, int32_t top_k_text, uint64_t seed) {
  st->smp.mode = mode;
  st->smp.temp = temp;
  st->smp.temp_text = temp_text;
  st->smp.top_k = top_k;
  st->smp.top_k_text = top_k_text;
  st->rng = seed > 1 ? seed : 1;
}

uint64_t orc_state_get_rng(const orc_state *st) { return st->rng; }

void orc_state_free(orc_state *st) {
  if (!st) return;
  free(st->kv_len); free(st->k); free(st->v); free(st);
}

/* Pre-fill a session: positions 0..n_pos-1 of every layer's window take the given
 * rows (already rotated keys; [L][n_pos][D], bf16 bits when kv_bits16, else f32),
 * and the clock jumps to n_pos without touching the ring (moshi_lm.rs,
 * `MoshiState::advance_clock`). */
int orc_state_set_kv(orc_state *st, int32_t n_pos, const void *k, const void *v,
                     int32_t kv_bits16) {
  if (n_pos < 0 || n_pos > st->context) return 1;
  for (int l = 0; l < st->layers; l++) {
    for (int p = 0; p < n_pos; p++) {
      for (int d = 0; d < st->dim; d++) {
        size_t src = ((size_t)l * n_pos + p) * st->dim + d;
        size_t dst = ((size_t)l * st->context + p) * st->dim + d;
        st->k[dst] = wat(k, kv_bits16, src);
        st->v[dst] = wat(v, kv_bits16, src);
      }
    }
    st->kv_len[l] = n_pos;
  }
  st->offset = n_pos;
  return 0;
}

void orc_state_get_ring(const orc_state *st, int64_t *ring /*[17][3]*/,
                        int64_t *offset) {
  memcpy(ring, st->ring, sizeof(st->ring));
  *offset = st->offset;
}

/* ---------------------------------------------------------------- model */

/* moshi_lm.rs, `temporal_step`: 32 pre-norm layers at position `pos` = offset,
 * then `out_norm`; x is the running residual (in: embedding sum). */
void orc_temporal_step(const orc_cfg *c, const orc_weights *w, orc_state *st,
                       float *x, float *tout) {
  const int D = c->dim, F = c->hidden, C = c->context, bf = c->w_bf16;
  const int64_t pos = st->offset;
  float *h = (float *)malloc(sizeof(float) * D);
  float *qkv = (float *)malloc(sizeof(float) * 3 * D);
  float *attn = (float *)malloc(sizeof(float) * D);
  float *proj = (float *)malloc(sizeof(float) * D);
  float *gate = (float *)malloc(sizeof(float) * 2 * F);
  float *gated = (float *)malloc(sizeof(float) * F);
  for (int l = 0; l < c->layers; l++) {
    orc_rms_norm(x, w->norm1 + (size_t)l * D, D, c->eps, h);
    orc_gemv(woff(w->in_proj, bf, (size_t)l * 3 * D * D), bf, 3 * D, D, h, qkv);
    float *q = qkv, *k = qkv + D, *v = qkv + 2 * D;
    orc_rope_row(q, D, pos, c->head_dim, c->rope_theta);
    orc_rope_row(k, D, pos, c->head_dim, c->rope_theta);
    /* push, then evict the oldest while the window is longer than the context */
    float *K = st->k + (size_t)l * C * D, *V = st->v + (size_t)l * C * D;
    int n = st->kv_len[l];
    if (n == C) {
      memmove(K, K + D, sizeof(float) * (size_t)(C - 1) * D);
      memmove(V, V + D, sizeof(float) * (size_t)(C - 1) * D);
      n = C - 1;
    }
    for (int d = 0; d < D; d++) {
      K[(size_t)n * D + d] = c->kv_bf16 ? round_to_bf16(k[d]) : k[d];
      V[(size_t)n * D + d] = c->kv_bf16 ? round_to_bf16(v[d]) : v[d];
    }
    st->kv_len[l] = n + 1;
    orc_attend(q, K, V, n + 1, c->heads, c->head_dim, attn);
    orc_gemv(woff(w->out_proj, bf, (size_t)l * D * D), bf, D, D, attn, proj);
    for (int d = 0; d < D; d++) x[d] += proj[d];
    orc_rms_norm(x, w->norm2 + (size_t)l * D, D, c->eps, h);
    orc_gemv(woff(w->gate_in, bf, (size_t)l * 2 * F * D), bf, 2 * F, D, h, gate);
    for (int j = 0; j < F; j++) gated[j] = orc_silu(gate[j]) * gate[F + j];
    orc_gemv(woff(w->gate_out, bf, (size_t)l * D * F), bf, D, F, gated, proj);
    for (int d = 0; d < D; d++) x[d] += proj[d];
  }
  orc_rms_norm(x, w->out_norm, D, c->eps, tout);
  free(h); free(qkv); free(attn); free(proj); free(gate); free(gated);
}

/* moshi_lm.rs, `depformer_cycle`: the 8 sequential codebook steps of one frame.
 * The per-frame K/V cache starts empty; step cb's input is
 * dep_in[cb] * tout + emb(prev), prev = the text token for cb 0, else the previous
 * codebook's token; DL layers with step-cb weights, shared norms, no positional
 * rotation; then linears[cb] (no norm) and an argmax.
 * `forced` (NULL, or [text, audio0..7]) replaces prev after each step, as in
 * rlx_lm.rs `depformer_forced_logits_rlx`; `tokens` are always the own argmaxes. */
static void depformer_cycle(const orc_cfg *c, const orc_weights *w, const float *tout,
                            int64_t text_token, const int32_t *forced,
                            float *logits /*[8][A]*/, int32_t *tokens /*[8]*/,
                            const orc_sampling *smp, uint64_t *rng) {
  const int D = c->dim, DD = c->ddim, DF = c->dhidden, A = c->audio_card;
  const int DL = c->dlayers, bf = c->w_bf16, Q = ORC_DEP_Q;
  float *kc = (float *)calloc((size_t)DL * Q * DD, sizeof(float));
  float *vc = (float *)calloc((size_t)DL * Q * DD, sizeof(float));
  float *x = (float *)malloc(sizeof(float) * DD);
  float *h = (float *)malloc(sizeof(float) * DD);
  float *qkv = (float *)malloc(sizeof(float) * 3 * DD);
  float *attn = (float *)malloc(sizeof(float) * DD);
  float *proj = (float *)malloc(sizeof(float) * DD);
  float *gate = (float *)malloc(sizeof(float) * 2 * DF);
  float *gated = (float *)malloc(sizeof(float) * DF);
  int64_t prev = forced ? (int64_t)forced[0] : text_token;
  for (int cb = 0; cb < Q; cb++) {
    orc_gemv(woff(w->dep_in, bf, (size_t)cb * DD * D), bf, DD, D, tout, x);
    if (cb == 0)
      orc_embed(w->dep_text_emb, bf, DD, prev, x);
    else
      orc_embed(woff(w->dep_emb, bf, (size_t)(cb - 1) * (A + 1) * DD), bf, DD, prev, x);
    for (int l = 0; l < DL; l++) {
      size_t ls = (size_t)l * Q + cb; /* [DL][8] weight set index */
      orc_rms_norm(x, w->dnorm1 + (size_t)l * DD, DD, c->eps, h);
      orc_gemv(woff(w->d_in_proj, bf, ls * 3 * DD * DD), bf, 3 * DD, DD, h, qkv);
      float *K = kc + (size_t)l * Q * DD, *V = vc + (size_t)l * Q * DD;
      memcpy(K + (size_t)cb * DD, qkv + DD, sizeof(float) * DD);
      memcpy(V + (size_t)cb * DD, qkv + 2 * DD, sizeof(float) * DD);
      orc_attend(qkv, K, V, cb + 1, c->dheads, c->dhead_dim, attn);
      orc_gemv(woff(w->d_out_proj, bf, ls * DD * DD), bf, DD, DD, attn, proj);
      for (int d = 0; d < DD; d++) x[d] += proj[d];
      orc_rms_norm(x, w->dnorm2 + (size_t)l * DD, DD, c->eps, h);
      orc_gemv(woff(w->d_gate_in, bf, ls * 2 * DF * DD), bf, 2 * DF, DD, h, gate);
      for (int j = 0; j < DF; j++) gated[j] = orc_silu(gate[j]) * gate[DF + j];
      orc_gemv(woff(w->d_gate_out, bf, ls * DD * DF), bf, DD, DF, gated, proj);
      for (int d = 0; d < DD; d++) x[d] += proj[d];
    }
    float *lg = logits + (size_t)cb * A;
    orc_gemv(woff(w->linears, bf, (size_t)cb * A * DD), bf, A, DD, x, lg);
    tokens[cb] = (int32_t)pick(smp, rng, lg, A, 0);
    prev = forced ? (int64_t)forced[1 + cb] : (int64_t)tokens[cb];
  }
  free(kc); free(vc); free(x); free(h); free(qkv); free(attn); free(proj);
  free(gate); free(gated);
}

void orc_depformer_cycle(const orc_cfg *c, const orc_weights *w, const float *tout,
                         int64_t text_token, const int32_t *forced,
                         float *logits /*[8][A]*/, int32_t *tokens /*[8]*/) {
  depformer_cycle(c, w, tout, text_token, forced, logits, tokens, NULL, NULL);
}

/* moshi_lm.rs, `step_ext` steps 1-3 (shared by `step_forced`): write the user stream at
 * its delays, gather the model input (INITIAL tokens while offset <= delay) and sum the
 * embeddings, the 16 audio streams in order, then text, into x (zeroed by the caller). */
static void gather_embed(const orc_cfg *c, const orc_weights *w, orc_state *st,
                         const int32_t *user, int64_t *input, float *x) {
  const int D = c->dim, V = c->text_card, A = c->audio_card, bf = c->w_bf16;
  for (int k = 0; k < ORC_DEP_Q; k++) {
    int s = ORC_DEP_Q + 1 + k;
    st->ring[s][(st->offset + ORC_DELAYS[s]) % ORC_CT] = user[k];
  }
  for (int s = 0; s < ORC_STREAMS; s++) {
    if (st->offset <= ORC_DELAYS[s])
      input[s] = (s == 0) ? (int64_t)V : (int64_t)A;
    else
      input[s] = st->ring[s][st->offset % ORC_CT];
  }
  for (int k = 0; k < 16; k++)
    orc_embed(woff(w->emb, bf, (size_t)k * (A + 1) * D), bf, D, input[1 + k], x);
  orc_embed(w->text_emb, bf, D, input[0], x);
}

/* moshi_lm.rs, `MoshiLm::step_forced` (the prompt-priming primitive): steps 1-3, the
 * temporal stack at pos = offset with its output discarded (only its K/V rows stay),
 * offset + 1, and the ring records the forced [text, agent0..7].  No text head and no
 * depformer run.  emb_sum: NULL or [D]. */
void orc_prime_step(const orc_cfg *c, const orc_weights *w, orc_state *st,
                    const int32_t *forced, const int32_t *user, float *emb_sum) {
  const int D = c->dim;
  int64_t input[ORC_STREAMS];
  float *x = (float *)calloc((size_t)D, sizeof(float));
  float *tout = (float *)malloc(sizeof(float) * D);
  gather_embed(c, w, st, user, input, x);
  if (emb_sum) memcpy(emb_sum, x, sizeof(float) * D);
  orc_temporal_step(c, w, st, x, tout);
  st->offset += 1;
  int pos = (int)(st->offset % ORC_CT);
  for (int s = 0; s <= ORC_DEP_Q; s++) st->ring[s][pos] = forced[s];
  free(x);
  free(tout);
}

/* moshi_lm.rs, `MoshiState::advance_clock` after the temporal consumed a precomputed
 * embedding row (the voice-prompt replay): the temporal stack on x at pos = offset, then
 * offset + 1; the ring is not touched. */
void orc_replay_step(const orc_cfg *c, const orc_weights *w, orc_state *st, const float *x_in) {
  const int D = c->dim;
  float *x = (float *)malloc(sizeof(float) * D);
  float *tout = (float *)malloc(sizeof(float) * D);
  memcpy(x, x_in, sizeof(float) * D);
  orc_temporal_step(c, w, st, x, tout);
  st->offset += 1;
  free(x);
  free(tout);
}

/* moshi_lm.rs, `MoshiState::snapshot`: an independent copy of the session (ring, offset,
 * K/V window, sampler). */
orc_state *orc_state_clone(const orc_state *st) {
  orc_state *o = (orc_state *)malloc(sizeof(orc_state));
  if (!o) return NULL;
  memcpy(o, st, sizeof(orc_state));
  size_t n = (size_t)st->layers * st->context * st->dim;
  o->kv_len = (int32_t *)malloc(sizeof(int32_t) * (size_t)st->layers);
  o->k = (float *)malloc(sizeof(float) * n);
  o->v = (float *)malloc(sizeof(float) * n);
  if (!o->kv_len || !o->k || !o->v) {
    free(o->kv_len); free(o->k); free(o->v); free(o);
    return NULL;
  }
  memcpy(o->kv_len, st->kv_len, sizeof(int32_t) * (size_t)st->layers);
  memcpy(o->k, st->k, sizeof(float) * n);
  memcpy(o->v, st->v, sizeof(float) * n);
  return o;
}

/* moshi_lm.rs, `step_ext` (steps 1-8) for one session.
 * user: [8] user-audio codes; forced: NULL or [9] = [text, audio0..7].
 * own: [9] the step's own argmax tokens [text, audio0..7].
 * out / has_out: the delay-realigned [text, audio0..7] once offset > max_delay.
 * Trace buffers (any may be NULL): input_tokens [17], emb_sum [D], tout [D],
 * text_logits [V], audio_logits [8][A]. */
void orc_step(const orc_cfg *c, const orc_weights *w, orc_state *st,
              const int32_t *user, const int32_t *forced, int32_t *own,
              int32_t *out, int32_t *has_out, int64_t *input_tokens,
              float *emb_sum, float *tout_o, float *text_logits_o,
              float *audio_logits_o) {
  const int D = c->dim, V = c->text_card, A = c->audio_card, bf = c->w_bf16;
  /* 1-3. user codes, gathered input, embedding sum */
  int64_t input[ORC_STREAMS];
  float *x = (float *)calloc((size_t)D, sizeof(float));
  gather_embed(c, w, st, user, input, x);
  if (emb_sum) memcpy(emb_sum, x, sizeof(float) * D);
  if (input_tokens) memcpy(input_tokens, input, sizeof(input));
  /* 4-5. temporal step and text head */
  float *tout = (float *)malloc(sizeof(float) * D);
  float *tl = (float *)malloc(sizeof(float) * V);
  float *al = (float *)malloc(sizeof(float) * ORC_DEP_Q * A);
  orc_temporal_step(c, w, st, x, tout);
  orc_gemv(w->text_linear, bf, V, D, tout, tl);
  int32_t text_token = (int32_t)pick(&st->smp, &st->rng, tl, V, 1);
  /* 6. depformer cycle */
  int32_t audio[ORC_DEP_Q];
  depformer_cycle(c, w, tout, text_token, forced, al, audio, &st->smp, &st->rng);
  /* 7. advance and self-feed (forced tokens are what the ring records) */
  st->offset += 1;
  int pos = (int)(st->offset % ORC_CT);
  st->ring[0][pos] = forced ? forced[0] : text_token;
  for (int cb = 0; cb < ORC_DEP_Q; cb++)
    st->ring[1 + cb][pos] = forced ? forced[1 + cb] : audio[cb];
  /* 8. delay-realigned output once past max_delay */
  if (st->offset > ORC_MAX_DELAY) {
    for (int s = 0; s <= ORC_DEP_Q; s++)
      out[s] = (int32_t)st->ring[s][(st->offset - ORC_MAX_DELAY + ORC_DELAYS[s]) % ORC_CT];
    *has_out = 1;
  } else {
    for (int s = 0; s <= ORC_DEP_Q; s++) out[s] = 0;
    *has_out = 0;
  }
  own[0] = text_token;
  for (int cb = 0; cb < ORC_DEP_Q; cb++) own[1 + cb] = audio[cb];
  if (tout_o) memcpy(tout_o, tout, sizeof(float) * D);
  if (text_logits_o) memcpy(text_logits_o, tl, sizeof(float) * V);
  if (audio_logits_o) memcpy(audio_logits_o, al, sizeof(float) * ORC_DEP_Q * A);
  free(x); free(tout); free(tl); free(al);
}

/* ---------------------------------------------------------------- misc */

void orc_set_threads(int32_t n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int32_t orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

float orc_round_to_bf16(float f) { return round_to_bf16(f); }
