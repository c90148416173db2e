// sampling.cuh -- device side of the token picks ("moshi_lm.rs", `pick`,
// `xorshift_u01`, `gumbel_full_pick`, `topk_sample`).
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace rqk {

// the state after n further xorshift64 steps: M^n s, from the columns of M^(2^k)
__device__ __forceinline__ uint64_t xs_advance(uint64_t s, uint32_t n, const uint64_t* jump) {
  for (int k = 0; n != 0u; ++k, n >>= 1) {
    if (!(n & 1u)) continue;
    const uint64_t* col = jump + k * 64;
    uint64_t y = 0ull;
#pragma unroll 8
    for (int b = 0; b < 64; ++b) y ^= __ldg(col + b) & (0ull - ((s >> b) & 1ull));
    s = y;
  }
  return s;
}

// "moshi_lm.rs", `xorshift_u01`: the top 53 bits of a generated value over 2^53
__device__ __forceinline__ double xs_u01(uint64_t x) {
  return (double)(x >> 11) * (1.0 / 9007199254740992.0);
}

// draws made before pick p of a frame (p = 0 text, 1 + cb codebook cb)
__device__ __forceinline__ uint32_t draws_before(const SampleParams& sp, int p) {
  if (sp.mode == SAMPLE_GUMBEL) return p == 0 ? 0u : (uint32_t)sp.V + (uint32_t)(p - 1) * sp.A;
  return (uint32_t)p;  // top-k: one draw per pick
}

// the key a row competes with in pick p: its logit (greedy, top-k), or "moshi_lm.rs"
// `gumbel_full_pick`'s score y / temp + g with g = -ln(-ln u) in f64 rounded to f32,
// u the row's own draw (at least 1e-300)
__device__ __forceinline__ unsigned long long pick_key(const SampleParams& sp, int b, int p,
                                                       float y, uint32_t row) {
  if (sp.mode != SAMPLE_GUMBEL) return argmax_key(y, row);
  const uint64_t x = xs_advance(sp.rng[b], draws_before(sp, p) + row + 1u, sp.jump);
  double u = xs_u01(x);
  u = u < 1e-300 ? 1e-300 : u;
  const float g = (float)(-log(-log(u)));
  const float temp = p == 0 ? sp.temp_text : sp.temp;
  return argmax_key(y / temp + g, row);
}

// CTA barriers for topk_pick_block
struct SyncBlock {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};
template <int N>
struct SyncNamed {  // named barrier 1 over the first N threads
  __device__ __forceinline__ void operator()() const { bar_sync(1, N); }
};

// ---------------------------------------------------------------- top-k pick
struct TopkShared {
  unsigned long long cand[kTopKMax];
  double p[kTopKMax];
  unsigned int hist[256];
  unsigned int wcount[32];
  unsigned int misc[4];
};

constexpr int kTkBatch = 8;  // logits loaded per thread before any is used

// f32 total order (-NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN) as an unsigned key
__device__ __forceinline__ uint32_t total_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// "moshi_lm.rs", `topk_sample` over logits lg[0..n) by the nthr threads tid of one CTA
// (`sync` a barrier of exactly those threads): the k largest logits in descending order
// (equal logits by ascending index), p_i = exp(((l_i - max) / temp) widened to f64)
// normalised by their sequential sum, and the first i where u - p_0 - ... - p_i <= 0.
// Returns the token in every thread.
template <typename Sync>
__device__ int topk_pick_block(const float* lg, int n, int k, float temp, double u, int tid,
                               int nthr, TopkShared& S, Sync sync) {
  k = k < 1 ? 1 : (k > n ? n : k);
  k = k > kTopKMax ? kTopKMax : k;
  // 1. the k-th largest total-order key T (radix select, 8 bits a pass)
  uint32_t prefix = 0u, mask = 0u;
  int remaining = k;  // how many of the keys matching the prefix are still needed
  unsigned int n_eq = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += nthr) S.hist[i] = 0u;
    sync();
    // kTkBatch loads in flight per thread; logits cluster in a few bins, so lanes with
    // equal bins add once, by their count
    for (int base = 0; base < n; base += kTkBatch * nthr) {
      uint32_t key[kTkBatch];
#pragma unroll
      for (int j = 0; j < kTkBatch; ++j) {
        const int i = base + j * nthr + tid;
        key[j] = i < n ? total_key(__ldcg(lg + i)) : 0u;
      }
#pragma unroll
      for (int j = 0; j < kTkBatch; ++j) {
        const int i = base + j * nthr + tid;
        const unsigned bin = (i < n && (key[j] & mask) == prefix) ? (key[j] >> shift) & 255u : 256u;
        const unsigned same = __match_any_sync(0xffffffffu, bin);
        if (bin < 256u && (tid & 31) == __ffs(same) - 1) atomicAdd(&S.hist[bin], __popc(same));
      }
    }
    sync();
    if (tid == 0) {
      int acc = 0, d = 255;
      for (; d > 0; --d) {
        if (acc + (int)S.hist[d] >= remaining) break;
        acc += (int)S.hist[d];
      }
      S.misc[0] = (unsigned)d;
      S.misc[1] = (unsigned)(remaining - acc);
      S.misc[2] = S.hist[d];
    }
    sync();
    prefix |= S.misc[0] << shift;
    mask |= 255u << shift;
    remaining = (int)S.misc[1];
    n_eq = S.misc[2];
    sync();  // misc is rewritten by the next pass
  }
  const uint32_t T = prefix;
  // 2. candidates: every key above T, then the `remaining` lowest indices equal to T
  if (tid == 0) S.misc[3] = 0u;
  sync();
  const bool all_eq = n_eq == (unsigned)remaining;
  for (int base = 0; base < n; base += kTkBatch * nthr) {
    uint32_t key[kTkBatch];
#pragma unroll
    for (int j = 0; j < kTkBatch; ++j) {
      const int i = base + j * nthr + tid;
      key[j] = i < n ? total_key(__ldcg(lg + i)) : 0u;
    }
#pragma unroll
    for (int j = 0; j < kTkBatch; ++j) {
      const int i = base + j * nthr + tid;
      if (i < n && (key[j] > T || (all_eq && key[j] == T))) {
        const unsigned slot = atomicAdd(&S.misc[3], 1u);
        if (slot < (unsigned)kTopKMax)  // exactly k keys qualify (counted by the passes)
          S.cand[slot] = ((unsigned long long)key[j] << 32) | (0xffffffffu - (uint32_t)i);
      }
    }
  }
  sync();
  if (!all_eq) {
    const int lane = tid & 31, warp = tid >> 5, nw = (nthr + 31) >> 5;
    int taken = 0;
    const int first = k - remaining;
    for (int base = 0; base < n && taken < remaining; base += nthr) {
      const int i = base + tid;
      const bool eq = i < n && total_key(__ldcg(lg + i)) == T;
      const unsigned bal = __ballot_sync(0xffffffffu, eq);
      if (lane == 0) S.wcount[warp] = __popc(bal);
      sync();
      int before = __popc(bal & ((1u << lane) - 1u)), total = 0;
      for (int w = 0; w < nw; ++w) {
        if (w < warp) before += (int)S.wcount[w];
        total += (int)S.wcount[w];
      }
      if (eq && taken + before < remaining)
        S.cand[first + taken + before] = ((unsigned long long)T << 32) | (0xffffffffu - (uint32_t)i);
      taken += total;
      sync();
    }
  }
  // 3. sort the k candidates (distinct keys) ascending; pad to a power of two with 0
  int P = 1;
  while (P < k) P <<= 1;
  for (int i = k + tid; i < P; i += nthr) S.cand[i] = 0ull;
  sync();
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P; i += nthr) {
        const int j = i ^ stride;
        if (j > i) {
          const unsigned long long a = S.cand[i], c = S.cand[j];
          if (((i & size) == 0) ? (a > c) : (a < c)) {
            S.cand[i] = c;
            S.cand[j] = a;
          }
        }
      }
      sync();
    }
  }
  // descending rank r is S.cand[P - 1 - r]
  // 4. probabilities in f64, their sequential sum, one draw
  for (int r = tid; r < k; r += nthr) {
    const int idx = (int)(0xffffffffu - (uint32_t)(S.cand[P - 1 - r] & 0xffffffffull));
    S.p[r] = (double)__ldcg(lg + idx);  // the logit, exactly
  }
  sync();
  if (tid == 0) {  // the page's max fold (NaN-ignoring f32 max from -inf)
    float mx = -__int_as_float(0x7f800000);
    for (int r = 0; r < k; ++r) mx = fmaxf(mx, (float)S.p[r]);
    S.misc[1] = __float_as_uint(mx);
  }
  sync();
  const float mx = __uint_as_float(S.misc[1]);
  for (int r = tid; r < k; r += nthr) S.p[r] = exp((double)(((float)S.p[r] - mx) / temp));
  sync();
  if (tid == 0) {  // the sum in order, then every p_i / sum in parallel
    double sum = 0.0;
    for (int r = 0; r < k; ++r) sum += S.p[r];
    S.misc[2] = (unsigned)__double2hiint(sum);
    S.misc[3] = (unsigned)__double2loint(sum);
  }
  sync();
  {
    const double sum = __hiloint2double((int)S.misc[2], (int)S.misc[3]);
    for (int r = tid; r < k; r += nthr) S.p[r] = S.p[r] / sum;
  }
  sync();
  if (tid == 0) {
    int tok = (int)(0xffffffffu - (uint32_t)(S.cand[P - k] & 0xffffffffull));
    double left = u;
    for (int r = 0; r < k; ++r) {
      left -= S.p[r];
      if (left <= 0.0) {
        tok = (int)(0xffffffffu - (uint32_t)(S.cand[P - 1 - r] & 0xffffffffull));
        break;
      }
    }
    S.misc[0] = (unsigned)tok;
  }
  sync();
  const int tok = (int)S.misc[0];
  sync();
  return tok;
}

}  // namespace rqk
