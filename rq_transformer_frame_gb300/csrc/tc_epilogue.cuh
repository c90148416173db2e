// tc_epilogue.cuh -- pieces shared by the tensor-core GEMM kernels (one launch per linear,
// and the persistent batched depformer): tile geometry, the fused epilogues of one
// 16-session chunk of an accumulator tile, and the tensor-memory read of a tile over the bf16 operand parts.
#pragma once

#include <cuda_bf16.h>

#include "kernels.h"
#include "sampling.cuh"
#include "tc_common.cuh"

namespace rqk {
namespace tcg {

constexpr int kThreads = 192;
constexpr int kBM = 128;  // rows of W per tile
constexpr int kBK = 64;   // K elements per stage (128 bytes of bf16)
constexpr int kABytes = kBM * kBK * 2;


__device__ __forceinline__ void store_kv_tc(void* base, size_t i, float v, int bf16) {
  if (bf16)
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(base)[i] = v;
}


// Fused epilogue of columns c0..c0+15 (sessions) of one 128-row tile, this thread's row m
// of the tile = tensor-memory lane m.  Mirrors the streaming GEMV's epilogues, batched.
struct EpiShared {
  float ex[2][64][16];                 // SiLU gate: multiplier rows -> gate rows
  unsigned long long key[4][64];       // argmax: best key per lane quarter and session
  float ss[4][64];                     // fused RMSNorm: sum of squares per lane quarter
  float inv[64];                       // fused RMSNorm: 1 / rms of each session's input
};

// The next GEMM's operand for a new residual value v of row `row`, session b (fused
// RMSNorm, see TcParams); `an` = alpha_next[row], loaded once by the caller (1 without).
__device__ __forceinline__ void feed_next(const TcParams& p, int row, bool valid, int b,
                                          float v, float an) {
  const TcPlan& pl = p.pl;
  if (valid)
    store_bf16_parts(p.opnd, (size_t)pl.NB * pl.n_out, (size_t)b * pl.n_out + row,
                     b < p.B ? v * an : 0.f);
}

// Sum over the warp's 32 rows of each of 16 per-lane values with 16 shuffles (a
// transposing butterfly: every step halves the values a lane keeps); the lanes with bit 0
// clear end with the sum for column ((lane >> 1) & 15) bit-reversed into place below.
__device__ __forceinline__ void tile_sumsq(float (&sq)[16], int lane, int q, int c0,
                                           EpiShared& es) {
  float w8[8], w4[4], w2[2];
  {
    const bool hi = (lane & 16) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float send = hi ? sq[i] : sq[i + 8];
      const float keep = hi ? sq[i + 8] : sq[i];
      w8[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  {
    const bool hi = (lane & 8) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float send = hi ? w8[i] : w8[i + 4];
      const float keep = hi ? w8[i + 4] : w8[i];
      w4[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
  }
  {
    const bool hi = (lane & 4) != 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float send = hi ? w4[i] : w4[i + 2];
      const float keep = hi ? w4[i + 2] : w4[i];
      w2[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
  }
  const bool hi = (lane & 2) != 0;
  float w1 = (hi ? w2[1] : w2[0]) + __shfl_xor_sync(0xffffffffu, hi ? w2[0] : w2[1], 2);
  w1 += __shfl_xor_sync(0xffffffffu, w1, 1);
  // column kept: bit 4 of the lane chose 8, bit 3 chose 4, bit 2 chose 2, bit 1 chose 1
  const int col = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 +
                  ((lane >> 1) & 1);
  if ((lane & 1) == 0) es.ss[q][c0 + col] = w1;
}

// Every read of a chunk's epilogue (tables, positions, tokens) is issued before its first
// store: the compiler may not move a load across a store to a possibly aliasing pointer,
// and one round trip to L2 per session and chunk made the batch-64 qkv epilogue cost
// three times the GEMM's main loop.
__device__ __forceinline__ void epilogue_chunk(const TcParams& p, const float (&d)[16], int c0,
                                               int tile, int m, int lane, int q, EpiShared& es,
                                               const float (&old0)[16]) {
  const TcPlan& pl = p.pl;
  const int B = p.B;
  const int epi = p.epi;
  if (epi == EPI_SWIGLU) {
    // "moshi_lm.rs": silu(gate_j) * mult_j; the multiplier rows (64..127) hand their
    // values to the gate rows (0..63) through shared memory (double-buffered by chunk)
    float(*ex)[16] = es.ex[(c0 >> 4) & 1];
    if (m >= 64) {
#pragma unroll
      for (int i = 0; i < 16; ++i) ex[m - 64][i] = d[i];
    }
    bar_sync(1, 128);
    const int j = tile * 64 + m;
    if (m < 64 && j < pl.n_out) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float g = d[i], mu = ex[m][i];
        store_bf16_parts(p.out_bf16, (size_t)pl.NB * p.outb_bs, (size_t)(c0 + i) * p.outb_bs + j,
                     g / (1.0f + expf(-g)) * mu);
      }
    }
    return;
  }
  const int row = tile * kBM + m;
  const bool valid = row < pl.n_out;
  const float an = (p.opnd && p.alpha_next && valid) ? __ldg(p.alpha_next + row) : 1.0f;
  if (epi == EPI_RESID || epi == EPI_STORE) {
    float sq[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float nv = 0.f;
      if (valid && c0 + i < B) {
        float* o = p.out + (size_t)(c0 + i) * p.out_bs + row;
        nv = (epi == EPI_RESID ? old0[i] : 0.f) + d[i];
        *o = nv;
      }
      sq[i] = nv * nv;
      if (p.opnd) feed_next(p, row, valid, c0 + i, nv, an);
    }
    if (p.ss_out) tile_sumsq(sq, lane, q, c0, es);
  } else if (epi == EPI_QKV) {
    // "moshi_lm.rs", `rope_row` on q, k at each session's position, K/V append
    const int D = pl.n_out / 3;
    const int region = row / D, col = row % D;
    const bool odd = (lane & 1) != 0;
    // each session's (cos, sin) of this pair and its cache slot, all loaded first
    float2 rr[16];
    int slot[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int b = c0 + i;
      const bool ok = valid && b < B;
      rr[i] = (ok && region < 2)
                  ? __ldg(p.rope + (size_t)b * (p.head_dim / 2) + (col % p.head_dim) / 2)
                  : make_float2(1.f, 0.f);
      slot[i] = (ok && region > 0) ? __ldg(p.offsets + b) : 0;
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int b = c0 + i;
      const float partner = __shfl_xor_sync(0xffffffffu, d[i], 1);
      if (!valid || b >= B) continue;
      float v = d[i];
      if (region < 2) {
        const float2 r = rr[i];
        const float re = odd ? partner : v, im = odd ? v : partner;
        v = odd ? re * r.y + im * r.x : re * r.x - im * r.y;
      }
      if (region == 0) {
        p.out[(size_t)b * p.out_bs + col] = v;
      } else {
        store_kv_tc(region == 1 ? p.kcache : p.vcache,
                    (size_t)b * p.kv_bs + (size_t)(slot[i] % p.context) * D + col, v,
                    p.kv_bf16);
      }
    }
  } else if (epi == EPI_DQKV) {
    const int DD = pl.n_out / 3;
    if (valid)
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int b = c0 + i;
        if (b >= B) continue;
        if (row < DD)
          p.out[(size_t)b * p.out_bs + row] = d[i];
        else if (row < 2 * DD)
          p.dk_out[(size_t)b * p.dkv_bs + row - DD] = d[i];
        else
          p.dv_out[(size_t)b * p.dkv_bs + row - 2 * DD] = d[i];
      }
  } else if (epi == EPI_DEPIN) {
    // "moshi_lm.rs", `embed` of the previous step's token: -1 adds nothing.  The tokens,
    // then the embedding values, are loaded for the whole chunk before any store.
    const IoLayout io{p.B};
    int tok[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int b = c0 + i;
      tok[i] = -1;
      if (valid && b < B)
        tok[i] = p.d_in[io.flag_off() + b]
                     ? p.d_in[io.forced_off() + (size_t)b * 9 + p.key_index]
                     : argmax_key_index(p.keys[(size_t)b * 9 + p.key_index]);
    }
    float e[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      e[i] = tok[i] != -1 ? __uint_as_float(((uint32_t)static_cast<const uint16_t*>(
                                                 p.emb)[(size_t)max(tok[i], 0) * pl.n_out + row])
                                             << 16)
                          : 0.f;
    float sq[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int b = c0 + i;
      float nv = 0.f;
      if (valid && b < B) {
        nv = d[i] + e[i];
        p.out[(size_t)b * p.out_bs + row] = nv;
      }
      sq[i] = nv * nv;
      if (p.opnd) feed_next(p, row, valid, b, nv, an);
    }
    if (p.ss_out) tile_sumsq(sq, lane, q, c0, es);
  } else if (epi == EPI_ARGMAX) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int b = c0 + i;
      unsigned long long k = 0ull;
      if (valid && b < B) {
        p.out[(size_t)b * p.out_bs + row] = d[i];
        k = pick_key(p.samp, b, p.key_index, d[i], (uint32_t)row);
      }
      k = warp_max_u64(k);
      if (lane == 0) es.key[q][b] = k;
    }
  }
}

// columns c0..c0+15 of this lane's accumulator row: (lo + mid) + hi of each session
template <int NB>
__device__ __forceinline__ void load_sum3(uint32_t taddr, int c0, float (&v)[16]) {
  float h[16], m[16];
  tc::tmem_ld16(taddr + (uint32_t)c0, h);
  tc::tmem_ld16(taddr + (uint32_t)(NB + c0), m);
  if (kOpndParts == 3) {
    tc::tmem_ld16(taddr + (uint32_t)(2 * NB + c0), v);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = (v[i] + m[i]) + h[i];
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = m[i] + h[i];
  }
}

}  // namespace tcg
}  // namespace rqk
