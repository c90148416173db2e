// gemv.cu -- weight-streaming GEMV with fused prologues and epilogues (sm_103a).
//
// Every linear of the decode step at batch 1 is y = W x with W [rows][K] read exactly
// once per frame ("inferencelayer 0.2.4 -- src/moshi_lm.rs", `Band::mv`), so the
// kernel is bound by HBM bandwidth.  Design:
//   * one CTA per SM (grid = #SMs; two CTAs of consecutive kernels fit on an SM),
//     each owning a contiguous run of row tiles, i.e. one contiguous byte range of W;
//   * a producer warp streams tiles with cp.async.bulk into an mbarrier ring of
//     shared-memory stages (L2 evict-first: weights are not reused within a frame);
//     the first stages are issued BEFORE griddepcontrol.wait, so with programmatic
//     dependent launch the weight stream of this GEMV overlaps the tail of the
//     previous kernel;
//   * 8 consumer warps keep their slice of x in registers (formed by the fused
//     prologue: plain, RMSNorm, or the depformer's tiny attention) and read each
//     weight element once from shared memory; per-warp partial sums of each row are
//     kept in shared memory and reduced in a fixed order (deterministic);
//   * the epilogue fuses what follows the linear on the page: residual add, SiLU gate,
//     rotary embedding + K/V append, depformer K/V append, logits + first-wins argmax,
//     depformer conditioning embedding.
#pragma once
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "sampling.cuh"

namespace rqk {

constexpr int kConsumers = kGemvConsumers;  // 8 consumer warps
constexpr int kThreads = 288;    // + 1 producer warp
constexpr int kMaxAttPairs = 32 * 8;

template <typename WT>
struct Chunk;

template <>
struct Chunk<uint16_t> {  // bf16 bit patterns
  static constexpr int V = 8;
  static constexpr bool kBand = false;
  using Table = uint16_t;
  static __host__ __device__ size_t row_bytes(int K) { return (size_t)K * 2; }
  static __device__ __forceinline__ float dot(const uint4 w, const float (&x)[8], float acc) {
    acc = fmaf(bf16lo(w.x), x[0], acc);
    acc = fmaf(bf16hi(w.x), x[1], acc);
    acc = fmaf(bf16lo(w.y), x[2], acc);
    acc = fmaf(bf16hi(w.y), x[3], acc);
    acc = fmaf(bf16lo(w.z), x[4], acc);
    acc = fmaf(bf16hi(w.z), x[5], acc);
    acc = fmaf(bf16lo(w.w), x[6], acc);
    acc = fmaf(bf16hi(w.w), x[7], acc);
    return acc;
  }
  static __device__ __forceinline__ void dot2(const uint4 w, const float (&x)[8], float& a,
                                              float& b) {
    a = fmaf(bf16lo(w.x), x[0], a);
    b = fmaf(bf16hi(w.x), x[1], b);
    a = fmaf(bf16lo(w.y), x[2], a);
    b = fmaf(bf16hi(w.y), x[3], b);
    a = fmaf(bf16lo(w.z), x[4], a);
    b = fmaf(bf16hi(w.z), x[5], b);
    a = fmaf(bf16lo(w.w), x[6], a);
    b = fmaf(bf16hi(w.w), x[7], b);
  }
  static __device__ __forceinline__ float elem(const void* base, size_t i) {
    return __uint_as_float(((uint32_t)(static_cast<const uint16_t*>(base)[i])) << 16);
  }
};

template <>
struct Chunk<float> {
  static constexpr int V = 4;
  static constexpr bool kBand = false;
  using Table = float;
  static __host__ __device__ size_t row_bytes(int K) { return (size_t)K * 4; }
  static __device__ __forceinline__ float dot(const uint4 w, const float (&x)[4], float acc) {
    acc = fmaf(__uint_as_float(w.x), x[0], acc);
    acc = fmaf(__uint_as_float(w.y), x[1], acc);
    acc = fmaf(__uint_as_float(w.z), x[2], acc);
    acc = fmaf(__uint_as_float(w.w), x[3], acc);
    return acc;
  }
  static __device__ __forceinline__ void dot2(const uint4 w, const float (&x)[4], float& a,
                                              float& b) {
    a = fmaf(__uint_as_float(w.x), x[0], a);
    b = fmaf(__uint_as_float(w.y), x[1], b);
    a = fmaf(__uint_as_float(w.z), x[2], a);
    b = fmaf(__uint_as_float(w.w), x[3], b);
  }
  static __device__ __forceinline__ float elem(const void* base, size_t i) {
    return static_cast<const float*>(base)[i];
  }
};

// Weight bands (kernels.h: codes, then one f32 scale per 32 values of the row).  Value i
// is (float)q_i * d, multiplied with x_i as the dequantized weight would be; the tables
// of a band model stay bf16.
template <>
struct Chunk<q8_t> {
  static constexpr int V = 16;  // 16 one-byte codes per 16-byte chunk: half a group
  static constexpr bool kBand = true;
  using Table = uint16_t;
  static __host__ __device__ size_t row_bytes(int K) { return band_row_bytes(BAND_Q8, 1, K); }
  static __device__ __forceinline__ size_t scale_off(int K, int c) {
    return (size_t)K + (size_t)(c >> 1) * 4;
  }
  // sum_i q_i x_i, then times d: each code becomes a float with one byte permute and one
  // add (2^23 + 128 + q has the bits 0x4B0000nn, nn = q + 128), no int-to-float convert
  static __device__ __forceinline__ void dot2s(const uint4 w, float d, const float (&x)[16],
                                               float& a, float& b) {
    const uint32_t u[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u,
                           w.w ^ 0x80808080u};
    float sa = 0.f, sb = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float q = __uint_as_float(__byte_perm(u[k], 0x4B000000u, 0x7640u + j)) -
                        8388736.0f;
        if (j & 1)
          sb = fmaf(q, x[4 * k + j], sb);
        else
          sa = fmaf(q, x[4 * k + j], sa);
      }
    a = fmaf(sa, d, a);
    b = fmaf(sb, d, b);
  }
};

// two f32 lanes in one 64-bit register pair, with the packed add and FMA of sm_100+
typedef unsigned long long gv_f32x2;
__device__ __forceinline__ gv_f32x2 gv_pack2(float a, float b) {
  gv_f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void gv_unpack2(gv_f32x2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ gv_f32x2 gv_add2(gv_f32x2 a, gv_f32x2 b) {
  gv_f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ void gv_fma2(gv_f32x2& d, gv_f32x2 a, gv_f32x2 b) {  // d += a * b
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

template <>
struct Chunk<q4_t> {
  static constexpr int V = 32;  // one group: byte i holds values i and i + 16
  static constexpr bool kBand = true;
  using Table = uint16_t;
  static __host__ __device__ size_t row_bytes(int K) { return band_row_bytes(BAND_Q4, 1, K); }
  static __device__ __forceinline__ size_t scale_off(int K, int c) {
    return (size_t)K / 2 + (size_t)c * 4;
  }
  // sum_i (q_i - 8) x_i, then times d: one mask per word of codes, one byte permute per
  // code (the bits 0x4B00000n are 2^23 + n) and, two at a time, one packed add
  static __device__ __forceinline__ void dot2s(const uint4 w, float d, const float (&x)[32],
                                               float& a, float& b) {
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    const gv_f32x2 off = gv_pack2(-8388616.0f, -8388616.0f);
    gv_f32x2 sl = gv_pack2(0.f, 0.f), sh = gv_pack2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t lo = u[k] & 0x0F0F0F0Fu, hi = (u[k] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        const gv_f32x2 l =
            gv_add2(gv_pack2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7640u + j)),
                             __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7641u + j))),
                    off);
        const gv_f32x2 h =
            gv_add2(gv_pack2(__uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7640u + j)),
                             __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7641u + j))),
                    off);
        gv_fma2(sl, l, gv_pack2(x[4 * k + j], x[4 * k + j + 1]));       // values 4k + j, +1
        gv_fma2(sh, h, gv_pack2(x[4 * k + j + 16], x[4 * k + j + 17]));  // the same + 16
      }
    }
    float p0, p1, p2, p3;
    gv_unpack2(sl, p0, p1);
    gv_unpack2(sh, p2, p3);
    a = fmaf(p0 + p1, d, a);
    b = fmaf(p2 + p3, d, b);
  }
};

__device__ __forceinline__ void store_kv(void* base, size_t i, float v, int bf16) {
  if (bf16)
    static_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(base)[i] = v;
}

// NCH: 16-byte chunks of x held per thread; RG: rows each thread accumulates per
// tile.  Small NCH leaves registers for two CTAs of this kernel plus two of the next
// one (programmatic dependent launch) on every SM.
template <int NCH>
struct GemvShape {
  static constexpr int RG = NCH <= 2 ? 2 : 1;
  static constexpr int MIN_BLOCKS = NCH <= 2 ? 4 : 2;
};

template <typename WT, int PRO, int EPI, int NCH>
__global__ void __launch_bounds__(kThreads, Chunk<WT>::kBand ? 2 : GemvShape<NCH>::MIN_BLOCKS)
    gemv_kernel(const GemvParams p) {
  constexpr int V = Chunk<WT>::V;
  constexpr int RG = Chunk<WT>::kBand ? (V * NCH <= 32 ? 2 : 1) : GemvShape<NCH>::RG;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_red[kConsumers / 32];
  __shared__ float s_att[kMaxAttPairs];
  __shared__ unsigned long long s_key[kThreads / 32];
  __shared__ volatile int s_abort;
  __shared__ int s_issued;

  const GemvPlan& pl = p.pl;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y;
  const int G = gridDim.x;
  const int t0 = (int)(((long long)pl.tiles * blockIdx.x) / G);
  const int t1 = (int)(((long long)pl.tiles * (blockIdx.x + 1)) / G);
  const int nt = t1 - t0;
  const int K = pl.K;
  const uint32_t row_bytes = (uint32_t)Chunk<WT>::row_bytes(K);
  const uint32_t tile_bytes = row_bytes * (uint32_t)pl.tile_rows;
  const int NS = pl.n_stages;
  const int wpg = pl.tpr >> 5;
  const int out_per_tile = (EPI == EPI_SWIGLU) ? (pl.tile_rows >> 1) : pl.tile_rows;

  uint8_t* stages = smem;
  float* part = reinterpret_cast<float*>(smem + (size_t)NS * tile_bytes);
  const int part_n = (pl.max_tiles * pl.tile_rows * wpg + 3) & ~3;
  uint64_t* full = reinterpret_cast<uint64_t*>(part + part_n);
  uint64_t* empty = full + NS;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumers / 32);
    }
    fence_barrier_init();
    s_abort = 0;
    s_issued = 0;
  }
  __syncthreads();
  pdl_trigger();

  if (warp == kConsumers / 32) {
    // ------------------------------------------------------------ producer warp
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      const uint8_t* W = static_cast<const uint8_t*>(p.W);
      int i = 0;
      for (; i < nt; ++i) {
        const int s = i % NS;
        if (i >= NS) {
          if (!mbar_wait(&empty[s], (uint32_t)(((i / NS) - 1) & 1))) {
            atomicOr(p.status, kDevTimeout);
            s_abort = 1;
            break;
          }
        }
        if (s_abort) break;
        const int r0 = (t0 + i) * out_per_tile;
        const int nv = min(out_per_tile, pl.n_out - r0);
        const uint32_t bytes = (uint32_t)nv * row_bytes;
        uint8_t* dst = stages + (size_t)s * tile_bytes;
        if (EPI == EPI_SWIGLU) {
          mbar_arrive_expect_tx(&full[s], 2u * bytes);
          bulk_g2s(dst, W + (size_t)r0 * row_bytes, bytes, &full[s], pol);
          bulk_g2s(dst + (size_t)out_per_tile * row_bytes,
                   W + (size_t)p.w_half + (size_t)r0 * row_bytes, bytes, &full[s],
                   pol);
        } else {
          mbar_arrive_expect_tx(&full[s], bytes);
          bulk_g2s(dst, W + (size_t)r0 * row_bytes, bytes, &full[s], pol);
        }
      }
      s_issued = i;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumer warps
    pdl_wait();
    const int g = tid / pl.tpr, tig = tid % pl.tpr;
    const int CC = K / V;
    float xr[NCH][V];
    const float* in = p.in + (size_t)b * p.in_bs;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = tig + j * pl.tpr;
#pragma unroll
      for (int v = 0; v < V; ++v) xr[j][v] = 0.f;
      if (PRO != PRO_DATTN && c < CC) {
#pragma unroll
        for (int v = 0; v < V; v += 4) {
          const float4 f = *reinterpret_cast<const float4*>(in + (size_t)c * V + v);
          xr[j][v] = f.x;
          xr[j][v + 1] = f.y;
          xr[j][v + 2] = f.z;
          xr[j][v + 3] = f.w;
        }
      }
    }
    if (PRO == PRO_RMS) {
      // "moshi_lm.rs", `rms_norm`: x * alpha * (1 / sqrt(eps + sum(x^2) / n)).
      // Every row group holds the whole vector: group 0's warps sum the squares from
      // registers.
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < NCH; ++j)
#pragma unroll
        for (int v = 0; v < V; ++v) ss = fmaf(xr[j][v], xr[j][v], ss);
      ss = warp_sum(ss);
      if (lane == 0) s_red[warp] = ss;
      bar_sync(1, kConsumers);
      float tot = 0.f;
      for (int w = 0; w < pl.tpr / 32; ++w) tot += s_red[w];
      const float inv = 1.0f / sqrtf(p.eps + tot / (float)K);
      const bool side = p.side_out != nullptr && blockIdx.x == 0 && g == 0;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int c = tig + j * pl.tpr;
        if (c < CC) {
#pragma unroll
          for (int v = 0; v < V; v += 4) {  // alpha rows are 16-byte aligned (dims % 8)
            const float4 a = *reinterpret_cast<const float4*>(p.alpha + c * V + v);
            xr[j][v] = xr[j][v] * a.x * inv;
            xr[j][v + 1] = xr[j][v + 1] * a.y * inv;
            xr[j][v + 2] = xr[j][v + 2] * a.z * inv;
            xr[j][v + 3] = xr[j][v + 3] * a.w * inv;
          }
          if (side) {
#pragma unroll
            for (int v = 0; v < V; ++v) p.side_out[(size_t)b * p.side_bs + c * V + v] = xr[j][v];
          }
        }
      }
    }
    if (PRO == PRO_DATTN) {
      // "moshi_lm.rs", `attend` over the depformer's per-frame keys 0..n_keys-1.
      // Scores: `tp` threads per (head, key) pair, float4 loads issued together, so
      // the whole prologue costs two dependent round trips to L2.
      const int nk = p.n_keys, dh = p.dheads, hd = p.dhead_dim;
      const float* q = p.dq + (size_t)b * p.dq_bs;
      const float* dk = p.dk + (size_t)b * p.dkv_bs;
      const float* dv = p.dv + (size_t)b * p.dkv_bs;
      const float scale = 1.0f / sqrtf((float)hd);
      const int npairs = dh * nk;
      int tp = 32;
      while (tp > 1 && tp * npairs > kConsumers) tp >>= 1;
      if (tp > hd / 4) tp = hd / 4;
      const int pr = tid / tp, sub = tid % tp;
      float d = 0.f;
      if (pr < npairs) {
        const int h = pr / nk, jk = pr % nk;
        const float4* q4 = reinterpret_cast<const float4*>(q + h * hd);
        const float4* k4 = reinterpret_cast<const float4*>(dk + (size_t)jk * K + h * hd);
#pragma unroll 8
        for (int e = sub; e < hd / 4; e += tp) {
          const float4 a = q4[e], c4 = k4[e];
          d = fmaf(a.x, c4.x, d);
          d = fmaf(a.y, c4.y, d);
          d = fmaf(a.z, c4.z, d);
          d = fmaf(a.w, c4.w, d);
        }
      }
      for (int o = tp >> 1; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (pr < npairs && sub == 0) s_att[(pr / nk) * 8 + pr % nk] = d * scale;
      bar_sync(1, kConsumers);
      if (tid < dh) {
        float mx = -__int_as_float(0x7f800000);
        for (int jk = 0; jk < nk; ++jk) mx = fmaxf(mx, s_att[tid * 8 + jk]);
        float den = 0.f;
        for (int jk = 0; jk < nk; ++jk) {
          const float e = expf(s_att[tid * 8 + jk] - mx);
          s_att[tid * 8 + jk] = e;
          den += e;
        }
        for (int jk = 0; jk < nk; ++jk) s_att[tid * 8 + jk] = s_att[tid * 8 + jk] / den;
      }
      bar_sync(1, kConsumers);
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int c = tig + j * pl.tpr;
        if (c < CC) {
          const int h = (c * V) / hd;  // a chunk never straddles two heads
          float o[V];
#pragma unroll
          for (int v = 0; v < V; ++v) o[v] = 0.f;
#pragma unroll
          for (int jk = 0; jk < 8; ++jk) {
            if (jk < nk) {
              const float pw = s_att[h * 8 + jk];
#pragma unroll
              for (int v = 0; v < V; v += 4) {
                const float4 f = *reinterpret_cast<const float4*>(dv + (size_t)jk * K + c * V + v);
                o[v] += pw * f.x;
                o[v + 1] += pw * f.y;
                o[v + 2] += pw * f.z;
                o[v + 3] += pw * f.w;
              }
            }
          }
#pragma unroll
          for (int v = 0; v < V; ++v) xr[j][v] = o[v];
        }
      }
    }

    // a tile is `rounds` rounds of the row groups (one round for bf16 / f32; band tiles
    // take several so that each bulk copy stays large)
    const int rstride = (kConsumers / pl.tpr) * RG;  // rows of one round
    const int rounds = Chunk<WT>::kBand ? pl.tile_rows / rstride : 1;
    for (int i = 0; i < nt; ++i) {
      if (s_abort) break;
      const int s = i % NS;
      if (!mbar_wait(&full[s], (uint32_t)((i / NS) & 1))) {
        atomicOr(p.status, kDevTimeout);
        s_abort = 1;
        break;
      }
      for (int rd = 0; rd < rounds; ++rd) {
        const int lr0 = rd * rstride + g * RG;  // this group's first row in the tile
        const uint8_t* row0 = stages + (size_t)s * tile_bytes + (size_t)lr0 * row_bytes;
        // two accumulators per row (even / odd elements) halve the FMA dependency chain
        float acc[RG][2];
#pragma unroll
        for (int r = 0; r < RG; ++r) acc[r][0] = acc[r][1] = 0.f;
        uint4 w[NCH][RG];
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int c = tig + j * pl.tpr;
#pragma unroll
          for (int r = 0; r < RG; ++r)
            w[j][r] = (c < CC) ? *reinterpret_cast<const uint4*>(row0 + (size_t)r * row_bytes +
                                                                 (size_t)c * 16)
                               : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int j = 0; j < NCH; ++j)
#pragma unroll
          for (int r = 0; r < RG; ++r) {
            if constexpr (Chunk<WT>::kBand) {
              const int c = tig + j * pl.tpr;
              const float d =
                  (c < CC) ? *reinterpret_cast<const float*>(row0 + (size_t)r * row_bytes +
                                                             Chunk<WT>::scale_off(K, c))
                           : 0.f;
              Chunk<WT>::dot2s(w[j][r], d, xr[j], acc[r][0], acc[r][1]);
            } else {
              Chunk<WT>::dot2(w[j][r], xr[j], acc[r][0], acc[r][1]);
            }
          }
        if (rd == rounds - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
        }
        float* pp = part + (size_t)(i * pl.tile_rows + lr0) * wpg + (warp % wpg);
        if (RG == 2) {
          // reduce two rows with five shuffles: lanes 0-15 end with row 0, 16-31 row 1
          const bool up = (lane & 16) != 0;
          const float r0 = acc[0][0] + acc[0][1];
          const float r1 = acc[RG - 1][0] + acc[RG - 1][1];
          float keep = up ? r1 : r0;
          const float send = up ? r0 : r1;
          keep += __shfl_xor_sync(0xffffffffu, send, 16);
          keep += __shfl_xor_sync(0xffffffffu, keep, 8);
          keep += __shfl_xor_sync(0xffffffffu, keep, 4);
          keep += __shfl_xor_sync(0xffffffffu, keep, 2);
          keep += __shfl_xor_sync(0xffffffffu, keep, 1);
          if (lane == 0) pp[0] = keep;
          if (lane == 16) pp[wpg] = keep;
        } else {
          const float r0 = warp_sum(acc[0][0] + acc[0][1]);
          if (lane == 0) pp[0] = r0;
        }
      }
    }
  }
  __syncthreads();

  if (s_abort) {
    // wind down: wait (bounded) for the copies still in flight into this CTA's stages
    if (tid == 0) {
      const int issued = s_issued;
      for (int i = max(0, issued - NS); i < issued; ++i)
        (void)mbar_wait(&full[i % NS], (uint32_t)((i / NS) & 1));
    }
    __syncthreads();
    return;
  }

  // ------------------------------------------------------------ epilogue
  const int tr = pl.tile_rows;
  const int nrows = nt * tr;
  auto yrow = [&](int lr) {
    float y = 0.f;
    for (int w = 0; w < wpg; ++w) y += part[(size_t)lr * wpg + w];
    return y;
  };
  auto grow = [&](int lr) { return (t0 + lr / tr) * tr + lr % tr; };

  if (EPI == EPI_STORE || EPI == EPI_RESID || EPI == EPI_DEPIN) {
    float* out = p.out + (size_t)b * p.out_bs;
    int prev = -1;
    if (EPI == EPI_DEPIN) {
      const IoLayout io{p.batch};
      const int forcing = p.d_in[io.flag_off() + b];
      prev = forcing ? p.d_in[io.forced_off() + (size_t)b * 9 + p.key_index]
                     : argmax_key_index(p.keys[(size_t)b * 9 + p.key_index]);
    }
    for (int lr = tid; lr < nrows; lr += kThreads) {
      const int row = grow(lr);
      if (row >= pl.n_out) continue;
      const float y = yrow(lr);
      if (EPI == EPI_STORE) out[row] = y;
      if (EPI == EPI_RESID) out[row] += y;
      if (EPI == EPI_DEPIN) {
        // "moshi_lm.rs", `embed`: -1 adds nothing, else row max(tok, 0)
        if (prev != -1)
          out[row] = y + Chunk<typename Chunk<WT>::Table>::elem(
                             p.emb, (size_t)max(prev, 0) * pl.n_out + row);
        else
          out[row] = y;
      }
    }
  } else if (EPI == EPI_SWIGLU) {
    // "moshi_lm.rs", `temporal_step`: silu(gate_j) * mult_j
    float* out = p.out + (size_t)b * p.out_bs;
    const int half = tr >> 1;
    for (int lr = tid; lr < nrows; lr += kThreads) {
      const int r = lr % tr;
      if (r >= half) continue;
      const int j = (t0 + lr / tr) * half + r;
      if (j >= pl.n_out) continue;
      const float gt = yrow(lr), mu = yrow(lr + half);
      out[j] = gt / (1.0f + expf(-gt)) * mu;
    }
  } else if (EPI == EPI_QKV) {
    // "moshi_lm.rs", `rope_row` on q and k at pos, then the K/V push at slot pos % C
    const int D = pl.n_out / 3;
    const int pos = p.offsets[b];
    const int slot = pos % p.context;
    const int hd = p.head_dim;
    for (int lr = 2 * tid; lr < nrows; lr += 2 * kThreads) {
      const int row = grow(lr);
      if (row >= pl.n_out) continue;
      float a = yrow(lr), c = yrow(lr + 1);
      const int region = row / D, col = row % D;
      if (region < 2) {
        const int ip = (col % hd) >> 1;
        const float freq = expf(-logf(p.rope_theta) * 2.0f * (float)ip / (float)hd);
        const float ang = freq * (float)pos;
        const float sn = sinf(ang), cs = cosf(ang);
        const float ra = a * cs - c * sn;
        const float rc = a * sn + c * cs;
        a = ra;
        c = rc;
      }
      if (region == 0) {
        p.out[(size_t)b * p.out_bs + col] = a;
        p.out[(size_t)b * p.out_bs + col + 1] = c;
      } else {
        void* cache = region == 1 ? p.kcache : p.vcache;
        const size_t base = (size_t)b * p.kv_bs + (size_t)slot * D + col;
        store_kv(cache, base, a, p.kv_bf16);
        store_kv(cache, base + 1, c, p.kv_bf16);
      }
    }
  } else if (EPI == EPI_DQKV) {
    const int DD = pl.n_out / 3;
    for (int lr = tid; lr < nrows; lr += kThreads) {
      const int row = grow(lr);
      if (row >= pl.n_out) continue;
      const float y = yrow(lr);
      if (row < DD)
        p.out[(size_t)b * p.out_bs + row] = y;
      else if (row < 2 * DD)
        p.dk_out[(size_t)b * p.dkv_bs + row - DD] = y;
      else
        p.dv_out[(size_t)b * p.dkv_bs + row - 2 * DD] = y;
    }
  } else if (EPI == EPI_ARGMAX) {
    float* out = p.out + (size_t)b * p.out_bs;
    unsigned long long best = 0ull;
    for (int lr = tid; lr < nrows; lr += kThreads) {
      const int row = grow(lr);
      if (row >= pl.n_out) continue;
      const float y = yrow(lr);
      out[row] = y;
      const unsigned long long k = pick_key(p.samp, b, p.key_index, y, (uint32_t)row);
      best = k > best ? k : best;
    }
    best = warp_max_u64(best);
    if (lane == 0) s_key[warp] = best;
    __syncthreads();
    if (tid == 0 && nt > 0) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kThreads / 32; ++w) m = s_key[w] > m ? s_key[w] : m;
      atomicMax(p.keys + (size_t)b * 9 + p.key_index, m);
    }
  }
}


}  // namespace rqk
