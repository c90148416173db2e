// frame_persistent.cuh -- the whole frame's linears and attentions in one cooperative
// launch (batch 1).  Instantiated by frame_persistent.cu (with token picks) and
// frame_persistent_greedy.cu (greedy frames).
//
// Every CTA walks the same op table (temporal layers, text head, the 8 depformer
// steps).  Between dependent ops the CTAs of the two-CTAs-per-SM launch meet at a grid
// barrier (one atomic counter, bounded spin); the one-CTA-per-SM launch (the depformer)
// instead polls tagged words, each value carrying the op that wrote it.  The weights of every op are known before the frame starts, so each
// CTA's producer warp streams the weight tiles it owns for ALL ops, in order, into one
// shared-memory ring with cp.async.bulk, running ahead of the consumers across op
// boundaries: HBM keeps streaming the next ops' weights while the consumers wait on a
// barrier, which removes the per-kernel drain and fill of a launch-per-op schedule.
// Consumers run the prologues / epilogues of the streaming GEMV (gemv_kernel.cuh)
// selected per op at run time, and the split-K decode attention as work items.
// Activations written by other CTAs are read with L2-only loads (ld.global.cg), or as
// tagged words with relaxed gpu-scope loads.
#pragma once
#include <cuda_bf16.h>

#include "gemv_kernel.cuh"

namespace rqk {
namespace pers {

constexpr int kCons = 256;    // consumer threads
constexpr int kThr = 288;     // + 1 producer warp
constexpr int kMaxNch = 2;  // long reductions are split into parts (GemvPlan::kparts)
// chunks of x a consumer thread holds: two for f32 / bf16 rows (4 or 8 values each), one
// for weight bands (16 q8 or 32 q4 values)
template <typename WT>
struct Nx {
  static constexpr int N = Chunk<WT>::kBand ? 1 : kMaxNch;
};
constexpr int kMaxStage = 1024;  // depformer attention output staged in shared memory (DD <= 1024)
#ifndef RQ_PERS_BURST_T
#define RQ_PERS_BURST_T 4
#endif
#ifndef RQ_PERS_STREAM_T
#define RQ_PERS_STREAM_T 4
#endif
#ifndef RQ_PERS_STREAM_BURST
#define RQ_PERS_STREAM_BURST 0
#endif
#ifndef RQ_PERS_STREAM_MIN
#define RQ_PERS_STREAM_MIN 4
#endif
// tile groups: resident tiles (ops of a few tiles per CTA) in bursts of kBurstT; the
// weight stream of long ops (more than kStreamMinTiles tiles per CTA) kStreamT at a time
// (4: once the two-CTA kernel ran without spills, groups of 4 measured 17 us per frame
// faster than 2)
constexpr int kBurstT = RQ_PERS_BURST_T;
#ifndef RQ_PERS_BURST_T_WIDE
#define RQ_PERS_BURST_T_WIDE 8
#endif
// the one-CTA-per-SM launch (the depformer) has the registers for bigger groups
constexpr int kBurstTWide = RQ_PERS_BURST_T_WIDE;
constexpr int kStreamT = RQ_PERS_STREAM_T;
constexpr bool kStreamBurst = RQ_PERS_STREAM_BURST != 0;
constexpr int kStreamMinTiles = RQ_PERS_STREAM_MIN;


// ---------------------------------------------------------------- grid barrier
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// one arrival of this CTA, after a CTA barrier: the release orders every thread's writes
// (made visible to it by that barrier) before the count.  A returning atom.add: on GB300
// (2 CTAs per SM, 304 CTAs) a grid barrier takes 1.23 us with it against 1.39 us with the
// reduction form red.add, which the memory system completes later.
__device__ __forceinline__ void grid_arrive(unsigned* bar) {
  [[maybe_unused]] unsigned old;
  asm volatile("atom.add.release.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(bar) : "memory");
}

// thread 0 of the consumers: wait until `target` CTAs have arrived (bounded by limit_ns)
__device__ __forceinline__ bool grid_wait(const unsigned* bar, unsigned target,
                                          uint64_t limit_ns) {
  if (ld_acquire(bar) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ld_acquire(bar) >= target) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ float ldcg(const float* p) { return __ldcg(p); }

// ---------------------------------------------------------------- tagged words
// The depformer launch (one CTA per SM) runs without grid barriers.  Every value that one
// CTA writes and another reads is one 64-bit word, (tag << 32) | f32 bits, stored by a
// single relaxed store; a reader polls the word until it carries the tag of the op that
// produces it.  An aligned 64-bit access is single-copy atomic, so a word is seen either
// old or new, never half of each, and a value needs no ordering against any other: the
// wait for the producer and the load of its output are one round trip instead of a
// barrier's arrival, its polling and then the load.  Tags are (frame epoch << 10) | the
// frame index of the producing op: words of earlier frames, and of earlier ops writing
// the same buffer, never match.  Buffers are reused safely because every op waits for
// the whole output of the op before it, so no CTA can be more than one op ahead of any
// CTA that still has to read what it would overwrite.
__device__ __forceinline__ void ll_st(float* base, size_t i, uint32_t tag, float v) {
  const unsigned long long w = ((unsigned long long)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(
                   reinterpret_cast<unsigned long long*>(base) + i),
               "l"(w)
               : "memory");
}
// two consecutive words (16-byte aligned)
__device__ __forceinline__ void ll_ld2(const float* base, size_t i, unsigned long long& a,
                                       unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];"
               : "=l"(a), "=l"(b)
               : "l"(reinterpret_cast<const unsigned long long*>(base) + i)
               : "memory");
}
__device__ __forceinline__ unsigned long long ll_ld1(const float* base, size_t i) {
  unsigned long long a;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];"
               : "=l"(a)
               : "l"(reinterpret_cast<const unsigned long long*>(base) + i)
               : "memory");
  return a;
}
__device__ __forceinline__ float ll_val(unsigned long long w) {
  return __uint_as_float((uint32_t)w);
}
__device__ __forceinline__ bool ll_is(unsigned long long w, uint32_t tag) {
  return (uint32_t)(w >> 32) == tag;
}

// the CTA's abort flag: raised by a wait that ran out (or by the producer), it ends every
// other wait of the CTA and, read at a CTA barrier, the op loop
__shared__ volatile int s_abort;
// the launch's wait limit (ns), set once by thread 0
__shared__ unsigned long long s_wait_lim;

// The launch's view of the tags: the epoch base and `flip` (all ones for the op a test
// stalls: it turns every tag that op waits for into one that nothing writes).
struct LLCtx {
  uint32_t ebase, flip;
  const PersParams& P;
  __device__ __forceinline__ uint32_t want(int op_index) const {
    return (ebase | (uint32_t)op_index) ^ flip;
  }
  // After an attempt that found a word without its tag: whether to try again.  The first
  // miss starts the clock (t0); on the wait limit it records a timeout and raises the
  // CTA's abort flag (the op's results are then garbage and the launch winds down).
  // Written as a loop in the caller, not a callback, so that the words polled stay in
  // registers.
  __device__ __forceinline__ bool again(uint64_t& t0) const {
    if (t0 == 0ull) {
      t0 = global_timer_ns();
      return true;
    }
    if (s_abort) return false;
    if (global_timer_ns() - t0 > s_wait_lim) {
      atomicOr(P.status, kDevTimeout);
      s_abort = 1;
      return false;
    }
    return true;
  }
  __device__ __forceinline__ float wait1(const float* base, size_t i, uint32_t tag) const {
    unsigned long long w;
    uint64_t t0 = 0ull;
    do {
      w = ll_ld1(base, i);
    } while (!ll_is(w, tag) && again(t0));
    return ll_val(w);
  }
};

// ---------------------------------------------------------------- tile consumer
// Sum each of R row values over the warp's 32 lanes with a transposing butterfly: at
// every halving step a lane keeps half of its values and adds its partner's copy of
// them, so R rows take R - 1 + (5 - log2 R) shuffles instead of 5 R.  Afterwards lanes
// [q * 32/R, (q + 1) * 32/R) all hold the full sum of row q (returned).
template <int R>
__device__ __forceinline__ float warp_sum_rows(float (&v)[R], int lane) {
#pragma unroll
  for (int n = R, o = 16; n > 1; n >>= 1, o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int m = 0; m < n / 2; ++m) {
      const float keep = up ? v[m + n / 2] : v[m];
      const float send = up ? v[m] : v[m + n / 2];
      v[m] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
#pragma unroll
  for (int o = 16 / R; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
  return v[0];
}

// one 16-byte chunk of a staged weight row times the thread's chunk of x: f32 / bf16
// values, or a weight band's codes times the scale of their group (read from the row)
template <typename WT>
__device__ __forceinline__ void tile_dot(const uint8_t* row, int Kw, int c, const uint4 w,
                                         const float (&x)[Chunk<WT>::V], float& a, float& b) {
  if constexpr (Chunk<WT>::kBand) {
    const float d = *reinterpret_cast<const float*>(row + Chunk<WT>::scale_off(Kw, c));
    Chunk<WT>::dot2s(w, d, x, a, b);
  } else {
    (void)row;
    (void)Kw;
    (void)c;
    Chunk<WT>::dot2(w, x, a, b);
  }
}

// Consume `nt` tiles of one GEMV op from the ring (slot `slot`, phase `ph` advance tile by
// tile), the CTA's tiles tb.. of the op, leaving one partial per (row, warp) in `part`.  Tiles go in
// groups of T with one butterfly over the group's 2T rows.  BURST (tiles already
// resident, the latency-bound depformer ops): every wait of a group, then every
// shared-memory load, the FMAs and the slots' release, so the chain of dependent
// latencies is paid once per group.  Otherwise (the weight stream): each tile is loaded
// and multiplied as soon as it lands and its slot goes back to the producer at once.
template <typename WT, int NCH, int T, bool BURST>
__device__ __forceinline__ bool consume_tiles(const GemvPlan& pl, int Kw, bool accumulate,
                                              int nt, int tb, int& slot, uint32_t& ph,
                                              uint8_t* ring, int slot_bytes, int NS,
                                              uint64_t* full, uint64_t* empty, float* part,
                                              const float (&xr)[Nx<WT>::N][Chunk<WT>::V],
                                              int g, int tig, int warp, int lane,
                                              uint64_t lim) {
  constexpr int RG = 2;  // rows per thread group and tile (every persistent plan)
  constexpr int R = T * RG;
  static_assert(NCH <= Nx<WT>::N, "x chunks held per thread");
  const uint32_t row_bytes = (uint32_t)Chunk<WT>::row_bytes(Kw);
  const int CC = Kw / Chunk<WT>::V;
  const int wpg = pl.tpr >> 5;
  for (int i0 = 0; i0 < nt; i0 += T) {
    float acc[R][2];
#pragma unroll
    for (int q = 0; q < R; ++q) acc[q][0] = acc[q][1] = 0.f;
    if (BURST) {
      int sl[T];
      const uint8_t* row0[T];
#pragma unroll
      for (int t = 0; t < T; ++t) {
        sl[t] = slot;
        row0[t] = ring + (size_t)slot * slot_bytes + (size_t)(g * RG) * row_bytes;
        if (i0 + t < nt) {
          if (!mbar_wait_for(&full[slot], ph, lim)) return false;
          if (++slot == NS) {
            slot = 0;
            ph ^= 1u;
          }
        }
      }
      uint4 w[T][NCH][RG];
#pragma unroll
      for (int t = 0; t < T; ++t)
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int c = tig + j * pl.tpr;
#pragma unroll
          for (int r = 0; r < RG; ++r)
            w[t][j][r] = (i0 + t < nt && c < CC)
                             ? *reinterpret_cast<const uint4*>(row0[t] + (size_t)r * row_bytes +
                                                               (size_t)c * 16)
                             : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
      for (int t = 0; t < T; ++t) {
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          const int c = tig + j * pl.tpr;
          // past the row: zero weights for f32 / bf16; a band code 0 stands for -8, skip
          if (Chunk<WT>::kBand && c >= CC) continue;
#pragma unroll
          for (int r = 0; r < RG; ++r)
            tile_dot<WT>(row0[t] + (size_t)r * row_bytes, Kw, c, w[t][j][r], xr[j],
                         acc[t * RG + r][0], acc[t * RG + r][1]);
        }
      }
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < T; ++t)
          if (i0 + t < nt) mbar_arrive(&empty[sl[t]]);
      }
    } else {
#pragma unroll
      for (int t = 0; t < T; ++t) {
        if (i0 + t < nt) {
          if (!mbar_wait_for(&full[slot], ph, lim)) return false;
          const uint8_t* row0 = ring + (size_t)slot * slot_bytes + (size_t)(g * RG) * row_bytes;
          uint4 w[NCH][RG];
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            const int c = tig + j * pl.tpr;
#pragma unroll
            for (int r = 0; r < RG; ++r)
              w[j][r] = c < CC ? *reinterpret_cast<const uint4*>(row0 + (size_t)r * row_bytes +
                                                                 (size_t)c * 16)
                               : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            const int c = tig + j * pl.tpr;
            if (Chunk<WT>::kBand && c >= CC) continue;  // see the burst path
#pragma unroll
            for (int r = 0; r < RG; ++r)
              tile_dot<WT>(row0 + (size_t)r * row_bytes, Kw, c, w[j][r], xr[j],
                           acc[t * RG + r][0], acc[t * RG + r][1]);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[slot]);
          if (++slot == NS) {
            slot = 0;
            ph ^= 1u;
          }
        }
      }
    }
    float v[R];
#pragma unroll
    for (int q = 0; q < R; ++q) v[q] = acc[q][0] + acc[q][1];
    const float sum = warp_sum_rows<R>(v, lane);
    // row q = t * RG + r of the group: tile i0 + t, row g * RG + r of that tile
    const int q = lane / (32 / R);
    const int t = q / RG, r = q % RG;
    if (lane % (32 / R) == 0 && i0 + t < nt) {
      float* pp = part + (size_t)((tb + i0 + t) * pl.tile_rows + g * RG + r) * wpg + (warp % wpg);
      *pp = accumulate ? *pp + sum : sum;
    }
  }
  return true;
}

// Tiles [ceil(T*c/G), ceil(T*(c+1)/G)) for CTA c: contiguous, balanced, and CTA 0
// always owns tile 0 (it writes the op's side output) even when T < G.
__device__ __forceinline__ void tile_range(const GemvPlan& pl, int& t0, int& t1) {
  const long long T = pl.tiles, G = gridDim.x;
  t0 = (int)((T * blockIdx.x + G - 1) / G);
  t1 = (int)((T * (blockIdx.x + 1) + G - 1) / G);
}

// ---------------------------------------------------------------- weight tile sequence
// One position in this CTA's sequence of weight tiles: every GEMV op's tile range, every
// reduction part of it, in op order -- the order the producer fills the ring in.
struct TileCur {
  int k, kp, t, t0, t1;
};

// from op c.k on, the first GEMV op with a tile for this CTA
template <typename WT>
__device__ __forceinline__ bool cur_seek(const PersParams& P, TileCur& c) {
  for (; c.k < P.n_ops; ++c.k) {
    const PersOp& op = P.ops[c.k];
    if (op.type != OPT_GEMV) continue;
    tile_range(P.plans[op.plan], c.t0, c.t1);
    if (c.t0 < c.t1) {
      c.kp = 0;
      c.t = c.t0;
      return true;
    }
  }
  return false;
}

template <typename WT>
__device__ __forceinline__ bool cur_next(const PersParams& P, TileCur& c) {
  if (++c.t < c.t1) return true;
  if (++c.kp < P.plans[P.ops[c.k].plan].kparts) {
    c.t = c.t0;
    return true;
  }
  ++c.k;
  return cur_seek<WT>(P, c);
}

// the source byte ranges of the tile at c, each with its offset in the ring slot:
// f(src, bytes, slot_offset); all 16-byte aligned, sizes multiples of 16
template <typename WT, typename F>
__device__ __forceinline__ void cur_ranges(const PersParams& P, const TileCur& c, F&& f) {
  const PersOp& op = P.ops[c.k];
  const GemvPlan& pl = P.plans[op.plan];
  const uint32_t row_bytes = (uint32_t)Chunk<WT>::row_bytes(pl.K);
  const bool paired = op.epi == EPI_SWIGLU;
  const int opt = paired ? pl.tile_rows / 2 : pl.tile_rows;
  const uint8_t* W = static_cast<const uint8_t*>(op.W);
  const int r0 = c.t * opt;
  const int nv = min(opt, pl.n_out - r0);
  if (pl.kparts > 1) {
    // per row, the part's columns are a strided window of W; a weight band's row part is
    // its codes, then its groups' scales (the layout of a Kw-column band row)
    const int k0 = c.kp * pl.kp_width;
    const int Kw = c.kp == pl.kparts - 1 ? pl.K - k0 : pl.kp_width;
    const uint32_t seg = (uint32_t)Chunk<WT>::row_bytes(Kw);
    for (int r = 0; r < nv; ++r) {
      const uint8_t* row = W + (size_t)(r0 + r) * row_bytes;
      if constexpr (Chunk<WT>::kBand) {
        const uint32_t sc = (uint32_t)Kw / 8u;          // f32 scale per 32 values
        const uint32_t cd = seg - sc;                   // code bytes of the part
        const uint32_t cd0 = (uint32_t)Chunk<WT>::row_bytes(k0) - (uint32_t)k0 / 8u;
        const uint32_t codes_row = row_bytes - (uint32_t)pl.K / 8u;
        f(row + cd0, cd, (uint32_t)r * seg);
        f(row + codes_row + (uint32_t)k0 / 8u, sc, (uint32_t)r * seg + cd);
      } else {
        f(row + (size_t)k0 * sizeof(WT), seg, (uint32_t)r * seg);
      }
    }
  } else if (paired) {
    const uint32_t bytes = (uint32_t)nv * row_bytes;
    f(W + (size_t)r0 * row_bytes, bytes, 0u);
    f(W + (size_t)op.w_half + (size_t)r0 * row_bytes, bytes, (uint32_t)opt * row_bytes);
  } else {
    f(W + (size_t)r0 * row_bytes, (uint32_t)nv * row_bytes, 0u);
  }
}

template <typename WT>
__device__ __forceinline__ uint32_t cur_bytes(const PersParams& P, const TileCur& c) {
  uint32_t n = 0;
  cur_ranges<WT>(P, c, [&](const uint8_t*, uint32_t bytes, uint32_t) { n += bytes; });
  return n;
}

// ---------------------------------------------------------------- prologue
// x for this op into registers: chunk j of thread (g, tig) covers columns
// [(tig + j*tpr)*V, +V).  Returns nothing; uses consumer barrier 1.  LL: the launch
// exchanges tagged words (wtag: this op's tag; lc: the tags it waits for).
template <typename WT, bool LL, bool PICKS>
__device__ __forceinline__ void form_x(const PersParams& P, const PersOp& op,
                                       const GemvPlan& pl, int nch, int k0, int Kw,
                                       float (&xr)[Nx<WT>::N][Chunk<WT>::V],
                                       const float (&ar)[Nx<WT>::N][Chunk<WT>::V], int g,
                                       int tig, int tid, int warp, int lane, float* s_red,
                                       int red_half, float* s_att, int forcing,
                                       const LLCtx& lc, uint32_t wtag,
                                       unsigned long long* s_key) {
  constexpr int V = Chunk<WT>::V;
  constexpr int NX = Nx<WT>::N;
  using TT = typename Chunk<WT>::Table;  // embedding tables: bf16 for weight bands
  const int K = pl.K, CC = Kw / V;
  const float* in = op.in + k0;  // this part's columns [k0, k0 + Kw)
  (void)tid;
  (void)wtag;
  (void)s_key;
  // tagged input: every chunk polled until all its words carry the producer's tag
  const bool tagged = LL && (op.pro == PRO_PLAIN || op.pro == PRO_RMS);
#pragma unroll
  for (int j = 0; j < NX; ++j) {
    const int c = tig + j * pl.tpr;
    if (op.pro != PRO_DATTN) {  // (the attention sets x at its end: fewer live registers)
#pragma unroll
      for (int v = 0; v < V; ++v) xr[j][v] = 0.f;
    }
    if (!tagged && op.pro != PRO_DATTN && j < nch && c < CC) {
#pragma unroll
      for (int v = 0; v < V; v += 4) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(in + (size_t)c * V + v));
        xr[j][v] = f.x;
        xr[j][v + 1] = f.y;
        xr[j][v + 2] = f.z;
        xr[j][v + 3] = f.w;
      }
    }
  }
  // the tagged launch loads an RMSNorm's alpha here, in flight with the poll of x (the
  // other launches load it before their grid barrier)
  float al[NX][V];
  if constexpr (LL && !Chunk<WT>::kBand) {
    if (op.pro == PRO_RMS || op.pro == PRO_RMS_EMB) {
#pragma unroll
      for (int j = 0; j < NX; ++j) {
        const int c = tig + j * pl.tpr;
#pragma unroll
        for (int v = 0; v < V; v += 4) {
          const float4 a = (j < nch && c < CC)
                               ? __ldg(reinterpret_cast<const float4*>(op.alpha + (size_t)c * V + v))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
          al[j][v] = a.x;
          al[j][v + 1] = a.y;
          al[j][v + 2] = a.z;
          al[j][v + 3] = a.w;
        }
      }
    }
  } else {
    (void)al;
  }
  if constexpr (LL) {
    if (tagged) {
      const uint32_t t = lc.want(op.tag_in);
      uint64_t t0 = 0ull;
      bool ok;
      do {
        ok = true;
#pragma unroll
        for (int j = 0; j < NX; ++j) {
          const int c = tig + j * pl.tpr;
          if (j < nch && c < CC) {
#pragma unroll
            for (int v = 0; v < V; v += 2) {
              unsigned long long a, b;
              ll_ld2(op.in, (size_t)k0 + (size_t)c * V + v, a, b);
              xr[j][v] = ll_val(a);
              xr[j][v + 1] = ll_val(b);
              ok &= ll_is(a, t) & ll_is(b, t);
            }
          }
        }
      } while (!ok && lc.again(t0));
    }
  }
  // (the depformer's prologues and its qkv epilogue exist only in the tagged, one-CTA-per-SM
  // instantiation: the two-CTA launch runs no depformer op, and without them it fits its
  // 96 registers with no spills -- measured 38 us per frame faster)
  if (LL && op.pro == PRO_RMS_EMB) {
    // a depformer step's input: dep_in[cb] . t (computed beside the text head) plus
    // "moshi_lm.rs", `embed` of the step's conditioning token (-1 adds nothing, else row
    // max(tok, 0)); CTA 0 keeps this x for the residuals
    const IoLayout io{1};
    int prev;
    if (LL && op.tag_key >= 0) {
      // the pick's key: the largest of the CTAs' tagged best keys (or the one slot a top-k
      // pick wrote).  Polled even when the token is forced: this op must not start before
      // every CTA is done with the op before it (the chain that keeps buffers safe).
      unsigned long long best = 0ull;
      if (tid < op.key_slots) {
        const float* sp = reinterpret_cast<const float*>(P.key_ll) +
                          ((size_t)op.key_index * gridDim.x + tid) * 4;
        const uint32_t t = lc.want(op.tag_key);
        unsigned long long a, b;
        uint64_t t0 = 0ull;
        do {
          ll_ld2(sp, 0, a, b);
        } while (!(ll_is(a, t) & ll_is(b, t)) && lc.again(t0));
        best = ((unsigned long long)(uint32_t)b << 32) | (uint32_t)a;
      }
      best = warp_max_u64(best);
      if (lane == 0) s_key[warp] = best;
      bar_sync(1, kCons);
      unsigned long long m = 0ull;
#pragma unroll
      for (int w = 0; w < kCons / 32; ++w) m = s_key[w] > m ? s_key[w] : m;
      prev = forcing ? P.d_in[io.forced_off() + op.key_index] : argmax_key_index(m);
    } else {
      prev = forcing ? P.d_in[io.forced_off() + op.key_index]
                     : argmax_key_index(__ldcg(P.keys + op.key_index));
    }
    const bool keep = op.side_out != nullptr && blockIdx.x == 0 && g == 0;
#pragma unroll
    for (int j = 0; j < NX; ++j) {
      const int c = tig + j * pl.tpr;
      if (j < nch && c < CC) {
        if (prev != -1) {
#pragma unroll
          for (int v = 0; v < V; ++v)
            xr[j][v] += Chunk<TT>::elem(op.emb, (size_t)max(prev, 0) * K + c * V + v);
        }
        if (keep) {
#pragma unroll
          for (int v = 0; v < V; ++v) {
            if constexpr (LL)
              ll_st(op.side_out, (size_t)c * V + v, wtag, xr[j][v]);
            else
              op.side_out[c * V + v] = xr[j][v];
          }
        }
      }
    }
  }
  if (op.pro == PRO_RMS || op.pro == PRO_RMS_EMB) {
    // "moshi_lm.rs", `rms_norm`: x * alpha * (1 / sqrt(eps + sum(x^2) / n)).  The factor
    // 1 / sqrt(...) is one scalar for the whole vector, so W (x * alpha * r) = r W (x *
    // alpha): the tiles run on x * alpha and the epilogue multiplies by r (rms_scale),
    // after the CTA barrier that follows the tiles -- the reduction is off the path from
    // x to the first tile.  Here each warp leaves its partial sum of squares in s_red:
    // every row group holds the whole vector, group 0's warps' partials cover it once.
    // s_red alternates between two halves op by op (the next op writes the other half).
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NX; ++j)
#pragma unroll
      for (int v = 0; v < V; ++v) ss = fmaf(xr[j][v], xr[j][v], ss);
    ss = warp_sum(ss);
    if (lane == 0) s_red[red_half * (kCons / 32) + warp] = ss;
#pragma unroll
    for (int j = 0; j < NX; ++j) {
      const int c = tig + j * pl.tpr;
      if (j < nch && c < CC) {
        if constexpr (Chunk<WT>::kBand) {
          // weight bands: x is one chunk of 16 / 32 values, too many registers to keep
          // alpha from before the grid barrier; it loads here (16-byte aligned rows)
#pragma unroll
          for (int v = 0; v < V; v += 4) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(op.alpha + c * V + v));
            xr[j][v] *= a.x;
            xr[j][v + 1] *= a.y;
            xr[j][v + 2] *= a.z;
            xr[j][v + 3] *= a.w;
          }
        } else if constexpr (LL) {
#pragma unroll
          for (int v = 0; v < V; ++v) xr[j][v] *= al[j][v];
        } else {
#pragma unroll
          for (int v = 0; v < V; ++v) xr[j][v] *= ar[j][v];  // loaded before the barrier
        }
      }
    }
  } else if (LL && op.pro == PRO_DATTN) {
    // "moshi_lm.rs", `attend` over the depformer's per-frame keys 0..n_keys-1.
    // hd/4 threads per head, one float4 of dimensions each: q and every key in one
    // round trip, scores reduced with shuffles, the softmax in registers, then the values
    // in one more round trip (loading them with the keys measured 10 us per frame slower
    // in the one-CTA-per-SM launch); the output is staged in shared memory and read back
    // in the chunk layout of x.
    const int nk = op.n_keys, dh = P.dheads, hd = P.dhead_dim;
    const float scale = 1.0f / sqrtf((float)hd);
    const int tph = hd / 4;
    const int hpp = kCons / tph;
    // a float4 of tagged words at element i of base, ok &= all four carry tag t
    auto ld4 = [&](const float* base, size_t i, uint32_t t, float4& f, bool& ok) {
      unsigned long long a, b, c, d;
      ll_ld2(base, i, a, b);
      ll_ld2(base, i + 2, c, d);
      f = make_float4(ll_val(a), ll_val(b), ll_val(c), ll_val(d));
      ok &= ll_is(a, t) & ll_is(b, t) & ll_is(c, t) & ll_is(d, t);
    };
    (void)ld4;
    for (int h0 = 0; h0 < dh; h0 += hpp) {
      const int h = h0 + tid / tph, sub = tid % tph;
      const bool act = h < dh;
      const size_t col = (size_t)h * hd + 4 * sub;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (LL) {
        // tagged: keys and values in groups of four, each group one round trip (with q in
        // the first), folded in with the running-max softmax (windows of up to four keys:
        // one round trip; eight tagged keys and values in flight would take more
        // registers than the launch has)
        float m = -__int_as_float(0x7f800000), l = 0.f;
        float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
        const uint32_t tq = lc.want(op.tag_in);
#pragma unroll
        for (int j0 = 0; j0 < 8; j0 += 4) {
          if (j0 > 0 && j0 >= nk) break;
          float4 kk[4], vv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) kk[i] = vv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (act) {
            uint64_t t0 = 0ull;
            bool ok;
            do {
              ok = true;
              if (j0 == 0) ld4(op.in, col, tq, q4, ok);  // (k0 is 0: x is one part)
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int j = j0 + i;
                if (j < nk) {
                  const uint32_t tj = lc.want(op.tag_kv + j * op.tag_kv_step);
                  ld4(op.dk, (size_t)j * K + col, tj, kk[i], ok);
                  ld4(op.dv, (size_t)j * K + col, tj, vv[i], ok);
                }
              }
            } while (!ok && lc.again(t0));
          }
          float sc[4];
          float mn = m;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float d = q4.x * kk[i].x;
            d = fmaf(q4.y, kk[i].y, d);
            d = fmaf(q4.z, kk[i].z, d);
            d = fmaf(q4.w, kk[i].w, d);
            for (int w = tph >> 1; w > 0; w >>= 1) d += __shfl_xor_sync(0xffffffffu, d, w);
            sc[i] = d * scale;
            if (j0 + i < nk) mn = fmaxf(mn, sc[i]);
          }
          const float corr = expf(m - mn);  // 0 for the first group (m = -inf)
          l *= corr;
          o.x *= corr;
          o.y *= corr;
          o.z *= corr;
          o.w *= corr;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (j0 + i < nk) {
              const float e = expf(sc[i] - mn);
              l += e;
              o.x = fmaf(e, vv[i].x, o.x);
              o.y = fmaf(e, vv[i].y, o.y);
              o.z = fmaf(e, vv[i].z, o.z);
              o.w = fmaf(e, vv[i].w, o.w);
            }
          }
          m = mn;
        }
        const float inv = 1.0f / l;
        o.x *= inv;
        o.y *= inv;
        o.z *= inv;
        o.w *= inv;
      } else {
        float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 kk[8];
        if (act) q4 = __ldcg(reinterpret_cast<const float4*>(in + col));
#pragma unroll
        for (int j = 0; j < 8; ++j)
          kk[j] = (act && j < nk) ? __ldcg(reinterpret_cast<const float4*>(op.dk + (size_t)j * K + col))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        float sc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float d = q4.x * kk[j].x;
          d = fmaf(q4.y, kk[j].y, d);
          d = fmaf(q4.z, kk[j].z, d);
          d = fmaf(q4.w, kk[j].w, d);
          for (int w = tph >> 1; w > 0; w >>= 1) d += __shfl_xor_sync(0xffffffffu, d, w);
          sc[j] = d * scale;
        }
        float mx = -__int_as_float(0x7f800000);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < nk) mx = fmaxf(mx, sc[j]);
        float den = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          sc[j] = (j < nk) ? expf(sc[j] - mx) : 0.f;
          den += sc[j];
        }
        float4 vv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          vv[j] = (act && j < nk) ? __ldcg(reinterpret_cast<const float4*>(op.dv + (size_t)j * K + col))
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j < nk) {
            const float w = sc[j] / den;
            o.x += w * vv[j].x;
            o.y += w * vv[j].y;
            o.z += w * vv[j].z;
            o.w += w * vv[j].w;
          }
        }
      }
      if (act) *reinterpret_cast<float4*>(s_att + col) = o;
    }
    bar_sync(1, kCons);
#pragma unroll
    for (int j = 0; j < NX; ++j) {
      const int c = tig + j * pl.tpr;
#pragma unroll
      for (int v = 0; v < V; ++v) xr[j][v] = (j < nch && c < CC) ? s_att[c * V + v] : 0.f;
    }
    bar_sync(1, kCons);  // the staging buffer is reused by the next op
  }
}

// The RMSNorm factor 1 / sqrt(eps + sum(x^2) / K) of an RMS op, from the per-warp sums
// form_x left (call after a CTA barrier that follows form_x); every thread sums them in
// the same order, so every thread gets the same value.
__device__ __forceinline__ float rms_scale(const PersParams& P, const GemvPlan& pl,
                                           const float* s_red, int red_half) {
  float rv[kCons / 32];
#pragma unroll
  for (int w = 0; w < kCons / 32; ++w) rv[w] = s_red[red_half * (kCons / 32) + w];
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kCons / 32; ++w)
    if (w < pl.tpr / 32) tot += rv[w];
  return 1.0f / sqrtf(P.eps + tot / (float)pl.K);
}

// ---------------------------------------------------------------- epilogue
// slot `cta` of pick `pick`'s tagged key halves (the readers take the largest key)
__device__ __forceinline__ void put_key_slot(const PersParams& P, int pick, int cta,
                                             uint32_t tag, unsigned long long key) {
  float* sp = reinterpret_cast<float*>(P.key_ll) + ((size_t)pick * gridDim.x + cta) * 4;
  const unsigned long long lo = ((unsigned long long)tag << 32) | (uint32_t)key;
  const unsigned long long hi = ((unsigned long long)tag << 32) | (uint32_t)(key >> 32);
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(sp), "l"(lo), "l"(hi)
               : "memory");
}

// Finish rows [t0*tr, (t0+nt)*tr) of one GEMV op from the per-warp partials (batch 1).
// LL: outputs other CTAs read are tagged words (wtag), the residual's other rows are
// polled (lc).
template <typename WT, bool PICKS, bool LL>
__device__ __forceinline__ void epilogue(const PersParams& P, const PersOp& op,
                                         const GemvPlan& pl, int t0, int nt, const float* part,
                                         int tid, int warp, int lane,
                                         unsigned long long* s_key, const float2* s_rope,
                                         float resid_old, int pos, float scale,
                                         const LLCtx& lc, uint32_t wtag) {
  const int tr = pl.tile_rows, wpg = pl.tpr >> 5;
  const int nrows = nt * tr;
  (void)lc;
  (void)wtag;
  auto put = [&](float* base, size_t i, float v) {
    if constexpr (LL)
      ll_st(base, i, wtag, v);
    else
      base[i] = v;
  };
  // the row's value: the partials (wpg <= 8, loaded together, added in order), times the
  // RMSNorm factor of an RMS op (1 otherwise)
  auto yrow = [&](int lr) {
    float pv[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) pv[w] = w < wpg ? part[(size_t)lr * wpg + w] : 0.f;
    float y = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) y += pv[w];
    return y * scale;
  };
  auto grow = [&](int lr) { return (t0 + lr / tr) * tr + lr % tr; };
  const int epi = op.epi;
  // (the op table adds a depformer step's embedding row in the first qkv's prologue,
  // PRO_RMS_EMB, so this kernel has no EPI_DEPIN)
  if (epi == EPI_STORE || epi == EPI_RESID) {
    for (int lr = tid; lr < nrows; lr += kCons) {
      const int row = grow(lr);
      if (row >= pl.n_out) continue;
      const float y = yrow(lr);
      if (epi == EPI_STORE) put(op.out, row, y);
      if (epi == EPI_RESID) {
        float old = resid_old;
        if (lr != tid) old = LL ? lc.wait1(op.out, row, lc.want(op.tag_res)) : ldcg(op.out + row);
        put(op.out, row, old + y);
      }
    }
  } else if (epi == EPI_SWIGLU) {
    const int half = tr >> 1;
    for (int lr = tid; lr < nrows; lr += kCons) {
      const int r = lr % tr;
      if (r >= half) continue;
      const int j = (t0 + lr / tr) * half + r;
      if (j >= pl.n_out) continue;
      const float gt = yrow(lr), mu = yrow(lr + half);
      put(op.out, j, gt / (1.0f + expf(-gt)) * mu);
    }
  } else if (!LL && epi == EPI_QKV) {  // (the temporal stack's: not in the tagged kernel)
    const int D = pl.n_out / 3;
    const int slot = pos % P.context;
    const int hd = P.head_dim;
    for (int lr = 2 * tid; lr < nrows; lr += 2 * kCons) {
      const int row = grow(lr);
      if (row >= pl.n_out) continue;
      float a = yrow(lr), c = yrow(lr + 1);
      const int region = row / D, col = row % D;
      if (region < 2) {
        const float2 r = s_rope[(col % hd) >> 1];  // (cos, sin) of this pair at pos
        const float cs = r.x, sn = r.y;
        const float ra = a * cs - c * sn;
        const float rc = a * sn + c * cs;
        a = ra;
        c = rc;
      }
      if (region == 0) {
        op.out[col] = a;
        op.out[col + 1] = c;
      } else {
        void* cache = region == 1 ? op.kcache : op.vcache;
        const size_t base = (size_t)slot * D + col;
        store_kv(cache, base, a, P.kv_bf16);
        store_kv(cache, base + 1, c, P.kv_bf16);
      }
    }
  } else if (LL && epi == EPI_DQKV) {
    const int DD = pl.n_out / 3;
    for (int lr = tid; lr < nrows; lr += kCons) {
      const int row = grow(lr);
      if (row >= pl.n_out) continue;
      const float y = yrow(lr);
      if (row < DD)
        put(op.out, row, y);
      else if (row < 2 * DD)
        put(op.dk_out, row - DD, y);
      else
        put(op.dv_out, row - 2 * DD, y);
    }
  } else if (epi == EPI_ARGMAX) {
    unsigned long long best = 0ull;
    for (int lr = tid; lr < nrows; lr += kCons) {
      const int row = grow(lr);
      if (row >= pl.n_out) continue;
      const float y = yrow(lr);
      op.out[row] = y;
      if (LL && op.side_out) ll_st(op.side_out, row, wtag, y);  // for the top-k pick
      const unsigned long long k = PICKS ? pick_key(P.samp, 0, op.key_index, y, (uint32_t)row)
                                         : argmax_key(y, (uint32_t)row);
      best = k > best ? k : best;
    }
    best = warp_max_u64(best);
    if (lane == 0) s_key[warp] = best;
    bar_sync(1, kCons);
    if (tid == 0) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kCons / 32; ++w) m = s_key[w] > m ? s_key[w] : m;
      if (!LL || !op.no_keymax) atomicMax(P.keys + op.key_index, m);
      if (LL && !op.no_keymax) put_key_slot(P, op.key_index, blockIdx.x, wtag, m);
    }
  }
}

// ---------------------------------------------------------------- attention items
// one lane's EPL elements of a K/V row as loaded (no conversion): the next key's row is
// fetched while the current one is used
template <typename KT, int EPL> struct KvRaw;
template <> struct KvRaw<uint16_t, 4> {
  uint2 u;
  __device__ __forceinline__ void load(const uint16_t* p) { u = __ldcg(reinterpret_cast<const uint2*>(p)); }
  __device__ __forceinline__ void get(float (&o)[4]) const {
    o[0] = bf16lo(u.x); o[1] = bf16hi(u.x); o[2] = bf16lo(u.y); o[3] = bf16hi(u.y);
  }
};
template <> struct KvRaw<uint16_t, 2> {
  unsigned u;
  __device__ __forceinline__ void load(const uint16_t* p) { u = __ldcg(reinterpret_cast<const unsigned*>(p)); }
  __device__ __forceinline__ void get(float (&o)[2]) const { o[0] = bf16lo(u); o[1] = bf16hi(u); }
};
template <> struct KvRaw<uint16_t, 1> {
  unsigned u;
  __device__ __forceinline__ void load(const uint16_t* p) {
    u = (unsigned)__ldcg(reinterpret_cast<const unsigned short*>(p));
  }
  __device__ __forceinline__ void get(float (&o)[1]) const { o[0] = __uint_as_float(u << 16); }
};
template <int EPL> struct KvRawF;
template <> struct KvRawF<4> {
  float4 f;
  __device__ __forceinline__ void load(const float* p) { f = __ldcg(reinterpret_cast<const float4*>(p)); }
  __device__ __forceinline__ void get(float (&o)[4]) const { o[0] = f.x; o[1] = f.y; o[2] = f.z; o[3] = f.w; }
};
template <> struct KvRawF<2> {
  float2 f;
  __device__ __forceinline__ void load(const float* p) { f = __ldcg(reinterpret_cast<const float2*>(p)); }
  __device__ __forceinline__ void get(float (&o)[2]) const { o[0] = f.x; o[1] = f.y; }
};
template <> struct KvRawF<1> {
  float f;
  __device__ __forceinline__ void load(const float* p) { f = __ldcg(p); }
  __device__ __forceinline__ void get(float (&o)[1]) const { o[0] = f; }
};
template <> struct KvRaw<float, 4> : KvRawF<4> {};
template <> struct KvRaw<float, 2> : KvRawF<2> {};
template <> struct KvRaw<float, 1> : KvRawF<1> {};

// "moshi_lm.rs", `attend` for one session: work item (head, split of kps positions)
// per group of 4 warps; the last group to finish a head merges its splits in order.
// The split length follows the window so that every group of the grid gets about one
// item (16..64 positions, a multiple of 16): short windows give each warp few keys, so
// the chain of dependent K/V loads per warp stays short.
template <typename KT, int EPL>
__device__ __forceinline__ void attn_items(const PersParams& P, const PersOp& op, int tid,
                                           int warp, int lane, float (*s_am)[4],
                                           float (*s_al)[4], float (*s_aacc)[4][EPL * 32],
                                           int* s_last, int pos) {
  constexpr int HD = EPL * 32;
  const int group = warp >> 2, wig = warp & 3, gt = tid & 127;
  const int len = min(pos + 1, P.context);
  const int first = pos + 1 - len;
  const int groups = (int)gridDim.x * 2;
  int kps = (len * P.H + groups - 1) / groups;
  kps = min(64, max(16, (kps + 15) & ~15));
  const int nsplit = (len + kps - 1) / kps;  // <= P.nsplit = ceil(C / 16)
  const int items = P.H * nsplit;
  const float scale = 1.0f / sqrtf((float)HD);
  const float ninf = -__int_as_float(0x7f800000);
  const size_t pstride = (size_t)HD + 2;
  for (int it = blockIdx.x * 2 + group; it < items; it += groups) {
    const int h = it % P.H, split = it / P.H;
    const int j0 = first + split * kps;
    const int j1 = min(j0 + kps, pos + 1);
    const KT* kb = static_cast<const KT*>(op.kcache) + (size_t)h * HD + lane * EPL;
    const KT* vb = static_cast<const KT*>(op.vcache) + (size_t)h * HD + lane * EPL;
    // keys of this warp in flight: one; two to four (a register ring) spill at this
    // kernel's 96-register cap and slow every op down more than they save here
    constexpr int KPF = 1;
    KvRaw<KT, EPL> kr[KPF], vr[KPF];  // this warp's first keys, issued before q
#pragma unroll
    for (int pf = 0; pf < KPF; ++pf) {
      const int j = j0 + wig + 4 * pf;
      if (j < j1) {
        const size_t off = (size_t)(j % P.context) * P.D;
        kr[pf].load(kb + off);
        vr[pf].load(vb + off);
      }
    }
    float q[EPL];
    {
      KvRawF<EPL> qr;
      qr.load(P.attn_q + (size_t)h * HD + lane * EPL);
      qr.get(q);
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) q[e] *= scale;
    float m = ninf, l = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    for (int jb = j0 + wig; jb < j1; jb += 4 * KPF)
#pragma unroll
    for (int pf = 0; pf < KPF; ++pf) {
      const int j = jb + 4 * pf;
      if (j >= j1) break;
      float k[EPL], v[EPL];
      kr[pf].get(k);
      vr[pf].get(v);
      if (j + 4 * KPF < j1) {  // this slot's next key, in flight during the others
        const size_t off = (size_t)((j + 4 * KPF) % P.context) * P.D;
        kr[pf].load(kb + off);
        vr[pf].load(vb + off);
      }
      float sc = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) sc = fmaf(q[e], k[e], sc);
      sc = warp_sum(sc);
      const float mn = fmaxf(m, sc);
      const float corr = expf(m - mn);
      const float pe = expf(sc - mn);
      l = l * corr + pe;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = acc[e] * corr + pe * v[e];
      m = mn;
    }
    if (lane == 0) {
      s_am[group][wig] = m;
      s_al[group][wig] = l;
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) s_aacc[group][wig][lane * EPL + e] = acc[e];
    bar_sync(2 + group, 128);
    float* part = P.part + ((size_t)h * P.nsplit + split) * pstride;
    if (gt < HD) {
      float M = ninf;
#pragma unroll
      for (int w = 0; w < 4; ++w) M = fmaxf(M, s_am[group][w]);
      float L = 0.f, A = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        if (s_al[group][w] > 0.f) {
          const float c = expf(s_am[group][w] - M);
          L += s_al[group][w] * c;
          A += s_aacc[group][w][gt] * c;
        }
      }
      if (nsplit == 1) {
        // the whole window is this item's split: its merge is the output (what the ordered
        // merge of one split gives, bit for bit), without the partial and the ticket
        P.attn_out[(size_t)h * HD + gt] = A / L;
      } else {
        part[2 + gt] = A;
        if (gt == 0) {
          part[0] = M;
          part[1] = L;
        }
      }
    }
    if (nsplit == 1) {  // (uniform) the group's shared staging is reused by its next item
      bar_sync(2 + group, 128);
      continue;
    }
    __threadfence();
    bar_sync(2 + group, 128);
    if (gt == 0) s_last[group] = (atomicAdd(&P.counters[h], 1) == nsplit - 1);
    bar_sync(2 + group, 128);
    if (s_last[group]) {
      __threadfence();
      const float* pb = P.part + (size_t)h * P.nsplit * pstride;
      if (gt < HD) {
        // splits in order, one pass: the running max rescales what was summed so far
        // (the loads of later splits do not wait on earlier ones)
        float M = ninf, L = 0.f, A = 0.f;
#pragma unroll 4
        for (int s = 0; s < nsplit; ++s) {
          const float ms = ldcg(pb + s * pstride), ls = ldcg(pb + s * pstride + 1);
          const float as = ldcg(pb + s * pstride + 2 + gt);
          const float mn = fmaxf(M, ms);
          const float co = expf(M - mn), cs = expf(ms - mn);
          L = L * co + ls * cs;
          A = A * co + as * cs;
          M = mn;
        }
        P.attn_out[(size_t)h * HD + gt] = A / L;
      }
      if (gt == 0) P.counters[h] = 0;
    }
    bar_sync(2 + group, 128);
  }
}

// ---------------------------------------------------------------- the kernel
// PICKS: with the token-pick ops (top-k, Gumbel scores); without them (greedy frames) the
// kernel is about a quarter smaller, which leaves more of its hot code in the SM's
// instruction caches (measured: 18 us less per Moshi-7B frame)
// MINB: CTAs per SM.  Two for the temporal stack's weight stream (16 consumer warps per
// SM keep up with HBM; the register cap follows from 2 x 288 threads: 96), one for the
// depformer's latency-bound small ops, which exchange tagged words instead of meeting at
// grid barriers.
template <typename WT, typename KT, int EPL, bool PICKS, int MINB>
__global__ void __launch_bounds__(kThr, MINB) frame_persistent_kernel(const PersParams P) {
  constexpr int V = Chunk<WT>::V;
  constexpr bool LL = MINB == 1;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_red[2 * (kCons / 32)];
  __shared__ __align__(16) float s_att[kMaxStage];
  __shared__ unsigned long long s_key[kCons / 32];
  __shared__ float2 s_rope[64];  // (cos, sin) of each rotary pair at this frame's position
  __shared__ float s_am[2][4], s_al[2][4];
  __shared__ float s_aacc[2][4][EPL * 32];
  __shared__ int s_last[2];
  __shared__ unsigned s_issued;
  // the consumers read op descriptors, plans and the launch's position from shared
  // memory: op k+1's descriptor is fetched during op k and published by its last CTA
  // barrier, so no op starts with a round trip to global memory for its own parameters
  __shared__ __align__(16) PersOp s_op[2];
  __shared__ __align__(16) GemvPlan s_plan[kPersMaxPlans];
  __shared__ int s_pos, s_forcing;
  __shared__ uint32_t s_ebase;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // wait limit of this launch (a test may shorten it), and the op whose barrier a test
  // makes unreachable (-1: none)
  const uint64_t lim = P.wait_ctl && P.wait_ctl[0] ? P.wait_ctl[0] : kWaitLimitNs;
  const int stall_op = P.wait_ctl ? (int)P.wait_ctl[1] - 1 - P.op_base : -1;
  const int NS = P.n_slots;
  uint8_t* ring = smem;
  float* part = reinterpret_cast<float*>(smem + (size_t)NS * P.slot_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(part + P.part_floats);
  uint64_t* empty = full + NS;
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCons / 32);
    }
    fence_barrier_init();
    s_abort = 0;
    s_issued = 0;
    s_wait_lim = lim;
  }
  __syncthreads();

  if (warp == kCons / 32) {
    // ------------------------------------------------ producer: every op's weight tiles
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      TileCur c{};
      bool more = cur_seek<WT>(P, c);
      uint32_t gi = 0;
      while (more) {
        const int s = (int)(gi % (uint32_t)NS);
        if (gi >= (uint32_t)NS &&
            !mbar_wait_for(&empty[s], ((gi / (uint32_t)NS) - 1u) & 1u, lim)) {
          atomicOr(P.status, kDevTimeout);
          s_abort = 1;
        }
        if (s_abort) break;
        uint8_t* dst = ring + (size_t)s * P.slot_bytes;
        mbar_arrive_expect_tx(&full[s], cur_bytes<WT>(P, c));
        cur_ranges<WT>(P, c, [&](const uint8_t* src, uint32_t bytes, uint32_t off) {
          bulk_g2s(dst + off, src, bytes, &full[s], pol);
        });
        ++gi;
        more = cur_next<WT>(P, c);
      }
      s_issued = gi;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ consumers: ops in order
    constexpr int kOpWords = (int)(sizeof(PersOp) / 8);
    constexpr int kPlanWords = (int)(sizeof(GemvPlan) * kPersMaxPlans / 4);
    static_assert(sizeof(PersOp) % 8 == 0 && kOpWords <= kCons, "op descriptor words");
    static_assert((sizeof(GemvPlan) * kPersMaxPlans) % 4 == 0 && kPlanWords <= kCons,
                  "plan words");
    const unsigned long long* ops64 = reinterpret_cast<const unsigned long long*>(P.ops);
    unsigned long long* s_op64 = reinterpret_cast<unsigned long long*>(s_op);
    if (tid < kPlanWords)
      reinterpret_cast<int*>(s_plan)[tid] = reinterpret_cast<const int*>(P.plans)[tid];
    if (tid < kOpWords) s_op64[tid] = ops64[tid];
    pdl_wait();
    if (tid == 0) {
      s_pos = P.offsets[0];
      s_forcing = P.d_in[IoLayout{1}.flag_off()];
      // the frame's first launch advances the epoch; the tagged launch reads it (after
      // the first launch has finished)
      if (P.epoch_bump && blockIdx.x == 0) atomicAdd(P.epoch, 1u);
      s_ebase = LL ? ld_acquire(P.epoch) << 10 : 0u;
    }
    if (!LL && tid < P.head_dim / 2) {
      // "moshi_lm.rs", `rope_row`: freq_i = exp(-ln(theta) * 2i / hd), angle freq_i * pos;
      // every layer rotates at the same position, so the pairs are computed once
      const float freq = expf(-logf(P.rope_theta) * 2.0f * (float)tid / (float)P.head_dim);
      const float ang = freq * (float)P.offsets[0];
      s_rope[tid] = make_float2(cosf(ang), sinf(ang));
    }
    bar_sync(1, kCons);
    const int pos = s_pos, forcing = s_forcing;
    LLCtx lc{s_ebase, 0u, P};
    int cslot = 0;       // ring slot of the next tile to consume
    uint32_t cph = 0u;   // and the phase its "full" barrier completes
    float xr[Nx<WT>::N][V];
    const bool stamp = P.trace != nullptr && blockIdx.x == 0 && tid == 0;
    float ar[Nx<WT>::N][V];  // an RMSNorm op's alpha, loaded before its grid barrier
    for (int k = 0; k < P.n_ops; ++k) {
      // op k+1's descriptor, loaded now, stored to shared memory at the end of op k
      const unsigned long long nxt =
          (tid < kOpWords && k + 1 < P.n_ops) ? ops64[(size_t)(k + 1) * kOpWords + tid] : 0ull;
      if constexpr (!Chunk<WT>::kBand && !LL) {  // constant alpha of an RMSNorm prologue
        const PersOp& op = s_op[k & 1];
        if (op.type == OPT_GEMV && (op.pro == PRO_RMS || op.pro == PRO_RMS_EMB)) {
          const GemvPlan& pl = s_plan[op.plan];
          const int tig = tid % pl.tpr, CC = pl.K / V;
#pragma unroll
          for (int j = 0; j < Nx<WT>::N; ++j) {
            const int c = tig + j * pl.tpr;
#pragma unroll
            for (int v = 0; v < V; ++v) ar[j][v] = (c < CC) ? op.alpha[c * V + v] : 0.f;
          }
        }
      }
      lc.flip = (LL && k == stall_op) ? 0xffffffffu : 0u;
      const uint32_t wtag = s_ebase | (uint32_t)(P.op_base + k);
      if (!LL && k > 0 && !s_op[k & 1].nobar) {
        const unsigned target = (unsigned)k * gridDim.x + (k == stall_op ? 1u : 0u);
        if (tid == 0 && !grid_wait(P.grid_bar, target, lim)) {
          atomicOr(P.status, kDevTimeout);
          s_abort = 1;
        }
        if (bar_or(1, kCons, s_abort != 0)) break;
      }
      if (stamp) P.trace[P.op_base + k] = global_timer_ns();
      const PersOp& op = s_op[k & 1];
      if (!LL && op.type == OPT_ATTN) {  // (the temporal attention: not in the tagged kernel)
        attn_items<KT, EPL>(P, op, tid, warp, lane, s_am, s_al, s_aacc, s_last, pos);
      } else if (PICKS && op.type == OPT_TOPK) {
        // "moshi_lm.rs", `topk_sample` for pick key_index over the logits the previous op
        // wrote, by CTA 0 (its partial-sum buffer holds the selection's scratch)
        if (blockIdx.x == 0) {
          const int pk = op.key_index;
          const float* lg = op.in;
          if constexpr (LL) {
            // gather the logits from their tagged copy (8 words per thread and round trip)
            const int n = pk == 0 ? P.samp.V : P.samp.A;
            const uint32_t t = lc.want(op.tag_in);
            for (int i0 = 0; i0 < n; i0 += 8 * kCons) {
              // (a value is stored as it loads; a retry stores it again)
              uint64_t t0 = 0ull;
              bool ok;
              do {
                ok = true;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const int i = i0 + e * kCons + tid;
                  if (i < n) {
                    const unsigned long long w = ll_ld1(op.in, i);
                    P.topk_scratch[i] = ll_val(w);
                    ok &= ll_is(w, t);
                  }
                }
              } while (!ok && lc.again(t0));
            }
            bar_sync(1, kCons);
            lg = P.topk_scratch;
          }
          const double u = xs_u01(xs_advance(P.samp.rng[0], draws_before(P.samp, pk) + 1u,
                                             P.samp.jump));
          TopkShared& S = *reinterpret_cast<TopkShared*>(part);
          const int tok = topk_pick_block(lg, pk == 0 ? P.samp.V : P.samp.A,
                                          pk == 0 ? P.samp.top_k_text : P.samp.top_k,
                                          pk == 0 ? P.samp.temp_text : P.samp.temp, u, tid,
                                          kCons, S, SyncNamed<kCons>{});
          if (tid == 0) {
            const unsigned long long key = argmax_key(__ldcg(lg + tok), (uint32_t)tok);
            P.keys[pk] = key;
            if (LL) put_key_slot(P, pk, 0, wtag, key);
          }
        }
      } else {
        const GemvPlan& pl = s_plan[op.plan];
        int t0, t1;
        tile_range(pl, t0, t1);
        const int nt = t1 - t0;
        if (nt > 0) {
          const int g = tid / pl.tpr, tig = tid % pl.tpr;
          float resid_old = 0.f;  // the residual's old value, fetched before the tiles
          if (op.epi == EPI_RESID && tid < nt * pl.tile_rows) {
            const int row = (t0 + tid / pl.tile_rows) * pl.tile_rows + tid % pl.tile_rows;
            if (row < pl.n_out)
              resid_old = LL ? lc.wait1(op.out, row, lc.want(op.tag_res)) : ldcg(op.out + row);
          }
          bool ok = true;
          for (int kp = 0; kp < pl.kparts && ok; ++kp) {
            // reduction part kp covers columns [k0, k0 + Kw); partials accumulate
            const int k0 = kp * pl.kp_width;
            const int Kw = kp == pl.kparts - 1 ? pl.K - k0 : pl.kp_width;
            const int nch = (Kw / V + pl.tpr - 1) / pl.tpr;
            form_x<WT, LL, PICKS>(P, op, pl, nch, k0, Kw, xr, ar, g, tig, tid, warp, lane, s_red,
                           k & 1, s_att, forcing, lc, wtag, s_key);
            constexpr int BT = MINB == 1 ? kBurstTWide : kBurstT;
            if (nch <= 1 && nt > 2) {
              // full groups of BT; a remainder of one or two tiles as its own small group
              // (its butterfly and loads sized for two tiles, not BT)
              const int rem = MINB == 1 && nt > BT && nt % BT <= 2 ? nt % BT : 0;
              ok = consume_tiles<WT, 1, BT, true>(pl, Kw, kp > 0, nt - rem, 0, cslot, cph,
                                                  ring, P.slot_bytes, NS, full, empty, part,
                                                  xr, g, tig, warp, lane, lim);
              if constexpr (MINB == 1) {  // (the other launch keeps its smaller code)
                if (ok && rem > 0)
                  ok = consume_tiles<WT, 1, 2, true>(pl, Kw, kp > 0, rem, nt - rem, cslot, cph,
                                                     ring, P.slot_bytes, NS, full, empty, part,
                                                     xr, g, tig, warp, lane, lim);
              }
            } else if (nch <= 1)
              ok = consume_tiles<WT, 1, 2, true>(pl, Kw, kp > 0, nt, 0, cslot, cph, ring,
                                                 P.slot_bytes, NS, full, empty, part, xr, g,
                                                 tig, warp, lane, lim);
            else if constexpr (Nx<WT>::N >= 2) {  // two x chunks (weight bands hold one)
              if (nt > kStreamMinTiles)
                ok = consume_tiles<WT, 2, kStreamT, kStreamBurst>(pl, Kw, kp > 0, nt, 0, cslot,
                                                                  cph, ring, P.slot_bytes, NS,
                                                                  full, empty, part, xr, g, tig,
                                                                  warp, lane, lim);
              else
                ok = consume_tiles<WT, 2, 2, true>(pl, Kw, kp > 0, nt, 0, cslot, cph, ring,
                                                   P.slot_bytes, NS, full, empty, part, xr, g,
                                                   tig, warp, lane, lim);
            }
          }
          if (!ok) {
            atomicOr(P.status, kDevTimeout);
            s_abort = 1;
          }
          // the producer may raise s_abort at any time: decide on one uniform answer
          if (bar_or(1, kCons, s_abort != 0)) break;
          const bool rms = op.pro == PRO_RMS || op.pro == PRO_RMS_EMB;
          const float scale = rms ? rms_scale(P, pl, s_red, k & 1) : 1.0f;
          if (!LL && op.pro == PRO_RMS && op.side_out != nullptr && blockIdx.x == 0 && g == 0) {
            // CTA 0 keeps the normalised vector (the head's transformer_out)
            constexpr int V2 = Chunk<WT>::V;
#pragma unroll
            for (int j = 0; j < Nx<WT>::N; ++j) {
              const int c = tig + j * pl.tpr;
              if (c < pl.K / V2) {
#pragma unroll
                for (int v = 0; v < V2; ++v) op.side_out[c * V2 + v] = xr[j][v] * scale;
              }
            }
          }
          epilogue<WT, PICKS, LL>(P, op, pl, t0, nt, part, tid, warp, lane, s_key, s_rope,
                                  resid_old, pos, scale, lc, wtag);
        } else if (LL && op.epi == EPI_ARGMAX && !op.no_keymax && tid == 0) {
          put_key_slot(P, op.key_index, blockIdx.x, wtag, 0ull);  // no rows here
        }
      }
      if (tid < kOpWords && k + 1 < P.n_ops) s_op64[((k + 1) & 1) * kOpWords + tid] = nxt;
      bar_sync(1, kCons);
      if (!LL && tid == 0) grid_arrive(P.grid_bar);
    }
    // end of the launch (tagged: when CTA 0 is done)
    if (stamp && !s_abort && (LL || grid_wait(P.grid_bar, (unsigned)P.n_ops * gridDim.x, lim)))
      P.trace[P.op_base + P.n_ops] = global_timer_ns();
  }
  __syncthreads();
  pdl_trigger();
  if (s_abort) {
    // wind down: wait for this CTA's copies still in flight, bounded by the default
    // limit (not a shortened one: the copies land on their own within microseconds)
    if (tid == 0) {
      const unsigned issued = s_issued;
      for (unsigned i = issued > (unsigned)NS ? issued - NS : 0u; i < issued; ++i)
        (void)mbar_wait(&full[i % NS], (i / NS) & 1u);
    }
    __syncthreads();
  }
}

template <typename WT, typename KT, int EPL, bool PICKS, int MINB>
cudaError_t launch_t(const PersParams& p, int grid, int smem, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kThr, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, frame_persistent_kernel<WT, KT, EPL, PICKS, MINB>, p);
}

template <typename WT, typename KT, int EPL, bool PICKS, int MINB>
int max_grid_t(int smem) {
  int per_sm = 0, dev = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, frame_persistent_kernel<WT, KT, EPL, PICKS, MINB>,
                                                    kThr, (size_t)smem) != cudaSuccess)
    return 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return per_sm * sms;
}

template <typename WT, typename KT, int EPL, bool PICKS, int MINB>
cudaError_t configure_t(int smem) {
  return cudaFuncSetAttribute(frame_persistent_kernel<WT, KT, EPL, PICKS, MINB>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

// Instantiation sets.  Two CTAs per SM (the temporal launch): frame_persistent.cu (with
// token picks), frame_persistent_greedy.cu, frame_persistent_band.cu.  One CTA per SM
// (the depformer launch, which runs no temporal attention, so one head-size variant):
// frame_persistent_dep.cu.
#define RQ_PERS_EXTERN(W, K, E, PK, MB)                                                    \
  extern template cudaError_t launch_t<W, K, E, PK, MB>(const PersParams&, int, int,        \
                                                        cudaStream_t, bool);                \
  extern template int max_grid_t<W, K, E, PK, MB>(int);                                    \
  extern template cudaError_t configure_t<W, K, E, PK, MB>(int);
#define RQ_PERS_INSTANTIATE(W, K, E, PK, MB)                                               \
  template cudaError_t launch_t<W, K, E, PK, MB>(const PersParams&, int, int, cudaStream_t, \
                                                 bool);                                     \
  template int max_grid_t<W, K, E, PK, MB>(int);                                           \
  template cudaError_t configure_t<W, K, E, PK, MB>(int);
#define RQ_PERS_ALL(M, PK)                                                                 \
  M(float, float, 1, PK, 2) M(float, float, 2, PK, 2) M(float, float, 4, PK, 2)            \
  M(uint16_t, uint16_t, 1, PK, 2) M(uint16_t, uint16_t, 2, PK, 2)                          \
  M(uint16_t, uint16_t, 4, PK, 2)
// weight bands (bf16 K/V), head_dim 64 and 128: frame_persistent_band.cu
#define RQ_PERS_BANDS(M, PK)                                                               \
  M(q8_t, uint16_t, 2, PK, 2) M(q8_t, uint16_t, 4, PK, 2) M(q4_t, uint16_t, 2, PK, 2)      \
  M(q4_t, uint16_t, 4, PK, 2)
#define RQ_PERS_DEP(M, PK)                                                                 \
  M(float, float, 1, PK, 1) M(uint16_t, uint16_t, 1, PK, 1) M(q8_t, uint16_t, 1, PK, 1)    \
  M(q4_t, uint16_t, 1, PK, 1)

}  // namespace pers

}  // namespace rqk
