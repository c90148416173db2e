// attn.cu -- split-K single-query decode attention over the temporal K/V window.
//
// "inferencelayer 0.2.4 -- src/moshi_lm.rs", `attend`: for each head,
// s_j = (q . k_j) / sqrt(head_dim) over the cached positions j of the window,
// p = softmax(s) with the maximum subtracted, o = sum_j p_j v_j.
//
// The window of session b holds positions [pos - len + 1, pos] with
// len = min(pos + 1, C); position j lives in cache slot j % C.  A work item is `kps`
// consecutive positions of one (session, head); a CTA keeps an online softmax
// (running max m, sum l, weighted values) per warp in registers, merges its warps in a
// fixed order and writes the item's partial (m, l, acc).  The last CTA of a (session,
// head) to finish -- found with an atomic ticket -- merges the partials in split order,
// so the result does not depend on which CTA finished last.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace rqk {

template <typename KT>
__device__ __forceinline__ float kv_load(const KT* p);
template <>
__device__ __forceinline__ float kv_load<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float kv_load<uint16_t>(const uint16_t* p) {
  return __uint_as_float(((uint32_t)*p) << 16);
}

// This lane's EPL consecutive elements of a K or V row in shared memory, widened to f32.
template <typename KT, int EPL>
__device__ __forceinline__ void load_row(const KT* r, float (&v)[EPL]) {
  if constexpr (sizeof(KT) == 2 && EPL == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(r);
    v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  } else if constexpr (sizeof(KT) == 2 && EPL == 2) {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(r);
    v[0] = bf16lo(u); v[1] = bf16hi(u);
  } else if constexpr (sizeof(KT) == 4 && EPL == 4) {
    const float4 f = *reinterpret_cast<const float4*>(r);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
  } else if constexpr (sizeof(KT) == 4 && EPL == 2) {
    const float2 f = *reinterpret_cast<const float2*>(r);
    v[0] = f.x; v[1] = f.y;
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] = kv_load<KT>(r + e);
  }
}

// The 16 elements of a K or V row in shared memory that lane gl of a G-lane group owns,
// widened to f32: 16-byte chunks c = 0.. at element c * G * EPC + gl * EPC (EPC elements
// per chunk), so the G lanes of a group read each chunk row contiguously (no bank
// conflicts).  Element e of the result is dimension dim16<KT>(e, gl, G).
template <typename KT>
__device__ __forceinline__ int dim16(int e, int gl, int G) {
  constexpr int EPC = 16 / sizeof(KT);
  return (e / EPC) * G * EPC + gl * EPC + (e % EPC);
}

template <typename KT>
__device__ __forceinline__ void load16(const KT* row, int gl, int G, float (&v)[16]) {
  constexpr int EPC = 16 / sizeof(KT);
#pragma unroll
  for (int c = 0; c < 16 / EPC; ++c) {
    const uint4 u = *reinterpret_cast<const uint4*>(row + c * G * EPC + gl * EPC);
    if constexpr (sizeof(KT) == 2) {
      v[8 * c + 0] = bf16lo(u.x); v[8 * c + 1] = bf16hi(u.x);
      v[8 * c + 2] = bf16lo(u.y); v[8 * c + 3] = bf16hi(u.y);
      v[8 * c + 4] = bf16lo(u.z); v[8 * c + 5] = bf16hi(u.z);
      v[8 * c + 6] = bf16lo(u.w); v[8 * c + 7] = bf16hi(u.w);
    } else {
      v[4 * c + 0] = __uint_as_float(u.x); v[4 * c + 1] = __uint_as_float(u.y);
      v[4 * c + 2] = __uint_as_float(u.z); v[4 * c + 3] = __uint_as_float(u.w);
    }
  }
}

// packed pair of f32 (two lanes of one 64-bit register pair) and its FMA
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pack2(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(f32x2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ void ffma2(f32x2& d, f32x2 a, f32x2 b) {  // d += a * b, per lane
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

// load16 as 8 packed pairs: pair i holds elements 2i, 2i + 1 (dimensions dim16(2i), +1)
template <typename KT>
__device__ __forceinline__ void load16p(const KT* row, int gl, int G, f32x2 (&v)[8]) {
  constexpr int EPC = 16 / sizeof(KT);
#pragma unroll
  for (int c = 0; c < 16 / EPC; ++c) {
    const uint4 u = *reinterpret_cast<const uint4*>(row + c * G * EPC + gl * EPC);
    if constexpr (sizeof(KT) == 2) {
      v[4 * c + 0] = pack2(bf16lo(u.x), bf16hi(u.x));
      v[4 * c + 1] = pack2(bf16lo(u.y), bf16hi(u.y));
      v[4 * c + 2] = pack2(bf16lo(u.z), bf16hi(u.z));
      v[4 * c + 3] = pack2(bf16lo(u.w), bf16hi(u.w));
    } else {
      v[2 * c + 0] = pack2(__uint_as_float(u.x), __uint_as_float(u.y));
      v[2 * c + 1] = pack2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
  }
}

// One work item = (session, split, head).  Splits are cut in cache-slot
// space: the window of session b is every slot when pos >= C, else slots 0..pos, so
// split s covers slots [s kps, min((s + 1) kps, min(pos + 1, C))) and never wraps.
// Softmax is order-free, so visiting the window in slot order rather than position
// order changes only the rounding.
struct AttnItem {
  int b, h, split, ns, j0, j1;
};

__device__ __forceinline__ bool attn_decode_item(const AttnParams& p, int it, AttnItem& x) {
  // head fastest: the items in flight at once read every head's slice of the same K/V
  // rows, so each row is fetched from DRAM as a whole
  x.h = it % p.H;
  const int bs = it / p.H;
  x.split = bs % p.nsplit;
  x.b = bs / p.nsplit;
  const int lim = min(p.offsets[x.b] + 1, p.C);
  x.ns = (lim + p.kps - 1) / p.kps;
  if (x.split >= x.ns) return false;
  x.j0 = x.split * p.kps;
  x.j1 = min(x.j0 + p.kps, lim);
  return true;
}

// The same items numbered densely: session b owns H * ns_b consecutive indices from
// pref[b] (pref = prefix sums over sessions, pref[0] = 0), split-major, head fastest.
// Every index is a real item, so the persistent grid never walks the empty splits
// beyond short windows (at position 50 of a 3000-slot cache, 46 of 47 splits).
constexpr int kAttnDenseMaxB = 256;  // sessions whose prefix sums fit the CTA's table

// item i of the dense numbering; `b` is a session at or before the item's (a CTA's items
// only move forward, so the walk from its previous item's session is short)
__device__ __forceinline__ void attn_dense_item(const AttnParams& p, const int* pref, int i,
                                                int& b, AttnItem& x) {
  while (b + 1 < p.batch && pref[b + 1] <= i) ++b;
  x.b = b;
  const int r = i - pref[b];
  x.h = r % p.H;
  x.split = r / p.H;
  const int lim = min(p.offsets[x.b] + 1, p.C);
  x.ns = (lim + p.kps - 1) / p.kps;
  x.j0 = x.split * p.kps;
  x.j1 = min(x.j0 + p.kps, lim);
}

#ifndef RQ_ATTN_STAGES
#define RQ_ATTN_STAGES 2
#endif
#ifndef RQ_ATTN_WARPS
#define RQ_ATTN_WARPS 4
#endif
constexpr int kAttnStages = RQ_ATTN_STAGES;  // K/V chunks per CTA (ring depth)
constexpr int kAttnMaxKps = 64;              // positions per work item, at most
constexpr int kAttnWarps = RQ_ATTN_WARPS;

// Persistent grid over the work items: each CTA takes items blockIdx.x, + gridDim.x, ...
// skipping splits beyond a session's window.  Thread 0 loads an item's K and V rows with
// one 2-D TMA box each ({head_dim, kps} out of the cache viewed as rows of D) into a
// kAttnStages-deep shared-memory ring, so the next items' chunks stream while this one
// is computed.  Within a warp, groups of head_dim / 16 lanes each take one key (16
// dimensions per lane), so a warp steps through 32 / (head_dim / 16) keys at once with
// log2(head_dim / 16) shuffles; each group keeps an online softmax in registers, the
// groups merge by a fixed butterfly, the warps in a fixed order into the item's partial
// (m, l, acc), combined per (session, head) by attn_merge_kernel.
template <typename KT, int EPL>
__global__ void __launch_bounds__(kAttnWarps * 32)
    attn_decode_kernel(const AttnParams p, const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap) {
  constexpr int HD = EPL * 32;
  constexpr int NS = kAttnStages, NW = kAttnWarps;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t s_full[NS];
  __shared__ int s_item[NS];
  __shared__ AttnItem s_info[NS];  // the item of each stage, decoded once by thread 0
  __shared__ float s_m[NW], s_l[NW];
  __shared__ float s_acc[NW][HD];
  __shared__ int s_pref[kAttnDenseMaxB + 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kps = p.kps;
  KT* const stage0 = reinterpret_cast<KT*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const size_t stage_elems = (size_t)2 * kps * HD;  // K rows then V rows
  const uint32_t stage_bytes = (uint32_t)(stage_elems * sizeof(KT));
  const bool dense = p.batch <= kAttnDenseMaxB;
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&s_full[i], 1);
    fence_barrier_init();
    tc::prefetch_tmap(&kmap);
    tc::prefetch_tmap(&vmap);
  }
  pdl_wait();
  if (dense && warp == 0) {
    // prefix sums of H * ns_b over the sessions, 32 sessions per warp scan step
    int run = 0;
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < p.batch) n = p.H * ((min(p.offsets[b] + 1, p.C) + kps - 1) / kps);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, n, o);
        if (lane >= o) n += t;
      }
      if (b < p.batch) s_pref[b + 1] = run + n;
      run += __shfl_sync(0xffffffffu, n, 31);
    }
    if (lane == 0) s_pref[0] = 0;
  }
  __syncthreads();
  const int total = dense ? s_pref[p.batch] : p.batch * p.H * p.nsplit;
  const uint64_t pol = l2_policy_evict_first();
  // thread 0 only: the next valid item at or after `it` (stride gridDim.x), then its load
  int last = blockIdx.x - (int)gridDim.x;  // last item index issued by this CTA
  int walk_b = 0;                          // dense numbering: session of that item
  auto issue_next = [&](int s) {
    AttnItem x;
    int it = last + (int)gridDim.x;
    const int G = (int)gridDim.x, per_b = p.nsplit * p.H;
    if (dense) {
      if (it < total) attn_dense_item(p, s_pref, it, walk_b, x);
    } else {
      while (it < total && !attn_decode_item(p, it, x)) {
        // past session b's window: every later split of b is empty too, so go to the
        // first item of session b + 1 in this CTA's stride class (it mod G fixed)
        const int base = (x.b + 1) * per_b;
        it = base + (((it - base) % G) + G) % G;
      }
    }
    s_item[s] = it;
    if (it >= total) return;
    s_info[s] = x;
    last = it;
    KT* const st = stage0 + (size_t)s * stage_elems;
    const int row = (int)(p.row_bs * x.b + p.row0 + x.j0);
    mbar_arrive_expect_tx(&s_full[s], stage_bytes);  // full boxes; tail rows unused
    tc::tma_load_2d(st, &kmap, x.h * HD, row, &s_full[s], pol);
    tc::tma_load_2d(st + (size_t)kps * HD, &vmap, x.h * HD, row, &s_full[s], pol);
  };
  if (tid == 0)
    for (int s = 0; s < NS; ++s) issue_next(s);
  __syncthreads();
  const float scale = 1.0f / sqrtf((float)HD);
  const float ninf = -__int_as_float(0x7f800000);
  for (int k = 0;; ++k) {
    const int s = k % NS;
    const int item = s_item[s];
    if (item >= total) break;
    const bool ok = mbar_wait(&s_full[s], (uint32_t)(k / NS) & 1u);
    if (__syncthreads_or(!ok)) {
      // a copy never landed: record it, wait (bounded) for the other stages, stop
      if (tid == 0) {
        if (p.status) atomicOr(p.status, kDevTimeout);
        for (int d = 1; d < NS; ++d)
          if (s_item[(k + d) % NS] < total)
            (void)mbar_wait(&s_full[(k + d) % NS], (uint32_t)((k + d) / NS) & 1u);
      }
      return;
    }
    const AttnItem cur = s_info[s];
    const int b = cur.b, h = cur.h, n = cur.j1 - cur.j0;
    // G lanes share one key, 16 dimensions each; a warp covers KPI keys per step
    constexpr int G = HD / 16, KPI = 32 / G;
    const int grp = lane / G, gl = lane % G;
    const KT* ks = stage0 + (size_t)s * stage_elems;
    const KT* vs = ks + (size_t)kps * HD;
    f32x2 q2[8];
    const float* qp = p.q + (size_t)b * p.D + (size_t)h * HD;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      q2[i] = pack2(qp[dim16<KT>(2 * i, gl, G)] * scale, qp[dim16<KT>(2 * i + 1, gl, G)] * scale);
    // pass 1: this warp's scores (key group grp takes key warp*KPI + st*NW*KPI + grp), max
    constexpr int kSteps = kAttnMaxKps / (NW * KPI) > 0 ? kAttnMaxKps / (NW * KPI) : 1;
    float sc[kSteps];
    float m = ninf;
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
      const int r = warp * KPI + st * NW * KPI + grp;  // uniform within the group
      float d = 0.f;
      if (r < n) {
        f32x2 kv[8];
        load16p<KT>(ks + (size_t)r * HD, gl, G, kv);
        f32x2 d2 = pack2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 8; ++i) ffma2(d2, q2[i], kv[i]);
        float dx, dy;
        unpack2(d2, dx, dy);
        d = dx + dy;
      }
#pragma unroll
      for (int o = G / 2; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      sc[st] = r < n ? d : ninf;
      m = fmaxf(m, sc[st]);
    }
#pragma unroll
    for (int o = G; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    // pass 2: exp against the warp's max (no per-key rescale), weighted values
    float l = 0.f;
    f32x2 acc2[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc2[i] = pack2(0.f, 0.f);
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
      const int r = warp * KPI + st * NW * KPI + grp;
      if (r < n) {
        const float pe = expf(sc[st] - m);
        l += pe;
        const f32x2 p2 = pack2(pe, pe);
        f32x2 vv[8];
        load16p<KT>(vs + (size_t)r * HD, gl, G, vv);
#pragma unroll
        for (int i = 0; i < 8; ++i) ffma2(acc2[i], p2, vv[i]);
      }
    }
    // merge the key groups (same max): plain sums in a fixed butterfly order
    float acc[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) unpack2(acc2[i], acc[2 * i], acc[2 * i + 1]);
#pragma unroll
    for (int o = G; o < 32; o <<= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
      for (int e = 0; e < 16; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
    }
    if (lane == 0) {
      s_m[warp] = m;
      s_l[warp] = l;
    }
    if (lane < G) {
#pragma unroll
      for (int e = 0; e < 16; ++e) s_acc[warp][dim16<KT>(e, gl, G)] = acc[e];
    }
    __syncthreads();  // every warp is done with this stage and has published its state
    if (tid == 0) issue_next(s);  // refill the stage just consumed
    // merge the warps in a fixed order into this split's partial (m, l, acc); a window
    // of one split is the whole result (the merge kernel skips it)
    if (tid < HD) {
      const size_t pstride = (size_t)HD + 2;
      float M = ninf;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w]);
      float L = 0.f, A = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        if (s_l[w] > 0.f) {
          const float c = expf(s_m[w] - M);
          L += s_l[w] * c;
          A += s_acc[w][tid] * c;
        }
      }
      if (cur.ns == 1) {
        const float o = A / L;
        const size_t i = (size_t)b * p.D + (size_t)h * HD + tid;
        p.out[i] = o;
        if (p.out_bf16) store_bf16_parts(p.out_bf16, (size_t)p.nb * p.D, i, o);
      } else {
        float* part = p.part + (((size_t)b * p.H + h) * p.nsplit + cur.split) * pstride;
        part[2 + tid] = A;
        if (tid == 0) {
          part[0] = M;
          part[1] = L;
        }
      }
    }
    __syncthreads();  // s_m / s_acc / s_item are reused by the next item
  }
  // dependents launch once this CTA is done: launched early, the merge kernel's blocks
  // would sit resident beside the streaming CTAs for the whole kernel
  pdl_trigger();
}

// Grid (head, session), head_dim threads: combine the partials of every split of the
// window in split order (deterministic) into o = sum_s A_s e^(M_s - M) / sum_s L_s e^(M_s - M).
__global__ void __launch_bounds__(128) attn_merge_kernel(const AttnParams p) {
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  if (tid >= p.hd) return;
  const int ns = (min(p.offsets[b] + 1, p.C) + p.kps - 1) / p.kps;
  if (ns == 1) return;  // the attention kernel wrote this (session, head) itself
  const size_t pstride = (size_t)p.hd + 2;
  const float* pb = p.part + ((size_t)b * p.H + h) * p.nsplit * pstride;
  float M = -__int_as_float(0x7f800000);
  for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, pb[sp * pstride]);
  float L = 0.f, A = 0.f;
  for (int sp = 0; sp < ns; ++sp) {
    const float c = expf(pb[sp * pstride] - M);
    L += pb[sp * pstride + 1] * c;
    A += pb[sp * pstride + 2 + tid] * c;
  }
  const float o = A / L;
  const size_t i = (size_t)b * p.D + (size_t)h * p.hd + tid;
  p.out[i] = o;
  if (p.out_bf16) store_bf16_parts(p.out_bf16, (size_t)p.nb * p.D, i, o);
}

// Resident CTAs per SM of one instantiation at `smem` bytes (sets the shared-memory
// attribute first).  Called outside stream capture by attn_configure, and lazily by the
// standalone entry points.
template <typename KT, int EPL>
static cudaError_t attn_occupancy(size_t smem, int* per_sm) {
  static int cached = 0;
  static size_t cached_smem = 0;
  if (cached == 0 || cached_smem != smem) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<KT, EPL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attn_decode_kernel<KT, EPL>,
                                                      kAttnWarps * 32, smem);
    if (e != cudaSuccess) return e;
    cached = n > 0 ? n : 1;
    cached_smem = smem;
  }
  *per_sm = cached;
  return cudaSuccess;
}

template <typename KT, int EPL>
static size_t attn_smem(int kps) {
  return (size_t)kAttnStages * 2 * kps * EPL * 32 * sizeof(KT) + 1024;  // K, V stages + align
}

template <typename KT, int EPL>
static cudaError_t launch_attn_t(const AttnParams& p, cudaStream_t s, bool pdl) {
  constexpr int HD = EPL * 32;
  const size_t smem = attn_smem<KT, EPL>(p.kps);
  int per_sm = 0, dev = 0, sms = 0;
  cudaError_t e = attn_occupancy<KT, EPL>(smem, &per_sm);
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  CUtensorMap kmap, vmap;
  const bool bf = sizeof(KT) == 2;
  if ((e = encode_tmap_2d(&kmap, bf, p.kbase, p.rows, p.D, HD, p.kps, false)) != cudaSuccess)
    return e;
  if ((e = encode_tmap_2d(&vmap, bf, p.vbase, p.rows, p.D, HD, p.kps, false)) != cudaSuccess)
    return e;
  const long long total = (long long)p.batch * p.H * p.nsplit;
  const long long grid = total < (long long)per_sm * sms ? total : (long long)per_sm * sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kAttnWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if ((e = cudaLaunchKernelEx(&cfg, attn_decode_kernel<KT, EPL>, p, kmap, vmap)) != cudaSuccess)
    return e;
  cudaLaunchConfig_t mc = {};
  mc.gridDim = dim3((unsigned)p.H, (unsigned)p.batch, 1);
  mc.blockDim = dim3(128, 1, 1);
  mc.stream = s;
  mc.attrs = attr;
  mc.numAttrs = 1;  // the merge always follows the attention kernel on the stream
  return cudaLaunchKernelEx(&mc, attn_merge_kernel, p);
}

cudaError_t attn_configure(int hd, bool kv_bf16, int kps) {
  int n = 0;
  switch (hd) {
    case 32:
      return kv_bf16 ? attn_occupancy<uint16_t, 1>(attn_smem<uint16_t, 1>(kps), &n)
                     : attn_occupancy<float, 1>(attn_smem<float, 1>(kps), &n);
    case 64:
      return kv_bf16 ? attn_occupancy<uint16_t, 2>(attn_smem<uint16_t, 2>(kps), &n)
                     : attn_occupancy<float, 2>(attn_smem<float, 2>(kps), &n);
    case 128:
      return kv_bf16 ? attn_occupancy<uint16_t, 4>(attn_smem<uint16_t, 4>(kps), &n)
                     : attn_occupancy<float, 4>(attn_smem<float, 4>(kps), &n);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn(const AttnParams& p, bool kv_bf16, cudaStream_t s, bool pdl) {
  if (p.kps < 1 || p.kps > kAttnMaxKps) return cudaErrorInvalidValue;
  switch (p.hd) {
    case 32:
      return kv_bf16 ? launch_attn_t<uint16_t, 1>(p, s, pdl) : launch_attn_t<float, 1>(p, s, pdl);
    case 64:
      return kv_bf16 ? launch_attn_t<uint16_t, 2>(p, s, pdl) : launch_attn_t<float, 2>(p, s, pdl);
    case 128:
      return kv_bf16 ? launch_attn_t<uint16_t, 4>(p, s, pdl) : launch_attn_t<float, 4>(p, s, pdl);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace rqk

// ---------------------------------------------------------------- standalone entry
#include "../../include/rq.h"

namespace {
constexpr int kStandaloneKps = rqk::kStandaloneAttnKps;  // positions per split, as in the frame

size_t partial_bytes(int B, int H, int hd, int C) {
  return rqk::standalone_attn_partial_bytes(B, H, hd, C);
}
}  // namespace

extern "C" size_t rq_attention_workspace_size(int32_t batch, int32_t heads, int32_t head_dim,
                                              int32_t context) {
  if (batch < 1 || heads < 1 || head_dim < 1 || context < 1) return 0;
  return partial_bytes(batch, heads, head_dim, context) + (size_t)batch * heads * sizeof(int);
}

extern "C" rq_status rq_attention(int32_t batch, int32_t heads, int32_t head_dim,
                                  int32_t context, int32_t kv_dtype, const float* q,
                                  const void* k, const void* v, const int32_t* positions,
                                  float* out, void* workspace, size_t workspace_bytes,
                                  void* cuda_stream) {
  using namespace rqk;
  if (batch < 1 || heads < 1 || context < 1 || batch > 65535 || heads > 65535)
    return RQ_ERR_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return RQ_ERR_UNSUPPORTED;
  if (kv_dtype != RQ_F32 && kv_dtype != RQ_BF16) return RQ_ERR_ARG;
  if (!q || !k || !v || !positions || !out || !workspace) return RQ_ERR_ARG;
  // the K/V rows are bulk-copied into shared memory: 16-byte aligned sources
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u) return RQ_ERR_ARG;
  if (workspace_bytes < rq_attention_workspace_size(batch, heads, head_dim, context))
    return RQ_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  AttnParams a{};
  a.q = q;
  a.kbase = k;
  a.vbase = v;
  a.rows = (long long)batch * context;
  a.row0 = 0;
  a.row_bs = context;
  a.offsets = positions;
  a.part = static_cast<float*>(workspace);
  a.counters = reinterpret_cast<int*>(static_cast<char*>(workspace) +
                                      partial_bytes(batch, heads, head_dim, context));
  a.out = out;
  a.D = heads * head_dim;
  a.H = heads;
  a.hd = head_dim;
  a.C = context;
  a.kps = kStandaloneKps;
  a.nsplit = (context + kStandaloneKps - 1) / kStandaloneKps;
  a.batch = batch;
  a.status = nullptr;
  if (cudaMemsetAsync(a.counters, 0, (size_t)batch * heads * sizeof(int), s) != cudaSuccess)
    return RQ_ERR_CUDA;
  return launch_attn(a, kv_dtype == RQ_BF16, s, false) == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}

// ---------------------------------------------------------------- batched depformer attention
namespace rqk {

// "moshi_lm.rs", `attend` over the depformer's per-frame keys 0..n_keys-1, for every
// session: one warp per (session, head), the head's dimensions spread over the lanes;
// writes the bf16 operand parts of the next tensor-core GEMM (parts nb rows apart).
// "moshi_lm.rs", `attend` over the depformer's per-frame keys 0..n_keys-1 (<= 8) for
// session b, head h: one warp, dimension e = lane + 32 i on lane `lane`.  The query, every
// key and then every value are loaded together (two round trips instead of one per key);
// the sums run in the same order as a key-by-key loop.
__global__ void __launch_bounds__(32) dattn_batched_kernel(const float* dq, long long dq_bs,
                                                           const float* dk, const float* dv,
                                                           long long dkv_bs, int n_keys,
                                                           int hd, int DD, uint16_t* out,
                                                           long long out_bs, int nb) {
  constexpr int kE = 4;  // head_dim <= 128
  const int b = blockIdx.x, h = blockIdx.y, lane = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const float* q = dq + (size_t)b * dq_bs + (size_t)h * hd;
  const float* K = dk + (size_t)b * dkv_bs + (size_t)h * hd;
  const float* Vv = dv + (size_t)b * dkv_bs + (size_t)h * hd;
  const float scale = 1.0f / sqrtf((float)hd);
  float qv[kE], kk[8][kE];
#pragma unroll
  for (int i = 0; i < kE; ++i) {
    const int e = lane + 32 * i;
    qv[i] = e < hd ? q[e] : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) kk[j][i] = (j < n_keys && e < hd) ? K[(size_t)j * DD + e] : 0.f;
  }
  float sc[8];
  float mx = -__int_as_float(0x7f800000);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float d = 0.f;
#pragma unroll
    for (int i = 0; i < kE; ++i)
      if (lane + 32 * i < hd) d = fmaf(qv[i], kk[j][i], d);
    sc[j] = warp_sum(d) * scale;
    if (j < n_keys) mx = fmaxf(mx, sc[j]);
  }
  float den = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sc[j] = j < n_keys ? expf(sc[j] - mx) : 0.f;
    den += sc[j];
  }
#pragma unroll
  for (int i = 0; i < kE; ++i) {
    const int e = lane + 32 * i;
#pragma unroll
    for (int j = 0; j < 8; ++j) kk[j][i] = (j < n_keys && e < hd) ? Vv[(size_t)j * DD + e] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < kE; ++i) {
    const int e = lane + 32 * i;
    if (e >= hd) continue;
    float o = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < n_keys) o += sc[j] / den * kk[j][i];
    store_bf16_parts(out, (size_t)nb * out_bs, (size_t)b * out_bs + (size_t)h * hd + e, o);
  }
}

cudaError_t launch_dattn_batched(const float* dq, long long dq_bs, const float* dk,
                                 const float* dv, long long dkv_bs, int n_keys, int B,
                                 int heads, int hd, uint16_t* out, long long out_bs, int nb,
                                 cudaStream_t s, bool pdl) {
  if (n_keys < 1 || n_keys > 8 || hd > 128) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B, (unsigned)heads, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, dattn_batched_kernel, dq, dq_bs, dk, dv, dkv_bs, n_keys, hd,
                            heads * hd, out, out_bs, nb);
}

}  // namespace rqk
