// attn.cu -- split-K single-query decode attention over the temporal K/V window.
//
// "inferencelayer 0.2.4 -- src/moshi_lm.rs", `attend`: for each head,
// s_j = (q . k_j) / sqrt(head_dim) over the cached positions j of the window,
// p = softmax(s) with the maximum subtracted, o = sum_j p_j v_j.
//
// The window of session b holds positions [pos - len + 1, pos] with
// len = min(pos + 1, C); position j lives in cache slot j % C.  Grid (split, head,
// session): each CTA covers `kps` consecutive positions with 4 warps (one key per
// warp per step, the head's dimensions spread over the lanes), keeps an online
// softmax (running max m, sum l, weighted values) in registers, merges its warps in a
// fixed order and writes a partial (m, l, acc).  The last CTA of a (session, head)
// to finish -- found with an atomic ticket -- merges the partials in split order, so
// the result does not depend on which CTA finished last.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace rqk {

template <typename KT>
__device__ __forceinline__ float kv_load(const KT* p);
template <>
__device__ __forceinline__ float kv_load<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float kv_load<uint16_t>(const uint16_t* p) {
  return __uint_as_float(((uint32_t)*p) << 16);
}

template <typename KT, int EPL>
__global__ void __launch_bounds__(128) attn_decode_kernel(const AttnParams p) {
  constexpr int HD = EPL * 32;
  __shared__ float s_m[4], s_l[4];
  __shared__ float s_acc[4][HD];
  __shared__ int s_last;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();
  pdl_wait();
  const int pos = p.offsets[b];
  const int len = min(pos + 1, p.C);
  const int first = pos + 1 - len;
  const int nsplit = (len + p.kps - 1) / p.kps;
  if (split >= nsplit) return;
  const int j0 = first + split * p.kps;
  const int j1 = min(j0 + p.kps, pos + 1);

  float q[EPL];
  const float* qp = p.q + (size_t)b * p.D + (size_t)h * HD + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; ++e) q[e] = qp[e];
  const float scale = 1.0f / sqrtf((float)HD);
  const float ninf = -__int_as_float(0x7f800000);
  float m = ninf, l = 0.f, acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  const KT* kb = static_cast<const KT*>(p.kc) + (size_t)b * p.kv_bs + (size_t)h * HD + lane * EPL;
  const KT* vb = static_cast<const KT*>(p.vc) + (size_t)b * p.kv_bs + (size_t)h * HD + lane * EPL;
  for (int j = j0 + warp; j < j1; j += 4) {
    const size_t off = (size_t)(j % p.C) * p.D;
    float k[EPL], v[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      k[e] = kv_load<KT>(kb + off + e);
      v[e] = kv_load<KT>(vb + off + e);
    }
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) s = fmaf(q[e], k[e], s);
    s = warp_sum(s) * scale;
    const float mn = fmaxf(m, s);
    const float corr = expf(m - mn);
    const float pe = expf(s - mn);
    l = l * corr + pe;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = acc[e] * corr + pe * v[e];
    m = mn;
  }
  if (lane == 0) {
    s_m[warp] = m;
    s_l[warp] = l;
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) s_acc[warp][lane * EPL + e] = acc[e];
  __syncthreads();

  const size_t pstride = (size_t)HD + 2;
  float* part = p.part + (((size_t)b * p.H + h) * p.nsplit + split) * pstride;
  if (tid < HD) {
    float M = ninf;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, s_m[w]);
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (s_l[w] > 0.f) {
        const float c = expf(s_m[w] - M);
        L += s_l[w] * c;
        A += s_acc[w][tid] * c;
      }
    }
    part[2 + tid] = A;
    if (tid == 0) {
      part[0] = M;
      part[1] = L;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int t = atomicAdd(&p.counters[b * p.H + h], 1);
    s_last = (t == nsplit - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const float* pb = p.part + ((size_t)b * p.H + h) * p.nsplit * pstride;
  if (tid < HD) {
    float M = ninf;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, __ldcg(pb + s * pstride));
    float L = 0.f, A = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float c = expf(__ldcg(pb + s * pstride) - M);
      L += __ldcg(pb + s * pstride + 1) * c;
      A += __ldcg(pb + s * pstride + 2 + tid) * c;
    }
    const float o = A / L;
    p.out[(size_t)b * p.D + (size_t)h * HD + tid] = o;
    if (p.out_bf16)
      store_bf16x3(p.out_bf16, (size_t)p.nb * p.D, (size_t)b * p.D + (size_t)h * HD + tid, o);
  }
  if (tid == 0) p.counters[b * p.H + h] = 0;
}

template <typename KT, int EPL>
static cudaError_t launch_attn_t(const AttnParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.nsplit, (unsigned)p.H, (unsigned)p.batch);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_decode_kernel<KT, EPL>, p);
}

cudaError_t launch_attn(const AttnParams& p, bool kv_bf16, cudaStream_t s, bool pdl) {
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
constexpr int kStandaloneKps = 64;  // positions per split, as in the frame

size_t partial_bytes(int B, int H, int hd, int C) {
  const size_t nsplit = (size_t)(C + kStandaloneKps - 1) / kStandaloneKps;
  return ((size_t)B * H * nsplit * (hd + 2) * sizeof(float) + 255) & ~(size_t)255;
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
  if (workspace_bytes < rq_attention_workspace_size(batch, heads, head_dim, context))
    return RQ_ERR_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  AttnParams a{};
  a.q = q;
  a.kc = k;
  a.vc = v;
  a.kv_bs = (long long)context * heads * head_dim;
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
// writes the bf16x3 operand of the next tensor-core GEMM (parts nb rows apart).
__global__ void __launch_bounds__(32) dattn_batched_kernel(const float* dq, long long dq_bs,
                                                           const float* dk, const float* dv,
                                                           long long dkv_bs, int n_keys,
                                                           int hd, int DD, uint16_t* out,
                                                           long long out_bs, int nb) {
  const int b = blockIdx.x, h = blockIdx.y, lane = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const float* q = dq + (size_t)b * dq_bs + (size_t)h * hd;
  const float* K = dk + (size_t)b * dkv_bs + (size_t)h * hd;
  const float* Vv = dv + (size_t)b * dkv_bs + (size_t)h * hd;
  const float scale = 1.0f / sqrtf((float)hd);
  float sc[8];
  float mx = -__int_as_float(0x7f800000);
  for (int j = 0; j < n_keys; ++j) {
    float d = 0.f;
    for (int e = lane; e < hd; e += 32) d = fmaf(q[e], K[(size_t)j * DD + e], d);
    sc[j] = warp_sum(d) * scale;
    mx = fmaxf(mx, sc[j]);
  }
  float den = 0.f;
  for (int j = 0; j < n_keys; ++j) {
    sc[j] = expf(sc[j] - mx);
    den += sc[j];
  }
  for (int e = lane; e < hd; e += 32) {
    float o = 0.f;
    for (int j = 0; j < n_keys; ++j) o += sc[j] / den * Vv[(size_t)j * DD + e];
    store_bf16x3(out, (size_t)nb * out_bs, (size_t)b * out_bs + (size_t)h * hd + e, o);
  }
}

cudaError_t launch_dattn_batched(const float* dq, long long dq_bs, const float* dk,
                                 const float* dv, long long dkv_bs, int n_keys, int B,
                                 int heads, int hd, uint16_t* out, long long out_bs, int nb,
                                 cudaStream_t s, bool pdl) {
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
