// prefill.cu -- the ring bookkeeping and embedding sums of T prompt steps of one session,
// ahead of the tensor-core temporal layers that run those T positions as one batch.
//
// "inferencelayer 0.2.4 -- src/moshi_lm.rs", `MoshiLm::step_forced` (the prompt-priming
// primitive: user codes written at their delays, the input gathered with INITIAL
// substitution and embedded, the temporal stack run, the ring recording the forced
// tokens) and `MoshiState::advance_clock` (the embedding replay: the clock moves, the
// ring is not touched).  The gathered inputs of step t depend only on the ring and the
// known forced / user codes of steps < t, never on model outputs, so all T steps'
// inputs are fixed before any layer runs.
#include "common.cuh"
#include "kernels.h"

namespace rqk {

namespace {

// One CTA: thread 0 walks the T steps of the ring in order; then the column positions
// and their rotary pairs.
__global__ void __launch_bounds__(128) prefill_ring_kernel(const PrefillParams p) {
  __shared__ int s_off0;
  const int tid = threadIdx.x, b = p.session;
  int32_t* ring = p.ring + (size_t)b * kStreams * kRing;
  if (tid == 0) {
    int off = p.offsets[b];
    s_off0 = off;
    if (p.forced != nullptr) {
      for (int t = 0; t < p.T; ++t) {
        const int32_t* user = p.user + (size_t)t * 8;
        for (int k = 0; k < 8; ++k) {
          const int s = 9 + k;
          ring[s * kRing + (off + stream_delay(s)) % kRing] = user[k];
        }
        for (int s = 0; s < kStreams; ++s) {
          const int d = stream_delay(s);
          p.tokens[(size_t)t * kStreams + s] =
              off <= d ? (s == 0 ? p.V : p.A) : ring[s * kRing + off % kRing];
        }
        ++off;
        for (int s = 0; s < 9; ++s) ring[s * kRing + off % kRing] = p.forced[(size_t)t * 9 + s];
      }
    }
    p.offsets[b] = s_off0 + p.T;
  }
  __syncthreads();
  const int half = p.head_dim / 2;
  for (int i = tid; i < p.T * half; i += blockDim.x) {
    const int t = i / half, j = i % half;
    const int pos = s_off0 + t;
    if (j == 0) p.pos[t] = pos;
    // "moshi_lm.rs", `rope_row`: freq_j = exp(-ln(theta) * 2j / hd), angle freq_j * pos
    const float freq = expf(-logf(p.rope_theta) * 2.0f * (float)j / (float)p.head_dim);
    const float ang = freq * (float)pos;
    p.rope[i] = make_float2(cosf(ang), sinf(ang));
  }
}

// Grid (ceil(D/256), T): the embedding sum of step t's gathered inputs, the 16 audio
// streams in order and then the text stream (`step_ext` step 3's order).
template <typename WT>
__global__ void __launch_bounds__(256) prefill_embed_kernel(const PrefillParams p) {
  const int t = blockIdx.y, col = blockIdx.x * 256 + threadIdx.x;
  if (col >= p.D) return;
  const int32_t* in = p.tokens + (size_t)t * kStreams;
  auto elem = [&](const void* table, size_t row) {
    if (sizeof(WT) == 2)
      return __uint_as_float(((uint32_t)static_cast<const uint16_t*>(table)[row * p.D + col]) << 16);
    return static_cast<const float*>(table)[row * p.D + col];
  };
  float acc = 0.f;
  for (int k = 0; k < 16; ++k) {
    const int tok = in[1 + k];
    if (tok == -1) continue;  // "moshi_lm.rs", `embed`: -1 adds nothing, else row max(tok, 0)
    acc += elem(p.emb, (size_t)k * (p.A + 1) + (size_t)(tok > 0 ? tok : 0));
  }
  const int tok = in[0];
  if (tok != -1) acc += elem(p.text_emb, (size_t)(tok > 0 ? tok : 0));
  p.x[(size_t)t * p.D + col] = acc;
}

}  // namespace

cudaError_t launch_prefill_begin(const PrefillParams& p, bool bf16, cudaStream_t s) {
  if (p.T < 1) return cudaErrorInvalidValue;
  prefill_ring_kernel<<<1, 128, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.forced == nullptr) return e;
  dim3 grid((unsigned)((p.D + 255) / 256), (unsigned)p.T);
  if (bf16)
    prefill_embed_kernel<uint16_t><<<grid, 256, 0, s>>>(p);
  else
    prefill_embed_kernel<float><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace rqk
