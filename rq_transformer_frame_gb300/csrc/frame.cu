// frame.cu -- the device-side ring cache: frame prologue (user write, gather with
// INITIAL substitution, summed embeddings) and frame epilogue (advance, self-feed,
// delay-realigned output), plus session reset.
//
// "inferencelayer 0.2.4 -- src/moshi_lm.rs", module doc "streams and delays" and
// `step_ext` steps 1-3 and 7-8; `embed` (ScaledEmbedding).
#include "common.cuh"
#include "kernels.h"
#include "sampling.cuh"

namespace rqk {

// Grid (ceil(D/256), B).  Every CTA gathers the 17 inputs itself from the ring as it
// was before this frame's user write: a user stream with delay 0 is read from the
// slot this frame writes, so it takes the user code directly; every other stream
// reads a slot nobody writes in this kernel.  CTA x == 0 performs the user write and
// clears the 9 argmax keys of the session.
template <typename WT>
__global__ void __launch_bounds__(256) frame_begin_kernel(const FrameParams p) {
  __shared__ int s_in[kStreams];
  const int b = blockIdx.y, tid = threadIdx.x;
  const IoLayout io{p.B};
  const int32_t* user = p.d_in + io.user_off() + (size_t)b * 8;
  const int off = p.offsets[b];
  int32_t* ring = p.ring + (size_t)b * kStreams * kRing;
  if (tid < kStreams) {
    const int s = tid, d = stream_delay(s);
    int tok;
    if (off <= d)
      tok = (s == 0) ? p.V : p.A;  // INITIAL while offset <= delay
    else if (s >= 9 && d == 0)
      tok = user[s - 9];           // written this frame at the slot read this frame
    else
      tok = ring[s * kRing + off % kRing];
    s_in[s] = tok;
  }
  if (blockIdx.x == 0) {
    if (tid < 8) {
      const int s = 9 + tid;
      ring[s * kRing + (off + stream_delay(s)) % kRing] = user[tid];
    }
    if (tid < 9) p.keys[(size_t)b * 9 + tid] = 0ull;
    if (tid == 0 && b == 0 && p.grid_bar) {
      p.grid_bar[0] = 0u;                // the temporal launch's grid barrier
      p.grid_bar[kPersDepBarWord] = 0u;  // the depformer launch's
    }
    if (p.rope && tid < p.head_dim / 2) {
      // "moshi_lm.rs", `rope_row`: freq_i = exp(-ln(theta) * 2i / hd), angle freq_i * pos
      const float freq = expf(-logf(p.rope_theta) * 2.0f * (float)tid / (float)p.head_dim);
      const float ang = freq * (float)off;
      p.rope[(size_t)b * (p.head_dim / 2) + tid] = make_float2(cosf(ang), sinf(ang));
    }
  }
  __syncthreads();
  pdl_trigger();
  const int col = blockIdx.x * 256 + tid;
  if (col >= p.D) return;
  const WT* emb = static_cast<const WT*>(p.emb);
  const WT* temb = static_cast<const WT*>(p.text_emb);
  float acc = 0.f;
  // audio streams 1..16 use tables 0..15 in order, then the text stream
  for (int k = 0; k < 16; ++k) {
    const int tok = s_in[1 + k];
    if (tok == -1) continue;
    const size_t row = (size_t)k * (p.A + 1) + (size_t)(tok > 0 ? tok : 0);
    if (sizeof(WT) == 2)
      acc += __uint_as_float(((uint32_t)reinterpret_cast<const uint16_t*>(emb)[row * p.D + col]) << 16);
    else
      acc += reinterpret_cast<const float*>(emb)[row * p.D + col];
  }
  {
    const int tok = s_in[0];
    if (tok != -1) {
      const size_t row = (size_t)(tok > 0 ? tok : 0);
      if (sizeof(WT) == 2)
        acc += __uint_as_float(((uint32_t)reinterpret_cast<const uint16_t*>(temb)[row * p.D + col]) << 16);
      else
        acc += reinterpret_cast<const float*>(temb)[row * p.D + col];
    }
  }
  p.x[(size_t)b * p.D + col] = acc;
  p.emb_sum[(size_t)b * p.D + col] = acc;
}

// One warp per session: decode the 9 argmax keys, advance the offset, write the
// generated (or forced) tokens at offset % 3 and read the realigned output at
// (offset - 1 + delay) % 3.
__global__ void __launch_bounds__(32) frame_end_kernel(const FrameParams p) {
  const int b = blockIdx.x, lane = threadIdx.x;
  pdl_wait();
  pdl_trigger();
  const IoLayout io{p.B};
  const int forcing = p.d_in[io.flag_off() + b];
  const int off1 = p.offsets[b] + 1;
  int32_t* ring = p.ring + (size_t)b * kStreams * kRing;
  int own = 0;
  if (lane < 9) {
    own = argmax_key_index(p.keys[(size_t)b * 9 + lane]);
    const int gen = forcing ? p.d_in[io.forced_off() + (size_t)b * 9 + lane] : own;
    ring[lane * kRing + off1 % kRing] = gen;
  }
  __syncwarp();
  if (lane < 9) {
    const int out = ring[lane * kRing + (off1 - kMaxDelay + stream_delay(lane)) % kRing];
    p.d_out[io.own_off() + (size_t)b * 9 + lane] = own;
    p.d_out[io.out_off() + (size_t)b * 9 + lane] = out;
  }
  __syncwarp();
  if (lane == 0) {
    p.d_has[b] = off1 > kMaxDelay ? 1 : 0;
    p.offsets[b] = off1;
    // the sampler moves past this frame's draws (one per logit of every Gumbel-max
    // pick, one per top-k pick)
    const SampleParams& sp = p.samp;
    if (sp.mode != SAMPLE_GREEDY) {
      const uint32_t draws =
          sp.mode == SAMPLE_GUMBEL ? (uint32_t)sp.V + 8u * (uint32_t)sp.A : 9u;
      sp.rng[b] = xs_advance(sp.rng[b], draws, sp.jump);
    }
  }
}

__global__ void reset_kernel(int32_t* ring, int32_t* offsets, int B, int session) {
  const int b = blockIdx.x;
  if (session >= 0 && b != session) return;
  for (int i = threadIdx.x; i < kStreams * kRing; i += blockDim.x)
    ring[(size_t)b * kStreams * kRing + i] = kUngenerated;
  if (threadIdx.x == 0) offsets[b] = 0;
}

__global__ void set_offset_kernel(int32_t* offsets, int session, int value) {
  offsets[session] = value;
}

cudaError_t launch_frame_begin(const FrameParams& p, bool bf16, cudaStream_t s) {
  dim3 grid((unsigned)((p.D + 255) / 256), (unsigned)p.B);
  if (bf16)
    frame_begin_kernel<uint16_t><<<grid, 256, 0, s>>>(p);
  else
    frame_begin_kernel<float><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_frame_end(const FrameParams& p, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.B, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, frame_end_kernel, p);
}

cudaError_t launch_reset(int32_t* ring, int32_t* offsets, int B, int session, cudaStream_t s) {
  reset_kernel<<<B, 64, 0, s>>>(ring, offsets, B, session);
  return cudaGetLastError();
}

cudaError_t launch_set_offset(int32_t* offsets, int session, int value, cudaStream_t s) {
  set_offset_kernel<<<1, 1, 0, s>>>(offsets, session, value);
  return cudaGetLastError();
}

}  // namespace rqk
