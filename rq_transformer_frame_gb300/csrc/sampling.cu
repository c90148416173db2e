// sampling.cu -- host side of the token picks and the standalone top-k pick kernel.
#include "sampling.cuh"

namespace rqk {

namespace {

// "moshi_lm.rs", `xorshift_u01`: one step of the generator (shifts 13, 7, 17)
uint64_t xs_step(uint64_t x) {
  x ^= x << 13;
  x ^= x >> 7;
  x ^= x << 17;
  return x;
}

// M y for the matrix given by its columns
uint64_t apply(const uint64_t* col, uint64_t y) {
  uint64_t r = 0;
  for (int b = 0; b < 64; ++b)
    if ((y >> b) & 1ull) r ^= col[b];
  return r;
}

__global__ void __launch_bounds__(256) topk_pick_kernel(const SampleParams sp, const float* logits,
                                                        long long ld, int n, int p,
                                                        unsigned long long* keys) {
  __shared__ TopkShared S;
  const int b = blockIdx.x;
  pdl_wait();
  const float* lg = logits + (size_t)b * ld;
  // top-k draws once per pick: draw draws_before + 1 of the frame
  const double u = xs_u01(xs_advance(sp.rng[b], draws_before(sp, p) + 1u, sp.jump));
  const int k = p == 0 ? sp.top_k_text : sp.top_k;
  const float temp = p == 0 ? sp.temp_text : sp.temp;
  const int tok = topk_pick_block(lg, n, k, temp, u, (int)threadIdx.x, 256, S, SyncBlock{});
  if (threadIdx.x == 0) keys[(size_t)b * 9 + p] = argmax_key(__ldcg(lg + tok), (uint32_t)tok);
  pdl_trigger();
}

}  // namespace

void xorshift_jump_table(uint64_t* table) {
  // level 0: column b of M is the step applied to the unit vector e_b (linearity)
  for (int b = 0; b < 64; ++b) table[b] = xs_step(1ull << b);
  // level k + 1: M^(2^(k+1)) e_b = M^(2^k) (M^(2^k) e_b)
  for (int k = 0; k + 1 < kXsLevels; ++k) {
    const uint64_t* cur = table + (size_t)k * 64;
    uint64_t* nxt = table + (size_t)(k + 1) * 64;
    for (int b = 0; b < 64; ++b) nxt[b] = apply(cur, cur[b]);
  }
}

long long frame_draws(const SampleParams& sp) {
  if (sp.mode == SAMPLE_GUMBEL) return (long long)sp.V + 8ll * sp.A;
  if (sp.mode == SAMPLE_TOPK) return 9;
  return 0;
}

cudaError_t launch_topk_pick(const SampleParams& sp, const float* logits, long long ld, int n,
                             int p, unsigned long long* keys, int B, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, topk_pick_kernel, sp, logits, ld, n, p, keys);
}

}  // namespace rqk
