// common.cuh -- device helpers shared by the kernels of the decode step (sm_103a).
//
// Inline PTX for the Blackwell data path: mbarrier-tracked bulk copies
// (cp.async.bulk global -> shared, completion by transaction bytes), programmatic
// dependent launch (griddepcontrol), an L2 evict-first policy for weights that are
// streamed exactly once per frame, and bounded waits that report a timeout instead
// of spinning forever.
#pragma once

#include <cuda_bf16.h>

#include "kernels.h"
#include <cuda_runtime.h>
#include <stdint.h>

namespace rqk {

// ---------------------------------------------------------------- model constants
// "inferencelayer 0.2.4 -- src/moshi_lm.rs", consts N_STREAMS, DEP_Q, DELAYS,
// MAX_DELAY, CT, UNGENERATED.
constexpr int kStreams = 17;
constexpr int kQ = 8;
constexpr int kRing = 3;
constexpr int kMaxDelay = 1;
constexpr int kUngenerated = -2;

// delay of stream s: text 0, generated audio [0,1x7], user audio [0,1x7]
__host__ __device__ __forceinline__ int stream_delay(int s) {
  return (s == 0 || s == 1 || s == 9) ? 0 : 1;
}

// ---------------------------------------------------------------- per-step io layout
// d_in (int32 words): user [B][8] | forced [B][9] | force flag [B]
// d_out (bytes):      own [B][9] int32 | out [B][9] int32 | has [B] uint8 (padded
//                     to 4) | status uint32
struct IoLayout {
  int B;
  __host__ __device__ size_t user_off() const { return 0; }
  __host__ __device__ size_t forced_off() const { return (size_t)B * 8; }
  __host__ __device__ size_t flag_off() const { return (size_t)B * 17; }
  __host__ __device__ size_t in_words() const { return (size_t)B * 18; }
  __host__ __device__ size_t own_off() const { return 0; }  // int32 words
  __host__ __device__ size_t out_off() const { return (size_t)B * 9; }
  __host__ __device__ size_t has_off_bytes() const { return (size_t)B * 18 * 4; }
  __host__ __device__ size_t status_off_bytes() const {
    return has_off_bytes() + (((size_t)B + 3) / 4) * 4;
  }
  __host__ __device__ size_t out_bytes() const { return status_off_bytes() + 4; }
};

// status bits written by kernels (the host maps them to rq_status)
enum : uint32_t { kDevTimeout = 1u, kDevBadInput = 2u };

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// non-blocking test of the same condition (the fast path when the phase is complete)
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every wait in these kernels is bounded: after kWaitLimitNs of wall time it
// returns false and the caller records kDevTimeout and winds down.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ bool mbar_wait_for(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  return mbar_wait_for(bar, parity, kWaitLimitNs);
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk copy global -> this CTA's shared memory; completes `bytes` on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// programmatic dependent launch
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// named barrier over the first `n` threads of the CTA (n a multiple of 32)
__device__ __forceinline__ void bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// bar.sync of n threads that also returns whether any of them passed `pred` true: the
// same answer in every thread, so a decision taken on it (leave a loop) stays uniform
// even while another warp may still change the flag behind `pred`
__device__ __forceinline__ bool bar_or(int id, int n, bool pred) {
  unsigned r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((unsigned)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0u;
}

// ---------------------------------------------------------------- numerics
// bf16 expansion of an f32 for the tensor-core operand: hi = bf16(x), mid = bf16(x - hi)
// (x - hi is exact), and with kOpndParts == 3 also lo = bf16(x - hi - mid).  Two parts keep
// 16 significant bits (relative representation error <= 2^-17); three parts are exact
// for every normal-range x (lo needs at most 8 significant bits).  A bf16 x bf16
// tensor-core product over the parts, accumulated in f32, sees hi + mid (+ lo).  Parts
// go to base[idx], base[ps + idx] (and base[2 ps + idx]).
__device__ __forceinline__ void store_bf16_parts(uint16_t* base, size_t ps, size_t idx, float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h);
  const __nv_bfloat16 m = __float2bfloat16_rn(r1);
  base[idx] = __bfloat16_as_ushort(h);
  base[ps + idx] = __bfloat16_as_ushort(m);
  if (kOpndParts == 3) {
    const float r2 = r1 - __bfloat162float(m);
    base[2 * ps + idx] = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
  }
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// First-wins argmax as a single 64-bit maximum ("moshi_lm.rs", `argmax`: strict '>'
// from (-inf, 0)).  High word: the value mapped to an unsigned order (NaN counts as
// -inf, -0 as +0); low word: ~index, so equal values prefer the smaller index.
// Every real key is > 0, the reset value.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  if (!(v == v)) v = -__int_as_float(0x7f800000);
  if (v == 0.0f) v = 0.0f;
  const uint32_t u = __float_as_uint(v);
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)o << 32) | (unsigned long long)(0xffffffffu - idx);
}

__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
  return (int)(0xffffffffu - (uint32_t)(k & 0xffffffffull));
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

}  // namespace rqk
