// quantize.cu -- rows of f32 or bf16 values into the q8 / q4 weight bands.
//
// "inferencelayer 0.2.4 -- src/moshi_lm.rs", `qn_roundtrip` and the Q4_0 layout noted at
// `q4_roundtrip`: per 32 consecutive values of a row, mx = the first value of the largest
// magnitude, d = mx / -(2^(bits-1)), id = 1/d (0 when d is 0), q = clamp(round(x * id))
// with round halving away from zero; the codes and d are stored (kernels.h, weight bands).
#include "common.cuh"
#include "kernels.h"

namespace rqk {

namespace {

// one warp per group, lane i holding value i of the group
__global__ void __launch_bounds__(256) quantize_band_kernel(int band, const void* src,
                                                            int src_bf16, long long rows,
                                                            int cols, uint8_t* dst) {
  const int lane = threadIdx.x & 31;
  const long long ng = (long long)cols / 32, total = rows * ng;
  const long long g = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (g >= total) return;  // whole warps leave together
  const long long r = g / ng;
  const int blk = (int)(g % ng);
  const size_t idx = (size_t)r * cols + (size_t)blk * 32 + lane;
  const float x = src_bf16
      ? __uint_as_float((uint32_t)static_cast<const uint16_t*>(src)[idx] << 16)
      : static_cast<const float*>(src)[idx];
  // the first value of the largest magnitude: |x| bits (NaN counts as 0), ties to the
  // lowest lane
  const float ax = fabsf(x);
  const uint32_t mag = (ax == ax) ? __float_as_uint(ax) : 0u;
  unsigned long long key = ((unsigned long long)mag << 32) | (uint32_t)(31 - lane);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long k2 = __shfl_xor_sync(0xffffffffu, key, o);
    key = k2 > key ? k2 : key;
  }
  const int winner = 31 - (int)(key & 0xffffffffu);
  const float mx = __shfl_sync(0xffffffffu, x, winner);
  const int bits = band == BAND_Q8 ? 8 : 4;
  const int qmin = -(1 << (bits - 1)), qmax = (1 << (bits - 1)) - 1;
  const float d = (key >> 32) == 0ull ? 0.f : mx / (float)qmin;
  const float id = d != 0.f ? 1.0f / d : 0.f;
  int q = (int)roundf(x * id);
  q = q < qmin ? qmin : (q > qmax ? qmax : q);
  const size_t row_bytes = band_row_bytes(band, 1, cols);
  uint8_t* row = dst + (size_t)r * row_bytes;
  const int hi = __shfl_down_sync(0xffffffffu, q, 16);  // lanes 0-15: value i + 16
  if (band == BAND_Q8) {
    row[(size_t)blk * 32 + lane] = (uint8_t)(int8_t)q;
  } else if (lane < 16) {
    row[(size_t)blk * 16 + lane] = (uint8_t)((q + 8) | ((hi + 8) << 4));
  }
  if (lane == 0) {
    const size_t codes = band == BAND_Q8 ? (size_t)cols : (size_t)cols / 2;
    *reinterpret_cast<float*>(row + codes + (size_t)blk * 4) = d;
  }
}

}  // namespace

cudaError_t launch_quantize_band(int band, const void* src, bool src_bf16, long long rows,
                                 int cols, void* dst, cudaStream_t s) {
  if ((band != BAND_Q8 && band != BAND_Q4) || cols <= 0 || cols % 32 != 0 || rows < 0)
    return cudaErrorInvalidValue;
  const long long groups = rows * (cols / 32);
  if (groups == 0) return cudaSuccess;
  const long long blocks = (groups * 32 + 255) / 256;
  quantize_band_kernel<<<(unsigned)blocks, 256, 0, s>>>(band, src, src_bf16 ? 1 : 0, rows, cols,
                                                        static_cast<uint8_t*>(dst));
  return cudaGetLastError();
}

}  // namespace rqk
