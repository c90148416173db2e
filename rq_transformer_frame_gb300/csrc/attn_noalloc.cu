// attn_noalloc.cu -- decode attention for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: a real-time audio thread, where an allocation
// can stall behind device-wide synchronization for an unbounded time and break the
// 80 ms frame deadline, and plug-in hosts that hand a component a fixed device-memory
// budget at start-up and forbid allocation afterwards.  rq_attention needs a scratch
// workspace from its caller; rq_attention_noalloc runs the same kernel with its scratch
// in a fixed array that lives in this library's device image instead.
//
// The array (kScratchBytes, 4 MiB) exists on every GPU that loads the library, until
// the process exits.  Host code cannot use the array's name as a device address (on the
// host it is only a stand-in), so the device address is looked up once per device with
// cudaGetSymbolAddress while that device is current, and that pointer is what the
// kernel receives.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/rq.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = 4u << 20;  // 4 MiB: partials + tickets
constexpr int kKps = 64;                     // positions per split, as in the frame
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device (looked up on first use).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t partial_bytes(int B, int H, int hd, int C) {
  const size_t nsplit = (size_t)(C + kKps - 1) / kKps;
  return ((size_t)B * H * nsplit * (hd + 2) * sizeof(float) + 255) & ~(size_t)255;
}

}  // namespace

extern "C" rq_status rq_attention_noalloc(int32_t batch, int32_t heads, int32_t head_dim,
                                          int32_t context, int32_t kv_dtype, const float* q,
                                          const void* k, const void* v,
                                          const int32_t* positions, float* out,
                                          void* cuda_stream) {
  using namespace rqk;
  if (batch < 1 || heads < 1 || context < 1 || batch > 65535 || heads > 65535)
    return RQ_ERR_ARG;
  if (head_dim != 32 && head_dim != 64 && head_dim != 128) return RQ_ERR_UNSUPPORTED;
  if (kv_dtype != RQ_F32 && kv_dtype != RQ_BF16) return RQ_ERR_ARG;
  if (!q || !k || !v || !positions || !out) return RQ_ERR_ARG;
  // the K/V rows are bulk-copied into shared memory: 16-byte aligned sources
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u) return RQ_ERR_ARG;
  const size_t part = partial_bytes(batch, heads, head_dim, context);
  const size_t need = part + (size_t)batch * heads * sizeof(int);
  if (need > kScratchBytes) return RQ_ERR_UNSUPPORTED;  // beyond the fixed scratch
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return RQ_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  AttnParams a{};
  a.q = q;
  a.kbase = k;
  a.vbase = v;
  a.rows = (long long)batch * context;
  a.row0 = 0;
  a.row_bs = context;
  a.offsets = positions;
  a.part = static_cast<float*>(scratch);
  a.counters = reinterpret_cast<int*>(static_cast<char*>(scratch) + part);
  a.out = out;
  a.D = heads * head_dim;
  a.H = heads;
  a.hd = head_dim;
  a.C = context;
  a.kps = kKps;
  a.nsplit = (context + kKps - 1) / kKps;
  a.batch = batch;
  a.status = nullptr;
  // the merge tickets must start at zero; the partials are always written before read
  if (cudaMemsetAsync(a.counters, 0, (size_t)batch * heads * sizeof(int), s) != cudaSuccess)
    return RQ_ERR_CUDA;
  return launch_attn(a, kv_dtype == RQ_BF16, s, false) == cudaSuccess ? RQ_OK : RQ_ERR_CUDA;
}
