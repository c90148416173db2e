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
// host it is only a stand-in), so the device address is looked up with
// cudaGetSymbolAddress while the device is current, and that pointer is what the
// kernel receives.  The address belongs to the CUDA context the library's module was
// loaded into: it is cached per device together with that context's unique id and
// looked up again whenever the current context is another one (after cudaDeviceReset,
// or under a caller's own driver-API context), so a stale address is never used.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/rq.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = 4u << 20;  // 4 MiB: partials + tickets
constexpr int kKps = rqk::kStandaloneAttnKps;  // positions per split, as rq_attention
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CachedAddr {
  unsigned long long ctx_id;  // unique id of the context the address belongs to
  void* addr;
};

std::mutex g_mu;
CachedAddr g_scratch[kMaxDevices] = {};
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

template <typename Fn>
bool driver_fn(const char* name, int version, Fn* out) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !f)
    return false;
  *out = reinterpret_cast<Fn>(f);
  return true;
}

// unique id of the calling thread's current context (0 if there is none yet)
cudaError_t current_ctx_id(unsigned long long* id) {
  *id = 0;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  if (!ctx) return cudaSuccess;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

// Device address of g_attn_scratch for the current device and context: looked up with
// cudaGetSymbolAddress on first use and whenever the current context has changed.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ctx_current && (!driver_fn("cuCtxGetCurrent", 4000, &g_ctx_current) ||
                         !driver_fn("cuCtxGetId", 12000, &g_ctx_id))) {
    g_ctx_current = nullptr;
    return cudaErrorNotSupported;
  }
  unsigned long long id = 0;
  if ((e = current_ctx_id(&id)) != cudaSuccess) return e;
  if (id == 0 || id != g_scratch[dev].ctx_id || !g_scratch[dev].addr) {
    void* p = nullptr;
    // makes the device's primary context current if the thread has none yet
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess) return e;
    if ((e = current_ctx_id(&id)) != cudaSuccess) return e;
    if (id == 0) return cudaErrorDeviceUninitialized;
    g_scratch[dev] = CachedAddr{id, p};
  }
  *out = g_scratch[dev].addr;
  return cudaSuccess;
}

size_t partial_bytes(int B, int H, int hd, int C) {
  return rqk::standalone_attn_partial_bytes(B, H, hd, C);
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
