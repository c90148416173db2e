// gemv_bf16.cu -- the GEMV kernels for bf16 weights (one translation unit per dtype
// so the two sets compile in parallel).
#include "gemv_launch.cuh"

namespace rqk {
template cudaError_t gemv_dispatch<uint16_t>(const GemvParams&, int, int, int, cudaStream_t, bool);
template cudaError_t gemv_configure<uint16_t>(int);
}  // namespace rqk
