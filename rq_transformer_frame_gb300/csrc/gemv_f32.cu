// gemv_f32.cu -- the GEMV kernels for f32 weights.
#include "gemv_launch.cuh"

namespace rqk {
template cudaError_t gemv_dispatch<float>(const GemvParams&, int, int, int, cudaStream_t, bool);
template cudaError_t gemv_configure<float>(int);
}  // namespace rqk
