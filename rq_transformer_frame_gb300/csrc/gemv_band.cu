// gemv_band.cu -- the GEMV kernels for the q8 and q4 weight bands.
#include "gemv_launch.cuh"

namespace rqk {
template cudaError_t gemv_dispatch<q8_t>(const GemvParams&, int, int, int, cudaStream_t, bool);
template cudaError_t gemv_configure<q8_t>(int);
template cudaError_t gemv_dispatch<q4_t>(const GemvParams&, int, int, int, cudaStream_t, bool);
template cudaError_t gemv_configure<q4_t>(int);
}  // namespace rqk
