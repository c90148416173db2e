// gemv_launch.cuh -- launch and configure helpers for the instantiated GEMV kernels.
#pragma once
#include "gemv_kernel.cuh"

namespace rqk {

template <typename WT, int PRO, int EPI, int NCH>
static cudaError_t gemv_launch_one(const GemvParams& p, int batch, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.pl.grid, (unsigned)batch, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)p.pl.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemv_kernel<WT, PRO, EPI, NCH>, p);
}

template <typename WT, int PRO, int EPI, int NCH>
static cudaError_t gemv_configure_one(int max_smem) {
  return cudaFuncSetAttribute(gemv_kernel<WT, PRO, EPI, NCH>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

// Every (prologue, epilogue) pair the decode step uses, for chunk counts 1 and 2;
// the long-reduction residual GEMV (K = hidden) also for 3, 4 and 6.
#define RQ_GEMV_PAIRS(X, NCH)                                               \
  X(PRO_RMS, EPI_QKV, NCH) X(PRO_PLAIN, EPI_RESID, NCH) X(PRO_RMS, EPI_SWIGLU, NCH) \
  X(PRO_RMS, EPI_ARGMAX, NCH) X(PRO_PLAIN, EPI_DEPIN, NCH) X(PRO_RMS, EPI_DQKV, NCH) \
  X(PRO_DATTN, EPI_RESID, NCH) X(PRO_PLAIN, EPI_ARGMAX, NCH) X(PRO_PLAIN, EPI_STORE, NCH)

template <typename WT>
cudaError_t gemv_dispatch(const GemvParams& p, int pro, int epi, int batch, cudaStream_t s,
                          bool pdl) {
  const int nch = p.pl.nch;
#define RQ_X(P, E, N) \
  if (pro == P && epi == E && nch == N) return gemv_launch_one<WT, P, E, N>(p, batch, s, pdl);
  RQ_GEMV_PAIRS(RQ_X, 1)
  RQ_GEMV_PAIRS(RQ_X, 2)
  RQ_X(PRO_PLAIN, EPI_RESID, 3)
  RQ_X(PRO_PLAIN, EPI_RESID, 4)
  RQ_X(PRO_PLAIN, EPI_RESID, 6)
#undef RQ_X
  return cudaErrorInvalidValue;
}

template <typename WT>
cudaError_t gemv_configure(int max_smem) {
  cudaError_t e = cudaSuccess, r;
#define RQ_X(P, E, N) \
  if ((r = gemv_configure_one<WT, P, E, N>(max_smem)) != cudaSuccess) e = r;
  RQ_GEMV_PAIRS(RQ_X, 1)
  RQ_GEMV_PAIRS(RQ_X, 2)
  RQ_X(PRO_PLAIN, EPI_RESID, 3)
  RQ_X(PRO_PLAIN, EPI_RESID, 4)
  RQ_X(PRO_PLAIN, EPI_RESID, 6)
#undef RQ_X
  return e;
}

}  // namespace rqk
