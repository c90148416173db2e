// frame_persistent.cu -- host side of the whole-frame cooperative kernel (batch 1): the
// instantiations with token picks, the launch dispatch and the tile plans.  The greedy
// instantiations are compiled in frame_persistent_greedy.cu.
#include "frame_persistent.cuh"

namespace rqk {
namespace pers {
RQ_PERS_ALL(RQ_PERS_EXTERN, false)
RQ_PERS_ALL(RQ_PERS_INSTANTIATE, true)
}  // namespace pers

#define RQ_PERS_DISPATCH(CALL)                                                  \
  switch (hd) {                                                                 \
    case 32: return bf16 ? CALL(uint16_t, uint16_t, 1) : CALL(float, float, 1); \
    case 64: return bf16 ? CALL(uint16_t, uint16_t, 2) : CALL(float, float, 2); \
    default: return bf16 ? CALL(uint16_t, uint16_t, 4) : CALL(float, float, 4); \
  }

// frames with token picks run the kernel with the pick ops, greedy frames the smaller one
cudaError_t launch_persistent(const PersParams& p, bool bf16, bool kv_bf16, int grid, int smem,
                              cudaStream_t s, bool pdl) {
  if (bf16 != kv_bf16) return cudaErrorInvalidValue;
  const int hd = p.head_dim;
  if (p.samp.mode != SAMPLE_GREEDY) {
#define RQ_L(W, K, E) pers::launch_t<W, K, E, true>(p, grid, smem, s, pdl)
    RQ_PERS_DISPATCH(RQ_L)
#undef RQ_L
  }
#define RQ_L(W, K, E) pers::launch_t<W, K, E, false>(p, grid, smem, s, pdl)
  RQ_PERS_DISPATCH(RQ_L)
#undef RQ_L
}

// the smaller of the two variants' co-resident grids
int persistent_max_grid(bool bf16, bool kv_bf16, int smem, int hd) {
  if (bf16 != kv_bf16) return 0;
  int a = 0, b = 0;
  {
    auto f = [&]() -> int {
#define RQ_M(W, K, E) pers::max_grid_t<W, K, E, true>(smem)
      RQ_PERS_DISPATCH(RQ_M)
#undef RQ_M
    };
    a = f();
  }
  {
    auto f = [&]() -> int {
#define RQ_M(W, K, E) pers::max_grid_t<W, K, E, false>(smem)
      RQ_PERS_DISPATCH(RQ_M)
#undef RQ_M
    };
    b = f();
  }
  return a < b ? a : b;
}

cudaError_t persistent_configure(bool bf16, bool kv_bf16, int smem, int hd) {
  if (bf16 != kv_bf16) return cudaErrorInvalidValue;
  cudaError_t e;
  {
    auto f = [&]() -> cudaError_t {
#define RQ_C(W, K, E) pers::configure_t<W, K, E, true>(smem)
      RQ_PERS_DISPATCH(RQ_C)
#undef RQ_C
    };
    if ((e = f()) != cudaSuccess) return e;
  }
  auto f = [&]() -> cudaError_t {
#define RQ_C(W, K, E) pers::configure_t<W, K, E, false>(smem)
    RQ_PERS_DISPATCH(RQ_C)
#undef RQ_C
  };
  return f();
}

GemvPlan plan_persistent(int n_out, int K, int es, bool paired, bool even_rows, int grid) {
  GemvPlan pl = plan_gemv(n_out, K, es, paired, even_rows, 1 << 24);
  const int V = 16 / es, CC = K / V;
  const int need = (CC + pl.tpr - 1) / pl.tpr;  // chunks per thread over the whole row
  if (need > 2 && !paired) {
    // parts of at most 2 chunks per thread; widths are multiples of 8 columns
    pl.kparts = (need + 1) / 2;
    int w = (K + pl.kparts - 1) / pl.kparts;
    w = (w + 7) & ~7;
    pl.kp_width = w;
    pl.nch = 2;
    pl.rg = 2;
    pl.tile_rows = (kGemvConsumers / pl.tpr) * 2;
    pl.tiles = (n_out + pl.tile_rows - 1) / pl.tile_rows;
    if ((K - (pl.kparts - 1) * w) <= 0 || (w / V + pl.tpr - 1) / pl.tpr > 2) pl.nch = 0;
  }
  pl.grid = grid;
  pl.max_tiles = (pl.tiles + grid - 1) / grid;
  pl.n_stages = 0;
  pl.smem = 0;
  return pl;
}

}  // namespace rqk
