// frame_persistent.cu -- host side of the whole-frame cooperative kernel (batch 1): the
// instantiations with token picks, the launch dispatch and the tile plans.  The greedy
// instantiations are compiled in frame_persistent_greedy.cu.
#include "frame_persistent.cuh"

namespace rqk {
namespace pers {
RQ_PERS_ALL(RQ_PERS_EXTERN, false)
RQ_PERS_BANDS(RQ_PERS_EXTERN, false)
RQ_PERS_BANDS(RQ_PERS_EXTERN, true)
RQ_PERS_DEP(RQ_PERS_EXTERN, false)
RQ_PERS_DEP(RQ_PERS_EXTERN, true)
RQ_PERS_ALL(RQ_PERS_INSTANTIATE, true)
}  // namespace pers

// The instantiation of a launch: weight type (0 f32, 1 bf16 -- the K/V cache of the same
// type -- or a weight band with bf16 K/V), the temporal head_dim (bands: 64 and 128), and
// CTAs per SM (MB 1: the depformer launch, one head-size variant).
#define RQ_PERS_DISPATCH(CALL, MB)                                                          \
  if (MB == 1) {                                                                            \
    if (wtype == BAND_Q8) return CALL(q8_t, uint16_t, 1, 1);                                \
    if (wtype == BAND_Q4) return CALL(q4_t, uint16_t, 1, 1);                                \
    return wtype == 1 ? CALL(uint16_t, uint16_t, 1, 1) : CALL(float, float, 1, 1);          \
  }                                                                                         \
  if (wtype == BAND_Q8 || wtype == BAND_Q4) {                                               \
    if (hd != 64 && hd != 128) return RQ_PERS_BAD;                                          \
    if (wtype == BAND_Q8)                                                                   \
      return hd == 64 ? CALL(q8_t, uint16_t, 2, 2) : CALL(q8_t, uint16_t, 4, 2);            \
    return hd == 64 ? CALL(q4_t, uint16_t, 2, 2) : CALL(q4_t, uint16_t, 4, 2);              \
  }                                                                                         \
  switch (hd) {                                                                             \
    case 32: return wtype == 1 ? CALL(uint16_t, uint16_t, 1, 2) : CALL(float, float, 1, 2);  \
    case 64: return wtype == 1 ? CALL(uint16_t, uint16_t, 2, 2) : CALL(float, float, 2, 2);  \
    default: return wtype == 1 ? CALL(uint16_t, uint16_t, 4, 2) : CALL(float, float, 4, 2);  \
  }

// weight / K/V types the persistent kernel takes: f32 / f32, bf16 / bf16, band / bf16
static bool types_ok(int wtype, bool kv_bf16) {
  if (wtype == BAND_Q8 || wtype == BAND_Q4) return kv_bf16;
  return (wtype == 1) == kv_bf16 && (wtype == 0 || wtype == 1);
}

// frames with token picks run the kernel with the pick ops, greedy frames the smaller one
cudaError_t launch_persistent(const PersParams& p, int wtype, bool kv_bf16, int grid, int smem,
                              cudaStream_t s, bool pdl, int minb) {
  if (!types_ok(wtype, kv_bf16) || (minb != 1 && minb != 2)) return cudaErrorInvalidValue;
  const int hd = p.head_dim;
#define RQ_PERS_BAD cudaErrorInvalidValue
  if (p.samp.mode != SAMPLE_GREEDY) {
#define RQ_L(W, K, E, MB) pers::launch_t<W, K, E, true, MB>(p, grid, smem, s, pdl)
    RQ_PERS_DISPATCH(RQ_L, minb)
#undef RQ_L
  }
#define RQ_L(W, K, E, MB) pers::launch_t<W, K, E, false, MB>(p, grid, smem, s, pdl)
  RQ_PERS_DISPATCH(RQ_L, minb)
#undef RQ_L
#undef RQ_PERS_BAD
}

// the smaller of the two variants' co-resident grids
int persistent_max_grid(int wtype, bool kv_bf16, int smem, int hd, int minb) {
  if (!types_ok(wtype, kv_bf16) || (minb != 1 && minb != 2)) return 0;
#define RQ_PERS_BAD 0
  auto a = [&]() -> int {
#define RQ_M(W, K, E, MB) pers::max_grid_t<W, K, E, true, MB>(smem)
    RQ_PERS_DISPATCH(RQ_M, minb)
#undef RQ_M
  };
  auto b = [&]() -> int {
#define RQ_M(W, K, E, MB) pers::max_grid_t<W, K, E, false, MB>(smem)
    RQ_PERS_DISPATCH(RQ_M, minb)
#undef RQ_M
  };
#undef RQ_PERS_BAD
  const int x = a(), y = b();
  return x < y ? x : y;
}

cudaError_t persistent_configure(int wtype, bool kv_bf16, int smem, int hd, int minb) {
  if (!types_ok(wtype, kv_bf16) || (minb != 1 && minb != 2)) return cudaErrorInvalidValue;
#define RQ_PERS_BAD cudaErrorInvalidValue
  auto a = [&]() -> cudaError_t {
#define RQ_C(W, K, E, MB) pers::configure_t<W, K, E, true, MB>(smem)
    RQ_PERS_DISPATCH(RQ_C, minb)
#undef RQ_C
  };
  auto b = [&]() -> cudaError_t {
#define RQ_C(W, K, E, MB) pers::configure_t<W, K, E, false, MB>(smem)
    RQ_PERS_DISPATCH(RQ_C, minb)
#undef RQ_C
  };
#undef RQ_PERS_BAD
  cudaError_t e = a();
  return e != cudaSuccess ? e : b();
}

// Weight bands: a part of a row is at most 256 chunks (one per consumer thread, so x
// stays one chunk of 16 q8 / 32 q4 values per thread) and a multiple of 128 columns (its
// codes and its groups' scales start on 16-byte boundaries).
static GemvPlan plan_persistent_band(int n_out, int K, int band, bool paired, int grid) {
  GemvPlan pl{};
  pl.n_out = n_out;
  pl.K = K;
  const int V = band == BAND_Q8 ? 16 : 32;
  int parts = (K / V + kGemvConsumers - 1) / kGemvConsumers;
  int w = K;
  if (parts > 1) {
    w = ((K + parts - 1) / parts + 127) & ~127;
    parts = (K + w - 1) / w;
  }
  int tpr = 32;
  while (tpr < w / V && tpr < kGemvConsumers) tpr <<= 1;
  pl.tpr = tpr;
  pl.nch = (w / V <= tpr && (K % 128) == 0) ? 1 : 0;
  pl.rg = 2;
  pl.tile_rows = (kGemvConsumers / tpr) * 2;
  const int per = paired ? pl.tile_rows / 2 : pl.tile_rows;
  pl.tiles = (n_out + per - 1) / per;
  pl.kparts = parts;
  pl.kp_width = w;
  pl.grid = grid;
  pl.max_tiles = (pl.tiles + grid - 1) / grid;
  pl.bytes = (double)n_out * (paired ? 2.0 : 1.0) * (double)band_row_bytes(band, 1, K);
  return pl;
}

GemvPlan plan_persistent(int n_out, int K, int es, bool paired, bool even_rows, int grid,
                         int band) {
  if (band != BAND_NONE) return plan_persistent_band(n_out, K, band, paired, grid);
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
