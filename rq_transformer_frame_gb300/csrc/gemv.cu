// gemv.cu -- host side of the streaming GEMV: tile plan and dispatch to the kernel
// instantiations compiled in gemv_bf16.cu / gemv_f32.cu / gemv_band.cu.
#include "kernels.h"

#ifndef RQ_GEMV_STAGE_BUDGET
#define RQ_GEMV_STAGE_BUDGET (48 * 1024)  // shared-memory bytes of one CTA's weight ring
#endif
#ifndef RQ_GEMV_MAX_STAGES
#define RQ_GEMV_MAX_STAGES 8
#endif
#ifndef RQ_BAND_STAGE_BYTES
#define RQ_BAND_STAGE_BYTES (24 * 1024)  // largest band stage (tile) built from rounds
#endif
#ifndef RQ_BAND_STAGE_BUDGET
#define RQ_BAND_STAGE_BUDGET (64 * 1024)  // band CTAs: two per SM
#endif
constexpr int kBandStageBytes = RQ_BAND_STAGE_BYTES;
constexpr int kBandStageBudget = RQ_BAND_STAGE_BUDGET;
#ifndef RQ_GEMV_CTAS_PER_SM
#define RQ_GEMV_CTAS_PER_SM 2
#endif

namespace rqk {

template <typename WT>
cudaError_t gemv_dispatch(const GemvParams& p, int pro, int epi, int batch, cudaStream_t s,
                          bool pdl);
template <typename WT>
cudaError_t gemv_configure(int max_smem);

constexpr int kMaxDynSmem = 200 * 1024;

static int nch_bucket(int n) {
  if (n <= 1) return 1;
  if (n <= 2) return 2;
  if (n <= 3) return 3;
  if (n <= 4) return 4;
  if (n <= 6) return 6;
  return 0;  // unsupported
}

GemvPlan plan_gemv(int n_out, int K, int es, bool paired, bool even_rows, int num_sms,
                   int band) {
  GemvPlan pl{};
  pl.n_out = n_out;
  pl.K = K;
  // values per 16-byte chunk: 4 f32, 8 bf16, 16 q8 codes, 32 q4 codes
  const int V = band == BAND_Q8 ? 16 : (band == BAND_Q4 ? 32 : 16 / es);
  const int CC = K / V;
  int tpr = kGemvConsumers;
  while (tpr > 32 && tpr > CC) tpr >>= 1;
  const int ng = kGemvConsumers / tpr;
  pl.nch = nch_bucket((CC + tpr - 1) / tpr);
  // rows per thread group and tile: two while a thread's x fits in 32 values (bands) or
  // 2 chunks (f32 / bf16)
  pl.rg = band == BAND_NONE ? (pl.nch <= 2 ? 2 : 1) : (V * pl.nch <= 32 ? 2 : 1);
  if (band != BAND_NONE && pl.nch > 3) pl.nch = 0;      // x in registers: <= 96 values
  if ((paired || even_rows) && ((ng * pl.rg) & 1)) pl.nch = 0;
  const int row_bytes = (int)band_row_bytes(band, es, K);
  pl.tpr = tpr;
  pl.tile_rows = ng * pl.rg;
  const int max_grid = num_sms * RQ_GEMV_CTAS_PER_SM;
  if (band != BAND_NONE) {
    // band rows are short: a tile takes several rounds of the row groups, so each bulk
    // copy stays large (a producer thread keeps only a few copies in flight), as long
    // as every CTA of the grid still gets a tile
    const int per = paired ? pl.tile_rows / 2 : pl.tile_rows;
    int rounds = 1;
    while (rounds < 4 && 2 * rounds * pl.tile_rows * row_bytes <= kBandStageBytes &&
           (n_out + 2 * rounds * per - 1) / (2 * rounds * per) >= max_grid)
      rounds *= 2;
    pl.tile_rows *= rounds;
  }
  const int out_per_tile = paired ? pl.tile_rows / 2 : pl.tile_rows;
  pl.tiles = (n_out + out_per_tile - 1) / out_per_tile;
  pl.grid = pl.tiles < max_grid ? pl.tiles : max_grid;
  pl.max_tiles = (pl.tiles + pl.grid - 1) / pl.grid;
  const int tile_bytes = pl.tile_rows * row_bytes;
  int ns = (band != BAND_NONE ? kBandStageBudget : RQ_GEMV_STAGE_BUDGET) / tile_bytes;
  ns = ns < 2 ? 2 : (ns > RQ_GEMV_MAX_STAGES ? RQ_GEMV_MAX_STAGES : ns);
  if (ns > pl.max_tiles) ns = pl.max_tiles < 1 ? 1 : pl.max_tiles;
  pl.n_stages = ns;
  const int wpg = tpr / 32;
  const int part_n = (pl.max_tiles * pl.tile_rows * wpg + 3) & ~3;
  pl.smem = ns * tile_bytes + part_n * 4 + 2 * ns * 8;
  pl.bytes = (double)n_out * (paired ? 2.0 : 1.0) * row_bytes;
  pl.kparts = 1;
  pl.kp_width = K;
  return pl;
}

int gemv_chunks_per_thread(const GemvPlan& pl, int) {
  return pl.nch == 0 ? 1 << 20 : pl.nch;
}

// Raise the dynamic shared-memory limit of every instantiation once per device,
// before any launch is captured into a graph.
cudaError_t gemv_configure_all() {
  cudaError_t e[4] = {gemv_configure<uint16_t>(kMaxDynSmem), gemv_configure<float>(kMaxDynSmem),
                      gemv_configure<q8_t>(kMaxDynSmem), gemv_configure<q4_t>(kMaxDynSmem)};
  for (cudaError_t x : e)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

cudaError_t launch_gemv(const GemvParams& p, int pro, int epi, int wtype, int batch,
                        cudaStream_t s, bool pdl) {
  if (p.pl.smem > kMaxDynSmem || p.pl.nch == 0) return cudaErrorInvalidValue;
  switch (wtype) {
    case 0: return gemv_dispatch<float>(p, pro, epi, batch, s, pdl);
    case 1: return gemv_dispatch<uint16_t>(p, pro, epi, batch, s, pdl);
    case BAND_Q8: return gemv_dispatch<q8_t>(p, pro, epi, batch, s, pdl);
    case BAND_Q4: return gemv_dispatch<q4_t>(p, pro, epi, batch, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rqk
