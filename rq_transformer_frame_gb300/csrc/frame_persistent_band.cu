// frame_persistent_band.cu -- the whole-frame kernel for weight-band models (q8 / q4
// matrices, bf16 tables and K/V), greedy and with token picks; compiled apart from the
// f32 / bf16 instantiations so the units build in parallel.
#include "frame_persistent.cuh"

namespace rqk {
namespace pers {
RQ_PERS_BANDS(RQ_PERS_INSTANTIATE, false)
RQ_PERS_BANDS(RQ_PERS_INSTANTIATE, true)
}  // namespace pers
}  // namespace rqk
