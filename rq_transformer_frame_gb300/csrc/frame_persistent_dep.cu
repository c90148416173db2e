// frame_persistent_dep.cu -- the depformer's cooperative launch: the same kernel at one
// CTA per SM (every weight type, greedy and with token picks); compiled apart so the
// units build in parallel.
#include "frame_persistent.cuh"

namespace rqk {
namespace pers {
RQ_PERS_DEP(RQ_PERS_INSTANTIATE, false)
RQ_PERS_DEP(RQ_PERS_INSTANTIATE, true)
}  // namespace pers
}  // namespace rqk
