// frame_persistent_greedy.cu -- the whole-frame kernel without the token-pick ops, for
// greedy frames; compiled apart from frame_persistent.cu so both build in parallel.
#include "frame_persistent.cuh"

namespace rqk {
namespace pers {
RQ_PERS_ALL(RQ_PERS_INSTANTIATE, false)
}  // namespace pers
}  // namespace rqk
