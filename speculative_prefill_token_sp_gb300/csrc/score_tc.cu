// Tensor-core (tcgen05 + TMA) scoring path -- placeholder until it lands.
#include "sp_common.cuh"

namespace sp {
bool score_tc_supported(const ScoreProblem&) { return false; }
size_t score_tc_ws_bytes(const ScoreProblem&) { return 0; }
sp_status score_tc_launch(const ScoreProblem&, void*, cudaStream_t) { return SP_EUNSUPPORTED; }
}  // namespace sp
