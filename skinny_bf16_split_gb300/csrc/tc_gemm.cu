// tc_gemm.cu -- tcgen05 tensor-core tactic (not yet implemented: rejected as invalid).
#include "internal.h"

namespace dep {
bool tc_valid(const dep_tactic_t &) { return false; }
int64_t tc_units(const dep_tactic_t &, int64_t, int64_t) { return 1; }
size_t tc_ws_per_cta(const dep_tactic_t &) { return 0; }
size_t tc_counters(const dep_tactic_t &, int64_t) { return 0; }
int tc_blocks_per_sm(const dep_tactic_t &) { return 0; }
cudaError_t tc_run(const dep_tactic_t &, const RunArgs &) { return cudaErrorNotSupported; }
}  // namespace dep
