// spin_score_tc.cu -- indexer score with one key shared by all heads, on tcgen05 tensor
// cores.  (Placeholder until the kernel lands: reports the shape as unsupported.)
#include "spin_common.cuh"
#include "spin_internal.h"

namespace spin {

bool score_tc_supported(const spin_config&, int) { return false; }

cudaError_t launch_score_tc(const spin_config&, const ScoreArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace spin
