// tcgen05 prefill scorer (not built yet: the launcher refuses).
#include "qsa_launch.h"

namespace qsa {

const bool kTcScorerReady = false;

cudaError_t launch_score_tc(const ScoreArgs &, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace qsa
