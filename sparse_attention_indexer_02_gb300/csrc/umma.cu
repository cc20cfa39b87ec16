// tcgen05 scorer (placeholder until the kernel lands): reports every shape as
// unsupported so the dispatch routes to the CUDA-core scorer.
#include "qsa_internal.h"

namespace qsa {

bool umma_supports(const qsa_paged_desc&, const char** why) {
  *why = "tcgen05 scorer not built";
  return false;
}

cudaError_t launch_umma(const ScoreParams&, cudaStream_t, const char** msg) {
  *msg = "tcgen05 scorer not built";
  return cudaErrorInvalidValue;
}

}  // namespace qsa
