// Lightning indexer on the tcgen05 tensor cores (filled in below).
#include "common.cuh"

namespace dsa {

bool indexer_tc_supported(const dsa_problem&) { return false; }

cudaError_t launch_indexer_tc(const dsa_problem&, const Plan&, int32_t*, uint32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace dsa
