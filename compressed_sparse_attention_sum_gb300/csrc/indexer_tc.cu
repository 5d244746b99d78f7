// Tensor-core (tcgen05) indexer score kernel: placeholder until written.
#include "csa_common.cuh"
#include "csa_kernels.h"
namespace csa {
bool indexer_tc_supported(int, int) { return false; }
cudaError_t launch_indexer_scores_tc(const void*, const void*, const float*, float*, int, int, int,
                                     int, int, int, int, int, int*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace csa
