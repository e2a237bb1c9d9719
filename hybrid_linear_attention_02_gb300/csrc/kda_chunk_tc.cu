// bf16 chunkwise KDA on tcgen05 tensor cores (dk = dv = 128, chunk = 64).
#include "kda_internal.h"

namespace kda {

bool chunk_tc_supported(const LaunchArgs& a) {
  (void)a;
  return false;
}

cudaError_t launch_chunk_tc(const LaunchArgs& a, cudaStream_t stream) {
  (void)a;
  (void)stream;
  return cudaErrorNotSupported;
}

}  // namespace kda
