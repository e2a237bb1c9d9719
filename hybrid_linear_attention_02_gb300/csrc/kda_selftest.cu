// Failure-detection self-test: the kernels' bounded mbarrier wait, run on a
// barrier that nothing ever arrives at, must give up after its limit, report
// KDA_ERR_TIMEOUT through dev_status and leave the context usable.  No fault,
// trap or unbounded loop is involved: the kernel returns once the limit passes.
#include "kda_chunk_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace {

__global__ void wait_timeout_kernel(int* dev_status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    abort_flag = 0;
    sm100::fence_mbar_init();
  }
  __syncthreads();
  chunk::Sync sync{&bar, &abort_flag};
  const bool ok = sync.wait_for(0, 0, limit_ns);   // phase 0 never completes
  if (!ok && threadIdx.x == 0 && dev_status) atomicExch(dev_status, KDA_ERR_TIMEOUT);
}

}  // namespace
}  // namespace kda

extern "C" KDA_API int kda_debug_wait_timeout(int* dev_status, unsigned timeout_us, void* stream) {
  if (!dev_status || timeout_us == 0 || timeout_us > 10000000u) return KDA_ERR_INVALID;
  kda::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      dev_status, static_cast<unsigned long long>(timeout_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
