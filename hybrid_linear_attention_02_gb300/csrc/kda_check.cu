// Precondition check of the inputs: every log-decay g in [g_min, 0] with
// g_min = -5 and every beta in [0, 1].
//
// The lower bound is the one of "[Paper Review] Kimi K3: Open Frontier
// Intelligence", section "Kimi Delta Attention (KDA)" (the scaled-sigmoid
// decay g = g_min * sigmoid(.)): it keeps a 16-token tile's log-decay above
// -80, so the tensor-core path's in-tile factors stay below e^80, inside the
// bf16 and fp32 range.  g > 0 would make alpha = e^g > 1 (no longer a forget
// gate) and beta outside [0, 1] breaks the erase-then-write reading of the
// same section.  NaN fails every comparison and is reported too.
//
// One pass over g and beta (HBM-bound, 16-byte loads for g); a warp that
// finds a value out of range sets *dev_status to KDA_ERR_RANGE unless it
// already holds an error.  Nothing traps.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ bool g_ok(float x) { return x >= -5.0f && x <= 0.0f; }
__device__ __forceinline__ bool beta_ok(float x) { return x >= 0.0f && x <= 1.0f; }

template <typename T>
__global__ void range_check_kernel(const T* __restrict__ g, long long n_g,
                                   const T* __restrict__ beta, long long n_beta,
                                   int* dev_status) {
  constexpr int kVec = 16 / sizeof(T);
  const long long n_vec = n_g / kVec;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long i0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  bool bad = false;
  for (long long i = i0; i < n_vec; i += stride) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(g) + i);
    const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
    for (int j = 0; j < kVec; ++j) bad |= !g_ok(to_f(e[j]));
  }
  for (long long i = n_vec * kVec + i0; i < n_g; i += stride) bad |= !g_ok(to_f(g[i]));
  for (long long i = i0; i < n_beta; i += stride) bad |= !beta_ok(to_f(beta[i]));
  if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0)
    atomicCAS(dev_status, 0, static_cast<int>(KDA_ERR_RANGE));
}

}  // namespace

cudaError_t launch_range_check(const void* g, const void* beta, long long tokens, int heads,
                               int dk, int dtype, int* dev_status, cudaStream_t stream) {
  const long long n_g = tokens * heads * dk, n_beta = tokens * heads;
  if (n_g == 0 && n_beta == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  const long long want = (n_g / 8 + 255) / 256;
  const unsigned grid = static_cast<unsigned>(want < 1 ? 1 : want < 8ll * sms ? want : 8ll * sms);
  if (dtype == KDA_BF16)
    range_check_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(g), n_g, static_cast<const __nv_bfloat16*>(beta),
        n_beta, dev_status);
  else
    range_check_kernel<float><<<grid, 256, 0, stream>>>(
        static_cast<const float*>(g), n_g, static_cast<const float*>(beta), n_beta, dev_status);
  return cudaGetLastError();
}

}  // namespace kda
