// KDA output epilogue as a separate pass: head-wise RMSNorm of each output row
// followed by the full-rank sigmoid gate ("[Paper Review] Kimi K3: Open
// Frontier Intelligence", section "Kimi Delta Attention (KDA)", paragraph
// "Full-rank gate"):
//   out[t, h, :] = o / sqrt(mean(o^2) + eps) * w * sigmoid(z[t, h, :])
// One warp per (token, head) row; each lane holds dv / 32 consecutive
// channels, so a warp moves one 256-byte bf16 row (dv = 128) per access.
// Used after the fused tensor-core kernel; the split form and the CUDA-core
// recurrence apply the same epilogue inside their own kernels.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kWarps = 8;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <typename T, int DV>
__global__ void __launch_bounds__(32 * kWarps)
    gate_epilogue_kernel(T* __restrict__ out, const T* __restrict__ z,
                         const float* __restrict__ w, float eps, long long rows) {
  constexpr int PER = DV / 32;
  const int lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  T* o_row = out + row * DV + PER * lane;
  const T* z_row = z + row * DV + PER * lane;
  float o[PER], ss = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    o[i] = to_f(o_row[i]);
    ss = fmaf(o[i], o[i], ss);
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, m);
  const float rinv = rsqrtf(ss * (1.f / DV) + eps);
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const float zz = to_f(z_row[i]);
    o_row[i] = from_f<T>(o[i] * rinv * w[PER * lane + i] / (1.f + __expf(-zz)));
  }
}

template <typename T, int DV>
cudaError_t launch_typed(const LaunchArgs& a, long long rows, cudaStream_t s) {
  const long long blocks = (rows + kWarps - 1) / kWarps;
  gate_epilogue_kernel<T, DV><<<static_cast<unsigned>(blocks), 32 * kWarps, 0, s>>>(
      static_cast<T*>(a.out), static_cast<const T*>(a.gate), a.gate_w, a.gate_eps, rows);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gate_epilogue(const LaunchArgs& a, cudaStream_t s) {
  const long long rows = a.total_tokens * a.heads;
  if (rows == 0 || !a.gate) return cudaSuccess;
  if (rows / kWarps >= (1ll << 31)) return cudaErrorInvalidValue;
  const bool f32 = a.dtype == KDA_F32;
  if (a.dv == 128)
    return f32 ? launch_typed<float, 128>(a, rows, s) : launch_typed<__nv_bfloat16, 128>(a, rows, s);
  if (a.dv == 64)
    return f32 ? launch_typed<float, 64>(a, rows, s) : launch_typed<__nv_bfloat16, 64>(a, rows, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
