// Composition of KDA segment transitions (the single-GPU form of the
// context parallelism in "[Paper Review] Kimi K3: Open Frontier
// Intelligence", section "Infrastructure: how to actually run
// trillion-scale"): a segment maps its entry state to S_end = M S_0 + H, and
// maps compose as (M2, H2) o (M1, H1) = (M2 M1, M2 H1 + H2).  Both are the one
// product below, in fp32 on CUDA cores (each is a single 128 x 128 x 128
// product per sequence-head pair, far from any bound).
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kKTile = 32;

// out[o, i] = M[o, i] S[o, i] (+ H[o, i]) for o < n_outer, i < n_inner, where
// pair (o, i) of each array sits at base + (o * stride_outer + i) * size.
template <int DK, int DV>
__global__ void __launch_bounds__(kThreads)
    transition_apply_kernel(const float* __restrict__ M, const float* __restrict__ H,
                            const float* __restrict__ S, float* __restrict__ out, int n_inner,
                            long long m_stride, long long s_stride, long long o_stride) {
  constexpr int RT = DK / 16, CT = DV / 16;   // rows x columns of out per thread
  __shared__ float mt[kKTile][DK + 1];              // M[:, k0 .. k0 + 31], transposed
  __shared__ __align__(16) float st[kKTile][DV];   // S[k0 .. k0 + 31, :]
  const int o = blockIdx.y, i = blockIdx.x;
  const float* m = M + (o * m_stride + i) * DK * DK;
  const float* s = S + (o * s_stride + i) * DK * DV;
  const float* hh = H ? H + (o * m_stride + i) * DK * DV : nullptr;
  float* y = out + (o * o_stride + i) * DK * DV;
  const int tr = threadIdx.x >> 4, tc = threadIdx.x & 15;
  float acc[RT][CT] = {};
  for (int k0 = 0; k0 < DK; k0 += kKTile) {
    for (int e = threadIdx.x; e < kKTile * DK; e += kThreads) {
      const int r = e / kKTile, kk = e % kKTile;
      mt[kk][r] = m[r * DK + k0 + kk];
    }
    for (int e = threadIdx.x; e < kKTile * DV; e += kThreads) {
      const int kk = e / DV, c = e % DV;
      st[kk][c] = s[(k0 + kk) * DV + c];
    }
    __syncthreads();
#pragma unroll 4
    for (int kk = 0; kk < kKTile; ++kk) {
      float a[RT], b[CT];
#pragma unroll
      for (int r = 0; r < RT; ++r) a[r] = mt[kk][RT * tr + r];
#pragma unroll
      for (int c = 0; c < CT; ++c) b[c] = st[kk][CT * tc + c];
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int c = 0; c < CT; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int c = 0; c < CT; ++c) {
      const int idx = (RT * tr + r) * DV + CT * tc + c;
      y[idx] = acc[r][c] + (hh ? hh[idx] : 0.f);
    }
}

template <int DK, int DV>
cudaError_t launch_typed(const float* M, const float* H, const float* S, float* out,
                         long long n_outer, int n_inner, long long m_stride, long long s_stride,
                         long long o_stride, cudaStream_t st) {
  if (n_outer <= 0 || n_inner <= 0) return cudaSuccess;
  if (n_outer > 65535 || n_inner > (1 << 30)) return cudaErrorInvalidValue;
  dim3 grid(n_inner, static_cast<unsigned>(n_outer));
  transition_apply_kernel<DK, DV><<<grid, kThreads, 0, st>>>(M, H, S, out, n_inner, m_stride,
                                                             s_stride, o_stride);
  return cudaGetLastError();
}

__global__ void segment_offsets_kernel(int* cu_seg, int n_seqs, long long seq_len, int n_seg,
                                       long long seg_len) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(n_seqs) * n_seg;
  if (i > total) return;
  if (i == total) {
    cu_seg[i] = static_cast<int>(n_seqs * seq_len);
    return;
  }
  const long long n = i / n_seg, s = i % n_seg;
  const long long off = s * seg_len < seq_len ? s * seg_len : seq_len;
  cu_seg[i] = static_cast<int>(n * seq_len + off);
}

}  // namespace

cudaError_t launch_segment_offsets(int* cu_seg, int n_seqs, long long seq_len, int n_segments,
                                   long long seg_len, cudaStream_t st) {
  const long long total = static_cast<long long>(n_seqs) * n_segments + 1;
  segment_offsets_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(
      cu_seg, n_seqs, seq_len, n_segments, seg_len);
  return cudaGetLastError();
}

cudaError_t launch_transition_apply_strided(const float* M, const float* H, const float* S,
                                            float* out, long long n_outer, int n_inner,
                                            long long m_stride, long long s_stride,
                                            long long o_stride, int dk, int dv,
                                            cudaStream_t st) {
  if (dk == 128 && dv == 128)
    return launch_typed<128, 128>(M, H, S, out, n_outer, n_inner, m_stride, s_stride, o_stride, st);
  if (dk == 64 && dv == 64)
    return launch_typed<64, 64>(M, H, S, out, n_outer, n_inner, m_stride, s_stride, o_stride, st);
  if (dk == 128 && dv == 64)
    return launch_typed<128, 64>(M, H, S, out, n_outer, n_inner, m_stride, s_stride, o_stride, st);
  if (dk == 64 && dv == 128)
    return launch_typed<64, 128>(M, H, S, out, n_outer, n_inner, m_stride, s_stride, o_stride, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_transition_apply(const float* M, const float* H, const float* S_in,
                                    float* S_out, long long pairs, int dk, int dv,
                                    cudaStream_t st) {
  // One row of `pairs` pairs (a grid dimension holds up to 2^30 of them here).
  if (pairs <= (1 << 30))
    return launch_transition_apply_strided(M, H, S_in, S_out, 1, static_cast<int>(pairs), 0, 0, 0,
                                           dk, dv, st);
  return cudaErrorInvalidValue;
}

}  // namespace kda
