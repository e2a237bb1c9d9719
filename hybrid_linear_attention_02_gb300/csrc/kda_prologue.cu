// KDA's input prologue in one pass ("[Paper Review] Kimi K3: Open Frontier
// Intelligence", section "Kimi Delta Attention (KDA)"):
//   q = L2norm(Swish(ShortConv_q(q_pre))),  k = L2norm(Swish(ShortConv_k(k_pre)))
//   g = g_min sigmoid(exp(A_h) z),  g_min = -5
// ShortConv is a depthwise causal convolution of 4 taps along each sequence
// (tap 3 on the current token, zero before the sequence's first token);
// L2norm(y) = y / sqrt(sum(y^2) + 1e-6) over the dk channels of a head.
// One warp per head and 4 consecutive tokens, each lane dk / 32 consecutive
// channels; the warp loads the 7 rows its taps read once per branch (the rows
// shared with the neighbouring warps come from L2), so HBM sees each input and
// output row about once.  Blocks whose tap rows all lie inside one sequence and
// inside the tensor (nearly all) run a path without per-tap masking or row
// clamping.
#include <cuda_bf16.h>

#include <type_traits>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kWarps = 8;         // heads per block
constexpr int kRowsPerWarp = 4;   // consecutive tokens per warp
constexpr int kTaps = 4;
constexpr float kGMin = -5.f;
constexpr float kNormEps = 1e-6f;

// PER consecutive elements as one vector access (8 or 16 bytes for PER = 4,
// 4 or 8 bytes for PER = 2); the row offsets keep them aligned.
template <int PER>
__device__ __forceinline__ void ldv(const __nv_bfloat16* p, float (&y)[PER]) {
  if constexpr (PER == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    y[0] = __uint_as_float(u.x << 16); y[1] = __uint_as_float(u.x & 0xFFFF0000u);
    y[2] = __uint_as_float(u.y << 16); y[3] = __uint_as_float(u.y & 0xFFFF0000u);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    y[0] = __uint_as_float(u << 16); y[1] = __uint_as_float(u & 0xFFFF0000u);
  }
}
template <int PER>
__device__ __forceinline__ void ldv(const float* p, float (&y)[PER]) {
  if constexpr (PER == 4) {
    const float4 u = *reinterpret_cast<const float4*>(p);
    y[0] = u.x; y[1] = u.y; y[2] = u.z; y[3] = u.w;
  } else {
    const float2 u = *reinterpret_cast<const float2*>(p);
    y[0] = u.x; y[1] = u.y;
  }
}
__device__ __forceinline__ uint32_t bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <int PER>
__device__ __forceinline__ void stv(__nv_bfloat16* p, const float (&y)[PER]) {
  if constexpr (PER == 4)
    *reinterpret_cast<uint2*>(p) = make_uint2(bf2(y[0], y[1]), bf2(y[2], y[3]));
  else
    *reinterpret_cast<uint32_t*>(p) = bf2(y[0], y[1]);
}
template <int PER>
__device__ __forceinline__ void stv(float* p, const float (&y)[PER]) {
  if constexpr (PER == 4)
    *reinterpret_cast<float4*>(p) = make_float4(y[0], y[1], y[2], y[3]);
  else
    *reinterpret_cast<float2*>(p) = make_float2(y[0], y[1]);
}

// First token of the sequence that holds token t.
__device__ __forceinline__ long long seq_start(const PrologueArgs& a, long long t) {
  if (a.cu_seqlens) {
    int lo = 0, hi = a.n_seqs;   // cu[lo] <= t < cu[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.cu_seqlens[mid] <= t) lo = mid;
      else hi = mid;
    }
    return a.cu_seqlens[lo];
  }
  if (a.seq_len <= 0) return 0;
  const unsigned sl = static_cast<unsigned>(a.seq_len);
  return static_cast<long long>(static_cast<unsigned>(t) / sl) * sl;
}

// Warp w of block (b, hb) handles head 8 hb + w and tokens 4 b .. 4 b + 3.
// Raw PER-element vectors (kept packed until used).
template <typename T, int PER>
struct Raw;
template <>
struct Raw<__nv_bfloat16, 4> { using type = uint2; };
template <>
struct Raw<__nv_bfloat16, 2> { using type = uint32_t; };
template <>
struct Raw<float, 4> { using type = float4; };
template <>
struct Raw<float, 2> { using type = float2; };

template <int PER, typename R>
__device__ __forceinline__ void unpack(const R& v, float (&y)[PER]) {
  ldv<PER>(reinterpret_cast<const typename std::conditional<
               sizeof(R) == 2 * PER, __nv_bfloat16, float>::type*>(&v), y);
}

// Rows of one warp: tokens tb .. tb + R - 1 of head h.  kInterior: every tap
// row lies inside the tensor and inside the sequence of the block's last
// token, so no tap is masked and no row index is clamped (the common case).
template <typename T, int DK, bool kInterior>
__device__ __forceinline__ void prologue_rows(const PrologueArgs& a, int h, long long tb) {
  constexpr int PER = DK / 32;
  constexpr int R = kRowsPerWarp;
  constexpr int WIN = R + kTaps - 1;
  using RawT = typename Raw<T, PER>::type;
  const int lane = threadIdx.x & 31;
  const long long n_tok = a.total_tokens;
  const int c0 = PER * lane;
  const long long rs = static_cast<long long>(a.heads) * DK;      // row stride
  const long long col = static_cast<long long>(h) * DK + c0;
  // Every load first: the tap windows of q and k (rows tb - 3 .. tb + R - 1)
  // and the z rows.
  RawT xw[2][WIN], zr[R];
#pragma unroll
  for (int br = 0; br < 2; ++br) {
    const T* x = static_cast<const T*>(br ? a.k_pre : a.q_pre);
#pragma unroll
    for (int i = 0; i < WIN; ++i) {
      long long src = tb - (kTaps - 1) + i;
      if (!kInterior) src = src < 0 ? 0 : src >= n_tok ? n_tok - 1 : src;
      xw[br][i] = *reinterpret_cast<const RawT*>(x + src * rs + col);
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const long long src = kInterior || tb + r < n_tok ? tb + r : n_tok - 1;
    zr[r] = *reinterpret_cast<const RawT*>(static_cast<const T*>(a.z) + src * rs + col);
  }
  long long t0[R];
  if (!kInterior) {
#pragma unroll
    for (int r = 0; r < R; ++r) t0[r] = tb + r < n_tok ? seq_start(a, tb + r) : tb + r;
  }

#pragma unroll
  for (int br = 0; br < 2; ++br) {
    const float* w = (br ? a.conv_k : a.conv_q) + col * kTaps;
    T* y_out = static_cast<T*>(br ? a.k : a.q) + col;
    float4 wt[PER];   // the 4 taps of each channel
#pragma unroll
    for (int u = 0; u < PER; ++u) wt[u] = __ldg(reinterpret_cast<const float4*>(w) + u);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const long long t = tb + r;
      float y[PER] = {};
#pragma unroll
      for (int i = 0; i < kTaps; ++i) {
        const bool on = kInterior || t - (kTaps - 1) + i >= t0[r];
        float xv[PER];
        unpack<PER>(xw[br][r + i], xv);
#pragma unroll
        for (int u = 0; u < PER; ++u) {
          const float wi = i == 0 ? wt[u].x : i == 1 ? wt[u].y : i == 2 ? wt[u].z : wt[u].w;
          y[u] = fmaf(on ? wi : 0.f, xv[u], y[u]);
        }
      }
      float ss = 0.f;
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        y[u] = __fdividef(y[u], 1.f + __expf(-y[u]));   // Swish
        ss = fmaf(y[u], y[u], ss);
      }
#pragma unroll
      for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, m);
      const float rinv = rsqrtf(ss + kNormEps);
#pragma unroll
      for (int u = 0; u < PER; ++u) y[u] *= rinv;
      if (kInterior || t < n_tok) stv<PER>(y_out + t * rs, y);
    }
  }
  const float scale = __expf(__ldg(a.a_log + h));
#pragma unroll
  for (int r = 0; r < R; ++r) {
    float zv[PER];
    unpack<PER>(zr[r], zv);
#pragma unroll
    for (int u = 0; u < PER; ++u) zv[u] = __fdividef(kGMin, 1.f + __expf(-scale * zv[u]));
    if (kInterior || tb + r < n_tok) stv<PER>(static_cast<T*>(a.g) + (tb + r) * rs + col, zv);
  }
}

// bf16: four blocks per SM (measured faster than the three that 77 registers
// allow, despite a few spilled bytes); fp32 keeps its registers.
template <typename T, int DK>
__global__ void __launch_bounds__(32 * kWarps, sizeof(T) == 2 ? 4 : 1) prologue_kernel(PrologueArgs a) {
  constexpr int R = kRowsPerWarp;
  const int h = blockIdx.y * kWarps + (threadIdx.x >> 5);
  if (h >= a.heads) return;
  const long long tb = static_cast<long long>(blockIdx.x) * R;   // first token
  const long long n_tok = a.total_tokens;
  const bool interior = tb >= kTaps - 1 && tb + R <= n_tok &&
                        seq_start(a, tb + R - 1) <= tb - (kTaps - 1);
  if (interior) prologue_rows<T, DK, true>(a, h, tb);
  else prologue_rows<T, DK, false>(a, h, tb);
}

template <typename T, int DK>
cudaError_t launch_typed(const PrologueArgs& a, cudaStream_t s) {
  const long long tblocks = (a.total_tokens + kRowsPerWarp - 1) / kRowsPerWarp;
  if (tblocks >= (1ll << 31)) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(tblocks), (a.heads + kWarps - 1) / kWarps);
  prologue_kernel<T, DK><<<grid, 32 * kWarps, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t s) {
  if (a.total_tokens == 0 || a.heads == 0) return cudaSuccess;
  const bool f32 = a.dtype == KDA_F32;
  if (a.dk == 128) return f32 ? launch_typed<float, 128>(a, s) : launch_typed<__nv_bfloat16, 128>(a, s);
  if (a.dk == 64) return f32 ? launch_typed<float, 64>(a, s) : launch_typed<__nv_bfloat16, 64>(a, s);
  return cudaErrorInvalidValue;
}

}  // namespace kda
