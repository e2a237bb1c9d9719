// KDA on CUDA cores, one token at a time, fp32 state held in registers.
//
// Per token (the update of "[Paper Review] Kimi K3: Open Frontier
// Intelligence", section "Kimi Delta Attention (KDA)", expanded):
//   S' = Diag(exp g) S;  u = S'^T k;  p = S'^T q;  delta = beta (v - u)
//   S  = S' + k delta^T;  o = S^T q = p + (q . k) delta
// One CTA owns one (sequence, head) state: 256 threads, thread (rg, cg) holds
// rows {rg + RG*m} x columns [4cg, 4cg+4) as float4s, so every state row is
// read and written by one warp as 512 contiguous bytes (dv = 128).  The two
// column reductions (u and p) go through shared memory, double-buffered by
// token parity so one token costs two barriers.
//
// With one token per sequence this is the decode step: the state streams in
// once and out once, in place.
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float load_in(const T* p, long long i);
template <>
__device__ __forceinline__ float load_in<float>(const float* p, long long i) {
  return __ldg(p + i);
}
template <>
__device__ __forceinline__ float load_in<__nv_bfloat16>(const __nv_bfloat16* p, long long i) {
  return __bfloat162float(p[i]);
}

template <typename T>
__device__ __forceinline__ void store_out4(T* p, long long i, float4 x);
template <>
__device__ __forceinline__ void store_out4<float>(float* p, long long i, float4 x) {
  *reinterpret_cast<float4*>(p + i) = x;
}
template <>
__device__ __forceinline__ void store_out4<__nv_bfloat16>(__nv_bfloat16* p, long long i,
                                                          float4 x) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(x.z, x.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p + i) = pk;
}

// kCkpt: also write the prefix-cache checkpoints; kGate: apply the output
// epilogue (head-wise RMSNorm, then the sigmoid gate) to every output row.
// Each is its own instantiation, so the plain prefill and decode code carries
// no extra test.
template <int DK, int DV, typename T, bool kCkpt, bool kGate>
__global__ void __launch_bounds__(kThreads) recurrent_kernel(LaunchArgs a) {
  constexpr int CG = DV / 4;       // float4 column groups
  constexpr int RG = kThreads / CG;  // row groups
  constexpr int RPT = DK / RG;     // state rows per thread
  static_assert(kThreads % CG == 0 && DK % RG == 0, "thread layout");

  __shared__ float s_q[2][DK], s_k[2][DK], s_a[2][DK], s_v[2][DV], s_b[2];
  __shared__ __align__(16) float s_ru[2][RG][DV];
  __shared__ __align__(16) float s_rp[2][RG][DV];
  __shared__ float s_rqk[2][RG];

  const T* __restrict__ q = static_cast<const T*>(a.q);
  const T* __restrict__ k = static_cast<const T*>(a.k);
  const T* __restrict__ v = static_cast<const T*>(a.v);
  const T* __restrict__ g = static_cast<const T*>(a.g);
  const T* __restrict__ beta = static_cast<const T*>(a.beta);
  T* __restrict__ out = static_cast<T*>(a.out);

  const int h = blockIdx.y;
  const int n = a.order ? a.order[blockIdx.x] : static_cast<int>(blockIdx.x);
  long long t0, t1;
  if (a.cu_seqlens) {
    t0 = a.cu_seqlens[n];
    t1 = a.cu_seqlens[n + 1];
  } else {
    t0 = static_cast<long long>(n) * a.seq_len;
    t1 = t0 + a.seq_len;
  }
  const int tid = threadIdx.x;
  const int cg = tid % CG, rg = tid / CG;
  const long long soff = (static_cast<long long>(n) * a.heads + h) * DK * DV;

  float4 S[RPT];
  if (a.init_state) {
    const float4* src = reinterpret_cast<const float4*>(a.init_state + soff);
#pragma unroll
    for (int m = 0; m < RPT; ++m) S[m] = __ldcs(src + (rg + RG * m) * CG + cg);
  } else {
#pragma unroll
    for (int m = 0; m < RPT; ++m) S[m] = make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // Tokens [s0, s1) of the sequence, one at a time.
  auto run = [&](long long s0, long long s1) {
    for (long long t = s0; t < s1; ++t) {
      const int b = static_cast<int>((t - t0) & 1);
      const long long rk = (t * a.heads + h) * DK, rv = (t * a.heads + h) * DV;
      for (int c = tid; c < DK; c += kThreads) {
        s_q[b][c] = load_in(q, rk + c);
        s_k[b][c] = load_in(k, rk + c);
        s_a[b][c] = expf(load_in(g, rk + c));
      }
      for (int j = tid; j < DV; j += kThreads) s_v[b][j] = load_in(v, rv + j);
      if (tid == 0) s_b[b] = load_in(beta, t * a.heads + h);
      __syncthreads();

      float4 pu = make_float4(0.f, 0.f, 0.f, 0.f), pp = pu;
      float pqk = 0.f;
#pragma unroll
      for (int m = 0; m < RPT; ++m) {
        const int c = rg + RG * m;
        const float al = s_a[b][c], kc = s_k[b][c], qc = s_q[b][c];
        S[m].x *= al; S[m].y *= al; S[m].z *= al; S[m].w *= al;
        pu.x = fmaf(S[m].x, kc, pu.x); pu.y = fmaf(S[m].y, kc, pu.y);
        pu.z = fmaf(S[m].z, kc, pu.z); pu.w = fmaf(S[m].w, kc, pu.w);
        pp.x = fmaf(S[m].x, qc, pp.x); pp.y = fmaf(S[m].y, qc, pp.y);
        pp.z = fmaf(S[m].z, qc, pp.z); pp.w = fmaf(S[m].w, qc, pp.w);
        pqk = fmaf(qc, kc, pqk);
      }
      *reinterpret_cast<float4*>(&s_ru[b][rg][4 * cg]) = pu;
      *reinterpret_cast<float4*>(&s_rp[b][rg][4 * cg]) = pp;
      if (cg == 0) s_rqk[b][rg] = pqk;
      __syncthreads();

      float4 u = make_float4(0.f, 0.f, 0.f, 0.f), p = u;
      float qk = 0.f;
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const float4 x = *reinterpret_cast<const float4*>(&s_ru[b][r][4 * cg]);
        const float4 y = *reinterpret_cast<const float4*>(&s_rp[b][r][4 * cg]);
        u.x += x.x; u.y += x.y; u.z += x.z; u.w += x.w;
        p.x += y.x; p.y += y.y; p.z += y.z; p.w += y.w;
        qk += s_rqk[b][r];
      }
      const float bt = s_b[b];
      const float4 vv = *reinterpret_cast<const float4*>(&s_v[b][4 * cg]);
      const float4 d = make_float4(bt * (vv.x - u.x), bt * (vv.y - u.y), bt * (vv.z - u.z),
                                   bt * (vv.w - u.w));
#pragma unroll
      for (int m = 0; m < RPT; ++m) {
        const float kc = s_k[b][rg + RG * m];
        S[m].x = fmaf(kc, d.x, S[m].x); S[m].y = fmaf(kc, d.y, S[m].y);
        S[m].z = fmaf(kc, d.z, S[m].z); S[m].w = fmaf(kc, d.w, S[m].w);
      }
      if (rg == 0) {
        float4 o = make_float4(fmaf(qk, d.x, p.x), fmaf(qk, d.y, p.y), fmaf(qk, d.z, p.z),
                               fmaf(qk, d.w, p.w));
        if constexpr (kGate) {
          // Threads rg == 0 are lanes 0 .. CG-1 of warp 0 and hold the whole row.
          constexpr unsigned kMask = CG == 32 ? 0xFFFFFFFFu : ((1u << CG) - 1u);
          float ss = o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w;
#pragma unroll
          for (int m = CG / 2; m > 0; m >>= 1) ss += __shfl_xor_sync(kMask, ss, m);
          const float rinv = rsqrtf(ss * (1.f / DV) + a.gate_eps);
          const T* __restrict__ zg = static_cast<const T*>(a.gate);
          const float4 wv = *reinterpret_cast<const float4*>(a.gate_w + 4 * cg);
          o.x *= rinv * wv.x / (1.f + __expf(-load_in(zg, rv + 4 * cg)));
          o.y *= rinv * wv.y / (1.f + __expf(-load_in(zg, rv + 4 * cg + 1)));
          o.z *= rinv * wv.z / (1.f + __expf(-load_in(zg, rv + 4 * cg + 2)));
          o.w *= rinv * wv.w / (1.f + __expf(-load_in(zg, rv + 4 * cg + 3)));
        }
        store_out4(out, rv + 4 * cg, o);
      }
    }
  };

  if constexpr (kCkpt) {
    // Segments of ckpt_interval tokens; after each full one, its checkpoint.
    const long long seg = a.ckpt_interval;
    for (long long s0 = t0; s0 < t1; s0 += seg) {
      const long long s1 = s0 + seg < t1 ? s0 + seg : t1;
      run(s0, s1);
      if (s1 - s0 == seg) {
        const long long row = a.ckpt_offsets[n] + (s1 - t0) / seg - 1;
        float4* dst = reinterpret_cast<float4*>(a.ckpt + (row * a.heads + h) * DK * DV);
#pragma unroll
        for (int m = 0; m < RPT; ++m) __stcs(dst + (rg + RG * m) * CG + cg, S[m]);
      }
    }
  } else {
    run(t0, t1);
  }

  if (a.final_state) {
    float4* dst = reinterpret_cast<float4*>(a.final_state + soff);
#pragma unroll
    for (int m = 0; m < RPT; ++m) __stcs(dst + (rg + RG * m) * CG + cg, S[m]);
  }
}

template <int DK, int DV>
cudaError_t launch_dims(const LaunchArgs& a, cudaStream_t s) {
  dim3 grid(a.n_seqs, a.heads);
  // Checkpoints and the output gate are separate entry points, never both.
  if (a.ckpt && a.gate) return cudaErrorInvalidValue;
  if (a.dtype == KDA_F32) {
    if (a.ckpt)
      recurrent_kernel<DK, DV, float, true, false><<<grid, kThreads, 0, s>>>(a);
    else if (a.gate)
      recurrent_kernel<DK, DV, float, false, true><<<grid, kThreads, 0, s>>>(a);
    else
      recurrent_kernel<DK, DV, float, false, false><<<grid, kThreads, 0, s>>>(a);
  } else {
    if (a.ckpt)
      recurrent_kernel<DK, DV, __nv_bfloat16, true, false><<<grid, kThreads, 0, s>>>(a);
    else if (a.gate)
      recurrent_kernel<DK, DV, __nv_bfloat16, false, true><<<grid, kThreads, 0, s>>>(a);
    else
      recurrent_kernel<DK, DV, __nv_bfloat16, false, false><<<grid, kThreads, 0, s>>>(a);
  }
  return cudaGetLastError();
}

// Rank sort of sequence lengths (descending, ties by index), one CTA.
__global__ void length_order_kernel(const int* __restrict__ cu, int n, int* __restrict__ order) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const int li = cu[i + 1] - cu[i];
    int rank = 0;
    for (int j = 0; j < n; ++j) {
      const int lj = cu[j + 1] - cu[j];
      rank += (lj > li) || (lj == li && j < i);
    }
    order[rank] = i;
  }
}

__global__ void identity_order_kernel(int n, int* __restrict__ order) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) order[i] = i;
}

}  // namespace

cudaError_t launch_recurrent(const LaunchArgs& a, cudaStream_t s) {
  if (a.n_seqs == 0 || a.heads == 0) return cudaSuccess;
  if (a.dk == 128 && a.dv == 128) return launch_dims<128, 128>(a, s);
  if (a.dk == 64 && a.dv == 64) return launch_dims<64, 64>(a, s);
  if (a.dk == 128 && a.dv == 64) return launch_dims<128, 64>(a, s);
  if (a.dk == 64 && a.dv == 128) return launch_dims<64, 128>(a, s);
  return cudaErrorInvalidValue;
}

constexpr int kMaxSortedSeqs = 8192;

cudaError_t launch_length_order(const int* cu, int n, int* order, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (n <= kMaxSortedSeqs)
    length_order_kernel<<<1, 1024, 0, s>>>(cu, n, order);
  else
    identity_order_kernel<<<(n + 255) / 256, 256, 0, s>>>(n, order);
  return cudaGetLastError();
}

}  // namespace kda
