// bf16 chunkwise KDA on tcgen05 tensor cores (dk = dv = 128, chunk C = 64).
//
// The chunkwise parallel form named in "[Paper Review] Kimi K3: Open Frontier
// Intelligence", section "Kimi Delta Attention (KDA)", written out from the
// recurrence.  For one (sequence, head) and one chunk of C tokens with state
// S0 entering it and G = inclusive cumulative sum of g along the chunk:
//   A  = strictly_lower(diag(beta) (k e^G)(k e^-G)^T),  T = (I + A)^-1
//   W  = T diag(beta) (k e^G),  U = T diag(beta) V - W S0
//   O  = (q e^G) S0 + lower_incl((q e^G)(k e^-G)^T) U
//   S_C = Diag(e^{G_C}) S0 + (k e^{G_C - G})^T U
// The same section's lower-bounded decay (g >= -5) keeps the cumulative
// log-decay of a 16-token tile above -80, so the masked intra-chunk products
// are formed per 16-token row tile a with the reference point R_a (the
// cumulative decay where tile a starts): rows use k e^{G - R_a} <= 1 and keys
// use k e^{R_a - G} < e^80, both inside the bf16/fp32 range.  Every product
// is then a dense tensor-core MMA, which is the point of that section.
//
// One CTA (256 threads) owns one (sequence, head) and walks its chunks in
// order with the fp32 state in registers (thread j of each warpgroup holds
// column j of S, half of the dk rows) and a bf16 copy of S^T in shared memory
// as the MMA operand.  Every MMA is M = 128 (cta_group::1) with bf16 operands
// and fp32 accumulators in TMEM:
//   AP  [K';Q'] (128 x dk)  x  Khat blocks (160 x dk)^T     -> A and P rows
//   W^T = Ktil^T (T')^T,   U0^T = V^T (T')^T                 (T' = T diag beta)
//   U^T = U0^T + S^T (-W)^T,   O^T = S^T Qtil^T
//   dS^T = U^T Kbar,   O^T += U^T P^T
// T = (I + A)^-1 is solved on CUDA cores in fp32 (16 x 16 diagonal blocks by
// forward substitution, then block merges).
#include <cuda_bf16.h>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory tiles (byte offsets from a 1024-aligned base).  bf16 tiles
// use the 128B-swizzled layout of sw128_off().
constexpr uint32_t kOffKQ = 0;                 // [K'; Q']        128 x 128
constexpr uint32_t kOffKH = kOffKQ + 32768;    // Khat blocks     160 x 128
constexpr uint32_t kOffKT = kOffKH + 40960;    // Ktil = k e^G     64 x 128
constexpr uint32_t kOffQT = kOffKT + 16384;    // Qtil = q e^G     64 x 128
constexpr uint32_t kOffKB = kOffQT + 16384;    // Kbar             64 x 128
constexpr uint32_t kOffV = kOffKB + 16384;     // V                64 x 128
constexpr uint32_t kOffP = kOffV + 16384;      // P                64 x 64
constexpr uint32_t kOffTB = kOffP + 8192;      // T diag(beta)     64 x 64
constexpr uint32_t kOffWT = kOffTB + 8192;     // -W^T            128 x 64
constexpr uint32_t kOffUT = kOffWT + 16384;    // U^T             128 x 64
constexpr uint32_t kOffS = kOffUT + 16384;     // S^T (bf16)      128 x 128
constexpr uint32_t kTileBytes = kOffS + 32768;
// fp32 work matrices and the output staging reuse tiles that are dead then.
constexpr int kLd = 65;                        // padded fp32 row length
constexpr uint32_t kOffA = kOffKH;             // A  64 x 65 fp32
constexpr uint32_t kOffT = kOffKH + 64 * kLd * 4;  // T 64 x 65 fp32
constexpr uint32_t kOffX = kOffKQ;             // merge scratch 64 x 65 fp32
constexpr uint32_t kOffO = kOffKQ;             // O staging 64 x 136 bf16
constexpr int kLdO = 136;
constexpr uint32_t kSmemBytes = kTileBytes + 1024;
static_assert(2 * 64 * kLd * 4 <= 40960, "A and T fit in the Khat tile");
static_assert(64 * kLdO * 2 <= 32768, "O staging fits in the [K';Q'] tile");

// TMEM columns (fp32, lane = M row).
constexpr uint32_t kColAP = 0;    // 160 columns
constexpr uint32_t kColW = 0;     // 64, after AP is read
constexpr uint32_t kColU = 64;    // 64
constexpr uint32_t kColDS = 0;    // 128, after W and U are read
constexpr uint32_t kColO = 160;   // 64
constexpr uint32_t kTmemCols = 256;

__device__ __forceinline__ int khat_block_row0(int a) { return 8 * a * (a + 1); }  // 0,16,48,96

__device__ __forceinline__ uint4 ldg16(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

__device__ __forceinline__ void st_tile8(uint8_t* tile, int row, int col, int rows,
                                         const float (&f)[8]) {
  *reinterpret_cast<uint4*>(tile + sw128_off(row, col, rows)) = pack8(f);
}

__device__ __forceinline__ void st_tile8_raw(uint8_t* tile, int row, int col, int rows, uint4 v) {
  *reinterpret_cast<uint4*>(tile + sw128_off(row, col, rows)) = v;
}

__global__ void __launch_bounds__(kThreads, 1) chunk_tc_kernel(LaunchArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ float s_gamma[kD];
  __shared__ float s_beta[kC];
  __shared__ uint64_t s_bar;
  __shared__ uint32_t s_tmem;

  const __nv_bfloat16* __restrict__ gq = static_cast<const __nv_bfloat16*>(args.q);
  const __nv_bfloat16* __restrict__ gk = static_cast<const __nv_bfloat16*>(args.k);
  const __nv_bfloat16* __restrict__ gv = static_cast<const __nv_bfloat16*>(args.v);
  const __nv_bfloat16* __restrict__ gg = static_cast<const __nv_bfloat16*>(args.g);
  const __nv_bfloat16* __restrict__ gb = static_cast<const __nv_bfloat16*>(args.beta);
  __nv_bfloat16* __restrict__ gout = static_cast<__nv_bfloat16*>(args.out);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = args.heads;
  const int h = blockIdx.y;
  const int n = args.order ? args.order[blockIdx.x] : static_cast<int>(blockIdx.x);
  long long t0, t1;
  if (args.cu_seqlens) {
    t0 = args.cu_seqlens[n];
    t1 = args.cu_seqlens[n + 1];
  } else {
    t0 = static_cast<long long>(n) * args.seq_len;
    t1 = t0 + args.seq_len;
  }

  if (warp == 0) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
  }

  // State: thread (sj, sh) holds S[c][sj] for c in [64 sh, 64 sh + 64).
  const int sj = tid & 127, sh = tid >> 7;
  const long long soff = (static_cast<long long>(n) * H + h) * kD * kD;
  float S[64];
#pragma unroll
  for (int i = 0; i < 64; ++i)
    S[i] = args.init_state ? __ldcs(args.init_state + soff + (64 * sh + i) * kD + sj) : 0.f;
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    float f[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) f[u] = S[8 * m + u];
    st_tile8(smem + kOffS, sj, 64 * sh + 8 * m, 128, f);
  }

  // Prep layout: thread (cg, rg) owns channels [8 cg, 8 cg + 8) of rows
  // [4 rg, 4 rg + 4); the 16 row groups of one channel group share a warp half.
  const int cg = tid >> 4, rg = tid & 15, ta = rg >> 2;
  const uint32_t kSeg = 0xFFFFFFFFu;

  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;
  uint32_t phase = 0;
  bool ok = true;

  auto wait_mma = [&]() -> bool {
    bool done = mbar_wait(&s_bar, phase);
    phase ^= 1u;
    done = __syncthreads_and(done) != 0;
    tc_fence_after();
    return done;
  };

  // Raw inputs of the current chunk, prefetched one chunk ahead.
  uint4 rq[4], rk[4], rgt[4], rv[4];
  float rb[4];
  auto load_chunk = [&](long long c0, int L) {
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int r = 4 * rg + m;
      if (r < L) {
        const long long off = ((c0 + r) * H + h) * kD + 8 * cg;
        rq[m] = ldg16(gq + off);
        rk[m] = ldg16(gk + off);
        rgt[m] = ldg16(gg + off);
        rv[m] = ldg16(gv + off);
        rb[m] = cg == 0 ? __bfloat162float(gb[(c0 + r) * H + h]) : 0.f;
      } else {
        rq[m] = rk[m] = rgt[m] = rv[m] = make_uint4(0, 0, 0, 0);
        rb[m] = 0.f;
      }
    }
  };

  const long long n_tok = t1 - t0;
  if (n_tok > 0) load_chunk(t0, static_cast<int>(n_tok < kC ? n_tok : kC));

  for (long long c0 = t0; c0 < t1 && ok; c0 += kC) {
    const int L = static_cast<int>((t1 - c0) < kC ? (t1 - c0) : kC);

    // ---- P1: cumulative log2-decay along the chunk, per channel.
    float G[4][8];
    {
      float gf[8];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        unpack8(rgt[m], gf);
#pragma unroll
        for (int j = 0; j < 8; ++j) G[m][j] = (m ? G[m - 1][j] : 0.f) + gf[j] * kLog2e;
      }
    }
    float incl[8], R[4][8], Rta[8], GC[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) incl[j] = G[3][j];
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float y = __shfl_up_sync(kSeg, incl[j], o, 16);
        if (rg >= o) incl[j] += y;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float excl = incl[j] - G[3][j];
#pragma unroll
      for (int m = 0; m < 4; ++m) G[m][j] += excl;
      R[0][j] = 0.f;
      R[1][j] = __shfl_sync(kSeg, incl[j], 3, 16);
      R[2][j] = __shfl_sync(kSeg, incl[j], 7, 16);
      R[3][j] = __shfl_sync(kSeg, incl[j], 11, 16);
      GC[j] = __shfl_sync(kSeg, incl[j], 15, 16);
      const float rt = __shfl_sync(kSeg, incl[j], (4 * ta + 15) & 15, 16);
      Rta[j] = ta ? rt : 0.f;  // reference of this thread's own row tile
    }

    // ---- P2: scaled operand tiles.
    {
      float eR[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) eR[j] = exp2f(Rta[j]);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int r = 4 * rg + m;
        float kf[8], qf[8], t1v[8], t2v[8];
        unpack8(rk[m], kf);
        unpack8(rq[m], qf);
        float e1[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) e1[j] = exp2f(G[m][j] - Rta[j]);
#pragma unroll
        for (int j = 0; j < 8; ++j) { t1v[j] = kf[j] * e1[j]; t2v[j] = qf[j] * e1[j]; }
        st_tile8(smem + kOffKQ, r, 8 * cg, 128, t1v);
        st_tile8(smem + kOffKQ, 64 + r, 8 * cg, 128, t2v);
#pragma unroll
        for (int j = 0; j < 8; ++j) { t1v[j] *= eR[j]; t2v[j] *= eR[j]; }
        st_tile8(smem + kOffKT, r, 8 * cg, 64, t1v);
        st_tile8(smem + kOffQT, r, 8 * cg, 64, t2v);
#pragma unroll
        for (int a2 = 0; a2 < 4; ++a2) {
          if (a2 < ta) continue;
#pragma unroll
          for (int j = 0; j < 8; ++j) t1v[j] = kf[j] * exp2f(R[a2][j] - G[m][j]);
          st_tile8(smem + kOffKH, khat_block_row0(a2) + r, 8 * cg, 160, t1v);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) t1v[j] = kf[j] * exp2f(GC[j] - G[m][j]);
        st_tile8(smem + kOffKB, r, 8 * cg, 64, t1v);
        st_tile8_raw(smem + kOffV, r, 8 * cg, 64, rv[m]);
        if (cg == 0) s_beta[r] = rb[m];
      }
      if (rg == 0) {
#pragma unroll
        for (int j = 0; j < 8; ++j) s_gamma[8 * cg + j] = exp2f(GC[j]);
      }
    }
    // Prefetch the next chunk's raw inputs (consumed at the top of the loop).
    if (c0 + kC < t1) {
      const long long rem = t1 - (c0 + kC);
      load_chunk(c0 + kC, static_cast<int>(rem < kC ? rem : kC));
    }
    fence_async_smem();
    __syncthreads();

    // ---- P3: masked intra-chunk products on the tensor cores.
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = umma_idesc_bf16(128, 160, 0, 0);
      const uint32_t aK = smem_u32(smem + kOffKQ), bK = smem_u32(smem + kOffKH);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t ad = umma_desc(aK + (s >> 2) * 128 * 128 + (s & 3) * 32, 16, 1024);
        const uint64_t bd = umma_desc(bK + (s >> 2) * 160 * 128 + (s & 3) * 32, 16, 1024);
        umma_bf16(tbase + kColAP, ad, bd, idesc, s > 0);
      }
      umma_commit(&s_bar);
    }
    // Zero the P tile while the MMA runs (only in-block entries get written).
    if (tid >= 128) {
      uint4* p = reinterpret_cast<uint4*>(smem + kOffP);
      for (int i = tid - 128; i < 8192 / 16; i += 128) p[i] = make_uint4(0, 0, 0, 0);
    }
    if (!(ok = wait_mma())) break;

    // ---- P4: read A (x beta, strictly lower) and P (lower inclusive).
    float* Am = reinterpret_cast<float*>(smem + kOffA);
    float* Tm = reinterpret_cast<float*>(smem + kOffT);
    float* Xm = reinterpret_cast<float*>(smem + kOffX);
    if (warp < 4) {
      const int row = tid;                 // TMEM lane
      const bool isP = row >= 64;
      const int r = row & 63, a = r >> 4;
      const int a0 = ((32 * warp) & 63) >> 4;  // first row tile of this warp
      const int lo = khat_block_row0(a0), hi = khat_block_row0(a0 + 1) + 16 * (a0 + 2);
      const int mylo = khat_block_row0(a), myn = 16 * (a + 1);
      const float br = s_beta[r];
      for (int cb = lo; cb < hi; cb += 16) {
        float v16[16];
        tmem_ld16(tmem_addr(tbase, 32 * warp, kColAP + cb), v16);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int i = cb + u - mylo;
          if (i < 0 || i >= myn) continue;
          if (!isP) {
            Am[r * kLd + i] = i < r ? br * v16[u] : 0.f;
          } else {
            const __nv_bfloat16 pv = __float2bfloat16_rn(i <= r ? v16[u] : 0.f);
            *reinterpret_cast<__nv_bfloat16*>(smem + kOffP + sw128_off(r, i, 64)) = pv;
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- P5: T = (I + A)^-1, fp32.
    if (tid < 64) {
      const int blk = tid >> 4, j = tid & 15;
      const float* Ab = Am + 16 * blk * kLd + 16 * blk;
      float x[16];
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < rr; ++i) acc = fmaf(Ab[rr * kLd + i], x[i], acc);
        x[rr] = rr == j ? 1.f : (rr < j ? 0.f : -acc);
      }
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) Tm[(16 * blk + rr) * kLd + 16 * blk + j] = x[rr];
    }
    __syncthreads();
#pragma unroll 1
    for (int d = 1; d < 4; ++d) {
      const int nel = (4 - d) * 256;
      for (int e = tid; e < nel; e += kThreads) {
        const int b = e >> 8, a = b + d, rr = (e >> 4) & 15, cc = e & 15;
        float acc = 0.f;
        for (int c = b; c < a; ++c) {
          const float* arow = Am + (16 * a + rr) * kLd + 16 * c;
          const float* tcol = Tm + (16 * c) * kLd + 16 * b + cc;
#pragma unroll
          for (int u = 0; u < 16; ++u) acc = fmaf(arow[u], tcol[u * kLd], acc);
        }
        Xm[(16 * a + rr) * kLd + 16 * b + cc] = acc;
      }
      __syncthreads();
      for (int e = tid; e < nel; e += kThreads) {
        const int b = e >> 8, a = b + d, rr = (e >> 4) & 15, cc = e & 15;
        const float* trow = Tm + (16 * a + rr) * kLd + 16 * a;
        const float* xcol = Xm + (16 * a) * kLd + 16 * b + cc;
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) acc = fmaf(trow[u], xcol[u * kLd], acc);
        Tm[(16 * a + rr) * kLd + 16 * b + cc] = -acc;
      }
      __syncthreads();
    }
    // T' = T diag(beta) as the bf16 B operand (rows r, K = i).
    for (int e = tid; e < 64 * 8; e += kThreads) {
      const int r = e >> 3, i0 = (e & 7) * 8;
      float f[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u;
        f[u] = (i >> 4) <= (r >> 4) ? Tm[r * kLd + i] * s_beta[i] : 0.f;
      }
      st_tile8(smem + kOffTB, r, i0, 64, f);
    }
    fence_async_smem();
    __syncthreads();

    // ---- P6: W^T = Ktil^T T'^T and U0^T = V^T T'^T.
    if (tid == 0) {
      tc_fence_after();
      const uint32_t idesc = umma_idesc_bf16(128, 64, 1, 0);
      const uint32_t aKT = smem_u32(smem + kOffKT), aV = smem_u32(smem + kOffV);
      const uint32_t bT = smem_u32(smem + kOffTB);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint64_t bd = umma_desc(bT + s * 32, 16, 1024);
        umma_bf16(tbase + kColW, umma_desc(aKT + s * 2048, 64 * 128, 1024), bd, idesc, s > 0);
        umma_bf16(tbase + kColU, umma_desc(aV + s * 2048, 64 * 128, 1024), bd, idesc, s > 0);
      }
      umma_commit(&s_bar);
    }
    if (!(ok = wait_mma())) break;

    // ---- P7: -W^T to shared memory (rows c, K = r) as an MN-major B operand.
    if (warp < 4) {
      const int c = tid;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float w32[32];
        tmem_ld32(tmem_addr(tbase, 32 * warp, kColW + 32 * half), w32);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float f[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) f[u] = -w32[8 * m + u];
          st_tile8(smem + kOffWT, c, 32 * half + 8 * m, 128, f);
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- P8: U^T += S^T (-W)^T;  O^T = S^T Qtil^T.
    if (tid == 0) {
      tc_fence_after();
      const uint32_t iU = umma_idesc_bf16(128, 64, 0, 1), iO = umma_idesc_bf16(128, 64, 0, 0);
      const uint32_t aS = smem_u32(smem + kOffS), bW = smem_u32(smem + kOffWT),
                     bQ = smem_u32(smem + kOffQT);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const uint64_t ad = umma_desc(aS + (s >> 2) * 128 * 128 + (s & 3) * 32, 16, 1024);
        umma_bf16(tbase + kColU, ad, umma_desc(bW + s * 2048, 128 * 128, 1024), iU, 1);
        umma_bf16(tbase + kColO, ad,
                  umma_desc(bQ + (s >> 2) * 64 * 128 + (s & 3) * 32, 16, 1024), iO, s > 0);
      }
      umma_commit(&s_bar);
    }
    if (!(ok = wait_mma())) break;

    // ---- P9: U^T to shared memory (rows j, K = i) as a K-major A operand.
    if (warp < 4) {
      const int j = tid;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float u32v[32];
        tmem_ld32(tmem_addr(tbase, 32 * warp, kColU + 32 * half), u32v);
        tmem_ld_wait();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          float f[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) f[u] = u32v[8 * m + u];
          st_tile8(smem + kOffUT, j, 32 * half + 8 * m, 128, f);
        }
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- P10: dS^T = U^T Kbar;  O^T += U^T P^T.
    if (tid == 0) {
      tc_fence_after();
      const uint32_t iS = umma_idesc_bf16(128, 128, 0, 1), iO = umma_idesc_bf16(128, 64, 0, 0);
      const uint32_t aU = smem_u32(smem + kOffUT), bKB = smem_u32(smem + kOffKB),
                     bP = smem_u32(smem + kOffP);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint64_t ad = umma_desc(aU + s * 32, 16, 1024);
        umma_bf16(tbase + kColDS, ad, umma_desc(bKB + s * 2048, 64 * 128, 1024), iS, s > 0);
        umma_bf16(tbase + kColO, ad, umma_desc(bP + s * 32, 16, 1024), iO, 1);
      }
      umma_commit(&s_bar);
    }
    if (!(ok = wait_mma())) break;

    // ---- P11: state update, bf16 state copy, outputs.
    {
      const uint32_t lane_base = 32 * (warp & 3);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float d32[32];
        tmem_ld32(tmem_addr(tbase, lane_base, kColDS + 64 * sh + 32 * half), d32);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const int i = 32 * half + u;
          S[i] = fmaf(s_gamma[64 * sh + i], S[i], d32[u]);
        }
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        float f[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) f[u] = S[8 * m + u];
        st_tile8(smem + kOffS, sj, 64 * sh + 8 * m, 128, f);
      }
      float o32[32];
      tmem_ld32(tmem_addr(tbase, lane_base, kColO + 32 * sh), o32);
      tmem_ld_wait();
      __nv_bfloat16* so = reinterpret_cast<__nv_bfloat16*>(smem + kOffO);
#pragma unroll
      for (int u = 0; u < 32; ++u) so[(32 * sh + u) * kLdO + sj] = __float2bfloat16_rn(o32[u]);
    }
    __syncthreads();
    for (int e = tid; e < 64 * 16; e += kThreads) {
      const int row = e >> 4, ch = e & 15;
      if (row < L) {
        const uint4 v = *reinterpret_cast<const uint4*>(smem + kOffO + row * kLdO * 2 + ch * 16);
        *reinterpret_cast<uint4*>(gout + ((c0 + row) * H + h) * kD + 8 * ch) = v;
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
  }

  if (!ok && tid == 0 && args.dev_status) atomicExch(args.dev_status, KDA_ERR_TIMEOUT);
  if (ok && args.final_state) {
#pragma unroll
    for (int i = 0; i < 64; ++i) __stcs(args.final_state + soff + (64 * sh + i) * kD + sj, S[i]);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

bool chunk_tc_supported(const LaunchArgs& a) {
  return a.dtype == KDA_BF16 && a.dk == kD && a.dv == kD && a.chunk == kC;
}

cudaError_t launch_chunk_tc(const LaunchArgs& a, cudaStream_t stream) {
  if (a.n_seqs == 0 || a.heads == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_seqs, a.heads);
  chunk_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kda
