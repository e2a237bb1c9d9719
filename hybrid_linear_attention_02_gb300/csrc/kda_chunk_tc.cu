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
// log-decay of a 16-token tile above -80.  The masked intra-chunk products
// are therefore formed per 16-token row tile a with the reference point R_a
// (the cumulative decay where tile a starts): rows use k e^{G - R_a} <= 1 and
// keys use k e^{R_a - G} < e^80, both inside the bf16/fp32 range, and every
// product is one dense tensor-core MMA.
//
// One CTA (384 threads) owns one (sequence, head) and walks its chunks in
// order.  The work of a chunk splits into a state-independent "prep" part and
// the serial state pass, and the two run concurrently on different warps:
//   prep  (warps 4..11) for chunk c+1:  cumulative decay, scaled operand tiles,
//         AP = [K';Q'] x Khat^T (one M=128 N=160 K=128 MMA), A and P rows,
//         T = (I + A)^-1 in fp32, W^T = Ktil^T T'^T and U0^T = V^T T'^T
//         (T' = T diag(beta)), -W^T to shared memory.
//   state (warps 0..3) for chunk c:  U^T = U0^T + S^T(-W)^T, O^T = S^T Qtil^T;
//         S <- Diag(e^{G_C}) S (fp32, in TMEM);  U^T -> bf16 in TMEM;
//         S^T += U^T Kbar, O^T += U^T P^T;  S^T -> bf16 in TMEM;  O -> out.
// The fp32 state lives in tensor memory for the whole sequence (the MMA adds
// dS onto the decayed state); its bf16 copy and U^T are A operands read from
// tensor memory.  Every MMA is M = 128 (cta_group::1), bf16 x bf16 -> fp32.
// Handoffs use mbarriers (a two-slot ring for the per-chunk tiles the state
// pass consumes).  Every wait is bounded; on expiry the CTA stops issuing
// work, reports KDA_ERR_TIMEOUT and exits.
// Raw q, k, v, g tiles of the next chunk arrive by TMA into tiles that are
// dead at that point (k and v into the [K';Q'] tile once the masked-product
// MMA has read it, q and g into the Qtil / Kbar slot the next chunk will
// overwrite in place), so the prefetch costs no extra shared memory.
//
// Building with -DKDA_PHASE_PROFILE records per-phase SM-clock totals of
// CTA (0, 0) in the device array kda_phase_clocks (instrumentation only).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

using namespace sm100;

constexpr int kC = 64;
constexpr int kD = 128;
constexpr int kStateThreads = 128;                  // warps 0..3
constexpr int kPrepThreads = 256;                   // warps 4..11
constexpr int kThreads = kStateThreads + kPrepThreads;
constexpr float kLog2e = 1.4426950408889634f;

// Shared-memory tiles (byte offsets from a 1024-aligned base); bf16 tiles use
// the 128B-swizzled layout of sw128_off().
constexpr uint32_t kOffKQ = 0;                 // [K'_a; Q'_a] for a = 0..3   128 x 128
constexpr uint32_t kOffKH = kOffKQ + 32768;    // Khat blocks                 160 x 128
constexpr uint32_t kOffKT = kOffKH + 40960;    // Ktil = k e^G                 64 x 128
constexpr uint32_t kOffV = kOffKT + 16384;     // V                            64 x 128
constexpr uint32_t kOffTB = kOffV + 16384;     // T diag(beta)                 64 x 64
constexpr uint32_t kOffQT = kOffTB + 8192;     // Qtil = q e^G, 2 slots        64 x 128
constexpr uint32_t kOffKB = kOffQT + 32768;    // Kbar, 2 slots                64 x 128
constexpr uint32_t kOffWT = kOffKB + 32768;    // -W^T                        128 x 64
constexpr uint32_t kOffP = kOffWT + 16384;     // P, 2 slots                   64 x 64
constexpr uint32_t kOffO = kOffP + 16384;      // O staging (row-major bf16)   64 x 128
constexpr uint32_t kTileBytes = kOffO + 16384;
// Raw tiles of the next chunk (TMA destinations, same swizzled layout).
constexpr uint32_t kOffRawK = kOffKQ;          // 64 x 128, dead once AP is done
constexpr uint32_t kOffRawV = kOffKQ + 16384;  // 64 x 128
// (raw q and g land in the Qtil and Kbar slot of their chunk.)
// Per-chunk scan sums and Khat factors live in the T' tile until P5 writes it.
constexpr uint32_t kOffTileTot = kOffTB;       // fp32 [4][128]
constexpr uint32_t kOffFac = kOffTB + 2048;    // fp32 [4][3][128]
static_assert(2048 + 4 * 3 * 128 * 4 <= 8192, "scan sums and factors fit in the T' tile");
constexpr uint32_t kSmemBytes = kTileBytes + 1024;
// fp32 work matrices of the inverse reuse the Khat tile once AP is done.
constexpr int kLdA = 68;                                 // 16-byte aligned rows
constexpr uint32_t kOffA = kOffKH;                       // A  64 x 68
constexpr uint32_t kOffT = kOffA + 64 * kLdA * 4;        // T  64 x 68
constexpr uint32_t kOffX = kOffT + 64 * kLdA * 4;        // X  3 x 16 x 20
static_assert(kOffX + 3 * 16 * 20 * 4 <= kOffKH + 40960, "inverse scratch fits");

// TMEM columns (512 allocated).
constexpr uint32_t kColAP = 0;     // 160 fp32: AP;  W^T reuses columns 0..63
constexpr uint32_t kColW = 0;
constexpr uint32_t kColU = 160;    // 64 fp32: U0^T, then U^T
constexpr uint32_t kColO = 224;    // 64 fp32: O^T
constexpr uint32_t kColS = 288;    // 128 fp32: S^T (lane j = value column, col = key row)
constexpr uint32_t kColSB = 416;   // 64: bf16 S^T, A operand
constexpr uint32_t kColUT = 480;   // 32: bf16 U^T, A operand
constexpr uint32_t kTmemCols = 512;

enum { kBarAP = 0, kBarWU, kBarFull0, kBarFull1, kBarEmpty0, kBarEmpty1, kBarMMA1, kBarUFree,
       kBarMMA2, kBarRaw, kNumBars };

#ifdef KDA_PHASE_PROFILE
__device__ unsigned long long kda_phase_clocks[32];
#define KDA_MARK(i)                                   \
  do {                                                \
    const unsigned long long now_ = clock64();        \
    prof_acc[i] += now_ - prof_t;                     \
    prof_t = now_;                                    \
  } while (0)
#else
#define KDA_MARK(i) ((void)0)
#endif

__device__ __forceinline__ int khat_row0(int a) { return 8 * a * (a + 1); }  // 0, 16, 48, 96

__device__ __forceinline__ void named_bar(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
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

__device__ __forceinline__ void st_tile8(uint8_t* tile, int row, int col, int rows,
                                         const float (&f)[8]) {
  *reinterpret_cast<uint4*>(tile + sw128_off(row, col, rows)) =
      make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

// Shared by all roles: a wait that also gives up once any thread has given up.
struct Sync {
  uint64_t* bars;
  volatile int* abort;
  __device__ __forceinline__ bool wait(int b, uint32_t parity) {
    if (*abort) return false;
    if (mbar_try_wait(&bars[b], parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
      if (mbar_try_wait(&bars[b], parity)) return true;
      if ((it & 255u) == 0) {
        if (*abort) return false;
        if (global_timer_ns() - t0 > 2000000000ull) {
          *abort = 1;
          return false;
        }
      }
    }
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_kernel(LaunchArgs args, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ __align__(16) float s_gamma[2][kD];     // e^{G_C} per channel, per slot
  __shared__ float s_beta[kC];
  __shared__ uint64_t s_bars[kNumBars];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

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
  const int n_chunks = static_cast<int>((t1 - t0 + kC - 1) / kC);

  if (warp == 0) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < kNumBars; ++b) mbar_init(&s_bars[b], 1);
    s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;
  Sync sync{s_bars, &s_abort};
#ifdef KDA_PHASE_PROFILE
  unsigned long long prof_acc[16] = {}, prof_t = clock64();
#endif

  if (tid < kStateThreads) {
    // =============================== state pass ===============================
    const int j = tid;                                   // TMEM lane = value column
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    const long long soff = (static_cast<long long>(n) * H + h) * kD * kD;
    __nv_bfloat16* __restrict__ gout = static_cast<__nv_bfloat16*>(args.out);

    // S^T[j][c] = S[c][j]: fp32 copy and bf16 operand copy.
#pragma unroll 1
    for (int cb = 0; cb < 4; ++cb) {
      uint32_t f[32], b[16];
#pragma unroll
      for (int u = 0; u < 32; ++u)
        f[u] = __float_as_uint(args.init_state ? __ldcs(args.init_state + soff +
                                                        (32 * cb + u) * kD + j)
                                               : 0.f);
#pragma unroll
      for (int u = 0; u < 16; ++u)
        b[u] = pack2(__uint_as_float(f[2 * u]), __uint_as_float(f[2 * u + 1]));
      tmem_st32(tbase + lane_base + kColS + 32 * cb, f);
      tmem_st16(tbase + lane_base + kColSB + 16 * cb, b);
    }
    tmem_st_wait();
    tc_fence_before();
    named_bar(1, kStateThreads);

#pragma unroll 1
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c & 1;
      const long long c0 = t0 + static_cast<long long>(c) * kC;
      const int L = static_cast<int>(t1 - c0 < kC ? t1 - c0 : kC);
      const bool ok_full = sync.wait(kBarFull0 + s, (c >> 1) & 1);
      KDA_MARK(0);
      tc_fence_after();
      if (j == 0 && ok_full) {
        // U^T += S^T (-W)^T ;  O^T = S^T Qtil^T      (K = dk = 128)
        const uint32_t iU = umma_idesc_bf16(128, 64, 0, 1), iO = umma_idesc_bf16(128, 64, 0, 0);
        const uint32_t bW = smem_u32(smem + kOffWT), bQ = smem_u32(smem + kOffQT + s * 16384);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const uint32_t aS = tbase + kColSB + 8 * t;
          umma_bf16_tmem_a(tbase + kColU, aS, umma_desc(bW + t * 2048, 128 * 128, 1024), iU, 1);
          umma_bf16_tmem_a(tbase + kColO, aS,
                           umma_desc(bQ + (t >> 2) * 64 * 128 + (t & 3) * 32, 16, 1024), iO,
                           t > 0);
        }
        umma_commit(&s_bars[kBarMMA1]);
      }
      KDA_MARK(1);
      // Decay the fp32 state in place: S <- Diag(e^{G_C}) S (MMA1 does not read it).
      if (ok_full) {
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          float v[32];
          tmem_ld32(tbase + lane_base + kColS + 32 * cb, v);
          tmem_ld_wait();
          uint32_t f[32];
#pragma unroll
          for (int u = 0; u < 32; u += 4) {
            const float4 gm = *reinterpret_cast<const float4*>(&s_gamma[s][32 * cb + u]);
            f[u] = __float_as_uint(v[u] * gm.x);
            f[u + 1] = __float_as_uint(v[u + 1] * gm.y);
            f[u + 2] = __float_as_uint(v[u + 2] * gm.z);
            f[u + 3] = __float_as_uint(v[u + 3] * gm.w);
          }
          tmem_st32(tbase + lane_base + kColS + 32 * cb, f);
        }
      }
      const bool ok1 = sync.wait(kBarMMA1, c & 1);
      KDA_MARK(2);
      tc_fence_after();
      if (ok1) {
        // U^T (fp32) -> bf16 A operand.
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tmem_ld32(tbase + lane_base + kColU + 32 * half, v);
          tmem_ld_wait();
          uint32_t b[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) b[u] = pack2(v[2 * u], v[2 * u + 1]);
          tmem_st16(tbase + lane_base + kColUT + 16 * half, b);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      named_bar(1, kStateThreads);
      if (j == 0 && ok1 && !s_abort) {
        mbar_arrive(&s_bars[kBarUFree]);
        tc_fence_after();
        // S^T += U^T Kbar (K = 64 tokens) ;  O^T += U^T P^T
        const uint32_t iS = umma_idesc_bf16(128, 128, 0, 1), iO = umma_idesc_bf16(128, 64, 0, 0);
        const uint32_t bK = smem_u32(smem + kOffKB + s * 16384),
                       bP = smem_u32(smem + kOffP + s * 8192);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t aU = tbase + kColUT + 8 * t;
          umma_bf16_tmem_a(tbase + kColS, aU, umma_desc(bK + t * 2048, 64 * 128, 1024), iS, 1);
          umma_bf16_tmem_a(tbase + kColO, aU, umma_desc(bP + t * 32, 16, 1024), iO, 1);
        }
        umma_commit(&s_bars[kBarEmpty0 + s]);
        umma_commit(&s_bars[kBarMMA2]);
      }
      KDA_MARK(3);
      const bool ok2 = sync.wait(kBarMMA2, c & 1);
      KDA_MARK(4);
      tc_fence_after();
      float o0[32], o1[32];
      if (ok2) {
        // New state -> bf16 operand copy; O^T -> registers.
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          float v[32];
          tmem_ld32(tbase + lane_base + kColS + 32 * cb, v);
          tmem_ld_wait();
          uint32_t b[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) b[u] = pack2(v[2 * u], v[2 * u + 1]);
          tmem_st16(tbase + lane_base + kColSB + 16 * cb, b);
        }
        tmem_ld32(tbase + lane_base + kColO, o0);
        tmem_ld32(tbase + lane_base + kColO + 32, o1);
        tmem_ld_wait();
      }
      tmem_st_wait();
      tc_fence_before();
      named_bar(1, kStateThreads);
      KDA_MARK(5);
      // O^T column j -> row-major staging, then 16-byte rows to global memory.
      if (ok2) {
        __nv_bfloat16* so = reinterpret_cast<__nv_bfloat16*>(smem + kOffO) + j;
#pragma unroll
        for (int r = 0; r < 32; ++r) so[r * kD] = __float2bfloat16_rn(o0[r]);
#pragma unroll
        for (int r = 0; r < 32; ++r) so[(32 + r) * kD] = __float2bfloat16_rn(o1[r]);
      }
      named_bar(1, kStateThreads);
      if (ok2) {
        __nv_bfloat16* dst = gout + (c0 * H + h) * kD;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int e = j + kStateThreads * i, r = e >> 4, ch = e & 15;
          if (r < L)
            *reinterpret_cast<uint4*>(dst + static_cast<long long>(r) * H * kD + 8 * ch) =
                *reinterpret_cast<const uint4*>(smem + kOffO + r * 256 + ch * 16);
        }
      }
      KDA_MARK(6);
    }
#ifdef KDA_PHASE_PROFILE
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) {
      for (int i = 0; i < 8; ++i) kda_phase_clocks[i] = prof_acc[i];
      kda_phase_clocks[24] = n_chunks;
    }
#endif
    if (!s_abort && args.final_state) {
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        float v[32];
        tmem_ld32(tbase + lane_base + kColS + 32 * cb, v);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 32; ++u) __stcs(args.final_state + soff + (32 * cb + u) * kD + j, v[u]);
      }
    }
  } else {
    // ================================== prep ==================================
    const int p = tid - kStateThreads;          // 0..255
    const int pw = p >> 5;                      // prep warp 0..7
    const int ta = pw & 3;                      // this warp's 16-token row tile
    const int cg = 8 * (pw >> 2) + (lane & 7);  // channel group: channels 8 cg .. 8 cg + 7
    const int r4 = lane >> 3;                   // rows 16 ta + 4 r4 + m, m = 0..3
    const int row0 = 16 * ta + 4 * r4;
    const bool leader = p == 0;                 // issues the prep MMAs
    const bool loader = p == 128;               // issues the raw-tile TMA loads
    const __nv_bfloat16* __restrict__ gb = static_cast<const __nv_bfloat16*>(args.beta);
    float* Am = reinterpret_cast<float*>(smem + kOffA);
    float* Tm = reinterpret_cast<float*>(smem + kOffT);
    float* Xm = reinterpret_cast<float*>(smem + kOffX);
    float* tile_tot = reinterpret_cast<float*>(smem + kOffTileTot);  // [4][128]
    float* fac = reinterpret_cast<float*>(smem + kOffFac);           // [4][3][128]

    auto chunk_len = [&](int c) {
      const long long rem = t1 - (t0 + static_cast<long long>(c) * kC);
      return static_cast<int>(rem < kC ? rem : kC);
    };
    // Raw q, k, v, g of chunk c: two 64-channel boxes each, by TMA.
    auto issue_raw = [&](int c) {
      const int s = c & 1;
      const int c0 = static_cast<int>(t0 + static_cast<long long>(c) * kC);
      uint64_t* bar = &s_bars[kBarRaw];
      mbar_arrive_expect_tx(bar, 4 * 16384);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        tma_load_3d(smem + kOffRawK + hf * 8192, &tm_k, 64 * hf, h, c0, bar);
        tma_load_3d(smem + kOffRawV + hf * 8192, &tm_v, 64 * hf, h, c0, bar);
        tma_load_3d(smem + kOffQT + s * 16384 + hf * 8192, &tm_q, 64 * hf, h, c0, bar);
        tma_load_3d(smem + kOffKB + s * 16384 + hf * 8192, &tm_g, 64 * hf, h, c0, bar);
      }
    };
    // beta of chunk c: the 16 threads of channel group 0 hold 4 rows each.
    float rb[4];
    auto load_beta = [&](int c) {
      const long long c0 = t0 + static_cast<long long>(c) * kC;
      const int L = chunk_len(c);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int r = row0 + m;
        rb[m] = (cg == 0 && r < L) ? __bfloat162float(gb[(c0 + r) * H + h]) : 0.f;
      }
    };
    if (n_chunks > 0) {
      if (loader) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_g);
        issue_raw(0);
      }
      load_beta(0);
    }

#pragma unroll 1
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c & 1;
      const int L = chunk_len(c);
      const bool ok_raw = sync.wait(kBarRaw, c & 1);
      KDA_MARK(8);
      // Raw rows of this chunk (rows past the end of the sequence read as 0).
      uint4 rq[4], rk[4], rgt[4], rv[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int r = row0 + m;
        const uint32_t off = sw128_off(r, 8 * cg, 64);
        if (r < L && ok_raw) {
          rgt[m] = *reinterpret_cast<const uint4*>(smem + kOffKB + s * 16384 + off);
          rq[m] = *reinterpret_cast<const uint4*>(smem + kOffQT + s * 16384 + off);
          rk[m] = *reinterpret_cast<const uint4*>(smem + kOffRawK + off);
          rv[m] = *reinterpret_cast<const uint4*>(smem + kOffRawV + off);
        } else {
          rgt[m] = rq[m] = rk[m] = rv[m] = make_uint4(0, 0, 0, 0);
        }
      }
      // ---- P1: cumulative decay (log2 units) along the chunk, per channel.
      float G[4][8];
      {
        float gf[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          unpack8(rgt[m], gf);
#pragma unroll
          for (int u = 0; u < 8; ++u) G[m][u] = (m ? G[m - 1][u] : 0.f) + gf[u] * kLog2e;
        }
      }
      // Scan the four 4-row groups of this tile (lanes 8 apart), then across tiles.
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        float tot = G[3][u];
        float y = __shfl_up_sync(0xFFFFFFFFu, tot, 8);
        if (r4 >= 1) tot += y;
        y = __shfl_up_sync(0xFFFFFFFFu, tot, 16);
        if (r4 >= 2) tot += y;
        const float excl = tot - G[3][u];
#pragma unroll
        for (int m = 0; m < 4; ++m) G[m][u] += excl;
        if (r4 == 3) tile_tot[ta * kD + 8 * cg + u] = tot;
      }
      // Tile sums are visible, and every raw k / v read is done before the
      // [K';Q'] tile is rewritten.
      named_bar(2, kPrepThreads);
      float R[4][8], GC[8];
      {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int a = 0; a < 4; ++a) {
#pragma unroll
          for (int u = 0; u < 8; ++u) R[a][u] = acc[u];
          const float4 t0v = *reinterpret_cast<const float4*>(&tile_tot[a * kD + 8 * cg]);
          const float4 t1v = *reinterpret_cast<const float4*>(&tile_tot[a * kD + 8 * cg + 4]);
          acc[0] += t0v.x; acc[1] += t0v.y; acc[2] += t0v.z; acc[3] += t0v.w;
          acc[4] += t1v.x; acc[5] += t1v.y; acc[6] += t1v.z; acc[7] += t1v.w;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) GC[u] = acc[u];
      }
      float Ra[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        Ra[u] = ta == 0 ? R[0][u] : ta == 1 ? R[1][u] : ta == 2 ? R[2][u] : R[3][u];
#pragma unroll
        for (int m = 0; m < 4; ++m) G[m][u] += Ra[u];
      }

      // ---- P2: scaled operand tiles (packed fp32 pairs, one rounding each).
      {
        uint8_t* qt = smem + kOffQT + s * 16384;
        uint8_t* kb = smem + kOffKB + s * 16384;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int r = row0 + m;
          *reinterpret_cast<uint4*>(smem + kOffV + sw128_off(r, 8 * cg, 64)) = rv[m];
          if (cg == 0) s_beta[r] = rb[m];
        }
        uint64_t eR[4], eC[4], Rp[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          eR[w] = f2_pack(ex2_fast(Ra[2 * w]), ex2_fast(Ra[2 * w + 1]));
          eC[w] = f2_pack(ex2_fast(GC[2 * w] - Ra[2 * w]), ex2_fast(GC[2 * w + 1] - Ra[2 * w + 1]));
          Rp[w] = f2_pack(Ra[2 * w], Ra[2 * w + 1]);
        }
        // Khat factors for the later key blocks, e^{R_{a2} - R_ta} <= 1, shared
        // by the warp (all its lanes are in tile ta).
        if (r4 == 0) {
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            const int a2 = ta + 1 + i;
            if (a2 < 4) {
              float f8[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const float ra2 = a2 == 1 ? R[1][u] : a2 == 2 ? R[2][u] : R[3][u];
                f8[u] = ex2_fast(ra2 - Ra[u]);
              }
              float* fr = fac + (ta * 3 + i) * kD + 8 * cg;
              *reinterpret_cast<float4*>(fr) = make_float4(f8[0], f8[1], f8[2], f8[3]);
              *reinterpret_cast<float4*>(fr + 4) = make_float4(f8[4], f8[5], f8[6], f8[7]);
            }
          }
          if (ta == 0) {
#pragma unroll
            for (int u = 0; u < 8; ++u) s_gamma[s][8 * cg + u] = ex2_fast(GC[u]);
          }
        }
        __syncwarp();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int r = row0 + m, rl = 4 * r4 + m;
          const uint32_t kw[4] = {rk[m].x, rk[m].y, rk[m].z, rk[m].w};
          const uint32_t qw[4] = {rq[m].x, rq[m].y, rq[m].z, rq[m].w};
          uint32_t okp[4], oqp[4], okt[4], oqt[4], okh[4], okb[4];
          uint64_t kh[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint64_t kp = bf16x2_to_f2(kw[w]), qp = bf16x2_to_f2(qw[w]);
            float dx, dy;
            f2_unpack(f2_sub(f2_pack(G[m][2 * w], G[m][2 * w + 1]), Rp[w]), dx, dy);
            const uint64_t e1 = f2_pack(ex2_fast(dx), ex2_fast(dy));    // e^{G - R_ta} <= 1
            const uint64_t ei = f2_pack(ex2_fast(-dx), ex2_fast(-dy));  // e^{R_ta - G} < e^80
            const uint64_t k1 = f2_mul(kp, e1), q1 = f2_mul(qp, e1);
            okp[w] = f2_to_bf16x2(k1);
            oqp[w] = f2_to_bf16x2(q1);
            okt[w] = f2_to_bf16x2(f2_mul(k1, eR[w]));
            oqt[w] = f2_to_bf16x2(f2_mul(q1, eR[w]));
            kh[w] = f2_mul(kp, ei);
            okh[w] = f2_to_bf16x2(kh[w]);
            okb[w] = f2_to_bf16x2(f2_mul(kh[w], eC[w]));
          }
          auto st4 = [&](uint32_t off_tile, int row, int rows, const uint32_t (&v)[4]) {
            *reinterpret_cast<uint4*>(smem + off_tile + sw128_off(row, 8 * cg, rows)) =
                make_uint4(v[0], v[1], v[2], v[3]);
          };
          st4(kOffKQ, 32 * ta + rl, 128, okp);
          st4(kOffKQ, 32 * ta + 16 + rl, 128, oqp);
          st4(kOffKT, r, 64, okt);
          st4(kOffKH, khat_row0(ta) + r, 160, okh);
          if (ok_raw) {
            *reinterpret_cast<uint4*>(qt + sw128_off(r, 8 * cg, 64)) =
                make_uint4(oqt[0], oqt[1], oqt[2], oqt[3]);
            *reinterpret_cast<uint4*>(kb + sw128_off(r, 8 * cg, 64)) =
                make_uint4(okb[0], okb[1], okb[2], okb[3]);
          }
#pragma unroll
          for (int i = 0; i < 3; ++i) {
            if (ta + 1 + i < 4) {
              const float* fr = fac + (ta * 3 + i) * kD + 8 * cg;
              const float4 f0 = *reinterpret_cast<const float4*>(fr);
              const float4 f1 = *reinterpret_cast<const float4*>(fr + 4);
              const uint64_t fp[4] = {f2_pack(f0.x, f0.y), f2_pack(f0.z, f0.w),
                                      f2_pack(f1.x, f1.y), f2_pack(f1.z, f1.w)};
              uint32_t ox[4];
#pragma unroll
              for (int w = 0; w < 4; ++w) ox[w] = f2_to_bf16x2(f2_mul(kh[w], fp[w]));
              st4(kOffKH, khat_row0(ta + 1 + i) + r, 160, ox);
            }
          }
        }
      }
      if (c + 1 < n_chunks) load_beta(c + 1);
      fence_async_smem();
      named_bar(2, kPrepThreads);
      KDA_MARK(9);

      // ---- P3: every masked intra-chunk product in one MMA.
      if (leader && !s_abort) {
        tc_fence_after();
        const uint32_t idesc = umma_idesc_bf16(128, 160, 0, 0);
        const uint32_t aK = smem_u32(smem + kOffKQ), bK = smem_u32(smem + kOffKH);
#pragma unroll
        for (int t = 0; t < 8; ++t)
          umma_bf16(tbase + kColAP, umma_desc(aK + (t >> 2) * 128 * 128 + (t & 3) * 32, 16, 1024),
                    umma_desc(bK + (t >> 2) * 160 * 128 + (t & 3) * 32, 16, 1024), idesc, t > 0);
        umma_commit(&s_bars[kBarAP]);
      }
      const bool ok_ap = sync.wait(kBarAP, c & 1);
      KDA_MARK(10);
      tc_fence_after();
      // Prefetch the next chunk's raw tiles: AP has read [K';Q'], and the
      // Qtil / Kbar slot of chunk c + 1 is free once the state pass of chunk
      // c - 1 has finished its last MMA.
      if (loader && c + 1 < n_chunks && ok_ap) {
        const bool ok_e = c < 1 || sync.wait(kBarEmpty0 + ((c + 1) & 1), ((c - 1) >> 1) & 1);
        if (ok_e) issue_raw(c + 1);
      }

      // ---- P4: A (x beta, strictly lower; fp32) and P (lower inclusive; bf16).
      if (pw < 4 && ok_ap) {
        // TMEM lane quarter pw holds rows [K'_pw; Q'_pw].
        const int a = pw, rl = lane & 15, r = 16 * a + rl;
        const bool isP = lane >= 16;
        const float br = s_beta[r];
        uint8_t* ptile = smem + kOffP + s * 8192;
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
          float v[16];
          if (blk <= a) {
            tmem_ld16(tbase + (static_cast<uint32_t>(32 * pw) << 16) + kColAP + khat_row0(a) +
                          16 * blk,
                      v);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const int i = 16 * blk + u;
              v[u] = isP ? (i <= r ? v[u] : 0.f) : (i < r ? br * v[u] : 0.f);
            }
          } else {
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = 0.f;
          }
          if (isP) {
            if (ok_raw) {
#pragma unroll
              for (int h8 = 0; h8 < 2; ++h8) {
                float f8[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) f8[u] = v[8 * h8 + u];
                st_tile8(ptile, r, 16 * blk + 8 * h8, 64, f8);
              }
            }
          } else {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<float4*>(&Am[r * kLdA + 16 * blk + 4 * q4]) =
                  make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
          }
        }
      }
      tc_fence_before();
      named_bar(2, kPrepThreads);

      KDA_MARK(11);
      // ---- P5: T = (I + A)^-1 in fp32; T' = T diag(beta) as bf16.
      if (p < 64) {
        const int blk = p >> 4, jj = p & 15;
        const float* Ab = Am + 16 * blk * kLdA + 16 * blk;
        float x[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < rr; ++i) acc = fmaf(Ab[rr * kLdA + i], x[i], acc);
          x[rr] = rr == jj ? 1.f : (rr < jj ? 0.f : -acc);
        }
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) Tm[(16 * blk + rr) * kLdA + 16 * blk + jj] = x[rr];
      }
      named_bar(2, kPrepThreads);
#pragma unroll 1
      for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;
        const int bi = p >> 6, b = bi, a = b + d, rr = (p >> 2) & 15, q = p & 3;
        if (bi < nb) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int cc = b; cc < a; ++cc) {
            const float* arow = Am + (16 * a + rr) * kLdA + 16 * cc;
            const float* tcol = Tm + (16 * cc) * kLdA + 16 * b + 4 * q;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
              const float av = arow[u];
              const float4 tv = *reinterpret_cast<const float4*>(tcol + u * kLdA);
              acc.x = fmaf(av, tv.x, acc.x); acc.y = fmaf(av, tv.y, acc.y);
              acc.z = fmaf(av, tv.z, acc.z); acc.w = fmaf(av, tv.w, acc.w);
            }
          }
          *reinterpret_cast<float4*>(&Xm[(bi * 16 + rr) * 20 + 4 * q]) = acc;
        }
        named_bar(2, kPrepThreads);
        if (bi < nb) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          const float* trow = Tm + (16 * a + rr) * kLdA + 16 * a;
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const float tv = trow[u];
            const float4 xv = *reinterpret_cast<const float4*>(&Xm[(bi * 16 + u) * 20 + 4 * q]);
            acc.x = fmaf(tv, xv.x, acc.x); acc.y = fmaf(tv, xv.y, acc.y);
            acc.z = fmaf(tv, xv.z, acc.z); acc.w = fmaf(tv, xv.w, acc.w);
          }
          *reinterpret_cast<float4*>(&Tm[(16 * a + rr) * kLdA + 16 * b + 4 * q]) =
              make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        named_bar(2, kPrepThreads);
      }
#pragma unroll
      for (int e = p; e < 64 * 8; e += kPrepThreads) {
        const int r = e >> 3, i0 = (e & 7) * 8;
        float f8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = i0 + u;
          f8[u] = (i >> 4) <= (r >> 4) ? Tm[r * kLdA + i] * s_beta[i] : 0.f;
        }
        st_tile8(smem + kOffTB, r, i0, 64, f8);
      }
      fence_async_smem();
      named_bar(2, kPrepThreads);

      KDA_MARK(12);
      // ---- P6: W^T = Ktil^T T'^T and U0^T = V^T T'^T (U0 goes where the state
      // pass accumulates U, once it has read the previous chunk's U).
      const bool ok_u = c < 1 || sync.wait(kBarUFree, (c - 1) & 1);
      if (leader && ok_u && !s_abort) {
        tc_fence_after();
        const uint32_t idesc = umma_idesc_bf16(128, 64, 1, 0);
        const uint32_t aKT = smem_u32(smem + kOffKT), aV = smem_u32(smem + kOffV),
                       bT = smem_u32(smem + kOffTB);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint64_t bd = umma_desc(bT + t * 32, 16, 1024);
          umma_bf16(tbase + kColW, umma_desc(aKT + t * 2048, 64 * 128, 1024), bd, idesc, t > 0);
          umma_bf16(tbase + kColU, umma_desc(aV + t * 2048, 64 * 128, 1024), bd, idesc, t > 0);
        }
        umma_commit(&s_bars[kBarWU]);
      }
      const bool ok_wu = sync.wait(kBarWU, c & 1);
      // -W^T may overwrite the shared tile once the state pass's first MMA of
      // the previous chunk is done.
      const bool ok_m1 = c < 1 || sync.wait(kBarMMA1, (c - 1) & 1);
      KDA_MARK(13);
      tc_fence_after();

      // ---- P7: -W^T (rows = key channel, K = token) as an MN-major B operand.
      if (pw < 4 && ok_wu && ok_m1) {
        const int cc = 32 * pw + lane;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float w[32];
          tmem_ld32(tbase + (static_cast<uint32_t>(32 * pw) << 16) + kColW + 32 * half, w);
          tmem_ld_wait();
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            float f8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) f8[u] = -w[8 * q8 + u];
            st_tile8(smem + kOffWT, cc, 32 * half + 8 * q8, 128, f8);
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      named_bar(2, kPrepThreads);
      if (leader && !s_abort) mbar_arrive(&s_bars[kBarFull0 + s]);
      KDA_MARK(14);
    }
#ifdef KDA_PHASE_PROFILE
    if (blockIdx.x == 0 && blockIdx.y == 0 && p == 0)
      for (int i = 8; i < 16; ++i) kda_phase_clocks[i] = prof_acc[i];
#endif
  }

  tc_fence_before();
  __syncthreads();
  if (s_abort && tid == 0 && args.dev_status) atomicExch(args.dev_status, KDA_ERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}


// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// [T, H, 128] bf16 viewed as a 3-D tensor (channel, head, token); one box is
// 64 channels x 1 head x 64 tokens, 128B-swizzled, zero-filled past T.
bool make_token_map(CUtensorMap* map, const void* base, int heads, long long tokens) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kD), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(tokens)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kD) * 2,
                                 static_cast<cuuint64_t>(heads) * kD * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kC)};
  const cuuint32_t elem[3] = {1, 1, 1};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_supported(const LaunchArgs& a) {
  return a.dtype == KDA_BF16 && a.dk == kD && a.dv == kD && a.chunk == kC &&
         a.total_tokens < (1ll << 31);
}

cudaError_t launch_chunk_tc(const LaunchArgs& a, cudaStream_t stream) {
  if (a.n_seqs == 0 || a.heads == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(chunk_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  CUtensorMap maps[4] = {};
  if (a.total_tokens > 0) {
    const void* bases[4] = {a.q, a.k, a.v, a.g};
    for (int i = 0; i < 4; ++i)
      if (!make_token_map(&maps[i], bases[i], a.heads, a.total_tokens))
        return cudaErrorInvalidValue;
  }
  dim3 grid(a.n_seqs, a.heads);
  chunk_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(a, maps[0], maps[1], maps[2], maps[3]);
  return cudaGetLastError();
}

#ifdef KDA_PHASE_PROFILE
// Copies the phase totals of the last profiled launch to the host (build with
// -DKDA_PHASE_PROFILE only).
extern "C" KDA_API int kda_debug_phase_clocks(unsigned long long* host) {
  return static_cast<int>(
      cudaMemcpyFromSymbol(host, kda_phase_clocks, sizeof(unsigned long long) * 32));
}
#endif

}  // namespace kda
