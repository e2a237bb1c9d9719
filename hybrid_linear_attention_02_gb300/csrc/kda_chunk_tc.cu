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
//         T = (I + A)^-1 in fp32 (block Neumann form), W^T = Ktil^T T'^T and U0^T = V^T T'^T
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
// dead at that point (k into the [K';Q'] tile once the masked-product MMA has
// read it, v into the V tile once U0 is done, q and g into the Qtil / Kbar
// slot the next chunk overwrites in place), so the prefetch costs no extra
// shared memory.
//
// Building with -DKDA_PHASE_PROFILE records per-phase SM-clock totals of
// CTA (0, 0) in the device array kda_phase_clocks (instrumentation only).
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "kda_internal.h"
#include "kda_sm100.cuh"
#include "kda_chunk_common.cuh"

namespace kda {
namespace {

using namespace sm100;
using namespace chunk;

constexpr int kStateThreads = 128;                  // warps 0..3
constexpr int kPrepThreads = 256;                   // warps 4..11
constexpr int kThreads = kStateThreads + kPrepThreads;
// Register split: the block launches with 168 per thread (384 x 168 = 64512);
// the state warpgroup gives up 80 per thread and the two prep warpgroups take
// 40 more each (128 x 88 + 256 x 208 = 64512).
constexpr int kStateRegs = 88;
constexpr int kPrepRegs = 208;
static_assert(kStateThreads * kStateRegs + kPrepThreads * kPrepRegs <= kThreads * 168,
              "register split fits the launch allocation");

// Shared-memory tiles (byte offsets from a 1024-aligned base); bf16 tiles use
// the 128B-swizzled layout of sw128_off().
constexpr uint32_t kOffKQ = 0;                 // [K'_a; Q'_a] for a = 0..3   128 x 128
constexpr uint32_t kOffKH = kOffKQ + 32768;    // Khat blocks                 160 x 128
constexpr uint32_t kOffKT = kOffKH + 40960;    // Ktil = k e^G                 64 x 128
constexpr uint32_t kOffV = kOffKT + 16384;     // V                            64 x 128
constexpr uint32_t kOffTB = kOffV + 16384;     // T diag(beta)                 64 x 64
constexpr uint32_t kOffQT = kOffTB + 8192;     // Qtil = q e^G, 2 slots        64 x 128
constexpr uint32_t kOffKB = kOffQT + 32768;    // Kbar (fp16), 2 slots         64 x 128
constexpr uint32_t kOffWT = kOffKB + 32768;    // -W^T                        128 x 64
constexpr uint32_t kOffP = kOffWT + 16384;     // P (fp16), 2 slots            64 x 64
constexpr uint32_t kOffO = kOffP + 16384;      // O staging (row-major bf16)   64 x 128
constexpr uint32_t kTileBytes = kOffO + 16384;
// Raw tiles of the next chunk (TMA destinations, same swizzled layout): k in
// the [K';Q'] tile once AP has read it, v straight into the V tile, q and g in
// the Qtil and Kbar slot of their chunk (overwritten in place).
constexpr uint32_t kOffRawK = kOffKQ;          // 64 x 128
// Per-chunk tile sums and per-(tile, channel) factors live in the T' tile
// until P5 writes it; the Khat block factors in the chunk's P slot until P4.
constexpr uint32_t kOffTileTot = kOffTB;              // fp32 [4][128]
constexpr uint32_t kOffTabR = kOffTB + 2048;          // fp32 [2][4][128]
static_assert(2048 + 2 * 4 * 128 * 4 <= 8192, "tile sums and factors fit in the T' tile");
static_assert(6 * 128 * 4 <= 8192, "Khat factors fit in a P slot");
constexpr uint32_t kSmemBytes = kTileBytes + 1024;
// fp32 work matrices of the inverse reuse the Khat tile once AP is done.
constexpr int kLdA = 68;                                 // 16-byte aligned rows
constexpr uint32_t kOffA = kOffKH;                       // A     64 x 68
constexpr int kLdB = 20;                                 // 16 x 16 blocks, 16-byte rows
constexpr uint32_t kOffD = kOffA + 64 * kLdA * 4;        // D     4 x 16 x 20
constexpr uint32_t kOffN = kOffD + 4 * 16 * kLdB * 4;    // N     6 x 16 x 20
constexpr uint32_t kOffN2 = kOffN + 6 * 16 * kLdB * 4;   // N^2   3 x 16 x 20
constexpr uint32_t kOffN3 = kOffN2 + 3 * 16 * kLdB * 4;  // N^3   16 x 20
constexpr uint32_t kOffAt = kOffN3 + 16 * kLdB * 4;      // A_aa^T 4 x 16 x 20
static_assert(kOffAt + 4 * 16 * kLdB * 4 <= kOffKH + 40960, "inverse scratch fits");

// TMEM columns (512 allocated).
constexpr uint32_t kColAP = 0;     // 160 fp32: AP;  W^T reuses columns 0..63
constexpr uint32_t kColW = 0;
constexpr uint32_t kColU = 160;    // 64 fp32: U0^T, then U^T
constexpr uint32_t kColO = 224;    // 64 fp32: O^T
constexpr uint32_t kColS = 288;    // 128 fp32: S^T (lane j = value column, col = key row)
constexpr uint32_t kColSB = 416;   // 64: bf16 S^T, A operand
constexpr uint32_t kColUT = 480;   // 32: fp16 U^T, A operand
constexpr uint32_t kTmemCols = 512;

enum { kBarAP = 0, kBarWU, kBarFull0, kBarFull1, kBarEmpty0, kBarEmpty1, kBarMMA1, kBarUFree,
       kBarMMA2, kBarRaw, kBarRawV, kBarDrainS, kBarDrainP, kNumBars };

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
  unsigned long long prof_acc[24] = {}, prof_t = clock64();
#endif

  if (tid < kStateThreads) {
    // =============================== state pass ===============================
    regs_dec<kStateRegs>();
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

    // Outputs of chunk cc leave from the staging tile as 16-byte rows.
    auto store_out = [&](int cc) {
      const long long c0 = t0 + static_cast<long long>(cc) * kC;
      const int L = static_cast<int>(t1 - c0 < kC ? t1 - c0 : kC);
      __nv_bfloat16* dst = gout + (c0 * H + h) * kD;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = j + kStateThreads * i, r = e >> 4, ch = e & 15;
        if (r < L)
          *reinterpret_cast<uint4*>(dst + static_cast<long long>(r) * H * kD + 8 * ch) =
              *reinterpret_cast<const uint4*>(smem + kOffO + r * 256 + ch * 16);
      }
    };
    bool prev_ok = false;

#pragma unroll 1
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c & 1;
      const bool ok_full = sync.wait_warp(kBarFull0 + s, (c >> 1) & 1);
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
      // The previous chunk's outputs leave while MMA1 runs.
      if (c > 0 && prev_ok) store_out(c - 1);
      // Decay the fp32 state in place: S <- Diag(e^{G_C}) S (MMA1 does not read it).
      if (ok_full) {
#pragma unroll 1
        for (int cb = 0; cb < 8; ++cb) {
          float v[16];
          tmem_ld16(tbase + lane_base + kColS + 16 * cb, v);
          tmem_ld_wait();
          uint32_t f[16];
#pragma unroll
          for (int u = 0; u < 16; u += 4) {
            const float4 gm = *reinterpret_cast<const float4*>(&s_gamma[s][16 * cb + u]);
            f[u] = __float_as_uint(v[u] * gm.x);
            f[u + 1] = __float_as_uint(v[u + 1] * gm.y);
            f[u + 2] = __float_as_uint(v[u + 2] * gm.z);
            f[u + 3] = __float_as_uint(v[u + 3] * gm.w);
          }
          tmem_st16(tbase + lane_base + kColS + 16 * cb, f);
        }
      }
      const bool ok1 = sync.wait_warp(kBarMMA1, c & 1);
      KDA_MARK(2);
      tc_fence_after();
      if (ok1) {
        // U^T (fp32) -> fp16 A operand (Kbar and P are fp16 too: the state
        // update S += Kbar^T U carries U = v_new - v_old where a write
        // replaces an old value, far larger than the state it leaves, and
        // fp16 rounds it 8x finer than bf16).
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tmem_ld32(tbase + lane_base + kColU + 32 * half, v);
          tmem_ld_wait();
          uint32_t b[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) b[u] = pack2_f16(v[2 * u], v[2 * u + 1]);
          tmem_st16(tbase + lane_base + kColUT + 16 * half, b);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      named_bar(1, kStateThreads);
      if (j == 0 && ok1 && !s_abort) {
        mbar_arrive(&s_bars[kBarUFree]);
        tc_fence_after();
        // S^T += U^T Kbar (K = 64 tokens) ;  O^T += U^T P^T   (fp16 operands)
        const uint32_t iS = umma_idesc_f16(128, 128, 0, 1), iO = umma_idesc_f16(128, 64, 0, 0);
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
      const bool ok2 = sync.wait_warp(kBarMMA2, c & 1);
      KDA_MARK(4);
      tc_fence_after();
      if (ok2) {
        // Prefix-cache checkpoint after this chunk (full chunks whose end is a
        // multiple of the checkpoint interval).
        const long long done = static_cast<long long>(c + 1) * kC;
        float* ck = nullptr;
        if (args.ckpt && done <= t1 - t0 && done % args.ckpt_interval == 0) {
          const long long row = args.ckpt_offsets[n] + done / args.ckpt_interval - 1;
          ck = args.ckpt + (row * H + h) * kD * kD + j;
        }
        // New state -> bf16 operand copy; O^T column j -> row-major staging.
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          float v[32];
          tmem_ld32(tbase + lane_base + kColS + 32 * cb, v);
          tmem_ld_wait();
          if (ck) {
#pragma unroll
            for (int u = 0; u < 32; ++u) __stcs(ck + (32 * cb + u) * kD, v[u]);
          }
          uint32_t b[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) b[u] = pack2(v[2 * u], v[2 * u + 1]);
          tmem_st16(tbase + lane_base + kColSB + 16 * cb, b);
        }
        __nv_bfloat16* so = reinterpret_cast<__nv_bfloat16*>(smem + kOffO) + j;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          float v[32];
          tmem_ld32(tbase + lane_base + kColO + 32 * half, v);
          tmem_ld_wait();
#pragma unroll
          for (int r = 0; r < 32; ++r) so[(32 * half + r) * kD] = __float2bfloat16_rn(v[r]);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      named_bar(1, kStateThreads);
      prev_ok = ok2;
      KDA_MARK(5);
    }
    if (n_chunks > 0 && prev_ok) store_out(n_chunks - 1);
#ifdef KDA_PHASE_PROFILE
    if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) {
      for (int i = 0; i < 8; ++i) kda_phase_clocks[i] = prof_acc[i];
      kda_phase_clocks[28] = n_chunks;
    }
#endif
    if (__all_sync(0xFFFFFFFFu, !s_abort) && args.final_state) {
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        float v[32];
        tmem_ld32(tbase + lane_base + kColS + 32 * cb, v);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 32; ++u) __stcs(args.final_state + soff + (32 * cb + u) * kD + j, v[u]);
      }
    }
    // After an abort, MMAs whose commit nobody waited for complete before
    // the block frees its TMEM (bounded).
    if (s_abort && j == 0) {
      umma_commit(&s_bars[kBarDrainS]);
      mbar_wait(&s_bars[kBarDrainS], 0, 100000000ull);
    }
  } else {
    // ================================== prep ==================================
    regs_inc<kPrepRegs>();
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
    float* Dm = reinterpret_cast<float*>(smem + kOffD);      // [4][16][kLdB]  T_aa
    float* Nm = reinterpret_cast<float*>(smem + kOffN);      // [6][16][kLdB]  T_aa A_ab
    float* N2m = reinterpret_cast<float*>(smem + kOffN2);    // [3][16][kLdB]
    float* N3m = reinterpret_cast<float*>(smem + kOffN3);    // [16][kLdB]
    float* Atm = reinterpret_cast<float*>(smem + kOffAt);    // [4][16][kLdB]  A_aa^T
    float* tile_tot = reinterpret_cast<float*>(smem + kOffTileTot);  // [4][128]
    float* tabR = reinterpret_cast<float*>(smem + kOffTabR);  // e^{R_a}, e^{G_C - R_a}: [2][4][128]

    auto chunk_len = [&](int c) {
      const long long rem = t1 - (t0 + static_cast<long long>(c) * kC);
      return static_cast<int>(rem < kC ? rem : kC);
    };
    // Raw k, q, g of chunk c (two 64-channel boxes each), by TMA.
    auto issue_raw = [&](int c) {
      const int s = c & 1;
      const int c0 = static_cast<int>(t0 + static_cast<long long>(c) * kC);
      uint64_t* bar = &s_bars[kBarRaw];
      mbar_arrive_expect_tx(bar, 3 * 16384);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        tma_load_3d(smem + kOffRawK + hf * 8192, &tm_k, 64 * hf, h, c0, bar);
        tma_load_3d(smem + kOffQT + s * 16384 + hf * 8192, &tm_q, 64 * hf, h, c0, bar);
        tma_load_3d(smem + kOffKB + s * 16384 + hf * 8192, &tm_g, 64 * hf, h, c0, bar);
      }
    };
    // Raw v of chunk c straight into the V operand tile.
    auto issue_raw_v = [&](int c) {
      const int c0 = static_cast<int>(t0 + static_cast<long long>(c) * kC);
      uint64_t* bar = &s_bars[kBarRawV];
      mbar_arrive_expect_tx(bar, 16384);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
        tma_load_3d(smem + kOffV + hf * 8192, &tm_v, 64 * hf, h, c0, bar);
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
    int last_raw = -1, last_rawv = -1;   // loader: last chunk its raw copies were issued for
    if (n_chunks > 0) {
      if (loader) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_g);
        if (!(args.debug_withhold == 3 && blockIdx.x == 0 && blockIdx.y == 0)) {
          issue_raw(0);   // (self-test: withheld, so the first raw tiles never arrive)
          last_raw = 0;
        }
        issue_raw_v(0);
        last_rawv = 0;
      }
      load_beta(0);
    }

#pragma unroll 1
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c & 1;
      const int L = chunk_len(c);
      // beta of this chunk to shared memory; the next chunk's load is in flight
      // for the whole iteration.
#pragma unroll
      for (int m = 0; m < 4; ++m)
        if (cg == 0) s_beta[row0 + m] = rb[m];
      if (c + 1 < n_chunks) load_beta(c + 1);
      const bool ok_raw = sync.wait_warp(kBarRaw, c & 1);
      KDA_MARK(8);
      // Raw rows of this chunk (rows past the end of the sequence read as 0).
      uint4 rq[4], rk[4];
      float G[4][8];
      {
        uint4 rgt[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int r = row0 + m;
          const uint32_t off = sw128_off(r, 8 * cg, 64);
          if (r < L && ok_raw) {
            rgt[m] = *reinterpret_cast<const uint4*>(smem + kOffKB + s * 16384 + off);
            rq[m] = *reinterpret_cast<const uint4*>(smem + kOffQT + s * 16384 + off);
            rk[m] = *reinterpret_cast<const uint4*>(smem + kOffRawK + off);
          } else {
            rgt[m] = rq[m] = rk[m] = make_uint4(0, 0, 0, 0);
          }
        }
        // ---- P1: decay accumulated from the start of this 16-token tile
        // (log2 units): G = cumsum(g) - R_ta, the exponent e1 and ei need.
        float gf[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          unpack8(rgt[m], gf);
#pragma unroll
          for (int u = 0; u < 8; ++u) G[m][u] = (m ? G[m - 1][u] : 0.f) + gf[u] * kLog2e;
        }
      }
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
      // Tile sums are visible, and every raw k read is done before the
      // [K';Q'] tile is rewritten.
      named_bar(2, kPrepThreads);
      // ---- Per-(tile, channel) factors, once per chunk (thread p <-> channel p):
      // e^{R_a}, e^{G_C - R_a}, the Khat block factors e^{R_{a2} - R_a}
      // (a2 > a) and e^{G_C}.  Split layout: entry c of a 128-vector sits at
      // (c & 4 ? 64 : 0) + 4 (c >> 3) + (c & 3), so the 16-byte reads of the
      // row loop are conflict-free.
      float* facs = reinterpret_cast<float*>(smem + kOffP + s * 8192);  // [6][128]
      if (p < kD) {
        const int cc = p;
        const int sc = (cc & 4 ? 64 : 0) + 4 * (cc >> 3) + (cc & 3);
        float tt[4], R[4], acc = 0.f;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          tt[a] = tile_tot[a * kD + cc];
          R[a] = acc;
          acc += tt[a];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          tabR[a * kD + sc] = ex2_fast(R[a]);
          tabR[(4 + a) * kD + sc] = ex2_fast(acc - R[a]);
        }
        // factor rows: (a, a2) = (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
        facs[0 * kD + sc] = ex2_fast(R[1] - R[0]);
        facs[1 * kD + sc] = ex2_fast(R[2] - R[0]);
        facs[2 * kD + sc] = ex2_fast(R[3] - R[0]);
        facs[3 * kD + sc] = ex2_fast(R[2] - R[1]);
        facs[4 * kD + sc] = ex2_fast(R[3] - R[1]);
        facs[5 * kD + sc] = ex2_fast(R[3] - R[2]);
        s_gamma[s][cc] = ex2_fast(acc);
      }
      named_bar(2, kPrepThreads);
      KDA_MARK(15);

      // ---- P2: scaled operand tiles (packed fp32 pairs, one rounding each).
      {
        uint8_t* qt = smem + kOffQT + s * 16384;
        uint8_t* kb = smem + kOffKB + s * 16384;
        const int sc0 = 4 * cg;  // split-layout index of channels 8cg..8cg+3 (+64: 8cg+4..)
        auto ld8 = [&](const float* t, uint64_t (&o)[4]) {
          const float4 lo = *reinterpret_cast<const float4*>(t + sc0);
          const float4 hi = *reinterpret_cast<const float4*>(t + 64 + sc0);
          o[0] = f2_pack(lo.x, lo.y);
          o[1] = f2_pack(lo.z, lo.w);
          o[2] = f2_pack(hi.x, hi.y);
          o[3] = f2_pack(hi.z, hi.w);
        };
        uint64_t eR[4], eC[4];
        ld8(tabR + ta * kD, eR);
        ld8(tabR + (4 + ta) * kD, eC);
        auto st4 = [&](uint32_t off_tile, int row, int rows, const uint32_t (&v)[4]) {
          *reinterpret_cast<uint4*>(smem + off_tile + sw128_off(row, 8 * cg, rows)) =
              make_uint4(v[0], v[1], v[2], v[3]);
        };
        uint64_t kh[4][4];   // Khat rows of this thread (fp32 pairs), for the later blocks
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int r = row0 + m, rl = 4 * r4 + m;
          const uint32_t kw[4] = {rk[m].x, rk[m].y, rk[m].z, rk[m].w};
          const uint32_t qw[4] = {rq[m].x, rq[m].y, rq[m].z, rq[m].w};
          uint32_t okp[4], oqp[4], okt[4], oqt[4], okh[4], okb[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint64_t kp = bf16x2_to_f2(kw[w]), qp = bf16x2_to_f2(qw[w]);
            const float dx = G[m][2 * w], dy = G[m][2 * w + 1];
            const uint64_t e1 = f2_pack(ex2_fast(dx), ex2_fast(dy));    // e^{G - R_ta} <= 1
            const uint64_t ei = f2_pack(ex2_fast(-dx), ex2_fast(-dy));  // e^{R_ta - G} < e^80
            const uint64_t k1 = f2_mul(kp, e1), q1 = f2_mul(qp, e1);
            okp[w] = f2_to_bf16x2(k1);
            oqp[w] = f2_to_bf16x2(q1);
            okt[w] = f2_to_bf16x2(f2_mul(k1, eR[w]));
            oqt[w] = f2_to_bf16x2(f2_mul(q1, eR[w]));
            kh[m][w] = f2_mul(kp, ei);
            okh[w] = f2_to_bf16x2(kh[m][w]);
            okb[w] = f2_to_f16x2(f2_mul(kh[m][w], eC[w]));
          }
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
        }
        // Later key blocks a2 > ta: Khat e^{R_a2 - R_ta}.
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          const int a2 = ta + 1 + i;
          if (a2 < 4) {
            const int frow = ta == 0 ? a2 - 1 : ta == 1 ? a2 + 1 : 5;
            uint64_t f[4];
            ld8(facs + frow * kD, f);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              uint32_t ox[4];
#pragma unroll
              for (int w = 0; w < 4; ++w) ox[w] = f2_to_bf16x2(f2_mul(kh[m][w], f[w]));
              st4(kOffKH, khat_row0(a2) + row0 + m, 160, ox);
            }
          }
        }
      }
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
      const bool ok_ap = sync.wait_warp(kBarAP, c & 1);
      KDA_MARK(10);
      tc_fence_after();
      // Prefetch the next chunk's raw k, q, g: AP has read [K';Q'], and the
      // Qtil / Kbar slot of chunk c + 1 is free once the state pass of chunk
      // c - 1 has finished its last MMA.
      if (loader && c + 1 < n_chunks && ok_ap) {
        const bool ok_e = c < 1 || sync.wait(kBarEmpty0 + ((c + 1) & 1), ((c - 1) >> 1) & 1);
        if (ok_e) {
          issue_raw(c + 1);
          last_raw = c + 1;
        }
      }

      // ---- P4: A (x beta, strictly lower; fp32) and P (lower inclusive; bf16).
      // Warps pw and pw + 4 share row tile pw & 3 (the same TMEM lanes): the
      // first takes column blocks 0 and 2, the second 1 and 3.  A's blocks
      // above the diagonal are never read, so only P's are written (as zeros);
      // A's diagonal blocks go out transposed, and the warp that holds one also
      // inverts it (P5's diagonal blocks).  The blocks of T' above the diagonal
      // are zeroed first (the factor tables there are dead).
      for (int e = p; e < 192; e += kPrepThreads) {
        const int pb = e >> 5, rr = (e >> 1) & 15, h8 = e & 1;
        const int a = pb < 3 ? 0 : pb < 5 ? 1 : 2;
        const int b = pb < 3 ? pb + 1 : pb < 5 ? pb - 1 : 3;
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        st_tile8(smem + kOffTB, 16 * a + rr, 16 * b + 8 * h8, 64, z);
      }
      if (ok_ap) {
        // TMEM lane quarter pw & 3 holds rows [K'_a; Q'_a].
        const int a = pw & 3, b0 = pw >> 2, rl = lane & 15, r = 16 * a + rl;
        const bool isP = lane >= 16;
        const float br = s_beta[r];
        uint8_t* ptile = smem + kOffP + s * 8192;
#pragma unroll
        for (int jb = 0; jb < 2; ++jb) {
          const int blk = b0 + 2 * jb;
          float v[16];
          if (blk <= a) {
            tmem_ld16(tbase + (static_cast<uint32_t>(32 * a) << 16) + kColAP + khat_row0(a) +
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
#pragma unroll
            for (int h8 = 0; h8 < 2; ++h8) {
              float f8[8];
#pragma unroll
              for (int u = 0; u < 8; ++u) f8[u] = v[8 * h8 + u];
              st_tile8_f16(ptile, r, 16 * blk + 8 * h8, 64, f8);
            }
          } else if (blk == a) {
#pragma unroll
            for (int u = 0; u < 16; ++u) Atm[(16 * a + u) * kLdB + rl] = v[u];
          } else if (blk < a) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              *reinterpret_cast<float4*>(&Am[r * kLdA + 16 * blk + 4 * q4]) =
                  make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
          }
        }
        // D_aa = (I + A_aa)^-1, column jj = lane by right-looking substitution:
        // once x_i is final it is taken off every later row, so the dependent
        // chain is one FMA per row.  Column i of A_aa is row i of its
        // transposed copy (the 16 lanes read the same words).
        __syncwarp();
        if (b0 == (a & 1) && lane < 16) {
          const int jj = lane;
          const float* At = Atm + 16 * a * kLdB;
          float y[16];
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) y[rr] = rr == jj ? 1.f : 0.f;
#pragma unroll
          for (int i = 0; i < 15; ++i) {
            const float xi = y[i];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if (4 * q + 3 > i) {
                const float4 w4 = *reinterpret_cast<const float4*>(At + i * kLdB + 4 * q);
                const float a4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  if (4 * q + u > i) y[4 * q + u] = fmaf(-a4[u], xi, y[4 * q + u]);
              }
            }
          }
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) Dm[(a * 16 + rr) * kLdB + jj] = y[rr];
        }
      }
      tc_fence_before();
      named_bar(2, kPrepThreads);
      KDA_MARK(11);

      // ---- P5: T = (I + A)^-1 in fp32, written as T' = T diag(beta) in bf16.
      // With D = blockdiag of the inverted 16 x 16 diagonal blocks and
      // N = D (strictly block-lower part of A), T = (I - N + N^2 - N^3) D.
      // Off-diagonal block pairs (a, b), a > b, are numbered
      // (1,0)=0 (2,0)=1 (2,1)=2 (3,0)=3 (3,1)=4 (3,2)=5; D is done (P4).  Block
      // products are 16 x 16 x 16, one warp each.
      KDA_MARK(16);
      // Block products, one warp per 16 x 16 x 16 product on warp-level tf32
      // tensor-core MMAs (m16n8k8, fp32 accumulate): acc[i] holds row
      // mg + 8 (i & 1), columns 8 (i >> 1) + 2 mt, + 1 of the output block.
      const int mg = (p & 31) >> 2, mt = p & 3;
      auto prod16 = [&](const float* X, int xs, const float* Y, int ys, float (&acc)[4][2]) {
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
          const uint32_t a0 = tf32_rna(X[mg * xs + 8 * ks + mt]);
          const uint32_t a1 = tf32_rna(X[(mg + 8) * xs + 8 * ks + mt]);
          const uint32_t a2 = tf32_rna(X[mg * xs + 8 * ks + mt + 4]);
          const uint32_t a3 = tf32_rna(X[(mg + 8) * xs + 8 * ks + mt + 4]);
#pragma unroll
          for (int nh = 0; nh < 2; ++nh) {
            const uint32_t b0 = tf32_rna(Y[(8 * ks + mt) * ys + 8 * nh + mg]);
            const uint32_t b1 = tf32_rna(Y[(8 * ks + mt + 4) * ys + 8 * nh + mg]);
            mma_m16n8k8_tf32(acc[2 * nh][0], acc[2 * nh][1], acc[2 * nh + 1][0],
                             acc[2 * nh + 1][1], a0, a1, a2, a3, b0, b1);
          }
        }
      };
      auto store_blk = [&](float* Z, const float (&acc)[4][2]) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<float2*>(Z + (mg + 8 * (i & 1)) * kLdB + 8 * (i >> 1) + 2 * mt) =
              make_float2(acc[i][0], acc[i][1]);
      };
      // Step 1: N_ab = D_aa A_ab (warps 0..5); diagonal blocks of T' (warps 6, 7).
      if (pw < 6) {
        const int blk = pw;
        const int a = blk < 1 ? 1 : blk < 3 ? 2 : 3;
        const int b = blk - (a * (a - 1)) / 2;
        float acc[4][2] = {};
        prod16(Dm + a * 16 * kLdB, kLdB, Am + 16 * a * kLdA + 16 * b, kLdA, acc);
        store_blk(Nm + blk * 16 * kLdB, acc);
      } else {
        for (int e = p - 192; e < 128; e += 64) {
          const int a = e >> 5, rr = (e >> 1) & 15, h8 = e & 1;
          float f8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int cc = 8 * h8 + u;
            f8[u] = Dm[(a * 16 + rr) * kLdB + cc] * s_beta[16 * a + cc];
          }
          st_tile8(smem + kOffTB, 16 * a + rr, 16 * a + 8 * h8, 64, f8);
        }
      }
      named_bar(2, kPrepThreads);
      KDA_MARK(17);
      // Step 2: N^2 blocks (2,0) = N21 N10, (3,1) = N32 N21, (3,0) = N31 N10 + N32 N20.
      if (pw < 3) {
        const int k2 = pw;
        float acc[4][2] = {};
        const int xa = k2 == 0 ? 2 : k2 == 1 ? 5 : 4, ya = k2 == 0 ? 0 : k2 == 1 ? 2 : 0;
        prod16(Nm + xa * 16 * kLdB, kLdB, Nm + ya * 16 * kLdB, kLdB, acc);
        if (k2 == 2) prod16(Nm + 5 * 16 * kLdB, kLdB, Nm + 1 * 16 * kLdB, kLdB, acc);
        store_blk(N2m + k2 * 16 * kLdB, acc);
      }
      named_bar(2, kPrepThreads);
      KDA_MARK(18);
      // Step 3: N^3 block (3,0) = N32 (N^2)_20 (warp 0), and M = -N + N^2 in
      // place of N for blocks (1,0) (2,0) (2,1) (3,1) (warps 1..7); N32, which
      // warp 0 reads, is negated in step 4 and M_30 is finished there too.
      if (pw == 0) {
        float acc[4][2] = {};
        prod16(Nm + 5 * 16 * kLdB, kLdB, N2m, kLdB, acc);
        store_blk(N3m, acc);
      } else {
        for (int e = p - 32; e < 4 * 64; e += kPrepThreads - 32) {
          const int bsel = e >> 6;                          // blocks 0, 1, 2, 4
          const int blk = bsel < 3 ? bsel : 4;
          const int k2 = blk == 1 ? 0 : blk == 4 ? 1 : -1;
          const int row = (e >> 2) & 15, q = e & 3;
          float4* nv = reinterpret_cast<float4*>(Nm + (blk * 16 + row) * kLdB + 4 * q);
          float4 m = *nv;
          m.x = -m.x; m.y = -m.y; m.z = -m.z; m.w = -m.w;
          if (k2 >= 0) {
            const float4 n2 = *reinterpret_cast<const float4*>(N2m + (k2 * 16 + row) * kLdB + 4 * q);
            m.x += n2.x; m.y += n2.y; m.z += n2.z; m.w += n2.w;
          }
          *nv = m;
        }
      }
      named_bar(2, kPrepThreads);
      KDA_MARK(19);
      // Step 4: T_ab = M_ab D_bb, times beta, into T' (warps 0..5; M_30 =
      // -N30 + N^2_30 - N^3_30 first, M_32 = -N_32).
      if (pw < 6) {
        const int blk = pw;
        const int a = blk < 1 ? 1 : blk < 3 ? 2 : 3;
        const int b = blk - (a * (a - 1)) / 2;
        if (blk == 3) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int row = mg + 8 * (i & 1), col = 8 * (i >> 1) + 2 * mt;
            float2* nv = reinterpret_cast<float2*>(Nm + (3 * 16 + row) * kLdB + col);
            const float2 n2 = *reinterpret_cast<const float2*>(N2m + (2 * 16 + row) * kLdB + col);
            const float2 n3 = *reinterpret_cast<const float2*>(N3m + row * kLdB + col);
            float2 m = *nv;
            m.x = n2.x - m.x - n3.x;
            m.y = n2.y - m.y - n3.y;
            *nv = m;
          }
          __syncwarp();
        }
        float acc[4][2] = {};
        prod16(Nm + blk * 16 * kLdB, kLdB, Dm + b * 16 * kLdB, kLdB, acc);
        const float sg = blk == 5 ? -1.f : 1.f;   // M_32 = -N_32
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = mg + 8 * (i & 1), col = 8 * (i >> 1) + 2 * mt;
          const float2 bv = *reinterpret_cast<const float2*>(&s_beta[16 * b + col]);
          *reinterpret_cast<uint32_t*>(smem + kOffTB + sw128_off(16 * a + row, 16 * b + col, 64)) =
              pack2(sg * acc[i][0] * bv.x, sg * acc[i][1] * bv.y);
        }
      }
      fence_async_smem();
      named_bar(2, kPrepThreads);

      KDA_MARK(12);
      // ---- P6: W^T = Ktil^T T'^T and U0^T = V^T T'^T (U0 goes where the state
      // pass accumulates U, once it has read the previous chunk's U).
      const bool ok_u = c < 1 || sync.wait_warp(kBarUFree, (c - 1) & 1);
      const bool ok_v = sync.wait_warp(kBarRawV, c & 1);
      if (leader && ok_u && ok_v && !s_abort) {
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
      const bool ok_wu = sync.wait_warp(kBarWU, c & 1);
      // The V tile is free: fetch the next chunk's v.
      if (loader && c + 1 < n_chunks && ok_wu) {
        issue_raw_v(c + 1);
        last_rawv = c + 1;
      }
      // -W^T may overwrite the shared tile once the state pass's first MMA of
      // the previous chunk is done.
      const bool ok_m1 = c < 1 || sync.wait_warp(kBarMMA1, (c - 1) & 1);
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
      for (int i = 8; i < 24; ++i) kda_phase_clocks[i] = prof_acc[i];
    if (blockIdx.x == 0 && blockIdx.y == 0 && p == 0) kda_phase_clocks[28] = n_chunks;
#endif
    // After an abort: raw copies nobody waited for, and MMAs whose commit
    // nobody waited for, land before the block frees its memory (bounded).
    if (s_abort) {
      if (loader && last_raw >= 0) mbar_wait(&s_bars[kBarRaw], last_raw & 1, 100000000ull);
      if (loader && last_rawv >= 0) mbar_wait(&s_bars[kBarRawV], last_rawv & 1, 100000000ull);
      if (leader) {
        umma_commit(&s_bars[kBarDrainP]);
        mbar_wait(&s_bars[kBarDrainP], 0, 100000000ull);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (s_abort && tid == 0 && args.dev_status) atomicExch(args.dev_status, KDA_ERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

}  // namespace

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// A requested chunk of 16 or 32 tokens is served by the 64-token chunks of
// the tensor-core kernels (each made of the same 16-token tiles): the chunk
// size only blocks the computation, the result is the same function.
bool chunk_tc_supported(const LaunchArgs& a) {
  return a.dtype == KDA_BF16 && a.dk == kD && a.dv == kD &&
         (a.chunk == 16 || a.chunk == 32 || a.chunk == kC) && a.total_tokens < (1ll << 31);
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
