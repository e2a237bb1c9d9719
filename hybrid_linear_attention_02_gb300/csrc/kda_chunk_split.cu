// bf16 chunkwise KDA on tcgen05 tensor cores (dk = dv = 128, chunk C = 64),
// split into a parallel preparation kernel and a serial state kernel.
//
// Same chunkwise form as the fused kernel (written out from the recurrence of
// "[Paper Review] Kimi K3: Open Frontier Intelligence", section "Kimi Delta
// Attention (KDA)"; G = in-chunk cumulative log-decay, T = (I + A)^-1):
//   A  = strictly_lower(diag(beta) (k e^G)(k e^-G)^T)
//   W  = T diag(beta) (k e^G),  U = T diag(beta) V - W S0
//   O  = (q e^G) S0 + lower_incl((q e^G)(k e^-G)^T) U
//   S_C = Diag(e^{G_C}) S0 + (k e^{G_C - G})^T U
// Everything but the last three lines' products with S0 and U is independent
// of the state.  With few (sequence, head) pairs, one CTA per pair leaves most
// SMs idle while each CTA's preparation chain is the bound, so here:
//
//  chunk_prep_kernel: persistent, two CTAs per SM, one chunk of one head per
//    iteration, over every chunk of every pair at once.  It runs the
//    state-independent chain (cumulative decay, scaled operand tiles, the
//    masked products A and P in one MMA, T by block-Neumann inversion,
//    W = T' Ktil by MMA) and writes one 66,048-byte record per chunk: the
//    byte images of the operand tiles the state pass reads (Qtil, -W, Kbar,
//    P, T' = T diag(beta)) and e^{G_C}.
//  chunk_state_kernel: one CTA per pair walks its chunks in order; a producer
//    warp streams records (1-D bulk copies) and v tiles (TMA) into a two-slot
//    ring, one warp issues every MMA, and eight warps (two per TMEM lane
//    quarter, each on half the columns) convert between the fp32 state
//    resident in TMEM and the bf16 operands:
//      U0^T = V^T T'^T                                     (MMA0, off the chain)
//      [O^T | U^T] = S^T [Qtil; -W]^T,  U^T += U0^T         (MMA1, N = 128)
//      S^T += U^T Kbar,  O^T += U^T P^T                      (MMA2, N = 128 + 64, fp16)
//    The serial chain per chunk is MMA1 -> U^T to bf16 -> MMA2 -> S^T to
//    bf16 (with the next chunk's decay Diag(e^{G_C}) applied to the fp32
//    copy in the same pass); the previous chunk's output stores run while
//    MMA1 executes.
//
// Records of a window of chunk indices [cw0, cw1) (per sequence) are laid out
// [sequence][head][chunk]; a long input runs as several windows with the
// state carried between them, which bounds the record buffer.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "kda_internal.h"
#include "kda_sm100.cuh"
#include "kda_chunk_common.cuh"

namespace kda {
namespace {

using namespace sm100;
using namespace chunk;

// ---- one chunk record: shared-memory operand images, 1024-aligned tiles.
// WQ: K-major B operand, N = 128 rows (rows 0..63 Qtil, rows 64..127 -W, one
//     per token) by K = 128 key channels; two 16 KB channel panels.
// KB: Kbar, one row per token: an MN-major B operand (N = 128 key channels
//     in two 64-channel panels, K = 64 tokens).
// P:  K-major B operand, 64 rows (one per output token) by K = 64 tokens.
// WQ and T' are bf16.  Kbar and P are fp16, like the U^T they multiply: the
// state update S += Kbar^T U carries U = v_new - v_old where a write replaces
// an old value (beta = 1), which can be far larger than the state it leaves;
// fp16's 10-bit mantissa keeps that update's rounding 8x below bf16's, at no
// extra MMA.  All three are bounded by 1 except U (saturated at +-65504).
constexpr uint32_t kRecWQ = 0;       // [Qtil; -W]        128 x 128
constexpr uint32_t kRecKB = 32768;   // Kbar (fp16)       64 x 128
constexpr uint32_t kRecP = 49152;    // P (fp16)          64 x 64
constexpr uint32_t kRecT = 57344;    // T' = T diag(beta) 64 x 64  (K-major B)
constexpr uint32_t kRecG = 65536;    // e^{G_C}, fp32 [128]
constexpr uint32_t kRecBytes = 66048;
constexpr uint32_t kRecSlot = 66560; // slot stride in shared memory (1024-aligned)
constexpr long long kPrepItemsPerCta = 4;    // overlapped windows: prep CTAs live this long

static_assert(kRecBytes == kSplitRecordBytes, "record size seen by the host");
static_assert(kC == kSplitChunk, "chunk size seen by the window planner");

// ---------------------------------------------------------------- prep kernel
constexpr int kPThreads = 256;
constexpr uint32_t kPOffKQ = 0;        // [K';Q'] 128 x 128; raw k at 0, raw q at 16384
constexpr uint32_t kPOffKH = 32768;    // Khat 160 x 128; then A + inverse scratch; then raw g
constexpr uint32_t kPOffKT = 73728;    // Ktil 64 x 128
// TB: [T'; 0] 128 x 64, the A operand of W = T' Ktil (rows 64..127 zero;
// before P4 they hold the tile sums and e^{R_a} tables).
constexpr uint32_t kPOffTB = 90112;
constexpr uint32_t kPTiles = 106496;
constexpr uint32_t kPSmem = kPTiles + 1024;
// The tables sit in the zero rows of [T'; 0], which the T' store never reads.
constexpr uint32_t kPOffTileTot = kPOffTB + 8192;   // fp32 [4][128]
constexpr uint32_t kPOffTabR = kPOffTB + 10240;     // fp32 [2][4][128]
constexpr uint32_t kPOffG = kPOffKH + 24576;        // raw g of the next item (after step 4)
constexpr int kLdA = 68;
constexpr uint32_t kPOffA = kPOffKH;                       // A   64 x 68 fp32
constexpr int kLdB = 20;
constexpr uint32_t kPOffD = kPOffA + 64 * kLdA * 4;        // D   4 x 16 x 20
constexpr uint32_t kPOffN = kPOffD + 4 * 16 * kLdB * 4;    // N   6 x 16 x 20
constexpr uint32_t kPOffN2 = kPOffN + 6 * 16 * kLdB * 4;   // N^2 3 x 16 x 20
constexpr uint32_t kPOffN3 = kPOffN2 + 3 * 16 * kLdB * 4;  // N^3 16 x 20
constexpr uint32_t kPOffAt = kPOffN3 + 16 * kLdB * 4;     // A_bb^T 4 x 16 x 20
static_assert(kPOffAt + 4 * 16 * kLdB * 4 <= kPOffKH + 40960, "inverse scratch fits");
constexpr uint32_t kPTmemCols = 256;   // AP: 160 fp32 columns; W (lanes 0..63) reuses 0..127
enum { kPBarAP = 0, kPBarW, kPBarRaw, kPBarDrain, kPNumBars };

// ---------------------------------------------------------------- state kernel
constexpr int kSStateWarps = 8;            // warps 0..7: state pass (TMEM <-> registers)
constexpr int kSStateThreads = 32 * kSStateWarps;
constexpr int kSProducerWarp = 8;          // records and v tiles into the ring
constexpr int kSMmaWarp = 9;               // issues every MMA
constexpr int kSThreads = 32 * 10;
constexpr int kSGateWarp = 10;             // gated variant: warps 10, 11 make the gate
constexpr int kSGateWarps = 2;             // tiles w * sigmoid(z), 32 rows each
constexpr int kSThreadsGated = 32 * (10 + kSGateWarps);
constexpr uint32_t kSOffRec = 0;           // 2 record slots
constexpr uint32_t kSOffV = 2 * kRecSlot;  // 2 v tiles 64 x 128
constexpr uint32_t kSOffO = kSOffV + 2 * 16384;  // O staging 64 x 128 (TMA store image)
constexpr uint32_t kSTiles = kSOffO + 16384;
constexpr uint32_t kSSmem = kSTiles + 1024;
constexpr uint32_t kSOffZ = kSTiles;           // gated variant: 2 gate tiles 64 x 128
constexpr uint32_t kSSmemGated = kSTiles + 2 * 16384 + 1024;
constexpr uint32_t kSColS = 0;     // 128 fp32: S^T (lane = value column, column = key row)
constexpr uint32_t kSColO = 128;   // 64 fp32: O^T  (MMA2 writes [S^T | O^T])
constexpr uint32_t kSColU = 192;   // 64 fp32: U^T  (MMA1 writes [O^T | U^T])
constexpr uint32_t kSColSB = 256;  // 64: bf16 S^T, A operand
constexpr uint32_t kSColUT = 320;  // 32: fp16 U^T, A operand
constexpr uint32_t kSColU0 = 352;  // 2 x 64 fp32: U0^T = V^T T'^T, by chunk parity
constexpr uint32_t kSTmemCols = 512;
enum { kSBarFull0 = 0, kSBarFull1, kSBarEmpty0, kSBarEmpty1, kSBarMMA1, kSBarMMA2, kSBarSB,
       kSBarUT, kSBarZFull0, kSBarZFull1, kSBarZEmpty0, kSBarZEmpty1, kSBarZReady0,
       kSBarZReady1, kSBarDrain, kSNumBars };

#ifdef KDA_PHASE_PROFILE
// Per-phase SM-clock totals of two state-pass threads of CTA (0, 0)
// (instrumentation builds only).
__device__ unsigned long long kda_split_clocks[32];
__device__ unsigned long long kda_prep_clocks[32];
#define KDA_SMARK(i)                                  \
  do {                                                \
    const unsigned long long now_ = clock64();        \
    prof_acc[i] += now_ - prof_t;                     \
    prof_t = now_;                                    \
  } while (0)
#else
#define KDA_SMARK(i) ((void)0)
#endif

// One step of a transposing butterfly sum across a warp: afterwards a[0..M)
// hold, for the half of the rows this lane keeps (the upper half when lane
// bit M is set), the sums over lane pairs M apart.  Steps 16 .. 1 over 32
// rows leave lane l with row l summed over all 32 lanes.
template <int M>
__device__ __forceinline__ void butterfly_step(float (&a)[16], int lane) {
  const bool up = lane & M;
#pragma unroll
  for (int i = 0; i < M; ++i) {
    const float send = up ? a[i] : a[i + M];
    const float keep = up ? a[i + M] : a[i];
    a[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, M);
  }
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                    ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ void seq_bounds(const LaunchArgs& a, int n, long long& t0,
                                           long long& t1) {
  if (a.cu_seqlens) {
    t0 = a.cu_seqlens[n];
    t1 = a.cu_seqlens[n + 1];
  } else {
    t0 = static_cast<long long>(n) * a.seq_len;
    t1 = t0 + a.seq_len;
  }
}

// cum[n] = H x (chunks of sequences m < n inside the window), n = 0..N; the
// records of sequence n start at cum[n].  Every thread of the block calls it.
__device__ void window_prefix(const LaunchArgs& a, const SplitWindow& w, int* cum) {
  const int N = a.n_seqs, H = a.heads;
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    long long t0, t1;
    seq_bounds(a, i, t0, t1);
    const long long nc = (t1 - t0 + kC - 1) / kC;
    const long long lo = nc < w.cw0 ? nc : w.cw0, hi = nc < w.cw1 ? nc : w.cw1;
    cum[i + 1] = H * static_cast<int>(hi - lo);
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 0; base < N; base += 32) {
      const int i = base + lane;
      int x = i < N ? cum[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
      }
      if (i < N) cum[i + 1] = carry + x;
      carry += __shfl_sync(0xFFFFFFFFu, x, 31);
    }
    if (lane == 0) cum[0] = 0;
  }
  __syncthreads();
}

struct Item {
  int n, h, c;          // sequence, head, chunk index within the sequence
  long long t0, t1;     // sequence token range
};

__device__ __forceinline__ Item decode_item(const LaunchArgs& a, const SplitWindow& w,
                                            const int* cum, int it) {
  int lo = 0, hi = a.n_seqs;  // cum[lo] <= it < cum[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cum[mid] <= it) lo = mid;
    else hi = mid;
  }
  Item r;
  r.n = lo;
  const int nck = (cum[lo + 1] - cum[lo]) / a.heads;
  const int local = it - cum[lo];
  r.h = local / nck;
  r.c = w.cw0 + local % nck;
  seq_bounds(a, lo, r.t0, r.t1);
  return r;
}

__global__ void __launch_bounds__(kPThreads, 2)
    chunk_prep_kernel(LaunchArgs args, SplitWindow win, const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ __align__(16) float facs[6 * kD];   // Khat block factors e^{R_a2 - R_a}
  __shared__ __align__(16) float s_beta[kC];
  __shared__ int s_cum[kSplitMaxSeqs + 1];
  __shared__ uint64_t s_bars[kPNumBars];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  // The state pass may be scheduled on SMs this grid frees (its loads of
  // the records wait for this grid's completion).
  pdl_launch_dependents();
  const int p = threadIdx.x, pw = p >> 5, lane = p & 31;
  const int H = args.heads;
  window_prefix(args, win, s_cum);
  const int n_items = s_cum[args.n_seqs];
  // Items of this CTA: a contiguous run of win.per_cta (short-lived CTAs that
  // free their SM often), or every gridDim.x-th item (a persistent grid).
  const int it0 = win.per_cta ? static_cast<int>(blockIdx.x) * win.per_cta
                              : static_cast<int>(blockIdx.x);
  const int it_step = win.per_cta ? 1 : static_cast<int>(gridDim.x);
  const int it_end = win.per_cta ? min(n_items, it0 + win.per_cta) : n_items;
  if (it0 >= it_end) return;   // uniform over the block

  if (pw == 0) {
    tmem_alloc(&s_tmem, kPTmemCols);
    tmem_relinquish();
  }
  if (p == 0) {
    for (int b = 0; b < kPNumBars; ++b) mbar_init(&s_bars[b], 1);
    s_abort = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;
  Sync sync{s_bars, &s_abort};

  const int ta = pw & 3;                      // this warp's 16-token row tile
  const int cg = 8 * (pw >> 2) + (lane & 7);  // channels 8 cg .. 8 cg + 7
  const int r4 = lane >> 3;                   // rows 16 ta + 4 r4 + m, m = 0..3
  const int row0 = 16 * ta + 4 * r4;
  const bool leader = p == 0;                 // issues MMAs and bulk stores
  const bool loader = p == 128;               // issues the raw-tile TMA loads
  const __nv_bfloat16* __restrict__ gb = static_cast<const __nv_bfloat16*>(args.beta);
  float* Am = reinterpret_cast<float*>(smem + kPOffA);
  float* Dm = reinterpret_cast<float*>(smem + kPOffD);
  float* Nm = reinterpret_cast<float*>(smem + kPOffN);
  float* N2m = reinterpret_cast<float*>(smem + kPOffN2);
  float* N3m = reinterpret_cast<float*>(smem + kPOffN3);
  float* Atm = reinterpret_cast<float*>(smem + kPOffAt);
  float* tile_tot = reinterpret_cast<float*>(smem + kPOffTileTot);
  float* tabR = reinterpret_cast<float*>(smem + kPOffTabR);

  // Raw k, q (into the [K';Q'] tile, free once the masked products are done)
  // and g (into the Ktil tile, free once W is done), two boxes each, all on
  // one barrier phase: the first call expects the bytes of both.
  auto issue_raw_kq = [&](const Item& x) {
    const int c0 = static_cast<int>(x.t0 + static_cast<long long>(x.c) * kC);
    uint64_t* bar = &s_bars[kPBarRaw];
    mbar_arrive_expect_tx(bar, 3 * 16384);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      tma_load_3d(smem + kPOffKQ + hf * 8192, &tm_k, 64 * hf, x.h, c0, bar);
      tma_load_3d(smem + kPOffKQ + 16384 + hf * 8192, &tm_q, 64 * hf, x.h, c0, bar);
    }
  };
  auto issue_raw_g = [&](const Item& x) {
    const int c0 = static_cast<int>(x.t0 + static_cast<long long>(x.c) * kC);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
      tma_load_3d(smem + kPOffG + hf * 8192, &tm_g, 64 * hf, x.h, c0, &s_bars[kPBarRaw]);
  };
  float rb[4];
  auto load_beta = [&](const Item& x) {
    const long long c0 = x.t0 + static_cast<long long>(x.c) * kC;
    const long long rem = x.t1 - c0;
    const int L = static_cast<int>(rem < kC ? rem : kC);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int r = row0 + m;
      rb[m] = (cg == 0 && r < L) ? __bfloat162float(gb[(c0 + r) * H + x.h]) : 0.f;
    }
  };

  Item cur = decode_item(args, win, s_cum, it0);
  int last_raw = -1;   // loader: the last raw-tile phase it issued copies for
  if (loader) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_g);
    if (!(args.debug_withhold == 2 && blockIdx.x == 0)) {
      issue_raw_kq(cur);
      issue_raw_g(cur);
      last_raw = 0;
    }
  }
  load_beta(cur);

  uint32_t k_iter = 0;
#ifdef KDA_PHASE_PROFILE
  unsigned long long prof_acc[16] = {}, prof_t = clock64();
#endif
#pragma unroll 1
  for (int it = it0; it < it_end; it += it_step, ++k_iter) {
    const uint32_t par = k_iter & 1;
    const long long c0 = cur.t0 + static_cast<long long>(cur.c) * kC;
    const int L = static_cast<int>(cur.t1 - c0 < kC ? cur.t1 - c0 : kC);
    uint8_t* rec = win.rec + static_cast<size_t>(it) * kRecBytes;
    const int it_next = it + it_step;
    // The next item, decoded now so that its loads are done by the masked
    // products' MMA, where its beta is fetched and its raw tiles are issued.
    Item nxt = cur;
    if (it_next < it_end) nxt = decode_item(args, win, s_cum, it_next);

#pragma unroll
    for (int m = 0; m < 4; ++m)
      if (cg == 0) s_beta[row0 + m] = rb[m];
    named_bar(2, kPThreads);
    KDA_SMARK(0);
    const bool ok_raw = sync.wait_warp(kPBarRaw, par);
    KDA_SMARK(1);

    uint4 rq[4], rk[4];
    float G[4][8];
    {
      uint4 rgt[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int r = row0 + m;
        const uint32_t off = sw128_off(r, 8 * cg, 64);
        if (r < L && ok_raw) {
          rgt[m] = *reinterpret_cast<const uint4*>(smem + kPOffG + off);
          rq[m] = *reinterpret_cast<const uint4*>(smem + kPOffKQ + 16384 + off);
          rk[m] = *reinterpret_cast<const uint4*>(smem + kPOffKQ + off);
        } else {
          rgt[m] = rq[m] = rk[m] = make_uint4(0, 0, 0, 0);
        }
      }
      // ---- P1: decay accumulated from the start of this 16-token tile (log2 units).
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
    // Tile sums are visible, and every raw read is done before the tiles are rewritten.
    named_bar(2, kPThreads);
    KDA_SMARK(2);
    // ---- Per-(tile, channel) factors, thread p <-> channel p; split layout as in
    // the fused kernel, so the 16-byte reads below are conflict-free.
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
      facs[0 * kD + sc] = ex2_fast(R[1] - R[0]);
      facs[1 * kD + sc] = ex2_fast(R[2] - R[0]);
      facs[2 * kD + sc] = ex2_fast(R[3] - R[0]);
      facs[3 * kD + sc] = ex2_fast(R[2] - R[1]);
      facs[4 * kD + sc] = ex2_fast(R[3] - R[1]);
      facs[5 * kD + sc] = ex2_fast(R[3] - R[2]);
      reinterpret_cast<float*>(rec + kRecG)[cc] = ex2_fast(acc);
    }
    // The previous item's bulk stores have read their sources: the T' rows
    // before P4 rewrites them, the staged -W before P2 rewrites Ktil.
    if (leader) bulk_wait_read_all();
    named_bar(2, kPThreads);
    KDA_SMARK(3);

    // ---- P2: scaled operand tiles; Qtil and Kbar go straight to the record.
    {
      const int sc0 = 4 * cg;
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
      auto st4 = [&](uint8_t* base, int row, int rows, const uint32_t (&v)[4]) {
        *reinterpret_cast<uint4*>(base + sw128_off(row, 8 * cg, rows)) =
            make_uint4(v[0], v[1], v[2], v[3]);
      };
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint64_t kh[4];
        const int r = row0 + m, rl = 4 * r4 + m;
        const uint32_t kw[4] = {rk[m].x, rk[m].y, rk[m].z, rk[m].w};
        const uint32_t qw[4] = {rq[m].x, rq[m].y, rq[m].z, rq[m].w};
        uint32_t okp[4], oqp[4], okt[4], okh[4], oqt[4], okb[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint64_t kp = bf16x2_to_f2(kw[w]), qp = bf16x2_to_f2(qw[w]);
          const float dx = G[m][2 * w], dy = G[m][2 * w + 1];
          const uint64_t e1 = f2_pack(ex2_fast(dx), ex2_fast(dy));
          const uint64_t ei = f2_pack(ex2_fast(-dx), ex2_fast(-dy));
          const uint64_t k1 = f2_mul(kp, e1), q1 = f2_mul(qp, e1);
          okp[w] = f2_to_bf16x2(k1);
          oqp[w] = f2_to_bf16x2(q1);
          okt[w] = f2_to_bf16x2(f2_mul(k1, eR[w]));
          oqt[w] = f2_to_bf16x2(f2_mul(q1, eR[w]));
          kh[w] = f2_mul(kp, ei);
          okh[w] = f2_to_bf16x2(kh[w]);
          okb[w] = f2_to_f16x2(f2_mul(kh[w], eC[w]));
        }
        st4(smem + kPOffKQ, 32 * ta + rl, 128, okp);
        st4(smem + kPOffKQ, 32 * ta + 16 + rl, 128, oqp);
        st4(smem + kPOffKT, r, 64, okt);
        st4(smem + kPOffKH, khat_row0(ta) + r, 160, okh);
        st4(rec + kRecWQ, r, 128, oqt);
        st4(rec + kRecKB, r, 64, okb);
#pragma unroll
        for (int i = 0; i < 3; ++i) {
          const int a2 = ta + 1 + i;
          if (a2 < 4) {
            const int frow = ta == 0 ? a2 - 1 : ta == 1 ? a2 + 1 : 5;
            uint64_t f[4];
            ld8(facs + frow * kD, f);
            uint32_t ox[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) ox[w] = f2_to_bf16x2(f2_mul(kh[w], f[w]));
            st4(smem + kPOffKH, khat_row0(a2) + r, 160, ox);
          }
        }
      }
    }
    fence_async_smem();
    named_bar(2, kPThreads);
    KDA_SMARK(4);

    // ---- P3: every masked intra-chunk product in one MMA (M=128, N=160, K=128).
    if (leader && !s_abort) {
      tc_fence_after();
      const uint32_t idesc = umma_idesc_bf16(128, 160, 0, 0);
      const uint32_t aK = smem_u32(smem + kPOffKQ), bK = smem_u32(smem + kPOffKH);
#pragma unroll
      for (int t = 0; t < 8; ++t)
        umma_bf16(tbase, umma_desc(aK + (t >> 2) * 128 * 128 + (t & 3) * 32, 16, 1024),
                  umma_desc(bK + (t >> 2) * 160 * 128 + (t & 3) * 32, 16, 1024), idesc, t > 0);
      umma_commit(&s_bars[kPBarAP]);
    }
    if (it_next < it_end) load_beta(nxt);
    const bool ok_ap = sync.wait_warp(kPBarAP, par);
    tc_fence_after();
    // [K';Q'] is dead: the next item's raw k and q may land.
    if (loader && ok_ap && it_next < it_end) {
      issue_raw_kq(nxt);
      last_raw = static_cast<int>(k_iter) + 1;
    }
    KDA_SMARK(5);

    // ---- P4: A (x beta, strictly lower; fp32, shared) and P (lower inclusive;
    // bf16, straight to the record).  Warps pw and pw + 4 share row tile
    // pw & 3 (the same TMEM lanes): the first takes column blocks 0 and 2, the
    // second 1 and 3.  A's blocks above the diagonal are never read, so only
    // P's are written (as zeros); A's diagonal blocks go out transposed, and
    // the warp that holds one also inverts it (P5 below).
    // The [T'; 0] tile's zeros (blocks above the diagonal, rows 64..127) go
    // in first: the factor tables that shared the tile are dead.
    for (int e = p; e < 192; e += kPThreads) {
      const int pb = e >> 5, rr = (e >> 1) & 15, h8 = e & 1;
      const int a = pb < 3 ? 0 : pb < 5 ? 1 : 2;
      const int b = pb < 3 ? pb + 1 : pb < 5 ? pb - 1 : 3;
      const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      st_tile8(smem + kPOffTB, 16 * a + rr, 16 * b + 8 * h8, 64, z);
    }
    for (int e = p; e < 512; e += kPThreads)
      *reinterpret_cast<uint4*>(smem + kPOffTB + 8192 + 16 * e) = make_uint4(0, 0, 0, 0);
    if (ok_ap) {
      const int a = pw & 3, b0 = pw >> 2, rl = lane & 15, r = 16 * a + rl;
      const bool isP = lane >= 16;
      const float br = s_beta[r];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int blk = b0 + 2 * j;
        float v[16];
        if (blk <= a) {
          tmem_ld16(tbase + (static_cast<uint32_t>(32 * a) << 16) + khat_row0(a) + 16 * blk, v);
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
            st_tile8_f16(rec + kRecP, r, 16 * blk + 8 * h8, 64, f8);
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
      // ---- P5 (diagonal blocks): D_aa = (I + A_aa)^-1, column jj = lane by
      // right-looking substitution: once x_i is final it is taken off every
      // later row, so the dependent chain is one FMA per row.  Column i of
      // A_aa is row i of its transposed copy (the 16 lanes read the same words).
      if (b0 == (a & 1)) {
        __syncwarp();
        if (lane < 16) {
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
    }
    tc_fence_before();
    named_bar(2, kPThreads);
    KDA_SMARK(6);
    // ---- P5: T = (I + A)^-1 = (I - N + N^2 - N^3) D in fp32 with N = D A
    // (strictly block-lower, N^4 = 0), written as T' = T diag(beta) in bf16.
    KDA_SMARK(7);
    // Block products, one warp per 16 x 16 x 16 product on warp-level tf32
    // tensor-core MMAs (m16n8k8, fp32 accumulate): acc[i] holds row
    // mg + 8 (i & 1), columns 8 (i >> 1) + 2 mt, + 1 of the output block.
    // Elementwise block work (step 4's M_30) has lane (i4, j2) take rows
    // 4 i4 .. + 3 and columns 2 j2, 2 j2 + 1.
    const int i4 = lane >> 3, j2 = lane & 7;
    const int mg = lane >> 2, mt = lane & 3;
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
          mma_m16n8k8_tf32(acc[2 * nh][0], acc[2 * nh][1], acc[2 * nh + 1][0], acc[2 * nh + 1][1],
                           a0, a1, a2, a3, b0, b1);
        }
      }
    };
    auto store_blk = [&](float* Z, const float (&acc)[4][2]) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float2*>(Z + (mg + 8 * (i & 1)) * kLdB + 8 * (i >> 1) + 2 * mt) =
            make_float2(acc[i][0], acc[i][1]);
    };
    // Off-diagonal block pairs (a, b), a > b: (1,0)=0 (2,0)=1 (2,1)=2 (3,0)=3 (3,1)=4 (3,2)=5.
    auto blk_a = [](int blk) { return blk < 1 ? 1 : blk < 3 ? 2 : 3; };
    auto blk_b = [](int blk) {
      const int a = blk < 1 ? 1 : blk < 3 ? 2 : 3;
      return blk - (a * (a - 1)) / 2;
    };
    // Step 1: N_ab = D_aa A_ab (warps 0..5); diagonal blocks of T' (warps 6, 7).
    if (pw < 6) {
      const int a = blk_a(pw), b = blk_b(pw);
      float acc[4][2] = {};
      prod16(Dm + a * 16 * kLdB, kLdB, Am + 16 * a * kLdA + 16 * b, kLdA, acc);
      store_blk(Nm + pw * 16 * kLdB, acc);
    } else {
      for (int e = p - 192; e < 128; e += 64) {
        const int a = e >> 5, rr = (e >> 1) & 15, h8 = e & 1;
        float f8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int cc = 8 * h8 + u;
          f8[u] = Dm[(a * 16 + rr) * kLdB + cc] * s_beta[16 * a + cc];
        }
        st_tile8(smem + kPOffTB, 16 * a + rr, 16 * a + 8 * h8, 64, f8);
      }
    }
    named_bar(2, kPThreads);
    KDA_SMARK(8);
    // Step 2: N^2 blocks (2,0) = N21 N10, (3,1) = N32 N21, and (3,0) = N31 N10
    // + N32 N20 as two halves (warps 2, 3; the second where A_bb^T was).
    if (pw < 4) {
      float acc[4][2] = {};
      const int xa = pw == 0 ? 2 : pw == 1 ? 5 : pw == 2 ? 4 : 5;
      const int ya = pw == 0 ? 0 : pw == 1 ? 2 : pw == 2 ? 0 : 1;
      prod16(Nm + xa * 16 * kLdB, kLdB, Nm + ya * 16 * kLdB, kLdB, acc);
      store_blk(pw < 3 ? N2m + pw * 16 * kLdB : Atm, acc);
    }
    named_bar(2, kPThreads);
    KDA_SMARK(9);
    // Step 3: N^3 block (3,0) = N32 (N^2)_20 (warp 0), and M = -N + N^2 in
    // place of N for blocks (1,0) (2,0) (2,1) (3,1) (warps 1..7); N32, which
    // warp 0 reads, is negated in step 4 and M_30 is finished there too.
    if (pw == 0) {
      float acc[4][2] = {};
      prod16(Nm + 5 * 16 * kLdB, kLdB, N2m, kLdB, acc);
      store_blk(N3m, acc);
    } else {
      for (int e = p - 32; e < 4 * 64; e += kPThreads - 32) {
        const int bsel = e >> 6;
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
    named_bar(2, kPThreads);
    KDA_SMARK(10);
    // Step 4: T_ab = M_ab D_bb, times beta, into T' (warps 0..5; M_30 =
    // -N30 + N^2_30 - N^3_30 first, M_32 = -N_32).
    if (pw < 6) {
      const int a = blk_a(pw), b = blk_b(pw);
      if (pw == 3) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = 4 * i4 + i;
          float2* nv = reinterpret_cast<float2*>(Nm + (3 * 16 + row) * kLdB + 2 * j2);
          const float2 n2 = *reinterpret_cast<const float2*>(N2m + (2 * 16 + row) * kLdB + 2 * j2);
          const float2 n2b = *reinterpret_cast<const float2*>(Atm + row * kLdB + 2 * j2);
          const float2 n3 = *reinterpret_cast<const float2*>(N3m + row * kLdB + 2 * j2);
          float2 m = *nv;
          m.x = n2.x + n2b.x - m.x - n3.x;
          m.y = n2.y + n2b.y - m.y - n3.y;
          *nv = m;
        }
        __syncwarp();
      }
      float acc[4][2] = {};
      prod16(Nm + pw * 16 * kLdB, kLdB, Dm + b * 16 * kLdB, kLdB, acc);
      const float sg = pw == 5 ? -1.f : 1.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = mg + 8 * (i & 1), col = 8 * (i >> 1) + 2 * mt;
        const float2 bv = *reinterpret_cast<const float2*>(&s_beta[16 * b + col]);
        *reinterpret_cast<uint32_t*>(smem + kPOffTB + sw128_off(16 * a + row, 16 * b + col, 64)) =
            pack2(sg * acc[i][0] * bv.x, sg * acc[i][1] * bv.y);
      }
    }
    fence_async_smem();
    named_bar(2, kPThreads);
    KDA_SMARK(11);
    // The inverse scratch is dead: the next item's raw g may land behind it.
    if (loader && ok_ap && it_next < it_end) issue_raw_g(nxt);
    // T' is final: it leaves for the record now (it stays the A operand of W).
    if (leader && !s_abort) {
      bulk_store(rec + kRecT, smem + kPOffTB, 8192);
      bulk_commit();
    }

    // ---- P6: [W; 0] = [T'; 0] Ktil (M=128, N=128, K=64): W rows in TMEM
    // lanes 0..63, columns 0..127.
    if (leader && !s_abort) {
      tc_fence_after();
      const uint32_t idesc = umma_idesc_bf16(128, 128, 0, 1);
      const uint32_t aT = smem_u32(smem + kPOffTB), bKT = smem_u32(smem + kPOffKT);
#pragma unroll
      for (int t = 0; t < 4; ++t)
        umma_bf16(tbase, umma_desc(aT + t * 32, 16, 1024),
                  umma_desc(bKT + t * 2048, 64 * 128, 1024), idesc, t > 0);
      umma_commit(&s_bars[kPBarW]);
    }
    const bool ok_w = sync.wait_warp(kPBarW, par);
    tc_fence_after();
    KDA_SMARK(12);

    // ---- P7: -W (row = token, column = key channel) to the record, where
    // its two 64-channel panels are rows 64..127 of the WQ panels.  Warps 0,
    // 1 take channels 0..63 and warps 4, 5 channels 64..127 of TMEM lanes
    // 0..63.  A lane holds one row, so the rows are staged in the Ktil tile
    // (dead once W is done; the leader's read wait before the next item's P2
    // orders its reuse) and leave as two 8 KB bulk copies, rather than as
    // 16-byte stores that each touch a different 128-byte line.
    if ((pw & 3) < 2) {
      if (ok_w) {
        const int t = 32 * (pw & 3) + lane, q0 = 2 * (pw >> 2);
        float w[2][32];
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tmem_ld32(tbase + (static_cast<uint32_t>(32 * (pw & 3)) << 16) + 32 * (q0 + j), w[j]);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {
            float f8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) f8[u] = -w[j][8 * q8 + u];
            st_tile8(smem + kPOffKT, t, 32 * (q0 + j) + 8 * q8, 64, f8);
          }
        fence_async_smem();
      }
      named_bar(3, 128);   // the four -W warps, whatever the wait returned
      if (leader && ok_w && !s_abort) {
        bulk_store(rec + kRecWQ + 8192, smem + kPOffKT, 8192);
        bulk_store(rec + kRecWQ + 16384 + 8192, smem + kPOffKT + 8192, 8192);
        bulk_commit();
      }
    }
    tc_fence_before();
    KDA_SMARK(13);
    cur = nxt;
  }
#ifdef KDA_PHASE_PROFILE
  if (blockIdx.x == 0 && (p == 0 || p == 160)) {
    for (int i = 0; i < 14; ++i) kda_prep_clocks[(p ? 16 : 0) + i] = prof_acc[i];
    if (p == 0) kda_prep_clocks[31] = k_iter;
  }
#endif
  if (leader) bulk_wait_all();
  // After an abort: raw-tile copies nobody waited for and MMAs whose commit
  // nobody waited for land before the block frees its memory (bounded).
  if (s_abort) {
    if (loader && last_raw >= 0) mbar_wait(&s_bars[kPBarRaw], last_raw & 1, 100000000ull);
    if (leader) {
      umma_commit(&s_bars[kPBarDrain]);
      mbar_wait(&s_bars[kPBarDrain], 0, 100000000ull);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (s_abort && p == 0 && args.dev_status) atomicExch(args.dev_status, KDA_ERR_TIMEOUT);
  if (pw == 0) tmem_dealloc(tbase, kPTmemCols);
}

// Variants: kGate also applies the output epilogue (head-wise RMSNorm, then
// the sigmoid gate) to every output row before it is stored, the gate tiles
// arriving by TMA beside the records; kTrans computes segment transitions
// (below) instead of outputs.  Each is its own instantiation.
template <bool kGate, bool kTrans>
__global__ void __launch_bounds__(kGate ? kSThreadsGated : kSThreads, 1)
    chunk_state_kernel(LaunchArgs args, SplitWindow win, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CUtensorMap tm_z) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  __shared__ int s_cum[kSplitMaxSeqs + 1];
  __shared__ uint64_t s_bars[kSNumBars];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
#ifdef KDA_PHASE_PROFILE
  __shared__ volatile unsigned long long s_ts[4];   // MMA1 / MMA2 issue, SB / UT hand-off
#endif
  __shared__ __align__(16) float s_rsum[2][4][32];   // gated: row sums of squares, per warp
  __shared__ __align__(16) float s_rinv[2][32];      // gated: 1 / rms of the chunk's rows
  __shared__ __align__(16) float s_gw[kD];           // gated: RMSNorm scale

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = args.heads;
  const int h = blockIdx.y;
  const int n = args.order ? args.order[blockIdx.x] : static_cast<int>(blockIdx.x);
  window_prefix(args, win, s_cum);
  long long t0, t1;
  seq_bounds(args, n, t0, t1);
  const int nck = (s_cum[n + 1] - s_cum[n]) / H;     // chunks of this pair in the window
  const int rbase = s_cum[n] + h * nck;
  const long long soff = (static_cast<long long>(n) * H + h) * kD * kD;
  // Transition mode (args.trans_M set, grid depth 2): z = 0 runs the chunks
  // from S_0 = 0 and leaves H in trans_H, z = 1 runs them from S_0 = I with
  // v = 0 and leaves M in trans_M (dk = dv); no outputs.  Between windows the
  // two buffers carry the partial maps.
  const int tmode = kTrans ? 1 + static_cast<int>(blockIdx.z) : 0;   // 0 off, 1 H, 2 M
  const bool vzero = tmode == 2;
  float* tbuf = tmode == 1 ? args.trans_H : args.trans_M;
  const float* src = tmode ? (win.first ? nullptr : tbuf)
                           : (win.first ? args.init_state : win.s_run);
  const bool src_identity = tmode == 2 && win.first;
  float* dst = tmode ? tbuf : (win.last ? args.final_state : win.s_run);

  if (nck == 0) {
    // No chunk of this pair in the window: carry its state (or map) through.
    if (dst && dst != src) {
      float4* d4 = reinterpret_cast<float4*>(dst + soff);
      const float4* s4 = reinterpret_cast<const float4*>(src + soff);
      for (int e = tid; e < kD * kD / 4; e += static_cast<int>(blockDim.x)) {
        const int r = (4 * e) / kD, c = (4 * e) % kD;
        d4[e] = src ? s4[e]
                    : src_identity ? make_float4(r == c, r == c + 1, r == c + 2, r == c + 3)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    return;
  }

  if (warp == 0) {
    tmem_alloc(&s_tmem, kSTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    for (int b = 0; b < kSNumBars; ++b)
      mbar_init(&s_bars[b], b == kSBarZReady0 || b == kSBarZReady1 ? kSGateWarps : 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if constexpr (kGate) {
    if (tid < kD) s_gw[tid] = args.gate_w[tid];   // the RMSNorm scale
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;
  Sync sync{s_bars, &s_abort};

  if (warp >= kSGateWarp) {
    // ================================ gate tiles ===============================
    // Off the serial chain: each chunk's gate tile becomes w * sigmoid(z) in
    // place as soon as it lands (sigmoid(x) = (1 + tanh(x / 2)) / 2; the tile
    // is bf16, far coarser than the approximation), ready before the chunk's
    // outputs leave.  Lane l of gate warp g takes the 8-column group l & 15
    // of rows 32 g + (l >> 4) + 2 i.
    if constexpr (kGate) {
      const int cgp = lane & 15, rg = 32 * (warp - kSGateWarp) + (lane >> 4);
      float gw8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) gw8[u] = s_gw[8 * cgp + u];
#pragma unroll 1
      for (int c = 0; c < nck; ++c) {
        const int zs = c & 1;
        if (!sync.wait_warp(kSBarZFull0 + zs, (c >> 1) & 1)) break;
        uint8_t* zt = smem + kSOffZ + zs * 16384;
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          uint4* pz = reinterpret_cast<uint4*>(zt + sw128_off(rg + 2 * i, 8 * cgp, 64));
          const uint4 zv = *pz;
          uint32_t wv[4] = {zv.x, zv.y, zv.z, zv.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            float lo, hi;
            f2_unpack(bf16x2_to_f2(wv[u]), lo, hi);
            lo = gw8[2 * u] * fmaf(0.5f, tanh_fast(0.5f * lo), 0.5f);
            hi = gw8[2 * u + 1] * fmaf(0.5f, tanh_fast(0.5f * hi), 0.5f);
            wv[u] = pack2(lo, hi);
          }
          *pz = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_bars[kSBarZReady0 + zs]);
      }
    }
  } else if (warp == kSProducerWarp) {
    // ================================ producer ================================
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      // Launched as a programmatic dependent of the preparation grid: its
      // records are complete and visible past this point.  Nothing else of
      // this kernel reads what that grid writes.
      pdl_wait();
      int last[2] = {-1, -1}, zlast[2] = {-1, -1};   // last chunk loaded into each slot
#pragma unroll 1
      for (int c = 0; c < nck; ++c) {
        const int s = c & 1;
        if (c >= 2 && !sync.wait(kSBarEmpty0 + s, ((c - 2) >> 1) & 1)) break;
        if (c == 0 && args.debug_withhold == 1 && win.first && blockIdx.x == 0 &&
            blockIdx.y == 0 && blockIdx.z == 0)
          continue;   // self-test: this record never arrives
        uint64_t* bar = &s_bars[kSBarFull0 + s];
        mbar_arrive_expect_tx(bar, kRecBytes + (vzero ? 0 : 16384));
        const uint8_t* rec = win.rec + static_cast<size_t>(rbase + c) * kRecBytes;
        uint8_t* slot = smem + kSOffRec + s * kRecSlot;
#pragma unroll
        for (int i = 0; i < 4; ++i) bulk_load(slot + 16384 * i, rec + 16384 * i, 16384, bar);
        bulk_load(slot + kRecG, rec + kRecG, kRecBytes - kRecG, bar);
        const int c0 = static_cast<int>(t0 + static_cast<long long>(win.cw0 + c) * kC);
        if (!vzero) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_3d(smem + kSOffV + s * 16384 + hf * 8192, &tm_v, 64 * hf, h, c0, bar);
        }
        last[s] = c;
        if constexpr (kGate) {
          // The gate tile of chunk c is read when its outputs leave, during
          // chunk c + 1; its slot is free once chunk c - 2's outputs have left.
          if (c >= 2 && !sync.wait(kSBarZEmpty0 + s, ((c - 2) >> 1) & 1)) break;
          uint64_t* zbar = &s_bars[kSBarZFull0 + s];
          mbar_arrive_expect_tx(zbar, 16384);
#pragma unroll
          for (int hf = 0; hf < 2; ++hf)
            tma_load_3d(smem + kSOffZ + s * 16384 + hf * 8192, &tm_z, 64 * hf, h, c0, zbar);
          zlast[s] = c;
        }
      }
      // After an abort, copies issued into a slot nobody waited on may still
      // be landing: wait for them (bounded) before the block can exit.
      if (s_abort) {
        for (int s = 0; s < 2; ++s) {
          if (last[s] >= 0) mbar_wait(&s_bars[kSBarFull0 + s], (last[s] >> 1) & 1, 100000000ull);
          if (zlast[s] >= 0)
            mbar_wait(&s_bars[kSBarZFull0 + s], (zlast[s] >> 1) & 1, 100000000ull);
        }
      }
    }
  } else if (warp == kSMmaWarp) {
    // ================================ MMA issue ===============================
    if (lane == 0) {
      // U0^T = V^T T'^T of the chunk in slot s, into U0 buffer s (state-independent).
      auto issue_mma0 = [&](int s) {
        const uint32_t idesc = umma_idesc_bf16(128, 64, 1, 0);
        const uint32_t aV = smem_u32(smem + kSOffV + s * 16384);
        const uint32_t bT = smem_u32(smem + kSOffRec + s * kRecSlot + kRecT);
#pragma unroll
        for (int t = 0; t < 4; ++t)
          umma_bf16(tbase + kSColU0 + 64 * s, umma_desc(aV + t * 2048, 64 * 128, 1024),
                    umma_desc(bT + t * 32, 16, 1024), idesc, t > 0);
      };
      bool ok = sync.wait(kSBarFull0, 0);
      if (ok && !vzero) {
        tc_fence_after();
        issue_mma0(0);
      }
#pragma unroll 1
      for (int c = 0; c < nck && ok; ++c) {
        const int s = c & 1;
        const uint8_t* slot = smem + kSOffRec + s * kRecSlot;
        // [O^T | U^T] = S^T [Qtil^T | -W^T]      (M = 128, N = 128, K = dk = 128)
        if (!sync.wait(kSBarSB, c & 1)) break;
        tc_fence_after();
#ifdef KDA_PHASE_PROFILE
        s_ts[0] = clock64();
#endif
        {
          const uint32_t idesc = umma_idesc_bf16(128, 128, 0, 0);
          const uint32_t bWQ = smem_u32(slot + kRecWQ);
#pragma unroll
          for (int t = 0; t < 8; ++t)
            umma_bf16_tmem_a(tbase + kSColO, tbase + kSColSB + 8 * t,
                             umma_desc(bWQ + (t >> 2) * 16384 + (t & 3) * 32, 16, 1024), idesc,
                             t > 0);
          umma_commit(&s_bars[kSBarMMA1]);
        }
        // S^T += U^T Kbar,  O^T += U^T P^T        (M = 128, N = 128 + 64, K = 64 tokens;
        // fp16 operands: U^T, Kbar and P, see the record layout above)
        if (!sync.wait(kSBarUT, c & 1)) break;
        tc_fence_after();
#ifdef KDA_PHASE_PROFILE
        s_ts[1] = clock64();
#endif
        {
          const uint32_t idesc_s = umma_idesc_f16(128, 128, 0, 1);
          const uint32_t idesc_o = umma_idesc_f16(128, 64, 0, 0);
          const uint32_t bKB = smem_u32(slot + kRecKB), bP = smem_u32(slot + kRecP);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            umma_bf16_tmem_a(tbase + kSColS, tbase + kSColUT + 8 * t,
                             umma_desc(bKB + t * 2048, 64 * 128, 1024), idesc_s, 1);
            umma_bf16_tmem_a(tbase + kSColO, tbase + kSColUT + 8 * t,
                             umma_desc(bP + t * 32, 16, 1024), idesc_o, 1);
          }
          umma_commit(&s_bars[kSBarEmpty0 + s]);
          umma_commit(&s_bars[kSBarMMA2]);
        }
        // The next chunk's U0^T runs while the state warps convert S^T.
        if (c + 1 < nck && !vzero) {
          if (!sync.wait(kSBarFull0 + (s ^ 1), ((c + 1) >> 1) & 1)) break;
          tc_fence_after();
          issue_mma0(s ^ 1);
        }
      }
      // Every MMA issued has completed before the block frees its TMEM.
      umma_commit(&s_bars[kSBarDrain]);
      mbar_wait(&s_bars[kSBarDrain], 0, 100000000ull);
    }
  } else {
    // =============================== state pass ===============================
    // Warp w reads TMEM lanes 32 (w & 3) .. + 31 (value columns j) and the
    // column half hf = w >> 2 of every TMEM matrix.
    const int q = warp & 3, hf = warp >> 2;
    const int j = 32 * q + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    __nv_bfloat16* __restrict__ gout = static_cast<__nv_bfloat16*>(args.out);

    // S^T[j][c] = S[c][j] for key rows c of this half: fp32 copy and bf16 copy.
#pragma unroll 1
    for (int cb = 0; cb < 2; ++cb) {
      const int c0 = 64 * hf + 32 * cb;
      uint32_t f[32], b[16];
#pragma unroll
      for (int u = 0; u < 32; ++u)
        f[u] = __float_as_uint(src ? __ldcs(src + soff + (c0 + u) * kD + j)
                                   : (src_identity && c0 + u == j ? 1.f : 0.f));
#pragma unroll
      for (int u = 0; u < 16; ++u)
        b[u] = pack2(__uint_as_float(f[2 * u]), __uint_as_float(f[2 * u + 1]));
      tmem_st32(tbase + lane_base + kSColS + c0, f);
      tmem_st16(tbase + lane_base + kSColSB + c0 / 2, b);
    }
    // Outputs of chunk cl, held as O^T column j, rows 32 hf .. + 31, in `ov`.
    // Lane pairs swap values so each lane holds two adjacent columns of every
    // other row.  A full chunk goes through the staging tile and one TMA
    // store per 64-column half; a sequence's ragged last chunk is written
    // row by row (the tile's tail rows belong to the next sequence).  Every
    // state thread calls it (it holds barriers); `live` is false once a wait
    // has failed.  With `defer`, a gated full chunk is only staged and the
    // call returns true: its epilogue pass (gated_finish) is still to run.
    float ov[32];
    // A full chunk with the output epilogue, in two parts.  Part one: the raw
    // outputs (bf16) to the staging tile, while MMA1 of the next chunk runs.
    // Part two, during the next chunk's MMA2 (the U^T hand-off's barrier has
    // made every thread's staged rows visible by then): 8 threads per row
    // (16 columns each, 16-byte vectors) take the row's sum of squares with 3
    // shuffles and scale it in place by 1 / rms times the gate tile's
    // w * sigmoid(z), then the TMA stores.
    auto gated_stage = [&](bool odd) {
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float a = ov[2 * k], b = ov[2 * k + 1];
        const float other = __shfl_xor_sync(0xFFFFFFFFu, odd ? a : b, 1);
        pk[k] = odd ? pack2(other, b) : pack2(a, other);
      }
      // The previous TMA store has read the staging tile.
      if (tid == 0) bulk_wait_read_all();
      named_bar(1, kSStateThreads);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int r = 32 * hf + 2 * k + (odd ? 1 : 0);
        *reinterpret_cast<uint32_t*>(smem + kSOffO + sw128_off(r, j & ~1, 64)) = pk[k];
      }
    };
    // Part two (after a barrier since part one).
    auto gated_finish = [&](int cl, bool live) {
      const long long c0 = t0 + static_cast<long long>(win.cw0 + cl) * kC;
      // The gate tile holds w * sigmoid(z) once the gate warps are done with it.
      if (!sync.wait_warp(kSBarZReady0 + (cl & 1), (cl >> 1) & 1)) live = false;
      const uint8_t* zt = smem + kSOffZ + (cl & 1) * 16384;
      const int sg = tid & 7;
#pragma unroll
      for (int rh = 0; rh < 2; ++rh) {
        const int r = (tid >> 3) + 32 * rh;
        uint4* po[2];
        uint4 ov4[2], gv4[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t off = sw128_off(r, 16 * sg + 8 * e, 64);
          po[e] = reinterpret_cast<uint4*>(smem + kSOffO + off);
          ov4[e] = *po[e];
          gv4[e] = *reinterpret_cast<const uint4*>(zt + off);
        }
        float x[16];
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          unpack8(ov4[e], *reinterpret_cast<float(*)[8]>(&x[8 * e]));
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) ss = fmaf(x[u], x[u], ss);
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 4);
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 2);
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, 1);
        const float rinv = rsqrtf(ss * (1.f / kD) + args.gate_eps);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float gz[8];
          unpack8(gv4[e], gz);
          uint32_t w4[4];
#pragma unroll
          for (int u = 0; u < 4; ++u)
            w4[u] = pack2(x[8 * e + 2 * u] * rinv * gz[2 * u],
                          x[8 * e + 2 * u + 1] * rinv * gz[2 * u + 1]);
          *po[e] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      fence_async_smem();
      named_bar(1, kSStateThreads);
      if (tid == 0) mbar_arrive(&s_bars[kSBarZEmpty0 + (cl & 1)]);   // gate tile read
      if (tid == 0 && live && !s_abort) {
        tma_store_3d(&tm_o, smem + kSOffO, 0, h, static_cast<int>(c0));
        tma_store_3d(&tm_o, smem + kSOffO + 8192, 64, h, static_cast<int>(c0));
        bulk_commit();
      }
    };
    auto emit_out = [&](int cl, bool live, bool defer) -> bool {
      const long long c0 = t0 + static_cast<long long>(win.cw0 + cl) * kC;
      const int L = static_cast<int>(t1 - c0 < kC ? t1 - c0 : kC);
      const bool odd = lane & 1;
      if constexpr (kGate) {
        if (L == kC) {
          gated_stage(odd);
          if (defer) return true;
          named_bar(1, kSStateThreads);
          gated_finish(cl, live);
          return false;
        }
        // (A sequence's ragged last chunk.)  Row sums of squares: a butterfly over the warp's 32 columns leaves
        // lane l with row 32 hf + l; the four warps of a column half meet in
        // shared memory.
        float a[16];
        {
          const bool up = lane & 16;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float lo = ov[i] * ov[i], hi = ov[i + 16] * ov[i + 16];
            a[i] = (up ? hi : lo) + __shfl_xor_sync(0xFFFFFFFFu, up ? lo : hi, 16);
          }
        }
        butterfly_step<8>(a, lane);
        butterfly_step<4>(a, lane);
        butterfly_step<2>(a, lane);
        butterfly_step<1>(a, lane);
        s_rsum[hf][q][lane] = a[0];
        named_bar(1, kSStateThreads);
        if (q == 0) {
          const float ss = s_rsum[hf][0][lane] + s_rsum[hf][1][lane] + s_rsum[hf][2][lane] +
                           s_rsum[hf][3][lane];
          s_rinv[hf][lane] = rsqrtf(ss * (1.f / kD) + args.gate_eps);
        }
        named_bar(1, kSStateThreads);
        // The gate tile holds w * sigmoid(z) once the gate warp is done with it.
        if (!sync.wait_warp(kSBarZReady0 + (cl & 1), (cl >> 1) & 1)) live = false;
        const uint8_t* zt = smem + kSOffZ + (cl & 1) * 16384;
#pragma unroll
        for (int r = 0; r < 32; r += 4) {
          const float4 ri = *reinterpret_cast<const float4*>(&s_rinv[hf][r]);
          const float rr[4] = {ri.x, ri.y, ri.z, ri.w};
#pragma unroll
          for (int u = 0; u < 4; ++u)
            ov[r + u] *= rr[u] * __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                                     zt + sw128_off(32 * hf + r + u, j, 64)));
        }
      }
      uint32_t pk[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float a = ov[2 * k], b = ov[2 * k + 1];
        const float other = __shfl_xor_sync(0xFFFFFFFFu, odd ? a : b, 1);
        pk[k] = odd ? pack2(other, b) : pack2(a, other);
      }
      if (L < kC) {
        __nv_bfloat16* base = gout + (c0 * H + h) * kD + (j & ~1);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int r = 32 * hf + 2 * k + (odd ? 1 : 0);
          if (live && r < L)
            *reinterpret_cast<uint32_t*>(base + static_cast<long long>(r) * H * kD) = pk[k];
        }
        if constexpr (kGate) {
          named_bar(1, kSStateThreads);   // every gate-tile read is done
          if (tid == 0) mbar_arrive(&s_bars[kSBarZEmpty0 + (cl & 1)]);
        }
        return false;
      }
      // The previous TMA store has read the staging tile.
      if (tid == 0) bulk_wait_read_all();
      named_bar(1, kSStateThreads);
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int r = 32 * hf + 2 * k + (odd ? 1 : 0);
        *reinterpret_cast<uint32_t*>(smem + kSOffO + sw128_off(r, j & ~1, 64)) = pk[k];
      }
      fence_async_smem();
      named_bar(1, kSStateThreads);
      if constexpr (kGate) {
        if (tid == 0) mbar_arrive(&s_bars[kSBarZEmpty0 + (cl & 1)]);   // gate tile read
      }
      if (tid == 0 && live && !s_abort) {
        tma_store_3d(&tm_o, smem + kSOffO, 0, h, static_cast<int>(c0));
        tma_store_3d(&tm_o, smem + kSOffO + 8192, 64, h, static_cast<int>(c0));
        bulk_commit();
      }
      return false;
    };

    // The fp32 state carries the first chunk's decay Diag(e^{G_C}) before
    // MMA2 adds onto it (later chunks get theirs in step E).
    bool ok = sync.wait_warp(kSBarFull0, 0);
    tmem_st_wait();
    if (ok) {
      const float* gam = reinterpret_cast<const float*>(smem + kSOffRec + kRecG);
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        const int c0 = 64 * hf + 32 * cb;
        float v[32];
        tmem_ld32(tbase + lane_base + kSColS + c0, v);
        tmem_ld_wait();
        uint32_t f[32];
#pragma unroll
        for (int u = 0; u < 32; u += 4) {
          const float4 gm = *reinterpret_cast<const float4*>(&gam[c0 + u]);
          f[u] = __float_as_uint(v[u] * gm.x);
          f[u + 1] = __float_as_uint(v[u + 1] * gm.y);
          f[u + 2] = __float_as_uint(v[u + 2] * gm.z);
          f[u + 3] = __float_as_uint(v[u + 3] * gm.w);
        }
        tmem_st32(tbase + lane_base + kSColS + c0, f);
      }
    }
    tmem_st_wait();
    tc_fence_before();
    named_bar(1, kSStateThreads);
#ifdef KDA_PHASE_PROFILE
    if (tid == 0) s_ts[2] = clock64();
#endif
    if (tid == 0) mbar_arrive(&s_bars[kSBarSB]);
    bool prev_ok = false;
    bool pend = false;   // gated: chunk c - 1 staged, its epilogue pass still to run
#ifdef KDA_PHASE_PROFILE
    unsigned long long hand[4] = {};   // SB->MMA1 issue, MMA1 exec, UT->MMA2 issue, MMA2 exec
#endif
#ifdef KDA_PHASE_PROFILE
    unsigned long long prof_acc[10] = {}, prof_t = clock64();
#endif

#pragma unroll 1
    for (int c = 0; c < nck; ++c) {
      const int s = c & 1;
      // (B) While MMA1 runs: the previous chunk's outputs.
      if (c > 0 && tmode == 0) pend = emit_out(c - 1, prev_ok, true);
      KDA_SMARK(0);
      // (C) U^T + U0^T (fp32) -> bf16 A operand, then hand it to MMA2.
      bool ok1 = ok && sync.wait_warp(kSBarMMA1, c & 1);
      tc_fence_after();
#ifdef KDA_PHASE_PROFILE
      if (tid == 0) {
        const unsigned long long now = clock64();
        hand[0] += s_ts[0] - s_ts[2];
        hand[1] += now - s_ts[0];
      }
#endif
      KDA_SMARK(1);
      if (ok1) {
        float v[32], w[32];
        tmem_ld32(tbase + lane_base + kSColU + 32 * hf, v);
        if (!vzero) tmem_ld32(tbase + lane_base + kSColU0 + 64 * s + 32 * hf, w);
        tmem_ld_wait();
        if (vzero) {
#pragma unroll
          for (int u = 0; u < 32; ++u) w[u] = 0.f;
        }
        uint32_t b[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          b[u] = pack2_f16(v[2 * u] + w[2 * u], v[2 * u + 1] + w[2 * u + 1]);
        tmem_st16(tbase + lane_base + kSColUT + 16 * hf, b);
      }
      tmem_st_wait();
      tc_fence_before();
      KDA_SMARK(2);
      named_bar(1, kSStateThreads);
#ifdef KDA_PHASE_PROFILE
      if (tid == 0) s_ts[3] = clock64();
#endif
      if (tid == 0 && ok1) mbar_arrive(&s_bars[kSBarUT]);
      // While MMA2 runs: the staged chunk's epilogue (the barrier above made
      // its rows visible).
      if constexpr (kGate) {
        if (pend) gated_finish(c - 1, prev_ok);
        pend = false;
      }
      KDA_SMARK(3);
      KDA_SMARK(4);
      // (E) Outputs to registers; new state -> bf16 operand copy (the serial
      // step) and, for the next chunk, the decayed fp32 state; checkpoints;
      // then hand the state to the next MMA1.
      const bool has_next = c + 1 < nck;
      const bool ok_next =
          !has_next || sync.wait_warp(kSBarFull0 + (s ^ 1), ((c + 1) >> 1) & 1);
      const bool ok2 = ok1 && sync.wait_warp(kSBarMMA2, c & 1);
      tc_fence_after();
#ifdef KDA_PHASE_PROFILE
      if (tid == 0) {
        const unsigned long long now = clock64();
        hand[2] += s_ts[1] - s_ts[3];
        hand[3] += now - s_ts[1];
      }
#endif
      KDA_SMARK(5);
      if (ok2) {
        const bool decay = has_next && ok_next;
        const float* gam =
            reinterpret_cast<const float*>(smem + kSOffRec + (s ^ 1) * kRecSlot + kRecG);
        const long long done = static_cast<long long>(win.cw0 + c + 1) * kC;
        float* ck = nullptr;
        if (args.ckpt && done <= t1 - t0 && done % args.ckpt_interval == 0) {
          const long long row = args.ckpt_offsets[n] + done / args.ckpt_interval - 1;
          ck = args.ckpt + (row * H + h) * kD * kD + j;
        }
        float sv[2][32];
        tmem_ld32(tbase + lane_base + kSColO + 32 * hf, ov);
        tmem_ld32(tbase + lane_base + kSColS + 64 * hf, sv[0]);
        tmem_ld32(tbase + lane_base + kSColS + 64 * hf + 32, sv[1]);
        tmem_ld_wait();
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          const int c0 = 64 * hf + 32 * cb;
          const float (&v)[32] = sv[cb];
          uint32_t b[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) b[u] = pack2(v[2 * u], v[2 * u + 1]);
          tmem_st16(tbase + lane_base + kSColSB + c0 / 2, b);
          if (decay) {
            uint32_t f[32];
#pragma unroll
            for (int u = 0; u < 32; u += 4) {
              const float4 gm = *reinterpret_cast<const float4*>(&gam[c0 + u]);
              f[u] = __float_as_uint(v[u] * gm.x);
              f[u + 1] = __float_as_uint(v[u + 1] * gm.y);
              f[u + 2] = __float_as_uint(v[u + 2] * gm.z);
              f[u + 3] = __float_as_uint(v[u + 3] * gm.w);
            }
            tmem_st32(tbase + lane_base + kSColS + c0, f);
          }
          if (ck) {
#pragma unroll
            for (int u = 0; u < 32; ++u) __stcs(ck + (c0 + u) * kD, v[u]);
          }
        }
      }
      KDA_SMARK(6);
      tmem_st_wait();
      tc_fence_before();
      KDA_SMARK(7);
      named_bar(1, kSStateThreads);
#ifdef KDA_PHASE_PROFILE
      if (tid == 0) s_ts[2] = clock64();
#endif
      if (tid == 0 && ok2 && ok_next && has_next) mbar_arrive(&s_bars[kSBarSB]);
      KDA_SMARK(8);
      prev_ok = ok2;
      ok = ok2 && ok_next;
    }
#ifdef KDA_PHASE_PROFILE
    if (blockIdx.x == 0 && blockIdx.y == 0 && (tid == 0 || tid == 64)) {
      for (int i = 0; i < 10; ++i) kda_split_clocks[(tid ? 10 : 0) + i] = prof_acc[i];
      if (tid == 0) {
        kda_split_clocks[30] = nck;
        for (int i = 0; i < 4; ++i) kda_split_clocks[20 + i] = hand[i];
      }
    }
#endif
    if (tmode == 0) emit_out(nck - 1, prev_ok, false);
    if (tid == 0) bulk_wait_all();
    if (__all_sync(0xFFFFFFFFu, !s_abort) && dst) {
      // After the last chunk the fp32 state carries no further decay.
#pragma unroll 1
      for (int cb = 0; cb < 2; ++cb) {
        const int c0 = 64 * hf + 32 * cb;
        float v[32];
        tmem_ld32(tbase + lane_base + kSColS + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 32; ++u) __stcs(dst + soff + (c0 + u) * kD + j, v[u]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (s_abort && tid == 0 && args.dev_status) atomicExch(args.dev_status, KDA_ERR_TIMEOUT);
  if (warp == 0) tmem_dealloc(tbase, kSTmemCols);
}

}  // namespace


namespace {

// The helper stream (highest priority) that runs the state kernels beside the
// caller's stream, and the events that order the two, one set per device.
constexpr int kEvRing = kSplitEvRing;
constexpr int kMaxDevices = 64;
struct SplitStreams {
  cudaStream_t state = nullptr;   // highest priority: overlapped windows' state passes
  cudaStream_t side = nullptr;    // lowest priority: a front-loaded call's second preparation
  cudaEvent_t fork = nullptr, join = nullptr;
  cudaEvent_t prep_done[kEvRing] = {}, state_done[kEvRing] = {};
  bool ready = false;
};
std::mutex g_split_mu;
SplitStreams g_split[kMaxDevices];

// Creates the device's helper stream and events on first use (call with
// g_split_mu held); nullptr if that fails.
SplitStreams* split_streams(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  SplitStreams& st = g_split[dev];
  if (st.ready) return &st;
  int least = 0, greatest = 0;
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) return nullptr;
  if (cudaStreamCreateWithPriority(&st.state, cudaStreamNonBlocking, greatest) != cudaSuccess ||
      cudaStreamCreateWithPriority(&st.side, cudaStreamNonBlocking, least) != cudaSuccess)
    return nullptr;
  bool ok = cudaEventCreateWithFlags(&st.fork, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&st.join, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kEvRing; ++i)
    ok = cudaEventCreateWithFlags(&st.prep_done[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&st.state_done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) return nullptr;
  st.ready = true;
  return &st;
}

}  // namespace


cudaError_t launch_chunk_split(const LaunchArgs& a, uint8_t* records, size_t record_bytes,
                               float* run_state, cudaStream_t stream) {
  if (a.n_seqs == 0 || a.heads == 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kPSmem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(chunk_state_kernel<false, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSSmem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(chunk_state_kernel<true, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSSmemGated));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(chunk_state_kernel<false, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSSmem));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  CUtensorMap maps[6] = {};
  const int n_maps = a.gate ? 6 : 5;
  if (a.total_tokens > 0) {
    const void* bases[6] = {a.q, a.k, a.v, a.g, a.out, a.gate};
    for (int i = 0; i < n_maps; ++i)
      if (!make_token_map(&maps[i], bases[i], a.heads, a.total_tokens))
        return cudaErrorInvalidValue;
  }
  SplitPlan P;
  if (!plan_split(a, record_bytes, sms, &P)) return cudaErrorInvalidValue;
  const long long pairs = P.pairs, max_chunks = P.max_chunks, item_bound_all = P.item_bound_all;
  const long long wc = P.wc, n_win = P.n_win, n_regions = P.n_regions;
  const bool overlap = P.overlap;
  const long long head = P.head;
  const size_t head_bytes = P.head_bytes;

  std::unique_lock<std::mutex> lock(g_split_mu, std::defer_lock);
  SplitStreams* st = nullptr;
  cudaStream_t s_state = stream;
  if (overlap || head) {
    lock.lock();
    st = split_streams(dev);
    if (!st) return cudaErrorUnknown;
  }
  if (overlap) {
    s_state = st->state;
    if ((e = cudaEventRecord(st->fork, stream)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(s_state, st->fork, 0)) != cudaSuccess) return e;
  }
  // The state pass of one window on stream s; with pdl, as a programmatic
  // dependent of the preparation just launched on s: its CTAs start on the
  // SMs the preparation's tail frees and set up while it finishes.
  auto launch_state = [&](const SplitWindow& win, cudaStream_t s, bool pdl) -> cudaError_t {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_seqs, a.heads, a.trans_M ? 2 : 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (a.trans_M) {
      cfg.blockDim = dim3(kSThreads);
      cfg.dynamicSmemBytes = kSSmem;
      return cudaLaunchKernelEx(&cfg, chunk_state_kernel<false, true>, a, win, maps[2], maps[4],
                                maps[5]);
    }
    if (a.gate) {
      cfg.blockDim = dim3(kSThreadsGated);
      cfg.dynamicSmemBytes = kSSmemGated;
      return cudaLaunchKernelEx(&cfg, chunk_state_kernel<true, false>, a, win, maps[2], maps[4],
                                maps[5]);
    }
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = kSSmem;
    return cudaLaunchKernelEx(&cfg, chunk_state_kernel<false, false>, a, win, maps[2], maps[4],
                              maps[5]);
  };
  auto launch_prep = [&](const SplitWindow& win, long long grid, cudaStream_t s) -> cudaError_t {
    if (grid <= 0) return cudaSuccess;
    chunk_prep_kernel<<<static_cast<unsigned>(grid), kPThreads, kPSmem, s>>>(a, win, maps[0],
                                                                              maps[1], maps[3]);
    return cudaGetLastError();
  };

  if (head) {
    // Front-loaded: prep(w0) and state(w0) on the caller's stream, the
    // latter a programmatic dependent (launched once every prep(w0) CTA has
    // started), so that its CTAs take the SMs prep(w0)'s tail frees before
    // anything else may be scheduled; prep(w1) on the lowest-priority side
    // stream once prep(w0) is complete, sized to the SMs the state pass
    // leaves; state(w1) on the caller's stream after both.
    SplitWindow w0{}, w1{};
    w0.rec = records;
    w0.cw0 = 0;
    w0.cw1 = static_cast<int>(head);
    w0.first = true;
    w0.s_run = run_state;
    w1.rec = records + head_bytes;
    w1.cw0 = static_cast<int>(head);
    w1.cw1 = static_cast<int>(max_chunks);
    w1.last = true;
    w1.s_run = run_state;
    const long long items0 = pairs * head < item_bound_all ? pairs * head : item_bound_all;
    long long items1 = pairs * (max_chunks - head);
    if (items1 > item_bound_all) items1 = item_bound_all;
    const long long grid0 = items0 < 2ll * sms ? items0 : 2ll * sms;
    if ((e = launch_prep(w0, grid0, stream)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(st->prep_done[0], stream)) != cudaSuccess) return e;
    if ((e = launch_state(w0, stream, grid0 > 0)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(st->side, st->prep_done[0], 0)) != cudaSuccess) return e;
    const long long free2 = 2ll * (sms - pairs);   // two CTAs on each SM the state pass leaves
    if ((e = launch_prep(w1, items1 < free2 ? items1 : free2, st->side)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(st->prep_done[1], st->side)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(stream, st->prep_done[1], 0)) != cudaSuccess) return e;
    return launch_state(w1, stream, false);
  }

  const size_t region_bytes = static_cast<size_t>(pairs * wc) * kRecBytes;
  for (long long w = 0; w < n_win || w == 0; ++w) {
    const long long cw0 = w * wc;
    SplitWindow win{};
    win.rec = records + static_cast<size_t>(w % n_regions) * region_bytes;
    win.cw0 = static_cast<int>(cw0);
    win.cw1 = static_cast<int>(cw0 + wc < max_chunks ? cw0 + wc : max_chunks);
    win.first = w == 0;
    win.last = w + 1 >= n_win;
    win.s_run = run_state;
    long long items = pairs * (win.cw1 - win.cw0);
    if (items > item_bound_all) items = item_bound_all;
    long long grid_p;
    if (overlap) {
      win.per_cta = kPrepItemsPerCta;
      grid_p = (items + kPrepItemsPerCta - 1) / kPrepItemsPerCta;
      if (w >= n_regions &&
          (e = cudaStreamWaitEvent(stream, st->state_done[(w - n_regions) % kEvRing], 0)) !=
              cudaSuccess)
        return e;
    } else {
      win.per_cta = 0;
      grid_p = items < 2ll * sms ? items : 2ll * sms;
    }
    if ((e = launch_prep(win, grid_p, stream)) != cudaSuccess) return e;
    if (overlap) {
      if ((e = cudaEventRecord(st->prep_done[w % kEvRing], stream)) != cudaSuccess) return e;
      if ((e = cudaStreamWaitEvent(s_state, st->prep_done[w % kEvRing], 0)) != cudaSuccess)
        return e;
    }
    if ((e = launch_state(win, s_state, !overlap && grid_p > 0)) != cudaSuccess) return e;
    if (overlap && (e = cudaEventRecord(st->state_done[w % kEvRing], s_state)) != cudaSuccess)
      return e;
  }
  if (overlap) {
    if ((e = cudaEventRecord(st->join, s_state)) != cudaSuccess) return e;
    if ((e = cudaStreamWaitEvent(stream, st->join, 0)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

#ifdef KDA_PHASE_PROFILE
extern "C" KDA_API int kda_debug_split_clocks(unsigned long long* host) {
  cudaError_t e = cudaMemcpyFromSymbol(host, kda_split_clocks, sizeof(unsigned long long) * 32);
  if (e == cudaSuccess)
    e = cudaMemcpyFromSymbol(host + 32, kda_prep_clocks, sizeof(unsigned long long) * 32);
  return static_cast<int>(e);
}
#endif

}  // namespace kda
