// Device helpers and constants shared by the chunkwise tensor-core kernels
// (the fused kernel and the split prep / state kernels), plus the host helper
// that describes a [T, H, 128] bf16 tensor to TMA.
#pragma once

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "kda_sm100.cuh"

namespace kda {

constexpr int kC = 64;    // chunk length (tokens)
constexpr int kD = 128;   // dk = dv
constexpr float kLog2e = 1.4426950408889634f;

// [T, H, 128] bf16 viewed as a 3-D tensor (channel, head, token); one box is
// 64 channels x 1 head x 64 tokens, 128B-swizzled, zero-filled past T.
bool make_token_map(CUtensorMap* map, const void* base, int heads, long long tokens);

namespace chunk {

using namespace sm100;

__device__ __forceinline__ int khat_row0(int a) { return 8 * a * (a + 1); }  // 0, 16, 48, 96

// fp32 -> tf32 (round to nearest, ties away), as the m16n8k8 MMA reads it.
__device__ __forceinline__ uint32_t tf32_rna(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// One warp: D (16 x 8, fp32) += A (16 x 8, tf32, row) * B (8 x 8, tf32, col),
// in the m16n8k8 fragment layouts (group g = lane / 4, t = lane % 4): a0..a3
// = A[g][t], A[g+8][t], A[g][t+4], A[g+8][t+4]; b0, b1 = B[t][g], B[t+4][g];
// d0..d3 = D[g][2t], D[g][2t+1], D[g+8][2t], D[g+8][2t+1].
__device__ __forceinline__ void mma_m16n8k8_tf32(float& d0, float& d1, float& d2, float& d3,
                                                 uint32_t a0, uint32_t a1, uint32_t a2,
                                                 uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

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

// (lo, hi) rounded to fp16 (nearest even, saturating at +-65504), packed
// low half first.
__device__ __forceinline__ uint32_t pack2_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void st_tile8(uint8_t* tile, int row, int col, int rows,
                                         const float (&f)[8]) {
  *reinterpret_cast<uint4*>(tile + sw128_off(row, col, rows)) =
      make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

__device__ __forceinline__ void st_tile8_f16(uint8_t* tile, int row, int col, int rows,
                                             const float (&f)[8]) {
  *reinterpret_cast<uint4*>(tile + sw128_off(row, col, rows)) =
      make_uint4(pack2_f16(f[0], f[1]), pack2_f16(f[2], f[3]), pack2_f16(f[4], f[5]),
                 pack2_f16(f[6], f[7]));
}

// Shared by all roles: a wait that also gives up once any thread has given up.
struct Sync {
  uint64_t* bars;
  volatile int* abort;
  __device__ __forceinline__ bool wait(int b, uint32_t parity) {
    return wait_for(b, parity, 2000000000ull);
  }
  // As wait, called by all 32 lanes of a warp: the result is the same on
  // every lane (one lane that gave up makes the warp give up), so it may
  // guard warp-collective work (.sync.aligned TMEM loads, __syncwarp).
  __device__ __forceinline__ bool wait_warp(int b, uint32_t parity) {
    return __all_sync(0xFFFFFFFFu, wait_for(b, parity, 2000000000ull));
  }
  // As wait, giving up after limit_ns of wall time (a compile-time constant
  // in the kernels, so it costs them no register).
  __device__ __forceinline__ bool wait_for(int b, uint32_t parity, uint64_t limit_ns) {
    if (*abort) return false;
    if (mbar_try_wait(&bars[b], parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
      // Suspended until the phase completes (or 20 us pass), not spinning.
      if (mbar_try_wait_sleep(&bars[b], parity, 20000u)) return true;
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort = 1;
        return false;
      }
    }
  }
};

}  // namespace chunk
}  // namespace kda
