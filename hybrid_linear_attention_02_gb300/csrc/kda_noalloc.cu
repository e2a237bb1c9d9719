// kda_chunk_fwd_noalloc: the prefill entry point for callers that cannot
// allocate device memory.
//
// kda_chunk_fwd asks the caller for a workspace (the longest-first order in
// which packed sequences are scheduled).  Some callers cannot provide one:
// a plugin inside an inference engine that owns every device buffer and
// hands out only the tensors it planned, or a serving loop that must not call
// cudaMalloc (it synchronises the device and fragments a pool that is sized
// once at start-up).  This entry point keeps that scratch in a fixed
// file-scope device array instead, so a call needs nothing beyond its inputs
// and outputs.
//
// The array holds kNoAllocMaxSeqs sequence indices (256 KiB).  Every GPU that
// loads the library keeps it until the process exits.  Host code must not
// hand the array's symbol to a kernel (on the host it is only a stand-in);
// its device address is looked up once per device with
// cudaGetSymbolAddress, on the first call made while that device is current.
#include <mutex>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kNoAllocMaxSeqs = KDA_NOALLOC_MAX_SEQS;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int g_seq_order[kNoAllocMaxSeqs];

std::mutex g_setup_mutex;
int* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_seq_order on the current device (set up once per device).
cudaError_t scratch_for_current_device(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_seq_order);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace kda

extern "C" int kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                     const void* beta, const float* init_state,
                                     const int* cu_seqlens, void* out, float* final_state,
                                     int chunk, const kda_dims* d, int* dev_status,
                                     void* stream) {
  if (!d) return KDA_ERR_INVALID;
  if (d->n_seqs < 0 || d->heads < 0 || d->total_tokens < 0 || d->dk <= 0 || d->dv <= 0)
    return KDA_ERR_INVALID;
  if (d->dtype != KDA_F32 && d->dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
  if ((d->dk != 64 && d->dk != 128) || (d->dv != 64 && d->dv != 128)) return KDA_ERR_UNSUPPORTED;
  if (d->heads > 65535 && d->n_seqs > 0) return KDA_ERR_UNSUPPORTED;
  if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_UNSUPPORTED;
  if (d->n_seqs > kda::kNoAllocMaxSeqs) return KDA_ERR_SCRATCH_LIMIT;
  if (d->n_seqs == 0 || d->heads == 0) return d->total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID;
  if (d->total_tokens > 0) {
    if (!q || !k || !v || !g || !beta || !out) return KDA_ERR_INVALID;
    if (!kda::aligned16(q) || !kda::aligned16(k) || !kda::aligned16(v) || !kda::aligned16(g) ||
        !kda::aligned16(out))
      return KDA_ERR_ALIGNMENT;
  }
  if ((init_state && !kda::aligned16(init_state)) ||
      (final_state && !kda::aligned16(final_state)))
    return KDA_ERR_ALIGNMENT;
  long long seq_len = 0;
  if (!cu_seqlens) {
    if (d->total_tokens % d->n_seqs != 0) return KDA_ERR_INVALID;
    seq_len = d->total_tokens / d->n_seqs;
  }

  kda::LaunchArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.init_state = init_state;
  a.final_state = final_state;
  a.cu_seqlens = cu_seqlens;
  a.seq_len = seq_len;
  a.out = out;
  a.order = nullptr;
  a.dev_status = dev_status;
  a.n_seqs = d->n_seqs; a.heads = d->heads; a.dk = d->dk; a.dv = d->dv;
  a.dtype = d->dtype; a.chunk = chunk; a.total_tokens = d->total_tokens;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cu_seqlens && d->n_seqs > 1) {
    int* order = nullptr;
    if (kda::scratch_for_current_device(&order) != cudaSuccess) return KDA_ERR_CUDA;
    // The order kernel writes every one of the n_seqs entries it is asked
    // for, so nothing left from an earlier call is read.
    if (kda::launch_length_order(cu_seqlens, d->n_seqs, order, s) != cudaSuccess)
      return KDA_ERR_CUDA;
    a.order = order;
  }
  const cudaError_t e =
      kda::chunk_tc_supported(a) ? kda::launch_chunk_tc(a, s) : kda::launch_recurrent(a, s);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
