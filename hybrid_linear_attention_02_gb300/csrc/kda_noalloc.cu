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
// each call looks up its device address with cudaGetSymbolAddress for the
// device current at the call.  The lookup is repeated on every call rather
// than cached, so a new context on the device (after cudaDeviceReset, say),
// where the module may load at another address, never sees a stale pointer.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kNoAllocMaxSeqs = KDA_NOALLOC_MAX_SEQS;

static __device__ __align__(256) int g_seq_order[kNoAllocMaxSeqs];

// Device address of g_seq_order in the current device's context.
cudaError_t scratch_for_current_device(int** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_seq_order);
  if (e != cudaSuccess) return e;
  *out = static_cast<int*>(p);
  return cudaSuccess;
}

}  // namespace
}  // namespace kda

extern "C" int kda_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const void* g,
                                     const void* beta, const float* init_state,
                                     const int* cu_seqlens, void* out, float* final_state,
                                     int chunk, const kda_dims* d, int* dev_status,
                                     void* stream) {
  // The same checks, in the same order, as kda_chunk_fwd; only the scratch
  // limit is this entry point's own.
  int rc = kda::check_prefill_head(q, k, v, g, beta, out, chunk, d);
  if (rc != KDA_OK) return rc;
  if (d->n_seqs > kda::kNoAllocMaxSeqs) return KDA_ERR_SCRATCH_LIMIT;
  long long seq_len = 0;
  bool nothing_to_do = false;
  rc = kda::check_prefill_tail(init_state, final_state, cu_seqlens, d, &seq_len,
                               &nothing_to_do);
  if (rc != KDA_OK || nothing_to_do) return rc;

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
