// C ABI of libkda.so: argument validation and dispatch.  Every check here
// runs on the host before any CUDA call, so an invalid call returns without
// touching the device.
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "kda_internal.h"

namespace {

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

bool supported_head_dim(int d) { return d == 64 || d == 128; }

}  // namespace

namespace kda {

int check_dims(const kda_dims* d) {
  if (!d) return KDA_ERR_INVALID;
  if (d->n_seqs < 0 || d->heads < 0 || d->total_tokens < 0 || d->dk <= 0 || d->dv <= 0)
    return KDA_ERR_INVALID;
  if (d->dtype != KDA_F32 && d->dtype != KDA_BF16) return KDA_ERR_UNSUPPORTED;
  if (!supported_head_dim(d->dk) || !supported_head_dim(d->dv)) return KDA_ERR_UNSUPPORTED;
  if (d->heads > 65535 && d->n_seqs > 0) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

int check_io_pointers(const void* q, const void* k, const void* v, const void* g,
                      const void* beta, const void* out, const kda_dims* d) {
  if (d->total_tokens == 0 || d->heads == 0) return KDA_OK;
  if (!q || !k || !v || !g || !beta || !out) return KDA_ERR_INVALID;
  // Vector loads and stores need 16-byte rows; rows are dk/dv elements long.
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(g, 16) ||
      !aligned(out, 16))
    return KDA_ERR_ALIGNMENT;
  return KDA_OK;
}

int check_prefill_head(const void* q, const void* k, const void* v, const void* g,
                       const void* beta, const void* out, int chunk, const kda_dims* d) {
  int rc = check_dims(d);
  if (rc != KDA_OK) return rc;
  if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_UNSUPPORTED;
  return check_io_pointers(q, k, v, g, beta, out, d);
}

int check_prefill_tail(const float* init_state, const float* final_state,
                       const int* cu_seqlens, const kda_dims* d, long long* seq_len,
                       bool* nothing_to_do) {
  *nothing_to_do = false;
  *seq_len = 0;
  const int N = d->n_seqs;
  if (N == 0 || d->heads == 0) {
    *nothing_to_do = true;
    return d->total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID;
  }
  if (!cu_seqlens) {
    if (d->total_tokens % N != 0) return KDA_ERR_INVALID;
    *seq_len = d->total_tokens / N;
  }
  if ((init_state && !aligned(init_state, 16)) || (final_state && !aligned(final_state, 16)))
    return KDA_ERR_ALIGNMENT;
  return KDA_OK;
}

}  // namespace kda

namespace {

using kda::LaunchArgs;
using kda::check_dims;
using kda::check_io_pointers;

constexpr size_t kWorkspaceAlign = 256;

size_t order_bytes(int n_seqs) {
  if (n_seqs <= 1) return 0;
  const size_t b = sizeof(int) * static_cast<size_t>(n_seqs);
  return (b + kWorkspaceAlign - 1) / kWorkspaceAlign * kWorkspaceAlign;
}

size_t align_up(size_t b) { return (b + kWorkspaceAlign - 1) / kWorkspaceAlign * kWorkspaceAlign; }

enum class Path { kRecurrent, kFused, kSplit };

// Which prefill kernels run for these dims (split only with room for its
// records in the workspace; KDA_CHUNK_PATH=fused|split overrides the default).
Path choose_path(const kda_dims* d, int chunk) {
  LaunchArgs a{};
  a.n_seqs = d->n_seqs; a.heads = d->heads; a.dk = d->dk; a.dv = d->dv;
  a.dtype = d->dtype; a.chunk = chunk; a.total_tokens = d->total_tokens;
  if (!kda::chunk_tc_supported(a)) return Path::kRecurrent;
  if (d->n_seqs > kda::kSplitMaxSeqs) return Path::kFused;
  const char* env = getenv("KDA_CHUNK_PATH");
  if (env && strcmp(env, "fused") == 0) return Path::kFused;
  if (env && strcmp(env, "split") == 0) return Path::kSplit;
  return static_cast<long long>(d->n_seqs) * d->heads <= kda::kSplitMaxPairs ||
                 d->n_seqs <= kda::kSplitAnyPairsSeqs
             ? Path::kSplit
             : Path::kFused;
}

// Split-path workspace after the order array: the carried state, then records.
size_t split_state_bytes(const kda_dims* d) {
  return align_up(static_cast<size_t>(d->n_seqs) * d->heads * d->dk * d->dv * sizeof(float));
}
size_t split_workspace_bytes(const kda_dims* d) {
  return split_state_bytes(d) + kda::split_record_bytes(d->n_seqs, d->total_tokens, d->heads);
}

}  // namespace

extern "C" {

int kda_version(void) { return 10000; }

const char* kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported dims, dtype or chunk size";
    case KDA_ERR_CUDA: return "CUDA call or kernel launch failed";
    case KDA_ERR_TIMEOUT: return "device wait timed out";
    case KDA_ERR_ALIGNMENT: return "buffer not 16-byte aligned";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_SCRATCH_LIMIT: return "more sequences than the no-alloc scratch array holds";
    case KDA_ERR_RANGE: return "input out of range: g outside [-5, 0] or beta outside [0, 1]";
    default: return "unknown status";
  }
}

size_t kda_chunk_fwd_workspace_size(const kda_dims* dims, int chunk) {
  if (check_dims(dims) != KDA_OK) return 0;
  size_t b = order_bytes(dims->n_seqs);
  if (dims->n_seqs > 0 && dims->heads > 0 && choose_path(dims, chunk) == Path::kSplit)
    b += split_workspace_bytes(dims);
  return b;
}

int kda_chunk_fwd_launch_count(const kda_dims* dims, int chunk, size_t workspace_bytes,
                               int varlen) {
  const int rc = check_dims(dims);
  if (rc != KDA_OK) return rc;
  if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_UNSUPPORTED;
  const int N = dims->n_seqs;
  if (N == 0 || dims->heads == 0) return 0;
  const size_t need = order_bytes(N);
  if (need > 0 && varlen && workspace_bytes < need) return KDA_ERR_WORKSPACE;   // as the call
  const int n_order = need > 0 && varlen ? 1 : 0;   // the length-order kernel
  const size_t split_min = need + split_state_bytes(dims) +
                           static_cast<size_t>(N) * dims->heads * kda::kSplitRecordBytes;
  if (choose_path(dims, chunk) != Path::kSplit || workspace_bytes < split_min)
    return n_order + 1;   // one fused or token-recurrence kernel
  size_t rec_bytes = workspace_bytes - need - split_state_bytes(dims);
  const size_t full = kda::split_record_bytes(N, dims->total_tokens, dims->heads);
  if (rec_bytes > full) rec_bytes = full;
  LaunchArgs a{};
  a.n_seqs = N; a.heads = dims->heads; a.dk = dims->dk; a.dv = dims->dv;
  a.dtype = dims->dtype; a.chunk = chunk; a.total_tokens = dims->total_tokens;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KDA_ERR_CUDA;
  const int c = kda::split_launch_count(a, rec_bytes, sms);
  return c < 0 ? KDA_ERR_WORKSPACE : n_order + c;
}

int kda_chunk_fwd_algorithm(const kda_dims* dims, int chunk) {
  const int rc = check_dims(dims);
  if (rc != KDA_OK) return rc;
  if (chunk != 16 && chunk != 32 && chunk != 64) return KDA_ERR_UNSUPPORTED;
  switch (choose_path(dims, chunk)) {
    case Path::kSplit: return KDA_ALGO_TCGEN05_SPLIT;
    case Path::kFused: return KDA_ALGO_TCGEN05;
    default: return KDA_ALGO_RECURRENT;
  }
}

}  // extern "C"

namespace {

// Optional parts of a prefill call: prefix-cache checkpoints (ckpt null: none)
// and the output epilogue (gate null: none).
struct Extras {
  float* ckpt = nullptr;
  const int* ckpt_offsets = nullptr;
  int ckpt_interval = 0;
  const void* gate = nullptr;
  const float* gate_w = nullptr;
  float gate_eps = 0.f;
  int withhold = 0;   // failure-detection self-test (see LaunchArgs::debug_withhold)
};

int check_gate(const void* gate, const float* gate_w, float eps) {
  if (!gate || !gate_w) return KDA_ERR_INVALID;
  if (!(eps >= 0.f) || eps > 3.0e38f) return KDA_ERR_INVALID;   // rejects NaN too
  if (!aligned(gate, 16) || !aligned(gate_w, 16)) return KDA_ERR_ALIGNMENT;
  return KDA_OK;
}

int chunk_fwd_impl(const void* q, const void* k, const void* v, const void* g, const void* beta,
                   const float* init_state, const int* cu_seqlens, void* out, float* final_state,
                   int chunk, const kda_dims* dims, void* workspace, size_t workspace_bytes,
                   int* dev_status, void* stream, const Extras& x) {
  float* ckpt = x.ckpt;
  const int* ckpt_offsets = x.ckpt_offsets;
  const int ckpt_interval = x.ckpt_interval;
  int rc = kda::check_prefill_head(q, k, v, g, beta, out, chunk, dims);
  if (rc != KDA_OK) return rc;
  if (ckpt) {
    if (!ckpt_offsets || ckpt_interval <= 0) return KDA_ERR_INVALID;
    if (ckpt_interval % 64 != 0) return KDA_ERR_UNSUPPORTED;
    if (!aligned(ckpt, 16)) return KDA_ERR_ALIGNMENT;
  }
  if (x.gate || x.gate_w) {
    if (dims->total_tokens > 0 && dims->heads > 0) {
      rc = check_gate(x.gate, x.gate_w, x.gate_eps);
      if (rc != KDA_OK) return rc;
    }
  }
  const int N = dims->n_seqs;
  long long seq_len = 0;
  bool nothing_to_do = false;
  rc = kda::check_prefill_tail(init_state, final_state, cu_seqlens, dims, &seq_len,
                               &nothing_to_do);
  if (rc != KDA_OK || nothing_to_do) return rc;
  const size_t need = order_bytes(N);
  if (need > 0 && cu_seqlens && (!workspace || workspace_bytes < need))
    return KDA_ERR_WORKSPACE;
  if (workspace && !aligned(workspace, kWorkspaceAlign)) return KDA_ERR_ALIGNMENT;

  LaunchArgs a{};
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.init_state = init_state;
  a.final_state = final_state;
  a.cu_seqlens = cu_seqlens;
  a.seq_len = seq_len;
  a.out = out;
  a.order = nullptr;
  a.dev_status = dev_status;
  a.n_seqs = N; a.heads = dims->heads; a.dk = dims->dk; a.dv = dims->dv;
  a.dtype = dims->dtype; a.chunk = chunk; a.total_tokens = dims->total_tokens;
  a.ckpt = ckpt;
  a.ckpt_offsets = ckpt ? ckpt_offsets : nullptr;
  a.ckpt_interval = ckpt ? ckpt_interval : 0;
  a.gate = x.gate;
  a.gate_w = x.gate_w;
  a.gate_eps = x.gate_eps;
  a.debug_withhold = x.withhold;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
#ifdef KDA_DEBUG_BOUNDS
  // Debug build: the inputs' range precondition is checked on the device
  // before the prefill runs (reported through dev_status, never trapped).
  if (dev_status && kda::launch_range_check(g, beta, dims->total_tokens, dims->heads, dims->dk,
                                            dims->dtype, dev_status, s) != cudaSuccess)
    return KDA_ERR_CUDA;
#endif
  if (need > 0 && cu_seqlens && N > 1) {   // one sequence: no order needed
    int* order = static_cast<int*>(workspace);
    if (kda::launch_length_order(cu_seqlens, N, order, s) != cudaSuccess) return KDA_ERR_CUDA;
    a.order = order;
  }
  cudaError_t e;
  Path path = choose_path(dims, chunk);
  if (x.withhold) {
    if (path == Path::kRecurrent) return KDA_ERR_UNSUPPORTED;
    path = x.withhold == 3 ? Path::kFused : Path::kSplit;
  }
  // The split form needs room for at least one record per pair after the
  // order array and the carried states; less room than the full size only
  // means more (smaller) windows.
  const size_t split_min = need + split_state_bytes(dims) +
                           static_cast<size_t>(N) * dims->heads * kda::kSplitRecordBytes;
  bool gate_done = path == Path::kRecurrent;   // the recurrence applies the epilogue itself
  if (x.withhold && path == Path::kSplit && !(workspace && workspace_bytes >= split_min))
    return KDA_ERR_WORKSPACE;
  if (path == Path::kSplit && workspace && workspace_bytes >= split_min) {
    gate_done = true;                          // so does the split form's state kernel
    uint8_t* ws = static_cast<uint8_t*>(workspace) + need;
    float* run = reinterpret_cast<float*>(ws);
    uint8_t* rec = ws + split_state_bytes(dims);
    size_t rec_bytes = workspace_bytes - need - split_state_bytes(dims);
    const size_t full = kda::split_record_bytes(N, dims->total_tokens, dims->heads);
    if (rec_bytes > full) rec_bytes = full;
    e = kda::launch_chunk_split(a, rec, rec_bytes, final_state ? final_state : run, s);
  } else if (path != Path::kRecurrent) {
    e = kda::launch_chunk_tc(a, s);
  } else {
    e = kda::launch_recurrent(a, s);
  }
  if (e == cudaSuccess && a.gate && !gate_done) e = kda::launch_gate_epilogue(a, s);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int decode_impl(const void* q, const void* k, const void* v, const void* g, const void* beta,
                float* state, void* out, const kda_dims* dims, int* dev_status, void* stream,
                const void* gate, const float* gate_w, float gate_eps);

}  // namespace

extern "C" {

int kda_chunk_fwd(const void* q, const void* k, const void* v, const void* g, const void* beta,
                  const float* init_state, const int* cu_seqlens, void* out, float* final_state,
                  int chunk, const kda_dims* dims, void* workspace, size_t workspace_bytes,
                  int* dev_status, void* stream) {
  return chunk_fwd_impl(q, k, v, g, beta, init_state, cu_seqlens, out, final_state, chunk, dims,
                        workspace, workspace_bytes, dev_status, stream, Extras{});
}

int kda_chunk_fwd_gated(const void* q, const void* k, const void* v, const void* g,
                        const void* beta, const float* init_state, const int* cu_seqlens,
                        const void* gate, const float* norm_weight, float eps, void* out,
                        float* final_state, int chunk, const kda_dims* dims, void* workspace,
                        size_t workspace_bytes, int* dev_status, void* stream) {
  if (!gate || !norm_weight) return KDA_ERR_INVALID;
  Extras x;
  x.gate = gate;
  x.gate_w = norm_weight;
  x.gate_eps = eps;
  return chunk_fwd_impl(q, k, v, g, beta, init_state, cu_seqlens, out, final_state, chunk, dims,
                        workspace, workspace_bytes, dev_status, stream, x);
}

int kda_chunk_fwd_checkpoints(const void* q, const void* k, const void* v, const void* g,
                              const void* beta, const float* init_state, const int* cu_seqlens,
                              void* out, float* final_state, int chunk, const kda_dims* dims,
                              void* workspace, size_t workspace_bytes, int* dev_status,
                              void* stream, float* checkpoints, const int* ckpt_offsets,
                              int ckpt_interval) {
  if (!checkpoints) return KDA_ERR_INVALID;
  Extras x;
  x.ckpt = checkpoints;
  x.ckpt_offsets = ckpt_offsets;
  x.ckpt_interval = ckpt_interval;
  return chunk_fwd_impl(q, k, v, g, beta, init_state, cu_seqlens, out, final_state, chunk, dims,
                        workspace, workspace_bytes, dev_status, stream, x);
}

size_t kda_chunk_transition_workspace_size(const kda_dims* dims) {
  if (check_dims(dims) != KDA_OK || dims->n_seqs <= 0 || dims->heads <= 0) return 0;
  return order_bytes(dims->n_seqs) + split_workspace_bytes(dims);
}

int kda_chunk_transition(const void* q, const void* k, const void* v, const void* g,
                         const void* beta, const int* cu_seqlens, float* trans_M, float* trans_H,
                         int chunk, const kda_dims* dims, void* workspace, size_t workspace_bytes,
                         int* dev_status, void* stream) {
  int rc = check_dims(dims);
  if (rc != KDA_OK) return rc;
  LaunchArgs a{};
  a.n_seqs = dims->n_seqs; a.heads = dims->heads; a.dk = dims->dk; a.dv = dims->dv;
  a.dtype = dims->dtype; a.chunk = chunk; a.total_tokens = dims->total_tokens;
  if (!kda::chunk_tc_supported(a) || dims->n_seqs > kda::kSplitMaxSeqs) return KDA_ERR_UNSUPPORTED;
  const int N = dims->n_seqs;
  if (N == 0 || dims->heads == 0) return dims->total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID;
  if (!trans_M || !trans_H) return KDA_ERR_INVALID;
  if (!aligned(trans_M, 16) || !aligned(trans_H, 16)) return KDA_ERR_ALIGNMENT;
  rc = check_io_pointers(q, k, v, g, beta, trans_H, dims);   // trans_H stands in for out
  if (rc != KDA_OK) return rc;
  long long seq_len = 0;
  if (!cu_seqlens) {
    if (dims->total_tokens % N != 0) return KDA_ERR_INVALID;
    seq_len = dims->total_tokens / N;
  }
  const size_t need = order_bytes(N);
  const size_t split_min = need + split_state_bytes(dims) +
                           static_cast<size_t>(N) * dims->heads * kda::kSplitRecordBytes;
  if (!workspace || workspace_bytes < split_min) return KDA_ERR_WORKSPACE;
  if (!aligned(workspace, kWorkspaceAlign)) return KDA_ERR_ALIGNMENT;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.cu_seqlens = cu_seqlens;
  a.seq_len = seq_len;
  a.out = trans_H;   // never written: transitions produce no outputs
  a.dev_status = dev_status;
  a.trans_M = trans_M;
  a.trans_H = trans_H;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (need > 0 && cu_seqlens && N > 1) {   // one sequence: no order needed
    if (kda::launch_length_order(cu_seqlens, N, reinterpret_cast<int*>(ws), s) != cudaSuccess)
      return KDA_ERR_CUDA;
    a.order = reinterpret_cast<int*>(ws);
  }
  size_t rec_bytes = workspace_bytes - need - split_state_bytes(dims);
  const size_t full = kda::split_record_bytes(N, dims->total_tokens, dims->heads);
  if (rec_bytes > full) rec_bytes = full;
  const cudaError_t e = kda::launch_chunk_split(a, ws + need + split_state_bytes(dims), rec_bytes,
                                                nullptr, s);
  return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_transition_apply(const float* M, const float* H, const float* S_in, float* S_out,
                         long long pairs, int dk, int dv, void* stream) {
  if (pairs < 0 || !((dk == 64 || dk == 128) && (dv == 64 || dv == 128))) {
    return pairs < 0 ? KDA_ERR_INVALID : KDA_ERR_UNSUPPORTED;
  }
  if (pairs == 0) return KDA_OK;
  if (!M || !S_in || !S_out) return KDA_ERR_INVALID;
  if (S_out == S_in || S_out == M) return KDA_ERR_INVALID;
  if (pairs > (1ll << 30)) return KDA_ERR_UNSUPPORTED;
  return kda::launch_transition_apply(M, H, S_in, S_out, pairs, dk, dv,
                                      static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KDA_OK
             : KDA_ERR_CUDA;
}

size_t kda_chunk_fwd_kcp_workspace_size(const kda_dims* dims, int n_segments) {
  if (check_dims(dims) != KDA_OK || n_segments < 1 || dims->n_seqs <= 0 || dims->heads <= 0)
    return 0;
  kda_dims sd = *dims;
  sd.n_seqs = dims->n_seqs * n_segments;
  const size_t pair = static_cast<size_t>(dims->dk) * dims->dv * sizeof(float);
  const size_t mats = align_up(static_cast<size_t>(sd.n_seqs) * dims->heads * pair);
  const size_t inner = std::max(kda_chunk_transition_workspace_size(&sd),
                                kda_chunk_fwd_workspace_size(&sd, 64));
  return align_up(sizeof(int) * (static_cast<size_t>(sd.n_seqs) + 1)) + 4 * mats + inner;
}

int kda_chunk_fwd_kcp(const void* q, const void* k, const void* v, const void* g,
                      const void* beta, const float* init_state, void* out, float* final_state,
                      int n_segments, const kda_dims* dims, void* workspace,
                      size_t workspace_bytes, int* dev_status, void* stream) {
  int rc = check_dims(dims);
  if (rc != KDA_OK) return rc;
  if (n_segments < 1) return KDA_ERR_INVALID;
  const int N = dims->n_seqs, H = dims->heads;
  if (N == 0 || H == 0) return dims->total_tokens == 0 ? KDA_OK : KDA_ERR_INVALID;
  if (dims->total_tokens % N != 0) return KDA_ERR_INVALID;
  if (dims->dk != dims->dv) return KDA_ERR_UNSUPPORTED;
  if (static_cast<long long>(N) * n_segments > kda::kSplitMaxSeqs) return KDA_ERR_UNSUPPORTED;
  kda_dims sd = *dims;
  sd.n_seqs = N * n_segments;
  LaunchArgs probe{};
  probe.n_seqs = sd.n_seqs; probe.heads = H; probe.dk = dims->dk; probe.dv = dims->dv;
  probe.dtype = dims->dtype; probe.chunk = 64; probe.total_tokens = dims->total_tokens;
  if (!kda::chunk_tc_supported(probe)) return KDA_ERR_UNSUPPORTED;
  rc = check_io_pointers(q, k, v, g, beta, out, dims);
  if (rc != KDA_OK) return rc;
  if ((init_state && !aligned(init_state, 16)) || (final_state && !aligned(final_state, 16)))
    return KDA_ERR_ALIGNMENT;
  const size_t need = kda_chunk_fwd_kcp_workspace_size(dims, n_segments);
  if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
  if (!aligned(workspace, kWorkspaceAlign)) return KDA_ERR_ALIGNMENT;

  // Workspace: segment offsets, then M, H, entry states and end states of
  // every segment, then the inner calls' workspace.
  const long long L = dims->total_tokens / N;
  const long long seg_len = ((L + n_segments - 1) / n_segments + 63) / 64 * 64;
  const size_t pair = static_cast<size_t>(dims->dk) * dims->dv;
  const size_t mats = align_up(static_cast<size_t>(sd.n_seqs) * H * pair * sizeof(float));
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* cu_seg = reinterpret_cast<int*>(ws);
  ws += align_up(sizeof(int) * (static_cast<size_t>(sd.n_seqs) + 1));
  float* Ms = reinterpret_cast<float*>(ws);
  float* Hs = reinterpret_cast<float*>(ws + mats);
  float* starts = reinterpret_cast<float*>(ws + 2 * mats);
  float* ends = reinterpret_cast<float*>(ws + 3 * mats);
  uint8_t* inner = ws + 4 * mats;
  const size_t inner_bytes = workspace_bytes - static_cast<size_t>(inner - static_cast<uint8_t*>(workspace));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t seq_bytes = static_cast<size_t>(H) * pair * sizeof(float);   // one sequence's states

  if (kda::launch_segment_offsets(cu_seg, N, L, n_segments, seg_len, s) != cudaSuccess)
    return KDA_ERR_CUDA;
  // 1. Every segment's transition (M, H), all segments at once.
  rc = kda_chunk_transition(q, k, v, g, beta, cu_seg, Ms, Hs, 64, &sd, inner, inner_bytes,
                            dev_status, stream);
  if (rc != KDA_OK) return rc;
  // 2. Entry states: segment 0 starts from init_state, segment s + 1 from
  //    M_s S_s + H_s (the composed prefix), for every sequence at once.
  cudaError_t e =
      init_state ? cudaMemcpy2DAsync(starts, n_segments * seq_bytes, init_state, seq_bytes,
                                     seq_bytes, N, cudaMemcpyDeviceToDevice, s)
                 : cudaMemset2DAsync(starts, n_segments * seq_bytes, 0, seq_bytes, N, s);
  if (e != cudaSuccess) return KDA_ERR_CUDA;
  const long long stride = static_cast<long long>(n_segments) * H;   // pairs between sequences
  for (int sg = 0; sg + 1 < n_segments; ++sg) {
    const size_t off = static_cast<size_t>(sg) * H * pair;
    e = kda::launch_transition_apply_strided(Ms + off, Hs + off, starts + off,
                                             starts + off + H * pair, N, H, stride, stride,
                                             stride, dims->dk, dims->dv, s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
  }
  // 3. Every segment from its entry state: outputs, and end states.
  rc = kda_chunk_fwd(q, k, v, g, beta, starts, cu_seg, out, ends, 64, &sd, inner, inner_bytes,
                     dev_status, stream);
  if (rc != KDA_OK) return rc;
  if (final_state) {
    e = cudaMemcpy2DAsync(final_state, seq_bytes,
                          reinterpret_cast<uint8_t*>(ends) + (n_segments - 1) * seq_bytes,
                          n_segments * seq_bytes, seq_bytes, N, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return KDA_ERR_CUDA;
  }
  return KDA_OK;
}

int kda_prologue(const void* q_pre, const void* k_pre, const void* z, const float* conv_q,
                 const float* conv_k, const float* a_log, const int* cu_seqlens, void* q, void* k,
                 void* g, const kda_dims* dims, void* stream) {
  int rc = check_dims(dims);
  if (rc != KDA_OK) return rc;
  const int N = dims->n_seqs;
  if (dims->total_tokens == 0 || dims->heads == 0) return KDA_OK;
  if (N <= 0) return KDA_ERR_INVALID;
  if (!q_pre || !k_pre || !z || !conv_q || !conv_k || !a_log || !q || !k || !g)
    return KDA_ERR_INVALID;
  const void* vec[] = {q_pre, k_pre, z, conv_q, conv_k, q, k, g};
  for (const void* p : vec)
    if (!aligned(p, 16)) return KDA_ERR_ALIGNMENT;
  long long seq_len = 0;
  if (!cu_seqlens) {
    if (dims->total_tokens % N != 0) return KDA_ERR_INVALID;
    seq_len = dims->total_tokens / N;
  }
  kda::PrologueArgs a{};
  a.q_pre = q_pre; a.k_pre = k_pre; a.z = z;
  a.conv_q = conv_q; a.conv_k = conv_k; a.a_log = a_log;
  a.cu_seqlens = cu_seqlens; a.seq_len = seq_len;
  a.q = q; a.k = k; a.g = g;
  a.n_seqs = N; a.heads = dims->heads; a.dk = dims->dk; a.dtype = dims->dtype;
  a.total_tokens = dims->total_tokens;
  return kda::launch_prologue(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KDA_OK
             : KDA_ERR_CUDA;
}

int kda_debug_chunk_fwd_withhold(int which, const void* q, const void* k, const void* v,
                                 const void* g, const void* beta, const float* init_state,
                                 void* out, float* final_state, const kda_dims* dims,
                                 void* workspace, size_t workspace_bytes, int* dev_status,
                                 void* stream) {
  if (which < 1 || which > 3 || !dev_status) return KDA_ERR_INVALID;
  Extras x;
  x.withhold = which;
  return chunk_fwd_impl(q, k, v, g, beta, init_state, nullptr, out, final_state, 64, dims,
                        workspace, workspace_bytes, dev_status, stream, x);
}

int kda_check_inputs(const void* g, const void* beta, const kda_dims* dims, int* dev_status,
                     void* stream) {
  const int rc = check_dims(dims);
  if (rc != KDA_OK) return rc;
  if (!dev_status) return KDA_ERR_INVALID;
  if (dims->total_tokens == 0 || dims->heads == 0) return KDA_OK;
  if (!g || !beta) return KDA_ERR_INVALID;
  if (!aligned(g, 16)) return KDA_ERR_ALIGNMENT;
  return kda::launch_range_check(g, beta, dims->total_tokens, dims->heads, dims->dk, dims->dtype,
                                 dev_status, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KDA_OK
             : KDA_ERR_CUDA;
}

int kda_debug_bounds_build(void) {
#ifdef KDA_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

int kda_decode_step_gated(const void* q, const void* k, const void* v, const void* g,
                          const void* beta, const void* gate, const float* norm_weight,
                          float eps, float* state, void* out, const kda_dims* dims,
                          int* dev_status, void* stream) {
  if (!gate || !norm_weight) return KDA_ERR_INVALID;
  return decode_impl(q, k, v, g, beta, state, out, dims, dev_status, stream, gate, norm_weight,
                     eps);
}

int kda_decode_step(const void* q, const void* k, const void* v, const void* g, const void* beta,
                    float* state, void* out, const kda_dims* dims, int* dev_status, void* stream) {
  return decode_impl(q, k, v, g, beta, state, out, dims, dev_status, stream, nullptr, nullptr,
                     0.f);
}

}  // extern "C"

namespace {

int decode_impl(const void* q, const void* k, const void* v, const void* g, const void* beta,
                float* state, void* out, const kda_dims* dims, int* dev_status, void* stream,
                const void* gate, const float* gate_w, float gate_eps) {
  int rc = check_dims(dims);
  if (rc != KDA_OK) return rc;
  if (dims->total_tokens != dims->n_seqs) return KDA_ERR_INVALID;
  if (dims->n_seqs == 0 || dims->heads == 0) return KDA_OK;
  rc = check_io_pointers(q, k, v, g, beta, out, dims);
  if (rc != KDA_OK) return rc;
  if (!state) return KDA_ERR_INVALID;
  if (!aligned(state, 16)) return KDA_ERR_ALIGNMENT;
  if (gate || gate_w) {
    rc = check_gate(gate, gate_w, gate_eps);
    if (rc != KDA_OK) return rc;
  }
  LaunchArgs a{};
  a.gate = gate;
  a.gate_w = gate_w;
  a.gate_eps = gate_eps;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.init_state = state;
  a.final_state = state;
  a.cu_seqlens = nullptr;
  a.seq_len = 1;
  a.out = out;
  a.order = nullptr;
  a.dev_status = dev_status;
  a.n_seqs = dims->n_seqs; a.heads = dims->heads; a.dk = dims->dk; a.dv = dims->dv;
  a.dtype = dims->dtype; a.chunk = 1; a.total_tokens = dims->total_tokens;
#ifdef KDA_DEBUG_BOUNDS
  if (dev_status && kda::launch_range_check(g, beta, dims->n_seqs, dims->heads, dims->dk,
                                            dims->dtype, dev_status,
                                            static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KDA_ERR_CUDA;
#endif
  return kda::launch_recurrent(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KDA_OK
             : KDA_ERR_CUDA;
}

}  // namespace
