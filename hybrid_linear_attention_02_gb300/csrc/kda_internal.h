// Internal declarations shared by the translation units of libkda.so.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Host-side argument checks shared by the entry points (kda_api.cu); each
// returns a kda_status.  check_dims: the shape record.  check_io_pointers:
// q, k, v, g, beta, out present and 16-byte aligned (unless there is no
// token).  check_prefill_head: check_dims, the chunk size, then the pointers.
// check_prefill_tail: an empty call (no sequence or no head) sets
// *nothing_to_do; otherwise the equal-length split when cu_seqlens is NULL
// (*seq_len) and the states' alignment.
int check_dims(const kda_dims* d);
int check_io_pointers(const void* q, const void* k, const void* v, const void* g,
                      const void* beta, const void* out, const kda_dims* d);
int check_prefill_head(const void* q, const void* k, const void* v, const void* g,
                       const void* beta, const void* out, int chunk, const kda_dims* d);
int check_prefill_tail(const float* init_state, const float* final_state,
                       const int* cu_seqlens, const kda_dims* d, long long* seq_len,
                       bool* nothing_to_do);

// Arguments of one prefill or decode launch, already validated on the host.
struct LaunchArgs {
  const void *q, *k, *v, *g, *beta;
  const float* init_state;  // nullable: zeros
  float* final_state;       // nullable
  const int* cu_seqlens;    // nullable: equal lengths seq_len
  long long seq_len;        // tokens per sequence when cu_seqlens is null
  void* out;
  const int* order;         // nullable: sequence processing order (longest first)
  int* dev_status;          // nullable
  int n_seqs, heads, dk, dv, dtype, chunk;
  long long total_tokens;
  float* ckpt;              // nullable: state after every ckpt_interval tokens
  const int* ckpt_offsets;  // [n_seqs + 1] first checkpoint row of each sequence
  int ckpt_interval;        // tokens between checkpoints (multiple of 64) or 0
  // Output epilogue (nullable gate: none): out = RMSNorm(o) * gate_w * sigmoid(gate).
  const void* gate;         // [T, H, dv] gate pre-activation, dtype of v
  const float* gate_w;      // [dv] RMSNorm scale
  float gate_eps;
  // Segment transitions (split form only; trans_M null: off): per (sequence,
  // head) M [dk, dk] and H [dk, dv] with S_end = M S_0 + H; no outputs.
  float* trans_M;
  float* trans_H;
  // Failure-detection self-test only (0 in every production call): one copy
  // is never issued, so the kernels' bounded waits expire.  1: the split
  // state kernel's first record of pair (0, 0); 2: the split preparation
  // kernel's first raw tiles in CTA 0; 3: the fused kernel's first raw tiles
  // in CTA (0, 0).
  int debug_withhold;
};

// fp32 CUDA-core kernel that walks the recurrence token by token with the
// state on chip.  Serves fp32 prefill, the shapes the tensor-core kernel does
// not cover, and (with one token per sequence) the decode step.
cudaError_t launch_recurrent(const LaunchArgs& a, cudaStream_t stream);

// The output epilogue as its own pass over `out` (in place): for every
// (token, head) row, out = out / sqrt(mean(out^2) + eps) * gate_w * sigmoid(gate).
cudaError_t launch_gate_epilogue(const LaunchArgs& a, cudaStream_t stream);

// S_out[p] = M[p] S_in[p] (+ H[p] when H is not null), fp32, for `pairs`
// independent (dk x dk) (dk x dv) products; S_out must not alias M or S_in.
cudaError_t launch_transition_apply(const float* M, const float* H, const float* S_in,
                                    float* S_out, long long pairs, int dk, int dv,
                                    cudaStream_t stream);

// The same over a grid of pairs: pair (o, i), o < n_outer, i < n_inner, of
// each array at base + (o * stride + i) * (its matrix size).
cudaError_t launch_transition_apply_strided(const float* M, const float* H, const float* S,
                                            float* out, long long n_outer, int n_inner,
                                            long long m_stride, long long s_stride,
                                            long long o_stride, int dk, int dv,
                                            cudaStream_t stream);

// cu_seg[n * P + s] = start of segment s of sequence n (equal-length sequences
// of L tokens cut into P segments of seg_len tokens, the last ones shorter or
// empty); cu_seg[N * P] = N * L.
cudaError_t launch_segment_offsets(int* cu_seg, int n_seqs, long long seq_len, int n_segments,
                                   long long seg_len, cudaStream_t stream);

// The input prologue: q, k from their pre-activations (4-tap causal depthwise
// convolution, Swish, L2 norm) and g = -5 sigmoid(exp(A_h) z).
struct PrologueArgs {
  const void *q_pre, *k_pre, *z;
  const float *conv_q, *conv_k;   // [H, dk, 4]
  const float* a_log;             // [H]
  const int* cu_seqlens;          // nullable: sequences of seq_len tokens
  long long seq_len;
  void *q, *k, *g;
  int n_seqs, heads, dk, dtype;
  long long total_tokens;
};
cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t stream);

// Sets *dev_status to KDA_ERR_RANGE (unless it holds an error already) when
// any g of [tokens, heads, dk] lies outside [-5, 0] or any beta of
// [tokens, heads] outside [0, 1] (NaN included).  g is 16-byte aligned.
cudaError_t launch_range_check(const void* g, const void* beta, long long tokens, int heads,
                               int dk, int dtype, int* dev_status, cudaStream_t stream);

// Writes order[0..N) = sequence indices by decreasing length (ties by index).
cudaError_t launch_length_order(const int* cu_seqlens, int n_seqs, int* order,
                                cudaStream_t stream);

// bf16 chunkwise tcgen05/TMA kernel (dk = dv = 128, chunk = 64).
bool chunk_tc_supported(const LaunchArgs& a);
cudaError_t launch_chunk_tc(const LaunchArgs& a, cudaStream_t stream);

// The same computation split into a parallel preparation kernel, which writes
// one record per chunk, and a serial state kernel (for few sequence-head
// pairs, or few sequences).  Records of a window of chunk indices [cw0, cw1)
// of every sequence; the state is carried between windows in s_run.
constexpr int kSplitMaxSeqs = 1024;              // sequences per call on this path
constexpr long long kSplitMaxPairs = 304;        // default: sequence-head pairs up to this,
constexpr int kSplitAnyPairsSeqs = 32;           // or any pair count with this many sequences
constexpr size_t kSplitRecordBytes = 66048;      // one chunk record
// Record buffer cap (bytes): pairs that leave half of a GB300's 152 SMs free
// run overlapped windows, for which a small buffer is best; otherwise windows
// run one after another and fewer of them is better.
constexpr long long kSplitOverlapPairs = 76;
constexpr size_t kSplitRecordBudgetOverlap = 2ull << 30;
constexpr size_t kSplitRecordBudget = 32ull << 30;

struct SplitWindow {
  uint8_t* rec;
  int cw0, cw1;
  bool first, last;
  float* s_run;        // state between windows (nullable with a single window)
  int per_cta;         // prep items per CTA (contiguous), or 0: strided over the grid
};

// Record-buffer bytes the split path needs for these sizes.
size_t split_record_bytes(int n_seqs, long long total_tokens, int heads);
constexpr int kSplitChunk = 64;                   // the split form's chunk length
constexpr long long kSplitMinWindowChunks = 64;   // overlapped windows: at least this many chunks
constexpr int kSplitEvRing = 64;                  // overlapped windows: events per device

// The window schedule of one split-form call (kda_split_plan.cu; no CUDA
// calls): plan_split fills it, false when the record buffer holds less than
// one record per pair.
struct SplitPlan {
  long long pairs = 0, cap_items = 0, max_chunks = 0, item_bound_all = 0;
  long long wc = 0, n_win = 0, n_regions = 0;   // windows of wc chunks, n_regions record regions
  bool overlap = false;                         // overlapped windows (helper stream)
  long long head = 0;      // > 0: front-loaded windows [0, head) and [head, max_chunks)
  size_t head_bytes = 0;   // records of the first front-loaded window
};
bool plan_split(const LaunchArgs& a, size_t record_bytes, int sms, SplitPlan* P);
// KDA_SPLIT_SERIAL=1: the split form's windows run one after another on the
// caller's stream (no helper stream).
bool split_serial_only();
// Kernels one launch_chunk_split call launches with this record buffer on a
// device of sms SMs (-1 if the buffer holds less than one record per pair).
int split_launch_count(const LaunchArgs& a, size_t record_bytes, int sms);
cudaError_t launch_chunk_split(const LaunchArgs& a, uint8_t* records, size_t record_bytes,
                               float* run_state, cudaStream_t stream);

}  // namespace kda
