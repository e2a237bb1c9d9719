// The split prefill's window schedule (host code only; the kernels and
// their launches live in kda_chunk_split.cu).  A call's chunks run in windows
// of chunk indices: serial windows one after another, overlapped windows
// whose preparation runs beside the previous window's state pass, or two
// front-loaded windows.  Which one, and how wide, follows from the pair
// count, the SM count and the record buffer the caller's workspace holds.
#include <stdlib.h>
#include <string.h>

#include "kda_internal.h"

namespace kda {

// KDA_SPLIT_SERIAL=1 runs the windows of the split form one after another on
// the caller's stream (no helper stream).
bool split_serial_only() {
  const char* v = getenv("KDA_SPLIT_SERIAL");
  return v && strcmp(v, "1") == 0;
}

size_t split_record_bytes(int n_seqs, long long total_tokens, int heads) {
  const long long pairs = static_cast<long long>(n_seqs) * heads;
  const long long bound = static_cast<long long>(heads) * (total_tokens / kSplitChunk + n_seqs);
  size_t cap = pairs <= kSplitOverlapPairs ? kSplitRecordBudgetOverlap : kSplitRecordBudget;
  if (const char* v = getenv("KDA_SPLIT_RECORD_GIB")) {   // tuning knob: the cap in GiB
    const long long g = atoll(v);
    if (g > 0) cap = static_cast<size_t>(g) << 30;
  }
  const long long budget = static_cast<long long>(cap / kSplitRecordBytes);
  long long items = bound < budget ? bound : budget;
  if (items < pairs) items = pairs;
  return static_cast<size_t>(items) * kSplitRecordBytes;
}

bool plan_split(const LaunchArgs& a, size_t record_bytes, int sms, SplitPlan* P) {
  const long long pairs = static_cast<long long>(a.n_seqs) * a.heads;
  const long long cap_items = static_cast<long long>(record_bytes / kSplitRecordBytes);
  if (cap_items < pairs) return false;
  const long long max_chunks = (a.total_tokens + kSplitChunk - 1) / kSplitChunk;   // of any one sequence
  const long long item_bound_all =
      static_cast<long long>(a.heads) * (a.total_tokens / kSplitChunk + a.n_seqs);

  // Overlapped form, for pairs that leave at least half the SMs to spare:
  // about eight windows of at least kSplitMinWindowChunks chunks, two or more of
  // which fit in the record buffer at once.  The preparation of window w + 1
  // (caller's stream, short-lived CTAs) then runs beside the state pass of
  // window w (helper stream, higher priority) on the SMs the state pass
  // leaves idle, and a window's record region is rewritten only after the
  // state pass that read it.
  long long wc = (max_chunks + 7) / 8;
  if (wc < kSplitMinWindowChunks) wc = kSplitMinWindowChunks;
  if (pairs * wc * 2 > cap_items) wc = cap_items / (2 * pairs);
  long long n_win = wc > 0 ? (max_chunks + wc - 1) / wc : 0;
  long long n_regions = wc > 0 ? cap_items / (pairs * wc) : 0;
  if (n_regions > kSplitEvRing / 2) n_regions = kSplitEvRing / 2;
  bool overlap = 2 * pairs <= sms && wc > 0 && n_win >= 2 && n_regions >= 2 && !a.trans_M;
  // KDA_SPLIT_WINDOW=n: overlapped windows of n chunks whatever the pair count
  // (a tuning knob); KDA_SPLIT_SERIAL=1: never overlap.
  if (const char* fw = getenv("KDA_SPLIT_WINDOW")) {
    const long long f = atoll(fw);
    if (f > 0 && pairs * f * 2 <= cap_items) {
      wc = f;
      n_win = (max_chunks + wc - 1) / wc;
      n_regions = cap_items / (pairs * wc);
      if (n_regions > kSplitEvRing / 2) n_regions = kSplitEvRing / 2;
      overlap = n_win >= 2;
    }
  }
  if (split_serial_only() || a.trans_M) overlap = false;
  if (!overlap) {
    if (cap_items >= item_bound_all) {
      // Every record of the call fits: one window over every chunk index
      // (max_chunks bounds each sequence by the total, so cap_items / pairs
      // would cut packed sequences into windows most of which hold nothing).
      wc = max_chunks > 0 ? max_chunks : 1;
      n_win = 1;
    } else {
      wc = cap_items / pairs;
      n_win = max_chunks > 0 ? (max_chunks + wc - 1) / wc : 1;
    }
    n_regions = 1;
  }
  // Front-loaded form, for pairs that fit on the SMs in one wave but leave
  // fewer than half of them free, when every record fits at once: a first
  // window of most of the chunks is prepared on every SM; its state pass
  // then runs beside the preparation of a short second window, two
  // persistent CTAs on each SM it leaves free, and the second state pass
  // ends the call.  The split balances the middle phase: a state-pass chunk
  // takes about 0.22 of a preparation item's CTA time (measured on these
  // kernels), so tail / head = 0.44 (SMs - pairs) / pairs.
  // KDA_SPLIT_TAIL=n sets the second window's chunks (0: off; a tuning knob).
  long long head = 0;
  size_t head_bytes = 0;
  if (!overlap && !split_serial_only() && !a.trans_M && 2 * pairs > sms &&
      8 * (sms - pairs) >= sms && max_chunks >= 16) {
    const double r = 0.44 * static_cast<double>(sms - pairs) / static_cast<double>(pairs);
    long long tail = static_cast<long long>(static_cast<double>(max_chunks) * r / (1.0 + r));
    if (const char* ft = getenv("KDA_SPLIT_TAIL")) tail = atoll(ft);
    if (tail >= 1 && tail < max_chunks) {
      const long long h0 = max_chunks - tail;
      const long long b0 = pairs * h0 < item_bound_all ? pairs * h0 : item_bound_all;
      const long long b1 = pairs * tail < item_bound_all ? pairs * tail : item_bound_all;
      if (b0 + b1 <= cap_items) {
        head = h0;
        head_bytes = static_cast<size_t>(b0) * kSplitRecordBytes;
      }
    }
  }

  P->pairs = pairs;
  P->cap_items = cap_items;
  P->max_chunks = max_chunks;
  P->item_bound_all = item_bound_all;
  P->wc = wc;
  P->n_win = n_win;
  P->n_regions = n_regions;
  P->overlap = overlap;
  P->head = head;
  P->head_bytes = head_bytes;
  return true;
}

int split_launch_count(const LaunchArgs& a, size_t record_bytes, int sms) {
  SplitPlan P;
  if (!plan_split(a, record_bytes, sms, &P)) return -1;
  if (P.head) return 4;   // two preparations, two state passes
  long long n = 0;
  for (long long w = 0; w < P.n_win || w == 0; ++w) {
    const long long cw0 = w * P.wc;
    const long long cw1 = cw0 + P.wc < P.max_chunks ? cw0 + P.wc : P.max_chunks;
    if (cw1 > cw0) ++n;   // the preparation (none for a window without chunks)
    ++n;                  // the state pass
  }
  return static_cast<int>(n);
}

}  // namespace kda
