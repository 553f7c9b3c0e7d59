// tsa_kernels.h -- argument blocks and launchers of the libtsa kernels
// (host <-> device contract inside the library; not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "tsa_internal.cuh"

namespace tsa {

// Per-head activity filter: a head takes part iff
// head_active == nullptr || head_active[b*Hq + h] == active_value.
//
// Key scan: logits of every active head; window logits go to wz, pool
// positions are emitted as (position, logit) pairs when their
// order-preserving logit key is >= the head's emission key.
// Pairs go to the head's dense list: every warp bump-allocates runs of 8
// slots from dense_n and pads the unused tail of its last run with sentinel
// pairs (position 0xffffffff).  The finish kernel counts the pairs' bins to
// find b* and checks the emission.
// With head_active set, the kernel waits for the previous grid (which wrote
// it) before it starts; otherwise its producer streams keys at once.
struct ScanArgs {
  const uint16_t* q;         // bf16 [B][Hq][128]
  KvView kv;
  const int32_t* lens;       // [B] device, or nullptr -> len_host + b * len_step
  int64_t len_host, len_step;
  int B, Hq;
  float scale;
  int n_init, n_recent;      // static window (logits to wz, not emitted)
  const int32_t* head_active;  // heads with head_active[bh] == active_value take part
  int active_value;            // (nullptr: every head); written by the previous kernel
  uint32_t* tile_ctr;        // (zeroed) dynamic tile claims
  const uint32_t* emit_key;   // [B][Hq] emission keys, persistent across calls (any value is safe)
  uint2* dense;              // [B][Hq][dense_stride] (position, logit bits)
  int32_t* dense_n;          // [B][Hq] x kCtrStride (zeroed) slots allocated (pairs + sentinels)
  int64_t dense_stride;      // >= l_cap + slack for the padding
  float* wz;                 // [B][Hq][wz_stride] window logits
  int wz_stride;
  int* status;
  // Bounded waits give up after wait_ns (0: the default limit).  Fault
  // injection for tests of the error path: with stall_first_copy set, CTA 0
  // never issues the copy of its first tile, so that its consumers' wait
  // runs out (bounded) and the call reports a timeout.
  long long wait_ns;
  int stall_first_copy;
  TraceBuf trace;
};
cudaError_t launch_scan(const ScanArgs& a, int grid, cudaStream_t st, bool pdl);

struct RetopkSeq;  // one sequence of a ReTopK step (below)

// Finish: one cluster of NC CTAs per (sequence, query head) takes every
// emitted pair as a candidate and selects the exact top-K among them with a
// cluster-wide radix on the 64-bit rank key; when fewer pairs than K were
// emitted it re-scores the head's keys to count every 11-bit bin, finds the
// threshold bin b* and re-emits the pairs with bin >= b* itself (same
// tensor-core arithmetic as the scan, so every logit is bit-identical); it
// stores the next call's emission key and attends over the window and the
// selected rows with the gamma merge.
struct FinishArgs {
  const uint16_t* q;         // bf16 [B][Hq][128] (re-emission only)
  KvView kv;
  const int32_t* lens;
  int64_t len_host, len_step;
  int B, Hq;
  float scale;
  int K, n_init, n_recent;
  int32_t* counts_out;       // [B][Hq] or nullptr: |selected set| = min(K, |P|)
  uint32_t* emit_key;        // [B][Hq] the scan's emission key; the next call's is stored
  float* emit_margin;        // [B][Hq] per-head margin of the emission key (persistent)
  uint32_t* tile_ctr;        // the scan's tile claims (cleared)
  int* status;               // sticky error bits: a timeout makes the outputs NaN
  uint2* dense;              // [B][Hq][dense_stride] emitted pairs
  int32_t* dense_n;
  int64_t dense_stride;
  uint64_t* spill;           // [B][Hq][dense_stride] candidates past shared memory
  const float* wz;           // window logits [B][Hq][wz_stride]
  int wz_stride;
  float* out;                // [B][Hq][128]
  float* lse_out;            // [B][Hq] or nullptr
  int32_t* topk_idx;         // [B][Hq] rows of topk_stride, or nullptr
  float* topk_score;         // same layout, or nullptr
  int64_t topk_stride;       // elements between heads' output rows (K for decode)
  // Given-set heads (all nullptr for decode): heads with path == 0 rescore
  // their mcand candidates cand (positions, rows of cand_cap) and select
  // among them (no bins, no emission key).  With seqs set (a ReTopK step)
  // every head of sequence b pushes (qbar_t, S_t) into the FIFO entry
  // seqs[b].fifo_head of its state (S_t written straight into the entry's
  // support row); attend_set leaves seqs null.
  const int32_t* path;
  const int32_t* mcand;
  const uint32_t* cand;
  int cand_cap;
  const float* push_qbar;    // [B][Hq][128]
  const RetopkSeq* seqs;     // [B] (device, written by the selector)
  int C;
  TraceBuf trace;
};
cudaError_t launch_finish(const FinishArgs& a, cudaStream_t st);

cudaError_t launch_lse_merge(const float* oa, const float* la, const float* ob,
                             const float* lb, float* oo, float* lo, int rows, int d,
                             cudaStream_t st);

// ReTopK ------------------------------------------------------------------
// One sequence of a ReTopK step: its FIFO state (caller memory) and this
// step's length, oldest entry and refresh flag.
struct RetopkSeq {
  float* qbar;               // [Hq][C][128]
  int32_t* sup;              // [Hq][C][K]
  int32_t* sup_n;            // [Hq][C]
  int64_t L;                 // cache length this step
  int32_t fifo_head;         // slot of the oldest entry (overwritten by this step)
  int32_t refresh;           // t % T_r == 0
};
constexpr int kMaxRetopkBatch = 64;  // sequences of one step (kernel-parameter table)

struct RetopkSelArgs {
  const uint16_t* q;         // bf16 [n][Hq][128]
  int n;                     // sequences
  RetopkSeq seq[kMaxRetopkBatch];
  int Hq, C, R, K, W;
  float tau;
  int bitmap_words;          // of the longest sequence
  // Long caches: the candidate bitmap lives in global memory, gbitmap_stride
  // words per head (all zero between steps: the compaction clears every word
  // it reads), and only its second level in shared memory; nullptr: both in
  // shared memory.
  uint32_t* gbitmap;
  int64_t gbitmap_stride;
  float* qbar_new;           // [n][Hq][128]
  int32_t* path;             // [n][Hq] 1 exact, 0 reuse
  uint32_t* cand;            // [n][Hq][cand_cap] ascending
  int32_t* mcand;            // [n][Hq]
  int cand_cap;              // R*K + W
  int32_t* path_out;         // optional copies
  int32_t* mcand_out;
  int32_t* cand_out;         // [n][Hq][cand_cap], -1 padded
  int32_t* lens_ws;          // [n] this step's lengths, for the scan and finish kernels
  RetopkSeq* seq_ws;         // [n] the table above, for the finish kernel's push
  TraceBuf trace;
};
cudaError_t launch_retopk_selector(const RetopkSelArgs& a, size_t smem, cudaStream_t st);

struct RetopkInitArgs {
  const uint16_t* prefill_q;     // [C][Hq][128]
  const int32_t* prefill_sup;    // [C][Hq][K]
  const int32_t* prefill_n;      // [C][Hq]
  int Hq, C, K;
  float* cache_qbar;
  int32_t* cache_sup;
  int32_t* cache_sup_n;
};
cudaError_t launch_retopk_init(const RetopkInitArgs& a, cudaStream_t st);

}  // namespace tsa
