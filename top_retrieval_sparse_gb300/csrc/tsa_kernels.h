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
  // Plain scan only (nullptr: none): [B][Hq][kH16Bins], zero before the
  // call (the finish kernel clears it); every emitted pair is counted in its
  // fine bin.
  uint32_t* hist16;
  // Bounded waits give up after wait_ns (0: the default limit).  Fault
  // injection for tests of the error path: with stall_first_copy set, CTA 0
  // never issues the copy of its first tile, so that its consumers' wait
  // runs out (bounded) and the call reports a timeout.
  long long wait_ns;
  int stall_first_copy;
  // Quantised scan (codes != nullptr): pool logits are the approximations
  // z^ = qts[bh] * sum_j qh[bh][j] c_ij from the offset-binary key codes
  // (same row geometry as kv.k, one byte per element), emitted against the
  // emission key in that domain; window rows are skipped (the finish
  // computes their logits from the bf16 keys).
  // The codes of each sequence's last q8_new rows are written by the
  // preceding kernel: the producer waits for it before copying them.
  const uint8_t* codes;
  const uint16_t* qh;        // fp16 [B][Hq][128]
  const float* qts;          // [B][Hq]
  int q8_new;
  TraceBuf trace;
};
cudaError_t launch_scan(const ScanArgs& a, int grid, cudaStream_t st, bool pdl);
int scan_grid_rows(bool q8);  // rows of one scan tile

// Quantised decode, first kernel: codes the last n_new rows of every
// sequence with the stored per-channel scales (raising err), then prepares
// every query head of the group: qh = fp16(q_j s_j / t), qts = t * scale and
// eps, a bound on |z - z^| for every row that holds for the tensor-core
// arithmetic of both the scan and the exact rescoring.
struct Q8PrepArgs {
  const uint16_t* q;         // bf16 [B][Hq][128]
  KvView kv;
  uint8_t* codes;
  const float* kscale;       // [B][Hkv][128]
  float* kerr;               // [B][Hkv][128]
  const int32_t* lens;
  int64_t len_host, len_step;
  int B, Hq, n_new;
  float scale;
  uint16_t* qh;              // fp16 [B][Hq][128]
  float* qts;                // [B][Hq]
  float* eps;                // [B][Hq]
};
cudaError_t launch_q8_prep(const Q8PrepArgs& a, cudaStream_t st, bool pdl);

// Quantised decode, between the scan and the finish: every emitted pair is
// rescored on the bf16 keys (the key scan's tensor-core arithmetic, so each
// logit is bit-identical to the plain scan's) and kept, with its exact logit,
// iff z >= k^ + eps; the others become sentinels.  A pool position that was
// not emitted has z <= z^ + eps < k^ + eps, so the kept pairs are exactly the
// pool positions with z >= k^ + eps (a plain emission with that key).  The
// window logits, which the quantised scan skips, are computed here too.  The
// work -- 32 pairs or window rows of one head -- is spread over the whole
// grid, so a head with a long list does not hold up the others.
struct Q8RescoreArgs {
  const uint16_t* q;         // bf16 [B][Hq][128]
  KvView kv;
  const int32_t* lens;
  int64_t len_host, len_step;
  int B, Hq;
  float scale;
  int n_init, n_recent;
  uint2* dense;              // [B][Hq][dense_stride]
  const int32_t* dense_n;    // [B][Hq] x kCtrStride
  int64_t dense_stride;
  const uint32_t* emit_key;  // [B][Hq] the scan's keys k^
  const float* eps;          // [B][Hq]
  float* wz;                 // [B][Hq][wz_stride]
  int wz_stride;
  TraceBuf trace;
};
constexpr int kQ8MaxHeads = 8192;  // B * Hq of one quantised call
cudaError_t launch_q8_rescore(const Q8RescoreArgs& a, int grid, cudaStream_t st);
// Key coding outside a decode step: fit (scales from the absolute maxima of
// rows [0, L_b), codes and errors of those rows) or append (codes of the last
// n_tail rows with the stored scales, errors raised).  kscale and kerr must
// be zero before a fit.
cudaError_t launch_q8_quantize(const KvView& kv, const int32_t* lens, int B, int64_t n_tail,
                               bool fit, uint8_t* codes, float* kscale, float* kerr,
                               cudaStream_t st);

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
  // The scan's fine histogram of the emitted pairs (plain decode; nullptr:
  // the finish counts the pairs' 11-bit bins itself); cleared here.
  uint32_t* hist16;
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
  // Quantised scan (decode only): the pairs were rescored (q8 rescore
  // kernel) and are the pool positions with z >= k^ + q8_eps[bh], k^ the
  // emission key the scan used; the next call's key is stored in the codes'
  // domain (minus eps).  nullptr: a plain scan.
  const float* q8_eps;
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
  int32_t fresh;             // slot the sequence's previous step wrote (-1: none)
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
