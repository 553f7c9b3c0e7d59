// finish.cu -- the rest of a decode step after the key scan, in one kernel:
// exact top-K selection from the pairs the scan emitted, softmax.V over the
// static window and over the selected rows, and the gamma1/gamma2 merge.
//
// "RetrievalAttention" Eq. 2 (the selected set: exact top-k by inner
// product, as in the Flat baseline, ties to the smaller position), Eq. 3
// (o_W and o_Omega over disjoint W and Omega, each with its local max) and
// Eq. 4-5 (o_t = g1 o_W + g2 o_Omega).
//
// One thread-block cluster of NC CTAs (NC = 8, 4 or 2, chosen at launch so
// that all clusters are resident at once, one CTA per SM; with more heads one
// CTA per head) per (sequence, query head):
//   0. the threshold bin b* is the largest bin whose suffix count of the
//      head's emitted pairs reaches K: from the scan's fine histogram (16 key
//      bits; every CTA reads it, no exchange), or -- a first call, an
//      emission key far below the logits -- every CTA counts the 11-bit bins
//      (top bits of the order-preserving logit key) of its slice of the
//      pairs and the counts are summed over the cluster (distributed shared
//      memory).  The scan emitted every pool position whose logit key is >=
//      the head's emission key, so when that is at least K pairs the K-th
//      largest key is among them and b* (and the selection below) is exact,
//      even if b*'s bin was emitted only in part; otherwise the cluster re-scores the
//      head's keys to count every bin, then re-emits the pool pairs with bin
//      >= b*, recomputing the logits with the scan's own tensor-core fragment
//      arithmetic so that every logit -- and so every bin -- is bit-identical
//      to the scan's;
//   1. each CTA reads its 1/NC slice of the head's pair list (the first
//      batch is already in flight during step 0): pairs above b* are
//      selected outright and kept in shared memory, pairs in b* are the
//      candidates; after the one cluster barrier every CTA copies all the
//      cluster's candidates through distributed shared memory;
//   2. every CTA finds the same exact threshold among the candidates: CTA
//      radix rounds of 11 bits on the 64-bit rank key (order-preserving
//      logit key, then ~position, so ties go to the smaller position);
//   3. the selected rows (window, above-b* pairs, selected candidates) are
//      split evenly over the cluster; each warp gathers V for its rows with
//      half-warp 16-byte loads, a spill-free batch of rows at a time,
//      keeping (max, sum, o) per set in base 2;
//      every CTA pushes its partials into rank 0's shared memory, and rank
//      0 applies Eq. 4-5 and stores the next call's emission key (the K-th
//      logit minus a margin).
// ReTopK steps use the same kernel: a reuse head has no pair list; each CTA
// rescores its share of the head's candidates A_t (exact logits e_i on the
// key rows), stores the keys into every CTA of the cluster, and all of them
// compete in the radix (no bins, no emission key); no head has a window, and
// rank 0 pushes (qbar_t, S_t) into the query-support FIFO.
// Launched as a programmatic dependent of the kernel that wrote the lists.
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

constexpr int kFinMaxCluster = 8;  // CTAs per head: 1, 2, 4 or 8 (chosen at launch)
constexpr int kSelCap = 2048;   // this CTA's above-b* pairs in shared memory
constexpr int kMyCap = 4096;    // this CTA's threshold-bin candidates in shared memory
constexpr int kAllCap = 16384;  // the cluster's threshold-bin candidates, copied locally (NC > 1)
constexpr int kPtabCap = 8192;  // pages of one sequence held in shared memory (single-CTA heads)
constexpr int kFinU = 8;        // pairs per thread per batch
// Rows a warp gathers (or rescores) at a time: lane l < rows holds row l and
// every lane keeps rows / 2 16-byte loads in registers.  32 rows held 64
// registers of loads and made the kernel spill, which serialised the loads;
// 24 fit the clustered decode instantiations, 16 the ReTopK ones and the
// single-CTA heads (whose page table in shared memory takes registers).
template <bool RT, int NC>
struct GatherRows {
  static constexpr int value = RT || NC == 1 ? 16 : 24;
};
constexpr int kRescoreRows = 16;
constexpr int kRankShift = 64 - kHistBits;  // b* = the rank key's top 11 bits
constexpr float kFinLog2e = 1.4426950408889634f;
constexpr float kFinLn2 = 0.6931471805599453f;

// NC CTAs per head (a cluster), W warps per CTA.  A single-CTA head reads
// its candidates in place, so it keeps no cluster-wide copy.
template <int NC, int W>
struct FinShared {
  uint64_t cand[NC > 1 ? kAllCap : 1];  // rank keys of all threshold-bin candidates, cluster order
  uint64_t mycand[kMyCap];        // this CTA's candidates (read by the cluster)
  uint2 sel[kSelCap];             // this CTA's above-b* pairs (position, logit bits)
  uint32_t hist[kHistBins];       // this CTA's bin counts, then the radix round histogram
  uint32_t chist[kHistBins];      // the cluster's bin counts (bins at or above a floor)
  float wo[W][2][kD];             // warp partials: [set][d], set 0 window, 1 selected
  float wm[W][2], wl[W][2];
  float mo[NC][2][kD];            // rank 0: the CTA partials, pushed by each CTA
  int32_t ptab[NC == 1 ? kPtabCap : 1];  // a single-CTA head: its sequence's page table
  float mm[NC][2], ml[NC][2];
  uint32_t warp_tot[32];
  int cnt[2];                     // read by the cluster: above-b* pairs, candidates
  int aoff[kFinMaxCluster + 1];   // cluster prefix of the above-b* counts
  int coff[kFinMaxCluster + 1];   // cluster prefix of the candidate counts
  int scal[8];
};

// Block-wide exclusive scan of one int per thread (all threads call).
template <int W, class Sh>
__device__ int fin_scan(int v, Sh& sh, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.warp_tot[wid] = (uint32_t)incl;
  __syncthreads();
  if (wid == 0) {
    const int w = lane < W ? (int)sh.warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < W) sh.warp_tot[lane] = (uint32_t)(wi - w);
    if (lane == W - 1) sh.scal[7] = wi;
  }
  __syncthreads();
  const int off = incl - v + (int)sh.warp_tot[wid];
  *total = sh.scal[7];
  __syncthreads();
  return off;
}

// Step 0: re-emit the pool pairs of head bh whose bin is >= ebin.  The CTA
// of cluster rank `rank` covers rows [L*rank/8, L*(rank+1)/8) in blocks of
// 16 rows per warp; fragments, k order and the final (c0 + c1) * scale are
// those of the key scan, so each logit equals the scan's bit for bit.
template <int W>
__device__ void reemit(const FinishArgs& a, int b, int h, int g, int G, int64_t L, int ebin,
                       int rank, int nc) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int gr = lane >> 2, tq = lane & 3;
  const int hl = h - g * G;
  const int bh = b * a.Hq + h;
  const int head0 = b * a.Hq + g * G;
  uint32_t qb[4][4];
  const uint16_t* qp = a.q + ((int64_t)head0 + (gr < G ? gr : 0)) * kD;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (gr < G) w = *reinterpret_cast<const uint4*>(qp + 8 * (4 * p + tq));
    qb[p][0] = w.x; qb[p][1] = w.y; qb[p][2] = w.z; qb[p][3] = w.w;
  }
  uint2* drow = a.dense + (int64_t)bh * a.dense_stride;
  const int64_t r0 = L * rank / nc, r1 = L * (rank + 1) / nc;
  const bool mine = tq == (hl >> 1);  // lanes holding head hl's column
  for (int64_t base = r0 + 16 * wid; base < r1; base += 16 * W) {
    const int64_t ia = base + gr, ib = base + gr + 8;
    uint4 W[4], X[4];
    const uint16_t* ka = a.kv.k + kv_row(a.kv, b, g, ia < r1 ? ia : r0);
    const uint16_t* kb = a.kv.k + kv_row(a.kv, b, g, ib < r1 ? ib : r0);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      W[p] = ia < r1 ? *reinterpret_cast<const uint4*>(ka + 8 * (4 * p + tq))
                     : make_uint4(0u, 0u, 0u, 0u);
      X[p] = ib < r1 ? *reinterpret_cast<const uint4*>(kb + 8 * (4 * p + tq))
                     : make_uint4(0u, 0u, 0u, 0u);
    }
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      mma_bf16(c0, W[p].x, X[p].x, W[p].y, X[p].y, qb[p][0], qb[p][1]);
      mma_bf16(c1, W[p].z, X[p].z, W[p].w, X[p].w, qb[p][2], qb[p][3]);
    }
    const bool odd = hl & 1;
    const float za = (odd ? c0[1] + c1[1] : c0[0] + c1[0]) * a.scale;
    const float zb = (odd ? c0[3] + c1[3] : c0[2] + c1[2]) * a.scale;
    const bool ea = mine && ia < r1 && !in_window(ia, L, a.n_init, a.n_recent) &&
                    (int)(f2key(za) >> kHistShift) >= ebin;
    const bool eb = mine && ib < r1 && !in_window(ib, L, a.n_init, a.n_recent) &&
                    (int)(f2key(zb) >> kHistShift) >= ebin;
    const unsigned ma = __ballot_sync(0xffffffffu, ea), mb = __ballot_sync(0xffffffffu, eb);
    const int cnt = __popc(ma) + __popc(mb);
    if (!cnt) continue;
    int64_t slot0 = 0;
    if (lane == 0) slot0 = atomicAdd(a.dense_n + (int64_t)bh * kCtrStride, cnt);
    slot0 = __shfl_sync(0xffffffffu, slot0, 0);
    const unsigned lt = (1u << lane) - 1u;
    if (ea) {
      const int64_t s = slot0 + __popc(ma & lt);
      if (s < a.dense_stride) drow[s] = make_uint2((uint32_t)ia, __float_as_uint(za));
    }
    if (eb) {
      const int64_t s = slot0 + __popc(ma) + __popc(mb & lt);
      if (s < a.dense_stride) drow[s] = make_uint2((uint32_t)ib, __float_as_uint(zb));
    }
  }
}

// The rare path's count: the 11-bit bins of head bh's pool logits on the
// rows of cluster rank `rank` (the rows and arithmetic of reemit), added to
// sh.hist (zeroed by the caller) with one shared atomic per distinct bin per
// warp instruction.
template <int W, class Sh>
__device__ void rescore_count(const FinishArgs& a, int b, int h, int g, int G, int64_t L,
                              int rank, int nc, Sh& sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int gr = lane >> 2, tq = lane & 3;
  const int hl = h - g * G;
  const int head0 = b * a.Hq + g * G;
  uint32_t qb[4][4];
  const uint16_t* qp = a.q + ((int64_t)head0 + (gr < G ? gr : 0)) * kD;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (gr < G) w = *reinterpret_cast<const uint4*>(qp + 8 * (4 * p + tq));
    qb[p][0] = w.x; qb[p][1] = w.y; qb[p][2] = w.z; qb[p][3] = w.w;
  }
  const int64_t r0 = L * rank / nc, r1 = L * (rank + 1) / nc;
  const bool mine = tq == (hl >> 1);
  for (int64_t base = r0 + 16 * wid; base < r1; base += 16 * W) {
    const int64_t ia = base + gr, ib = base + gr + 8;
    uint4 W4[4], X4[4];
    const uint16_t* ka = a.kv.k + kv_row(a.kv, b, g, ia < r1 ? ia : r0);
    const uint16_t* kb = a.kv.k + kv_row(a.kv, b, g, ib < r1 ? ib : r0);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      W4[p] = ia < r1 ? *reinterpret_cast<const uint4*>(ka + 8 * (4 * p + tq))
                      : make_uint4(0u, 0u, 0u, 0u);
      X4[p] = ib < r1 ? *reinterpret_cast<const uint4*>(kb + 8 * (4 * p + tq))
                      : make_uint4(0u, 0u, 0u, 0u);
    }
    float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      mma_bf16(c0, W4[p].x, X4[p].x, W4[p].y, X4[p].y, qb[p][0], qb[p][1]);
      mma_bf16(c1, W4[p].z, X4[p].z, W4[p].w, X4[p].w, qb[p][2], qb[p][3]);
    }
    const bool odd = hl & 1;
    const float za = (odd ? c0[1] + c1[1] : c0[0] + c1[0]) * a.scale;
    const float zb = (odd ? c0[3] + c1[3] : c0[2] + c1[2]) * a.scale;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t i = k ? ib : ia;
      const bool ok = mine && i < r1 && !in_window(i, L, a.n_init, a.n_recent);
      const uint32_t bin = ok ? f2key(k ? zb : za) >> kHistShift : 0xffffffffu;
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (ok && __ffs(peers) - 1 == lane) atomicAdd(&sh.hist[bin], (uint32_t)__popc(peers));
    }
  }
}

// A given candidate set's logits (a ReTopK reuse head's A_t, or attend_set's
// rows) on candidates [c0, c1), as rank keys into this CTA's candidate list
// (shared memory, then the top of the slice's spill area).  A warp takes
// kRescoreRows candidates at a time: lane l < kRescoreRows holds candidate
// base + l's position; key rows are read by half-warps (16 lanes x 16
// bytes), two rows per load, all loads in flight before any is used.  A position at or past L is never read:
// its logit is -inf (it is not attended) and the status word flags it.
template <int W, int NC, class Sh>
__device__ void reuse_logits(const FinishArgs& a, int b, int bh, int g, int64_t c0, int64_t c1,
                             int64_t L, Sh& sh, uint64_t* spill, bool push) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int half = lane >> 4, col = 8 * (lane & 15);
  const uint4 qw = *reinterpret_cast<const uint4*>(a.q + (int64_t)bh * kD + col);
  const float qv[8] = {bf_lo(qw.x), bf_hi(qw.x), bf_lo(qw.y), bf_hi(qw.y),
                       bf_lo(qw.z), bf_hi(qw.z), bf_lo(qw.w), bf_hi(qw.w)};
  const uint32_t* crow = a.cand + (int64_t)bh * a.cand_cap;
  for (int64_t base = c0 + kRescoreRows * wid; base < c1; base += kRescoreRows * W) {
    const int64_t j = lane < kRescoreRows ? base + lane : c1;
    const uint32_t pos = j < c1 ? crow[j] : 0u;
    const bool inside = (int64_t)pos < L;
    if (__any_sync(0xffffffffu, j < c1 && !inside) && lane == 0) atomicOr(a.status, kStatusBadLength);
    uint4 kv4[kRescoreRows / 2];
#pragma unroll
    for (int k = 0; k < kRescoreRows / 2; ++k) {
      const int r = 2 * k + half;
      const uint32_t pk = __shfl_sync(0xffffffffu, pos, r);
      kv4[k] = base + r < c1 && (int64_t)pk < L
                   ? *reinterpret_cast<const uint4*>(a.kv.k + kv_row(a.kv, b, g, pk) + col)
                   : make_uint4(0u, 0u, 0u, 0u);
    }
    float mine = 0.f;  // lane l ends with the logit of candidate base + l
#pragma unroll
    for (int k = 0; k < kRescoreRows / 2; ++k) {
      const uint4 w = kv4[k];
      float acc = qv[0] * bf_lo(w.x);
      acc = fmaf(qv[1], bf_hi(w.x), acc);
      acc = fmaf(qv[2], bf_lo(w.y), acc);
      acc = fmaf(qv[3], bf_hi(w.y), acc);
      acc = fmaf(qv[4], bf_lo(w.z), acc);
      acc = fmaf(qv[5], bf_hi(w.z), acc);
      acc = fmaf(qv[6], bf_lo(w.w), acc);
      acc = fmaf(qv[7], bf_hi(w.w), acc);
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      // lanes 0-15 hold row 2k's logit, lanes 16-31 row 2k+1's
      const float e0 = __shfl_sync(0xffffffffu, acc, 0), e1 = __shfl_sync(0xffffffffu, acc, 16);
      if (lane == 2 * k) mine = e0;
      if (lane == 2 * k + 1) mine = e1;
    }
    if (j < c1) {
      const uint64_t v = rank_key(inside ? mine * a.scale : -INFINITY, pos);
      if constexpr (NC > 1) {
        if (push) {  // candidate j of every CTA's copy of the cluster's candidates
#pragma unroll
          for (int c = 0; c < NC; ++c) st_dsmem_u64(&sh.cand[j], (uint32_t)c, v);
          continue;
        }
      }
      const int64_t i = j - c0;
      if (i < kMyCap) sh.mycand[i] = v;
      else spill[c1 - 1 - (i - kMyCap)] = v;
    }
  }
}

// The rare path, out of line so that the kernel's common path keeps a small
// instruction footprint: the emission key missed part of the top-K.  The
// cluster re-scores the head's keys to count every 11-bit bin, takes the
// threshold bin b* (the largest bin whose suffix count reaches `need`; with
// `all`, bin 0: the whole pool is selected) and re-emits the head's pool
// pairs with bin >= b*.  Every CTA of the cluster calls it; returns b*
// (-1 with `all`).
template <int NC, int W>
__device__ __noinline__ int reemit_head(const FinishArgs& a, FinShared<NC, W>& sh, int b, int h,
                                        int g, int G, int64_t L, int rank, int need, bool all) {
  constexpr int kFinThreads = 32 * W;
  constexpr int kBpt = kHistBins / kFinThreads;
  const int tid = threadIdx.x;
  const int bh = b * a.Hq + h;
  int bstar = -1;
  cluster_sync_all();  // every CTA has read the old list size and the remote counts
  if (!all) {
    for (int q = tid; q < kHistBins; q += kFinThreads) sh.hist[q] = 0;
    __syncthreads();
    rescore_count<W>(a, b, h, g, G, L, rank, NC, sh);
    __syncthreads();
    cluster_sync_all();  // every CTA's counts are complete
    for (int q = tid; q < kHistBins; q += kFinThreads) {
      uint32_t c = sh.hist[q];
#pragma unroll
      for (int r = 1; r < NC; ++r) c += ld_dsmem_u32(&sh.hist[q], (uint32_t)((rank + r) % NC));
      sh.chist[q] = c;
    }
    __syncthreads();
    // thread t holds bins 2047 - kBpt*t - r, r < kBpt
    uint32_t c[kBpt], mine = 0;
#pragma unroll
    for (int r = 0; r < kBpt; ++r) {
      c[r] = sh.chist[kHistBins - 1 - kBpt * tid - r];
      mine += c[r];
    }
    if (tid == 0) sh.scal[0] = 0;
    int tot;
    uint32_t acc = (uint32_t)fin_scan<W>((int)mine, sh, &tot);
#pragma unroll
    for (int r = 0; r < kBpt; ++r) {
      if (acc < (uint32_t)need && acc + c[r] >= (uint32_t)need)
        sh.scal[0] = kHistBins - 1 - kBpt * tid - r;
      acc += c[r];
    }
    __syncthreads();
    bstar = sh.scal[0];  // exists: the pool holds more than need positions
    __syncthreads();
    cluster_sync_all();  // the remote counts have been read
  }
  if (rank == 0 && tid == 0) {
    a.dense_n[(int64_t)bh * kCtrStride] = 0;
    __threadfence();
  }
  cluster_sync_all();
  reemit<W>(a, b, h, g, G, L, all ? 0 : bstar, rank, NC);
  __threadfence();
  cluster_sync_all();
  return bstar;
}

// RT: a ReTopK step (reuse heads, the FIFO push); Q8: a decode step after
// the quantised scan and the rescoring (the emission key in the codes'
// domain); the plain decode instantiation carries neither.
template <int NC, int W, bool RT, bool Q8>
__global__ void __launch_bounds__(32 * W, 16 / W) finish_kernel(FinishArgs a) {
  static_assert(!(RT && Q8), "a ReTopK step scans bf16 keys");
  constexpr int kFinWarps = W, kFinThreads = 32 * W;
  constexpr int kBpt = kHistBins / kFinThreads;  // histogram bins per thread: 4 or 8
  static_assert(kBpt % 4 == 0 && kFinThreads >= 2 * kD, "block shape");
  TraceScope trace(a.trace, kTrFinish);         // start, waited, threshold found, exit
  TraceScope phases(a.trace, kTrFinishPhases);  // start, decided, slice read, rows gathered
  extern __shared__ __align__(16) uint8_t fin_smem[];
  FinShared<NC, W>& sh = *reinterpret_cast<FinShared<NC, W>*>(fin_smem);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int rank = blockIdx.x;  // cluster rank (the cluster spans gridDim.x)
  const int bh = blockIdx.y;
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int G = a.Hq / a.kv.Hkv;
  const int g = h / G;
  // A single-CTA head of a paged cache keeps its sequence's page table in
  // shared memory, so that a V row's address needs no dependent global load
  // (the table is an input: it is read before the scan completes).
  bool ptab_ok = false;
  if constexpr (NC == 1 && !RT) {  // (a ReTopK step's lengths come from the selector)
    if (a.kv.page_table) {
      const int64_t Lq = seq_len(a.lens, a.len_host, a.len_step, b, a.kv.l_cap);
      const int64_t np = (Lq + (1 << a.kv.page_shift) - 1) >> a.kv.page_shift;
      if (np <= kPtabCap) {
        const int32_t* pt = a.kv.page_table + (int64_t)b * a.kv.pt_stride;
        for (int64_t q = tid; q < np; q += kFinThreads) sh.ptab[q] = __ldg(pt + q);
        ptab_ok = true;
      }
      __syncthreads();
    }
  }
  // element offset of V/K row i of this head's KV head
  auto row_off = [&](int64_t i) -> int64_t {
    if (ptab_ok) {
      const int64_t page = sh.ptab[i >> a.kv.page_shift];
      const int64_t r = i & ((1 << a.kv.page_shift) - 1);
      return (((page * a.kv.Hkv + g) << a.kv.page_shift) + r) * kD;
    }
    return kv_row(a.kv, b, g, i);
  };
  // (No V row is prefetched into L2 anywhere in this kernel: the window's
  // rows before the dependency wait, the selected rows once classified and
  // each gather batch's successor were each measured slower than the plain
  // loads -- 128K step 56.4 -> 55.4 us without all three.)
  pdl_wait();     // pairs and window logits come from the scan
  pdl_trigger();  // the next kernel may be scheduled (it writes nothing
                  // this kernel reads until this kernel has completed)
  trace.mark(1);

  // The first decisions' inputs sit at fixed addresses: the status word, the
  // list size, the emission key and margin factor and, on a ReTopK step, the
  // head's path and candidate count are all requested before any is used
  // (with the sequence length), not one after another.
  const int status_in = __ldcg(a.status);
  const int64_t n_in = __ldcg(a.dense_n + (int64_t)bh * kCtrStride);
  uint32_t ekey = __ldcg(a.emit_key + bh);
  const float mg_in = __ldcg(a.emit_margin + bh);
  // the rescored pairs are the pool positions with z >= k^ + eps
  if constexpr (Q8) ekey = q8_exact_key(ekey, __ldcg(a.q8_eps + bh));
  const int path_in = RT ? __ldcg(a.path + bh) : 1;
  const int mc_in = RT ? __ldcg(a.mcand + bh) : 0;
  // A reuse head's CTAs store its rescored candidates into each other's
  // shared memory before their first cluster barrier: every CTA of the
  // cluster must have started (the wait is below, after the first loads).
  if constexpr (RT && NC > 1) cluster_arrive_relaxed();
  // the scan's fine histogram of this head's emitted pairs (plain decode):
  // thread t holds bins kH16Bins - 1 - kH16Bpt t - r, from the top
  constexpr int kH16Bpt = kH16Bins / kFinThreads;
  static_assert(kH16Bins % kFinThreads == 0, "fine bins per thread");
  const bool fine_in = !RT && !Q8 && a.hist16 != nullptr;
  uint32_t* hrow = fine_in ? a.hist16 + (int64_t)bh * kH16Bins : nullptr;
  uint32_t h16[kH16Bpt];
#pragma unroll
  for (int r = 0; r < kH16Bpt; ++r)
    h16[r] = fine_in ? __ldcg(hrow + kH16Bins - 1 - kH16Bpt * tid - r) : 0u;

  if constexpr (RT && NC > 1) cluster_wait();

  // A bounded wait of the key scan (this call's, or an earlier one on this
  // workspace: the bit is sticky until the host reads it) gave up: the lists
  // and histograms are incomplete.  Every CTA reads the same word, so the
  // whole grid takes this path: NaN outputs, the counters cleared for the next
  // call, no FIFO push (the ReTopK state keeps its previous entry).
  if (status_in & kStatusTimeout) {
    if (rank == 0) {
      const float nan = __int_as_float(0x7fc00000);
      if (tid < kD) a.out[(int64_t)bh * kD + tid] = nan;
      if (tid == 0 && a.lse_out) a.lse_out[bh] = nan;
      if (!RT)
        for (int q = tid; q < a.K; q += kFinThreads) {
          if (a.topk_idx) a.topk_idx[(int64_t)bh * a.topk_stride + q] = -1;
          if (a.topk_score) a.topk_score[(int64_t)bh * a.topk_stride + q] = nan;
        }
      if (tid == 0) {
        a.dense_n[(int64_t)bh * kCtrStride] = 0;
        if (bh == 0) *a.tile_ctr = 0;
      }
      if (fine_in)
        for (int q = tid; q < kH16Bins; q += kFinThreads) hrow[q] = 0u;
    }
    return;
  }
  const int64_t L = seq_len(a.lens, a.len_host, a.len_step, b, a.kv.l_cap);
  const int64_t nw = window_count(L, a.n_init, a.n_recent);
  // a ReTopK reuse head selects among its |A_t| rescored candidates
  const bool reuse = RT && path_in == 0;
  const int mcand = mc_in < a.cand_cap ? mc_in : a.cand_cap;
  const int64_t P = reuse ? (int64_t)mcand : L - nw;
  const int need = (int64_t)a.K < P ? a.K : (int)P;
  uint64_t* spill = a.spill + (int64_t)bh * a.dense_stride;
  const uint2* lrow = a.dense + (int64_t)bh * a.dense_stride;

  // The first batch of this CTA's slice of the list is in flight while the
  // threshold bin is found (it is discarded if the list is re-emitted).
  int64_t n = need > 0 ? n_in : 0;
  if (n > a.dense_stride) n = a.dense_stride;
  int64_t s0 = n * rank / NC, s1 = n * (rank + 1) / NC;
  uint2 pre[kFinU];
#pragma unroll
  for (int u = 0; u < kFinU; ++u) {
    const int64_t jj = s0 + u * kFinThreads + tid;
    pre[u] = jj < s1 ? __ldcg(lrow + jj) : make_uint2(0xffffffffu, 0u);
  }

  // ---- 0. threshold bin b* and the emission check ----
  // The largest bin whose suffix count reaches tgt[k], over a count array in
  // shared memory restricted to bins >= floor (-1: no such bin).
  auto suffix_bins = [&](const uint32_t* cnt, int floor, const uint32_t (&tgt)[2],
                         int (&fb)[2]) -> uint32_t {
    uint32_t c[kBpt], mine = 0;
#pragma unroll
    for (int r = 0; r < kBpt; ++r) {
      const int bin = kHistBins - 1 - kBpt * tid - r;
      c[r] = bin >= floor ? cnt[bin] : 0u;
      mine += c[r];
    }
    if (tid == 0) sh.scal[0] = sh.scal[1] = -1;
    int tot;
    const uint32_t excl = (uint32_t)fin_scan<W>((int)mine, sh, &tot);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      uint32_t acc = excl;
#pragma unroll
      for (int r = 0; r < kBpt; ++r) {
        if (acc < tgt[k] && acc + c[r] >= tgt[k]) sh.scal[k] = kHistBins - 1 - kBpt * tid - r;
        acc += c[r];
      }
    }
    __syncthreads();
    fb[0] = sh.scal[0];
    fb[1] = sh.scal[1];
    __syncthreads();  // scal is rewritten later
    return (uint32_t)tot;
  };
  // The cluster's counts of bins >= floor into sh.chist.  After the cluster
  // barrier every CTA reads the others' sh.hist: none may rewrite it before
  // the next cluster barrier.
  auto cluster_counts = [&](int floor) {
    cluster_sync_all();
    for (int q = floor + tid; q < kHistBins; q += kFinThreads) {
      uint32_t c = sh.hist[q];
#pragma unroll
      for (int r = 1; r < NC; ++r) c += ld_dsmem_u32(&sh.hist[q], (uint32_t)((rank + r) % NC));
      sh.chist[q] = c;
    }
    __syncthreads();
  };
  // b*: with `fine`, a fine bin relative to hb0 (the scan's histogram);
  // otherwise an 11-bit bin of the logit key (counted here); -1 selects every
  // pair
  int bstar = -1, redo = 0, ebin = 0;
  bool fine = false;
  uint32_t pred_above = 0, pred_cand = 0;  // the histogram's counts above b* and in it
  const uint32_t hb0 = ekey >> kH16Shift;
  const int used = need > 0 ? (int)(ekey >> kHistShift) : 0;  // the emission key's bin
  const uint32_t tgt[2] = {(uint32_t)need, (uint32_t)need};
  if (need > 0 && !reuse && fine_in) {
    // The scan counted every emitted pair in its fine bin: b* is the largest
    // fine bin whose suffix count reaches need, with no pass over the list
    // and no exchange between the cluster's CTAs.
    uint32_t mine = 0;
#pragma unroll
    for (int r = 0; r < kH16Bpt; ++r) mine += h16[r];
    if (tid == 0) sh.scal[0] = -1;
    int tot;
    uint32_t acc = (uint32_t)fin_scan<W>((int)mine, sh, &tot);
#pragma unroll
    for (int r = 0; r < kH16Bpt; ++r) {
      if (acc < (uint32_t)need && acc + h16[r] >= (uint32_t)need) {
        sh.scal[0] = kH16Bins - 1 - kH16Bpt * tid - r;
        sh.scal[1] = (int)acc;
        sh.scal[2] = (int)h16[r];
      }
      acc += h16[r];
    }
    __syncthreads();
    const int fb = sh.scal[0];
    pred_above = (uint32_t)sh.scal[1];
    pred_cand = (uint32_t)sh.scal[2];
    __syncthreads();  // scal is rewritten later
    fine = false;
    if (need < P) {
      if (fb < 0) {  // fewer than K pairs emitted: the re-emission counts 11-bit bins
        redo = 1;
      } else if (fb < kH16Bins - 1) {
        fine = true;
        bstar = fb;
      }  // else b* is the last fine bin, which holds everything above it (a first
         // call, or a far-off emission key): the 11-bit bins are counted below
    } else {  // every pool position is selected: all of them must have been emitted
      redo = (int64_t)tot < P;
      fine = !redo;
      pred_above = (uint32_t)tot;
      pred_cand = 0;
    }
  }
  if (need > 0 && !reuse && !fine && !redo) {  // (a reuse head has no bins: all its candidates compete)
    // the bins of this CTA's slice of the emitted pairs (the first batch is
    // in registers), one shared atomic per distinct bin per warp instruction;
    // every emitted pair's bin is >= the emission key's
    for (int q = used + tid; q < kHistBins; q += kFinThreads) sh.hist[q] = 0;
    __syncthreads();
    for (int64_t jb = s0; jb < s1; jb += kFinThreads * kFinU) {
#pragma unroll
      for (int u = 0; u < kFinU; ++u) {
        const int64_t jj = jb + u * kFinThreads + tid;
        const uint2 pv = jb == s0 ? pre[u]
                                  : (jj < s1 ? __ldcg(lrow + jj) : make_uint2(0xffffffffu, 0u));
        const bool ok = pv.x != 0xffffffffu;
        const uint32_t bin = ok ? f2key(__uint_as_float(pv.y)) >> kHistShift : 0xffffffffu;
        const unsigned peers = __match_any_sync(0xffffffffu, bin);
        if (ok && __ffs(peers) - 1 == lane) atomicAdd(&sh.hist[bin], (uint32_t)__popc(peers));
      }
    }
    __syncthreads();
    cluster_counts(used);
    int fb[2];
    const uint32_t total = suffix_bins(sh.chist, used, tgt, fb);
    if (need < P) {
      bstar = fb[0];  // -1: fewer than K pairs emitted, b* lies below the emission key
      redo = bstar < 0;
      ebin = bstar;
    } else {  // every pool position is selected: all of them must have been emitted
      redo = (int64_t)total < P;
      ebin = 0;
    }
  }
  phases.mark(1);
  trace.info = (uint32_t)min(n, (int64_t)0x7fffffff);
  phases.info = ((uint32_t)redo << 31) | ((uint32_t)(bstar & 0x7fff) << 16) | (uint32_t)used;
  // ---- re-emission when the emission key missed the top-K (rare) ----
  if (redo) {  // uniform over the cluster
    const int bs = reemit_head<NC, W>(a, sh, b, h, g, G, L, rank, need, need >= P);
    if (need < P) bstar = ebin = bs;
  }

  // ---- 1. this CTA's slice of the pair list ----
  // Pairs above b* are this CTA's selected rows; pairs in b* are candidates.
  // After one cluster barrier every CTA copies all the cluster's candidates
  // (a few thousand at most in practice) through distributed shared memory.
  int nmy = 0, nmc = 0;
  if (need > 0) {
    if (redo) {  // the list was re-emitted: new size, new slice
      n = __ldcg(a.dense_n + (int64_t)bh * kCtrStride);
      if (n > a.dense_stride) n = a.dense_stride;
      s0 = n * rank / NC;
      s1 = n * (rank + 1) / NC;
    }
    for (int64_t jb = s0; jb < s1; jb += kFinThreads * kFinU) {
      uint2 pv[kFinU];
#pragma unroll
      for (int u = 0; u < kFinU; ++u) {
        const int64_t jj = jb + u * kFinThreads + tid;
        pv[u] = jb == s0 && !redo ? pre[u]
                                  : (jj < s1 ? __ldcg(lrow + jj) : make_uint2(0xffffffffu, 0u));
      }
      uint64_t v[kFinU];
      uint32_t selm = 0u, cndm = 0u;
#pragma unroll
      for (int u = 0; u < kFinU; ++u) {
        v[u] = 0;
        if (pv[u].x != 0xffffffffu) {
          v[u] = rank_key(__uint_as_float(pv[u].y), pv[u].x);
          int bin;
          if (fine) {  // (emitted keys are >= the emission key: d >= 0)
            const int dd = (int)(uint32_t)(v[u] >> (32 + kH16Shift)) - (int)hb0;
            bin = dd < 0 ? -1 : (dd < kH16Bins ? dd : kH16Bins - 1);
          } else {
            bin = (int)(v[u] >> kRankShift);
          }
          if (bstar < 0 || bin > bstar) selm |= 1u << u;
          else if (bin == bstar) cndm |= 1u << u;
        }
      }
      int tot;
      const int off = fin_scan<W>((__popc(selm) << 16) | __popc(cndm), sh, &tot);
      int i1 = nmy + (off >> 16), i2 = nmc + (off & 0xffff);
#pragma unroll
      for (int u = 0; u < kFinU; ++u) {
        if ((selm >> u) & 1u) {  // slice-relative spill from the bottom
          if (i1 < kSelCap) sh.sel[i1] = pv[u];
          else spill[s0 + (i1 - kSelCap)] = v[u];
          ++i1;
        } else if ((cndm >> u) & 1u) {  // ... and from the top
          if (i2 < kMyCap) sh.mycand[i2] = v[u];
          else spill[s1 - 1 - (i2 - kMyCap)] = v[u];
          ++i2;
        }
      }
      nmy += tot >> 16;
      nmc += tot & 0xffff;
    }
  }
  // A reuse head whose A_t fits the cluster's candidate copy: every CTA
  // stores its share's keys at their A_t index into every CTA's copy before
  // the cluster barrier, so nothing is exchanged after it.
  const bool rpush = NC > 1 && reuse && mcand <= kAllCap;
  if (need > 0 && reuse) {  // this CTA's share of A_t, rescored: every one a candidate
    n = mcand;  // the candidate index space (spill layout as for a list slice)
    s0 = n * rank / NC;
    s1 = n * (rank + 1) / NC;
    reuse_logits<W, NC>(a, b, bh, g, s0, s1, L, sh, spill, rpush);
    nmc = (int)(s1 - s0);
    __syncthreads();
  }
  if (tid == 0) {
    sh.cnt[0] = nmy;
    sh.cnt[1] = nmc;
  }
  phases.mark(2);
  cluster_sync_all();  // every CTA's lists and counts are complete
  if (wid == 0) {
    int ca = 0, cc = 0;
    if (lane < NC && rpush) {  // no pairs; each CTA's share of A_t
      cc = (int)((int64_t)mcand * (lane + 1) / NC - (int64_t)mcand * lane / NC);
    } else if (lane < NC) {
      ca = (int)ld_dsmem_u32(reinterpret_cast<const uint32_t*>(&sh.cnt[0]), lane);
      cc = (int)ld_dsmem_u32(reinterpret_cast<const uint32_t*>(&sh.cnt[1]), lane);
    }
    int ia = ca, ic = cc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ya = __shfl_up_sync(0xffffffffu, ia, o), yc = __shfl_up_sync(0xffffffffu, ic, o);
      if (lane >= o) {
        ia += ya;
        ic += yc;
      }
    }
    if (lane < NC) {
      sh.aoff[lane + 1] = ia;
      sh.coff[lane + 1] = ic;
    }
    if (lane == 0) sh.aoff[0] = sh.coff[0] = 0;
  }
  __syncthreads();
  const int nabove = sh.aoff[NC], ncand = sh.coff[NC];
  // The fine histogram has been read by every CTA of the cluster: clear it
  // for the next call.  Its counts must equal the classification's.
  if (fine_in && rank == 0) {
    for (int q = tid; q < kH16Bins; q += kFinThreads) hrow[q] = 0u;
    if (fine && tid == 0 && ((uint32_t)nabove != pred_above || (uint32_t)ncand != pred_cand))
      atomicOr(a.status, kStatusCheck);
  }
  // Every CTA of the cluster has read the head's list size and key: clear
  // the counters for the next call (the workspace contract).
  if (rank == 0 && tid == 0) {
    a.dense_n[(int64_t)bh * kCtrStride] = 0;
    if (bh == 0) *a.tile_ctr = 0;
  }
  // candidate j of the cluster (cluster order): CTA c's list, local index i
  auto cand_remote = [&](int jc) -> uint64_t {
    int c = 0;
#pragma unroll
    for (int k = 1; k < NC; ++k) c += jc >= sh.coff[k] ? 1 : 0;
    const int i = jc - sh.coff[c];
    if (i < kMyCap) return ld_dsmem_u64(&sh.mycand[i], (uint32_t)c);
    const int64_t c1 = n * (c + 1) / NC;
    return __ldcg(spill + (c1 - 1 - (i - kMyCap)));
  };
  if constexpr (NC > 1) {  // eight remote loads in flight per thread before any is stored
    constexpr int kCopyU = 8;
    const int lim = rpush ? 0 : ncand < kAllCap ? ncand : kAllCap;
    for (int jb = 0; jb < lim; jb += kFinThreads * kCopyU) {
      uint64_t v[kCopyU];
#pragma unroll
      for (int u = 0; u < kCopyU; ++u) {
        const int jc = jb + u * kFinThreads + tid;
        v[u] = jc < lim ? cand_remote(jc) : 0ull;
      }
#pragma unroll
      for (int u = 0; u < kCopyU; ++u) {
        const int jc = jb + u * kFinThreads + tid;
        if (jc < lim) sh.cand[jc] = v[u];
      }
    }
  }
  __syncthreads();
  auto cand_at = [&](int jc) -> uint64_t {
    if constexpr (NC == 1) {  // a single CTA reads its own list in place
      return jc < kMyCap ? sh.mycand[jc] : __ldcg(spill + (n - 1 - (jc - kMyCap)));
    } else {
      return jc < kAllCap ? sh.cand[jc] : cand_remote(jc);
    }
  };

  // ---- 2. the threshold among the candidates (same result in every CTA) ----
  // cmode 0: no candidate selected, 1: all, 2: those with rank key >= T
  int cmode = 0;
  uint64_t T = 0;
  const int need_rem = need - nabove;
  if (need > 0 && (bstar >= 0 || reuse) && need_rem > 0) {
    if (need_rem >= ncand) {
      cmode = 1;
    } else {
      cmode = 2;
      // the candidates share b*'s 11 bits, or its 16 key bits (a reuse
      // head's, or those of the last fine bin: no known bits)
      uint64_t prefix = 0ull, mask = 0ull;
      int shift = 64;
      if (!reuse && !fine) {
        prefix = (uint64_t)bstar << kRankShift;
        mask = (uint64_t)(kHistBins - 1) << kRankShift;
        shift = kRankShift;
      } else if (!reuse && bstar < kH16Bins - 1) {
        prefix = (uint64_t)(hb0 + (uint32_t)bstar) << (32 + kH16Shift);
        mask = 0xffffull << (32 + kH16Shift);
        shift = 32 + kH16Shift;
      }
      int match = ncand, rem = need_rem;
      while (true) {
        if (match <= rem) {  // everything still matching is selected
          T = prefix;
          break;
        }
        const int db = shift < kHistBits ? shift : kHistBits;
        shift -= db;
        const uint32_t dmask = (1u << db) - 1u;
        for (int q = tid; q < kHistBins; q += kFinThreads) sh.hist[q] = 0;
        __syncthreads();
        for (int jc = tid; jc < ncand; jc += kFinThreads) {
          const uint64_t v = cand_at(jc);
          if ((v & mask) == prefix) atomicAdd(&sh.hist[(uint32_t)(v >> shift) & dmask], 1u);
        }
        __syncthreads();
        // thread t: bins nb-1-kBpt*t-r (from the top); digits past nb are empty
        const int nb = 1 << db;
        uint32_t c[kBpt], mine = 0;
#pragma unroll
        for (int r = 0; r < kBpt; ++r) {
          const int bin = nb - 1 - kBpt * tid - r;
          c[r] = bin >= 0 ? sh.hist[bin] : 0u;
          mine += c[r];
        }
        int tot;
        const uint32_t excl = (uint32_t)fin_scan<W>((int)mine, sh, &tot);
        if (excl < (uint32_t)rem && excl + mine >= (uint32_t)rem) {
          uint32_t acc = excl;
#pragma unroll
          for (int r = 0; r < kBpt; ++r) {
            if (acc < (uint32_t)rem && acc + c[r] >= (uint32_t)rem) {
              sh.scal[2] = nb - 1 - kBpt * tid - r;  // threshold digit d*
              sh.scal[3] = (int)acc;              // candidates above it
              sh.scal[4] = (int)c[r];             // candidates equal to it
            }
            acc += c[r];
          }
        }
        __syncthreads();
        const uint32_t dstar = (uint32_t)sh.scal[2];
        rem -= sh.scal[3];
        match = sh.scal[4];
        __syncthreads();  // scal is rewritten by the next round
        prefix |= (uint64_t)dstar << shift;
        mask |= (uint64_t)dmask << shift;
        if (rem == 0) {  // the digits above d* were exactly enough
          T = prefix + (1ull << shift);
          break;
        }
        if (shift == 0) {
          T = prefix;
          break;
        }
      }
    }
  }
  auto cand_selected = [&](uint64_t v) -> bool { return cmode == 1 || (cmode == 2 && v >= T); };
  trace.mark(2);

  // ---- 3. softmax.V over this CTA's rows ----
  // The cluster's rows in one index space -- the window, then the above-b*
  // pairs in cluster order (CTA c's i-th pair at nw + aoff[c] + i), then the
  // candidates (absent when not selected) -- split evenly over the CTAs and
  // their warps; a row held by another CTA is read through distributed
  // shared memory.
  const int Rtot = (int)nw + nabove + (cmode != 0 ? ncand : 0);
  const int c0r = (int)((int64_t)Rtot * rank / NC), c1r = (int)((int64_t)Rtot * (rank + 1) / NC);
  const int w0 = c0r + (int)((int64_t)(c1r - c0r) * wid / kFinWarps);
  const int w1 = c0r + (int)((int64_t)(c1r - c0r) * (wid + 1) / kFinWarps);
  const uint16_t* vbase = a.kv.page_table ? a.kv.v : a.kv.v + kv_row(a.kv, b, g, 0);
  const float* wzrow = a.wz + (int64_t)bh * a.wz_stride;
  constexpr int kGatherRows = GatherRows<RT, NC>::value;
  // kGatherRows rows per warp at a time: lane l < kGatherRows holds row
  // base + l's position and logit; V rows are read by half-warps (16 lanes x
  // 16 bytes = one row), so load k brings rows base + 2k (lanes 0-15) and
  // base + 2k + 1 (lanes 16-31), and each lane accumulates 8 columns,
  // 8 * (lane % 16) onwards.
  const int half = lane >> 4, col = 8 * (lane & 15);
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[2][8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[0][e] = o[1][e] = 0.f;
  // row j of the cluster's index space: position, logit, set (0 window, 1
  // selected) and whether it is attended (an unselected candidate is not)
  auto row_meta = [&](int j, int& pos, float& z, int& set, bool& lv) {
    z = -INFINITY;
    pos = 0;
    set = 0;
    lv = false;
    if (j >= w1) return;
    if (j < nw) {  // window row: its logit is loaded after the V loads issue
      pos = (int)window_pos(j, L, a.n_init, a.n_recent);
      lv = true;
    } else if (j < nw + nabove) {
      const int k = j - (int)nw;
      int c = 0;
#pragma unroll
      for (int q = 1; q < NC; ++q) c += k >= sh.aoff[q] ? 1 : 0;
      const int li = k - sh.aoff[c];
      if (li < kSelCap) {
        const uint64_t pr = c == rank ? *reinterpret_cast<const uint64_t*>(&sh.sel[li])
                                      : ld_dsmem_u64(reinterpret_cast<const uint64_t*>(&sh.sel[li]),
                                                     (uint32_t)c);
        pos = (int)(uint32_t)pr;
        z = __uint_as_float((uint32_t)(pr >> 32));
      } else {
        const uint64_t v = __ldcg(spill + n * c / NC + (li - kSelCap));
        pos = (int)rank_pos(v);
        z = key2f((uint32_t)(v >> 32));
      }
      set = 1;
      lv = true;
    } else {
      const uint64_t v = cand_at(j - (int)nw - nabove);
      if (cand_selected(v) && (int64_t)rank_pos(v) < L) {  // (given sets: only rows < L)
        pos = (int)rank_pos(v);
        z = key2f((uint32_t)(v >> 32));
        lv = true;
      }
      set = 1;
    }
  };
  float nz;
  int npos, nset;
  bool nlv;
  row_meta(lane < kGatherRows ? w0 + lane : w1, npos, nz, nset, nlv);
  for (int base = w0; base < w1; base += kGatherRows) {
    const float z0 = nz;
    const int pos = npos, set = nset;
    const bool lv = nlv;
    const int j = base + lane;
    // the next batch's row: fetch its description now
    row_meta(lane < kGatherRows ? base + kGatherRows + lane : w1, npos, nz, nset, nlv);
    float z = z0;
    const unsigned live = __ballot_sync(0xffffffffu, lv);
    const unsigned sel1 = __ballot_sync(0xffffffffu, set == 1);
    uint4 vv[kGatherRows / 2];
#pragma unroll
    for (int k = 0; k < kGatherRows / 2; ++k) {
      const int r = 2 * k + half;
      const int pk = __shfl_sync(0xffffffffu, pos, r);
      const uint16_t* vr =
          a.kv.page_table ? a.kv.v + row_off(pk) : vbase + (int64_t)pk * kD;
      vv[k] = ((live >> r) & 1u) ? __ldg(reinterpret_cast<const uint4*>(vr + col))
                                 : make_uint4(0u, 0u, 0u, 0u);
    }
    if (lv && j < nw) z = __ldcg(wzrow + j);
    z = lv ? z * kFinLog2e : -INFINITY;
    // chunk maxima per set, rescale, then each lane weights its own row
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      const float bm = warp_max(set == st ? z : -INFINITY);
      if (bm > m[st]) {
        const float sc = m[st] == -INFINITY ? 0.f : exp2f(m[st] - bm);
        l[st] *= sc;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[st][e] *= sc;
        m[st] = bm;
      }
    }
    const float p = lv ? exp2f(z - (set ? m[1] : m[0])) : 0.f;
    l[0] += warp_sum(set == 0 ? p : 0.f);
    l[1] += warp_sum(set == 1 ? p : 0.f);
#pragma unroll
    for (int k = 0; k < kGatherRows / 2; ++k) {
      if (!((live >> (2 * k)) & 3u)) continue;  // warp-uniform: both rows absent
      const int r = 2 * k + half;
      const float pr = __shfl_sync(0xffffffffu, p, r);  // 0 for an absent row
      const uint4 w = vv[k];
      const float v[8] = {bf_lo(w.x), bf_hi(w.x), bf_lo(w.y), bf_hi(w.y),
                          bf_lo(w.z), bf_hi(w.z), bf_lo(w.w), bf_hi(w.w)};
      if ((sel1 >> r) & 1u) {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[1][e] = fmaf(pr, v[e], o[1][e]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[0][e] = fmaf(pr, v[e], o[0][e]);
      }
    }
  }
  // the two half-warps hold the same columns for different rows
#pragma unroll
  for (int st = 0; st < 2; ++st)
#pragma unroll
    for (int e = 0; e < 8; ++e) o[st][e] += __shfl_xor_sync(0xffffffffu, o[st][e], 16);
  // combine the warps of this CTA
  phases.mark(3);
#pragma unroll
  for (int st = 0; st < 2; ++st) {
    if (lane == 0) {
      sh.wm[wid][st] = m[st];
      sh.wl[wid][st] = l[st];
    }
    if (lane < 16) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sh.wo[wid][st][col + e] = o[st][e];
    }
  }
  __syncthreads();
  if (tid < 2 * kD) {
    const int st = tid / kD, t = tid % kD;  // (set, element)
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kFinWarps; ++w) M = fmaxf(M, sh.wm[w][st]);
    float acc = 0.f, lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kFinWarps; ++w) {
        if (sh.wm[w][st] == -INFINITY) continue;
        const float e = exp2f(sh.wm[w][st] - M);
        acc = fmaf(e, sh.wo[w][st][t], acc);
        lsum = fmaf(e, sh.wl[w][st], lsum);
      }
    }
    // push this CTA's partial into rank 0's shared memory
    st_dsmem(&sh.mo[rank][st][t], 0, acc);
    if (t == 0) {
      st_dsmem(&sh.mm[rank][st], 0, M);
      st_dsmem(&sh.ml[rank][st], 0, lsum);
    }
  }
  // a ReTopK step writes S_t straight into the FIFO entry it overwrites
  int32_t* ofifo = nullptr;
  if (RT && a.seqs) {  // the record was written by the selector, complete since pdl_wait
    const RetopkSeq* sq = a.seqs + b;
    int32_t* sup = reinterpret_cast<int32_t*>(
        __ldcg(reinterpret_cast<const unsigned long long*>(&sq->sup)));
    ofifo = sup + ((int64_t)h * a.C + __ldcg(&sq->fifo_head)) * a.K;
  }
  const bool want_idx = a.topk_idx != nullptr || a.topk_score != nullptr || ofifo != nullptr;
  cluster_sync_all();  // every CTA's partial is in rank 0's shared memory; after this
                       // barrier no CTA reads another CTA's shared memory (but see below)

  // ---- rank 0: Eq. 4-5 over the cluster's partials ----
  if (rank == 0 && tid < kD) {
    float mc[2][NC], lc[2][NC], oc[2][NC];
#pragma unroll
    for (int c = 0; c < NC; ++c)
#pragma unroll
      for (int st = 0; st < 2; ++st) {
        mc[st][c] = sh.mm[c][st];
        lc[st][c] = sh.ml[c][st];
        oc[st][c] = sh.mo[c][st][tid];
      }
    float zt[2], lsum[2], osum[2];
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < NC; ++c) M = fmaxf(M, mc[st][c]);
      float ls = 0.f, os = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const float e = mc[st][c] == -INFINITY ? 0.f : exp2f(mc[st][c] - M);
          ls = fmaf(e, lc[st][c], ls);
          os = fmaf(e, oc[st][c], os);
        }
      }
      zt[st] = M;  // z~1 (window), z~2 (selected), base 2
      lsum[st] = ls;
      osum[st] = os;
    }
    float outv = 0.f, lse = -INFINITY;
    const bool eW = !(lsum[0] > 0.f), eO = !(lsum[1] > 0.f);
    if (!(eW && eO)) {
      const float z = eW ? zt[1] : (eO ? zt[0] : fmaxf(zt[0], zt[1]));
      const float aW = eW ? 0.f : exp2f(zt[0] - z);
      const float aO = eO ? 0.f : exp2f(zt[1] - z);
      const float den = aW * lsum[0] + aO * lsum[1];
      outv = (aW * osum[0] + aO * osum[1]) / den;  // g1 o_W + g2 o_Omega
      lse = (z + log2f(den)) * kFinLn2;
    }
    a.out[(int64_t)bh * kD + tid] = outv;
    if (tid == 0 && a.lse_out) a.lse_out[bh] = lse;
  }
  // ---- optional top-K outputs: each CTA writes its above-b* pairs at its
  // cluster offset; rank 0 appends the selected candidates in cluster order ----
  if (want_idx) {
    int32_t* oidx = a.topk_idx ? a.topk_idx + (int64_t)bh * a.topk_stride : nullptr;
    float* osc = a.topk_score ? a.topk_score + (int64_t)bh * a.topk_stride : nullptr;
    for (int li = tid; li < nmy; li += kFinThreads) {
      const int i = sh.aoff[rank] + li;
      int32_t pos;
      float z;
      if (li < kSelCap) {
        pos = (int32_t)sh.sel[li].x;
        z = __uint_as_float(sh.sel[li].y);
      } else {
        const uint64_t v = __ldcg(spill + s0 + (li - kSelCap));
        pos = (int32_t)rank_pos(v);
        z = key2f((uint32_t)(v >> 32));
      }
      if (i < a.K) {
        if (oidx) oidx[i] = pos;
        if (ofifo) ofifo[i] = pos;
        if (osc) osc[i] = z;
      }
    }
    if (rank == 0) {
      if (cmode != 0) {
        int done = 0;
        for (int jb = 0; jb < ncand; jb += kFinThreads) {
          const int jc = jb + tid;
          uint64_t v = 0;
          const bool s = jc < ncand && cand_selected(v = cand_at(jc));
          int tot;
          const int r = fin_scan<W>(s ? 1 : 0, sh, &tot);
          const int at = nabove + done + r;
          if (s && at < a.K) {
            if (oidx) oidx[at] = (int32_t)rank_pos(v);
            if (ofifo) ofifo[at] = (int32_t)rank_pos(v);
            if (osc) osc[at] = key2f((uint32_t)(v >> 32));
          }
          done += tot;
        }
      }
      for (int q = (need > 0 ? need : 0) + tid; q < a.K; q += kFinThreads) {
        if (oidx) oidx[q] = -1;
        if (ofifo) ofifo[q] = -1;
        if (osc) osc[q] = -INFINITY;
      }
    }
  }
  if (a.counts_out && rank == 0 && tid == 0) a.counts_out[bh] = need > 0 ? need : 0;
  // The length contract (0 <= lens[b] <= l_cap) is checked here: an
  // out-of-range length was clamped by both kernels; flag it for the host.
  if (a.lens && rank == 0 && h == 0 && tid == 0) {
    const int32_t Lr = a.lens[b];
    if (Lr < 0 || (int64_t)Lr > a.kv.l_cap) atomicOr(a.status, kStatusBadLength);
  }
  // The next call's emission key: the K-th logit z_T (the threshold's logit,
  // or the lower edge of b*'s bin when all its candidates were taken) minus a
  // margin f * 0.2 * (|z_T| + 1).  Across the decode steps of the synthetic
  // workloads the K-th logit fell by at most 16 % of |z| + 1 from one step to
  // the next, and a margin of 0.2 (|z| + 1) emits about 2.5 K pairs.  The
  // per-head factor f doubles after a re-emission (at most 8) and decays back
  // to 1 by 10 % per call.  Any stored value is safe: only the cost depends
  // on it.
  if (need > 0 && !reuse && rank == 0 && tid == 0) {  // read by every CTA long before this point
    float f = mg_in;
    if (!(f >= 1.f) || !(f <= 8.f)) f = 1.f;  // a new or unset state
    f = redo ? fminf(2.f * f, 8.f) : fmaxf(1.f, 0.9f * f);
    uint32_t next = 0u;
    if (need < P && bstar >= 0) {
      const uint32_t fedge = min(hb0 + (uint32_t)bstar, 0xffffu) << kH16Shift;
      const float zref = cmode == 2 ? key2f((uint32_t)(T >> 32))
                         : fine     ? key2f(fedge)
                                    : key2f((uint32_t)bstar << kHistShift);
      float ze = zref - f * 0.2f * (fabsf(zref) + 1.f);
      if constexpr (Q8) ze = __fsub_rd(ze, __ldcg(a.q8_eps + bh));  // the codes' domain
      next = ze == ze && fabsf(ze) < INFINITY ? f2key(ze) : 0u;
    }
    a.emit_key[bh] = next;
    a.emit_margin[bh] = f;
  }
  if (RT && a.seqs && rank == 0) {  // ReTopK: (qbar_t, S_t) over the oldest FIFO entry
    const RetopkSeq* sq = a.seqs + b;
    float* qbar = reinterpret_cast<float*>(
        __ldcg(reinterpret_cast<const unsigned long long*>(&sq->qbar)));
    int32_t* sup_n = reinterpret_cast<int32_t*>(
        __ldcg(reinterpret_cast<const unsigned long long*>(&sq->sup_n)));
    const int64_t hc = (int64_t)h * a.C + __ldcg(&sq->fifo_head);
    if (tid < kD) qbar[hc * kD + tid] = a.push_qbar[(int64_t)bh * kD + tid];
    if (tid == 0) sup_n[hc] = need > 0 ? need : 0;
  }
  // Candidates past rank 0's copy are read from the other CTAs: keep them
  // resident until rank 0 has written the outputs (a uniform decision).
  if (NC > 1 && want_idx && cmode != 0 && ncand > kAllCap) cluster_sync_all();
}

template <int NC, int W, bool RT, bool Q8 = false>
static cudaError_t launch_finish_t(const FinishArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(FinShared<NC, W>);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(NC, a.B * a.Hq);
  cfg.blockDim = dim3(32 * W);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(finish_kernel<NC, W, RT, Q8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return cudaLaunchKernelEx(&cfg, finish_kernel<NC, W, RT, Q8>, a);
}

// Cluster size: the largest of 8, 4, 2 whose CTAs for every head (one CTA of
// 16 warps per SM: 512 threads x 128 registers) fill at most 85 % of the SMs.
// A cluster must sit in one GPC, so a nearly full device places fewer large
// clusters than its SM count suggests: 32 clusters of 8 CTAs at two per SM
// left two clusters for a second wave.  With more heads than that every
// decode head is one CTA of 8 warps, two per SM (one CTA of 16 warps per head
// was measured 7 us slower on 16 paged sequences of 32 heads), and every
// ReTopK head one CTA of 16 warps (8 warps: 4 sequences' batched step 35.3 ->
// 40.2 us).
cudaError_t launch_finish(const FinishArgs& a, cudaStream_t st) {
  static int sms[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (!sms[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    sms[dev] = v > 0 ? v : 148;
  }
  const int64_t heads = (int64_t)a.B * a.Hq;
  const int64_t slots = (int64_t)sms[dev] * 85 / 100;
  const int nc = heads * 8 <= slots ? 8 : heads * 4 <= slots ? 4 : heads * 2 <= slots ? 2 : 1;
  if (a.path) {  // a ReTopK step
    switch (nc) {
      case 8: return launch_finish_t<8, 16, true>(a, st);
      case 4: return launch_finish_t<4, 16, true>(a, st);
      case 2: return launch_finish_t<2, 16, true>(a, st);
      default: return launch_finish_t<1, 16, true>(a, st);
    }
  }
  if (a.q8_eps) {  // a decode step after the quantised scan
    switch (nc) {
      case 8: return launch_finish_t<8, 16, false, true>(a, st);
      case 4: return launch_finish_t<4, 16, false, true>(a, st);
      case 2: return launch_finish_t<2, 16, false, true>(a, st);
      default: return launch_finish_t<1, 8, false, true>(a, st);
    }
  }
  switch (nc) {
    case 8: return launch_finish_t<8, 16, false>(a, st);
    case 4: return launch_finish_t<4, 16, false>(a, st);
    case 2: return launch_finish_t<2, 16, false>(a, st);
    default: return launch_finish_t<1, 8, false>(a, st);
  }
}

}  // namespace tsa
