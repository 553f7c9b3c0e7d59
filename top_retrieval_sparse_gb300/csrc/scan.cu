// scan.cu -- GQA key scan: z[h][i] = scale * q_h . k_{g(h), i} for every key.
//
// "RetrievalAttention" Eq. 1 logits and the Flat (exact KNN) scan; ReTopK's
// exact path ("Exact Top-K" e_{t,i}).  Each bf16 key row is read from HBM
// once per KV head and used for all query heads of its group.
//
// Design (sm_103a):
//   * persistent CTAs (one per SM), each owning a contiguous range of 256-row
//     tiles, balanced over the (sequence, KV head) units that have an active
//     query head;
//   * warp-specialised: one producer warp streams tiles global -> shared by
//     1-D bulk copies (cp.async.bulk with an L2 evict-first hint) into a
//     3-stage ring (64 KiB stages) with full/empty mbarriers; 16 consumer
//     warps never synchronise per tile (a paged cache issues one copy per
//     page segment of a tile);
//   * the contraction [16 keys x 128] . [128 x 8 heads] runs on the tensor
//     cores (mma.m16n8k16, bf16 in, fp32 accumulate): each warp owns 16 rows
//     of a tile, keys are the M operand and the (padded) query heads of the
//     group the N operand.  The reduction index is permuted identically in
//     both operands so that every lane reads its A fragment of two k-steps
//     as one contiguous 16-byte shared load (rows are 256 bytes apart, so a
//     load phase sees a 2-way bank conflict);
//   * pool positions (outside the static window) whose bin -- the top 11
//     bits of the order-preserving logit key -- is >= the head's hint bin
//     are emitted as (position, logit) pairs into the head's dense list; each
//     warp bump-allocates runs of 8 slots (one global atomic per run) and
//     pads the tail of its last run with sentinels -- no logit array is
//     written or re-read; window logits are written out;
//   * every emitted pair is also counted, with one global reduction, in its
//     fine bin -- 16 key bits, relative to the emission key -- of the head's
//     histogram, from which the finish kernel takes the threshold bin b*
//     without a pass over the pairs; when the emission fell short, or b* is
//     the histogram's last bin (which holds everything above it), the finish
//     kernel counts the pairs' 11-bit bins itself or re-scores the head's keys
//     and re-emits: exactness never depends on the hint, only the cost does.
//     (A shared-memory histogram of every pool position cost the consumers as
//     much as the emission; counting only the emitted pairs, ~5 % of the
//     rows, costs nothing measurable);
//   * a plain scan of every head loads its first unit's query fragments, an
//     input of the call, before the dependency wait.
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

constexpr int kScanWarps = 16;                     // consumer warps
constexpr int kConsumers = 32 * kScanWarps;
constexpr int kScanThreads = kConsumers + 32;      // + one producer warp
constexpr int kTileBytes = 16 * kScanWarps * kRowBytes;  // 64 KiB
constexpr int kStages = 3;
// Tile geometry: bf16 rows (256 bytes, one m16 block per consumer warp) or
// key codes (128 bytes, two m16 blocks per consumer warp).
template <bool Q8>
struct Geom {
  static constexpr int kRB = Q8 ? kD : kRowBytes;   // bytes per row
  static constexpr int kTR = kTileBytes / kRB;      // rows per tile
  static constexpr int kNB = kTR / (16 * kScanWarps);  // m16 blocks per warp
};

size_t scan_smem_bytes() {
  return (size_t)kStages * kTileBytes + 2 * kStages * 8 + (kMaxUnits + 1) * 4 + 64;
}

__device__ __forceinline__ uint32_t u4_word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

template <bool Q8>
__global__ void __launch_bounds__(kScanThreads, 1) scan_kernel(ScanArgs a) {
  constexpr int kTileRows = Geom<Q8>::kTR, kRB = Geom<Q8>::kRB, kNB = Geom<Q8>::kNB;
  TraceScope trace(a.trace, kTrScan);
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kTileBytes);
  uint64_t* empty = full + kStages;
  int* unit_tiles = reinterpret_cast<int*>(empty + kStages);  // prefix over units
  __shared__ volatile int s_abort;
  __shared__ int stage_tile[kStages];  // tile of each ring stage (-1: no more tiles)

  if (a.head_active) pdl_wait();  // the activity flags come from the previous grid
  pdl_trigger();
  const int tid = threadIdx.x;
  const int G = a.Hq / a.kv.Hkv;
  const int nunits = a.B * a.kv.Hkv;

  // ---- prefix of tiles over (sequence, KV head) units with an active head ----
  // With an activity filter the block first marks the units with an active
  // head (every head's flag read at once, one thread each).
  if (a.head_active) {
    for (int u = tid; u < nunits; u += kScanThreads) unit_tiles[u] = 0;
    __syncthreads();
    for (int i = tid; i < nunits * G; i += kScanThreads)
      if (a.head_active[i] == a.active_value) unit_tiles[i / G] = 1;
    __syncthreads();
  }
  if (tid < 32) {
    int run = 0;
    for (int base = 0; base < nunits; base += 32) {
      const int u = base + tid;
      int tiles = 0;
      if (u < nunits) {
        const int b = u / a.kv.Hkv;
        const bool act = !a.head_active || unit_tiles[u] != 0;
        const int64_t L = seq_len(a.lens, a.len_host, a.len_step, b, a.kv.l_cap);
        tiles = act ? (int)((L + kTileRows - 1) / kTileRows) : 0;
      }
      int incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      if (u < nunits) unit_tiles[u] = run + incl - tiles;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (tid == 0) unit_tiles[nunits] = run;
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kScanWarps);
    }
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();

  // Contiguous static ranges; with 8 or more tiles per CTA the last 5 % (10 %
  // from 64 tiles per CTA) are claimed one tile at a time (global counter) by
  // whichever CTA is free first, so that CTAs that start later (their SM was
  // still running the previous kernel) or get a smaller share of HBM
  // bandwidth end no later.  A claimed tile may switch the warp to another
  // (sequence, KV head) unit: the warp closes its emission runs and reloads
  // the query fragments, nothing more (measured at 128K, 27 tiles per CTA:
  // 5 % dynamic -1.2 us per step, 10 % -1.1 us).
  const int total = unit_tiles[nunits];
  if (total == 0) return;
  const int grid = gridDim.x;
  const int dyn = total >= 64 * grid ? total / 10 : total >= 8 * grid ? total / 20 : 0;
  const int stat = total - dyn;
  const int t_begin = (int)((int64_t)stat * blockIdx.x / grid);
  const int t_end = (int)((int64_t)stat * (blockIdx.x + 1) / grid);

  // global tile index -> unit (last unit whose first tile is <= t)
  auto locate = [&](int t) {
    int lo = 0, hi = nunits - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (unit_tiles[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    return lo;
  };

  const int warp = tid >> 5, lane = tid & 31;
  const long long lim = a.wait_ns > 0 ? a.wait_ns : kWaitLimitNs;

  // ======================= producer warp: the bulk-copy ring ==================
  // Lane 0 waits for free stages and arms the full barrier; a contiguous tile
  // is one copy (lane 0), a paged tile one copy per page, issued by the lanes
  // in parallel so that the page-table reads overlap (tiles start on a page
  // boundary: 256 and 512 rows are multiples of every page size).
  if (warp == kScanWarps) {
    const uint64_t pol = policy_evict_first();
    int next_static = t_begin;
    int claim = -1;  // lane 0: dynamic claim requested one tile ahead (-1: none)
    // the claim counter is cleared by the previous grid: claims wait for it
    bool waited = a.head_active != nullptr;
    int j = 0;
    bool marker = false;
    bool codes_ready = !Q8 || a.q8_new <= 0;  // (warp-uniform)
    for (;; ++j) {
      const int s = j % kStages;
      int go = 1, t = -1;
      if (lane == 0) {
        if (j >= kStages &&
            !mbar_wait_or_abort(&empty[s], (uint32_t)((j / kStages - 1) & 1), &s_abort, lim)) {
          s_abort = 1;
          go = 0;
        }
        if (s_abort) go = 0;
        if (go) {
          if (next_static < t_end) {
            t = next_static++;
          } else if (dyn > 0) {
            if (!waited) {
              pdl_wait();
              waited = true;
            }
            const int c = claim >= 0 ? claim : (int)atomicAdd(a.tile_ctr, 1u);
            claim = -1;
            t = c < dyn ? stat + c : -1;
          }
          // the next tile is a dynamic one: claim it now, so that the
          // atomic's round trip overlaps the wait for a free stage
          if (t >= 0 && next_static >= t_end && dyn > 0) {
            if (!waited) {
              pdl_wait();
              waited = true;
            }
            claim = (int)atomicAdd(a.tile_ctr, 1u);
          }
          stage_tile[s] = t;
          if (t < 0) mbar_arrive(&full[s]);  // no more tiles: release the consumers
        }
      }
      go = __shfl_sync(0xffffffffu, go, 0);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (!go) break;
      if (t < 0) {
        marker = true;
        break;
      }
      const int unit = locate(t);
      const int tile = t - unit_tiles[unit];
      const int b = unit / a.kv.Hkv, g = unit % a.kv.Hkv;
      const int64_t L = seq_len(a.lens, a.len_host, a.len_step, b, a.kv.l_cap);
      const int64_t r0 = (int64_t)tile * kTileRows;
      const int64_t r1 = r0 + kTileRows < L ? r0 + kTileRows : L;
      const uint32_t bytes = (uint32_t)(r1 - r0) * kRB;
      uint8_t* dst = ring + s * kTileBytes;
      // fault injection (tests only): the first stage is never armed or filled
      if (a.stall_first_copy && blockIdx.x == 0 && j == 0) continue;
      // the newest rows' codes are written by the preceding kernel
      if (!codes_ready && r1 > L - a.q8_new) {
        pdl_wait();
        codes_ready = true;
      }
      auto src = [&](int64_t r) -> const void* {
        if constexpr (Q8) return a.codes + kv_row(a.kv, b, g, r);
        else return a.kv.k + kv_row(a.kv, b, g, r);
      };
      if (lane == 0) {
        fence_proxy_async();
        mbar_expect_tx(&full[s], bytes);
      }
      __syncwarp();
      if (!a.kv.page_table) {
        if (lane == 0) bulk_g2s(dst, src(r0), bytes, &full[s], pol);
      } else {
        const int64_t ps = (int64_t)1 << a.kv.page_shift;
        const int nseg = (int)((r1 - r0 + ps - 1) >> a.kv.page_shift);  // <= 32
        for (int k = lane; k < nseg; k += 32) {
          const int64_t r = r0 + (int64_t)k * ps;
          const int64_t e = r + ps < r1 ? r + ps : r1;
          fence_proxy_async();
          bulk_g2s(dst + (r - r0) * kRB, src(r), (uint32_t)(e - r) * kRB, &full[s], pol);
        }
      }
    }
    // copies of the last (up to kStages) tiles may still be landing; after the
    // end marker, the stage it used had been seen consumed
    if (lane == 0)
      for (int jj = j - kStages + (marker ? 1 : 0) > 0 ? j - kStages + (marker ? 1 : 0) : 0; jj < j;
           ++jj)
        (void)mbar_wait(&full[jj % kStages], (uint32_t)((jj / kStages) & 1), lim);
    return;
  }

  // ============================ consumer warps ================================
  // Launched as a programmatic dependent, the scan streams keys while the
  // previous kernel finishes; its consumers read the query fragments of their
  // first unit (inputs of the call) before the dependency wait, and hints,
  // counters, pairs and logits only after that kernel has completed.
  const int gr = lane >> 2;  // A rows gr, gr+8 / B column (query head) gr
  const int tq = lane & 3;   // k-slot group / C columns 2tq, 2tq+1

  // B fragments of head gr: bf16, d in [8(4p+tq), +8) for p < 4; or, for
  // the codes, fp16 qh with d in [16 tq, +16) then [64 + 16 tq, +16)
  uint32_t qb[4][4];
  float qts[2] = {0.f, 0.f};    // codes: logit factors of heads 2tq, 2tq+1
  bool on[2] = {false, false};  // heads 2tq, 2tq+1 are active
  // emission thresholds of heads 2tq, 2tq+1 as floats: z >= thr exactly when
  // f2key(z) >= the head's key (-inf: every logit; NaN: an inactive head)
  float ethr[2] = {__int_as_float(0x7fc00000), __int_as_float(0x7fc00000)};
  uint32_t hbase[2] = {0u, 0u};  // fine-histogram base bins (emission key >> 16)
  bool lane_on = false;         // lane h < G: head h takes part (run owner)
  int run_ptr = 0;              // lane h < G: next free slot of this warp's run for head h
  int run_left = 0;             //            slots left in that run
  int cur_unit = -1, unit_end = 0, cur_b = 0, cur_g = 0, head0 = 0;
  int64_t cur_L = 0;
  bool aborted = false;

  // this warp leaves the current unit: pad the unused tail of its runs with
  // sentinels
  auto close_runs = [&]() {
    if (lane < G && run_left > 0) {
      uint2* row = a.dense + (int64_t)(head0 + lane) * a.dense_stride;
      for (int k = 0; k < run_left; ++k)
        if ((int64_t)run_ptr + k < a.dense_stride) row[run_ptr + k] = make_uint2(0xffffffffu, 0u);
    }
    run_ptr = 0;
    run_left = 0;
  };
  // entering a unit (each warp on its own: no barrier): what depends only on
  // the call's inputs -- heads, length, query fragments ...
  auto enter_inputs = [&](int unit) {
    cur_unit = unit;
    unit_end = unit_tiles[unit + 1];
    cur_b = unit / a.kv.Hkv;
    cur_g = unit % a.kv.Hkv;
    head0 = cur_b * a.Hq + cur_g * G;
    cur_L = seq_len(a.lens, a.len_host, a.len_step, cur_b, a.kv.l_cap);  // < 2^31
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int hl = 2 * tq + e;
      on[e] = hl < G && (!a.head_active || a.head_active[head0 + hl] == a.active_value);
    }
    lane_on = lane < G && (!a.head_active || a.head_active[head0 + lane] == a.active_value);
    if constexpr (Q8) {
      const uint16_t* qp = a.qh + ((int64_t)head0 + (gr < G ? gr : 0)) * kD;
#pragma unroll
      for (int p = 0; p < 4; ++p) {  // p: dims 16 tq + 8p (p < 2), 64 + 16 tq + 8 (p - 2)
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (gr < G) w = __ldcg(reinterpret_cast<const uint4*>(qp + 64 * (p >> 1) + 16 * tq +
                                                              8 * (p & 1)));
        qb[p][0] = w.x; qb[p][1] = w.y; qb[p][2] = w.z; qb[p][3] = w.w;
      }
    } else {
      const uint16_t* qp = a.q + ((int64_t)head0 + (gr < G ? gr : 0)) * kD;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (gr < G) w = *reinterpret_cast<const uint4*>(qp + 8 * (4 * p + tq));
        qb[p][0] = w.x; qb[p][1] = w.y; qb[p][2] = w.z; qb[p][3] = w.w;
      }
    }
  };
  // ... and what the previous kernel wrote: the emission keys (and the
  // codes' logit factors)
  auto enter_state = [&]() {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int bh = head0 + 2 * tq + e;
      const uint32_t ek = on[e] ? __ldcg(a.emit_key + bh) : 0u;
      // keys at or below f2key(-inf) admit every finite logit
      ethr[e] = !on[e] ? __int_as_float(0x7fc00000) : ek <= 0x007fffffu ? -INFINITY : key2f(ek);
      hbase[e] = ek >> kH16Shift;
      if constexpr (Q8) qts[e] = on[e] ? __ldcg(a.qts + bh) : 0.f;
    }
  };
  // a plain scan of every head reads its first unit's query before the wait
  const bool early = !Q8 && !a.head_active && t_begin < t_end;
  if (early) enter_inputs(locate(t_begin));
  pdl_wait();
  if (early) enter_state();
  for (int j = 0;; ++j) {
    const int s = j % kStages;
    if (!mbar_wait_or_abort(&full[s], (uint32_t)((j / kStages) & 1), &s_abort, lim)) {
      s_abort = 1;
      aborted = true;
      break;
    }
    const int t = stage_tile[s];  // written by the producer before it armed the stage
    if (t < 0) break;             // no more tiles (same stage, same j, for every warp)
    if (t >= unit_end) {  // entering a new unit
      const int unit = locate(t);
      if (cur_unit >= 0) close_runs();
      enter_inputs(unit);
      enter_state();
    }
    const int tile = t - unit_tiles[cur_unit];
    if (j == 0) trace.mark(1);
    // ---- 16 keys x 8 heads on the tensor cores, per m16 block ----
    // C: (row gr, head 2tq), (row gr, head 2tq+1), (row gr+8, 2tq), (row gr+8, 2tq+1)
    float zb[kNB][4];
    if constexpr (Q8) {
      // lane: rows gr, gr+8 of each block, bytes [16 tq, +16) and [64 + 16 tq,
      // +16); all loads first, so the stage is released before the math.  In
      // k-step m, dims 4m..4m+3 of the lane's 32 (word m%4 of chunk m/4) are
      // the k-slots (2tq, 2tq+1, 2tq+8, 2tq+9), and qb holds qh in that order.
      const uint8_t* wb = ring + s * kTileBytes + warp * kNB * 16 * kD;
      uint4 R[kNB][4];
#pragma unroll
      for (int blk = 0; blk < kNB; ++blk)
#pragma unroll
        for (int c = 0; c < 4; ++c)
          R[blk][c] = *reinterpret_cast<const uint4*>(wb + (blk * 16 + gr + 8 * (c >> 1)) * kD +
                                                      64 * (c & 1) + 16 * tq);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with stage s
#pragma unroll
      for (int blk = 0; blk < kNB; ++blk) {
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint32_t wa = u4_word(R[blk][m >> 2], m & 3);
          const uint32_t wc = u4_word(R[blk][2 + (m >> 2)], m & 3);
          mma_f16((m & 1) ? c1 : c0, codes_lo_f16x2(wa), codes_lo_f16x2(wc), codes_hi_f16x2(wa),
                  codes_hi_f16x2(wc), qb[m >> 1][2 * (m & 1)], qb[m >> 1][2 * (m & 1) + 1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) zb[blk][e] = (c0[e] + c1[e]) * qts[e & 1];
      }
    } else {
      const uint8_t* wb = ring + s * kTileBytes + warp * 16 * kRowBytes;
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint4 W = *reinterpret_cast<const uint4*>(wb + gr * kRowBytes + 16 * (4 * p + tq));
        const uint4 X =
            *reinterpret_cast<const uint4*>(wb + (gr + 8) * kRowBytes + 16 * (4 * p + tq));
        mma_bf16(c0, W.x, X.x, W.y, X.y, qb[p][0], qb[p][1]);
        mma_bf16(c1, W.z, X.z, W.w, X.w, qb[p][2], qb[p][3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with stage s
#pragma unroll
      for (int e = 0; e < 4; ++e) zb[0][e] = (c0[e] + c1[e]) * a.scale;
    }
#pragma unroll
    for (int blk = 0; blk < kNB; ++blk) {
      // row indices fit in 32 bits (l_cap < 2^31)
      const int Lc = (int)cur_L;
      const int rb = tile * kTileRows + (warp * kNB + blk) * 16;
      const int rowA = rb + gr;
      const float* zv = zb[blk];
      unsigned emit = 0u;
      if (rb >= a.n_init && rb + 16 <= Lc - a.n_recent) {  // a pool block (warp-uniform)
#pragma unroll
        for (int e = 0; e < 4; ++e) emit |= (zv[e] >= ethr[e & 1] ? 1u : 0u) << e;
      } else {  // meets the window or the end of the sequence
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = rowA + ((e >> 1) << 3);
          if (on[e & 1] && i < Lc) {
            if (in_window(i, Lc, a.n_init, a.n_recent)) {
              // (the rescoring computes the codes' window logits exactly)
              if constexpr (!Q8) {
                const int wa = a.n_init < Lc ? a.n_init : Lc;
                const int lo = Lc - a.n_recent > wa ? Lc - a.n_recent : wa;
                const int wj = i < wa ? i : wa + (i - lo);
                a.wz[(int64_t)(head0 + 2 * tq + (e & 1)) * a.wz_stride + wj] = zv[e];
              }
            } else if (zv[e] >= ethr[e & 1]) {
              emit |= 1u << e;
            }
          }
        }
      }
      if (!__any_sync(0xffffffffu, emit)) continue;  // nothing to emit in this block
      // emission: per head, this warp's pairs of the tile (rows gr, then
      // gr+8, by lane) continue its current run; lane h extends the run by
      // bump allocation (one atomic per 8 slots) and broadcasts where they go
      unsigned m[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) m[e] = __ballot_sync(0xffffffffu, (emit >> e) & 1u);
      if (m[0] | m[1] | m[2] | m[3]) {
        int p1 = 0, p2 = 0, take = 0;  // slots fit in 32 bits (lists are < 2^31)
        if (lane_on) {  // lane = head in group
          const unsigned M = 0x11111111u << (lane >> 1);
          const unsigned ma = (lane & 1) ? m[1] : m[0], mb = (lane & 1) ? m[3] : m[2];
          const int cnt = __popc(ma & M) + __popc(mb & M);
          if (cnt) {
            take = cnt < run_left ? cnt : run_left;
            p1 = run_ptr;
            const int over = cnt - take;
            if (over > 0) {
              // runs of 8 within a static range; a dynamic tile is a visit of
              // its own: it rounds its pairs up to a 32-byte sector only
              const int size = t < stat ? (over + 7) & ~7 : (over + 3) & ~3;
              p2 = atomicAdd(&a.dense_n[(int64_t)(head0 + lane) * kCtrStride], size);
              run_ptr = p2 + over;
              run_left = size - over;
            } else {
              run_ptr += cnt;
              run_left -= cnt;
            }
          }
        }
        const unsigned M = 0x11111111u << tq;
        const unsigned lt = (1u << lane) - 1u;
#pragma unroll
        for (int par = 0; par < 2; ++par) {
          if (!(m[par] | m[par + 2])) continue;  // warp-uniform: no pair of this parity
          const int src = 2 * tq + par;  // lane owning head 2tq+par's run
          const int q1 = __shfl_sync(0xffffffffu, p1, src);
          const int q2 = __shfl_sync(0xffffffffu, p2, src);
          const int qt = __shfl_sync(0xffffffffu, take, src);
          const int below = __popc(m[par] & M);
          uint2* drow = a.dense + (int64_t)(head0 + src) * a.dense_stride;
#pragma unroll
          for (int hi = 0; hi < 2; ++hi) {
            const int e = par + 2 * hi;
            if (!((emit >> e) & 1u)) continue;
            const int r = hi == 0 ? __popc(m[par] & M & lt) : below + __popc(m[par + 2] & M & lt);
            const int slot = r < qt ? q1 + r : q2 + (r - qt);
            if (slot < a.dense_stride)
              drow[slot] = make_uint2((uint32_t)(rowA + 8 * hi), __float_as_uint(zv[e]));
            if constexpr (!Q8) {
              if (a.hist16) {  // (the key is >= the emission key: the bin is >= 0)
                const uint32_t fb =
                    min((f2key(zv[e]) >> kH16Shift) - hbase[par], (uint32_t)kH16Bins - 1u);
                atomicAdd(a.hist16 + (int64_t)(head0 + src) * kH16Bins + fb, 1u);
              }
            }
          }
        }
      }
    }
  }

  // a warp whose bounded wait expired reports it; its pairs are incomplete
  if (aborted) {
    if (lane == 0) atomicOr(a.status, kStatusTimeout);
    return;
  }
  trace.mark(2);
  if (cur_unit >= 0) close_runs();
}

template <bool Q8>
static cudaError_t launch_scan_t(const ScanArgs& a, int grid, cudaStream_t st, bool pdl) {
  const size_t smem = scan_smem_bytes();
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(scan_kernel<Q8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kScanThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, scan_kernel<Q8>, a);
}

int scan_tile_rows() { return Geom<false>::kTR; }
int scan_grid_rows(bool q8) { return q8 ? Geom<true>::kTR : Geom<false>::kTR; }
int scan_tile_warps() { return kScanWarps; }

cudaError_t launch_scan(const ScanArgs& a, int grid, cudaStream_t st, bool pdl) {
  return a.codes ? launch_scan_t<true>(a, grid, st, pdl) : launch_scan_t<false>(a, grid, st, pdl);
}

}  // namespace tsa
