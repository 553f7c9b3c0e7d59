// scan.cu -- GQA key scan: z[h][i] = scale * q_h . k_{g(h), i} for every key.
//
// "RetrievalAttention" Eq. 1 logits and the Flat (exact KNN) scan; ReTopK's
// exact path ("Exact Top-K" e_{t,i}).  Each bf16 key row is read from HBM
// once per KV head and used for all query heads of its group.
//
// Design (sm_103a):
//   * persistent CTAs, a contiguous range of 64-row tiles each, balanced over
//     the (sequence, KV head) units with at least one active query head;
//   * tiles stream global -> shared by 1-D bulk copies (cp.async.bulk with an
//     L2 evict-first hint) into a 4-stage ring completed on mbarriers; a paged
//     cache issues one copy per page segment of a tile;
//   * 8 lanes cooperate on one 256-byte row (16 elements each, two 16-byte
//     shared loads at lane*16 and 128+lane*16: conflict-free), packed fp32x2
//     FMAs against the group's queries held in registers, then a
//     reduce-scatter over the 8 lanes leaves one (row, head) logit per lane;
//   * the pass-1 radix histogram (top 11 bits of the order-preserving key) of
//     every active head is built in shared memory over positions outside the
//     static window and flushed to global memory with one atomic per
//     non-empty bin.
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

constexpr int kScanThreads = 256;
constexpr int kTileRows = 64;
constexpr int kStages = 4;
constexpr int kTileBytes = kTileRows * kRowBytes;  // 16 KiB

template <int GP>
struct ScanShape {
  static constexpr int HG = GP > 4 ? 4 : GP;        // heads per head-group
  static constexpr int NHG = GP / HG;               // head-groups (1 or 2)
  static constexpr int TPG = kScanThreads / NHG;    // threads per head-group
  static constexpr int RPP = TPG / 8;               // rows per pass
  static constexpr int R = kTileRows / RPP;         // rows per thread per tile
  static constexpr int NV = R * HG;                 // values per lane before reduce
  static constexpr int NOUT = NV >= 8 ? NV / 8 : 1; // values per lane after reduce
};

template <int GP>
size_t scan_smem_bytes() {
  return (size_t)kStages * kTileBytes + (size_t)GP * kHistBins * 4 + kStages * 8 +
         (kMaxUnits + 1) * 4 + 64;
}

// Reduce NV per-lane partial sums across the 8 lanes of a row group.
// After the call lane `lr` holds NOUT complete sums in v[0..NOUT); their
// original indices are base + i, with base returned.
template <int NV>
__device__ __forceinline__ int reduce8(float (&v)[NV], int lr) {
  int base = 0;
  int cur = NV;
#pragma unroll
  for (int mask = 4; mask >= 1; mask >>= 1) {
    if (cur >= 2) {
      const int half = cur / 2;
      const bool bit = (lr & mask) != 0;
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) {
        if (i < half) {
          float send = bit ? v[i] : v[i + half];
          float keep = bit ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
        }
      }
      if (bit) base += half;
      cur = half;
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
    }
  }
  return base;
}

template <int GP>
__global__ void __launch_bounds__(kScanThreads) scan_kernel(ScanArgs a) {
  using S = ScanShape<GP>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kStages * kTileBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(hist + GP * kHistBins);
  int* unit_tiles = reinterpret_cast<int*>(full + kStages);  // prefix over units

  const int tid = threadIdx.x;
  const int G = a.Hq / a.kv.Hkv;
  const int nunits = a.B * a.kv.Hkv;

  // ---- prefix of tiles over (sequence, KV head) units with an active head ----
  if (tid < 32) {
    int run = 0;
    for (int base = 0; base < nunits; base += 32) {
      const int u = base + tid;
      int tiles = 0;
      if (u < nunits) {
        const int b = u / a.kv.Hkv, g = u % a.kv.Hkv;
        bool act = true;
        if (a.head_active) {
          act = false;
          for (int j = 0; j < G; ++j)
            act |= a.head_active[b * a.Hq + g * G + j] == a.active_value;
        }
        const int64_t L = seq_len(a.lens, a.len_host, b, a.kv.l_cap);
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
  for (int i = tid; i < GP * kHistBins; i += kScanThreads) hist[i] = 0;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int total = unit_tiles[nunits];
  const int t_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int t_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  const int ntile = t_end - t_begin;
  if (ntile <= 0) return;

  // global tile index -> (unit, tile within the unit)
  auto locate = [&](int t, int& unit, int& tile) {
    int lo = 0, hi = nunits - 1;
    while (lo < hi) {  // last unit whose first tile is <= t
      const int mid = (lo + hi + 1) >> 1;
      if (unit_tiles[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    unit = lo;
    tile = t - unit_tiles[lo];
  };

  const uint64_t pol = policy_evict_first();
  // producer (thread 0): stream tile t into stage s
  auto issue = [&](int t, int s) {
    int unit, tile;
    locate(t, unit, tile);
    const int b = unit / a.kv.Hkv, g = unit % a.kv.Hkv;
    const int64_t L = seq_len(a.lens, a.len_host, b, a.kv.l_cap);
    const int64_t r0 = (int64_t)tile * kTileRows;
    const int64_t r1 = r0 + kTileRows < L ? r0 + kTileRows : L;
    const uint32_t bytes = (uint32_t)(r1 - r0) * kRowBytes;
    mbar_expect_tx(&full[s], bytes);
    uint8_t* dst = ring + s * kTileBytes;
    if (!a.kv.page_table) {
      bulk_g2s(dst, a.kv.k + kv_row(a.kv, b, g, r0), bytes, &full[s], pol);
    } else {
      const int64_t ps = (int64_t)1 << a.kv.page_shift;
      for (int64_t r = r0; r < r1;) {
        const int64_t pe = ((r >> a.kv.page_shift) + 1) * ps;
        const int64_t e = pe < r1 ? pe : r1;
        bulk_g2s(dst + (r - r0) * kRowBytes, a.kv.k + kv_row(a.kv, b, g, r),
                 (uint32_t)(e - r) * kRowBytes, &full[s], pol);
        r = e;
      }
    }
  };

  if (tid == 0) {
    const int pre = ntile < kStages ? ntile : kStages;
    for (int j = 0; j < pre; ++j) issue(t_begin + j, j);
  }

  // thread roles
  const int hgi = tid / S::TPG;  // head-group index
  const int t2 = tid % S::TPG;
  const int lr = t2 & 7;         // lane within the 8-lane row group
  const int rp = t2 >> 3;        // row within a pass

  float2 qf[S::HG][8];           // this lane's 16 query elements, per head
  unsigned act_bits = 0;         // heads (of this head-group) that are active
  int cur_unit = -1, cur_b = 0, cur_g = 0;
  int64_t cur_L = 0;

  auto flush_hist = [&](int unit) {
    const int b = unit / a.kv.Hkv, g = unit % a.kv.Hkv;
    for (int i = tid; i < GP * kHistBins; i += kScanThreads) {
      const uint32_t c = hist[i];
      if (c) {
        const int hl = i / kHistBins;
        atomicAdd(&a.hist[(int64_t)(b * a.Hq + g * G + hl) * kHistBins + (i % kHistBins)], c);
        hist[i] = 0;
      }
    }
  };

  int j = 0;
  for (; j < ntile; ++j) {
    const int s = j % kStages;
    const int t = t_begin + j;
    int unit, tile;
    locate(t, unit, tile);
    if (unit != cur_unit) {
      if (cur_unit >= 0) {
        __syncthreads();
        flush_hist(cur_unit);
        __syncthreads();
      }
      cur_unit = unit;
      cur_b = unit / a.kv.Hkv;
      cur_g = unit % a.kv.Hkv;
      cur_L = seq_len(a.lens, a.len_host, cur_b, a.kv.l_cap);
      act_bits = 0;
#pragma unroll
      for (int i = 0; i < S::HG; ++i) {
        const int hl = hgi * S::HG + i;
        const int h = cur_g * G + (hl < G ? hl : 0);
        if (hl < G && (!a.head_active || a.head_active[cur_b * a.Hq + h] == a.active_value))
          act_bits |= 1u << i;
        const uint16_t* qp = a.q + ((int64_t)cur_b * a.Hq + h) * kD;
        const uint4 w0 = *reinterpret_cast<const uint4*>(qp + lr * 8);
        const uint4 w1 = *reinterpret_cast<const uint4*>(qp + 64 + lr * 8);
        const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
          qf[i][e] = hl < G ? make_float2(bf_lo(ws[e]), bf_hi(ws[e])) : make_float2(0.f, 0.f);
      }
    }
    const bool ok = mbar_wait(&full[s], (uint32_t)((j / kStages) & 1));
    if (__syncthreads_or(!ok)) break;  // uniform decision: leave on timeout

    const uint8_t* tileb = ring + s * kTileBytes;
    const int64_t r0 = (int64_t)tile * kTileRows;
    float v[S::NV];
#pragma unroll
    for (int k = 0; k < S::R; ++k) {
      const uint8_t* rb = tileb + (rp + k * S::RPP) * kRowBytes;
      const uint4 w0 = *reinterpret_cast<const uint4*>(rb + lr * 16);
      const uint4 w1 = *reinterpret_cast<const uint4*>(rb + 128 + lr * 16);
      const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      float2 acc[S::HG];
#pragma unroll
      for (int i = 0; i < S::HG; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float2 kk = make_float2(bf_lo(ws[e]), bf_hi(ws[e]));
#pragma unroll
        for (int i = 0; i < S::HG; ++i) ffma2(acc[i], kk, qf[i][e]);
      }
#pragma unroll
      for (int i = 0; i < S::HG; ++i) v[k * S::HG + i] = acc[i].x + acc[i].y;
    }
    const int base = reduce8<S::NV>(v, lr);
    // lanes holding a duplicate of a value (NV < 8) do not write it
    const bool owner = (S::NV >= 8) || ((lr & (8 / S::NV - 1)) == 0);
#pragma unroll
    for (int o = 0; o < S::NOUT; ++o) {
      const int idx = base + o;
      const int k = idx / S::HG;
      const int il = idx % S::HG;
      const int64_t i = r0 + rp + k * S::RPP;
      if (owner && ((act_bits >> il) & 1u) && i < cur_L) {
        const int hl = hgi * S::HG + il;
        const int h = cur_g * G + hl;
        const float z = v[o] * a.scale;
        a.scores[((int64_t)cur_b * a.Hq + h) * a.score_stride + i] = z;
        if (!in_window(i, cur_L, a.n_init, a.n_recent))
          atomicAdd(&hist[hl * kHistBins + (f2key(z) >> kHistShift)], 1u);
      }
    }
    __syncthreads();  // stage s fully consumed
    if (tid == 0 && j + kStages < ntile) {
      fence_proxy_async();
      issue(t + kStages, s);
    }
  }

  if (j < ntile) {  // a bounded wait expired: report, drain in-flight copies, leave
    if (tid == 0) {
      atomicOr(a.status, kStatusTimeout);
      const int last = ntile < j + kStages ? ntile : j + kStages;
      for (int jj = j; jj < last; ++jj)
        (void)mbar_wait(&full[jj % kStages], (uint32_t)((jj / kStages) & 1));
    }
    __syncthreads();
    return;
  }
  __syncthreads();
  if (cur_unit >= 0) flush_hist(cur_unit);
}

template <int GP>
static cudaError_t launch_scan_t(const ScanArgs& a, int grid, cudaStream_t st) {
  const size_t smem = scan_smem_bytes<GP>();
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(scan_kernel<GP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  scan_kernel<GP><<<grid, kScanThreads, smem, st>>>(a);
  return cudaGetLastError();
}

int scan_padded_group(int G) { return G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8; }

int scan_ctas_per_sm(int G) {
  const int GP = scan_padded_group(G);
  size_t smem = GP == 1 ? scan_smem_bytes<1>() : GP == 2 ? scan_smem_bytes<2>()
              : GP == 4 ? scan_smem_bytes<4>() : scan_smem_bytes<8>();
  int per = (int)((227 * 1024 + 1024) / (smem + 1024));
  return per < 1 ? 1 : per;
}

cudaError_t launch_scan(const ScanArgs& a, int grid, cudaStream_t st) {
  const int G = a.Hq / a.kv.Hkv;
  switch (scan_padded_group(G)) {
    case 1: return launch_scan_t<1>(a, grid, st);
    case 2: return launch_scan_t<2>(a, grid, st);
    case 4: return launch_scan_t<4>(a, grid, st);
    default: return launch_scan_t<8>(a, grid, st);
  }
}

}  // namespace tsa
