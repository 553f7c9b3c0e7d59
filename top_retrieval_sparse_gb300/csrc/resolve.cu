// resolve.cu -- exact top-K from the pairs the key scan emitted.
//
// "RetrievalAttention" Eq. 2 (the selected set, top-k by inner product as in
// the Flat baseline) with W and Omega disjoint (Eq. 3); ReTopK's exact path
// S_t = TopK(e, K).  Ties go to the smaller position.
//
// The scan emitted, for every head, the (position, logit) pairs of all pool
// positions whose radix bin is at least its emission bin into the head's
// dense list (sentinel-padded runs), and checked that this bin does not
// exceed the threshold bin b* -- so the list holds the whole top-K.  One CTA
// per head reads the list once, coalesced: pairs above b* are selected
// outright, pairs in b* are compacted into shared memory (a global spill past
// its capacity) and the remaining need is met by a CTA radix select on the
// 64-bit value (order-preserving logit key, ~position) with b*'s 11 bits
// known.  Launched as a programmatic dependent of the scan.
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

constexpr int kResThreads = 512;
constexpr int kResCache = 16384;  // threshold-bin candidates in shared memory (128 KiB)

struct ResShared {
  RadixScratch rs;
  int slot;   // selected so far
  int ncand;  // threshold-bin candidates
  int total;
};

// Block-wide exclusive scan of one value per thread; returns the thread's
// offset and writes the block total to *total.  All threads call.
__device__ int block_excl_scan(int v, uint32_t* warp_tot, int* total) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[wid] = (uint32_t)incl;
  __syncthreads();
  if (wid == 0) {
    constexpr int nw = kResThreads / 32;
    const int w = lane < nw ? (int)warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) warp_tot[lane] = (uint32_t)(wi - w);
    if (lane == nw - 1) *total = wi;
  }
  __syncthreads();
  const int off = incl - v + (int)warp_tot[wid];
  __syncthreads();
  return off;
}

__global__ void __launch_bounds__(kResThreads) resolve_kernel(ResolveArgs a) {
  TraceScope trace(a.trace, kTrSelect);
  extern __shared__ __align__(16) uint64_t cache[];
  __shared__ ResShared sh;
  const int tid = threadIdx.x;
  const int bh = blockIdx.x;
  const int b = bh / a.Hq;
  pdl_wait();     // the emitted pairs come from the scan
  pdl_trigger();  // the attention kernel may be scheduled
  trace.mark(1);
  if (a.head_active && a.head_active[bh] != a.active_value) return;

  const int64_t L = seq_len(a.lens, a.len_host, b, a.l_cap);
  const int64_t P = L - window_count(L, a.n_init, a.n_recent);
  const int need = (int)(a.K < P ? a.K : P);
  int32_t* sidx = a.sel_idx + (int64_t)bh * a.K;
  float* sz = a.sel_z + (int64_t)bh * a.K;
  if (need > 0) {
    int64_t n64 = __ldcg(a.dense_n + bh);
    if (n64 > a.dense_stride) n64 = a.dense_stride;
    const int n = (int)n64;
    const uint2* row = a.dense + (int64_t)bh * a.dense_stride;
    uint64_t* spill = a.spill + (int64_t)bh * a.dense_stride;
    const int bstar = __ldcg(a.bstar + bh);  // -1: every emitted pool position is selected
    if (tid == 0) {
      sh.slot = 0;
      sh.ncand = 0;
    }
    __syncthreads();
    constexpr int kU = 8;  // pairs in flight per thread
    int base_sel = 0, base_cand = 0;  // running totals (block-uniform)
    for (int jb = 0; jb < n; jb += kResThreads * kU) {
      uint2 pv[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int j = jb + u * kResThreads + tid;
        pv[u] = j < n ? __ldcg(row + j) : make_uint2(0xffffffffu, 0u);
      }
      uint64_t v[kU];
      uint32_t sel = 0u, cnd = 0u;  // bit masks over the kU pairs
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        v[u] = 0;
        if (pv[u].x != 0xffffffffu) {
          v[u] = rank_key(__uint_as_float(pv[u].y), pv[u].x);
          const int bin = (int)(v[u] >> (64 - kHistBits));
          if (bstar < 0 || bin > bstar) sel |= 1u << u;
          else if (bin == bstar) cnd |= 1u << u;
        }
      }
      // one block scan of (selected << 16 | candidates) per batch
      const int packed = (__popc(sel) << 16) | __popc(cnd);
      const int off = block_excl_scan(packed, sh.rs.warp_tot, &sh.total);
      const int tot = sh.total;
      int s1 = base_sel + (off >> 16), s2 = base_cand + (off & 0xffff);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if ((sel >> u) & 1u) {
          if (s1 < need) {
            sidx[s1] = (int32_t)rank_pos(v[u]);
            sz[s1] = key2f((uint32_t)(v[u] >> 32));
          }
          ++s1;
        } else if ((cnd >> u) & 1u) {
          if (s2 < kResCache) cache[s2] = v[u];
          else if (s2 - kResCache < a.dense_stride) spill[s2 - kResCache] = v[u];
          ++s2;
        }
      }
      base_sel += tot >> 16;
      base_cand += tot & 0xffff;
    }
    if (tid == 0) {
      sh.slot = base_sel;
      sh.ncand = base_cand;
    }
    __syncthreads();
    trace.mark(2);
    const int above = sh.slot < need ? sh.slot : need;
    int nc = sh.ncand;
    if (nc > kResCache + a.dense_stride) nc = (int)(kResCache + a.dense_stride);
    __syncthreads();
    if (bstar >= 0 && above < need) {
      auto val = [&](int j) -> uint64_t {
        return j < kResCache ? cache[j] : __ldcg(spill + (j - kResCache));
      };
      auto emit = [&](uint64_t v) {
        const int s = atomicAdd(&sh.slot, 1);
        if (s < need) {
          sidx[s] = (int32_t)rank_pos(v);
          sz[s] = key2f((uint32_t)(v >> 32));
        }
      };
      const uint64_t prefix = (uint64_t)bstar << (64 - kHistBits);
      const uint64_t mask = (uint64_t)(kHistBins - 1) << (64 - kHistBits);
      cta_radix_select(nc, need - above, prefix, mask, 64 - kHistBits, val, emit, sh.rs);
    }
  }
  for (int64_t j = (need > 0 ? need : 0) + tid; j < a.K; j += kResThreads) {
    sidx[j] = -1;
    sz[j] = -INFINITY;
  }
  if (tid == 0) a.sel_n[bh] = need > 0 ? need : 0;
}

cudaError_t launch_resolve(const ResolveArgs& a, cudaStream_t st) {
  const size_t smem = (size_t)kResCache * sizeof(uint64_t);
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(resolve_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.Hq);
  cfg.blockDim = dim3(kResThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, resolve_kernel, a);
}

}  // namespace tsa
