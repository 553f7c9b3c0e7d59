// select.cu -- exact top-K of the logits outside the static window.
//
// "RetrievalAttention" Eq. 2 (the selected set I, top-k by inner product,
// Flat baseline) with W and Omega disjoint (Eq. 3); ReTopK's exact path
// S_t = TopK(e, K).  Ties go to the smaller position.
//
// Two-pass multi-CTA radix select on the order-preserving fp32 key:
//   pass 1 (fused into the key scan): 11-bit histogram per head;
//   this kernel, one grid row per head, many CTAs per row:
//     - every CTA finds the threshold bin b* (largest bin whose suffix count
//       reaches `need`) from the histogram,
//     - streams its chunk of logits once (16-byte loads): positions above b*
//       are selected outright, positions in b* become candidates (warp-
//       aggregated slot reservation),
//     - the last CTA of the row (ticket) resolves the candidates exactly with
//       a CTA radix select on the 64-bit (key, ~position) value, shared-memory
//       resident when they fit, and pads the outputs.
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

constexpr int kSelThreads = 512;
constexpr int kCandSmem = 8192;  // candidates cached in shared memory

struct SelShared {
  RadixScratch rs;
  uint32_t bins[kHistBins];
  int bstar;
  int above;
  int last;
  int slot;
};

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a) {
  extern __shared__ __align__(16) uint64_t cand_cache[];
  __shared__ SelShared sh;
  const int tid = threadIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / a.Hq;
  if (a.head_active && a.head_active[bh] != a.active_value) return;

  const int64_t L = seq_len(a.lens, a.len_host, b, a.l_cap);
  const int64_t P = L - window_count(L, a.n_init, a.n_recent);
  const int64_t need = a.K < P ? a.K : P;
  const bool all_in = need == P;  // every pool position is selected (incl. P = 0)

  // ---- threshold bin from the pass-1 histogram ----
  if (!all_in) {
    const uint32_t* hh = a.hist + (int64_t)bh * kHistBins;
    for (int i = tid; i < kHistBins; i += kSelThreads) sh.bins[i] = hh[i];
    __syncthreads();
    // suffix search: 512 threads x 4 bins from the top
    constexpr int per = kHistBins / kSelThreads;
    uint32_t mine = 0;
#pragma unroll
    for (int r = 0; r < per; ++r) mine += sh.bins[kHistBins - 1 - (tid * per + r)];
    uint32_t incl = mine;
    const int lane = tid & 31, wid = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.rs.warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const uint32_t w = lane < kSelThreads / 32 ? sh.rs.warp_tot[lane] : 0;
      uint32_t wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      if (lane < kSelThreads / 32) sh.rs.warp_tot[lane] = wi - w;
    }
    __syncthreads();
    const uint32_t excl = incl - mine + sh.rs.warp_tot[wid];
    if (excl < (uint32_t)need && excl + mine >= (uint32_t)need) {
      uint32_t acc = excl;
      for (int r = 0; r < per; ++r) {
        const int bin = kHistBins - 1 - (tid * per + r);
        const uint32_t c = sh.bins[bin];
        if (acc + c >= (uint32_t)need) {
          sh.bstar = bin;
          sh.above = (int)acc;
          break;
        }
        acc += c;
      }
    }
    __syncthreads();
  }
  const uint32_t bstar = all_in ? 0u : (uint32_t)sh.bstar;

  // ---- filter this CTA's chunk ----
  const float* zrow = a.scores + (int64_t)bh * a.score_stride;
  int32_t* sidx = a.sel_idx + (int64_t)bh * a.K;
  float* sz = a.sel_z + (int64_t)bh * a.K;
  uint32_t* crow = a.cand + (int64_t)bh * a.score_stride;
  const int64_t c0 = (int64_t)blockIdx.x * a.chunk;
  const int64_t c1 = c0 + a.chunk < L ? c0 + a.chunk : L;
  if (need > 0) {
    for (int64_t base = c0; base < c1; base += 4 * kSelThreads) {
      const int64_t i0 = base + 4 * tid;
      float zz[4] = {0.f, 0.f, 0.f, 0.f};
      if (i0 + 3 < c1) {
        const float4 f = *reinterpret_cast<const float4*>(zrow + i0);
        zz[0] = f.x; zz[1] = f.y; zz[2] = f.z; zz[3] = f.w;
      } else {
        for (int e = 0; e < 4; ++e)
          if (i0 + e < c1) zz[e] = zrow[i0 + e];
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t i = i0 + e;
        const bool valid = i < c1 && !in_window(i, L, a.n_init, a.n_recent);
        const uint32_t bin = f2key(zz[e]) >> kHistShift;
        const bool take = valid && (all_in || bin > bstar);
        const bool maybe = valid && !all_in && bin == bstar;
        const int s1 = warp_reserve(take, &a.sel_n[bh]);
        if (take && s1 < need) {  // bound holds by construction; guarded anyway
          sidx[s1] = (int32_t)i;
          sz[s1] = zz[e];
        }
        const int s2 = warp_reserve(maybe, &a.cand_n[bh]);
        if (maybe && s2 < L) crow[s2] = (uint32_t)i;
      }
    }
  }

  // ---- last CTA of this head resolves the threshold bin ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t t = atomicAdd(&a.ticket[bh], 1u);
    sh.last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (!sh.last) return;
  __threadfence();

  int n_above = *((volatile int32_t*)&a.sel_n[bh]);
  int n_c = *((volatile int32_t*)&a.cand_n[bh]);
  if (n_above > need) n_above = (int)need;
  if (n_c > L) n_c = (int)L;
  const int need_c = (int)need - n_above;
  if (tid == 0) sh.slot = n_above;
  __syncthreads();
  if (need_c > 0) {
    const bool in_smem = n_c <= kCandSmem;
    if (in_smem)
      for (int j = tid; j < n_c; j += kSelThreads) {
        const uint32_t p = ((volatile uint32_t*)crow)[j];
        cand_cache[j] = rank_key(zrow[p], p);
      }
    __syncthreads();
    auto val = [&](int j) -> uint64_t {
      if (in_smem) return cand_cache[j];
      const uint32_t p = ((volatile uint32_t*)crow)[j];
      return rank_key(zrow[p], p);
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
    cta_radix_select(n_c, need_c, prefix, mask, 64 - kHistBits, val, emit, sh.rs);
  }
  for (int64_t j = need + tid; j < a.K; j += kSelThreads) {
    sidx[j] = -1;
    sz[j] = -INFINITY;
  }
  if (tid == 0) {
    a.sel_n[bh] = (int32_t)need;
    a.ticket[bh] = 0;
  }
}

cudaError_t launch_select(const SelectArgs& a, int chunks, cudaStream_t st) {
  const size_t smem = (size_t)kCandSmem * sizeof(uint64_t);
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(select_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  dim3 grid(chunks, a.B * a.Hq);
  select_kernel<<<grid, kSelThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tsa
