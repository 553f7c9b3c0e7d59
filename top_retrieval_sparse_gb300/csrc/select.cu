// select.cu -- exact top-K of the logits outside the static window.
//
// "RetrievalAttention" Eq. 2 (the selected set I, top-k by inner product,
// Flat baseline) with W and Omega disjoint (Eq. 3); ReTopK's exact path
// S_t = TopK(e, K).  Ties go to the smaller position.
//
// Two-pass multi-CTA radix select on the order-preserving fp32 key:
//   pass 1 (fused into the key scan): 11-bit histogram per head, turned into
//   the threshold bin b* (largest bin whose suffix count reaches `need`) by
//   the scan CTA that completes the head's KV unit;
//   this kernel, one grid row per head, many CTAs per row (launched as a
//   programmatic dependent of the scan):
//     - streams its chunk of logits once (16-byte loads, held in registers):
//       positions above b* are selected outright, positions in b* become
//       candidates; slots come from one block scan and one atomic per CTA,
//     - the last CTA of the row (ticket) resolves the candidates exactly with
//       a CTA radix select on the 64-bit (key, ~position) value, shared-memory
//       resident when they fit, and pads the outputs.
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

constexpr int kSelThreads = 256;
constexpr int kSelPer = 32;                          // positions per thread
constexpr int kSelChunk = kSelThreads * kSelPer;     // positions per CTA (8192)
constexpr int kCandSmem = 4096;                      // candidates cached in shared memory

struct SelShared {
  RadixScratch rs;
  int last;
  int slot;
  int base_take;
  int base_cand;
};

__global__ void __launch_bounds__(kSelThreads) select_kernel(SelectArgs a) {
  TraceScope trace(a.trace, kTrSelect);
  extern __shared__ __align__(16) uint64_t cand_cache[];
  __shared__ SelShared sh;
  const int tid = threadIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / a.Hq;
  pdl_wait();     // logits and threshold bins come from the key scan
  pdl_trigger();  // let the attention kernel start its window splits
  if (a.head_active && a.head_active[bh] != a.active_value) return;

  const int64_t L = seq_len(a.lens, a.len_host, b, a.l_cap);
  const int64_t P = L - window_count(L, a.n_init, a.n_recent);
  const int64_t need = a.K < P ? a.K : P;
  const bool all_in = need == P;  // every pool position is selected (incl. P = 0)
  const uint32_t bstar = all_in ? 0u : (uint32_t)__ldcg(a.bstar + bh);

  // ---- filter this CTA's chunk: values in registers, one atomic per CTA ----
  const float* zrow = a.scores + (int64_t)bh * a.score_stride;
  int32_t* sidx = a.sel_idx + (int64_t)bh * a.K;
  float* sz = a.sel_z + (int64_t)bh * a.K;
  uint32_t* crow = a.cand + (int64_t)bh * a.score_stride;
  const int64_t c0 = (int64_t)blockIdx.x * kSelChunk;
  const int64_t c1 = c0 + kSelChunk < L ? c0 + kSelChunk : L;
  if (need > 0 && c0 < c1) {
    float zz[kSelPer];
    uint32_t take = 0u, maybe = 0u;
#pragma unroll
    for (int k = 0; k < kSelPer / 4; ++k) {
      const int64_t i0 = c0 + 4 * (tid + (int64_t)k * kSelThreads);
      if (i0 + 3 < c1) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(zrow + i0));
        zz[4 * k] = f.x; zz[4 * k + 1] = f.y; zz[4 * k + 2] = f.z; zz[4 * k + 3] = f.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) zz[4 * k + e] = i0 + e < c1 ? zrow[i0 + e] : 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < kSelPer / 4; ++k) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int64_t i = c0 + 4 * (tid + (int64_t)k * kSelThreads) + e;
        const bool valid = i < c1 && !in_window(i, L, a.n_init, a.n_recent);
        const uint32_t bin = f2key(zz[4 * k + e]) >> kHistShift;
        if (valid && (all_in || bin > bstar)) take |= 1u << (4 * k + e);
        else if (valid && bin == bstar) maybe |= 1u << (4 * k + e);
      }
    }
    // block exclusive scan of (takes << 16 | candidates)
    const uint32_t mine = ((uint32_t)__popc(take) << 16) | (uint32_t)__popc(maybe);
    const int lane = tid & 31, wid = tid >> 5;
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.rs.warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const uint32_t w = lane < kSelThreads / 32 ? sh.rs.warp_tot[lane] : 0u;
      uint32_t wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      if (lane < kSelThreads / 32) sh.rs.warp_tot[lane] = wi - w;
      if (lane == kSelThreads / 32 - 1) {  // CTA totals -> one atomic per counter
        sh.base_take = (wi >> 16) ? atomicAdd(&a.sel_n[bh], (int)(wi >> 16)) : 0;
        sh.base_cand = (wi & 0xffffu) ? atomicAdd(&a.cand_n[bh], (int)(wi & 0xffffu)) : 0;
      }
    }
    __syncthreads();
    const uint32_t excl = incl - mine + sh.rs.warp_tot[wid];
    int st = sh.base_take + (int)(excl >> 16);
    int sc = sh.base_cand + (int)(excl & 0xffffu);
#pragma unroll
    for (int k = 0; k < kSelPer / 4; ++k) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int bit = 4 * k + e;
        const int64_t i = c0 + 4 * (tid + (int64_t)k * kSelThreads) + e;
        if ((take >> bit) & 1u) {
          if (st < need) {  // bound holds by construction; guarded anyway
            sidx[st] = (int32_t)i;
            sz[st] = zz[bit];
          }
          ++st;
        } else if ((maybe >> bit) & 1u) {
          if (sc < L) crow[sc] = (uint32_t)i;
          ++sc;
        }
      }
    }
  }

  // ---- last CTA of this head resolves the threshold bin ----
  trace.mark(1);
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t t = atomicAdd(&a.ticket[bh], 1u);
    sh.last = (t == gridDim.x - 1);
  }
  __syncthreads();
  if (!sh.last) return;
  __threadfence();
  trace.mark(2);

  int n_above = __ldcg(&a.sel_n[bh]);
  int n_c = __ldcg(&a.cand_n[bh]);
  if (n_above > need) n_above = (int)need;
  if (n_c > L) n_c = (int)L;
  const int need_c = (int)need - n_above;
  if (tid == 0) sh.slot = n_above;
  __syncthreads();
  if (need_c > 0) {
    const bool in_smem = n_c <= kCandSmem;
    if (in_smem)
      for (int j = tid; j < n_c; j += kSelThreads) {
        const uint32_t p = __ldcg(crow + j);
        cand_cache[j] = rank_key(zrow[p], p);
      }
    __syncthreads();
    auto val = [&](int j) -> uint64_t {
      if (in_smem) return cand_cache[j];
      const uint32_t p = __ldcg(crow + j);
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

int select_chunk() { return kSelChunk; }

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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(chunks, a.B * a.Hq);
  cfg.blockDim = dim3(kSelThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, select_kernel, a);
}

}  // namespace tsa
