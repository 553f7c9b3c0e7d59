// resolve.cu -- exact top-K from the pairs the key scan emitted.
//
// "RetrievalAttention" Eq. 2 (the selected set, top-k by inner product as in
// the Flat baseline) with W and Omega disjoint (Eq. 3); ReTopK's exact path
// S_t = TopK(e, K).  Ties go to the smaller position.
//
// The scan emitted, for every head, the (position, logit) pairs of all pool
// positions whose radix bin is at least its emission bin, and checked that
// this bin does not exceed the threshold bin b* -- so the emitted pairs hold
// the whole top-K.  One CTA per head keeps the min(K, |pool|) largest by the
// 64-bit value (order-preserving logit key, ~position) with a CTA radix
// select over the pairs, held in shared memory when they fit.  Launched as a
// programmatic dependent of the scan.
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

constexpr int kResThreads = 512;
constexpr int kResCache = 12288;  // pairs cached in shared memory (96 KiB)

struct ResShared {
  RadixScratch rs;
  int slot;
};

__global__ void __launch_bounds__(kResThreads) resolve_kernel(ResolveArgs a) {
  TraceScope trace(a.trace, kTrSelect);
  extern __shared__ __align__(16) uint64_t cache[];
  __shared__ ResShared sh;
  const int tid = threadIdx.x;
  const int bh = blockIdx.x;
  const int b = bh / a.Hq;
  pdl_wait();     // the emitted pairs and counts come from the scan
  pdl_trigger();  // let the attention kernel start its window splits
  if (a.head_active && a.head_active[bh] != a.active_value) return;

  const int64_t L = seq_len(a.lens, a.len_host, b, a.l_cap);
  const int64_t P = L - window_count(L, a.n_init, a.n_recent);
  const int need = (int)(a.K < P ? a.K : P);
  int32_t* sidx = a.sel_idx + (int64_t)bh * a.K;
  float* sz = a.sel_z + (int64_t)bh * a.K;
  if (need > 0) {
    int64_t n64 = __ldcg(a.emit_n + bh);
    if (n64 > a.cand_stride) n64 = a.cand_stride;
    const int n = (int)n64;
    const uint2* row = a.cand + (int64_t)bh * a.cand_stride;
    const bool in_smem = n <= kResCache;
    if (in_smem)
      for (int j = tid; j < n; j += kResThreads) {
        const uint2 p = __ldcg(row + j);
        cache[j] = rank_key(__uint_as_float(p.y), p.x);
      }
    if (tid == 0) sh.slot = 0;
    __syncthreads();
    trace.mark(1);
    auto val = [&](int j) -> uint64_t {
      if (in_smem) return cache[j];
      const uint2 p = __ldcg(row + j);
      return rank_key(__uint_as_float(p.y), p.x);
    };
    auto emit = [&](uint64_t v) {
      const int s = atomicAdd(&sh.slot, 1);
      if (s < need) {
        sidx[s] = (int32_t)rank_pos(v);
        sz[s] = key2f((uint32_t)(v >> 32));
      }
    };
    cta_radix_select(n, need, 0ull, 0ull, 64, val, emit, sh.rs);
    trace.mark(2);
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
