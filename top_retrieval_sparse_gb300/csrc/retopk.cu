// retopk.cu -- ReTopK reuse path ("Recall Before You Rank: Similarity-Guided
// Top-K Reuse for Efficient Long-Context Attention", method sections 1-5 and
// "GPU Kernel": fused selector, indexed QK, candidate top-K).
//
// selector  (one CTA per (sequence, query head)): qbar = q/|q|; rho_c = qbar . qbar_c over
//           the C cached queries; exact path iff max rho < tau or a refresh
//           step; otherwise the R most similar entries (ties: older entry
//           first), the union of their supports and the last W positions as a
//           bitmap over the cache's positions (in shared memory up to 1.5 M
//           positions, else in the workspace) with a second level in shared
//           memory, compacted in ascending order -> A_t, M_t.
// The indexed QK on A_t, the candidate top-K and the sparse softmax.V are
// the finish kernel's (finish.cu), for reuse heads as for exact ones.
// init      fills the FIFO from the last C prefill queries and their supports.
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

constexpr int kMaxC = 64;

// 1024 threads: the support loads of the union and the compaction's walk
// over the bitmap are latency chains split over the CTA's threads.
constexpr int kSelectorThreads = 1024;

// Supports entries per thread prefetched before the dependency wait (R*K
// beyond kPre * 1024 entries are loaded after it).
constexpr int kPre = 8;

__global__ void __launch_bounds__(kSelectorThreads) retopk_selector_kernel(RetopkSelArgs a) {
  TraceScope trace(a.trace, kTrSelector);  // start, waited, union built, exit
  extern __shared__ __align__(16) uint32_t sbits[];
  __shared__ __align__(16) float qs[kD];
  __shared__ float rho[kMaxC];
  __shared__ float red[kSelectorThreads / 32];
  __shared__ int stab[kMaxC];    // the stable entries' top-R, by rank
  __shared__ int stab_n[kMaxC];  // their support sizes
  __shared__ int s_path, s_fresh_in;
  __shared__ uint32_t wtot[kSelectorThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int bh = blockIdx.x;  // (sequence, query head) of the batch
  const int b = bh / a.Hq, h = bh % a.Hq;
  const RetopkSeq& sq = a.seq[b];
  const int64_t L = sq.L;
  const float* cache_qbar = sq.qbar;
  const int32_t* cache_sup = sq.sup;
  const int32_t* cache_sup_n = sq.sup_n;
  // The FIFO entry the previous step of this sequence wrote (-1: none) may
  // belong to a kernel still running: it is read after the dependency wait.
  // Every other entry was written by a kernel that has completed (the
  // previous kernel of the stream waited for it), so its query, support size
  // and support are read -- and the stable entries' top R chosen -- first.
  const int fresh = sq.fresh;

  // 1. normalise the query
  float x = 0.f;
  if (tid < kD) {
    x = __uint_as_float((uint32_t)a.q[(int64_t)bh * kD + tid] << 16);
    qs[tid] = x;
  }
  float ss = warp_sum(x * x);
  if (lane == 0) red[wid] = ss;
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int w = 0; w < kSelectorThreads / 32; ++w) t += red[w];
    red[0] = t;
  }
  __syncthreads();
  const float nrm = sqrtf(red[0]);
  // the bitmap of step 4: this CTA's shared memory (cleared now), or for a
  // long cache the head's zeroed words in the workspace.  A second level
  // (one bit per bitmap word, always in shared memory) marks the words that
  // hold a bit.
  const int nwords = (int)((L + 31) >> 5);
  const int nl2 = (nwords + 31) >> 5;
  const bool gbm = a.gbitmap != nullptr;
  uint32_t* bitmap = gbm ? a.gbitmap + (int64_t)bh * a.gbitmap_stride : sbits;
  uint32_t* l2 = gbm ? sbits : sbits + nwords;
  for (int w = tid; w < (gbm ? nl2 : nwords + nl2); w += kSelectorThreads) sbits[w] = 0u;
  if (tid < kD) qs[tid] = nrm > 0.f ? qs[tid] / nrm : 0.f;
  __syncthreads();

  // 2. cosine against the cached queries (warp w: entries w and w + 32; all of
  //    a warp's loads are issued before any is used) -- the stable ones now
  constexpr int kPer = kMaxC / (kSelectorThreads / 32);  // entries per warp, at most
  auto cosine = [&](bool fresh_pass) {
    float4 qv[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int c = wid + k * (kSelectorThreads / 32);
      const bool mine = c < a.C && ((c == fresh) == fresh_pass);
      qv[k] = mine ? *reinterpret_cast<const float4*>(cache_qbar + ((int64_t)h * a.C + c) * kD +
                                                      lane * 4)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float4 mq = *reinterpret_cast<const float4*>(qs + lane * 4);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int c = wid + k * (kSelectorThreads / 32);
      float acc = mq.x * qv[k].x;
      acc = fmaf(mq.y, qv[k].y, acc);
      acc = fmaf(mq.z, qv[k].z, acc);
      acc = fmaf(mq.w, qv[k].w, acc);
      acc = warp_sum(acc);
      if (lane == 0 && c < a.C && ((c == fresh) == fresh_pass)) rho[c] = acc;
    }
  };
  cosine(false);
  __syncthreads();
  // the stable entries' top R: a stable entry is taken iff fewer than R stable
  // entries beat it (larger rho, or equal rho and older)
  const int nst = fresh >= 0 ? a.C - 1 : a.C;  // stable entries
  const int Rs = a.R < nst ? a.R : nst;
  if (tid < a.C && tid != fresh) {
    const float rc = rho[tid];
    const int agec = (tid - sq.fifo_head + a.C) % a.C;  // 0 = oldest
    int beat = 0;
    for (int c = 0; c < a.C; ++c) {
      if (c == fresh) continue;
      const float r = rho[c];
      const int age = (c - sq.fifo_head + a.C) % a.C;
      beat += (r > rc || (r == rc && age < agec)) ? 1 : 0;
    }
    if (beat < Rs) {  // ranks are distinct: one entry per rank
      stab[beat] = tid;
      stab_n[beat] = cache_sup_n[(int64_t)h * a.C + tid];
    }
  }
  __syncthreads();
  // their supports as one flat index space of Rs*K entries (entries past a
  // support's size are -1), in registers
  int32_t pre[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int j = tid + u * kSelectorThreads;
    pre[u] = -1;
    if (j < Rs * a.K) {
      const int r = j / a.K, i = j - r * a.K;
      if (i < stab_n[r]) pre[u] = cache_sup[((int64_t)h * a.C + stab[r]) * a.K + i];
    }
  }

  // the cache and this step's buffers belong to the previous step's kernels
  // until they have completed; the key scan may be scheduled from here on
  pdl_wait();
  pdl_trigger();
  trace.mark(1);
  if (h == 0 && tid == 0) {  // this step's length and FIFO entry, for the next kernels
    a.lens_ws[b] = (int32_t)L;
    a.seq_ws[b] = sq;
  }
  if (tid < kD) a.qbar_new[(int64_t)bh * kD + tid] = qs[tid];
  // the fresh entry's support size and first kSelectorThreads entries,
  // requested with its query: the newest query is usually the most similar,
  // and its support is then part of the union
  int fsn = 0;
  int32_t fsup0 = -1;
  if (fresh >= 0) {
    fsn = cache_sup_n[(int64_t)h * a.C + fresh];
    if (tid < a.K) fsup0 = cache_sup[((int64_t)h * a.C + fresh) * a.K + tid];
  }
  if (fresh >= 0) cosine(true);
  __syncthreads();

  // 3. fallback / refresh decision; the final top R: the fresh entry is in
  //    iff fewer than R entries beat it, and then it displaces the stable R-th
  if (wid == 0) {
    float mx = -INFINITY;
    int nb = 0;  // stable entries that beat the fresh one
    const float rf = fresh >= 0 ? rho[fresh] : 0.f;
    const int agef = fresh >= 0 ? (fresh - sq.fifo_head + a.C) % a.C : 0;
    for (int c = lane; c < a.C; c += 32) {
      mx = fmaxf(mx, rho[c]);
      const int age = (c - sq.fifo_head + a.C) % a.C;
      if (fresh >= 0 && c != fresh && (rho[c] > rf || (rho[c] == rf && age < agef))) ++nb;
    }
    mx = warp_max(mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) nb += __shfl_xor_sync(0xffffffffu, nb, o);
    const int path = (mx < a.tau || sq.refresh) ? 1 : 0;
    if (lane == 0) {
      s_path = path;
      a.path[bh] = path;
      if (a.path_out) a.path_out[bh] = path;
      s_fresh_in = fresh >= 0 && nb < a.R ? 1 : 0;
    }
  }
  __syncthreads();
  uint32_t* crow = a.cand + (int64_t)bh * a.cand_cap;
  if (s_path) {
    if (tid == 0) {
      a.mcand[bh] = 0;
      if (a.mcand_out) a.mcand_out[bh] = (int32_t)L;
    }
    if (a.cand_out)
      for (int j = tid; j < a.cand_cap; j += kSelectorThreads)
        a.cand_out[(int64_t)bh * a.cand_cap + j] = -1;
    return;
  }

  // 4. bitmap union of the recalled supports and the recent window
  const int fin = s_fresh_in;
  const int keep = fin && Rs == a.R ? Rs - 1 : Rs;  // stable supports kept
  auto mark = [&](int32_t p) {
    if (p >= 0 && p < L) {
      atomicOr(&bitmap[p >> 5], 1u << (p & 31));
      atomicOr(&l2[p >> 10], 1u << ((p >> 5) & 31));
    }
  };
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int j = tid + u * kSelectorThreads;
    if (j < keep * a.K) mark(pre[u]);
  }
  for (int j = kPre * kSelectorThreads + tid; j < keep * a.K; j += kSelectorThreads) {
    const int r = j / a.K, i = j - r * a.K;  // past the prefetched entries
    if (i < stab_n[r]) mark(cache_sup[((int64_t)h * a.C + stab[r]) * a.K + i]);
  }
  if (fin)
    for (int i = tid; i < fsn && i < a.K; i += kSelectorThreads)
      mark(i == tid ? fsup0 : cache_sup[((int64_t)h * a.C + fresh) * a.K + i]);
  const int64_t lo = L - a.W > 0 ? L - a.W : 0;
  for (int64_t p = lo + tid; p < L; p += kSelectorThreads) mark((int32_t)p);
  __syncthreads();
  trace.mark(2);

  // 5. ascending compaction: each thread owns a contiguous range of bitmap
  // words (of second-level words when the bitmap is in the workspace: only
  // the words they mark are read, and cleared), counts their bits, and after
  // one block scan writes its positions in order.
  const int nunits = gbm ? nl2 : nwords;
  const int per = (nunits + kSelectorThreads - 1) / kSelectorThreads;
  const int q0 = tid * per;
  const int q1 = q0 + per < nunits ? q0 + per : nunits;
  uint32_t cnt = 0;
  if (gbm) {
    for (int q = q0; q < q1; ++q)
      for (uint32_t m = l2[q]; m; m &= m - 1) cnt += __popc(bitmap[(q << 5) + __ffs(m) - 1]);
  } else {
    for (int q = q0; q < q1; ++q) cnt += __popc(bitmap[q]);
  }
  uint32_t incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wtot[wid] = incl;
  __syncthreads();
  if (wid == 0) {  // exclusive scan of the warp totals
    const uint32_t t = wtot[lane];
    uint32_t inc = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += y;
    }
    wtot[lane] = inc - t;
    if (lane == 31) {
      a.mcand[bh] = (int32_t)inc;
      if (a.mcand_out) a.mcand_out[bh] = (int32_t)inc;
    }
  }
  __syncthreads();
  uint32_t pos = incl - cnt + wtot[wid];
  auto emit_word = [&](int w) {
    const uint32_t word = bitmap[w];
    if (gbm) bitmap[w] = 0u;  // the workspace bitmap is all zero again after the step
    for (uint32_t bits = word; bits; bits &= bits - 1) {
      if (pos < (uint32_t)a.cand_cap) crow[pos] = ((uint32_t)w << 5) + __ffs(bits) - 1;
      ++pos;
    }
  };
  if (gbm) {
    for (int q = q0; q < q1; ++q)
      for (uint32_t m = l2[q]; m; m &= m - 1) emit_word((q << 5) + __ffs(m) - 1);
  } else {
    for (int q = q0; q < q1; ++q) emit_word(q);
  }
  if (a.cand_out) {
    __syncthreads();
    const int m = a.mcand[bh];
    for (int j = tid; j < a.cand_cap; j += kSelectorThreads)
      a.cand_out[(int64_t)bh * a.cand_cap + j] = j < m ? (int32_t)crow[j] : -1;
  }
}

cudaError_t launch_retopk_selector(const RetopkSelArgs& a, size_t smem, cudaStream_t st) {
  static size_t configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev < 64 && configured[dev] < smem) {
    cudaError_t e = cudaFuncSetAttribute(retopk_selector_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured[dev] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n * a.Hq);
  cfg.blockDim = dim3(kSelectorThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, retopk_selector_kernel, a);
}

__global__ void retopk_init_kernel(RetopkInitArgs a) {
  __shared__ float red[kD / 32];
  const int c = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int64_t src = (int64_t)c * a.Hq + h;
  const float x = __uint_as_float((uint32_t)a.prefill_q[src * kD + tid] << 16);
  const float ss = warp_sum(x * x);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  const float nrm = sqrtf(red[0] + red[1] + red[2] + red[3]);
  const int64_t hc = (int64_t)h * a.C + c;
  a.cache_qbar[hc * kD + tid] = nrm > 0.f ? x / nrm : 0.f;
  int n = a.prefill_n[src];
  n = n < 0 ? 0 : (n > a.K ? a.K : n);
  for (int j = tid; j < a.K; j += kD)
    a.cache_sup[hc * a.K + j] = j < n ? a.prefill_sup[src * a.K + j] : -1;
  if (tid == 0) a.cache_sup_n[hc] = n;
}

cudaError_t launch_retopk_init(const RetopkInitArgs& a, cudaStream_t st) {
  dim3 grid(a.C, a.Hq);
  retopk_init_kernel<<<grid, kD, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace tsa
