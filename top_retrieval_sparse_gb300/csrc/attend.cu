// attend.cu -- softmax.V over the static window and the selected set, and the
// gamma1/gamma2 log-sum-exp merge.
//
// "RetrievalAttention" Eq. 3 (o_W with local max z~1, o_Omega with local max
// z~2) and Eq. 4-5 (o_t = g1 o_W + g2 o_Omega, g_j = e^(z~j - z~) l_j / sum).
// ReTopK: sparse softmax-V over S_t and the query-support cache push.
//
// One grid row per (sequence, query head); each CTA owns a split of 64 rows
// (window splits first, then selected splits).  A warp gathers 16 rows of V
// (256-byte rows, 8 bytes per lane, all loads issued before use) and keeps
// (m, l, o) with its own max, in base 2 (logits times log2 e, weights by
// exp2); the CTA combines its warps and writes the split partial.  The last CTA of the row (ticket) merges the window splits
// into (o_W, z~1, l_W), the selected splits into (o_Omega, z~2, l_Omega),
// applies Eq. 4-5 and, on a ReTopK step, pushes (qbar, S_t) into the FIFO.
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

constexpr int kAttThreads = 128;
constexpr int kAttWarps = kAttThreads / 32;
constexpr int kSplitRows = 64;
constexpr int kRowsPerWarp = kSplitRows / kAttWarps;  // 16
constexpr int kPartStride = kD + 2;                   // o[128], m, l
constexpr int kMaxSplits = 1024;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttShared {
  float wm[kAttWarps];
  float wl[kAttWarps];
  float wo[kAttWarps][kD];
  float sw[kMaxSplits];  // per-split merge weights (last CTA)
  float sm[kMaxSplits];  // per-split maxima
  float sl[kMaxSplits];  // per-split sums
  int last;
};

__global__ void __launch_bounds__(kAttThreads) attend_kernel(AttendArgs a) {
  TraceScope trace(a.trace, kTrAttend);
  __shared__ AttShared sh;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int bh = blockIdx.y;
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int g = h / (a.Hq / a.kv.Hkv);
  const int s = blockIdx.x;
  const int nsplit = a.n_wsplit + a.n_ssplit;
  const int64_t L = seq_len(a.lens, a.len_host, b, a.kv.l_cap);

  // ---- rows of this split ----
  const bool is_win = s < a.n_wsplit;
  // window splits read only the scan's logits: with early_window they run
  // before the selection kernel (the programmatic predecessor) has finished
  if (!(is_win && a.early_window)) pdl_wait();
  int64_t nrows;
  int64_t j0;
  if (is_win) {
    nrows = window_count(L, a.n_init, a.n_recent);
    j0 = (int64_t)s * kSplitRows;
  } else {
    nrows = a.sel_n[bh];
    j0 = (int64_t)(s - a.n_wsplit) * kSplitRows;
  }
  const int64_t jw = j0 + wid * kRowsPerWarp;  // this warp's first row
  // logits are carried in base 2 (z * log2 e) so each weight is one exp2
  float z = -INFINITY;
  int64_t pos = 0;
  if (lane < kRowsPerWarp && jw + lane < nrows) {
    const int64_t j = jw + lane;
    if (is_win) {
      pos = window_pos(j, L, a.n_init, a.n_recent);
      z = __ldcg(a.wz + (int64_t)bh * a.wz_stride + j);
    } else {
      pos = a.sel_idx[(int64_t)bh * a.K + j];
      z = a.sel_z[(int64_t)bh * a.K + j];
    }
    z *= kLog2e;
  }
  const float m = warp_max(z);
  float l = 0.f;
  float o[4] = {0.f, 0.f, 0.f, 0.f};
  if (m != -INFINITY) {
    const uint16_t* vbase = a.kv.page_table ? a.kv.v : a.kv.v + kv_row(a.kv, b, g, 0);
    uint2 vv[kRowsPerWarp];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const int pk = __shfl_sync(0xffffffffu, (int)pos, k);
      const bool valid = jw + k < nrows;
      const uint16_t* row = a.kv.page_table ? vbase + kv_row(a.kv, b, g, pk)
                                            : vbase + (int64_t)pk * kD;
      vv[k] = valid ? __ldg(reinterpret_cast<const uint2*>(row + lane * 4)) : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
      const float zk = __shfl_sync(0xffffffffu, z, k);
      const float p = (jw + k < nrows) ? exp2f(zk - m) : 0.f;
      l += p;
      o[0] = fmaf(p, bf_lo(vv[k].x), o[0]);
      o[1] = fmaf(p, bf_hi(vv[k].x), o[1]);
      o[2] = fmaf(p, bf_lo(vv[k].y), o[2]);
      o[3] = fmaf(p, bf_hi(vv[k].y), o[3]);
    }
  }
  if (lane == 0) {
    sh.wm[wid] = m;
    sh.wl[wid] = l;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) sh.wo[wid][lane * 4 + e] = o[e];
  __syncthreads();

  // ---- combine warps -> split partial (o unnormalised w.r.t. its max) ----
  {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttWarps; ++w) M = fmaxf(M, sh.wm[w]);
    float acc = 0.f, lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttWarps; ++w) {
        if (sh.wm[w] == -INFINITY) continue;
        const float e = exp2f(sh.wm[w] - M);
        acc = fmaf(e, sh.wo[w][tid], acc);
        lsum = fmaf(e, sh.wl[w], lsum);
      }
    }
    float* pp = a.part + ((int64_t)bh * nsplit + s) * kPartStride;
    pp[tid] = acc;
    if (tid == 0) {
      pp[kD] = M;
      pp[kD + 1] = lsum;
    }
  }

  // ---- last CTA of the row merges (Eq. 4-5) ----
  trace.mark(1);
  if (is_win && a.early_window) pdl_wait();
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const uint32_t t = atomicAdd(&a.ticket[bh], 1u);
    sh.last = (t == (uint32_t)nsplit - 1);
  }
  __syncthreads();
  if (!sh.last) return;
  __threadfence();
  trace.mark(2);

  const float* part = a.part + (int64_t)bh * nsplit * kPartStride;
  // split maxima and sums, loaded in parallel (L2: written by other CTAs)
  for (int i = tid; i < nsplit; i += kAttThreads) {
    sh.sm[i] = __ldcg(part + (int64_t)i * kPartStride + kD);
    sh.sl[i] = __ldcg(part + (int64_t)i * kPartStride + kD + 1);
  }
  __syncthreads();
  // z~1 (window) and z~2 (selected): maxima of the split maxima
  float z1 = -INFINITY, z2 = -INFINITY;
  for (int i = 0; i < a.n_wsplit; ++i) z1 = fmaxf(z1, sh.sm[i]);
  for (int i = a.n_wsplit; i < nsplit; ++i) z2 = fmaxf(z2, sh.sm[i]);
  // per-split rescale to its set's max
  for (int i = tid; i < nsplit; i += kAttThreads) {
    const float mi = sh.sm[i];
    const float zref = i < a.n_wsplit ? z1 : z2;
    sh.sw[i] = mi == -INFINITY ? 0.f : exp2f(mi - zref);
  }
  __syncthreads();
  float lW = 0.f, lO = 0.f, oW = 0.f, oO = 0.f;
  for (int i = 0; i < a.n_wsplit; ++i) {
    const float w = sh.sw[i];
    lW = fmaf(w, sh.sl[i], lW);
    oW = fmaf(w, __ldcg(part + (int64_t)i * kPartStride + tid), oW);
  }
  for (int i = a.n_wsplit; i < nsplit; ++i) {
    const float w = sh.sw[i];
    lO = fmaf(w, sh.sl[i], lO);
    oO = fmaf(w, __ldcg(part + (int64_t)i * kPartStride + tid), oO);
  }
  // gamma merge: z~ = max(z~1, z~2); den = sum over W u Omega of e^(z - z~)
  float outv = 0.f, lse = -INFINITY;
  const bool eW = !(lW > 0.f), eO = !(lO > 0.f);
  if (!(eW && eO)) {
    const float zt = eW ? z2 : (eO ? z1 : fmaxf(z1, z2));
    const float aW = eW ? 0.f : exp2f(z1 - zt);
    const float aO = eO ? 0.f : exp2f(z2 - zt);
    const float den = aW * lW + aO * lO;
    // g1 o_W + g2 o_Omega with o_W = oW / lW, g1 = aW lW / den (same for Omega)
    outv = (aW * oW + aO * oO) / den;
    lse = (zt + log2f(den)) * kLn2;  // back to natural log
  }
  a.out[(int64_t)bh * kD + tid] = outv;
  if (tid == 0 && a.lse_out) a.lse_out[bh] = lse;

  if (a.push_qbar) {  // ReTopK: push (qbar_t, S_t) over the oldest FIFO entry
    const int64_t hc = (int64_t)h * a.C + a.slot;
    a.cache_qbar[hc * kD + tid] = a.push_qbar[(int64_t)h * kD + tid];
    const int n = a.sel_n[bh];
    for (int j = tid; j < a.K; j += kAttThreads)
      a.cache_sup[hc * a.K + j] = j < n ? a.sel_idx[(int64_t)bh * a.K + j] : -1;
    if (tid == 0) a.cache_sup_n[hc] = n;
  }
  if (tid == 0) a.ticket[bh] = 0;
}

cudaError_t launch_attend(const AttendArgs& a, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_wsplit + a.n_ssplit, a.B * a.Hq);
  cfg.blockDim = dim3(kAttThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attend_kernel, a);
}

int attend_split_rows() { return kSplitRows; }
int attend_max_splits() { return kMaxSplits; }

// ----------------------------------------------------------- lse_merge
// Eq. 4-5 on precomputed (o, lse) partials.  One CTA per row: every thread
// reads the row's lse values before the barrier and writes after it, so the
// outputs may alias the inputs.
__global__ void lse_merge_kernel(const float* oa, const float* la, const float* ob,
                                 const float* lb, float* oo, float* lo, int d) {
  const int64_t r = blockIdx.x;
  const float xa = la[r], xb = lb[r];
  const bool ea = xa == -INFINITY, eb = xb == -INFINITY;
  float wa = 0.f, wb = 0.f, lse = -INFINITY, inv = 0.f;
  if (!(ea && eb)) {
    const float zt = ea ? xb : (eb ? xa : fmaxf(xa, xb));
    wa = ea ? 0.f : expf(xa - zt);
    wb = eb ? 0.f : expf(xb - zt);
    const float den = wa + wb;
    inv = 1.f / den;
    lse = zt + logf(den);
  }
  __syncthreads();
  for (int j = threadIdx.x; j < d; j += blockDim.x) {
    const int64_t e = r * d + j;
    oo[e] = (ea && eb) ? 0.f : (wa * oa[e] + wb * ob[e]) * inv;
  }
  if (threadIdx.x == 0) lo[r] = lse;
}

cudaError_t launch_lse_merge(const float* oa, const float* la, const float* ob,
                             const float* lb, float* oo, float* lo, int rows, int d,
                             cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  int th = ((d + 31) / 32) * 32;
  if (th > 1024) th = 1024;
  lse_merge_kernel<<<rows, th, 0, st>>>(oa, la, ob, lb, oo, lo, d);
  return cudaGetLastError();
}

}  // namespace tsa
