// attend.cu -- softmax.V over the static window and the selected set, and the
// gamma1/gamma2 log-sum-exp merge.
//
// "RetrievalAttention" Eq. 3 (o_W with local max z~1, o_Omega with local max
// z~2) and Eq. 4-5 (o_t = g1 o_W + g2 o_Omega, g_j = e^(z~j - z~) l_j / sum).
// ReTopK: sparse softmax-V over S_t and the query-support cache push.
//
// One thread-block cluster of 8 CTAs per (sequence, query head).  The
// head's rows -- window positions first, then the selected ones -- are split
// evenly over the 8 CTAs and, within a CTA, over 8 warps.  A warp takes its
// rows 32 at a time: one round of (position, logit) loads, then all 32 V rows
// (256-byte rows, 8 bytes per lane) in flight before any is used; it keeps
// running (max, sum, o) separately for the window and the selected rows, in
// base 2 (logits times log2 e, weights by exp2).  Each CTA
// combines its warps in shared memory; after a cluster barrier the rank-0 CTA
// reads the 8 CTA partials through distributed shared memory, forms
// (o_W, z~1, l_W) and (o_Omega, z~2, l_Omega), applies Eq. 4-5 and, on a
// ReTopK step, pushes (qbar, S_t) into the FIFO.  A second cluster barrier
// keeps every CTA's shared memory alive until rank 0 has read it.  Launched
// as a programmatic dependent of the top-K kernel.
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

constexpr int kAttCluster = 8;                 // CTAs per head
constexpr int kAttWarps = 8;
constexpr int kAttThreads = 32 * kAttWarps;
constexpr int kBatch = 16;                     // rows in flight per warp
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttPart {                               // [0] window rows, [1] selected rows
  float m[2], l[2];
  float o[2][kD];
};

// Merge (m1, l1, o1) into (m0, l0, o0) for one lane's 4 output elements.
__device__ __forceinline__ void merge4(float& m0, float& l0, float (&o0)[4], float m1, float l1,
                                       const float (&o1)[4]) {
  if (m1 == -INFINITY) return;
  if (m0 == -INFINITY) {
    m0 = m1; l0 = l1;
#pragma unroll
    for (int e = 0; e < 4; ++e) o0[e] = o1[e];
    return;
  }
  const float M = fmaxf(m0, m1);
  const float a0 = exp2f(m0 - M), a1 = exp2f(m1 - M);
  l0 = a0 * l0 + a1 * l1;
#pragma unroll
  for (int e = 0; e < 4; ++e) o0[e] = a0 * o0[e] + a1 * o1[e];
  m0 = M;
}

__global__ void __launch_bounds__(kAttThreads) attend_kernel(AttendArgs a) {
  TraceScope trace(a.trace, kTrAttend);
  __shared__ AttPart part;
  __shared__ float wm[kAttWarps][2], wl[kAttWarps][2];
  __shared__ float wo[kAttWarps][2][kD];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int rank = blockIdx.x;  // cluster rank (the cluster spans gridDim.x)
  const int bh = blockIdx.y;
  const int b = bh / a.Hq, h = bh % a.Hq;
  const int g = h / (a.Hq / a.kv.Hkv);
  pdl_wait();  // selected rows come from the top-K kernel
  trace.mark(1);

  const int64_t L = seq_len(a.lens, a.len_host, b, a.kv.l_cap);
  const int64_t nw = a.window ? window_count(L, a.n_init, a.n_recent) : 0;
  // with a window the selected count is min(K, |pool|); otherwise (ReTopK)
  // it comes from the selection kernels
  const int64_t ns = a.window ? (a.K < L - nw ? a.K : L - nw) : a.sel_n[bh];
  const int64_t R = nw + ns;
  const int64_t c0 = R * rank / kAttCluster, c1 = R * (rank + 1) / kAttCluster;
  const int64_t w0 = c0 + (c1 - c0) * wid / kAttWarps, w1 = c0 + (c1 - c0) * (wid + 1) / kAttWarps;
  const uint16_t* vbase = a.kv.page_table ? a.kv.v : a.kv.v + kv_row(a.kv, b, g, 0);
  const float* wzrow = a.wz + (int64_t)bh * a.wz_stride;
  const int32_t* srow = a.sel_idx + (int64_t)bh * a.K;
  const float* szrow = a.sel_z + (int64_t)bh * a.K;

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float o[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  // chunks of 32 rows: one round of (position, logit) loads, then all 32 V
  // rows in flight before any is used
  for (int64_t base = w0; base < w1; base += 2 * kBatch) {
    float z = -INFINITY;
    int pos = 0, set = 0;
    if (base + lane < w1) {
      const int64_t j = base + lane;
      if (j < nw) {
        pos = (int)window_pos(j, L, a.n_init, a.n_recent);
        z = __ldcg(wzrow + j);
      } else {
        pos = srow[j - nw];
        z = szrow[j - nw];
        set = 1;
      }
      z *= kLog2e;
    }
    uint2 vv[2 * kBatch];
#pragma unroll
    for (int k = 0; k < 2 * kBatch; ++k) {
      const int pk = __shfl_sync(0xffffffffu, pos, k);
      const uint16_t* row = a.kv.page_table ? vbase + kv_row(a.kv, b, g, pk)
                                            : vbase + (int64_t)pk * kD;
      vv[k] = base + k < w1 ? __ldg(reinterpret_cast<const uint2*>(row + lane * 4))
                            : make_uint2(0u, 0u);
    }
    // chunk maxima per set, then rescale the running partials
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      const float bm = warp_max(set == st ? z : -INFINITY);
      if (bm > m[st]) {
        const float sc = m[st] == -INFINITY ? 0.f : exp2f(m[st] - bm);
        l[st] *= sc;
#pragma unroll
        for (int e = 0; e < 4; ++e) o[st][e] *= sc;
        m[st] = bm;
      }
    }
#pragma unroll
    for (int k = 0; k < 2 * kBatch; ++k) {
      const float zk = __shfl_sync(0xffffffffu, z, k);
      const int sk = __shfl_sync(0xffffffffu, set, k);
      if (zk == -INFINITY) continue;  // row past the range (warp-uniform)
      const float mk = sk ? m[1] : m[0];
      const float p = exp2f(zk - mk);
      const float v0 = bf_lo(vv[k].x), v1 = bf_hi(vv[k].x), v2 = bf_lo(vv[k].y),
                  v3 = bf_hi(vv[k].y);
      if (sk) {
        l[1] += p;
        o[1][0] = fmaf(p, v0, o[1][0]); o[1][1] = fmaf(p, v1, o[1][1]);
        o[1][2] = fmaf(p, v2, o[1][2]); o[1][3] = fmaf(p, v3, o[1][3]);
      } else {
        l[0] += p;
        o[0][0] = fmaf(p, v0, o[0][0]); o[0][1] = fmaf(p, v1, o[0][1]);
        o[0][2] = fmaf(p, v2, o[0][2]); o[0][3] = fmaf(p, v3, o[0][3]);
      }
    }
  }
  // ---- combine the warps of this CTA ----
#pragma unroll
  for (int st = 0; st < 2; ++st) {
    if (lane == 0) {
      wm[wid][st] = m[st];
      wl[wid][st] = l[st];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) wo[wid][st][lane * 4 + e] = o[st][e];
  }
  __syncthreads();
  if (tid < 2 * kD) {
    const int st = tid / kD, t = tid % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttWarps; ++w) M = fmaxf(M, wm[w][st]);
    float acc = 0.f, lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttWarps; ++w) {
        if (wm[w][st] == -INFINITY) continue;
        const float e = exp2f(wm[w][st] - M);
        acc = fmaf(e, wo[w][st][t], acc);
        lsum = fmaf(e, wl[w][st], lsum);
      }
    }
    part.o[st][t] = acc;
    if (t == 0) {
      part.m[st] = M;
      part.l[st] = lsum;
    }
  }
  trace.mark(2);
  cluster_sync_all();  // every CTA's partial is in its shared memory

  // ---- rank 0: Eq. 4-5 over the cluster's partials ----
  if (rank == 0 && tid < kD) {
    float zt[2], lsum[2], osum[2];
    float mc[2][kAttCluster], lc[2][kAttCluster], oc[2][kAttCluster];
#pragma unroll
    for (int c = 0; c < kAttCluster; ++c)  // all remote loads first
#pragma unroll
      for (int st = 0; st < 2; ++st) {
        mc[st][c] = ld_dsmem(&part.m[st], c);
        lc[st][c] = ld_dsmem(&part.l[st], c);
        oc[st][c] = ld_dsmem(&part.o[st][tid], c);
      }
#pragma unroll
    for (int st = 0; st < 2; ++st) {
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < kAttCluster; ++c) M = fmaxf(M, mc[st][c]);
      float ls = 0.f, os = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int c = 0; c < kAttCluster; ++c) {
          const float e = mc[st][c] == -INFINITY ? 0.f : exp2f(mc[st][c] - M);
          ls = fmaf(e, lc[st][c], ls);
          os = fmaf(e, oc[st][c], os);
        }
      }
      zt[st] = M;  // z~1 (window), z~2 (selected)
      lsum[st] = ls;
      osum[st] = os;
    }
    // gamma merge: z~ = max(z~1, z~2); den = sum over W u Omega of e^(z - z~)
    float outv = 0.f, lse = -INFINITY;
    const bool eW = !(lsum[0] > 0.f), eO = !(lsum[1] > 0.f);
    if (!(eW && eO)) {
      const float z = eW ? zt[1] : (eO ? zt[0] : fmaxf(zt[0], zt[1]));
      const float aW = eW ? 0.f : exp2f(zt[0] - z);
      const float aO = eO ? 0.f : exp2f(zt[1] - z);
      const float den = aW * lsum[0] + aO * lsum[1];
      // g1 o_W + g2 o_Omega with o_X = osum_X / l_X and g_X = a_X l_X / den
      outv = (aW * osum[0] + aO * osum[1]) / den;
      lse = (z + log2f(den)) * kLn2;  // back to natural log
    }
    a.out[(int64_t)bh * kD + tid] = outv;
    if (tid == 0 && a.lse_out) a.lse_out[bh] = lse;
    if (a.push_qbar) {  // ReTopK: push (qbar_t, S_t) over the oldest FIFO entry
      const int64_t hc = (int64_t)h * a.C + a.slot;
      a.cache_qbar[hc * kD + tid] = a.push_qbar[(int64_t)h * kD + tid];
      const int n = (int)ns;
      for (int j = tid; j < a.K; j += kD)
        a.cache_sup[hc * a.K + j] = j < n ? srow[j] : -1;
      if (tid == 0) a.cache_sup_n[hc] = n;
    }
  }
  cluster_sync_all();  // rank 0 has finished reading remote shared memory
}

cudaError_t launch_attend(const AttendArgs& a, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kAttCluster, a.B * a.Hq);
  cfg.blockDim = dim3(kAttThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kAttCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attend_kernel, a);
}

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
