// q8.cu -- int8 key codes and the query preparation of the quantised scan.
//
// "RetrievalAttention" review, Appendix C "CPU memory minimization" (8-bit
// scalar quantisation of the key vectors) and the future-work item "Scalar
// quantization of KV vectors with accuracy-preservation guarantees" (the
// scheme is left open; per-channel symmetric is the one used here).  Codes
// halve the bytes of the key scan; exactness is kept by rescoring (the
// finish kernel), so the selected set is the one the bf16 scan selects.
//
// Per (sequence, KV head, channel j):
//   s_j  = maxabs_j / 127 (binary32 division, over the fitted rows)
//   c_ij = clamp(rint(k_ij / s_j), -127, 127) (binary32 quotient, ties to
//          even; 0 where s_j = 0), stored as the byte c + 128
//   e_j  >= max_i |k_ij - s_j c_ij| (an upper bound of the exact error)
// A row appended later uses the stored s_j; past 127 s_j it saturates and
// its error raises e_j.
//
// Logit bound.  With t = max_j |q_j s_j| (1 if that is 0), qh_j =
// fp16(q_j s_j / t) and delta_j = q_j s_j - t qh_j (exact in double):
//   z_i - z^_i = scale (sum_j q_j (k_ij - s_j c_ij) + sum_j delta_j c_ij)
//   |z_i - z^_i| <= scale (sum_j |q_j| e_j + 127 sum_j |delta_j|)
// for the exact sums.  Both sides are computed on the tensor cores with fp32
// accumulation (bf16 q.k for z, fp16 qh.c for z^); each result is taken to
// be within 2^-12 of the sum of its terms' magnitudes (a wide margin over
// binary32 accumulation of 128 products), so
//   eps = scale (sum_j |q_j| e_j + 127 sum_j |delta_j|
//                + 2^-12 (sum_j |q_j| (127 s_j + e_j) + 127 t sum_j |qh_j|))
// rounded up.  |k_ij| <= 127 s_j + e_j bounds the bf16 terms.
#include <cuda_fp16.h>

#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

namespace {

constexpr int kQ8Rows = 1024;  // rows per block of the coding kernels

// One code (offset binary) and an upper bound of its error |k - s c|: the
// fused multiply-add rounds the exact difference once, so |r| (1 + 2^-23)
// bounds it.
__device__ __forceinline__ uint8_t q8_code(float k, float s, float& e) {
  float c = 0.f;
  if (s != 0.f) c = fminf(fmaxf(rintf(__fdiv_rn(k, s)), -127.f), 127.f);
  const float r = fmaf(-s, c, k);
  e = __fmul_ru(fabsf(r), 1.0f + 0x1p-23f);
  return (uint8_t)((int)c + 128);
}

// Maxima of |k| per (sequence, KV head, channel) over rows [0, L_b), as the
// bits of non-negative floats (their integer order is the float order).
__global__ void __launch_bounds__(kD) q8_absmax_kernel(KvView kv, const int32_t* lens, int B,
                                                       uint32_t* maxbits) {
  const int unit = blockIdx.x, b = unit / kv.Hkv, g = unit % kv.Hkv, j = threadIdx.x;
  const int64_t L = seq_len(lens, 0, 0, b, kv.l_cap);
  const int64_t r0 = (int64_t)blockIdx.y * kQ8Rows;
  const int64_t r1 = r0 + kQ8Rows < L ? r0 + kQ8Rows : L;
  float m = 0.f;
  for (int64_t i = r0; i < r1; ++i) {
    const uint16_t h = kv.k[kv_row(kv, b, g, i) + j];
    m = fmaxf(m, fabsf(__uint_as_float((uint32_t)h << 16)));
  }
  if (r0 < r1) atomicMax(maxbits + (int64_t)unit * kD + j, __float_as_uint(m));
}

// Codes of rows [lo_b, L_b): lo_b = 0 when fitting (the scale is the stored
// maximum / 127), else L_b - n_tail; errors raised with atomicMax.
__global__ void __launch_bounds__(kD) q8_code_kernel(KvView kv, const int32_t* lens, int B,
                                                     int64_t n_tail, int fit, uint8_t* codes,
                                                     const float* kscale, float* kerr) {
  const int unit = blockIdx.x, b = unit / kv.Hkv, g = unit % kv.Hkv, j = threadIdx.x;
  const int64_t L = seq_len(lens, 0, 0, b, kv.l_cap);
  const int64_t lo = fit ? 0 : (L - n_tail > 0 ? L - n_tail : 0);
  const int64_t r0 = lo + (int64_t)blockIdx.y * kQ8Rows;
  const int64_t r1 = r0 + kQ8Rows < L ? r0 + kQ8Rows : L;
  if (r0 >= r1) return;
  const float sv = kscale[(int64_t)unit * kD + j];
  const float s = fit ? __fdiv_rn(sv, 127.f) : sv;
  float emax = 0.f;
  for (int64_t i = r0; i < r1; ++i) {
    const int64_t o = kv_row(kv, b, g, i) + j;
    float e;
    codes[o] = q8_code(__uint_as_float((uint32_t)kv.k[o] << 16), s, e);
    emax = fmaxf(emax, e);
  }
  atomicMax(reinterpret_cast<uint32_t*>(kerr) + (int64_t)unit * kD + j, __float_as_uint(emax));
}

__global__ void q8_scale_kernel(float* kscale, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) kscale[i] = __fdiv_rn(kscale[i], 127.f);
}

// Block-wide sums of four doubles over the 128 threads (all threads call).
__device__ void q8_sum4(double (&v)[4], double (*red)[4]) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o);
  __syncthreads();
  if (lane == 0)
#pragma unroll
    for (int k = 0; k < 4; ++k) red[w][k] = v[k];
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = red[0][k] + red[1][k] + red[2][k] + red[3][k];
}

__global__ void __launch_bounds__(kD) q8_prep_kernel(Q8PrepArgs a) {
  __shared__ double red[4][4];
  __shared__ float rmax[4];
  const int unit = blockIdx.x, b = unit / a.kv.Hkv, g = unit % a.kv.Hkv, j = threadIdx.x;
  const int lane = j & 31, w = j >> 5;
  const int G = a.Hq / a.kv.Hkv;
  const int64_t L = seq_len(a.lens, a.len_host, a.len_step, b, a.kv.l_cap);
  const float s = a.kscale[(int64_t)unit * kD + j];
  float e = a.kerr[(int64_t)unit * kD + j];
  // the newest rows' codes (this thread owns channel j of its unit)
  if (a.n_new > 0) {
    const int64_t lo = L - a.n_new > 0 ? L - a.n_new : 0;
    for (int64_t i = lo; i < L; ++i) {
      const int64_t o = kv_row(a.kv, b, g, i) + j;
      float ei;
      a.codes[o] = q8_code(__uint_as_float((uint32_t)a.kv.k[o] << 16), s, ei);
      e = fmaxf(e, ei);
    }
    a.kerr[(int64_t)unit * kD + j] = e;
  }
  __half qhv[kMaxGroup];
  float qtsv[kMaxGroup], epsv[kMaxGroup];
  for (int hl = 0; hl < G; ++hl) {
    const int bh = b * a.Hq + g * G + hl;
    const float qj = __uint_as_float((uint32_t)a.q[(int64_t)bh * kD + j] << 16);
    const double v = (double)qj * (double)s;  // exact: 8 x 24 significant bits
    float m = warp_max(fabsf((float)v));
    if (lane == 0) rmax[w] = m;
    __syncthreads();
    m = fmaxf(fmaxf(rmax[0], rmax[1]), fmaxf(rmax[2], rmax[3]));
    __syncthreads();
    const float t = m > 0.f ? m : 1.f;
    const __half qh = __float2half_rn((float)(v / (double)t));
    const double dl = v - (double)t * (double)__half2float(qh);
    const double aq = fabs((double)qj);
    double acc[4] = {aq * (double)e, fabs(dl), aq * (127.0 * (double)s + (double)e),
                     fabs((double)__half2float(qh))};
    q8_sum4(acc, red);
    const double bound = (double)a.scale * (acc[0] + 127.0 * acc[1] +
                                            0x1p-12 * (acc[2] + 127.0 * (double)t * acc[3]));
    qhv[hl] = qh;
    qtsv[hl] = t * a.scale;
    epsv[hl] = __double2float_ru(bound * (1.0 + 0x1p-20));
  }
  // The previous call's finish kernel may still read eps: write after it
  // has completed (everything above only read this call's inputs).
  pdl_wait();
  pdl_trigger();
  for (int hl = 0; hl < G; ++hl) {
    const int bh = b * a.Hq + g * G + hl;
    reinterpret_cast<__half*>(a.qh)[(int64_t)bh * kD + j] = qhv[hl];
    if (j == 0) {
      a.qts[bh] = qtsv[hl];
      a.eps[bh] = epsv[hl];
    }
  }
}

constexpr int kRsWarps = 8;  // rescore kernel: warps per CTA, two CTAs per SM

// A unit of the rescoring: 32 consecutive pairs of head bh's list, or 32
// consecutive window positions of head bh.
struct RsUnit {
  int bh;
  bool pairs;
  int r0, r1;  // rows [r0, min(r0 + 32, r1)) of the list / the window (< 2^31)
  int L;
};

__global__ void __launch_bounds__(32 * kRsWarps, 2) q8_rescore_kernel(Q8RescoreArgs a) {
  extern __shared__ int rs_sh[];  // [B*Hq + 1] units before head bh, then [B*Hq] pairs
  TraceScope trace(a.trace, kTrQ8Rescore);
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int gr = lane >> 2, tq = lane & 3;
  const int BH = a.B * a.Hq, G = a.Hq / a.kv.Hkv;
  int* rs_pre = rs_sh;
  int* rs_np = rs_sh + BH + 1;
  pdl_wait();  // the pairs and list sizes come from the scan
  pdl_trigger();
  trace.mark(1);
  // units of 32 rows per head: its pairs, then its window positions
  if (wid == 0) {
    int run = 0;
    for (int base = 0; base < BH; base += 32) {
      const int bh = base + lane;
      int u = 0;
      if (bh < BH) {
        int64_t np = __ldcg(a.dense_n + (int64_t)bh * kCtrStride);
        if (np > a.dense_stride) np = a.dense_stride;
        const int64_t L = seq_len(a.lens, a.len_host, a.len_step, bh / a.Hq, a.kv.l_cap);
        const int64_t nw = window_count(L, a.n_init, a.n_recent);
        rs_np[bh] = (int)np;
        u = (int)((np + 31) / 32 + (nw + 31) / 32);
      }
      int incl = u;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (bh < BH) rs_pre[bh] = run + incl - u;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) rs_pre[BH] = run;
  }
  __syncthreads();
  const int total = rs_pre[BH];
  auto unit_of = [&](int u) -> RsUnit {
    int lo = 0, hi = BH - 1;  // the head whose units contain u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (rs_pre[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    RsUnit r;
    r.bh = lo;
    r.L = (int)seq_len(a.lens, a.len_host, a.len_step, lo / a.Hq, a.kv.l_cap);
    const int np = rs_np[lo];
    const int up = (np + 31) / 32, lu = u - rs_pre[lo];
    r.pairs = lu < up;
    r.r0 = 32 * (r.pairs ? lu : lu - up);
    r.r1 = r.pairs ? np : (int)window_count(r.L, a.n_init, a.n_recent);
    return r;
  };
  // positions of a unit's rows gr + 8k (0xffffffff: none)
  auto unit_pos = [&](const RsUnit& r, uint32_t (&pos)[4]) {
    const uint2* lrow = a.dense + (int64_t)r.bh * a.dense_stride;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = r.r0 + gr + 8 * k;
      if (j >= r.r1) pos[k] = 0xffffffffu;
      else pos[k] = r.pairs ? __ldcg(&lrow[j].x)
                            : (uint32_t)window_pos(j, r.L, a.n_init, a.n_recent);
    }
  };
  const int stride = gridDim.x * kRsWarps;
  int u = blockIdx.x * kRsWarps + wid;
  if (u >= total) return;
  RsUnit cur = unit_of(u);
  uint32_t pos[4];
  unit_pos(cur, pos);
  int64_t cur_head0 = -1;
  uint32_t qb[4][4];
  for (; u < total; u += stride) {
    // the next unit's positions are requested before this unit's rows
    RsUnit nxt = cur;
    uint32_t npos[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
    if (u + stride < total) {
      nxt = unit_of(u + stride);
      unit_pos(nxt, npos);
    }
    const int bh = cur.bh, b = bh / a.Hq, h = bh % a.Hq, g = h / G, hl = h - g * G;
    const int64_t head0 = (int64_t)b * a.Hq + g * G;
    if (head0 != cur_head0) {
      load_q_frag(a.q, head0, G, qb);
      cur_head0 = head0;
    }
    bool ok[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) ok[k] = pos[k] != 0xffffffffu && pos[k] < (uint32_t)cur.L;
    // rows gr + 8k of the 32: lane (gr, tq) reads 16 bytes of each at
    // 8(4p + tq), all 16 loads in flight before the first product
    uint4 R[4][4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint16_t* kr = a.kv.k + kv_row(a.kv, b, g, ok[k] ? pos[k] : 0);
#pragma unroll
      for (int p = 0; p < 4; ++p)
        R[k][p] = ok[k] ? *reinterpret_cast<const uint4*>(kr + 8 * (4 * p + tq))
                        : make_uint4(0u, 0u, 0u, 0u);
    }
    float z[4];
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {  // the key scan's fragments, k order and (c0 + c1) * scale
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint4 X = R[2 * blk][p], Y = R[2 * blk + 1][p];
        mma_bf16(c0, X.x, Y.x, X.y, Y.y, qb[p][0], qb[p][1]);
        mma_bf16(c1, X.z, Y.z, X.w, Y.w, qb[p][2], qb[p][3]);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int e = 2 * r + (hl & 1);
        z[2 * blk + r] = (c0[e] + c1[e]) * a.scale;
      }
    }
    if (tq == (hl >> 1)) {  // lanes holding head hl's column write
      if (cur.pairs) {
        uint2* lrow = a.dense + (int64_t)bh * a.dense_stride;
        const uint32_t ekz = q8_exact_key(__ldcg(a.emit_key + bh), __ldcg(a.eps + bh));
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (pos[k] != 0xffffffffu) {
            const bool keep = ok[k] && f2key(z[k]) >= ekz;
            lrow[cur.r0 + gr + 8 * k] =
                keep ? make_uint2(pos[k], __float_as_uint(z[k])) : make_uint2(0xffffffffu, 0u);
          }
      } else {
        float* wzrow = a.wz + (int64_t)bh * a.wz_stride;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (ok[k]) wzrow[cur.r0 + gr + 8 * k] = z[k];
      }
    }
    cur = nxt;
#pragma unroll
    for (int k = 0; k < 4; ++k) pos[k] = npos[k];
  }
}

}  // namespace

cudaError_t launch_q8_rescore(const Q8RescoreArgs& a, int grid, cudaStream_t st) {
  const int BH = a.B * a.Hq;
  if (BH == 0) return cudaSuccess;
  const size_t smem = (size_t)(2 * BH + 1) * 4;
  static int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(q8_rescore_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)((2 * kQ8MaxHeads + 1) * 4));
    if (e != cudaSuccess) return e;
    configured[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(32 * kRsWarps);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, q8_rescore_kernel, a);
}

cudaError_t launch_q8_prep(const Q8PrepArgs& a, cudaStream_t st, bool pdl) {
  if (a.B == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B * a.kv.Hkv);
  cfg.blockDim = dim3(kD);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, q8_prep_kernel, a);
}

cudaError_t launch_q8_quantize(const KvView& kv, const int32_t* lens, int B, int64_t n_tail,
                               bool fit, uint8_t* codes, float* kscale, float* kerr,
                               cudaStream_t st) {
  const int units = B * kv.Hkv;
  if (units == 0) return cudaSuccess;
  const int64_t rows = fit ? kv.l_cap : (n_tail < kv.l_cap ? n_tail : kv.l_cap);
  if (rows <= 0) return cudaSuccess;
  const dim3 grid(units, (unsigned)((rows + kQ8Rows - 1) / kQ8Rows));
  if (fit) {
    q8_absmax_kernel<<<grid, kD, 0, st>>>(kv, lens, B, reinterpret_cast<uint32_t*>(kscale));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  q8_code_kernel<<<grid, kD, 0, st>>>(kv, lens, B, n_tail, fit ? 1 : 0, codes, kscale, kerr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !fit) return e;
  const int n = units * kD;
  q8_scale_kernel<<<(n + 255) / 256, 256, 0, st>>>(kscale, n);
  return cudaGetLastError();
}

}  // namespace tsa
