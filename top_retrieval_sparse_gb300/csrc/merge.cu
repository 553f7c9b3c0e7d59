// merge.cu -- the gamma1/gamma2 merge of two attention partials given as
// (o, lse) pairs: "RetrievalAttention" Eq. 4-5 (o = g1 o_a + g2 o_b with
// g_j = e^(lse_j - lse) and lse = log(e^lse_a + e^lse_b)).  The decode path
// merges inside its finish kernel; this is the library's merge for partials
// computed elsewhere (e.g. a dense attention over other keys).
#include "tsa_internal.cuh"
#include "tsa_kernels.h"

namespace tsa {

// One CTA per row.  A partial with lse = -inf is empty; two empty partials
// give o = 0 and lse = -inf.  Each output element depends only on the same
// element of the inputs, so the outputs may alias the inputs.
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
  __syncthreads();  // every thread has read the row's lse values
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
