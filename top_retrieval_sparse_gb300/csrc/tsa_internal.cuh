// tsa_internal.cuh -- device helpers shared by the libtsa kernels.
//
// Decode-step top-K sparse attention ("RetrievalAttention: Accelerating
// Long-Context LLM Inference via Vector Retrieval", Eq. 1-5, Flat exact
// top-k) and ReTopK reuse ("Recall Before You Rank", method sections 1-5).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tsa {

constexpr int kD = 128;                         // head dimension (only size compiled)
constexpr int kRowBytes = kD * 2;               // one bf16 K or V row
constexpr int kHistBits = 11;                   // pass-1 radix digit
constexpr int kHistBins = 1 << kHistBits;
constexpr int kHistShift = 32 - kHistBits;
constexpr int kMaxGroup = 8;                    // query heads per KV head
constexpr int kMaxUnits = 512;                  // B * Hkv limit of one call
// Each head's pair-list fill counter sits in its own 128-byte line: the
// slot atomics of all heads then spread over the L2 slices instead of
// queueing in one.
constexpr int kCtrStride = 32;
// Fine per-head histogram of the emitted pairs (plain key scan): bin of a
// pair = (its logit key >> 16) minus (the emission key >> 16), the last bin
// also holding everything above it.  16 key bits resolve a logit to 1/128 of
// its binade, so the threshold bin holds a few dozen pairs, not thousands.
constexpr int kH16Bins = 1024;
constexpr int kH16Shift = 16;
constexpr long long kWaitLimitNs = 1000000000;  // bounded waits: 1 s


// Status word bits written by kernels into the workspace (sticky: only the
// host clears them, through tsa_workspace_status).
constexpr int kStatusTimeout = 1;    // a bounded wait expired: the call's outputs are NaN
constexpr int kStatusBadLength = 2;  // a sequence length outside [0, l_cap] was clamped
constexpr int kStatusCheck = 4;      // an internal consistency check of a selection failed

// ---------------------------------------------------------------- encoding
// Order-preserving key of an fp32 value: a > b  <=>  key(a) > key(b).
// -0 is folded into +0 first, so equal logits have equal keys.
__device__ __forceinline__ uint32_t f2key(float f) {
  f = f + 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}
// Rank key of (logit, position): larger logit first, then smaller position.
__device__ __forceinline__ uint64_t rank_key(float z, uint32_t pos) {
  return ((uint64_t)f2key(z) << 32) | (uint64_t)(0xffffffffu - pos);
}
__device__ __forceinline__ uint32_t rank_pos(uint64_t v) {
  return 0xffffffffu - (uint32_t)(v & 0xffffffffu);
}

// bf16x2 word -> (low element, high element) as fp32 (exact).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ------------------------------------------------------------- KV address
struct KvView {
  const uint16_t* k;          // bf16 bits
  const uint16_t* v;
  const int32_t* page_table;  // nullptr: contiguous
  int page_shift;             // log2(page_size) (paged)
  int max_pages;
  int64_t l_cap;
  int Hkv;
  // Rows between sequences (contiguous: Hkv * l_cap) and page-table entries
  // between sequences (paged: max_pages); 0 makes every sequence index read
  // sequence 0's cache (several queries of one sequence as a batch).
  int64_t seq_rows;
  int64_t pt_stride;
};

// Element offset of row i of KV head g of sequence b.
__device__ __forceinline__ int64_t kv_row(const KvView& kv, int b, int g, int64_t i) {
  if (kv.page_table) {
    int64_t page = kv.page_table[(int64_t)b * kv.pt_stride + (i >> kv.page_shift)];
    int64_t r = i & ((1 << kv.page_shift) - 1);
    return (((page * kv.Hkv + g) << kv.page_shift) + r) * kD;
  }
  return ((int64_t)b * kv.seq_rows + (int64_t)g * kv.l_cap + i) * kD;
}

// Sequence length (lens[b], or len_host + b * len_step without a lens
// array), clamped to [0, cap] so that no position past the cache is ever
// addressed.
__device__ __forceinline__ int64_t seq_len(const int32_t* lens, int64_t len_host,
                                           int64_t len_step, int b, int64_t cap) {
  int64_t L = lens ? (int64_t)lens[b] : len_host + (int64_t)b * len_step;
  return L < 0 ? 0 : (L > cap ? cap : L);
}

// Window W_t = [0, n_init) u [L - n_recent, L), clipped (static pattern W).
__device__ __forceinline__ bool in_window(int64_t i, int64_t L, int n_init, int n_recent) {
  return i < n_init || i >= L - n_recent;
}
__device__ __forceinline__ int64_t window_count(int64_t L, int n_init, int n_recent) {
  int64_t a = n_init < L ? n_init : L;
  int64_t lo = L - n_recent > a ? L - n_recent : a;
  return a + (L - lo);
}
// j-th window position in ascending order (j < window_count).
__device__ __forceinline__ int64_t window_pos(int64_t j, int64_t L, int n_init, int n_recent) {
  int64_t a = n_init < L ? n_init : L;
  if (j < a) return j;
  int64_t lo = L - n_recent > a ? L - n_recent : a;
  return lo + (j - a);
}

// ------------------------------------------------ programmatic launch
// Dependent-launch control (sm_90+): a kernel launched with programmatic
// stream serialization may start before its predecessor finishes; it must
// call pdl_wait() before touching the predecessor's results.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// -------------------------------------------------------------- PTX: TMA
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait on an mbarrier phase: false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if ((long long)(globaltimer_ns() - t0) > limit_ns) return false;
  }
}
// Bounded wait that also gives up as soon as *abort is set (CTA-wide stop).
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t* bar, uint32_t parity,
                                                   volatile int* abort,
                                                   long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if ((long long)(globaltimer_ns() - t0) > limit_ns) return false;
  }
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---------------------------------------------------------- tensor cores
// D += A * B, m16n8k16, bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two offset-binary key codes (bytes 0-1, or 2-3, of w: u = c + 128) as an
// fp16x2 word holding the integers c exactly: the byte becomes the low
// mantissa bits of 1024 (0x6400 | u = 1024 + u) and 1152 is subtracted
// (exact: every value involved is an integer below 2048).
__device__ __forceinline__ uint32_t codes_lo_f16x2(uint32_t w) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(r) : "r"(w), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(r) : "r"(0x64806480u));
  return r;
}
__device__ __forceinline__ uint32_t codes_hi_f16x2(uint32_t w) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(r) : "r"(w), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(r) : "r"(0x64806480u));
  return r;
}

// B fragments of the query heads of group [head0, head0 + G) for the key
// scan's bf16 contraction: lane (gr, tq) holds head gr's dims [8(4p+tq), +8)
// for p < 4 (zero for gr >= G).
__device__ __forceinline__ void load_q_frag(const uint16_t* q, int64_t head0, int G,
                                            uint32_t (&qb)[4][4]) {
  const int lane = threadIdx.x & 31, gr = lane >> 2, tq = lane & 3;
  const uint16_t* qp = q + (head0 + (gr < G ? gr : 0)) * kD;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (gr < G) w = *reinterpret_cast<const uint4*>(qp + 8 * (4 * p + tq));
    qb[p][0] = w.x; qb[p][1] = w.y; qb[p][2] = w.z; qb[p][3] = w.w;
  }
}

// The emission key of the exact logits that a quantised emission with key
// k^ (order-preserving key; 0 admits everything) guarantees, for a logit
// error bound eps: f2key(k^ + eps), the sum rounded up (NaN: nothing).
__device__ __forceinline__ uint32_t q8_exact_key(uint32_t khat, float eps) {
  if (khat == 0u) return 0u;
  const float kz = __fadd_ru(key2f(khat), eps);
  return kz == kz ? f2key(kz) : 0xffffffffu;
}


// ------------------------------------------------------------- clusters
// Full barrier over the thread-block cluster (release / acquire: shared and
// global writes before it are visible to the cluster's threads after it).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n"
               "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// Loads from the shared memory of CTA `cta` of this cluster (distributed
// shared memory): p is the address of the same variable in this CTA.
__device__ __forceinline__ uint32_t ld_dsmem_u32(const uint32_t* p, uint32_t cta) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(cta));
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}
// Stores into the shared memory of CTA `cta` of this cluster.
__device__ __forceinline__ void st_dsmem(float* p, uint32_t cta, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(cta));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}
// Stores into the shared memory of CTA `cta` of this cluster.
__device__ __forceinline__ void st_dsmem_u64(uint64_t* p, uint32_t cta, uint64_t v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(cta));
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(remote), "l"(v) : "memory");
}
// The two halves of a cluster barrier, for a barrier whose wait comes later
// (every thread of the cluster calls both, in this order, before its next
// cluster barrier).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ uint64_t ld_dsmem_u64(const uint64_t* p, uint32_t cta) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(p)), "r"(cta));
  uint64_t v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(remote) : "memory");
  return v;
}

// ------------------------------------------------------------- tracing
// Optional per-CTA timeline: when a kernel's argument block carries a trace
// buffer, thread 0 of every CTA appends one record with the kernel id, the
// CTA, its SM and up to four %globaltimer stamps (start, two phase marks,
// exit).  Off (nullptr) costs one predicate per CTA.
struct TraceRec {
  uint32_t kernel, block, smid, pad;
  uint64_t t[4];
};
struct TraceBuf {
  uint32_t* count;   // records appended so far
  TraceRec* rec;
  uint32_t cap;
};

__device__ __forceinline__ uint32_t smid_u32() {
  uint32_t r;
  asm volatile("mov.u32 %0, %smid;" : "=r"(r));
  return r;
}

struct TraceScope {
  TraceBuf tb;
  bool on;
  uint32_t kernel;
  uint32_t info = 0;  // kernel-specific word stored in the record's pad field
  uint64_t t[4];
  __device__ TraceScope(const TraceBuf& b, uint32_t k) : tb(b), kernel(k) {
    on = b.rec != nullptr && threadIdx.x == 0;
    t[0] = t[1] = t[2] = t[3] = 0;
    if (on) t[0] = globaltimer_ns();
  }
  __device__ void mark(int i) {
    if (on) t[i] = globaltimer_ns();
  }
  __device__ ~TraceScope() {
    if (on) {
      if (!t[3]) t[3] = globaltimer_ns();
      const uint32_t slot = atomicAdd(tb.count, 1u);
      if (slot < tb.cap) {
        TraceRec r;
        r.kernel = kernel;
        r.block = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
        r.smid = smid_u32();
        r.pad = info;
        for (int i = 0; i < 4; ++i) r.t[i] = t[i];
        tb.rec[slot] = r;
      }
    }
  }
};
enum TraceKernel : uint32_t {  // 2, 3, 5 and 6 are retired ids
  kTrScan = 1, kTrSelector = 4, kTrFinish = 7, kTrFinishPhases = 8, kTrQ8Rescore = 9
};

// ------------------------------------------------------ warp/block utils
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace tsa
