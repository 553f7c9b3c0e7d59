// noalloc.cu -- sparse_attn_decode_noalloc: the decode step with its scratch
// memory in a fixed array that the library itself owns on every device.
//
// The decode step needs scratch global memory (histograms, per-head lists of
// candidate (position, logit) pairs, the selected set) beyond its inputs and
// outputs.  sparse_attn_decode takes that scratch from the caller.  Some
// callers cannot provide it: a serving engine that hands nearly all device
// memory to its own KV-cache pool at start-up and forbids later allocations,
// or a plain C host without an allocator of its own for whom cudaMalloc (which
// may synchronise the device) is not allowed inside its decode loop.  This
// entry point serves them: the scratch is a file-scope device array of
// kScratchBytes, created when the library's module is loaded on a device and
// kept until the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/tsa.h"

namespace tsa {
int report_error(int code, const char* msg);
int validate_decode(const void* q, const tsa_kv* kv, const int32_t* lens, int B, int Hq,
                    int Hkv, int d, int K, int n_init, int n_recent, float scale,
                    const float* out);
size_t decode_zero_bytes(int B, int Hq, int Hkv, int64_t l_cap, int K, int n_init, int n_recent);
}  // namespace tsa

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB per device
constexpr int kMaxDevices = 64;

// Device memory; in host code this name is only a stand-in for the symbol
// (never a device address): host code asks the runtime for the address.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device, looked up once per device.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tsa::report_error(TSA_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return tsa::report_error(TSA_ERR_INVALID_ARG, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p)
      return tsa::report_error(TSA_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e)
                                                              : "scratch address is NULL");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TSA_OK;
}

}  // namespace

extern "C" {

size_t tsa_noalloc_scratch_bytes(void) { return kScratchBytes; }

int sparse_attn_decode_noalloc(const void* q, const tsa_kv* kv, const int32_t* lens, int B,
                               int Hq, int Hkv, int d, int K, int n_init, int n_recent,
                               float scale, float* out, float* lse_out, int32_t* topk_idx,
                               float* topk_score, void* stream) {
  // The same host checks as sparse_attn_decode first: an invalid call
  // touches neither the array nor the stream.
  int rc = tsa::validate_decode(q, kv, lens, B, Hq, Hkv, d, K, n_init, n_recent, scale, out);
  if (rc != TSA_OK) return rc;
  if (B == 0) return sparse_attn_decode(q, kv, lens, B, Hq, Hkv, d, K, n_init, n_recent,
                                        scale, out, lse_out, topk_idx, topk_score, nullptr, 0,
                                        stream);
  const size_t need = tsa_decode_workspace_size(B, Hq, Hkv, d, kv->l_cap, K, n_init, n_recent);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof msg,
             "problem needs %zu bytes of scratch; sparse_attn_decode_noalloc holds %zu "
             "(use sparse_attn_decode with a caller workspace)",
             need, kScratchBytes);
    return tsa::report_error(TSA_ERR_WORKSPACE, msg);
  }
  void* scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc != TSA_OK) return rc;
  // Calls of any size share the array, so the counters that must start at
  // zero (and the status word) are cleared on the stream every time; the rest
  // needs no initialisation.
  if (kv->l_cap > 0) {
    const cudaError_t e =
        cudaMemsetAsync(scratch, 0, tsa::decode_zero_bytes(B, Hq, Hkv, kv->l_cap, K, n_init,
                                                           n_recent),
                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return tsa::report_error(TSA_ERR_CUDA, cudaGetErrorString(e));
  }
  return sparse_attn_decode(q, kv, lens, B, Hq, Hkv, d, K, n_init, n_recent, scale, out,
                            lse_out, topk_idx, topk_score, scratch, kScratchBytes, stream);
}

}  // extern "C"
