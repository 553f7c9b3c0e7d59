/*
 * tsa.h -- C ABI of libtsa: decode-step top-K sparse attention on one GB300.
 *
 * One decode step of one attention layer: for every query head, score the
 * query against every key of the cache, keep the exact top-K keys outside a
 * static window of initial + recent tokens, attend over those K rows and over
 * the window separately, and merge the two partial results with the
 * log-sum-exp rescale.  A second entry point runs ReTopK's reuse path, which
 * recalls candidate keys from a per-head cache of past queries instead of
 * scanning every key on most steps.
 *
 * Sources (page title, section / equation):
 *   [RA]  "RetrievalAttention: Accelerating Long-Context LLM Inference via
 *         Vector Retrieval": Eq. 1, Eq. 2, Eq. 3, Eq. 4-5, the "Flat"
 *         exact-KNN baseline, "CPU-GPU Co-Execution" (static pattern W),
 *         Appendix B.2 Algorithm 1 (per-step window update).
 *   [RTK] "Recall Before You Rank: Similarity-Guided Top-K Reuse for
 *         Efficient Long-Context Attention" (ReTopK): sections 1-5 of the
 *         method (query-support cache, similar-query recall, candidate set,
 *         exact re-ranking, fallback and refresh) and "GPU Kernel".
 *   [RA-review] the English review of RetrievalAttention: Appendix C "CPU
 *         memory minimization" and the future-work item "Scalar
 *         quantization of KV vectors with accuracy-preservation
 *         guarantees" (8-bit scalar quantisation of the keys).
 *
 * Conventions shared by every entry point
 *   - Element types: q, K, V are bf16 (IEEE binary16-brain, 2 bytes);
 *     outputs are fp32; indices are int32 token positions (0-based).
 *   - Head dimension d must be 128 (the only compiled size).
 *   - GQA: query head h reads KV head h / (Hq / Hkv); Hq % Hkv == 0,
 *     Hq / Hkv <= 8, B * Hkv <= 512 and B * Hq <= 65535.
 *   - Ownership: the caller allocates every buffer (device memory unless
 *     stated) and the workspace, and owns the stream.  No entry point
 *     allocates, frees or prints, and none but tsa_workspace_status
 *     synchronises; launches are asynchronous on `stream` (a cudaStream_t;
 *     NULL = legacy default stream).
 *   - Errors: every call returns a tsa_status.  Arguments are validated on
 *     the host before any launch; on an error nothing is launched and
 *     tsa_last_error() describes the problem (thread-local).  Launch
 *     failures are reported as TSA_ERR_CUDA.  Faults inside a kernel surface
 *     through the stream as usual CUDA errors.  What the kernels detect
 *     themselves (a bounded wait that expired, a length outside the cache)
 *     goes into a sticky status word in the workspace, which
 *     tsa_workspace_status() reads after the calls have run.
 *   - Concurrency: calls that share a workspace or a ReTopK state must be
 *     ordered on one stream.
 */
#ifndef TSA_H
#define TSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define TSA_API __attribute__((visibility("default")))
#else
#define TSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum tsa_status {
  TSA_OK = 0,
  TSA_ERR_INVALID_ARG = -1, /* a size, pointer or layout argument is invalid */
  TSA_ERR_WORKSPACE = -2,   /* workspace pointer NULL/misaligned or too small */
  TSA_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed           */
  TSA_ERR_STATE = -4,       /* ReTopK state handle invalid or not initialised */
  TSA_ERR_DEVICE_CHECK = -5,/* a device-side check flagged bad input          */
  TSA_ERR_TIMEOUT = -6      /* a bounded device wait expired (status word)    */
} tsa_status;

/* KV cache of one layer.
 *
 * Contiguous layout (page_table == NULL):
 *   k, v: bf16 [B][Hkv][l_cap][128]; sequence b, KV head g, position i at
 *   element ((b*Hkv + g)*l_cap + i)*128.
 * Paged layout (page_table != NULL):
 *   k, v: bf16 [num_pages][Hkv][page_size][128]; page_table: int32
 *   [B][max_pages] (device); position i of sequence b lives in page
 *   page_table[b*max_pages + i/page_size] at row i % page_size.
 *   page_size is a power of two in [16, 256]; l_cap = max_pages*page_size.
 * Base pointers must be 16-byte aligned.  Positions >= the sequence length
 * are never read. */
typedef struct tsa_kv {
  const void* k;
  const void* v;
  const int32_t* page_table;
  int32_t page_size;
  int32_t max_pages;
  int64_t l_cap;
} tsa_kv;

/* Human-readable description of the last error on this thread ("" if none). */
TSA_API const char* tsa_last_error(void);

/* Version string of the library build. */
TSA_API const char* tsa_version(void);

/* Number of kernels this library has launched in this process so far (all
 * threads, all entry points; a memset of workspace counters is not a
 * kernel and is not counted). */
TSA_API unsigned long long tsa_kernel_launches(void);

/* Per-stage timing (optional, thread-local).  With n >= 4 cudaEvent_t
 * handles (cast to void*), every later sparse_attn_decode / retopk_step call
 * on this thread records, on the call's stream, events[0] before its first
 * kernel, events[1] after the key scan, events[2] at once after events[1]
 * (the selection is the finish kernel's) and events[3] after the finish
 * kernel (selection, attention and merge; on ReTopK steps also the reuse
 * heads' rescoring and the FIFO push).  Events between kernels cost the overlap of their
 * launches.  events == NULL (or n == 0) turns it off.  The events stay owned
 * by the caller. */
TSA_API int tsa_set_stage_events(void* const* events, int n);

/* Per-CTA kernel timeline (optional, thread-local).  `buf` is device memory
 * (64-byte aligned) holding a uint32 record count at offset 0, which the
 * caller zeroes, followed from offset 64 by records of 48 bytes:
 *   uint32 kernel (1 key scan, 4 ReTopK selector, 7 finish (selection +
 *   attention), 8 finish phases; 2, 3, 5 and 6 are unused), uint32 CTA
 *   (linear block index), uint32 SM id, uint32 info (kernel 7: pairs the
 *   scan emitted for the head; kernel 8: bit 31 re-emission, bits 16-30
 *   the threshold bin, bits 0-15 the emission bin used; else 0),
 *   uint64 t[4] (%globaltimer ns: start, two kernel-specific phase marks
 *   or 0, exit; kernel 4: start, dependency wait over, candidate bitmap
 *   built, exit; kernel 8: start, threshold bin found, list read, rows
 *   gathered).
 * Later calls on this thread append one record per CTA while it fits.
 * buf == NULL (or too small) turns tracing off. */
TSA_API int tsa_set_trace(void* buf, size_t bytes);

/* ------------------------------------------------------------------ */
/* sparse_attn_decode -- [RA] Eq. 1-5 with an exact ("Flat") top-K Omega.
 *
 * For each sequence b (length L_b = lens[b], the newest token included)
 * and query head h:
 *   z_i   = scale * q_h . k_i                       for i < L_b   (Eq. 1)
 *   W     = [0, n_init) u [L_b - n_recent, L_b), clipped        (static W)
 *   Omega = the K positions of [0, L_b) \ W with the largest z,
 *           ties to the smaller position; all of it if smaller than K
 *   o_W, o_Omega: softmax-weighted V over W and Omega (Eq. 3)
 *   out   = g1 o_W + g2 o_Omega, lse = log sum_{W u Omega} e^z  (Eq. 4-5)
 *
 * q:          bf16 [B][Hq][128] (device)
 * kv:         the cache (see tsa_kv); read only
 * lens:       int32 [B] (device), 0 <= lens[b] <= kv->l_cap
 * K:          top-K budget (>= 0); n_init, n_recent >= 0
 * scale:      logit scale (1/sqrt(128) for standard attention)
 * out:        fp32 [B][Hq][128] (device)
 * lse_out:    fp32 [B][Hq] or NULL; -inf when W u Omega is empty
 * topk_idx:   int32 [B][Hq][K] or NULL: Omega in unspecified order, padded
 *             with -1 when fewer than K positions exist
 * topk_score: fp32 [B][Hq][K] or NULL: z of topk_idx (padding: -inf)
 * workspace:  device scratch of at least tsa_decode_workspace_size() bytes,
 *             256-byte aligned, zero-filled (e.g. cudaMemsetAsync 0) before
 *             its first use.  Every call leaves it ready for the next call
 *             with the same B, Hq, Hkv, l_cap, K, n_init and n_recent, so
 *             it is reused as is; zero it again before other sizes and after
 *             a call that failed.  It also keeps per-head state
 *             that speeds up the next call (never its result): use one
 *             workspace per layer.
 * Device-detected errors (read them with tsa_workspace_status):
 *   - every wait inside the kernels is bounded (1 s); if one expires the
 *     kernel gives up, the call's out / lse / topk_score are NaN and
 *     topk_idx is -1, the workspace stays consistent, and the status word
 *     keeps TSA_ERR_TIMEOUT: every later call on the workspace also outputs
 *     NaN until tsa_workspace_status(..., clear = 1) has cleared it;
 *   - a lens[b] outside [0, l_cap] is clamped to that range and reported as
 *     TSA_ERR_DEVICE_CHECK (the outputs are those of the clamped length).
 * Returns TSA_OK or an error; see the conventions above. */
TSA_API size_t tsa_decode_workspace_size(int B, int Hq, int Hkv, int d, int64_t l_cap,
                                 int K, int n_init, int n_recent);

TSA_API int sparse_attn_decode(const void* q, const tsa_kv* kv, const int32_t* lens,
                       int B, int Hq, int Hkv, int d, int K, int n_init,
                       int n_recent, float scale, float* out, float* lse_out,
                       int32_t* topk_idx, float* topk_score, void* workspace,
                       size_t ws_bytes, void* stream);

/* sparse_attn_decode_noalloc -- sparse_attn_decode without a caller
 * workspace.  The pages have no counterpart: this is a library service.
 *
 * For callers that cannot allocate device memory when they decode: a serving
 * engine that gives nearly all device memory to its KV-cache pool at start-up
 * and allows no later allocation, or a host for which cudaMalloc (it may
 * synchronise the device) is off limits inside the decode loop.  The scratch
 * lives in one array of tsa_noalloc_scratch_bytes() (32 MiB) of device
 * memory per device, which the library's module holds from the time it is
 * loaded on that device until the process exits.
 *
 * Same arguments and results as sparse_attn_decode, minus the workspace.
 *   - Problems whose tsa_decode_workspace_size() exceeds the array are
 *     rejected with TSA_ERR_WORKSPACE (nothing launched).  The size grows as
 *     B*Hq*16*(l_cap + 65536) bytes plus 12 KiB per head: B*Hq = 4 fits
 *     caches up to about 458 K positions, B*Hq = 16 about 65 K, and
 *     B*Hq >= 32 fits none.
 *   - The arguments are checked as in sparse_attn_decode before the array
 *     or the stream is touched.
 *   - Each call clears the array's status word with its counters, so a
 *     timeout shows as NaN outputs of that call only.
 *   - The first call on a device looks the array's device address up
 *     (cudaGetSymbolAddress, with that device current), which may load the
 *     library's module; make that first call before any stream capture.
 *   - Every call on a device, from any thread or stream, uses the same
 *     array, which keeps the previous call's contents; each call clears the
 *     counters that must start at zero on its stream.  Calls that overlap on
 *     the GPU race: order them on one stream.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
TSA_API size_t tsa_noalloc_scratch_bytes(void);

TSA_API int sparse_attn_decode_noalloc(const void* q, const tsa_kv* kv,
                       const int32_t* lens, int B, int Hq, int Hkv, int d, int K,
                       int n_init, int n_recent, float scale, float* out,
                       float* lse_out, int32_t* topk_idx, float* topk_score,
                       void* stream);

/* ------------------------------------------------------------------ */
/* int8 key codes and the quantised decode -- [RA-review] Appendix C "CPU
 * memory minimization" (8-bit scalar quantisation of the key vectors,
 * scheme left open) and the future-work item "Scalar quantization of KV
 * vectors with accuracy-preservation guarantees" (per-channel symmetric is
 * the scheme used here; the worry there -- quantised keys shift the top-K --
 * is removed by rescoring: the result is that of the bf16 keys).
 *
 * tsa_kq8: a quantised copy of a cache's keys, caller memory.
 *   codes: uint8, the row geometry of kv->k with one byte per element
 *          (contiguous [B][Hkv][l_cap][128], or paged [pages][Hkv]
 *          [page_size][128] through kv->page_table); the code c in
 *          [-127, 127] of k_ij is stored as the byte c + 128.  16-byte
 *          aligned.
 *   scale: fp32 [B][Hkv][128], the step s_j of each channel.
 *   err:   fp32 [B][Hkv][128], an upper bound of |k_ij - s_j c_ij| over
 *          every coded row of the channel.
 *   Per channel: s_j = maxabs_j / 127 (binary32 division, maxabs over the
 *   fitted rows), c_ij = clamp(rint(k_ij / s_j), -127, 127) (binary32
 *   quotient, ties to even; c = 0 where s_j = 0). */
typedef struct tsa_kq8 {
  void* codes;
  float* scale;
  float* err;
} tsa_kq8;

/* tsa_quantize_keys -- codes of a cache's keys.
 *   fit = 1: for each (sequence b, KV head, channel) s_j from the rows
 *            [0, lens[b]), then codes and err of those rows (n_tail unused);
 *   fit = 0: codes of the last n_tail rows [lens[b] - n_tail, lens[b])
 *            (clipped at 0) with the stored scales; err is raised to cover
 *            them (a value past 127 s_j saturates; its error counts).
 * lens: int32 [B] (device), 0 <= lens[b] <= kv->l_cap.  Launches up to three
 * kernels (and two memsets with fit) on `stream`; reads kv->k only.
 * Returns TSA_OK or an error (nothing launched on an argument error). */
TSA_API int tsa_quantize_keys(const tsa_kv* kv, const tsa_kq8* kq, const int32_t* lens,
                              int B, int Hkv, int d, int64_t n_tail, int fit,
                              void* stream);

/* sparse_attn_decode_q8 -- sparse_attn_decode with the pool scanned through
 * the key codes (128 bytes a key row instead of 256).
 *
 * Same arguments, contract and results as sparse_attn_decode: the selected
 * set Omega, topk_idx / topk_score (the logits of the bf16 keys, bit for bit
 * those sparse_attn_decode reports) and, up to the order of fp32 sums, out and
 * lse.  The codes must cover rows [0, lens[b] - n_new) of every sequence
 * when the call starts; the call first codes the last n_new rows (as
 * tsa_quantize_keys with fit = 0), so a decode loop that appends one key a
 * step passes n_new = 1.
 * How: per query head a bound eps on |z_i - z^_i| (z^ the logit of the codes)
 * is computed from err, the scales and the query; the scan emits the pool
 * positions with z^ >= k^ (the head's emission key); the finish kernel
 * rescores every emitted position on the bf16 keys and keeps those with
 * z >= k^ + eps, which are all the pool positions with such a logit; when
 * they are fewer than K it rescans the head's bf16 keys (slow, exact).
 * workspace: tsa_decode_q8_workspace_size() bytes, same rules as
 * sparse_attn_decode's (a q8 workspace is not interchangeable with a plain
 * one). */
TSA_API size_t tsa_decode_q8_workspace_size(int B, int Hq, int Hkv, int d, int64_t l_cap,
                                            int K, int n_init, int n_recent);

TSA_API int sparse_attn_decode_q8(const void* q, const tsa_kv* kv, const tsa_kq8* kq,
                                  int n_new, const int32_t* lens, int B, int Hq, int Hkv,
                                  int d, int K, int n_init, int n_recent, float scale,
                                  float* out, float* lse_out, int32_t* topk_idx,
                                  float* topk_score, void* workspace, size_t ws_bytes,
                                  void* stream);

/* tsa_workspace_status -- the device-side status of a decode or ReTopK
 * workspace.  The pages have no counterpart: this is error reporting.
 *
 * Synchronises `stream` (the only entry point that does), then reads the
 * workspace's status word (written by the kernels of earlier calls on it):
 *   TSA_OK               nothing was flagged;
 *   TSA_ERR_TIMEOUT      a bounded wait expired in some call (its outputs,
 *                        and those of every later call, are NaN);
 *   TSA_ERR_DEVICE_CHECK a device-side check flagged bad input (a sequence
 *                        length outside [0, l_cap], clamped).
 * With clear != 0 the word is reset to zero, so the next call runs normally
 * (the rest of the workspace needs no reset).  workspace: the pointer given
 * to sparse_attn_decode or retopk_step (256-byte aligned). */
TSA_API int tsa_workspace_status(void* workspace, int clear, void* stream);

/* tsa_inject_scan_stall -- fault injection for tests of the error path.
 *
 * Makes the next sparse_attn_decode or retopk_step call on this thread
 * wait at most wait_limit_ns (1 .. 1e9) in its key scan, and makes the
 * scan's first CTA withhold the copy of its first key tile, so that the
 * bounded waits of that CTA expire: the call then reports TSA_ERR_TIMEOUT
 * through tsa_workspace_status, with NaN outputs, and the device stays
 * usable.  One call only; 0 cancels a pending injection.  Nothing is
 * launched by this function. */
TSA_API int tsa_inject_scan_stall(long long wait_limit_ns);

/* sparse_attn_decode_shard -- one shard of a sequence split over devices
 * ([RA] Eq. 4-5: partial attentions over disjoint sets merge exactly).
 *
 * The cache `kv` (B = 1) holds positions [pos_offset, pos_offset +
 * shard_len) of a sequence of global_len positions, local row i being global
 * position pos_offset + i.  For each query head this computes, over the
 * shard's rows, what sparse_attn_decode computes over a whole cache, with the
 * static window taken in global positions ([0, n_init) u [global_len -
 * n_recent, global_len), met by the shard in a prefix and a suffix of it):
 *   topk_idx / topk_score: the shard's local top-K outside the window, as
 *     LOCAL row indices (add pos_offset for global positions) and logits;
 *   out / lse_out: attention over the shard's window rows and that local
 *     top-K (Eq. 4-5).
 * A split decode step: every shard runs this, the shards exchange their K
 * (logit, global position) pairs per head, every shard keeps the pairs of the
 * global top-K that it holds and runs attend_set over them plus its window
 * rows, and lse_merge folds the shards' (out, lse).
 * q: bf16 [Hq][128]; out fp32 [Hq][128]; lse_out fp32 [Hq] or NULL;
 * topk_idx int32 [Hq][K] or NULL; topk_score fp32 [Hq][K] or NULL.
 * 0 <= shard_len <= kv->l_cap, pos_offset >= 0, pos_offset + shard_len <=
 * global_len.  workspace: tsa_decode_workspace_size(1, Hq, Hkv, d, l_cap, K,
 * n_init, n_recent) bytes, as for sparse_attn_decode. */
TSA_API int sparse_attn_decode_shard(const void* q, const tsa_kv* kv, int64_t shard_len,
                                     int64_t pos_offset, int64_t global_len, int Hq, int Hkv,
                                     int d, int K, int n_init, int n_recent, float scale,
                                     float* out, float* lse_out, int32_t* topk_idx,
                                     float* topk_score, void* workspace, size_t ws_bytes,
                                     void* stream);

/* attend_set -- attention over a given set of rows ([RA] Eq. 3: the partial
 * o_Omega over a set Omega chosen elsewhere).
 *
 * For each sequence b and query head h: z_i = scale * q_h . k_i for the
 * counts[b][h] positions positions[b][h][0 .. counts-1] (rows of this
 * cache), out = softmax(z) . V over them, lse = log sum e^z (an empty set:
 * out 0, lse -inf).  No window is added; each listed row counts once per
 * listing.  q: bf16 [B][Hq][128]; positions: int32 [B][Hq][M] (device),
 * entries past counts ignored; counts: int32 [B][Hq] (device), 0..M;
 * out fp32 [B][Hq][128]; lse_out fp32 [B][Hq] or NULL.  A position outside
 * [0, kv->l_cap) is never read: it is left out and reported as
 * TSA_ERR_DEVICE_CHECK by tsa_workspace_status.  1 <= M <= 2^24.
 * workspace: tsa_attend_set_workspace_size(B, Hq, M) bytes, 256-byte
 * aligned, zero-filled before its first use (calls leave it ready). */
TSA_API size_t tsa_attend_set_workspace_size(int B, int Hq, int M);
TSA_API int attend_set(const void* q, const tsa_kv* kv, int B, int Hq, int Hkv, int d,
                       const int32_t* positions, const int32_t* counts, int M, float scale,
                       float* out, float* lse_out, void* workspace, size_t ws_bytes,
                       void* stream);

/* ------------------------------------------------------------------ */
/* lse_merge -- [RA] Eq. 4-5 on precomputed partials.
 *
 * For each row r < rows, merges two attention partials over disjoint key
 * sets, each given as (o, lse) with lse = log sum e^z over its set:
 *   lse = log(e^lse_a + e^lse_b)
 *   o   = e^(lse_a - lse) o_a + e^(lse_b - lse) o_b
 * A partial with lse = -inf is empty and gets weight 0; if both are empty
 * the row's o is 0 and lse is -inf.
 * o_a, o_b, o_out: fp32 [rows][d]; lse_a, lse_b, lse_out: fp32 [rows]
 * (device).  o_out may alias o_a or o_b; lse_out may alias lse_a or lse_b.
 * d: 1 .. 1024. */
TSA_API int lse_merge(const float* o_a, const float* lse_a, const float* o_b,
              const float* lse_b, float* o_out, float* lse_out, int rows,
              int d, void* stream);

/* ------------------------------------------------------------------ */
/* ReTopK -- [RTK] per-head query-support reuse for one sequence.
 *
 * State (per layer): for every query head a FIFO of C entries (qbar, S):
 * qbar a normalised past query (fp32 [128]), S its final top-K positions.
 * Step t (counted from 0 by the state) with query q and cache length L_t:
 *   qbar_t = q / |q|;  rho_c = qbar_t . qbar_c  for the C entries
 *   exact path if max rho < tau  or  t % T_r == 0:
 *       S_t = exact top-K of all L_t keys (no window)
 *   reuse path otherwise:
 *       R_t = the R entries of largest rho (ties: older entry first)
 *       A_t = Unique(U_{c in R_t} S_c  u  [L_t - W, L_t))      (ascending)
 *       S_t = top-K of A_t by e_i = scale * q . k_i (ties: smaller
 *             position); all of A_t when |A_t| <= K
 *   out = softmax(e_{S_t}) . V_{S_t}   (no window merge)
 *   push (qbar_t, S_t) into the FIFO, evicting the oldest entry.
 *
 * The state lives in caller-owned device memory of retopk_state_size()
 * bytes (256-byte aligned); the opaque host handle holds sizes, pointers,
 * the step counter and the FIFO head. */
typedef struct tsa_retopk tsa_retopk;

TSA_API size_t retopk_state_size(int Hq, int d, int K, int C);

/* Create a handle over `state_mem`.  Hyper-parameters: 1 <= R <= C <= 64,
 * K >= 1, W >= 0, T_r >= 1, R*K + W <= 8192, tau any float (tau > 1: always
 * exact; tau <= -1 with a large T_r: reuse after step 0).  max_len bounds
 * every later L_t and sizes the workspace: the candidate union is a bitmap
 * over the positions with a second level of one bit per 32-bit word; one CTA
 * keeps both in shared memory up to 1.5 M positions (192 KiB), and for
 * longer caches the bitmap lives in the workspace (max_len / 8 bytes per
 * query head) with only the second level in shared memory: max_len <=
 * 50331648.  Nothing is launched. */
TSA_API int retopk_create(tsa_retopk** st, int Hq, int Hkv, int d, int K, int C,
                  int R, int W, float tau, int T_r, int64_t max_len,
                  void* state_mem, size_t state_bytes);

/* Fill the FIFO from the last C prefill queries: prefill_q bf16 [C][Hq][128]
 * (row c is the query of prefill position L0-C+c; c = 0 is the oldest
 * entry) and their supports prefill_supports int32 [C][Hq][K] with sizes
 * prefill_counts int32 [C][Hq] (entries past a count are ignored).  All
 * device pointers.  Resets the step counter to 0. */
TSA_API int retopk_init(tsa_retopk* st, const void* prefill_q,
                const int32_t* prefill_supports, const int32_t* prefill_counts,
                void* stream);

/* Workspace needed by retopk_step for caches up to max_len keys: device
 * scratch, 256-byte aligned, zero-filled before the handle's first step.
 * Like the decode workspace it keeps per-head state that speeds up the next
 * step (never its result), so one workspace serves one handle. */
TSA_API size_t retopk_workspace_size(const tsa_retopk* st);

/* One decode step (see above).  q: bf16 [Hq][128]; kv: this layer's cache
 * with B = 1 (lens are the host value `len`, 1 <= len <= min(kv->l_cap,
 * max_len)); out: fp32 [Hq][128].  Optional outputs (NULL to skip):
 *   support_out int32 [Hq][K] (S_t, unspecified order, -1 padded; a copy
 *     of the FIFO entry this step pushed),
 *   path_out int32 [Hq] (1 exact, 0 reuse),
 *   mcand_out int32 [Hq] (|A_t| on the reuse path, len on the exact path),
 *   cand_out int32 [Hq][R*K+W] (A_t ascending, -1 padded; reuse heads only),
 *   lse_out fp32 [Hq].
 * Advances the step counter and the FIFO head.  (The same as
 * retopk_step_batched with one handle.)  If a bounded wait of the
 * step's key scan expires (see tsa_workspace_status), out and lse are NaN
 * and the FIFO entry is not rewritten (it keeps an older entry): restore
 * the state memory and counters from a copy taken before the step to redo
 * it. */
TSA_API int retopk_step(tsa_retopk* st, const void* q, const tsa_kv* kv, int64_t len,
                float scale, float* out, int32_t* support_out,
                int32_t* path_out, int32_t* mcand_out, int32_t* cand_out,
                float* lse_out, void* workspace, size_t ws_bytes,
                void* stream);

/* retopk_prefill_supports -- the FIFO's initial supports ([RTK] method
 * section 1: the cache starts from the last C prefill queries; the same exact
 * prefill-query top-K is [RA]'s attention-aware index, phase 1).
 *
 * For the last C prefill queries of one sequence -- query c (0 = oldest) at
 * position p_c = L0 - C + c -- and every query head h: the exact top-K of
 * z_i = scale * q_{c,h} . k_i over the causal prefix i in [0, p_c] (no
 * window), ties to the smaller position.  One call runs one key scan and one
 * selection for all C * Hq (query, head) pairs: the queries are a batch of C
 * sequences that all read this sequence's cache (each still reads its own
 * prefix of keys).
 * q_prefill:  bf16 [C][Hq][128] (device), the layout retopk_init takes
 * kv:         the sequence's cache (B = 1), L0 <= kv->l_cap, C <= L0
 * supports:   int32 [C][Hq][K] (device): the positions, unspecified order,
 *             padded with -1 past min(K, p_c + 1)
 * counts:     int32 [C][Hq] (device) or NULL: min(K, p_c + 1)
 * workspace:  retopk_prefill_workspace_size() bytes, 256-byte aligned,
 *             zero-filled before its first use; like the decode workspace
 *             it keeps per-head emission state between calls (a first call
 *             emits every key and costs more).
 * Limits as sparse_attn_decode with B = C (C * Hkv <= 512, C * Hq <= 65535).
 * Device-detected errors: tsa_workspace_status. */
TSA_API size_t retopk_prefill_workspace_size(int C, int Hq, int Hkv, int d, int64_t l_cap,
                                             int K);
TSA_API int retopk_prefill_supports(const void* q_prefill, const tsa_kv* kv, int64_t L0, int C,
                                    int Hq, int Hkv, int d, int K, float scale,
                                    int32_t* supports, int32_t* counts, void* workspace,
                                    size_t ws_bytes, void* stream);

/* retopk_step_batched -- one decode step of n sequences at once, each with
 * its own ReTopK state (continuous batching: any set of initialised handles,
 * in any order, may form a call; a sequence joins after retopk_init on its
 * handle and retires by no longer being passed).
 *
 * handles: n distinct handles (1 <= n <= 64) with equal Hq, Hkv, K, C, R, W,
 *   tau, T_r and max_len; each keeps its own step counter and FIFO head
 *   (both advance by one).
 * q: bf16 [n][Hq][128]; kv: the n sequences' caches in call order (B = n:
 *   contiguous [n][Hkv][l_cap][128], or paged with page-table rows in call
 *   order); lens: host int64 [n], 1 <= lens[b] <= min(l_cap, max_len).
 * Per sequence b everything is as for retopk_step (its path decisions, A_t,
 * S_t, output and FIFO push use only its own state and cache).  Outputs are
 * retopk_step's with a leading [n] (out fp32 [n][Hq][128]; support_out int32
 * [n][Hq][K]; path_out, mcand_out int32 [n][Hq]; cand_out int32
 * [n][Hq][R*K+W]; lse_out fp32 [n][Hq]; optional ones NULL to skip).
 * workspace: retopk_batched_workspace_size(handles[0], n_max) bytes for any
 *   n <= n_max, 256-byte aligned, zero-filled before its first use; it keeps
 *   per-row emission state (only the cost depends on it).  Its layout follows
 *   from ws_bytes (the most sequences it holds), so pass the same ws_bytes
 *   with a workspace on every call. */
TSA_API size_t retopk_batched_workspace_size(const tsa_retopk* proto, int n_max);
TSA_API int retopk_step_batched(tsa_retopk* const* handles, int n, const void* q,
                                const tsa_kv* kv, const int64_t* lens, float scale, float* out,
                                int32_t* support_out, int32_t* path_out, int32_t* mcand_out,
                                int32_t* cand_out, float* lse_out, void* workspace,
                                size_t ws_bytes, void* stream);

/* Host-side counters of the handle (for checkpointing). */
TSA_API int retopk_get_counters(const tsa_retopk* st, int64_t* t, int32_t* fifo_head);
TSA_API int retopk_set_counters(tsa_retopk* st, int64_t t, int32_t fifo_head);

/* Free the host handle only; the state memory belongs to the caller. */
TSA_API int retopk_destroy(tsa_retopk* st);

#ifdef __cplusplus
}
#endif
#endif
