/*
 * asp.h - C ABI of the coverage-selected sparse paged decode library (libasp.so).
 *
 * One decode step of long-context attention reads, for every (request, layer,
 * KV head), only the pages that a coverage rule selects: the smallest set of
 * pages whose estimated attention mass reaches a fraction gamma. Attention then
 * runs over those ragged per-head page lists, with every thread block deriving
 * its own share of the work from the list lengths on the device, so that a
 * whole step can be captured in one CUDA graph with no host-side plan.
 *
 * Sources: the MOIRA abstract on the page "Adaptive DHiSparse: Speculative
 * Decoding over a Load-Adaptive KV Hierarchy" (thelatestinai.com/papers/
 * 2610.13708) defines the coverage rule, the per-(request, layer, KV head,
 * step) page lists and self-planning attention. The page estimate is a
 * Quest-style bound; Quest is named in the abstract on the page "HiSparse:
 * scaling sparse attention decoding with hierarchical KV cache"
 * (scholarbro.com/p/47450-...). The pages print no interface: the calls below
 * are this library's own.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers: every tensor pointer is a DEVICE pointer (cudaMalloc'd or
 *   equivalent) that the caller owns. The library never allocates or frees
 *   memory and never synchronises inside the hot calls (asp_page_summarize,
 *   asp_coverage_select, asp_sparse_decode), so they may be captured into a
 *   CUDA graph. All work is enqueued on `stream`.
 * - bf16 tensors are passed as uint16_t bit patterns.
 * - Errors: arguments are checked on the host before any launch; a bad one
 *   returns a negative asp_status and launches nothing. Problems that only
 *   the device can see (an out-of-range block-table or list entry, a length
 *   beyond the request) set bits in a sticky device error word inside the
 *   workspace; the kernel then skips the offending page or clamps the length
 *   and never traps. Read and clear the word with asp_get_device_error.
 * - Shapes supported: head_dim d in {64, 128}; page_size P in {16, 32, 64};
 *   num_kv_heads Hkv in {1, 2, 4, 8}; GQA group g = Hq / Hkv in {1, 2, 4, 8};
 *   batch * Hkv <= 4096 segments; max_pages <= 1<<20;
 *   batch * Hkv * (max_pages + 128) < 2^31 and num_phys_pages * Hkv * P < 2^31
 *   (int32 page-space and cache-row indices). Anything else returns
 *   ASP_EUNSUPPORTED.
 * - The current CUDA device when a call is made must be the device that owns
 *   the pointers.
 * - Tracing: every call opens an NVTX range named after itself (e.g.
 *   "asp_sparse_decode"), so a profiler that reads NVTX attributes each
 *   kernel to the call that launched it.
 */
#ifndef ASP_H_
#define ASP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ASP_ABI_VERSION 1

typedef enum asp_status {
  ASP_OK = 0,
  ASP_EINVAL = -1,        /* null pointer, bad gamma/budget/scale, inconsistent sizes */
  ASP_EUNSUPPORTED = -2,  /* shape outside the supported set listed above */
  ASP_EWORKSPACE = -3,    /* workspace pointer null, misaligned (256 B) or too small */
  ASP_ECUDA = -4,         /* a CUDA runtime call or kernel launch failed */
  ASP_EDEVICE = -5        /* asp_get_device_error found a non-zero device error word */
} asp_status;

/* Bits of the device error word (see asp_get_device_error). */
#define ASP_DEVERR_PAGE_RANGE 0x1u /* block_table entry outside [0, num_phys_pages): page skipped */
#define ASP_DEVERR_LIST_RANGE 0x2u /* lists entry outside [0, N_b): page skipped */
#define ASP_DEVERR_LEN_RANGE 0x4u  /* lens[b,h] outside [0, N_b]: clamped */
#define ASP_DEVERR_SEQ_RANGE 0x8u  /* seq_lens[b] outside [0, max_pages*P]: clamped */
#define ASP_DEVERR_TIMEOUT 0x10u   /* a bounded on-chip wait ran out: the kernel stopped early */

/* A cudaStream_t, passed as an opaque pointer. NULL is the legacy default stream. */
typedef void* asp_stream;

/*
 * Paged KV cache of ONE layer, plus its page summaries.
 *
 *   k_cache, v_cache : bf16 [num_phys_pages, Hkv, P, d]. The (page, head) block
 *                      of P*d values is contiguous. Only asp_page_summarize in
 *                      APPEND mode writes them.
 *   summaries        : bf16 [batch, Hkv, max_pages, 2, d], in LOGICAL page
 *                      order: entry (b, h, p) summarises logical page p < N_b
 *                      of request b for KV head h; row 0 is the channel
 *                      minimum of K over the page's valid tokens, row 1 the
 *                      maximum. Each (request, KV head) segment's summaries
 *                      are one contiguous run, so the estimate pass streams
 *                      them sequentially. Written by asp_page_summarize, read
 *                      by asp_coverage_select.
 *   block_table      : int32 [batch, max_pages]; entry (b, p) is the physical
 *                      page holding logical page p of request b. Shared by all
 *                      heads and layers. Only entries p < N_b are read.
 *   seq_lens         : int32 [batch]; T_b, the tokens of request b (counting the
 *                      token being decoded). N_b = ceil(T_b / P) pages; the last
 *                      page is partial when T_b % P != 0.
 *   query head h uses KV head h / g (the group's heads are contiguous).
 */
typedef struct asp_paged_kv {
  uint16_t* k_cache;
  uint16_t* v_cache;
  uint16_t* summaries;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t batch;          /* B */
  int32_t num_q_heads;    /* Hq */
  int32_t num_kv_heads;   /* Hkv */
  int32_t head_dim;       /* d */
  int32_t page_size;      /* P (tokens per page) */
  int32_t max_pages;      /* columns of block_table and of the page lists */
  int32_t num_phys_pages; /* rows of k_cache / v_cache */
} asp_paged_kv;

/* Library ABI version (ASP_ABI_VERSION of the build). */
int32_t asp_abi_version(void);

/* Human-readable name of a status code (static string). */
const char* asp_status_string(asp_status status);

/*
 * Workspace bytes needed by asp_coverage_select / asp_sparse_decode /
 * asp_page_summarize for this shape on the CURRENT device (the decode grid
 * is sized from its SM count). Writes the size to *bytes. The workspace is a
 * caller-owned device buffer, 256-byte aligned, that must be zeroed once with
 * asp_workspace_init before first use. It holds the device error word,
 * per-call scratch (page scores, the decode's partial results) that every
 * call rewrites before reading, and one arrival count per segment that the
 * decode leaves at zero when it ends, so graph replay is safe. Calls that
 * share one workspace must be ordered on one stream; after a device error
 * (asp_get_device_error non-zero) zero it again with asp_workspace_init.
 */
asp_status asp_workspace_size(const asp_paged_kv* kv, size_t* bytes);

/* Zeroes the whole workspace, device error word included (async on `stream`). */
asp_status asp_workspace_init(void* ws, size_t ws_bytes, asp_stream stream);

/*
 * Page summaries: channel-wise min and max of K per (page, KV head).
 * Definition: the Quest page summary used by the estimate of the coverage
 * rule (MOIRA abstract; Quest as named in the HiSparse abstract).
 *
 * mode ASP_SUMMARIZE_BULK (0): for every request b and logical page p < N_b,
 *   recompute summaries[b, h, p] from the valid tokens (positions < T_b) of
 *   physical page block_table[b, p]. k_new / v_new must be NULL.
 * mode ASP_SUMMARIZE_APPEND (1): seq_lens already count one new token per
 *   request (T_b >= 1). Writes k_new[b,h,:] / v_new[b,h,:] (bf16 [B, Hkv, d])
 *   into slot (T_b-1) % P of page (T_b-1) / P of k_cache / v_cache, and folds
 *   the new key into summaries[b, h, (T_b-1) / P] (a fresh page, slot 0, takes
 *   the key as both its min and max). Idempotent, so replaying it is safe.
 * Requests with T_b == 0 are skipped. Out-of-range table entries set
 * ASP_DEVERR_PAGE_RANGE and skip the page.
 */
#define ASP_SUMMARIZE_BULK 0
#define ASP_SUMMARIZE_APPEND 1
asp_status asp_page_summarize(const asp_paged_kv* kv, int32_t mode,
                              const uint16_t* k_new, const uint16_t* v_new,
                              void* ws, size_t ws_bytes, asp_stream stream);

/*
 * Coverage selection (MOIRA abstract: a coverage rule keeps the smallest set
 * of pages whose estimated attention mass reaches gamma, per request, layer,
 * KV head and step).
 *
 * For each segment (b, kv head h), with g query heads q[b, h*g .. h*g+g-1]:
 *   score  s[p] = (1/sqrt(d)) * max over the group of
 *                 sum_i max(q_i * min_pi, q_i * max_pi)        (fp32)
 *   mass   softmax of s over the N_b pages
 *   rank   score descending, ties to the lower logical page id
 *   keep   the smallest prefix of the ranking whose mass reaches gamma
 *          (gamma >= 1 keeps all N_b pages); budget > 0 instead keeps the
 *          top min(budget, N_b) pages (fixed-budget comparison mode).
 * q      : fp32 [B, Hq, d].
 * gamma  : in (0, 1]; ignored when budget > 0.
 * lists  : int32 [B, Hkv, max_pages] out; row (b,h) receives the kept logical
 *          page ids in ascending order; entries past lens[b,h] are untouched.
 * lens   : int32 [B, Hkv] out; the kept count (0 only when T_b == 0).
 * Masses are summed in 64-bit fixed point, so the result is deterministic.
 * Reads summaries, seq_lens and q only (not block_table or the K/V pages):
 * run asp_page_summarize after any change to the cache first.
 */
asp_status asp_coverage_select(const asp_paged_kv* kv, const float* q, float gamma,
                               int32_t budget, int32_t* lists, int32_t* lens,
                               void* ws, size_t ws_bytes, asp_stream stream);

/*
 * How asp_coverage_select (append = 0) or asp_coverage_select_append
 * (append = 1) runs this shape on the CURRENT device: *kernels receives the
 * number of kernels one call launches, *cluster_ctas the CTAs per segment of
 * the one-pass cluster kernel (0: a score pass, then one select CTA per
 * segment). Segments of 64 to 8192 pages take the cluster kernel when the
 * device runs all of its clusters at once: a cluster of 1, 2 or 4 CTAs per segment
 * streams the segment's summaries, keeps the scores on chip and selects
 * through distributed shared memory. Both paths compute the same scores
 * and select the same pages. Launches nothing.
 */
asp_status asp_select_plan(const asp_paged_kv* kv, float gamma, int32_t budget, int32_t append,
                           int32_t* kernels, int32_t* cluster_ctas);

/*
 * APPEND and coverage selection in one pass: the same result as
 * asp_page_summarize(kv, ASP_SUMMARIZE_APPEND, k_new, v_new, ...) followed by
 * asp_coverage_select(kv, q, gamma, budget, lists, lens, ...), with the
 * append done inside the score kernel (no separate launch per layer and
 * step). The score kernel's warp that streams a segment's last page first
 * writes the new token's K and V rows into slot (T_b-1) % P of page
 * (T_b-1) / P and folds the key into that page's summary, then reads it.
 * k_new, v_new : bf16 [B, Hkv, d], 16-byte aligned. seq_lens already count
 * the new token; requests with T_b == 0 are skipped. Idempotent, like APPEND.
 * Errors and outputs as for the two calls it replaces.
 */
asp_status asp_coverage_select_append(const asp_paged_kv* kv, const uint16_t* k_new,
                                      const uint16_t* v_new, const float* q, float gamma,
                                      int32_t budget, int32_t* lists, int32_t* lens, void* ws,
                                      size_t ws_bytes, asp_stream stream);

/*
 * Page scores alone: the estimate that asp_coverage_select ranks (MOIRA
 * abstract: "estimated attention mass" per page; the Quest bound as named in
 * the HiSparse abstract), for diagnostics such as the captured mass of a
 * fixed page budget. For each segment (b, kv head h) and page p < N_b:
 *   scores[b, h, p] = (1/sqrt(d)) * max over the group of
 *                     sum_i max(q_i * min_pi, q_i * max_pi)        (fp32)
 * q      : fp32 [B, Hq, d], 16-byte aligned.
 * scores : fp32 [B, Hkv, max_pages] out; entries p >= N_b are untouched.
 * Runs the same kernel as asp_coverage_select's first pass; the workspace
 * supplies only the device error word.
 */
asp_status asp_page_scores(const asp_paged_kv* kv, const float* q, float* scores, void* ws,
                           size_t ws_bytes, asp_stream stream);

/*
 * Self-planning sparse attention (MOIRA abstract: each thread block derives
 * its own share of the work from the list lengths, so the step stays inside
 * the CUDA graph).
 *
 * For each query head h of segment (b, h/g), exact softmax attention over the
 * valid tokens of the listed pages:
 *   out[b,h,:] = sum_t softmax_t(sm_scale * q[b,h].k_t) v_t
 *   lse[b,h]   = log sum_t exp(sm_scale * q[b,h].k_t)
 * One kernel launch: a fixed number of CTAs (one per SM); each loads the
 * lengths, splits the concatenated lists by weight (a list's first page
 * weighs more than the others) and attends over its slice. A CTA whose slice
 * holds a whole segment writes out/lse itself; otherwise it leaves a partial
 * (max, sum, unnormalised output) in the workspace, and the last CTA of the
 * segment to finish combines its partials by log-sum-exp, in CTA order. A
 * segment with lens 0 gets out = 0, lse = -inf.
 * K/V are bf16; the products run on tensor cores with fp32 accumulation and
 * the probabilities are rounded to bf16 for the P.V product.
 * lists, lens : as written by asp_coverage_select (any order within a list).
 * out : fp32 [B, Hq, d]; lse : fp32 [B, Hq] (natural log).
 */
asp_status asp_sparse_decode(const asp_paged_kv* kv, const float* q,
                             const int32_t* lists, const int32_t* lens, float sm_scale,
                             float* out, float* lse,
                             void* ws, size_t ws_bytes, asp_stream stream);

/*
 * asp_coverage_select without a workspace. The paper has no counterpart: this
 * entry point exists for callers that cannot allocate device memory, such as
 * an engine that owns all GPU memory through its own pool and passes plugins
 * only their input and output buffers, or a loop that must not allocate once
 * running. It computes exactly what asp_coverage_select computes (same
 * kernels, same arguments and outputs) and calls no allocating routine.
 *
 * Its scratch (the per-page scores) is a fixed array inside libasp.so that
 * every GPU loading the library holds until exit: 4 MiB + 256 B. Shapes with
 * batch * num_kv_heads * max_pages > ASP_NOALLOC_MAX_SCORES are rejected with
 * ASP_EUNSUPPORTED before any device work. The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress with that device
 * current); make that first call before any stream capture. All calls share
 * the array and it keeps the last call's contents; calls that overlap on the
 * GPU (other streams, other host threads) race on it, so serialise them.
 * dev_error: optional device word; device-detected range problems are OR-ed
 * into it as ASP_DEVERR_* bits and the caller clears it. With NULL they go to
 * a spare word inside the library's array that no call reads back: device
 * error bits are then discarded.
 */
#define ASP_NOALLOC_MAX_SCORES (1u << 20)
asp_status asp_coverage_select_noalloc(const asp_paged_kv* kv, const float* q, float gamma,
                                       int32_t budget, int32_t* lists, int32_t* lens,
                                       uint32_t* dev_error, asp_stream stream);

/*
 * Synchronises `stream`, copies the device error word into *code_out
 * (0 = none; else a mask of ASP_DEVERR_* bits), clears it and returns
 * ASP_EDEVICE if it was non-zero, else ASP_OK. After an error, call
 * asp_workspace_init before reusing the workspace. Not capturable.
 */
asp_status asp_get_device_error(void* ws, uint32_t* code_out, asp_stream stream);

/*
 * Self-test of failure detection (the pages have no counterpart). Every
 * on-chip wait in this library is bounded: after 2 s it gives up, sets
 * ASP_DEVERR_TIMEOUT in the device error word and the kernel returns, so a
 * stuck copy never hangs the GPU. This call launches one small kernel whose
 * thread waits, through the same bounded wait, on a shared-memory barrier
 * that nothing completes: about 2 s later it sets the bit and returns, with
 * nothing in flight. Read the result with asp_get_device_error; the context
 * stays usable. ws: an initialised workspace (256-byte aligned, >= 256 B).
 */
asp_status asp_selftest_wait_timeout(void* ws, size_t ws_bytes, asp_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* ASP_H_ */
