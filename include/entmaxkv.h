/*
 * entmaxkv.h -- C ABI of libentmaxkv, the GB300 (sm_103a) EntmaxKV decode step.
 *
 * The method is "EntmaxKV: Support-Aware Decoding for Entmax Attention"
 * (gist.science technical summary; arXiv abstract on the mlsanity.com index
 * page). A decode step scores the pages of a paged KV cache from per-page key
 * metadata (summary §2A), selects candidate pages (§2B: top-k by a bounding-
 * box bound, or a Gaussian estimate τ̂ of the entmax threshold with margin Δ),
 * and runs exact α-entmax attention over the selected pages only (§2C):
 *
 *   s_i = q·k_i/√d,  z_i = (α−1)·s_i,  p_i = [z_i − τ]_+^{1/(α−1)},  Σ p_i = 1,
 *   o = Σ_i p_i v_i.
 *
 * Conventions for every call:
 *   - Pointers marked (device) point to CUDA device memory the CALLER owns
 *     and keeps alive until the work queued on `stream` has finished. The
 *     library allocates nothing and keeps no state between calls.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). All work is queued asynchronously on it; outputs are valid
 *     once the stream has been synchronised. No call synchronises.
 *   - Argument errors are found on the host and returned at once; nothing is
 *     queued then. Errors found by a kernel (a block-table entry out of
 *     range, an append past the block table, ...) are OR-ed as
 *     ENTMAXKV_DEV_* bits into the caller's device status word
 *     (entmaxkv_cache.status, may be NULL). Nothing prints, traps or throws.
 *   - No kernel spins: kernels never wait on other kernels or on flags. The
 *     entmax split-K blocks add their sums into `out` with float atomics, so
 *     the last bits of `out` depend on the order blocks finish in; the
 *     softmax split-K combine uses a "last block to finish combines" counter.
 */
#ifndef ENTMAXKV_H
#define ENTMAXKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ENTMAXKV_VERSION 4

/* Return codes of every call. */
typedef enum {
  ENTMAXKV_OK = 0,
  ENTMAXKV_ERR_INVALID_ARG = 1,       /* a NULL, negative or inconsistent argument   */
  ENTMAXKV_ERR_UNSUPPORTED = 2,       /* a valid but unimplemented shape/dtype/alpha */
  ENTMAXKV_ERR_WORKSPACE_TOO_SMALL = 3,
  ENTMAXKV_ERR_CUDA = 4               /* a CUDA launch or memset failed              */
} entmaxkv_status;

/* Bits a kernel ORs into the device status word. */
#define ENTMAXKV_DEV_BAD_PAGE_TABLE  0x1u  /* block-table entry outside [0, num_phys_pages): page skipped   */
#define ENTMAXKV_DEV_CAPACITY        0x2u  /* append past max_pages_per_seq, or Gaussian cap overflow       */
#define ENTMAXKV_DEV_TAUHAT_NOCONV   0x4u  /* the τ̂ solve stopped at its iteration limit                    */
#define ENTMAXKV_DEV_CAND_OVERFLOW   0x8u  /* informational: the exact-τ solve used its slow full-scan path */
#define ENTMAXKV_DEV_TAU_NOCONV      0x10u /* the exact-τ solve stopped at its iteration limit              */
#define ENTMAXKV_DEV_BAD_SEQ_ID      0x20u /* a seq_ids entry outside [0, max_seqs): that sequence skipped  */
#define ENTMAXKV_DEV_TIMEOUT         0x40u /* a bounded wait on an asynchronous copy ran out (about
                                              4M polls); the block waited for its copies in flight,
                                              stopped early, and its results are incomplete             */

/* KV storage types. */
#define ENTMAXKV_F32  0
#define ENTMAXKV_BF16 1

/* Page-selection policies (summary §2B) and the in-run baselines (§4). */
#define ENTMAXKV_POLICY_FULL     0  /* every page: full-cache α-entmax                      */
#define ENTMAXKV_POLICY_TOPK     1  /* the k = budget/page_size pages with the largest bound */
#define ENTMAXKV_POLICY_GAUSSIAN 2  /* pages whose estimated max clears τ̂ − Δ               */
#define ENTMAXKV_POLICY_SOFTMAX  3  /* full-cache softmax (FlashDecoding-style baseline)     */
#define ENTMAXKV_POLICY_SOFTMAX_TOPK 4  /* softmax over the top-k pages (the softmax side of the
                                           summary's comparison at equal budget, §1/§4)     */

/* Decode flags. */
#define ENTMAXKV_FLAG_DENSE_V 0x1u  /* read every selected V page even where all p_i = 0
                                       (the dense full-cache entmax baseline); without it a
                                       page whose scores all sit at or below τ is skipped,
                                       which is exact since its weights are 0.            */
#define ENTMAXKV_FLAG_EXACT_DELTA 0x2u  /* also compute the exact dropped mass
                                         δ = 1 − Σ_{i kept} p_i^full (summary §3: the
                                         mass of the full-cache α-entmax outside the
                                         kept pages) by a full-cache pass over every
                                         K page; a diagnostic, not for timed steps.
                                         The workspace must then hold
                                         entmaxkv_workspace_bytes_flags(...) bytes. */

#define ENTMAXKV_FLAG_EXPIRE_WAITS 0x100u  /* diagnostic, for testing the device-side
                                          timeout path: the Gaussian page scorer's
                                          waits for its staged copies give up at once
                                          instead of polling, as a wait that runs out
                                          of its bound does. The scorer then raises
                                          ENTMAXKV_DEV_TIMEOUT, waits (bounded) for
                                          the copies it issued and stops; the decode
                                          completes with every page unscored, so out
                                          is 0, n_sel 0 and tau NaN. Never set it for
                                          real work.                              */

/* What the delta output of a decode holds (entmaxkv_delta_kind). */
#define ENTMAXKV_DELTA_ZERO      0  /* FULL, SOFTMAX: nothing is dropped            */
#define ENTMAXKV_DELTA_CERTIFIED 1  /* TOPK: an upper bound on the dropped mass      */
#define ENTMAXKV_DELTA_MODEL     2  /* GAUSSIAN: the page model's estimate           */
#define ENTMAXKV_DELTA_EXACT     3  /* any policy with ENTMAXKV_FLAG_EXACT_DELTA     */

/*
 * Cache geometry. Supported: head_dim ∈ {64, 128}; page_size ∈ {16, 32};
 * 1 ≤ group ≤ 8 (query heads per KV head; query head h reads KV head h/group).
 */
typedef struct {
  int32_t num_kv_heads;       /* Hkv                                           */
  int32_t group;              /* g = Hq / Hkv                                  */
  int32_t head_dim;           /* d                                             */
  int32_t page_size;          /* P tokens per page                             */
  int32_t max_seqs;           /* rows of the block table / entries of seq_lens */
  int32_t max_pages_per_seq;  /* row length of the block table                 */
  int32_t num_phys_pages;     /* pages in the K/V pools                        */
  int32_t kv_dtype;           /* ENTMAXKV_F32 or ENTMAXKV_BF16                 */
} entmaxkv_config;

/*
 * The paged cache: caller-owned device buffers (summary §2A: the cache is
 * split into pages; each page keeps k_min/k_max and the mean and variance of
 * its keys). Layouts, row-major:
 *   k_pool, v_pool [num_phys_pages][num_kv_heads][page_size][head_dim]  kv_dtype
 *   kmin, kmax     [num_phys_pages][num_kv_heads][head_dim]             kv_dtype
 *   mean, m2       [num_phys_pages][num_kv_heads][head_dim]             float32
 *       (m2 = Σ (k − mean)² over the page's valid tokens; var = m2 / n_p)
 *   block_table    [max_seqs][max_pages_per_seq] int32: logical page → physical page
 *   seq_lens       [max_seqs] int32 valid tokens per sequence
 *   status         one uint32 the kernels OR ENTMAXKV_DEV_* bits into (may be NULL)
 *   mean_bf16, m2_bf16  [num_phys_pages][num_kv_heads][head_dim] bfloat16, or both NULL:
 *                  round-to-nearest-even copies of mean and m2, which append
 *                  keeps in step. When present, the Gaussian scorer streams
 *                  these instead of the fp32 arrays (half the bytes, summary §4:
 *                  the cost moves to page selection). The fp32 arrays stay the
 *                  ones appends merge into, so no rounding accumulates.
 * Metadata of a page covers its valid tokens only and is written by
 * entmaxkv_append; a partial last page holds n_p = len − P·(pages−1) tokens.
 * Every pool and metadata array starts on a 16-byte boundary (the kernels
 * move whole 16-byte vectors and page slabs); a misaligned pointer is
 * rejected with ENTMAXKV_ERR_INVALID_ARG before any launch.
 */
typedef struct {
  void* k_pool;
  void* v_pool;
  void* kmin;
  void* kmax;
  float* mean;
  float* m2;
  const int32_t* block_table;
  int32_t* seq_lens;
  uint32_t* status;
  void* mean_bf16;
  void* m2_bf16;
} entmaxkv_cache;

/* Library version (ENTMAXKV_VERSION). */
int32_t entmaxkv_version(void);

/* Static text for a return code; never NULL. */
const char* entmaxkv_status_string(int32_t status);

/*
 * Append n_tokens tokens to each of n_seqs sequences (summary §2A: the page
 * metadata the scorers read is maintained as keys are written).
 *   k, v     (device) [n_seqs][num_kv_heads][n_tokens][head_dim], kv_dtype
 *   seq_ids  (device) [n_seqs] distinct sequence rows, or NULL for 0..n_seqs−1
 * For sequence b with old length L, token t goes to logical page (L+t)/P,
 * slot (L+t)%P, through the block table; the caller must have filled the
 * block-table entries of every page being written. Each touched page's
 * kmin/kmax (exact element min/max) and mean/m2 (float32; a partly filled
 * page is merged with the Chan et al. pairwise update) are updated, then
 * seq_lens[seq] += n_tokens. A page past max_pages_per_seq or a block-table
 * entry out of range is skipped and flagged on the device status word.
 * n_tokens == 0 or n_seqs == 0 queues nothing and returns OK.
 */
int32_t entmaxkv_append(const entmaxkv_config* cfg, const entmaxkv_cache* cache,
                        const void* k, const void* v, const int32_t* seq_ids,
                        int32_t n_seqs, int32_t n_tokens, void* stream);

/*
 * Bytes of device workspace entmaxkv_decode needs for n_seqs sequences under
 * `policy` and `budget_tokens`. Returns 0 for invalid arguments.
 */
size_t entmaxkv_workspace_bytes(const entmaxkv_config* cfg, int32_t n_seqs,
                                int32_t policy, int32_t budget_tokens);

/*
 * Workspace bytes for a decode with the given flags: entmaxkv_workspace_bytes
 * for flags without ENTMAXKV_FLAG_EXACT_DELTA; with it, that plus a second
 * region laid out for the full-cache policy. 0 for an invalid configuration.
 */
size_t entmaxkv_workspace_bytes_flags(const entmaxkv_config* cfg, int32_t n_seqs, int32_t policy,
                                      int32_t budget_tokens, uint32_t flags);

/* The ENTMAXKV_DELTA_* kind of the delta output of a decode with this policy
 * and these flags; -1 for an unknown policy. */
int32_t entmaxkv_delta_kind(int32_t policy, uint32_t flags);

/*
 * Copy the cache's device status word (the ENTMAXKV_DEV_* bits the kernels
 * have raised) to *status_out after the work queued on `stream` has finished
 * (this call synchronises the stream). With clear ≠ 0 the word is reset to 0
 * afterwards. Returns ENTMAXKV_ERR_INVALID_ARG when the cache has no status
 * word or status_out is NULL, ENTMAXKV_ERR_CUDA when a CUDA call fails.
 */
int32_t entmaxkv_read_status(const entmaxkv_cache* cache, uint32_t* status_out, int32_t clear,
                             void* stream);

/*
 * Whether the GAUSSIAN policy supports this α (summary §2B.2: the
 * normalisation equation at entmax order α). α ∈ {1.5, 2} use closed forms;
 * any other α > 1 uses fits of the partial moments E[(t + Z)_+^ν] that this
 * call (or the first decode with that α) builds on the host, about 0.1-0.4 s,
 * and caches (the 8 most recently used orders; a caller cycling through more
 * rebuilds on each miss); they must pass a 1e-6 relative check. Returns 1 or
 * 0. Host only: no CUDA call.
 */
int32_t entmaxkv_gaussian_alpha_supported(float alpha);

/*
 * Diagnostic: the fitted J_ν(t) = E[(t + Z)_+^ν], Z ~ N(0, 1), for
 * ν = β − order (β = 1/(α−1); order 0, 1, or 2 when β > 1), at the n points
 * t[i] (host arrays), computed on the host in the float arithmetic the
 * kernels use, into out[i]. Returns ENTMAXKV_ERR_UNSUPPORTED when α has no
 * fits (α ∈ {1.5, 2}, which use closed forms, or fits that fail their check)
 * and ENTMAXKV_ERR_INVALID_ARG for a bad order, count or pointer. Host only.
 */
int32_t entmaxkv_moment_fit_eval(float alpha, int32_t order, const float* t, int32_t n, float* out);

/*
 * One decode step for n_seqs sequences (summary §2A-§2C; δ from §3).
 *   q          (device) [n_seqs][Hq][head_dim], kv_dtype (Hq = Hkv·group)
 *   seq_ids    (device) [n_seqs] sequence rows, or NULL for 0..n_seqs−1
 *   alpha      α > 1; ignored by SOFTMAX and SOFTMAX_TOPK. GAUSSIAN uses closed
 *              forms at α ∈ {1.5, 2} and, at any other α, fits of the partial
 *              moments E[(t + Z)_+^ν] that the first call with that α builds on
 *              the host (about 0.1-0.4 s, cached for later calls). The fits
 *              are checked to 1e-6 relative; an α whose fits fail that check
 *              (outside about [1.14, 6]) returns ENTMAXKV_ERR_UNSUPPORTED.
 *   policy     ENTMAXKV_POLICY_*
 *   budget_tokens  TOPK, SOFTMAX_TOPK: k = budget_tokens / page_size pages (must be ≥ 1);
 *                  GAUSSIAN: a cap in tokens (0 = none; on overflow the pages
 *                  with the largest margin max_h(M̂_p − threshold_h) are kept,
 *                  ties to the lower index, and ENTMAXKV_DEV_CAPACITY is set);
 *                  FULL/SOFTMAX: ignored
 *   margin     Δ in score units (GAUSSIAN)
 *   flags      ENTMAXKV_FLAG_*
 *   workspace  (device) ≥ entmaxkv_workspace_bytes_flags(...) bytes, 256-byte
 *              aligned; contents need no initialisation and are scratch
 *              afterwards. One workspace must not be shared by decodes that
 *              may run concurrently.
 * Outputs (device; any may be NULL except out):
 *   out        [n_seqs][Hq][head_dim] float32
 *   page_ids   [n_seqs][Hkv][page_ids_stride] int32: selected logical page
 *              ids, ascending (FULL/SOFTMAX: every page)
 *   n_sel      [n_seqs][Hkv] int32 selected pages
 *   tau        [n_seqs][Hq] float32: the exact α-entmax threshold over the
 *              kept tokens on the z scale (SOFTMAX, SOFTMAX_TOPK: log Σ exp(s_i)
 *              over the kept tokens); NaN for an empty kept set
 *   delta      [n_seqs][Hq] float32 dropped mass: FULL/SOFTMAX 0; TOPK the
 *              certified bound min(1, Σ_dropped n_p·[(α−1)U_p − τ]_+^β);
 *              GAUSSIAN the page model's estimate of the dropped mass: it
 *              is not certified and can be far below the true dropped mass
 *              (a single outlier token raises a page's true score spread
 *              much more than the per-coordinate variances show); use
 *              ENTMAXKV_FLAG_EXACT_DELTA for the exact value;
 *              SOFTMAX_TOPK the certified bound D/(1 + D) with
 *              D = Σ_dropped n_p·exp(U_p − log Σ_kept exp(s_i));
 *              with ENTMAXKV_FLAG_EXACT_DELTA, for every policy, the exact
 *              max(0, 1 − Σ_{i in the kept pages} p_i^full)
 * page_ids_stride must be ≥ the most pages the policy can select
 * (TOPK, SOFTMAX_TOPK: k; GAUSSIAN: the cap in pages, or max_pages_per_seq; otherwise
 * max_pages_per_seq) when page_ids is not NULL.
 * An empty sequence yields out = 0, tau = NaN, delta = 0, n_sel = 0.
 */
int32_t entmaxkv_decode(const entmaxkv_config* cfg, const entmaxkv_cache* cache,
                        const void* q, const int32_t* seq_ids, int32_t n_seqs,
                        float alpha, int32_t policy, int32_t budget_tokens,
                        float margin, uint32_t flags,
                        void* workspace, size_t workspace_bytes,
                        float* out, int32_t* page_ids, int32_t page_ids_stride,
                        int32_t* n_sel, float* tau, float* delta, void* stream);

/*
 * entmaxkv_decode with CUDA events recorded between its stages, for timing
 * one kernel on the stream it runs on. `events` holds ENTMAXKV_STAGE_EVENTS
 * cudaEvent_t handles (as void*) created by the caller: events[0] is recorded
 * before the first stage and events[i+1] after stage i, where the stages are
 *   0 workspace clear, 1 page scoring (bbox or Gaussian), 2 selection (top-k,
 *   τ̂ + bits, Gaussian cap), 3 pass A (K pages, scores, exact τ),
 *   4 pass B (V pages, output) or the softmax kernel.
 * A stage a policy does not run records back-to-back events. Everything else
 * is as entmaxkv_decode.
 */
#define ENTMAXKV_STAGE_EVENTS 6
int32_t entmaxkv_decode_profiled(const entmaxkv_config* cfg, const entmaxkv_cache* cache,
                                 const void* q, const int32_t* seq_ids, int32_t n_seqs,
                                 float alpha, int32_t policy, int32_t budget_tokens,
                                 float margin, uint32_t flags,
                                 void* workspace, size_t workspace_bytes,
                                 float* out, int32_t* page_ids, int32_t page_ids_stride,
                                 int32_t* n_sel, float* tau, float* delta, void* stream,
                                 void* const* events);

/*
 * Where the decode keeps its intermediate results inside the workspace, so
 * that tests and tools can read the page scores, τ̂ and the selection of the
 * last decode. Offsets are in bytes from the workspace base; a region the
 * policy does not use has offset SIZE_MAX. Layouts:
 *   bbox_u     float [n_seqs][Hq][max_pages_per_seq]   U_p per query head
 *   bbox_uhat  float [n_seqs][Hkv][max_pages_per_seq]  max over the group
 *   gauss_ms   float2 [n_seqs][Hq][max_pages_per_seq]  (m_p, ς_p) = (α−1)(μ_p, σ_p)
 *   tauhat     float [n_seqs][Hq]                      τ̂ on the z scale
 *   sel_bitmap uint32 [n_seqs][Hkv][ceil(max_pages_per_seq/32)]
 *   tauhat_iters int32 [n_seqs][Hq]                    iterations of the τ̂ solve
 */
typedef struct {
  size_t bbox_u, bbox_uhat, gauss_ms, tauhat, sel_bitmap;
  size_t tauhat_iters;
  size_t page_zmax;    /* float [n_seqs][Hkv][cap_pages][group]: max z of each kept page
                          (index = rank in page_ids), SIZE_MAX for SOFTMAX        */
  int32_t cap_pages;   /* most pages one (sequence, KV head) can keep              */
  int32_t splits;      /* most blocks per (sequence, KV head) of the decode kernels
                          (a launch uses fewer on a device with fewer SMs)         */
  size_t total;
  size_t z_scores;     /* float [n_seqs][Hkv][cap_pages][page_size][group]: z = (α−1)·s of
                          every token of each kept page (index = rank in page_ids), −inf
                          past a page's valid tokens; SIZE_MAX for SOFTMAX policies  */
} entmaxkv_workspace_view;

int32_t entmaxkv_workspace_layout(const entmaxkv_config* cfg, int32_t n_seqs,
                                  int32_t policy, int32_t budget_tokens,
                                  entmaxkv_workspace_view* view);

/*
 * Full-cache softmax decode for callers that cannot allocate device memory.
 * No passage of the EntmaxKV pages corresponds to this call: it exists for
 * embedders such as custom allocators' own callbacks, graph-building code
 * that must not allocate, or runtimes whose device memory is owned by someone
 * else, which cannot provide the scratch entmaxkv_decode needs.
 *
 * It runs the same computation as entmaxkv_decode with
 * policy = ENTMAXKV_POLICY_SOFTMAX (out [n_seqs][Hq][head_dim] float32 and
 * lse [n_seqs][Hq] = log Σ exp(s_i), lse may be NULL), but its scratch is a
 * fixed array inside the library of entmaxkv_noalloc_scratch_bytes() bytes
 * (8 MiB), which every GPU that loads the library holds until the process
 * exits. It calls no cudaMalloc/cudaFree and no allocating library routine.
 *   - Shapes whose softmax workspace (entmaxkv_workspace_bytes(cfg, n_seqs,
 *     ENTMAXKV_POLICY_SOFTMAX, 0)) exceeds that size are rejected with
 *     ENTMAXKV_ERR_WORKSPACE_TOO_SMALL before anything is queued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture. The address is kept for the process, so
 *     the library must not be used across a reset of that device
 *     (cudaDeviceReset, or another library resetting the primary context),
 *     after which the array may live elsewhere.
 *   - Every call shares the one array: calls that may overlap on the GPU
 *     (different streams, or different host threads) race and must be
 *     serialised by the caller. The counters the decode relies on are cleared
 *     at the start of each call; the array keeps the last call's partial sums.
 */
size_t entmaxkv_noalloc_scratch_bytes(void);
int32_t entmaxkv_decode_softmax_noalloc(const entmaxkv_config* cfg, const entmaxkv_cache* cache,
                                        const void* q, const int32_t* seq_ids, int32_t n_seqs,
                                        float* out, float* lse, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* ENTMAXKV_H */
