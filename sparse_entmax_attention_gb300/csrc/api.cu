// api.cu -- the extern "C" entry points of libentmaxkv: argument checks,
// workspace layout and the launch chain of one decode step.
#include <math.h>
#include <string.h>

#include <atomic>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace ekv {

// The workspace is laid out for at most this many decode blocks per launch,
// whatever the device; a launch uses one wave of 2 blocks per SM of the
// current device, capped at the layout's count.
constexpr int kLayoutBlocks = 2048;

// Streaming multiprocessors of the current device, queried once per device
// (0 when the query fails).
constexpr int kMaxDevices = 64;
static std::atomic<int> g_sms[kMaxDevices];

static int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = g_sms[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 0;
  g_sms[dev].store(n, std::memory_order_relaxed);
  return n;
}

// The driver's tensor-map encoder, looked up once through the runtime.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<void*> fn{nullptr};
  void* f = fn.load(std::memory_order_acquire);
  if (f) return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !f)
    return nullptr;
  fn.store(f, std::memory_order_release);
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// The bf16 V pool [nphys][Hkv][P][D] as a 3-D tensor (dim, KV head · token,
// page) read in boxes of 64 dims × P tokens × 1 page with 128-byte swizzle:
// one box per 64 dims of a (page, KV head) slab. The pool is 16-byte aligned
// (checked with the cache).
cudaError_t make_v_map(CUtensorMap* map, const void* v_pool, int nphys, int Hkv, int P, int D) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hkv * P, (cuuint64_t)nphys};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * P * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)P, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v_pool), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

struct Layout {
  size_t zmax, cnt_a, cnt_b, cand_cnt, kept_mass, dbar, bitmap, ctrl_end;
  size_t tauhat, tau_ws, nsel_ws, sel_list, sel_pp, vlist, vcount, bbox_u, bbox_uhat, gauss_ms, cand, z, pmax, partial, diag, mslot;
  size_t total;
  int splits, cap_pages, words, kpages, gcap, pstride, mslots;
};

static size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

static int check_config(const entmaxkv_config* c) {
  if (!c) return ENTMAXKV_ERR_INVALID_ARG;
  if (c->num_kv_heads < 1 || c->group < 1 || c->max_seqs < 1 || c->max_pages_per_seq < 1 ||
      c->num_phys_pages < 1 || c->num_kv_heads > 65535)
    return ENTMAXKV_ERR_INVALID_ARG;
  if (c->kv_dtype != ENTMAXKV_F32 && c->kv_dtype != ENTMAXKV_BF16) return ENTMAXKV_ERR_INVALID_ARG;
  if (c->group > 8) return ENTMAXKV_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return ENTMAXKV_ERR_UNSUPPORTED;
  if (c->page_size != 16 && c->page_size != 32) return ENTMAXKV_ERR_UNSUPPORTED;
  if ((long long)c->max_pages_per_seq * c->page_size > 0x7fffffffLL) return ENTMAXKV_ERR_UNSUPPORTED;
  return ENTMAXKV_OK;
}

static int check_cache(const entmaxkv_cache* k) {
  if (!k || !k->k_pool || !k->v_pool || !k->kmin || !k->kmax || !k->mean || !k->m2 ||
      !k->block_table || !k->seq_lens)
    return ENTMAXKV_ERR_INVALID_ARG;
  if ((k->mean_bf16 == nullptr) != (k->m2_bf16 == nullptr)) return ENTMAXKV_ERR_INVALID_ARG;
  const void* arrays[] = {k->k_pool, k->v_pool, k->kmin, k->kmax, k->mean, k->m2, k->mean_bf16, k->m2_bf16};
  for (const void* p : arrays)
    if ((uintptr_t)p & 15u) return ENTMAXKV_ERR_INVALID_ARG;
  return ENTMAXKV_OK;
}

static int compute_layout(const entmaxkv_config* c, int S, int policy, int budget, Layout& L) {
  int st = check_config(c);
  if (st) return st;
  if (S < 1 || S > 65535) return ENTMAXKV_ERR_INVALID_ARG;
  if (policy < ENTMAXKV_POLICY_FULL || policy > ENTMAXKV_POLICY_SOFTMAX_TOPK) return ENTMAXKV_ERR_INVALID_ARG;
  const int Hkv = c->num_kv_heads, G = c->group, Hq = Hkv * G, D = c->head_dim, P = c->page_size;
  const int maxp = c->max_pages_per_seq;
  memset(&L, 0, sizeof(L));
  L.words = (maxp + 31) / 32;
  L.kpages = 0;
  L.gcap = 0;
  int cap = maxp;
  const bool topk = policy == ENTMAXKV_POLICY_TOPK || policy == ENTMAXKV_POLICY_SOFTMAX_TOPK;
  if (topk) {
    if (budget < P) return ENTMAXKV_ERR_INVALID_ARG;
    L.kpages = budget / P;
    cap = L.kpages < maxp ? L.kpages : maxp;
  } else if (policy == ENTMAXKV_POLICY_GAUSSIAN) {
    if (budget < 0) return ENTMAXKV_ERR_INVALID_ARG;
    if (budget > 0) {
      L.gcap = budget / P;
      if (L.gcap < 1) return ENTMAXKV_ERR_INVALID_ARG;
      cap = L.gcap < maxp ? L.gcap : maxp;
    }
  }
  L.cap_pages = cap;
  const long long units = (long long)S * Hkv;
  long long splits = (cap + 7) / 8;
  // entmax top-k's pass B also sums the certified dropped-mass bound over
  // every page of the row: at least 512 pages of that per block (not for
  // softmax top-k, whose last block merges one partial per split)
  if (policy == ENTMAXKV_POLICY_TOPK && splits < (maxp + 511) / 512) splits = (maxp + 511) / 512;
  long long tgt = (kLayoutBlocks + units - 1) / units;
  if (splits > tgt) splits = tgt;
  const bool bitmap = topk || policy == ENTMAXKV_POLICY_GAUSSIAN;
  const long long need = (cap + kListCap - 1) / kListCap;
  if (bitmap && splits < need) splits = need;
  if (splits < 1) splits = 1;
  if (splits > 65535) return ENTMAXKV_ERR_UNSUPPORTED;
  L.splits = (int)splits;
  const bool entmax = policy != ENTMAXKV_POLICY_SOFTMAX && policy != ENTMAXKV_POLICY_SOFTMAX_TOPK;
  const size_t nq = (size_t)S * Hq, nk = (size_t)S * Hkv;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = up256(off + bytes); return o; };
  const size_t none = (size_t)-1;
  L.zmax = take(nq * 4);
  L.cnt_a = take(nk * 4);
  L.cnt_b = take(nk * 4);
  L.cand_cnt = take(nq * 4);
  L.kept_mass = take(nq * 4);
  L.dbar = take(nq * 4);
  L.bitmap = bitmap ? take(nk * L.words * 4) : none;
  L.ctrl_end = off;
  L.tauhat = policy == ENTMAXKV_POLICY_GAUSSIAN ? take(nq * 4) : none;
  L.tau_ws = take(nq * 8);
  L.nsel_ws = take(nk * 4);
  L.sel_list = bitmap ? take(nk * (size_t)cap * 4) : none;
  L.bbox_u = topk ? take(nq * (size_t)maxp * 4) : none;
  L.bbox_uhat = topk ? take(nk * (size_t)maxp * 4) : none;
  L.gauss_ms = policy == ENTMAXKV_POLICY_GAUSSIAN ? take(nq * (size_t)maxp * 8) : none;
  L.sel_pp = entmax ? take(nk * (size_t)cap * 8) : none;
  L.vlist = entmax ? take(nk * (size_t)cap * 16) : none;
  L.vcount = entmax ? take(nk * 4) : none;
  L.cand = entmax ? take(nq * (size_t)cap * 8) : none;
  L.z = entmax ? take(nk * (size_t)cap * P * G * 4) : none;
  L.pmax = entmax ? take(nk * (size_t)cap * G * 4) : none;
  L.pstride = (G * D + 4 * G + 3) & ~3;  // acc [G][D], then 4 floats per head
  L.partial = entmax ? none : take(nk * (size_t)L.splits * L.pstride * 4);
  L.diag = take(nq * 4);
  L.mslots = gauss_grid_x(maxp, Hkv, S, 0);
  L.mslot = policy == ENTMAXKV_POLICY_GAUSSIAN ? take(nq * (size_t)L.mslots * 4)
            : topk                               ? take(nk * (size_t)L.mslots * 4)
                                                 : none;
  L.total = off;
  return ENTMAXKV_OK;
}

template <typename T>
static T* at(void* base, size_t off) {
  return off == (size_t)-1 ? nullptr : reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

// Point the workspace members of `a` at the regions of layout L in ws.
static void bind_workspace(DecodeArgs& a, void* ws, const Layout& L) {
  a.splits = L.splits;
  a.cap_pages = L.cap_pages;
  a.kpages = L.kpages;
  a.gcap = L.gcap;
  a.words = L.words;
  a.zmax = at<uint32_t>(ws, L.zmax);
  a.cnt_a = at<int32_t>(ws, L.cnt_a);
  a.cnt_b = at<int32_t>(ws, L.cnt_b);
  a.cand_cnt = at<int32_t>(ws, L.cand_cnt);
  a.kept_mass = at<float>(ws, L.kept_mass);
  a.dbar = at<float>(ws, L.dbar);
  a.bitmap = at<uint32_t>(ws, L.bitmap);
  a.tauhat = at<float>(ws, L.tauhat);
  a.tau_ws = at<double>(ws, L.tau_ws);
  a.nsel_ws = at<int32_t>(ws, L.nsel_ws);
  a.sel_list = at<int32_t>(ws, L.sel_list);
  a.sel_pp = at<int2>(ws, L.sel_pp);
  a.vlist = at<int4>(ws, L.vlist);
  a.vcount = at<int32_t>(ws, L.vcount);
  a.bbox_u = at<float>(ws, L.bbox_u);
  a.bbox_uhat = at<float>(ws, L.bbox_uhat);
  a.gauss_ms = at<float2>(ws, L.gauss_ms);
  a.cand = at<int2>(ws, L.cand);
  a.z = at<float>(ws, L.z);
  a.pmax = at<float>(ws, L.pmax);
  a.partial = at<float>(ws, L.partial);
  a.pstride = L.pstride;
  a.diag = at<int32_t>(ws, L.diag);
  a.mslot = at<uint32_t>(ws, L.mslot);
  a.mslots = L.mslots;
  a.ctrl = reinterpret_cast<uint4*>(ws);
  a.ctrl_vec = (int)(L.ctrl_end / 16);
}

// The full-cache policy whose result defines the exact dropped mass.
static int full_policy_of(int policy) {
  return policy == ENTMAXKV_POLICY_SOFTMAX_TOPK ? ENTMAXKV_POLICY_SOFTMAX : ENTMAXKV_POLICY_FULL;
}

// Bytes of the workspace with the given flags (0 for an invalid
// configuration); L gets the policy's layout, LF the full-cache one that the
// exact dropped mass needs.
static size_t total_bytes(const entmaxkv_config* c, int S, int policy, int budget, uint32_t flags,
                          Layout& L, Layout& LF) {
  if (compute_layout(c, S, policy, budget, L) != ENTMAXKV_OK) return 0;
  if (!(flags & ENTMAXKV_FLAG_EXACT_DELTA) || policy == ENTMAXKV_POLICY_SOFTMAX ||
      policy == ENTMAXKV_POLICY_FULL)
    return L.total;
  if (compute_layout(c, S, full_policy_of(policy), 0, LF) != ENTMAXKV_OK) return 0;
  return up256(L.total) + LF.total;
}

// Blocks per (sequence, KV head) of one decode launch: one wave of 2 blocks
// per SM over all units, at most one per 8 kept pages and at most the
// layout's count, but at least enough that no block holds more than kListCap
// pages of a bitmap policy (the layout's lower bound).
static int launch_splits(const Layout& L, int S, int Hkv, int policy, int sms) {
  const long long units = (long long)S * Hkv;
  long long splits = (L.cap_pages + 7) / 8;
  const long long row = 32LL * L.words;  // the table's row, rounded up to a bitmap word
  if (policy == ENTMAXKV_POLICY_TOPK && splits < (row + 511) / 512) splits = (row + 511) / 512;  // (as in the layout)
  // one wave of 2 blocks per SM; two waves' worth when several sequences
  // (of unequal lengths) share the launch
  const long long tgt = ((S > 1 ? 4LL : 2LL) * sms + units - 1) / units;
  if (splits > tgt) splits = tgt;
  // The softmax kernel's page list must hold a block's whole share of the
  // top-k selection; pass A's continues in the global selection list.
  const long long need = (L.cap_pages + kListCap - 1) / kListCap;
  if (policy == ENTMAXKV_POLICY_SOFTMAX_TOPK && splits < need) splits = need;
  if (splits > L.splits) splits = L.splits;
  return splits < 1 ? 1 : (int)splits;
}

}  // namespace ekv

using namespace ekv;

extern "C" {

int32_t entmaxkv_version(void) { return ENTMAXKV_VERSION; }

const char* entmaxkv_status_string(int32_t s) {
  switch (s) {
    case ENTMAXKV_OK: return "ok";
    case ENTMAXKV_ERR_INVALID_ARG: return "invalid argument";
    case ENTMAXKV_ERR_UNSUPPORTED: return "unsupported shape, dtype or alpha";
    case ENTMAXKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small or misaligned";
    case ENTMAXKV_ERR_CUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

size_t entmaxkv_workspace_bytes(const entmaxkv_config* cfg, int32_t n_seqs, int32_t policy,
                                int32_t budget_tokens) {
  Layout L;
  if (compute_layout(cfg, n_seqs, policy, budget_tokens, L) != ENTMAXKV_OK) return 0;
  return L.total;
}

size_t entmaxkv_workspace_bytes_flags(const entmaxkv_config* cfg, int32_t n_seqs, int32_t policy,
                                      int32_t budget_tokens, uint32_t flags) {
  Layout L, LF;
  return total_bytes(cfg, n_seqs, policy, budget_tokens, flags, L, LF);
}

int32_t entmaxkv_delta_kind(int32_t policy, uint32_t flags) {
  switch (policy) {
    case ENTMAXKV_POLICY_FULL:
    case ENTMAXKV_POLICY_SOFTMAX: return ENTMAXKV_DELTA_ZERO;
    case ENTMAXKV_POLICY_TOPK:
    case ENTMAXKV_POLICY_SOFTMAX_TOPK:
      return (flags & ENTMAXKV_FLAG_EXACT_DELTA) ? ENTMAXKV_DELTA_EXACT : ENTMAXKV_DELTA_CERTIFIED;
    case ENTMAXKV_POLICY_GAUSSIAN:
      return (flags & ENTMAXKV_FLAG_EXACT_DELTA) ? ENTMAXKV_DELTA_EXACT : ENTMAXKV_DELTA_MODEL;
    default: return -1;
  }
}

int32_t entmaxkv_read_status(const entmaxkv_cache* cache, uint32_t* status_out, int32_t clear,
                             void* stream) {
  if (!cache || !cache->status || !status_out) return ENTMAXKV_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(status_out, cache->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(cache->status, 0, sizeof(uint32_t), s);
  return e == cudaSuccess ? ENTMAXKV_OK : ENTMAXKV_ERR_CUDA;
}

int32_t entmaxkv_workspace_layout(const entmaxkv_config* cfg, int32_t n_seqs, int32_t policy,
                                  int32_t budget_tokens, entmaxkv_workspace_view* view) {
  if (!view) return ENTMAXKV_ERR_INVALID_ARG;
  Layout L;
  const int st = compute_layout(cfg, n_seqs, policy, budget_tokens, L);
  if (st) return st;
  view->bbox_u = L.bbox_u;
  view->bbox_uhat = L.bbox_uhat;
  view->gauss_ms = L.gauss_ms;
  view->tauhat = L.tauhat;
  view->sel_bitmap = L.bitmap;
  view->tauhat_iters = policy == ENTMAXKV_POLICY_GAUSSIAN ? L.diag : (size_t)-1;
  view->page_zmax = L.pmax;
  view->cap_pages = L.cap_pages;
  view->splits = L.splits;
  view->total = L.total;
  view->z_scores = L.z;
  return ENTMAXKV_OK;
}

int32_t entmaxkv_append(const entmaxkv_config* cfg, const entmaxkv_cache* cache, const void* k,
                        const void* v, const int32_t* seq_ids, int32_t n_seqs, int32_t n_tokens,
                        void* stream) {
  int st = check_config(cfg);
  if (st) return st;
  if ((st = check_cache(cache))) return st;
  if (n_seqs < 0 || n_tokens < 0 || n_seqs > 65535) return ENTMAXKV_ERR_INVALID_ARG;
  if (n_seqs == 0 || n_tokens == 0) return ENTMAXKV_OK;
  if (!k || !v) return ENTMAXKV_ERR_INVALID_ARG;
  if ((long long)n_tokens > (long long)cfg->max_pages_per_seq * cfg->page_size)
    return ENTMAXKV_ERR_INVALID_ARG;
  AppendArgs a;
  a.Hkv = cfg->num_kv_heads;
  a.D = cfg->head_dim;
  a.P = cfg->page_size;
  a.maxp = cfg->max_pages_per_seq;
  a.nphys = cfg->num_phys_pages;
  a.max_seqs = cfg->max_seqs;
  a.n_seqs = n_seqs;
  a.n_tokens = n_tokens;
  a.k = k;
  a.v = v;
  a.seq_ids = seq_ids;
  a.k_pool = cache->k_pool;
  a.v_pool = cache->v_pool;
  a.kmin = cache->kmin;
  a.kmax = cache->kmax;
  a.mean = cache->mean;
  a.m2 = cache->m2;
  a.mean_lo = static_cast<__nv_bfloat16*>(cache->mean_bf16);
  a.m2_lo = static_cast<__nv_bfloat16*>(cache->m2_bf16);
  a.block_table = cache->block_table;
  a.seq_lens = cache->seq_lens;
  a.status = cache->status;
  return launch_append(a, cfg->kv_dtype, (cudaStream_t)stream) == cudaSuccess ? ENTMAXKV_OK
                                                                             : ENTMAXKV_ERR_CUDA;
}

static int32_t decode_impl(const entmaxkv_config* cfg, const entmaxkv_cache* cache, const void* q,
                           const int32_t* seq_ids, int32_t n_seqs, float alpha, int32_t policy,
                           int32_t budget_tokens, float margin, uint32_t flags, void* workspace,
                           size_t workspace_bytes, float* out, int32_t* page_ids,
                           int32_t page_ids_stride, int32_t* n_sel, float* tau, float* delta,
                           void* stream, void* const* events) {
  int st = check_config(cfg);
  if (st) return st;
  if ((st = check_cache(cache))) return st;
  if (n_seqs < 0) return ENTMAXKV_ERR_INVALID_ARG;
  if (n_seqs == 0) return ENTMAXKV_OK;
  if (!q || !out) return ENTMAXKV_ERR_INVALID_ARG;
  const bool soft = policy == ENTMAXKV_POLICY_SOFTMAX || policy == ENTMAXKV_POLICY_SOFTMAX_TOPK;
  const bool topk = policy == ENTMAXKV_POLICY_TOPK || policy == ENTMAXKV_POLICY_SOFTMAX_TOPK;
  if (!soft && !(alpha > 1.0f && isfinite(alpha)))
    return ENTMAXKV_ERR_INVALID_ARG;
  if (policy == ENTMAXKV_POLICY_GAUSSIAN && !isfinite(margin)) return ENTMAXKV_ERR_INVALID_ARG;
  Layout L, LF;
  if ((st = compute_layout(cfg, n_seqs, policy, budget_tokens, L))) return st;
  const size_t need = total_bytes(cfg, n_seqs, policy, budget_tokens, flags, L, LF);
  const bool exact_delta = need != L.total;  // a second, full-cache region follows
  if (!workspace || ((uintptr_t)workspace & 255u) || workspace_bytes < need)
    return ENTMAXKV_ERR_WORKSPACE_TOO_SMALL;
  if (page_ids && page_ids_stride < L.cap_pages) return ENTMAXKV_ERR_INVALID_ARG;

  DecodeArgs a;
  memset(&a, 0, sizeof(a));
  a.Hkv = cfg->num_kv_heads;
  a.G = cfg->group;
  a.Hq = a.Hkv * a.G;
  a.D = cfg->head_dim;
  a.P = cfg->page_size;
  a.maxp = cfg->max_pages_per_seq;
  a.nphys = cfg->num_phys_pages;
  a.max_seqs = cfg->max_seqs;
  a.S = n_seqs;
  a.words = L.words;
  a.policy = policy;
  a.splits = L.splits;
  a.cap_pages = L.cap_pages;
  a.kpages = L.kpages;
  a.gcap = L.gcap;
  a.flags = flags;
  const float al = soft ? 2.0f : alpha;
  a.alpha = al;
  a.a1 = al - 1.0f;
  a.beta = (float)(1.0 / ((double)al - 1.0));
  a.inv_sqrt_d = (float)(1.0 / sqrt((double)a.D));
  a.zscale = (float)(((double)al - 1.0) / sqrt((double)a.D));
  a.margin_z = (float)(((double)al - 1.0) * (double)margin);
  // The Gaussian selector at an order without closed forms takes its partial
  // moments from fits built on the host for this β (cached); an order whose
  // fits miss their accuracy check is refused before anything is queued.
  if (policy == ENTMAXKV_POLICY_GAUSSIAN && al != 1.5f && al != 2.0f &&
      moment_fit_for(a.beta, &a.fit))
    return ENTMAXKV_ERR_UNSUPPORTED;
  // Every argument is checked; the launch shapes come from the device.
  const int sms = device_sms();
  if (sms < 1) return ENTMAXKV_ERR_CUDA;
  a.k_pool = cache->k_pool;
  a.v_pool = cache->v_pool;
  a.kmin = cache->kmin;
  a.kmax = cache->kmax;
  a.mean = cache->mean;
  a.m2 = cache->m2;
  a.mean_lo = static_cast<const __nv_bfloat16*>(cache->mean_bf16);
  a.m2_lo = static_cast<const __nv_bfloat16*>(cache->m2_bf16);
  a.block_table = cache->block_table;
  a.seq_lens = cache->seq_lens;
  a.status = cache->status;
  a.q = q;
  a.seq_ids = seq_ids;
  a.out = out;
  a.page_ids = page_ids;
  a.page_ids_stride = page_ids_stride;
  a.n_sel_out = n_sel;
  a.tau_out = tau;
  a.delta_out = delta;
  bind_workspace(a, workspace, L);
  a.splits = launch_splits(L, n_seqs, cfg->num_kv_heads, policy, sms);
  // The dry runs of pass A's tail only pay when the grid is one wave: with
  // more, the tail's code is already in L2 by the time a last block runs it,
  // and a dry run keeps a block from the next wave.
  a.dry_tail = (long long)a.splits * cfg->num_kv_heads * n_seqs <= 2LL * sms;
  a.mslots = gauss_grid_x(cfg->max_pages_per_seq, cfg->num_kv_heads, n_seqs, sms);
  // the bf16 bounding box also leaves each scoring block's largest bound
  a.bbox_slots = topk && cfg->kv_dtype == ENTMAXKV_BF16 ? a.mslots : 0;

  cudaStream_t s = (cudaStream_t)stream;
  auto mark = [&](int i) -> cudaError_t {
    return events ? cudaEventRecord((cudaEvent_t)events[i], s) : cudaSuccess;
  };
  cudaError_t e = mark(0);
  // The selective policies' first kernel clears the control words itself.
  if (e == cudaSuccess && !topk && policy != ENTMAXKV_POLICY_GAUSSIAN)
    e = cudaMemsetAsync(workspace, 0, L.ctrl_end, s);
  if (e == cudaSuccess) e = mark(1);
  const int dt = cfg->kv_dtype;
  // stage 1: page scoring
  if (e == cudaSuccess) {
    if (topk) e = launch_bbox(a, dt, sms, s);
    else if (policy == ENTMAXKV_POLICY_GAUSSIAN) e = launch_gauss(a, dt, sms, s);
  }
  if (e == cudaSuccess) e = mark(2);
  // stage 2: selection
  if (e == cudaSuccess) {
    if (topk) {
      e = launch_topk(a, 0, s);
    } else if (policy == ENTMAXKV_POLICY_GAUSSIAN) {
      e = launch_tauhat(a, s);
      if (e == cudaSuccess && L.gcap > 0) e = launch_topk(a, 1, s);
    }
  }
  if (e == cudaSuccess) e = mark(3);
  // stage 3: pass A
  if (e == cudaSuccess && !soft) e = launch_pass_a(a, dt, s);
  if (e == cudaSuccess) e = mark(4);
  // stage 4: pass B or the softmax kernel
  if (e == cudaSuccess) e = soft ? launch_softmax(a, dt, s) : launch_pass_b(a, dt, s);
  if (e == cudaSuccess) e = mark(5);
  // exact dropped mass: the full-cache solve in the second region (entmax:
  // pass A, for τ and z of every page; softmax: the full softmax, for its
  // log-normaliser), then the dropped mass from both
  if (e == cudaSuccess && exact_delta) {
    void* ws2 = static_cast<char*>(workspace) + up256(L.total);
    DecodeArgs f = a;
    f.policy = full_policy_of(policy);
    f.out = static_cast<float*>(nullptr);
    f.flags = 0;
    f.page_ids = nullptr;
    f.n_sel_out = nullptr;
    f.tau_out = nullptr;
    f.delta_out = nullptr;
    bind_workspace(f, ws2, LF);
    f.splits = launch_splits(LF, n_seqs, cfg->num_kv_heads, f.policy, sms);
    f.dry_tail = (long long)f.splits * cfg->num_kv_heads * n_seqs <= 2LL * sms;
    f.mslots = 0;
    e = cudaMemsetAsync(ws2, 0, LF.ctrl_end, s);
    if (e == cudaSuccess) e = soft ? launch_softmax(f, dt, s) : launch_pass_a(f, dt, s);
    if (e == cudaSuccess) e = launch_exact_delta(a, f, s);
  }
  return e == cudaSuccess ? ENTMAXKV_OK : ENTMAXKV_ERR_CUDA;
}

int32_t entmaxkv_decode(const entmaxkv_config* cfg, const entmaxkv_cache* cache, const void* q,
                        const int32_t* seq_ids, int32_t n_seqs, float alpha, int32_t policy,
                        int32_t budget_tokens, float margin, uint32_t flags, void* workspace,
                        size_t workspace_bytes, float* out, int32_t* page_ids,
                        int32_t page_ids_stride, int32_t* n_sel, float* tau, float* delta,
                        void* stream) {
  return decode_impl(cfg, cache, q, seq_ids, n_seqs, alpha, policy, budget_tokens, margin, flags,
                     workspace, workspace_bytes, out, page_ids, page_ids_stride, n_sel, tau, delta,
                     stream, nullptr);
}

int32_t entmaxkv_decode_profiled(const entmaxkv_config* cfg, const entmaxkv_cache* cache,
                                 const void* q, const int32_t* seq_ids, int32_t n_seqs,
                                 float alpha, int32_t policy, int32_t budget_tokens, float margin,
                                 uint32_t flags, void* workspace, size_t workspace_bytes,
                                 float* out, int32_t* page_ids, int32_t page_ids_stride,
                                 int32_t* n_sel, float* tau, float* delta, void* stream,
                                 void* const* events) {
  if (!events) return ENTMAXKV_ERR_INVALID_ARG;
  for (int i = 0; i < ENTMAXKV_STAGE_EVENTS; ++i)
    if (!events[i]) return ENTMAXKV_ERR_INVALID_ARG;
  return decode_impl(cfg, cache, q, seq_ids, n_seqs, alpha, policy, budget_tokens, margin, flags,
                     workspace, workspace_bytes, out, page_ids, page_ids_stride, n_sel, tau, delta,
                     stream, events);
}

}  // extern "C"
