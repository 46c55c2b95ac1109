// common.cuh -- shared device helpers and the argument blocks of the
// libentmaxkv kernels (sm_103a). Internal: not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>
#include <math_constants.h>
#include <stdint.h>

#include "entmaxkv.h"
#include "mills_poly.cuh"

namespace ekv {

constexpr int kThreads = 256;       // decode / scoring blocks: 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kSolveCap = 8192;     // candidate scores the τ solver keeps in shared memory
constexpr int kListCap = 1024;      // selected pages one decode block handles
constexpr int kTauhatCluster = 8;   // most blocks per τ̂ cluster (one cluster per query head)
constexpr int kTauhatBlockPages = 4096;  // pages one τ̂ block keeps in registers (16 a thread)
constexpr int kTopkCluster = 8;     // blocks per top-k cluster (one cluster per (sequence, KV head))

// Chebyshev fits of J_ν(t) = E[(t + Z)_+^ν], Z ~ N(0, 1), for the Gaussian
// selector at an entmax order other than α ∈ {1.5, 2} (β = 1/(α−1)); the
// orders are ν = β, β − 1 and, for β > 1, β − 2 (F and its first two
// τ-derivatives). Built on the host per β (moment_fit.cu) and passed with the
// kernel arguments, so the kernels read the coefficients from constant memory.
//   t ≤ 0:  J_ν(t) = φ(x)·u^{ν+1}·Σ_k cl[k]·T_k(w),  x = min(−t, 12),
//           u = 1/(1 + x/3), w = 2.5u − 1.5 (φ at the true −t);
//   0 < t ≤ 16:  J_ν(t) = (1 + t)^ν·Σ_k cr[k]·T_k(t/8 − 1), or with rlog set
//           2^{ν·log2(1 + t) + Σ_k cr[k]·T_k(t/8 − 1)};
//   t > 16: J_ν(t) = t^ν·(1 + Σ_{k=1..5} ca[k−1]·t^{−2k}).
constexpr int kFitN = 33;  // Chebyshev coefficients per fit (degree 32)
struct MomentFit {
  float cl[3][kFitN];
  float cr[3][kFitN];
  float ca[3][5];
  float nu[3];
  int rlog[3];  // the right fit is of log2 J_ν(t)/(1 + t)^ν
  int orders;  // 0: the closed forms (β ∈ {1, 2}); 2: no second derivative (β ≤ 1); 3
};

// Everything a decode kernel needs, passed by value (well under 4 KB).
struct DecodeArgs {
  // geometry
  int Hkv, G, Hq, D, P, maxp, nphys, max_seqs, S, words;
  int policy, splits, cap_pages, kpages, gcap;
  int dry_tail;        // pass A's blocks that are not last warm the tail's code (one-wave grids)
  uint32_t flags;
  float alpha, a1, beta, zscale, inv_sqrt_d, margin_z;
  // cache
  const void* k_pool;
  const void* v_pool;
  const void* kmin;
  const void* kmax;
  const float* mean;
  const float* m2;
  const __nv_bfloat16* mean_lo;  // bf16 copies of mean and m2 the Gaussian scorer streams, or null
  const __nv_bfloat16* m2_lo;
  const int32_t* block_table;
  const int32_t* seq_lens;
  uint32_t* status;
  // inputs
  const void* q;
  const int32_t* seq_ids;
  // outputs
  float* out;
  int32_t* page_ids;
  int page_ids_stride;
  int32_t* n_sel_out;
  float* tau_out;
  float* delta_out;
  // workspace: zeroed at the start of every decode
  uint32_t* zmax;      // [S][Hq]   ordered-encoded max z
  int32_t* cnt_a;      // [S][Hkv]  blocks of pass A done
  int32_t* cnt_b;      // [S][Hkv]  blocks of pass B done
  int32_t* cand_cnt;   // [S][Hq]   candidate pages listed
  float* kept_mass;    // [S][Hq]   Gaussian model mass of the kept pages
  float* dbar;         // [S][Hq]   top-k certified dropped mass
  uint32_t* bitmap;    // [S][Hkv][words]
  // workspace: written before it is read in every decode
  float* tauhat;       // [S][Hq]
  double* tau_ws;      // [S][Hq]   exact τ (double)
  int32_t* nsel_ws;    // [S][Hkv]
  int32_t* sel_list;   // [S][Hkv][cap_pages]
  int2* sel_pp;        // [S][Hkv][cap_pages] (logical, physical) page of each rank; phys −1: unreadable
  int4* vlist;         // [S][Hkv][cap_pages] (rank, logical page, physical page, 0) of the ranks whose
                       //   page max clears τ for some head, rank ascending
  int32_t* vcount;     // [S][Hkv] entries of vlist; −1: not built (pass B scans the ranks itself)
  float* bbox_u;       // [S][Hq][maxp]
  float* bbox_uhat;    // [S][Hkv][maxp]
  float2* gauss_ms;    // [S][Hq][maxp]
  int2* cand;          // [S][Hq][cap_pages] candidate pages: (rank, page max z bits)
  float* z;            // [S][Hkv][cap_pages][P][G]
  float* pmax;         // [S][Hkv][cap_pages][G]
  float* partial;      // [S][Hkv][splits][pstride]: acc [G][D], then (m, l) per head
  int pstride;         // floats per split partial: G·D + 2G rounded up to 4
  int32_t* diag;       // [S][Hq] τ̂ iterations (Gaussian)
  uint32_t* mslot;     // [S][Hq][mslots] ordered-encoded max m of each scoring block (Gaussian);
                       // [S][Hkv][mslots] its largest bound Û (top-k, bf16 bounding box)
  int mslots;          // scoring blocks per (sequence, 8 KV heads) row
  int bbox_slots;      // top-k: block maxima of Û in mslot (mslots), 0 when none were written
  uint4* ctrl;         // the workspace words zeroed before each decode's counters are used
  int ctrl_vec;        // their count in 16-byte units
  MomentFit fit;       // Gaussian selector at a general α (orders == 0 otherwise)
};

struct AppendArgs {
  int Hkv, D, P, maxp, nphys, max_seqs, n_seqs, n_tokens;
  const void* k;
  const void* v;
  const int32_t* seq_ids;
  void* k_pool;
  void* v_pool;
  void* kmin;
  void* kmax;
  float* mean;
  float* m2;
  __nv_bfloat16* mean_lo;  // bf16 copies kept in step with mean and m2, or null
  __nv_bfloat16* m2_lo;
  const int32_t* block_table;
  int32_t* seq_lens;
  uint32_t* status;
};

// ---------------------------------------------------------------------------
// small helpers

// Zero the decode's control words (counters, maxima, bitmap) with every block
// of the launching grid taking a slice; run by the first kernel of a policy.
__device__ __forceinline__ void clear_ctrl_slice(uint4* ctrl, int n_vec) {
  const int nb = gridDim.x * gridDim.y * gridDim.z;
  const int b = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const int per = (n_vec + nb - 1) / nb;
  const int lo = b * per, hi = min(n_vec, lo + per);
  for (int i = lo + (int)threadIdx.x; i < hi; i += blockDim.x) ctrl[i] = make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ void raise_flag(uint32_t* st, uint32_t bit) {
  if (st) atomicOr(st, bit);
}

// Order-preserving map float -> uint32 (for atomicMax on floats). 0 is below
// every encoded value and stands for "no value yet" (−inf).
__device__ __forceinline__ uint32_t ord_enc(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord_dec(uint32_t o) {
  if (o == 0u) return -CUDART_INF_F;
  uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(u);
}

// bf16 pair in one 32-bit word -> floats (exact).
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_min_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// D = A·B + D for one m16n8k16 tile, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte load of data no kernel writes while it runs (K/V pages, metadata);
// it is read once, so it skips L1 allocation.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// Sequence row of decode slot s, validated (−1 and flagged when invalid).
__device__ __forceinline__ int seq_row(const int32_t* seq_ids, int s, int max_seqs, uint32_t* st) {
  int seq = seq_ids ? seq_ids[s] : s;
  if (seq < 0 || seq >= max_seqs) {
    raise_flag(st, ENTMAXKV_DEV_BAD_SEQ_ID);
    return -1;
  }
  return seq;
}

// Valid length of a sequence clamped to its block-table row.
__device__ __forceinline__ int seq_len_clamped(const int32_t* lens, int seq, int maxp, int P,
                                               uint32_t* st) {
  if (seq < 0) return 0;
  int L = lens[seq];
  long long cap = (long long)maxp * P;
  if (L < 0) L = 0;
  if ((long long)L > cap) {
    raise_flag(st, ENTMAXKV_DEV_CAPACITY);
    L = (int)cap;
  }
  return L;
}

// Physical page of logical page lp, or −1 (flagged) when out of range.
__device__ __forceinline__ int phys_page(const int32_t* bt, int seq, int lp, int maxp, int nphys,
                                         uint32_t* st) {
  int ph = bt[(size_t)seq * maxp + lp];
  if (ph < 0 || ph >= nphys) {
    raise_flag(st, ENTMAXKV_DEV_BAD_PAGE_TABLE);
    return -1;
  }
  return ph;
}

// [x]_+^β for the β of the decode (β = 2 and 1 exactly, else powf).
__device__ __forceinline__ float pos_pow(float x, float beta) {
  x = fmaxf(x, 0.0f);
  if (beta == 2.0f) return x * x;
  if (beta == 1.0f) return x;
  return x > 0.0f ? powf(x, beta) : 0.0f;
}

// E[(a + σZ)_+^β] and its derivative in a, Z ~ N(0,1), for β ∈ {1, 2}:
//   β = 1:  a·Φ(t) + σ·φ(t),          d/da = Φ(t)
//   β = 2:  (a²+σ²)·Φ(t) + a·σ·φ(t),  d/da = 2(a·Φ(t) + σ·φ(t)),   t = a/σ.
__device__ __forceinline__ void gauss_moment(float a, float sg, bool beta2, float& g, float& dg) {
  if (!(sg > 0.0f)) {
    float ap = fmaxf(a, 0.0f);
    g = beta2 ? ap * ap : ap;
    dg = beta2 ? 2.0f * ap : (a > 0.0f ? 1.0f : 0.0f);
    return;
  }
  float t = a / sg;
  float Phi = normcdff(t);
  float phi = 0.3989422804014327f * expf(-0.5f * t * t);
  if (beta2) {
    g = (a * a + sg * sg) * Phi + a * sg * phi;
    dg = 2.0f * (a * Phi + sg * phi);
  } else {
    g = a * Phi + sg * phi;
    dg = Phi;
  }
}

// E[(a + σZ)_+^β] for Z ~ N(0, 1) and its first two derivatives in a, for
// β ∈ {1, 2}, without special functions. With t = a/σ, x = |t|:
//   H1(t) = t·Φ(t) + φ(t),  H(t) = (1 + t²)·Φ(t) + t·φ(t),
//   G = σ²·H, G' = 2σ·H1, G'' = 2Φ  (β = 2);  G = σ·H1, G' = Φ, G'' = φ/σ  (β = 1).
// For t ≤ 0: Φ = φ(x)·R(x), H1 = φ(x)·A(x), H = φ(x)·B(x) with the smooth,
// cancellation-free R, A, B of mills_poly.cuh (polynomials in u = 1/(1+x/3));
// for t > 0 the reflections Φ(t) = 1 − Φ(−t), H1(t) = t + H1(−t),
// H(t) = 1 + t² − H(−t). Relative error of each function below ~5e-7.
template <int N>
__device__ __forceinline__ float horner(const float (&c)[N], float w) {
  float r = c[N - 1];
#pragma unroll
  for (int i = N - 2; i >= 0; --i) r = fmaf(r, w, c[i]);
  return r;
}

__device__ __forceinline__ void gauss_moment2(float a, float sg, float inv_sg, bool beta2, float& g,
                                              float& dg, float& d2g) {
  if (!(sg > 0.0f)) {  // point mass at a
    const float ap = fmaxf(a, 0.0f);
    g = beta2 ? ap * ap : ap;
    dg = beta2 ? 2.0f * ap : (a > 0.0f ? 1.0f : 0.0f);
    d2g = beta2 ? (a > 0.0f ? 2.0f : 0.0f) : 0.0f;
    return;
  }
  constexpr float cR[EKV_MILLS_DEG + 1] = {EKV_MILLS_R};
  constexpr float cA[EKV_MILLS_DEG + 1] = {EKV_MILLS_A};
  constexpr float cB[EKV_MILLS_DEG + 1] = {EKV_MILLS_B};
  const float t = a * inv_sg;
  const float x = fabsf(t);
  // u and φ need only the accuracy of the fits (relative 4.4e-7): the PTX
  // approximate reciprocal (within about 1 ulp) and base-2 exponential
  // (relative error about 2^-22; it flushes to 0 below 2^-126, where every
  // moment is negligible) are enough, and each is a single instruction.
  float u;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(u) : "f"(fmaf(fminf(x, EKV_MILLS_XMAX), 0.33333334f, 1.0f)));
  const float w = fmaf(2.5f, u, -1.5f);
  float e2;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e2) : "f"(-0.72134752f * x * x));
  const float phi = 0.3989422804f * e2;
  const float pu = phi * u;
  const float R = pu * horner(cR, w);
  const float A = pu * u * horner(cA, w);
  const bool left = t <= 0.0f;
  const float Phi = left ? R : 1.0f - R;
  const float H1 = left ? A : t + A;
  if (beta2) {
    const float B = pu * u * u * horner(cB, w);
    const float H = left ? B : fmaf(t, t, 1.0f) - B;
    g = sg * sg * H;
    dg = 2.0f * sg * H1;
    d2g = 2.0f * Phi;
  } else {
    g = sg * H1;
    dg = Phi;
    d2g = phi * inv_sg;
  }
}

// Σ_k c[k]·T_k(x) (Clenshaw), x ∈ [−1, 1], coefficients in constant memory.
__device__ __forceinline__ float clenshaw(const float (&c)[kFitN], float x) {
  const float x2 = 2.0f * x;
  float b1 = 0.0f, b2 = 0.0f;
#pragma unroll 4
  for (int k = kFitN - 1; k >= 1; --k) {
    const float b = fmaf(x2, b1, c[k] - b2);
    b2 = b1;
    b1 = b;
  }
  return fmaf(x, b1, c[0] - b2);
}

// J_ν(t) of order fit.nu[k] from its fits (layout at MomentFit), as
// 2^E·M: the caller adds the exponent of its power of ς to E before one ex2,
// so ς^p·J stays in range where ς^p and J alone would not (a page with a tiny
// ς has t ~ 2^24, and t^ν alone overflows for ν > 5). Powers and φ use the
// single-instruction base-2 logarithm and exponential (relative error about
// 2^-22), inside the fits' accuracy.
__device__ __forceinline__ void jfit(const MomentFit& F, int k, float t, float& E, float& M) {
  const float nu = F.nu[k];
  float l2;
  if (t <= 0.0f) {
    const float x = -t, xc = fminf(x, 12.0f);
    const float u = 1.0f / (1.0f + xc * 0.33333334f);
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(u));
    E = fmaf(-0.72134752f, x * x, (nu + 1.0f) * l2);
    M = 0.3989422804f * clenshaw(F.cl[k], fmaf(2.5f, u, -1.5f));
    return;
  }
  if (t <= 16.0f) {
    const float c = clenshaw(F.cr[k], fmaf(t, 0.125f, -1.0f));
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(1.0f + t));
    E = F.rlog[k] ? fmaf(nu, l2, c) : nu * l2;
    M = F.rlog[k] ? 1.0f : c;
    return;
  }
  const float it2 = 1.0f / (t * t);
  M = fmaf(it2, fmaf(it2, fmaf(it2, fmaf(it2, fmaf(it2, F.ca[k][4], F.ca[k][3]), F.ca[k][2]),
                               F.ca[k][1]), F.ca[k][0]), 1.0f);
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(t));
  E = nu * l2;
}

// ς^p·J_ν(t) for the fit of order k: one ex2 of the summed exponent (a
// vanishing multiplier gives 0 whatever the exponent).
__device__ __forceinline__ float spow_j(const MomentFit& F, int k, float t, float p, float lsg) {
  float E, M, e;
  jfit(F, k, t, E, M);
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(fmaf(p, lsg, E)));
  return M != 0.0f ? e * M : 0.0f;
}

// The general-order counterpart of gauss_moment2, for Z ~ N(m, ς²) against τ,
// with t = (m − τ)/ς and lsg = log2 ς (ς > 0):
//   g = E[(Z − τ)_+^β] = ς^β·J_β(t);
//   dg = β·ς^{β−1}·J_{β−1}(t), minus the τ-derivative of g (as gauss_moment2);
//   d2g = β(β−1)·ς^{β−2}·J_{β−2}(t), its second τ-derivative (0 when β ≤ 1,
//   where it does not exist).
__device__ __forceinline__ void gauss_moment_gen(const MomentFit& F, float beta, float t, float lsg,
                                                 float& g, float& dg, float& d2g) {
  g = spow_j(F, 0, t, beta, lsg);
  dg = beta * spow_j(F, 1, t, beta - 1.0f, lsg);
  d2g = F.orders == 3 ? beta * (beta - 1.0f) * spow_j(F, 2, t, beta - 2.0f, lsg) : 0.0f;
}

// E[(a + σZ)_+^β] alone at a general order (σ = 0: the point mass a_+^β).
__device__ __forceinline__ float gauss_mass_gen(const MomentFit& F, float beta, float a, float sg) {
  if (!(sg > 0.0f)) return a > 0.0f ? powf(a, beta) : 0.0f;
  float l2;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l2) : "f"(sg));
  return spow_j(F, 0, a / sg, beta, l2);
}

// ---------------------------------------------------------------------------
// Bulk asynchronous copies (global -> shared) completed on an mbarrier.

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// Bulk prefetch of a contiguous global range into L2 (16-byte aligned start,
// size a multiple of 16).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete; false when `limit`
// polls ran out (the caller flags ENTMAXKV_DEV_TIMEOUT). A limit of 0 gives
// up at once (ENTMAXKV_FLAG_EXPIRE_WAITS).
constexpr int kPollLimit = 1 << 22;
__device__ __forceinline__ bool mbar_wait_limit(uint64_t* bar, uint32_t parity, int limit) {
  for (int i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  return mbar_wait_limit(bar, parity, kPollLimit);
}
// The phase parity of the n-th fill (counted from 1) of a stage of a ring of
// nst stages whose fills are issued in order, stage = fill index % nst: a
// stopped ring waits for these to land before its block exits.
__device__ __forceinline__ int ring_fills(int n_issued, int st, int nst) {
  return n_issued > st ? (n_issued - st + nst - 1) / nst : 0;
}
// size bytes from global src to shared dst (both 16-byte aligned, size a
// multiple of 16), completing `size` transaction bytes on bar.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t size, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(size), "r"(smem_u32(bar))
      : "memory");
}

// Tiled tensor copies (TMA). A 3-D map over the V pool [page][KV head ·
// token][dim] of bf16 moves one page's slab of a KV head as boxes of
// P rows × 64 dims (128-byte rows, 128-byte swizzle: the 16-byte chunk c of
// row t lands at chunk c ^ (t & 7)), so an ldmatrix over 8 rows of one chunk
// column touches 8 different bank groups. The destination is 1024-byte
// aligned; the box's x coordinate (0 or 64 dims) is 128-byte aligned.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}
// Byte offset of 16-byte chunk c (0..7) of row t in a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t swz128(int t, int c) { return (uint32_t)(t * 128 + ((c ^ (t & 7)) << 4)); }
// Four transposed 8×8 b16 tiles: lanes 8j..8j+7 give the row addresses of
// tile j, and register j returns it, as mma's A or B fragments want it.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3,
                                              uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// bf16 pair (lo in the low half) from two floats, rounded to nearest.
__device__ __forceinline__ uint32_t bf2_rn(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
// x = hi + lo with hi = bf16(x) and lo = bf16(x − hi): 16 significant bits
// of x, so a bf16 × bf16 product accumulated in fp32 sees x to about 2^-16.
__device__ __forceinline__ void bf16_split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = bf2_rn(x0 - __low2float(h), x1 - __high2float(h));
}

// Packed fp32 pairs (two lanes of a 64-bit register) and the sm_100-family
// paired FMA: d = a·b + c on both halves.
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float f2_sum(unsigned long long v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return lo + hi;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_splat(float c) { return f2_pack(c, c); }

// Block-wide exclusive scan of one int per thread (blockDim multiple of 32).
// Returns the sum below this thread; `total` receives the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* sh, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? sh[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) sh[lane] = w;
  }
  __syncthreads();
  total = sh[nw - 1];
  const int before = (warp > 0 ? sh[warp - 1] : 0) + x - v;
  __syncthreads();
  return before;
}

// ---------------------------------------------------------------------------
// Launches. Every kernel is launched through cudaLaunchKernelEx and starts
// with pdl_enter(): griddepcontrol.wait returns once the previous grid in the
// stream has completed and its memory is visible (at once when the launch
// did not allow programmatic overlap), then the next grid is allowed to
// launch. A launch with pdl = true lets its blocks be scheduled while the
// previous kernel drains; since every kernel waits before its first access,
// each waits transitively for all earlier ones.
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Raise a kernel's dynamic shared memory limit to at least `bytes` on the
// current device, remembering what was set, so that a decode's launches make
// no attribute call after the first one (host time per decode).
inline cudaError_t ensure_smem(const void* kernel, int bytes) {
  struct Entry {
    const void* fn;
    int dev, bytes;
  };
  static Entry table[256];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  int slot = -1;
  for (int i = 0; i < used; ++i)
    if (table[i].fn == kernel && table[i].dev == dev) {
      if (table[i].bytes >= bytes) return cudaSuccess;
      slot = i;
    }
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (slot < 0 && used < 256) slot = used++;
  if (slot >= 0) table[slot] = Entry{kernel, dev, bytes};
  return cudaSuccess;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Policies whose selection is a bitmap of pages (top-k, Gaussian, softmax top-k).
__device__ __forceinline__ bool uses_bitmap(int policy) {
  return policy == ENTMAXKV_POLICY_TOPK || policy == ENTMAXKV_POLICY_GAUSSIAN ||
         policy == ENTMAXKV_POLICY_SOFTMAX_TOPK;
}

// This block's share [lo, hi) of the n_sel selected pages; for bitmap
// policies the page ids of that share go to list[0 .. hi−lo), the ranks
// past kListCap of a longer share to spill[rank] (none without spill: the
// caller's split count keeps its shares within kListCap).
__device__ __forceinline__ void block_page_range(const DecodeArgs& a, int s, int kvh, int n_pages, int split,
                                 int* list, int* sh_scan, int& n_sel, int& lo, int& hi,
                                 int* spill = nullptr) {
  if (!uses_bitmap(a.policy)) {
    n_sel = n_pages;
    lo = (int)(((long long)n_sel * split) / a.splits);
    hi = (int)(((long long)n_sel * (split + 1)) / a.splits);
    return;
  }
  // Every word of the row is read, so the loads need not wait for the
  // sequence length: the decode clears the bitmap before any bit is set, and
  // no bit past the sequence's last page is ever set.
  const uint32_t* bm = a.bitmap + ((size_t)s * a.Hkv + kvh) * a.words;
  const int W = a.words;
  const int wpt = (W + kThreads - 1) / kThreads;
  const int w0 = threadIdx.x * wpt;
  int cnt = 0;
  for (int j = 0; j < wpt; ++j)
    if (w0 + j < W) cnt += __popc(bm[w0 + j]);
  int total;
  int r = block_exclusive_scan(cnt, sh_scan, total);
  n_sel = total;
  lo = (int)(((long long)n_sel * split) / a.splits);
  hi = (int)(((long long)n_sel * (split + 1)) / a.splits);
  for (int j = 0; j < wpt; ++j) {
    if (w0 + j >= W || r >= hi) break;
    uint32_t bits = bm[w0 + j];
    while (bits) {
      const int b = __ffs(bits) - 1;
      if (r >= lo && r < hi) {
        if (r - lo < kListCap) list[r - lo] = (w0 + j) * 32 + b;
        else if (spill) spill[r] = (w0 + j) * 32 + b;
      }
      ++r;
      bits &= bits - 1u;
    }
  }
  __syncthreads();
}

// Host: the fits for order β (cached); 0 when they pass their accuracy check.
int moment_fit_for(float beta, MomentFit* out);

// Launchers (one translation unit each).
cudaError_t launch_append(const AppendArgs& a, int kv_dtype, cudaStream_t st);
cudaError_t launch_bbox(const DecodeArgs& a, int kv_dtype, int sms, cudaStream_t st);
cudaError_t launch_gauss(const DecodeArgs& a, int kv_dtype, int sms, cudaStream_t st);
int gauss_grid_x(int maxp, int Hkv, int S, int sms);
cudaError_t launch_tauhat(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_topk(const DecodeArgs& a, int mode, cudaStream_t st);
// The V pool's tensor map for pass B and the softmax kernel (bf16 pools).
cudaError_t make_v_map(CUtensorMap* map, const void* v_pool, int nphys, int Hkv, int P, int D);
cudaError_t launch_exact_delta(const DecodeArgs& m, const DecodeArgs& f, cudaStream_t st);
cudaError_t launch_pass_a(const DecodeArgs& a, int kv_dtype, cudaStream_t st);
cudaError_t launch_pass_b(const DecodeArgs& a, int kv_dtype, cudaStream_t st);
cudaError_t launch_softmax(const DecodeArgs& a, int kv_dtype, cudaStream_t st);

}  // namespace ekv
