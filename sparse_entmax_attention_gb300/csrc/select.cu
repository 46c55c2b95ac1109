// select.cu -- candidate page selection (EntmaxKV, gist.science technical
// summary §2B).
//
// Gaussian-aware selection (§2B.2): solve the approximate normalisation
// equation for τ̂ from the page statistics, then keep the pages whose
// estimated maximum score clears τ̂ lowered by the margin Δ. Here
//   F(τ) = Σ_p n_p·E[(Z_p − τ)_+^β],  Z_p ~ N(m_p, ς_p²),  F(τ̂) = 1,
// solved by safeguarded Halley steps on log F (cubic convergence; Newton
// when the Halley step is not usable) inside a bracket [lo, hi] (lo starts at
// max_p m_p − 1, where F ≥ 1 by Jensen's inequality; a step leaving the
// bracket is replaced by bisection). Each query head gets one
// cluster of kTauhatCluster blocks; every iteration each block sums its share
// of pages, the blocks exchange partial sums through distributed shared
// memory, and every block takes the same step from the same totals. Then a
// page is kept when m_p + ς_p·sqrt(2 ln n_p) ≥ τ̂ − (α−1)Δ (the estimated
// maximum M̂_p = μ_p + σ_p·sqrt(2 ln n_p) against τ̂/(α−1) − Δ, on the z scale);
// a KV head keeps the union over its query heads, as bits in a bitmap.
//
// Top-k selection (§2B.1): the k pages with the largest bound (max over the
// group's query heads), ties to the lower logical page index, by an 8-bit
// radix select over order-preserving keys, in a cluster of blocks per
// (sequence, KV head) that exchange digit histograms through distributed
// shared memory (rows of up to kTopkClusterKeys pages), else in one block.
// The one-block select also enforces an optional cap on the Gaussian
// selection, keyed by the margin max_h (M̂_p − threshold_h) of the selected
// pages.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace ekv {

constexpr int kTauhatIters = 60;

__device__ __forceinline__ int page_tokens(int p, int n_pages, int L, int P) {
  return p == n_pages - 1 ? L - p * P : P;
}

__device__ __forceinline__ float sqrt_2ln(int n, int P, float c_full) {
  return n == P ? c_full : sqrtf(2.0f * logf((float)n));
}

using u64 = unsigned long long;

template <int N>
__device__ __forceinline__ u64 horner_x2(const float (&c)[N], u64 w) {
  u64 r = f2_splat(c[N - 1]);
#pragma unroll
  for (int i = N - 2; i >= 0; --i) r = f2_fma(r, w, f2_splat(c[i]));
  return r;
}

// The moments of gauss_moment2 for two pages at once, in packed f32x2
// arithmetic (one instruction for both pages wherever the step is a plain
// add, multiply or fused multiply-add), accumulated with the pages' token
// counts into (F, D1, D2) pairs. For β = 2 the D1 and D2 pairs come out
// halved. The branches on the sign of t become arithmetic on h = [t > 0]:
//   Φ = σ·R + h,  H1 = A + h·t,  H = σ·B + h·(1 + t²),  σ = 1 − 2h,
// with R, A, B the Mills-ratio forms at x = |t| (R → Q(x) on the left,
// 1 − Q(x) on the right, and likewise for the first and second partial
// moments). Every input must be finite with ς > 0 (the caller floors ς).
template <bool B2>
__device__ __forceinline__ void moments_x2(u64 mb, u64 sr, u64 ir, u64 nr, u64 noff, u64& f,
                                           u64& d1, u64& d2) {
  constexpr float cR[EKV_MILLS_DEG + 1] = {EKV_MILLS_R};
  constexpr float cA[EKV_MILLS_DEG + 1] = {EKV_MILLS_A};
  constexpr float cB[EKV_MILLS_DEG + 1] = {EKV_MILLS_B};
  const u64 t = f2_mul(f2_add(mb, noff), ir);
  float t0, t1;
  f2_unpack(t, t0, t1);
  const u64 y = f2_fma(f2_pack(fminf(fabsf(t0), EKV_MILLS_XMAX), fminf(fabsf(t1), EKV_MILLS_XMAX)),
                       f2_splat(0.33333334f), f2_splat(1.0f));
  float y0, y1, u0, u1;
  f2_unpack(y, y0, y1);
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(u0) : "f"(y0));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(u1) : "f"(y1));
  const u64 u = f2_pack(u0, u1);
  const u64 w = f2_fma(u, f2_splat(2.5f), f2_splat(-1.5f));
  const u64 tt = f2_mul(t, t);
  float a0, a1, e0, e1;
  f2_unpack(f2_mul(tt, f2_splat(-0.72134752f)), a0, a1);  // −t²/(2 ln 2)
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(a0));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(a1));
  const u64 phi = f2_mul(f2_pack(e0, e1), f2_splat(0.3989422804f));
  const u64 pu = f2_mul(phi, u);
  const u64 pu2 = f2_mul(pu, u);
  const u64 R = f2_mul(pu, horner_x2(cR, w));
  const u64 A = f2_mul(pu2, horner_x2(cA, w));
  const u64 h = f2_pack(t0 > 0.0f ? 1.0f : 0.0f, t1 > 0.0f ? 1.0f : 0.0f);
  const u64 sg = f2_fma(h, f2_splat(-2.0f), f2_splat(1.0f));
  const u64 Phi = f2_fma(sg, R, h);
  const u64 H1 = f2_fma(h, t, A);
  if (B2) {
    const u64 B = f2_mul(f2_mul(pu2, u), horner_x2(cB, w));
    const u64 H = f2_fma(sg, B, f2_fma(h, tt, h));
    f = f2_fma(nr, f2_mul(f2_mul(sr, sr), H), f);  // n·ς²·H
    d1 = f2_fma(nr, f2_mul(sr, H1), d1);            // n·ς·H1  (D1/2)
    d2 = f2_fma(nr, Phi, d2);                       // n·Φ     (D2/2)
  } else {
    f = f2_fma(nr, f2_mul(sr, H1), f);   // n·ς·H1
    d1 = f2_fma(nr, Phi, d1);            // n·Φ
    d2 = f2_fma(nr, f2_mul(phi, ir), d2);  // n·φ/ς
  }
}

// All arithmetic is float, on offsets from base = max_p m_p − 1 (each page's
// m_p − base is formed once), so every τ̂ is base + off with off = O(1).
// Per iteration each warp publishes its partial (F, F', F'') in shared memory;
// after one cluster barrier every warp of every block reads all
// kTauhatCluster·kWarps partials over distributed shared memory, sums them in
// a fixed butterfly order and takes the same step: all copies of the state
// stay bit-identical without further synchronisation.
// MODE 0: β = 1, 1: β = 2 (closed forms, packed), 2: any other β (the fits of
// a.fit, one page at a time; Newton steps when β ≤ 1, where F has no second
// derivative).
template <int MODE>
__global__ void __launch_bounds__(kThreads, 2) tauhat_kernel(DecodeArgs a, int cls) {
  constexpr bool B2 = MODE == 1;
  pdl_enter();
  constexpr int kParts = kTauhatCluster * kWarps / 32;  // partials per lane after the exchange
  static_assert(kTauhatCluster * kWarps % 32 == 0, "whole partials per lane");
  cg::cluster_group cluster = cg::this_cluster();
  // Every warp of the cluster pushes its partial (F, D1, D2) into this slot
  // of every block, so after the cluster barrier all reads are local. The
  // slots of ranks the cluster does not have stay zero.
  __shared__ float4 slot[2][kTauhatCluster * kWarps];
  __shared__ float wmax_sh[kWarps];
  const int h = blockIdx.y, s = blockIdx.z;
  const int kvh = h / a.G;
  const int rank = (int)cluster.block_rank(), C = (int)cluster.num_blocks();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Every block of a cluster takes the same early exits, so no cluster
  // barrier is ever left waiting.
  const int seq = seq_row(a.seq_ids, s, a.max_seqs, nullptr);
  const int L = seq_len_clamped(a.seq_lens, seq, a.maxp, a.P, nullptr);
  const int n_pages = (L + a.P - 1) / a.P;
  if (n_pages == 0) return;
  if ((cls == 1 && n_pages > kTauhatBlockPages) || (cls == 2 && n_pages <= kTauhatBlockPages)) return;
  for (int i = tid; i < 2 * kTauhatCluster * kWarps; i += kThreads) {
    const int e = i % (kTauhatCluster * kWarps);
    if (e >= C * kWarps) slot[i / (kTauhatCluster * kWarps)][e] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  const float2* ms = a.gauss_ms + ((size_t)s * a.Hq + h) * a.maxp;
  const int words = (n_pages + 31) / 32;
  const int chunk = ((words + C - 1) / C) * 32;
  const int p_lo = rank * chunk, p_hi = min(n_pages, p_lo + chunk);

  // This thread's pages stay in registers for every iteration (kRegPages
  // each, which covers C·kTauhatBlockPages pages per query head), as pairs
  // for the packed arithmetic; pages beyond that are re-read from memory.
  // Their loads are issued before the maximum is known. An empty slot holds
  // a finite page of zero weight far below every threshold.
  constexpr int kRegPages = kTauhatBlockPages / kThreads, kPairs = kRegPages / 2;
  float mb[kRegPages], sr[kRegPages], nr[kRegPages];
#pragma unroll
  for (int k = 0; k < kRegPages; ++k) {
    const int p = p_lo + tid + k * kThreads;
    // (an empty slot: far below every threshold, yet with ς = 1 after the
    // floor below, so no power of ς overflows at a large β)
    float2 v = make_float2(-3.0e4f, 1.0f);
    nr[k] = 0.0f;
    if (p < p_hi) {
      v = ms[p];
      nr[k] = (float)page_tokens(p, n_pages, L, a.P);
    }
    mb[k] = v.x;
    sr[k] = v.y;
  }
  // M = max_p m_p from the scoring blocks' maxima, split over the block
  float M = -CUDART_INF_F;
  const uint32_t* ms_slots = a.mslot + ((size_t)s * a.Hq + h) * a.mslots;
  for (int i = tid; i < a.mslots; i += kThreads) M = fmaxf(M, ord_dec(__ldcg(ms_slots + i)));
  M = warp_max(M);
  if (lane == 0) wmax_sh[warp] = M;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wmax_sh[w]);
  if (!(M > -CUDART_INF_F)) return;  // no readable page
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
  const float base = M - 1.0f;
  // ς is floored at 2^-24·max(1, |m − base|): a point mass (ς = 0) then
  // becomes a Gaussian whose moments differ from the point mass's by
  // O(ς²) ≈ 1e-14 relative, and t = (m − τ)/ς stays finite, so the packed
  // evaluation needs no branch per page.
  u64 mb2[kPairs], sr2[kPairs], ir2[kPairs], nr2[kPairs];
#pragma unroll
  for (int k = 0; k < kRegPages; ++k) {
    mb[k] -= base;
    sr[k] = fmaxf(sr[k], 0x1p-24f * fmaxf(1.0f, fabsf(mb[k])));
  }
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    mb2[i] = f2_pack(mb[2 * i], mb[2 * i + 1]);
    sr2[i] = f2_pack(sr[2 * i], sr[2 * i + 1]);
    ir2[i] = f2_pack(__frcp_rn(sr[2 * i]), __frcp_rn(sr[2 * i + 1]));
    nr2[i] = f2_pack(nr[2 * i], nr[2 * i + 1]);
  }
  float lo = 0.0f, hi = CUDART_INF_F, off = 0.0f;  // offsets from base; F(lo) ≥ 1
  bool converged = false;
  int it = 0;
  for (; it < kTauhatIters; ++it) {
    float f = 0.0f, df = 0.0f, d2f = 0.0f;
    if constexpr (MODE == 2) {
#pragma unroll
      for (int i = 0; i < kPairs; ++i) {
        float m0, m1, s0, s1, i0, i1, n0, n1;
        f2_unpack(mb2[i], m0, m1);
        f2_unpack(sr2[i], s0, s1);
        f2_unpack(ir2[i], i0, i1);
        f2_unpack(nr2[i], n0, n1);
        float g, dg, d2g, l0, l1;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l0) : "f"(s0));
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(l1) : "f"(s1));
        gauss_moment_gen(a.fit, a.beta, (m0 - off) * i0, l0, g, dg, d2g);
        f = fmaf(n0, g, f);
        df = fmaf(n0, dg, df);
        d2f = fmaf(n0, d2g, d2f);
        gauss_moment_gen(a.fit, a.beta, (m1 - off) * i1, l1, g, dg, d2g);
        f = fmaf(n1, g, f);
        df = fmaf(n1, dg, df);
        d2f = fmaf(n1, d2g, d2f);
      }
    } else {
      u64 f2 = 0ull, df2 = 0ull, d2f2 = 0ull;
      const u64 noff = f2_splat(-off);
#pragma unroll
      for (int i = 0; i < kPairs; ++i) moments_x2<B2>(mb2[i], sr2[i], ir2[i], nr2[i], noff, f2, df2, d2f2);
      f = f2_sum(f2);
      df = f2_sum(df2);
      d2f = f2_sum(d2f2);
      if (B2) {
        df *= 2.0f;
        d2f *= 2.0f;
      }
    }
    for (int p = p_lo + tid + kRegPages * kThreads; p < p_hi; p += kThreads) {
      const float2 v = ms[p];
      float g, dg, d2g;
      if constexpr (MODE == 2) {
        const float mk = v.x - base, sk = fmaxf(v.y, 0x1p-24f * fmaxf(1.0f, fabsf(mk)));
        float lk;
        asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(lk) : "f"(sk));
        gauss_moment_gen(a.fit, a.beta, (mk - off) / sk, lk, g, dg, d2g);
      } else {
        gauss_moment2((v.x - base) - off, v.y, v.y > 0.0f ? 1.0f / v.y : 0.0f, B2, g, dg, d2g);
      }
      const float np = (float)page_tokens(p, n_pages, L, a.P);
      f = fmaf(np, g, f);
      df = fmaf(np, dg, df);
      d2f = fmaf(np, d2g, d2f);
    }
    f = warp_sum(f);
    df = warp_sum(df);
    d2f = warp_sum(d2f);
    // Before the first push every block of the cluster must be running (the
    // arrive was posted after the early exits). A slot half is rewritten two
    // iterations later, and no block gets there before every block has passed
    // the next barrier, i.e. finished reading it.
    if (it == 0) asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
    if (lane < C)
      cluster.map_shared_rank(&slot[it & 1][0], lane)[rank * kWarps + warp] = make_float4(f, df, d2f, 0.0f);
    cluster.sync();
    float F = 0.0f, D1 = 0.0f, D2 = 0.0f;  // F, −dF/dτ, d²F/dτ²
#pragma unroll
    for (int q = 0; q < kParts; ++q) {  // a fixed order: every warp sums alike
      const float4 e = slot[it & 1][lane + 32 * q];
      F += e.x;
      D1 += e.y;
      D2 += e.z;
    }
    F = warp_sum(F);
    D1 = warp_sum(D1);
    D2 = warp_sum(D2);
    if (F >= 1.0f) lo = off;
    else hi = off;
    float next;
    bool stop;
    if (F == 1.0f) {
      next = off;
      stop = true;
    } else {
      // Halley on g = log F: g' = −D1/F, g'' = D2/F − g'²; Newton when not
      // usable. A step below the tolerance ends the solve (in float it may not
      // even move off, so it must not be judged against the bracket). The
      // step is computed with the fast log and divide: F itself is evaluated
      // exactly at every point, and the last step, which is not re-evaluated,
      // inherits only the fast log's absolute error near F = 1 (about 2^-21,
      // divided by |g'| ≈ 2–5), under the solve's tolerance.
      next = CUDART_NAN_F;
      stop = false;
      const float tol = 1e-6f * fmaxf(1.0f, fabsf(base + off));
      if (F > 0.0f && D1 > 0.0f) {
        const float rF = __frcp_rn(F);
        const float g = __logf(F), g1 = -D1 * rF, g2 = D2 * rF - g1 * g1;
        // (a negative den selects the Newton step: no second derivative for β ≤ 1)
        const float den = (MODE != 2 || a.fit.orders == 3) ? 2.0f * g1 * g1 - g * g2 : -1.0f;
        const float newton = -__fdividef(g, g1);
        const float step = den > 0.0f ? -2.0f * __fdividef(g * g1, den) : newton;
        if (fabsf(step) <= tol) {
          next = off + step;
          stop = true;
        } else {
          next = off + step;
          if (!(next > lo && next < hi)) {
            next = off + newton;
          } else if (den > 0.0f && step * step * fabsf(step) <= 1e-2f * tol) {
            // Halley converges cubically: the error left after this step is
            // about K·step³ (K ≈ 0.1 on page-score models), far below tol,
            // so the confirming evaluation is skipped.
            stop = true;
          }
        }
      }
      if (!stop) {
        if (!(next > lo && next < hi)) next = isinf(hi) ? lo + 1.0f : 0.5f * (lo + hi);
        stop = fabsf(next - off) <= tol || (hi - lo) <= tol;
      }
    }
    off = next;
    if (stop) {
      converged = true;
      break;
    }
  }
  // Every block leaves the loop at the same iteration with the same state,
  // and all pushes into this block landed before the last barrier: no
  // block touches another's shared memory from here on.
  if (rank == 0 && tid == 0) {
    a.tauhat[(size_t)s * a.Hq + h] = base + off;
    a.diag[(size_t)s * a.Hq + h] = it + 1;
    if (!converged) raise_flag(a.status, ENTMAXKV_DEV_TAUHAT_NOCONV);
  }
  // Selection bits from the cached pages: for each k the warp's lanes hold 32
  // consecutive pages starting on a bitmap word. Keep p iff
  // m_p + ς_p·sqrt(2 ln n_p) ≥ τ̂ − (α−1)Δ, here on offsets from base.
  const float thr = off - a.margin_z;
  const float c_full = sqrtf(2.0f * logf((float)a.P));
  uint32_t* bm = a.bitmap + ((size_t)s * a.Hkv + kvh) * a.words;
#pragma unroll
  for (int k = 0; k < kRegPages; ++k) {
    const int p0 = p_lo + warp * 32 + k * kThreads;
    if (p0 >= p_hi) break;
    const int p = p0 + lane;
    float m_lo, m_hi, s_lo, s_hi, n_lo, n_hi;
    f2_unpack(mb2[k / 2], m_lo, m_hi);
    f2_unpack(sr2[k / 2], s_lo, s_hi);
    f2_unpack(nr2[k / 2], n_lo, n_hi);
    const float mk = k & 1 ? m_hi : m_lo, sk = k & 1 ? s_hi : s_lo, nk = k & 1 ? n_hi : n_lo;
    const bool sel = p < p_hi && mk + sk * sqrt_2ln((int)nk, a.P, c_full) >= thr;
    const uint32_t bits = __ballot_sync(0xffffffffu, sel);
    if (lane == 0 && bits) atomicOr(&bm[p0 >> 5], bits);
  }
  for (int p0 = p_lo + warp * 32 + kRegPages * kThreads; p0 < p_hi; p0 += kThreads) {
    const int p = p0 + lane;
    bool sel = false;
    if (p < p_hi) {
      const float2 v = ms[p];
      sel = (v.x - base) + v.y * sqrt_2ln(page_tokens(p, n_pages, L, a.P), a.P, c_full) >= thr;
    }
    const uint32_t bits = __ballot_sync(0xffffffffu, sel);
    if (lane == 0 && bits) atomicOr(&bm[p0 >> 5], bits);
  }
}

// ---------------------------------------------------------------------------
// top-k

// mode 0: key = bounding-box bound max over the group (bbox_uhat).
// mode 1: key = margin max_h (m + ς·sqrt(2 ln n) − (τ̂_h − (α−1)Δ)) of a page the
//         Gaussian rule selected, −inf for the others.
__device__ __forceinline__ float page_key(const DecodeArgs& a, int mode, int s, int kvh, int p,
                                          int n, int L, const uint32_t* bm, const float* thr,
                                          float c_full) {
  if (mode == 0) return a.bbox_uhat[((size_t)s * a.Hkv + kvh) * a.maxp + p];
  if (!((bm[p >> 5] >> (p & 31)) & 1u)) return -CUDART_INF_F;
  const float cn = sqrt_2ln(page_tokens(p, n, L, a.P), a.P, c_full);
  float best = -CUDART_INF_F;
  for (int h = 0; h < a.G; ++h) {
    const float2 v = a.gauss_ms[((size_t)s * a.Hq + (size_t)kvh * a.G + h) * a.maxp + p];
    best = fmaxf(best, v.x + v.y * cn - thr[h]);
  }
  return best;
}

// Keys of up to kTopkKeys pages are computed once and kept in shared memory
// for the radix passes; longer rows recompute them from global memory.
constexpr int kTopkKeys = 48 * 1024;

__global__ void __launch_bounds__(1024) topk_kernel(DecodeArgs a, int mode) {
  pdl_enter();
  extern __shared__ uint32_t keys_sh[];  // [min(maxp, kTopkKeys)] order-preserving keys
  __shared__ int hist[256];
  __shared__ int sh_scan[32];
  __shared__ float thr[8];
  __shared__ uint32_t sh_prefix, sh_mask, sh_kmin, sh_kmax;
  __shared__ int sh_remaining, sh_eq_count;
  const int kvh = blockIdx.x, s = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seq = seq_row(a.seq_ids, s, a.max_seqs, tid == 0 ? a.status : nullptr);
  const int L = seq_len_clamped(a.seq_lens, seq, a.maxp, a.P, tid == 0 ? a.status : nullptr);
  const int n = (L + a.P - 1) / a.P;
  uint32_t* bm = a.bitmap + ((size_t)s * a.Hkv + kvh) * a.words;
  const float c_full = sqrtf(2.0f * logf((float)a.P));
  const bool staged = n <= kTopkKeys && n <= a.maxp;
  int k;
  if (mode == 0) {
    k = min(a.kpages, n);
    if (k == n) {  // keep every page
      for (int p0 = warp * 32; p0 < n; p0 += 1024) {
        const uint32_t bits = __ballot_sync(0xffffffffu, p0 + lane < n);
        if (lane == 0) bm[p0 >> 5] = bits;
      }
      return;
    }
  } else {
    int cnt = 0;
    for (int w = tid; w < (n + 31) / 32; w += 1024) cnt += __popc(bm[w]);
    int total;
    block_exclusive_scan(cnt, sh_scan, total);
    k = a.gcap;
    if (total <= k) return;  // within the cap: selection stands
    if (tid == 0) raise_flag(a.status, ENTMAXKV_DEV_CAPACITY);
    if (tid < a.G) thr[tid] = a.tauhat[(size_t)s * a.Hq + (size_t)kvh * a.G + tid] - a.margin_z;
  }
  if (tid == 0) {
    sh_kmin = 0xffffffffu;
    sh_kmax = 0u;
    sh_remaining = k;
  }
  __syncthreads();
  auto key_of = [&](int p) -> uint32_t {
    return staged ? keys_sh[p] : ord_enc(page_key(a, mode, s, kvh, p, n, L, bm, thr, c_full));
  };
  // Every key once from global memory (eight loads in flight a thread), kept
  // in shared memory when it fits, with the smallest and largest key.
  {
    uint32_t lo_k = 0xffffffffu, hi_k = 0u;
    for (int p0 = 0; p0 < n; p0 += 8 * 1024) {
      uint32_t kk[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int p = p0 + u * 1024 + tid;
        kk[u] = p < n ? ord_enc(page_key(a, mode, s, kvh, p, n, L, bm, thr, c_full)) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int p = p0 + u * 1024 + tid;
        if (p < n) {
          if (staged) keys_sh[p] = kk[u];
          lo_k = min(lo_k, kk[u]);
          hi_k = max(hi_k, kk[u]);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo_k = min(lo_k, __shfl_xor_sync(0xffffffffu, lo_k, o));
      hi_k = max(hi_k, __shfl_xor_sync(0xffffffffu, hi_k, o));
    }
    if (lane == 0) {
      atomicMin(&sh_kmin, lo_k);
      atomicMax(&sh_kmax, hi_k);
    }
  }
  __syncthreads();
  // Radix select of the k-th largest key, 8 bits a pass, starting below the
  // leading bits every key shares (keys of similar scores agree in sign and
  // exponent, so a first digit there would put them all in one bin).
  const uint32_t kmin = sh_kmin, kmax = sh_kmax;
  const int rb = (kmin ^ kmax) ? 32 - __clz((int)(kmin ^ kmax)) : 0;  // bits below the common prefix
  if (tid == 0) {
    sh_mask = rb >= 32 ? 0u : (0xffffffffu << rb);
    sh_prefix = kmin & sh_mask;
    sh_eq_count = n;  // (all keys equal: every page ties at T = kmin)
  }
  __syncthreads();
  for (int sh = rb - 8; rb > 0; sh -= 8) {
    const int shift = sh > 0 ? sh : 0;  // the last digit may overlap the decided bits
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    const uint32_t prefix = sh_prefix, mask = sh_mask;
    for (int p = tid; p < n; p += 1024) {
      const uint32_t key = key_of(p);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits 255−8l … 248−8l (descending); find where the count
      // from the top reaches `remaining`.
      int cnt[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = hist[255 - 8 * lane - j];
        tot += cnt[j];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - tot;
      const int rem = sh_remaining;
      if (excl < rem && incl >= rem) {
        int run = excl;
        for (int j = 0; j < 8; ++j) {
          if (run + cnt[j] >= rem) {
            const uint32_t digit = 255u - 8u * lane - j;
            sh_prefix = prefix | (digit << shift);
            sh_mask = mask | (255u << shift);
            sh_remaining = rem - run;
            sh_eq_count = cnt[j];
            break;
          }
          run += cnt[j];
        }
      }
    }
    __syncthreads();
    if (shift == 0) break;
  }
  // T is the k-th largest key: keep every key > T and the `remaining`
  // lowest-index pages with key == T.
  const uint32_t T = sh_prefix;
  const int remaining = sh_remaining;
  const bool split_ties = sh_eq_count > remaining;
  if (mode == 0 && !split_ties) {
    // no tie to split and no bitmap read back: each warp writes its words
    // without block barriers
    for (int p0 = warp * 32; p0 < n; p0 += 1024) {
      const int p = p0 + lane;
      const uint32_t bits = __ballot_sync(0xffffffffu, p < n && key_of(p) >= T);
      if (lane == 0) bm[p0 >> 5] = bits;
    }
    return;
  }
  __syncthreads();  // every thread has read the selection state
  int taken = 0;    // ties kept so far (block-uniform)
  for (int base = 0; base < n; base += 1024) {
    const int p = base + tid;
    const uint32_t key = p < n ? key_of(p) : 0u;
    bool sel = p < n && key > T;
    const bool eq = p < n && key == T;
    if (!split_ties) {
      sel = sel || eq;
    } else {
      int tot;
      const int before = block_exclusive_scan(eq ? 1 : 0, sh_scan, tot);
      sel = sel || (eq && taken + before < remaining);
      taken += tot;
    }
    const uint32_t bits = __ballot_sync(0xffffffffu, sel);
    __syncthreads();  // mode 1 reads the bitmap it is rewriting
    if (lane == 0 && base + warp * 32 < n) bm[p >> 5] = bits;
    __syncthreads();
  }
}

// Top-k by bound (mode 0) over a cluster of kTopkCluster blocks per
// (sequence, KV head). Block r owns the pages [r·chunk, (r+1)·chunk), chunk a
// whole number of bitmap words, and keeps its keys in registers (page
// p_lo + j·kTopkThreads + tid in slot j). The smallest and largest key and,
// per 8-bit digit, every block's histogram are pushed into all blocks of the
// cluster through distributed shared memory; after one cluster barrier each
// block sums the same histograms in the same order and takes the same digit,
// so every block ends with the same k-th largest key T. Keys equal to T are
// kept lowest page first: the last digit's histograms already hold each
// block's count of them, which gives this block's offset among the ties.
constexpr int kTopkThreads = 1024, kTopkKpt = 8, kTopkCand = 256;
constexpr int kTopkClusterKeys = kTopkCluster * kTopkThreads * kTopkKpt;

__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads)
    topk_cluster_kernel(DecodeArgs a) {
  pdl_enter();
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ int hist[2][256];                     // this block's histogram, one per digit parity
  __shared__ int all_hist[2][kTopkCluster][256];  // pushed by every block, one half per digit parity
  __shared__ int tot_sh[256], bef_sh[256];         // per digit: cluster total, total in lower blocks
  __shared__ uint2 all_mm[kTopkCluster];           // every block's (smallest, largest) key
  __shared__ uint2 warp_mm[kTopkThreads / 32];
  __shared__ int sh_scan[32];
  __shared__ uint32_t sh_prefix, sh_mask;
  __shared__ int sh_remaining, sh_eq_count, sh_eq_before;
  __shared__ uint32_t sh_tlo;
  __shared__ int cand_n, all_cnt[kTopkCluster];
  __shared__ uint2 cand_loc[kTopkCand];              // this block's (key, page) at or above T_lo
  __shared__ __align__(16) uint2 all_cand[kTopkCluster][kTopkCand];  // every block's, pushed
  const int kvh = blockIdx.y, s = blockIdx.z;
  const int rank = (int)cluster.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // The blocks split the table's row (max_pages_per_seq), so each block's key
  // loads go out before the sequence length is known; keys past the length
  // are masked afterwards.
  const int chunk = (((a.maxp + 31) / 32 + kTopkCluster - 1) / kTopkCluster) * 32;
  const int p_lo = rank * chunk;
  const float* u = a.bbox_uhat + ((size_t)s * a.Hkv + kvh) * a.maxp;
  uint32_t key[kTopkKpt];
#pragma unroll
  for (int j = 0; j < kTopkKpt; ++j) {
    const int p = p_lo + j * kTopkThreads + tid;
    key[j] = p < a.maxp ? ord_enc(__ldcg(u + p)) : 0u;
  }
  if (tid < 256) hist[0][tid] = hist[1][tid] = 0;
  // the scoring blocks' largest bounds (fast path below), loaded with the keys
  const int nbm = a.bbox_slots;
  uint32_t bmv = 0u;  // 0: below every encoded key
  if (tid < nbm && nbm <= kTopkThreads) bmv = __ldcg(a.mslot + ((size_t)s * a.Hkv + kvh) * a.mslots + tid);
  // Every block of the cluster takes the same exits, so no cluster barrier
  // is left waiting.
  const int seq = seq_row(a.seq_ids, s, a.max_seqs, (rank == 0 && tid == 0) ? a.status : nullptr);
  const int L = seq_len_clamped(a.seq_lens, seq, a.maxp, a.P, (rank == 0 && tid == 0) ? a.status : nullptr);
  const int n = (L + a.P - 1) / a.P;
  const int p_hi = min(n, p_lo + chunk);
  uint32_t* bm = a.bitmap + ((size_t)s * a.Hkv + kvh) * a.words;
  const int k = min(a.kpages, n);
  if (k == n) {  // keep every page (also n = 0)
    for (int p0 = p_lo + warp * 32; p0 < p_hi; p0 += kTopkThreads) {
      const uint32_t bits = __ballot_sync(0xffffffffu, p0 + lane < p_hi);
      if (lane == 0) bm[p0 >> 5] = bits;
    }
    return;
  }
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
  // Fast path. When the bounding-box kernel left each scoring block's largest
  // bound and there are at least k of them, the k-th largest of those maxima,
  // T_lo, is a lower bound of the k-th largest key: k distinct pages reach
  // it. Only keys ≥ T_lo can be kept; each block pushes those (key, page)
  // pairs to every block, and every block ranks the union by (key
  // descending, page ascending), which is exactly the top-k order with ties
  // to the lower page. A block with more than kTopkCand of them sends the
  // whole cluster (all blocks see the same counts) down the radix path, and
  // so does a union of more than kTopkThreads candidates.
  // (k well below the count of maxima keeps T_lo tight and the candidates few)
  bool fast = nbm > 0 && nbm <= kTopkThreads && 4 * k <= nbm;  // uniform over the cluster
  bool waited = false;
  if (fast) {
    // T_lo: the lower edge of the 8-bit bin (below the leading bits all the
    // maxima share) that holds the k-th largest maximum, so at least k
    // maxima, and with them k pages, reach it
    uint32_t mlo = tid < nbm ? bmv : 0xffffffffu, mhi = bmv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      mlo = min(mlo, __shfl_xor_sync(0xffffffffu, mlo, o));
      mhi = max(mhi, __shfl_xor_sync(0xffffffffu, mhi, o));
    }
    if (lane == 0) warp_mm[warp] = make_uint2(mlo, mhi);
    if (tid == 0) {
      sh_tlo = 0u;
      cand_n = 0;
    }
    __syncthreads();
    if (warp == 0) {
      uint2 m = warp_mm[lane];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        m.x = min(m.x, __shfl_xor_sync(0xffffffffu, m.x, o));
        m.y = max(m.y, __shfl_xor_sync(0xffffffffu, m.y, o));
      }
      if (lane == 0) {
        sh_prefix = m.x;
        sh_mask = m.y;
      }
    }
    __syncthreads();
    const uint32_t bmin = sh_prefix, bmax = sh_mask;
    const int brb = (bmin ^ bmax) ? 32 - __clz((int)(bmin ^ bmax)) : 0;  // bits below the shared prefix
    const int bsh = brb > 8 ? brb - 8 : 0;
    if (tid < nbm) atomicAdd(&hist[0][(bmv >> bsh) & 255u], 1);
    __syncthreads();
    if (warp == 0) {
      int cnt[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = hist[0][255 - 8 * lane - j];
        tot += cnt[j];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - tot;
      if (excl < k && incl >= k) {
        int jj = 7;
#pragma unroll
        for (int j = 7; j >= 0; --j) {
          int before = excl;
#pragma unroll
          for (int i = 0; i < j; ++i) before += cnt[i];
          if (before + cnt[j] >= k) jj = j;
        }
        const uint32_t digit = 255u - 8u * lane - jj;
        const uint32_t keep = brb >= 32 ? 0u : (0xffffffffu << brb);  // the shared prefix
        sh_tlo = (bmin & keep) | (digit << bsh);
      }
    }
    __syncthreads();
    if (tid < 256) hist[0][tid] = 0;  // (the radix path below starts from a clear histogram)
    const uint32_t tlo = sh_tlo;
    fast = tlo > ord_enc(-CUDART_INF_F);  // (k scoring blocks saw a readable page)
    if (fast) {
#pragma unroll
      for (int j = 0; j < kTopkKpt; ++j) {
        const int p = p_lo + j * kTopkThreads + tid;
        if (p < p_hi && key[j] >= tlo) {
          const int i = atomicAdd(&cand_n, 1);
          if (i < kTopkCand) cand_loc[i] = make_uint2(key[j], (uint32_t)p);
        }
      }
      __syncthreads();
      const int nc = cand_n;
      // every block of the cluster is running before the first push
      asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
      waited = true;
      const int nsend = min(nc, kTopkCand);
      if (tid < kTopkCluster) cluster.map_shared_rank(&all_cnt[0], tid)[rank] = nc;
      for (int i = tid; i < kTopkCluster * nsend; i += kTopkThreads) {
        const int r = i / nsend, q = i - r * nsend;
        cluster.map_shared_rank(&all_cand[0][0], r)[rank * kTopkCand + q] = cand_loc[q];
      }
      cluster.sync();
      int C = 0;
      bool over = false;
#pragma unroll
      for (int r = 0; r < kTopkCluster; ++r) {
        over = over || all_cnt[r] > kTopkCand;
        C += all_cnt[r];
      }
      over = over || C < k || C > kTopkThreads;  // (C < k cannot happen: k pages reach T_lo)
      if (!over) {
        // the candidates packed at the front of all_cand (read into
        // registers, then written: 2 a thread at most), padded to an even
        // count with a pair that ranks below every other
        uint2* flat = &all_cand[0][0];
        uint2 mine[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i = tid + u * kTopkThreads;
          if (i < C) {
            int r = 0, q = i;
            while (q >= all_cnt[r]) q -= all_cnt[r++];
            mine[u] = all_cand[r][q];
          }
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int i = tid + u * kTopkThreads;
          if (i < C) flat[i] = mine[u];
        }
        if (tid == 0 && (C & 1)) flat[C] = make_uint2(0u, 0xffffffffu);
        __syncthreads();
        // T = the candidate of rank k − 1 (every rank is unique: pages are)
        const uint4* c4 = reinterpret_cast<const uint4*>(flat);
        const int C2 = (C + 1) / 2;
        for (int i = tid; i < C; i += kTopkThreads) {
          const uint2 ci = flat[i];
          int rk = 0;
#pragma unroll 4
          for (int j2 = 0; j2 < C2; ++j2) {
            const uint4 w = c4[j2];  // two candidates
            rk += (w.x > ci.x || (w.x == ci.x && w.y < ci.y)) ? 1 : 0;
            rk += (w.z > ci.x || (w.z == ci.x && w.w < ci.y)) ? 1 : 0;
          }
          if (rk == k - 1) {
            sh_prefix = ci.x;
            sh_eq_before = (int)ci.y;
          }
        }
        __syncthreads();
        const uint32_t T = sh_prefix;
        const int Tp = sh_eq_before;
#pragma unroll
        for (int j = 0; j < kTopkKpt; ++j) {
          const int p0 = p_lo + j * kTopkThreads;
          if (p0 >= p_hi) continue;  // block-uniform
          const int p = p0 + tid;
          const bool sel = p < p_hi && (key[j] > T || (key[j] == T && p <= Tp));
          const uint32_t bits = __ballot_sync(0xffffffffu, sel);
          if (lane == 0 && p0 + warp * 32 < p_hi) bm[p >> 5] = bits;
        }
        return;  // no block touches another's shared memory after the barrier
      }
      fast = false;
    }
  }
  uint32_t lo_k = 0xffffffffu, hi_k = 0u;
#pragma unroll
  for (int j = 0; j < kTopkKpt; ++j) {
    if (p_lo + j * kTopkThreads + tid < p_hi) {
      lo_k = min(lo_k, key[j]);
      hi_k = max(hi_k, key[j]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo_k = min(lo_k, __shfl_xor_sync(0xffffffffu, lo_k, o));
    hi_k = max(hi_k, __shfl_xor_sync(0xffffffffu, hi_k, o));
  }
  if (lane == 0) warp_mm[warp] = make_uint2(lo_k, hi_k);
  __syncthreads();
  // every block of the cluster is running before the first push
  if (!waited) asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
  if (warp == 0) {
    uint2 m = warp_mm[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      m.x = min(m.x, __shfl_xor_sync(0xffffffffu, m.x, o));
      m.y = max(m.y, __shfl_xor_sync(0xffffffffu, m.y, o));
    }
    if (lane < kTopkCluster) cluster.map_shared_rank(&all_mm[0], lane)[rank] = m;
  }
  cluster.sync();
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int r = 0; r < kTopkCluster; ++r) {
    kmin = min(kmin, all_mm[r].x);
    kmax = max(kmax, all_mm[r].y);
  }
  // Radix select of the k-th largest key, 8 bits a pass, below the leading
  // bits that every key shares.
  const int rb = (kmin ^ kmax) ? 32 - __clz((int)(kmin ^ kmax)) : 0;
  uint32_t mask = rb >= 32 ? 0u : (0xffffffffu << rb);
  uint32_t prefix = kmin & mask;
  int remaining = k, eq_count = n, eq_before = min(p_lo, n);  // (all keys equal: every page ties)
  int par = 0;
  for (int sh = rb - 8; rb > 0; sh -= 8, par ^= 1) {
    const int shift = sh > 0 ? sh : 0;  // the last digit may overlap the decided bits
#pragma unroll
    for (int j = 0; j < kTopkKpt; ++j)
      if (p_lo + j * kTopkThreads + tid < p_hi && (key[j] & mask) == prefix)
        atomicAdd(&hist[par][(key[j] >> shift) & 255u], 1);
    __syncthreads();
    // A half of all_hist is rewritten two digits later, and no block gets
    // there before every block has passed the next barrier, i.e. finished
    // reading it. The other local half was pushed before the last barrier,
    // so it is cleared for the next digit now.
    for (int i = tid; i < 256 * kTopkCluster; i += kTopkThreads)
      cluster.map_shared_rank(&all_hist[par][rank][0], i >> 8)[i & 255] = hist[par][i & 255];
    if (tid < 256) hist[par ^ 1][tid] = 0;
    cluster.sync();
    if (tid < 256) {  // per digit: the cluster's count, and the count in the blocks below this one
      int t = 0, b = 0;
#pragma unroll
      for (int r = 0; r < kTopkCluster; ++r) {
        const int v = all_hist[par][r][tid];
        t += v;
        b += r < rank ? v : 0;
      }
      tot_sh[tid] = t;
      bef_sh[tid] = b;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns digits 255−8l … 248−8l (descending)
      int cnt[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = tot_sh[255 - 8 * lane - j];
        tot += cnt[j];
      }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - tot;
      if (excl < remaining && incl >= remaining) {
        int run = excl, jj = 7;
#pragma unroll
        for (int j = 7; j >= 0; --j) {  // the first digit (from the top) where the count reaches it
          int before = excl;
#pragma unroll
          for (int i = 0; i < j; ++i) before += cnt[i];
          if (before + cnt[j] >= remaining) {
            jj = j;
            run = before;
          }
        }
        const uint32_t digit = 255u - 8u * lane - jj;
        sh_prefix = prefix | (digit << shift);
        sh_mask = mask | (255u << shift);
        sh_remaining = remaining - run;
        sh_eq_count = tot_sh[digit];
        sh_eq_before = bef_sh[digit];
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    mask = sh_mask;
    remaining = sh_remaining;
    eq_count = sh_eq_count;
    eq_before = sh_eq_before;
    if (shift == 0) break;
  }
  // T = prefix is the k-th largest key: keep every key > T and the
  // `remaining` lowest-index pages with key == T (eq_before of them lie in
  // the blocks below this one).
  const uint32_t T = prefix;
  const bool split_ties = eq_count > remaining;
  int taken = eq_before;
#pragma unroll
  for (int j = 0; j < kTopkKpt; ++j) {
    const int p0 = p_lo + j * kTopkThreads;
    if (p0 >= p_hi) continue;  // block-uniform
    const int p = p0 + tid;
    const bool valid = p < p_hi;
    bool sel = valid && key[j] > T;
    const bool eq = valid && key[j] == T;
    if (!split_ties) {
      sel = sel || eq;
    } else {
      int tot;
      const int before = block_exclusive_scan(eq ? 1 : 0, sh_scan, tot);
      sel = sel || (eq && taken + before < remaining);
      taken += tot;
    }
    const uint32_t bits = __ballot_sync(0xffffffffu, sel);
    if (lane == 0 && p0 + warp * 32 < p_hi) bm[p >> 5] = bits;
  }
}

// One launch of the τ̂ kernel with clusters of C blocks; cls selects the
// sequences it solves (0 all, 1 those of at most kTauhatBlockPages pages,
// 2 the longer ones).
static cudaError_t launch_tauhat_c(const DecodeArgs& a, int C, int cls, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, a.Hq, a.S);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.fit.orders) return cudaLaunchKernelEx(&cfg, tauhat_kernel<2>, a, cls);
  if (a.beta == 2.0f) return cudaLaunchKernelEx(&cfg, tauhat_kernel<1>, a, cls);
  return cudaLaunchKernelEx(&cfg, tauhat_kernel<0>, a, cls);
}

// A cluster holds the longest row's pages in its blocks' registers (up to
// kTauhatCluster blocks). With several sequences and rows longer than one
// block, the sequences that fit one block are solved by single-block
// clusters in a launch of their own: a short sequence then takes one block
// and no cluster barrier, instead of C blocks mostly without pages.
cudaError_t launch_tauhat(const DecodeArgs& a, cudaStream_t st) {
  int C = (a.maxp + kTauhatBlockPages - 1) / kTauhatBlockPages;
  C = C < 1 ? 1 : (C > kTauhatCluster ? kTauhatCluster : C);
  cudaError_t e;
  if (a.S > 1 && C > 1) {
    e = launch_tauhat_c(a, 1, 1, st);
    if (e == cudaSuccess) e = launch_tauhat_c(a, C, 2, st);
  } else {
    e = launch_tauhat_c(a, C, 0, st);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_topk(const DecodeArgs& a, int mode, cudaStream_t st) {
  if (mode == 0 && a.maxp <= kTopkClusterKeys) {
    launch_k(false, topk_cluster_kernel, dim3(kTopkCluster, a.Hkv, a.S), dim3(kTopkThreads), 0, st, a);
    return cudaGetLastError();
  }
  dim3 grid(a.Hkv, a.S);
  const int smem = 4 * (a.maxp < kTopkKeys ? a.maxp : kTopkKeys);
  const cudaError_t e = ensure_smem((const void*)topk_kernel, smem);
  if (e != cudaSuccess) return e;
  launch_k(false, topk_kernel, dim3(grid), dim3(1024), (size_t)smem, st, a, mode);
  return cudaGetLastError();
}

}  // namespace ekv
