// decode.cu -- sparse α-entmax attention over the selected pages (EntmaxKV,
// gist.science technical summary §2C), the exact threshold, and the
// full-cache entmax baseline (§4) as the same kernels over every page.
//
// For each (sequence, KV head) the selected pages are split evenly over
// `splits` blocks ("split-K").
//   pass A  gathers each selected K page (16-byte loads straight into the
//           MMA fragment registers), scores it for the g query heads of the
//           group (bf16: m16n8k16 MMA, tokens × heads, fp32 accumulate; fp32:
//           CUDA-core dot products) on the z = (α−1)·q·k/√d scale, stores
//           z and each page's max z, and publishes the block's max z. Every
//           token that can be in the support has z > max z − 1 (τ ≥ z_max − 1),
//           so each block also emits its tokens above (its best known max − 1)
//           as candidates. The last block to finish solves the exact τ of each
//           query head from the candidates (one warp per head).
//   pass B  gathers V only for pages with some z above τ (all pages for the
//           dense baseline), accumulates Σ p_i v_i with p_i = [z_i − τ]_+^β
//           (bf16: V by TMA tensor copies into swizzled shared memory and
//           out^T = V^T·p on the tensor cores, p split into bf16 hi + lo;
//           fp32: CUDA-core FMA), and adds each block's sums into the output
//           rows (zeroed by pass A) with vector float atomics; the order of
//           those additions, and so the last bits of the output, vary from
//           run to run.
// Exact τ: τ solves Σ_i [z_i − τ]_+^β = 1. Starting from τ = z_max − 1
// (where the sum is ≥ 1) Newton steps on this convex decreasing function stay
// below the root; after each step the closed-form root on the current support
// S = {z > τ} is tried (β = 2: Σ_S (z−t)² = 1, β = 1: Σ_S (z−t) = 1) and
// accepted once it lies in [τ, min_S z], which makes it the exact root.
#include "common.cuh"
#include "page_scores.cuh"

namespace ekv {

constexpr int kTauIters = 64;

// ---------------------------------------------------------------------------
// Exact τ of one query head by one warp. Candidates are the scores above
// T0 = z_max − 1 (no other score can carry weight); normally they sit in
// shared memory, and only when they do not fit does the solver walk the
// candidate pages in global memory on every iteration.

struct SolveSrc {
  const float* zs;      // compacted candidates (shared memory)
  int m;
  bool big;             // candidates did not fit: walk the candidate pages instead
  const int2* pages;    // candidate pages (rank, page max bits)
  int np;
  const float* zbase;   // z of this (sequence, KV head): [rank][P][G]
  int P, G, hg;
  float T0;             // every score that can carry weight is above T0
};

template <class F>
__device__ __forceinline__ void for_each_cand(const SolveSrc& S, F&& f) {
  const int lane = threadIdx.x & 31;
  if (!S.big) {
    for (int i = lane; i < S.m; i += 32) f(S.zs[i]);
    return;
  }
  for (int k0 = 0; k0 < S.np; k0 += 32) {
    const int k = k0 + lane;
    const int2 e = k < S.np ? __ldcg(S.pages + k) : make_int2(0, __float_as_int(-CUDART_INF_F));
    uint32_t bits = __ballot_sync(0xffffffffu, __int_as_float(e.y) > S.T0);
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      const int rank = __shfl_sync(0xffffffffu, e.x, b);
      const float* zr = S.zbase + (size_t)rank * S.P * S.G;
      for (int t = lane; t < S.P; t += 32) {
        const float v = __ldcg(zr + t * S.G + S.hg);
        if (v > S.T0) f(v);
      }
    }
  }
}

// Float accumulation per candidate (GB300 runs FP64 at a small fraction of
// the FP32 rate): τ is carried as a double and split into hi + lo floats so
// that y = z − τ keeps its accuracy; only the per-iteration totals are double.
// Other orders: Newton inside a bracket [lo, hi] kept by the sign of the
// normaliser minus 1 (for β < 1 it is concave, so a step from below can
// overshoot the root, and a step leaving the bracket is replaced by
// bisection); it ends when the step or the bracket is below the tolerance.
__device__ double solve_tau_warp(const SolveSrc& S, double tau0, float beta, bool& ok) {
  double tau = tau0;
  double lo = tau0, hi = CUDART_INF;
  ok = false;
  const bool b2 = beta == 2.0f, b1 = beta == 1.0f;
  for (int it = 0; it < kTauIters; ++it) {
    const float th = (float)tau, tl = (float)(tau - (double)th);
    float kf = 0.0f, s1f = 0.0f, s2f = 0.0f, sbf = 0.0f, sb1f = 0.0f, mnf = CUDART_INF_F;
    for_each_cand(S, [&](float zf) {
      const float y = (zf - th) - tl;
      if (y > 0.0f) {
        kf += 1.0f;
        s1f += y;
        s2f = fmaf(y, y, s2f);
        mnf = fminf(mnf, y);
        if (!b2 && !b1) {
          sbf += powf(y, beta);
          sb1f += powf(y, beta - 1.0f);
        }
      }
    });
    const float k = warp_sum(kf), s1 = warp_sum(s1f), s2 = warp_sum(s2f);
    const float sb = warp_sum(sbf), sb1 = warp_sum(sb1f);
    const float mn = warp_min_f(mnf);
    if (!b2 && !b1) {
      const float tol = 1e-7f * fmaxf(1.0f, fabsf((float)tau));
      if (k == 0.0f || sb < 1.0f) hi = tau;  // above the root (no score above τ counts as 0 < 1)
      else lo = tau;
      if (k > 0.0f) {
        const float step = (sb - 1.0f) / (beta * sb1);
        if (fabsf(step) <= tol) {
          tau += (double)step;
          ok = true;
          break;
        }
        const double nt = tau + (double)step;
        tau = (nt > lo && nt < hi) ? nt : 0.5 * (lo + hi);
      } else {
        tau = 0.5 * (lo + hi);
      }
      if (hi - lo <= (double)tol) {
        ok = true;
        break;
      }
      continue;
    }
    if (k == 0.0f) break;  // cannot happen while τ < z_max
    float step;
    if (b2) {
      // root t = τ + δ of Σ_S (y − δ)² = 1 on the branch δ ≤ min y, in the
      // conjugate form δ = (s2 − 1)/(s1 + sqrt(s1² − k(s2 − 1))) (no cancellation)
      const float disc = s1 * s1 - k * (s2 - 1.0f);
      if (disc >= 0.0f) {
        const float d = (s2 - 1.0f) / (s1 + sqrtf(disc));
        if (d >= -1e-7f && d <= mn * (1.0f + 1e-6f) + 1e-7f) {
          tau += (double)d;
          ok = true;
          break;
        }
      }
      step = (s2 - 1.0f) / (2.0f * s1);
    } else if (b1) {
      const float d = (s1 - 1.0f) / k;
      if (d >= -1e-7f && d <= mn * (1.0f + 1e-6f) + 1e-7f) {
        tau += (double)d;
        ok = true;
        break;
      }
      step = d;
    } else {
      step = 0.0f;  // (other orders take the bracketed branch above)
    }
    if (!(step > 1e-7f * fmaxf(1.0f, fabsf((float)tau)))) {  // converged to float resolution
      if (step > 0.0f) tau += (double)step;
      ok = true;
      break;
    }
    tau += (double)step;
  }
  return tau;
}

// Exact threshold of at most 32 values (β = 1 or 2) without iterating. Lane i
// takes the set {z_j ≥ z_i} and its closed-form root δ_i (β = 2: Σ (y − δ)² = 1
// on the branch δ ≤ min y, in the conjugate form; β = 1: Σ (y − δ) = 1), with
// y = z − base > 0. A root that does not exceed its set's smallest value is a
// lower bound of the threshold (the normaliser is ≥ 1 there), and the root of
// the true support is the threshold itself, so the threshold is the largest
// such root. Float arithmetic: about 1e-6 from the exact value. Returns NaN
// for an empty set.
__device__ __forceinline__ float direct_tau_warp(const float* zs, int m, float base, bool b2) {
  const int lane = threadIdx.x & 31;
  const float yi = lane < m ? zs[lane] - base : -CUDART_INF_F;
  float k = 0.0f, s1 = 0.0f, s2 = 0.0f;
#pragma unroll 8
  for (int j = 0; j < 32; ++j) {
    const float yj = __shfl_sync(0xffffffffu, yi, j);
    if (yj >= yi) {
      k += 1.0f;
      s1 += yj;
      s2 = fmaf(yj, yj, s2);
    }
  }
  float d = -CUDART_INF_F;
  if (lane < m) {
    float r = CUDART_NAN_F;
    if (b2) {
      const float disc = s1 * s1 - k * (s2 - 1.0f);
      if (disc >= 0.0f) r = (s2 - 1.0f) / (s1 + sqrtf(disc));
    } else {
      r = (s1 - 1.0f) / k;
    }
    if (r <= yi) d = r;
  }
  d = warp_max(d);
  return m > 0 ? base + d : CUDART_NAN_F;
}

// ---------------------------------------------------------------------------

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 2) pass_a_kernel(DecodeArgs a) {
  pdl_enter();
  __shared__ int list[kListCap];
  __shared__ int phys_sh[kListCap];
  __shared__ int sh_scan[32];
  __shared__ float qs[8][D];
  __shared__ float wmax[kWarps][8];
  __shared__ float kept_sh[8];
  __shared__ float thr_sh[8];
  __shared__ int last_sh;
  // Page maxima of the block's pages [rank][G] during the page loop; in the
  // last block, the τ solver's page and score candidates.
  __shared__ __align__(16) float pool[kSolveCap];
  static_assert(kListCap * 8 <= kSolveCap, "page maxima of a block fit the pool");
  __shared__ float T0_sh[8], tlb_sh[8];
  __shared__ int nc_sh[8], np_sh[8], nz_sh[8], off_sh[9];
  __shared__ float tauf_sh[8], km_sh[8];
  __shared__ int vcnt_sh, spec_all_sh;
  const int split = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G, P = a.P;
  const int seq = seq_row(a.seq_ids, s, a.max_seqs, tid == 0 ? a.status : nullptr);
  const int L = seq_len_clamped(a.seq_lens, seq, a.maxp, P, tid == 0 ? a.status : nullptr);
  const int n_pages = (L + P - 1) / P;
  if (tid < 8) kept_sh[tid] = 0.0f;  // published by the barriers of the page range
  const size_t skv = (size_t)s * a.Hkv + kvh;
  const size_t hq0 = (size_t)s * a.Hq + (size_t)kvh * G;  // first query head of the group
  // q depends on nothing: its loads overlap the page range's
  uint32_t bq[D / 16][2];
  if constexpr (sizeof(T) == 2) {
    load_q_bfrag<D>((const __nv_bfloat16*)a.q + hq0 * D, G, lane, bq);
  } else {
    for (int i = tid; i < G * D; i += kThreads) qs[i / D][i % D] = ((const float*)a.q)[hq0 * D + i];
  }
  int n_sel, lo, hi;
  // a share longer than the list continues in the selection's global list
  int* spill = uses_bitmap(a.policy) ? a.sel_list + (size_t)s * a.Hkv * a.cap_pages + (size_t)kvh * a.cap_pages
                                     : nullptr;
  block_page_range(a, s, kvh, n_pages, split, list, sh_scan, n_sel, lo, hi, spill);
  const bool bitmap = uses_bitmap(a.policy);
  auto page_of = [&](int i) { return i < kListCap ? list[i] : spill[lo + i]; };
  const bool beta2 = a.beta == 2.0f;
  const bool gauss = a.policy == ENTMAXKV_POLICY_GAUSSIAN;
  if (split == 0 && a.out)  // pass B adds its blocks' sums into these rows
    for (int e = tid; e < G * a.D; e += kThreads) a.out[hq0 * a.D + e] = 0.0f;
  if (split == 0 && tid == 0) {
    a.nsel_ws[skv] = n_sel;
    if (a.n_sel_out) a.n_sel_out[skv] = n_sel;
  }
  // Every page of the block is looked up at once, and the K slabs of each
  // warp's next kAhead pages are kept requested into L2 by bulk prefetches
  // (≤ kAhead·8 pages a block in flight, well inside L2 for a full grid).
  constexpr int kAhead = 3;
  const bool staged = hi - lo <= kListCap;
  const uint32_t slab_bytes = (uint32_t)(P * D * sizeof(T));
  auto k_slab = [&](int ph) {
    return (const char*)a.k_pool + ((size_t)ph * a.Hkv + kvh) * slab_bytes;
  };
  // One item per (page, head of the group) for the Gaussian policy (its
  // kept model mass), one per page otherwise; the head-0 item of a page also
  // records and looks up the page. Loads of both kinds are in flight together.
  const int GI = gauss ? G : 1;
  for (int e = tid; e < (hi - lo) * GI; e += kThreads) {
    const int i = e / GI, h = e - i * GI;
    const int page = bitmap ? page_of(i) : lo + i;
    float2 v = make_float2(0.0f, 0.0f);
    float th = 0.0f;
    if (gauss) {  // summary §2B.2: 1 − kept model mass estimates the dropped mass δ
      v = a.gauss_ms[(hq0 + h) * a.maxp + page];
      th = a.tauhat[hq0 + h];
    }
    if (h == 0) {
      if (bitmap) a.sel_list[skv * a.cap_pages + lo + i] = page;
      if (a.page_ids) a.page_ids[skv * a.page_ids_stride + lo + i] = page;
      if (staged) {
        const int ph = phys_page(a.block_table, seq, page, a.maxp, a.nphys, a.status);
        phys_sh[i] = ph;
        if (ph >= 0 && i < kAhead * kWarps) prefetch_l2_bulk(k_slab(ph), slab_bytes);
      }
    }
    if (gauss) {
      float g, dg;
      if (a.fit.orders) g = gauss_mass_gen(a.fit, a.beta, v.x - th, v.y);
      else gauss_moment(v.x - th, v.y, beta2, g, dg);
      atomicAdd(&kept_sh[h], (float)min(P, L - page * P) * g);
    }
  }
  __syncthreads();

  float wm[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) wm[h] = -CUDART_INF_F;
  for (int i = warp; i < hi - lo; i += kWarps) {
    const int rank = lo + i;
    const int page = bitmap ? page_of(i) : rank;
    const int ph = staged ? phys_sh[i] : phys_page(a.block_table, seq, page, a.maxp, a.nphys, lane == 0 ? a.status : nullptr);
    if (staged && lane == 0 && i + kAhead * kWarps < hi - lo) {
      const int ph_next = phys_sh[i + kAhead * kWarps];
      if (ph_next >= 0) prefetch_l2_bulk(k_slab(ph_next), slab_bytes);
    }
    const int nv = min(P, L - page * P);
    float* zb = a.z + (skv * a.cap_pages + rank) * (size_t)P * G;
    float* pm = a.pmax + (skv * a.cap_pages + rank) * (size_t)G;
    if (lane == 0) a.sel_pp[skv * a.cap_pages + rank] = make_int2(page, ph);
    if (ph < 0) {  // unreadable page: no scores
      for (int e = lane; e < P * G; e += 32) zb[e] = -CUDART_INF_F;
      if (lane < G) {
        pm[lane] = -CUDART_INF_F;
        if (staged) pool[i * G + lane] = -CUDART_INF_F;
      }
      continue;
    }
    const size_t slab_off = ((size_t)ph * a.Hkv + kvh) * P * D;
    if constexpr (sizeof(T) == 2) {
      float zf[2][4];
      page_scores_bf16<D>((const __nv_bfloat16*)a.k_pool + slab_off, P, nv, bq, a.zscale, lane, zf);
      const int r = lane >> 2, c = lane & 3, h0 = 2 * c, h1 = h0 + 1;
      float pm0 = -CUDART_INF_F, pm1 = -CUDART_INF_F;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        if (16 * mt >= P) break;
        const int t0 = 16 * mt + r, t1 = t0 + 8;
        if (h1 < G && (G & 1) == 0) {  // even G: the pair is 8-byte aligned
          *reinterpret_cast<float2*>(zb + t0 * G + h0) = make_float2(zf[mt][0], zf[mt][1]);
          *reinterpret_cast<float2*>(zb + t1 * G + h0) = make_float2(zf[mt][2], zf[mt][3]);
        } else {
          if (h0 < G) {
            zb[t0 * G + h0] = zf[mt][0];
            zb[t1 * G + h0] = zf[mt][2];
          }
          if (h1 < G) {
            zb[t0 * G + h1] = zf[mt][1];
            zb[t1 * G + h1] = zf[mt][3];
          }
        }
        pm0 = fmaxf(pm0, fmaxf(zf[mt][0], zf[mt][2]));
        pm1 = fmaxf(pm1, fmaxf(zf[mt][1], zf[mt][3]));
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, o));
        pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, o));
      }
      if (r == 0) {
        if (h0 < G) pm[h0] = pm0;
        if (h1 < G) pm[h1] = pm1;
        if (staged) {
          if (h0 < G) pool[i * G + h0] = pm0;
          if (h1 < G) pool[i * G + h1] = pm1;
        }
      }
      // lane c keeps the running max of heads 2c, 2c+1 in wm[0], wm[1]
      wm[0] = fmaxf(wm[0], pm0);
      wm[1] = fmaxf(wm[1], pm1);
    } else {
      float zt[8];
      page_scores_f32<D>((const float*)a.k_pool + slab_off, nv, qs, G, a.zscale, lane, zt);
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h < G) {
          if (lane < P) zb[lane * G + h] = zt[h];
          const float m = warp_max(zt[h]);
          if (lane == 0) {
            pm[h] = m;
            if (staged) pool[i * G + h] = m;
          }
          wm[h] = fmaxf(wm[h], m);
        }
      }
    }
  }
  // block max z per head → global max; candidate threshold per head
  if constexpr (sizeof(T) == 2) {
    if (lane < 4) {
      wmax[warp][2 * lane] = wm[0];
      wmax[warp][2 * lane + 1] = wm[1];
    }
  } else {
    if (lane == 0)
      for (int h = 0; h < 8; ++h) wmax[warp][h] = wm[h];
  }
  __syncthreads();
  if (tid < G) {
    float m = -CUDART_INF_F;
    const float ks = kept_sh[tid];
    for (int w = 0; w < kWarps; ++w) m = fmaxf(m, wmax[w][tid]);
    float gm = m;
    if (m > -CUDART_INF_F) {
      const uint32_t old = atomicMax(&a.zmax[hq0 + tid], ord_enc(m));
      gm = fmaxf(m, ord_dec(old));
    }
    thr_sh[tid] = gm - 1.0f;
    if (gauss && ks != 0.0f) atomicAdd(&a.kept_mass[hq0 + tid], ks);
  }
  __syncthreads();
  // candidate pages: those whose max clears (best known max − 1). Lane l
  // checks rank l of the warp's 32 for every head at once; lane h then
  // reserves head h's slots, so each chunk costs one load and one atomic
  // round trip.
  for (int i0 = warp * 32; i0 < hi - lo; i0 += kThreads) {
    const int i = i0 + lane;
    const bool in = i < hi - lo;
    const int rank = lo + i;
    const float* pm = staged ? pool + (in ? i : 0) * G : a.pmax + (skv * a.cap_pages + (in ? rank : lo)) * (size_t)G;
    float pmv[8];
#pragma unroll
    for (int hg = 0; hg < 8; ++hg) pmv[hg] = (in && hg < G) ? pm[hg] : -CUDART_INF_F;
    uint32_t mine = 0u, bits[8];
    bool cand = false;
#pragma unroll
    for (int hg = 0; hg < 8; ++hg) {
      const bool c = hg < G && pmv[hg] > thr_sh[hg];
      cand = cand || c;
      bits[hg] = __ballot_sync(0xffffffffu, c);
      if (lane == hg) mine = bits[hg];
    }
    // Only candidate pages can need V (τ ≥ z_max − 1): request their V slabs
    // into L2 now, so that pass B finds them there.
    if (cand && staged && phys_sh[i] >= 0)
      prefetch_l2_bulk((const char*)a.v_pool + ((size_t)phys_sh[i] * a.Hkv + kvh) * slab_bytes, slab_bytes);
    int base = 0;
    if (mine) base = atomicAdd(&a.cand_cnt[hq0 + lane], __popc(mine));
#pragma unroll
    for (int hg = 0; hg < 8; ++hg) {
      const int b = __shfl_sync(0xffffffffu, base, hg);
      if ((bits[hg] >> lane) & 1u)  // a page enters a head's list at most once
        a.cand[(hq0 + hg) * a.cap_pages + b + __popc(bits[hg] & ((1u << lane) - 1u))] =
            make_int2(rank, __float_as_int(pmv[hg]));
    }
  }
  // the last block of this (sequence, KV head) solves τ
  __threadfence();
  __syncthreads();
  if (tid == 0) last_sh = atomicAdd(&a.cnt_a[skv], 1) == a.splits - 1;
  __syncthreads();
  // A block that is not the last runs the tail below once as a dry run:
  // every candidate's rank reads as 0 and each head's list as at most one
  // entry, so all its loads stay in bounds and it is short, and it stores
  // nothing to global memory. The tail runs once per decode, after the
  // scorer's stream has left none of its code in L2; the dry runs bring that
  // code into L2 (and into their SMs' instruction caches) before the last
  // block needs it. Grids of more than one wave skip them (a.dry_tail).
  const bool dry = !last_sh;
  if (dry && (a.cap_pages <= 0 || !a.dry_tail)) return;
  __threadfence();
  // Exact τ of the G query heads, block-parallel:
  //  A  keep the listed candidate pages whose max clears T0 = z_max − 1
  //     (all heads' lists at once, a thread per entry);
  //  B  τ_lb = exact threshold of (a subset of) those page maxima: they are
  //     real token scores, so their normaliser is below the full one, τ ≥ τ_lb;
  //  C  gather the scores above τ_lb from the pages whose max clears τ_lb
  //     (a thread per 8 tokens of a page, every head at once);
  //  D  one warp per head solves exactly on that set, starting from τ_lb.
  // Shared pool: page maxima [G][capP], their ranks [G][capP], scores [G][capZ].
  const int capP = kSolveCap / 4 / G;
  const int capZ = kSolveCap / 2 / G;
  float* pv = pool;
  int* pr = reinterpret_cast<int*>(pool + kSolveCap / 4);
  float* zc = pool + kSolveCap / 2;
  const float* zbase = a.z + skv * a.cap_pages * (size_t)P * G;
  const int2* clist = a.cand + hq0 * a.cap_pages;
  // Thread tid also loads, with the counts, entries js + k·SPT (k < kSlots)
  // of head hs's list (fixed slots; stale past the count, so used only below
  // it). When every list fits its slots, step A needs no further load, and a
  // thread whose entry clears T0 starts the page's (page, phys) lookup for the
  // V list at once.
  constexpr int kSlots = 4;
  const int SPT = kThreads / G, SPH = kSlots * SPT;  // slots per head
  const int hs = tid / SPT, js = tid - hs * SPT;
  int2 ce[kSlots];
#pragma unroll
  for (int k = 0; k < kSlots; ++k) {
    ce[k] = make_int2(0, __float_as_int(-CUDART_INF_F));
    if (hs < G && js + k * SPT < a.cap_pages) ce[k] = __ldcg(clist + (size_t)hs * a.cap_pages + js + k * SPT);
    if (dry) ce[k].x = 0;
  }
  // V-list page bitmap over the selection's ranks (the page-id arrays are free now)
  const int Wv = (n_sel + 31) >> 5;
  uint32_t* vb = reinterpret_cast<uint32_t*>(phys_sh);
  if (Wv <= kListCap)
    for (int i = tid; i < Wv; i += kThreads) vb[i] = 0u;
  if (tid < G) {
    const float zm = ord_dec(__ldcg(&a.zmax[hq0 + tid]));
    T0_sh[tid] = zm > -CUDART_INF_F ? zm - 1.0f : CUDART_INF_F;
    nc_sh[tid] = min(__ldcg(&a.cand_cnt[hq0 + tid]), dry ? 1 : a.cap_pages);
    km_sh[tid] = gauss ? __ldcg(&a.kept_mass[hq0 + tid]) : 0.0f;
    np_sh[tid] = 0;
    nz_sh[tid] = 0;
  }
  __syncthreads();
  if (tid == 0) {
    int t = 0;
    bool fits = dry || Wv <= kListCap;
    for (int h = 0; h < G; ++h) {
      off_sh[h] = t;
      t += nc_sh[h];
      fits = fits && nc_sh[h] <= SPH;
    }
    off_sh[G] = t;
    spec_all_sh = fits;
    vcnt_sh = 0;
  }
  __syncthreads();
  const bool spec_all = spec_all_sh;
  uint32_t kept = 0u;  // bit k: slot k's entry clears T0 (spec_all only)
  int2 kpp[kSlots];
  if (spec_all) {  // A, from the slots
#pragma unroll
    for (int k = 0; k < kSlots; ++k) {
      kpp[k] = make_int2(0, -1);
      if (hs < G && js + k * SPT < nc_sh[hs] && __int_as_float(ce[k].y) > T0_sh[hs]) {
        kept |= 1u << k;
        kpp[k] = __ldcg(&a.sel_pp[skv * a.cap_pages + ce[k].x]);  // consumed after D
        const int pos = atomicAdd(&np_sh[hs], 1);
        if (pos < capP) {
          pv[hs * capP + pos] = __int_as_float(ce[k].y);
          pr[hs * capP + pos] = ce[k].x;
        }
      }
    }
  } else {
    for (int e = tid; e < off_sh[G]; e += kThreads) {  // A
      int h = 0;
      while (e >= off_sh[h + 1]) ++h;
      const int2 c = __ldcg(clist + (size_t)h * a.cap_pages + (e - off_sh[h]));
      if (__int_as_float(c.y) > T0_sh[h]) {
        const int pos = atomicAdd(&np_sh[h], 1);
        if (pos < capP) {
          pv[h * capP + pos] = __int_as_float(c.y);
          pr[h * capP + pos] = c.x;
        }
      }
    }
  }
  __syncthreads();
  if (warp < G) {  // B
    const int h = warp;
    float tlb = T0_sh[h];
    const int np = min(np_sh[h], capP);
    if (np > 0 && np <= 32 && (a.beta == 2.0f || a.beta == 1.0f)) {
      // a lower bound needs no more than float accuracy: the direct root,
      // lowered by a margin well above its error
      const float tb = direct_tau_warp(pv + h * capP, np, tlb, a.beta == 2.0f);
      if (tb > tlb) tlb = fmaxf(tlb, tb - 1e-5f * fmaxf(1.0f, fabsf(tb)));
    } else if (np > 0) {
      SolveSrc src;
      src.zs = pv + h * capP;
      src.m = np;
      src.big = false;
      bool ok;
      const float tb = (float)solve_tau_warp(src, (double)T0_sh[h], a.beta, ok);
      // the solve ends within its tolerance on either side of the root
      if (tb > tlb) tlb = fmaxf(tlb, tb - 1e-5f * fmaxf(1.0f, fabsf(tb)));
    }
    if (lane == 0) tlb_sh[h] = tlb;
  }
  // C walks the kept pages of A, or a head's whole list where A overflowed
  const int cpp = P / 8;  // 8-token pieces per page
  if (tid == 0) {
    int t = 0;
    for (int h = 0; h < G; ++h) {
      off_sh[h] = t;
      t += (np_sh[h] <= capP ? np_sh[h] : nc_sh[h]) * cpp;
    }
    off_sh[G] = t;
  }
  __syncthreads();
  for (int e = tid; e < off_sh[G]; e += kThreads) {  // C
    int h = 0;
    while (e >= off_sh[h + 1]) ++h;
    const int j = (e - off_sh[h]) / cpp, piece = (e - off_sh[h]) - j * cpp;
    int rank;
    float pmv;
    if (np_sh[h] <= capP) {
      rank = pr[h * capP + j];
      pmv = pv[h * capP + j];
    } else {
      const int2 c = __ldcg(clist + (size_t)h * a.cap_pages + j);
      rank = c.x;
      pmv = __int_as_float(c.y);
    }
    const float tlb = tlb_sh[h];
    if (!(pmv > tlb)) continue;
    const float* zr = zbase + ((size_t)rank * P + 8 * piece) * G + h;
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcg(zr + u * G);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (v[u] > tlb) {
        const int pos = atomicAdd(&nz_sh[h], 1);
        if (pos < capZ) zc[h * capZ + pos] = v[u];
      }
    }
  }
  __syncthreads();
  if (warp < G) {  // D
    const int hg = warp;
    const size_t hs = hq0 + hg;
    float tau_f = CUDART_NAN_F;
    double tau_d = CUDART_NAN;
    if (T0_sh[hg] < CUDART_INF_F) {
      SolveSrc src;
      src.zs = zc + hg * capZ;
      src.m = nz_sh[hg];
      src.big = nz_sh[hg] > capZ;
      src.pages = clist + (size_t)hg * a.cap_pages;
      src.np = nc_sh[hg];
      src.zbase = zbase;
      src.P = P;
      src.G = G;
      src.hg = hg;
      src.T0 = tlb_sh[hg];
      if (src.big && lane == 0 && !dry) raise_flag(a.status, ENTMAXKV_DEV_CAND_OVERFLOW);
      // With few scores the direct root, lowered by a margin above its error,
      // starts the solve just below τ: usually one closed-form check on the
      // final support ends it.
      double t0 = (double)src.T0;
      if (!src.big && src.m <= 32 && (a.beta == 2.0f || a.beta == 1.0f)) {
        const float td = direct_tau_warp(src.zs, src.m, src.T0, a.beta == 2.0f);
        if (td > src.T0) t0 = fmax(t0, (double)td - 1e-5 * fmax(1.0, fabs((double)td)));
      }
      bool ok;
      tau_d = solve_tau_warp(src, t0, a.beta, ok);
      if (!ok && lane == 0 && !dry) raise_flag(a.status, ENTMAXKV_DEV_TAU_NOCONV);
      tau_f = (float)tau_d;
    }
    if (lane == 0) tauf_sh[hg] = tau_f;
    if (lane == 0 && !dry) {
      a.tau_ws[hs] = tau_d;
      if (a.tau_out) a.tau_out[hs] = tau_f;
      if (a.delta_out) {
        if (a.policy == ENTMAXKV_POLICY_GAUSSIAN)
          a.delta_out[hs] = L > 0 ? fminf(1.0f, fmaxf(0.0f, 1.0f - km_sh[hg])) : 0.0f;
        else if (a.policy == ENTMAXKV_POLICY_FULL)
          a.delta_out[hs] = 0.0f;
      }
    }
  }
  // The pages pass B must read: some head's page max above its τ. τ ≥ T0, so
  // every such page is among the pages step A kept (in shared memory unless
  // a head overflowed, then in its global candidate list). They are marked
  // in a rank bitmap (in the score region, free after D), read back in rank
  // order into a shared list over the page maxima (free now), and written
  // out with their logical and physical pages.
  __syncthreads();  // the solves are done with the scores; τ of every head is in tauf_sh
  if (spec_all) {
    // Every page of the V list is the page of some kept slot entry (its max
    // clears τ_h ≥ T0_h); the first entry to set the page's bit writes it,
    // with the (page, phys) its thread looked up in step A.
#pragma unroll
    for (int k = 0; k < kSlots; ++k) {
      if (((kept >> k) & 1u) && __int_as_float(ce[k].y) > tauf_sh[hs]) {
        const uint32_t bit = 1u << (ce[k].x & 31);
        if (!(atomicOr(&vb[ce[k].x >> 5], bit) & bit)) {
          const int pos = atomicAdd(&vcnt_sh, 1);
          if (!dry) a.vlist[skv * a.cap_pages + pos] = make_int4(ce[k].x, kpp[k].x, kpp[k].y, 0);
        }
      }
    }
    __syncthreads();
    if (tid == 0 && !dry) a.vcount[skv] = vcnt_sh;
    return;
  }
  if (dry) return;  // (a dry run always takes the path above)
  const int W = (n_sel + 31) >> 5;
  uint32_t* vbm = reinterpret_cast<uint32_t*>(zc);
  int* vls = reinterpret_cast<int*>(pool);
  if (W > kSolveCap / 2) {  // more ranks than the region holds bits: pass B scans them itself
    if (tid == 0) a.vcount[skv] = -1;
    return;
  }
  for (int i = tid; i < W; i += kThreads) vbm[i] = 0u;
  if (tid == 0) {
    int t = 0;
    for (int h = 0; h < G; ++h) {
      off_sh[h] = t;
      t += np_sh[h] <= capP ? np_sh[h] : nc_sh[h];
    }
    off_sh[G] = t;
  }
  __syncthreads();
  for (int e = tid; e < off_sh[G]; e += kThreads) {
    int h = 0;
    while (e >= off_sh[h + 1]) ++h;
    const int j = e - off_sh[h];
    int rank;
    float pmv;
    if (np_sh[h] <= capP) {
      rank = pr[h * capP + j];
      pmv = pv[h * capP + j];
    } else {
      const int2 c = __ldcg(clist + (size_t)h * a.cap_pages + j);
      rank = c.x;
      pmv = __int_as_float(c.y);
    }
    if (pmv > tauf_sh[h]) atomicOr(&vbm[rank >> 5], 1u << (rank & 31));
  }
  __syncthreads();
  const int wpt = (W + kThreads - 1) / kThreads, w0 = tid * wpt;
  int cnt = 0;
  for (int j = 0; j < wpt && w0 + j < W; ++j) cnt += __popc(vbm[w0 + j]);
  int total;
  int r = block_exclusive_scan(cnt, sh_scan, total);
  if (total > kSolveCap / 2) {  // the shared list would overrun the bitmap
    if (tid == 0) a.vcount[skv] = -1;
    return;
  }
  for (int j = 0; j < wpt && w0 + j < W; ++j) {
    uint32_t bits = vbm[w0 + j];
    while (bits) {
      vls[r++] = (w0 + j) * 32 + __ffs(bits) - 1;
      bits &= bits - 1u;
    }
  }
  __syncthreads();
  for (int i = tid; i < total; i += kThreads) {  // all lookups in flight together
    const int rank = vls[i];
    const int2 pp = __ldcg(&a.sel_pp[skv * a.cap_pages + rank]);
    a.vlist[skv * a.cap_pages + i] = make_int4(rank, pp.x, pp.y, 0);
  }
  if (tid == 0) a.vcount[skv] = total;
}

// ---------------------------------------------------------------------------

template <typename T>
struct VTraits;
template <>
struct VTraits<float> {
  static constexpr int VEC = 4;
  __device__ static void unpack(const uint4& r, float (&v)[4]) {
    v[0] = __uint_as_float(r.x);
    v[1] = __uint_as_float(r.y);
    v[2] = __uint_as_float(r.z);
    v[3] = __uint_as_float(r.w);
  }
};
template <>
struct VTraits<__nv_bfloat16> {
  static constexpr int VEC = 8;
  __device__ static void unpack(const uint4& r, float (&v)[8]) {
    v[0] = bf_lo(r.x); v[1] = bf_hi(r.x);
    v[2] = bf_lo(r.y); v[3] = bf_hi(r.y);
    v[4] = bf_lo(r.z); v[5] = bf_hi(r.z);
    v[6] = bf_lo(r.w); v[7] = bf_hi(r.w);
  }
};

// Pass B: for each kept page with some z above τ (every page with
// ENTMAXKV_FLAG_DENSE_V) the warp requests the page's V slab into its shared
// buffer (bf16: two TMA tensor boxes with 128-byte swizzle; fp32: one bulk
// copy), stages the page's z beside it, forms p once per (token, head), and
// accumulates p·v: bf16 on the tensor cores (V^T by ldmatrix.trans, p as
// bf16 hi + lo), fp32 with paired FMA in registers.
template <typename T, int D, int GP>
__global__ void __launch_bounds__(kThreads, GP <= 4 ? 2 : 1)
    pass_b_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap vmap) {
  pdl_enter();
  constexpr bool MMA = sizeof(T) == 2;           // bf16 pages: p·v on the tensor cores
  constexpr int VEC = VTraits<T>::VEC, LPR = D / VEC, TG = 32 / LPR;
  constexpr int MAXT = 32 / TG;                  // rows per lane in a 32-token page
  __shared__ double tau_sh[GP];
  __shared__ __align__(16) float zs[kWarps][32 * 8];
  __shared__ __align__(16) float red[kWarps][GP][D];
  __shared__ float dsum[kWarps][GP];
  __shared__ int list_sh[kListCap];
  __shared__ uint64_t vbar[kWarps];
  // fp32: [kWarps][P][D]; bf16: [kWarps][D/64][P][128 B] swizzled boxes, from a
  // 1024-byte boundary
  extern __shared__ __align__(128) unsigned char vstage[];
  __shared__ int scan_sh[32];
  __shared__ int last_sh;
  const int split = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G, P = a.P;
  const int dc = lane % LPR, tg = lane / LPR;
  const int seq = seq_row(a.seq_ids, s, a.max_seqs, nullptr);
  const int L = seq_len_clamped(a.seq_lens, seq, a.maxp, P, nullptr);
  const int n_pages = (L + P - 1) / P;
  const bool bitmap = uses_bitmap(a.policy);
  const size_t skv = (size_t)s * a.Hkv + kvh;
  const size_t hq0 = (size_t)s * a.Hq + (size_t)kvh * G;
  const int n_sel = bitmap ? __ldcg(&a.nsel_ws[skv]) : n_pages;
  const int lo = (int)(((long long)n_sel * split) / a.splits);
  const int hi = (int)(((long long)n_sel * (split + 1)) / a.splits);
  if (tid < GP) tau_sh[tid] = tid < G ? __ldcg(&a.tau_ws[hq0 + tid]) : CUDART_INF;
  const bool dense = (a.flags & ENTMAXKV_FLAG_DENSE_V) != 0;
  // Pass A's count of pages that need V, and this warp's entry of its list at
  // the fixed position block·kWarps + warp (where it is whenever the list
  // holds at most kWarps pages a block), both loaded with the values above so
  // the V copy can be issued after one round trip.
  const int vc = dense ? -1 : __ldcg(&a.vcount[skv]);
  const int spec_i = split * kWarps + warp;
  int4 spec_e = make_int4(0, 0, -1, 0);
  if (!dense && spec_i < a.cap_pages) spec_e = __ldcg(&a.vlist[skv * a.cap_pages + spec_i]);
  __syncthreads();
  float tau[GP];   // bf16 pages: p from fp32 z − τ
  double taud[GP]; // fp32 pages: p from z − τ in double (z's own rounding only)
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    taud[h] = tau_sh[h];
    tau[h] = (float)taud[h];
  }
  unsigned long long accp[GP][VEC / 2];  // fp32: pairs of columns, for the paired FMA
#pragma unroll
  for (int h = 0; h < GP; ++h)
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) accp[h][i] = 0ull;
  // bf16: out^T = V^T·p per m16n8k16 tile (16 dims × 8 heads, 16 tokens deep);
  // lane l holds dims 16m + l/4 (+8) of heads 2(l%4), 2(l%4) + 1
  float cacc[MMA ? D / 16 : 1][4];
#pragma unroll
  for (int m = 0; m < (MMA ? D / 16 : 1); ++m) cacc[m][0] = cacc[m][1] = cacc[m][2] = cacc[m][3] = 0.0f;
  float* zw = zs[warp];

  // One page: its V slab (P rows × D) arrives in this warp's shared buffer
  // by one bulk copy completing on the warp's mbarrier, its z is staged next
  // to it, and a compact row loop accumulates p·v in fp32 (lane: VEC columns
  // of rows tg, tg+TG, ...). The loop is kept small on purpose: it runs once
  // per page, usually with cold instruction caches.
  const uint32_t vs_base = (smem_u32(vstage) + 1023u) & ~1023u;
  unsigned char* vbase = vstage + (vs_base - smem_u32(vstage));
  T* vbuf = reinterpret_cast<T*>(MMA ? vbase : vstage) + (size_t)warp * P * D;
  if (lane == 0) {
    mbar_init(&vbar[warp], 1);
    mbar_fence_init();
  }
  __syncwarp();
  uint32_t vphase = 0u;
  bool stuck = false;  // a copy did not arrive within the bound (warp-uniform)
  auto do_page = [&](int rank, int pg, int ph) {
    if (stuck) return;
    const int nv = min(P, L - pg * P);
    const uint32_t bytes = (uint32_t)(P * D * sizeof(T));
    if (lane == 0) {
      mbar_expect_tx(&vbar[warp], bytes);
      if constexpr (MMA) {
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tma_load_3d(reinterpret_cast<unsigned char*>(vbuf) + hf * P * 128, &vmap, 64 * hf, kvh * P, ph,
                      &vbar[warp]);
      } else {
        bulk_g2s(vbuf, (const T*)a.v_pool + ((size_t)ph * a.Hkv + kvh) * P * D, bytes, &vbar[warp]);
      }
    }
    const float* zb = a.z + (skv * a.cap_pages + rank) * (size_t)P * G;
#pragma unroll
    for (int u = 0; u < 2; ++u) {  // P·G ≤ 256 floats: two float4 per lane at most
      const int e = 4 * lane + 128 * u;
      if (e < P * G) *reinterpret_cast<float4*>(zw + e) = __ldcg(reinterpret_cast<const float4*>(zb + e));
    }
    __syncwarp();  // the staged z is visible to the whole warp
    // p of every (row, head) once, in place: [z − τ_h]_+^β, 0 past the valid rows
    for (int e = lane; e < P * G; e += 32) {
      const int t = e / G, h = e - t * G;
      float th = tau[0];
      double thd = taud[0];
#pragma unroll
      for (int hh = 1; hh < GP; ++hh)
        if (h == hh) {
          th = tau[hh];
          thd = taud[hh];
        }
      const float zv = zw[e];
      zw[e] = t >= nv ? 0.0f
                      : (sizeof(T) == 4 ? pos_pow((float)((double)zv - thd), a.beta) : pos_pow(zv - th, a.beta));
    }
    __syncwarp();
    const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&vbar[warp], vphase));
    if (!ok) {
      stuck = true;
      return;
    }
    vphase ^= 1u;
    if constexpr (MMA) {
      unsigned char* vb = reinterpret_cast<unsigned char*>(vbuf);
      if (nv < P) {  // token slots past the sequence's end: zero, so p = 0 meets no NaN
        for (int e = lane; e < (D / 64) * (P - nv) * 8; e += 32) {
          const int hf = e / ((P - nv) * 8), rem = e - hf * (P - nv) * 8;
          *reinterpret_cast<uint4*>(vb + hf * P * 128 + (nv + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }
      const int c = lane & 3, r = lane >> 2;
      const uint32_t vb_s = smem_u32(vb);
#pragma unroll
      for (int ks = 0; ks < P / 16; ++ks) {
        // B = p (tokens × heads): tokens 16ks + 2c (+1) and +8, head r
        const int t0 = 16 * ks + 2 * c;
        const bool hv = r < G;
        uint32_t bh0, bl0, bh1, bl1;
        bf16_split2(hv ? zw[t0 * G + r] : 0.0f, hv ? zw[(t0 + 1) * G + r] : 0.0f, bh0, bl0);
        bf16_split2(hv ? zw[(t0 + 8) * G + r] : 0.0f, hv ? zw[(t0 + 9) * G + r] : 0.0f, bh1, bl1);
        // A = V^T (dims × tokens): lane i addresses token 16ks + i%8 (+8 for
        // tiles 2, 3) in the 16-byte chunk of dims 16m (+8 for tiles 1, 3)
        const int tr = 16 * ks + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
        for (int m = 0; m < D / 16; ++m) {
          const int ch = 2 * m + ((lane >> 3) & 1);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(a0, a1, a2, a3, vb_s + (ch >> 3) * P * 128 + swz128(tr, ch & 7));
          mma_bf16(cacc[m], a0, a1, a2, a3, bh0, bh1);
          mma_bf16(cacc[m], a0, a1, a2, a3, bl0, bl1);
        }
      }
      __syncwarp();  // the buffer and zw are refilled for the next page
      return;
    }
    const T* vrow = vbuf + dc * VEC;
#pragma unroll 2
    for (int u = 0; u < MAXT; ++u) {
      const int t = tg + TG * u;
      if (t < nv) {
        float v[VEC];
        VTraits<T>::unpack(*reinterpret_cast<const uint4*>(vrow + (size_t)t * D), v);
        unsigned long long vp[VEC / 2];
#pragma unroll
        for (int i = 0; i < VEC / 2; ++i) vp[i] = f2_pack(v[2 * i], v[2 * i + 1]);
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          if (h < G) {
            const float pw = zw[t * G + h];
            const unsigned long long pp = f2_pack(pw, pw);
#pragma unroll
            for (int i = 0; i < VEC / 2; ++i) accp[h][i] = f2_fma(pp, vp[i], accp[h][i]);
          }
        }
      }
    }
    __syncwarp();  // the buffer and zw are refilled for the next page
  };

  // Pages that need V: some head's page max above its τ (every page with
  // ENTMAXKV_FLAG_DENSE_V). Unless every page needs V, each block lists those
  // ranks of the whole selection in rank order (a thread checks up to 32
  // consecutive ranks, one scan places them); the first `parts` blocks take
  // even shares of the list, a warp per page, so pages that cluster in rank
  // still spread over the grid, and only those blocks add to the output. Larger
  // selections are walked in the block's own rank range, kListCap ranks at a
  // time. Either way the block's pages sit in list_sh in rank order.
  int parts = a.splits;
  bool global_list = false;
  bool spec_ok = false;  // this block's share starts at split·kWarps: the warps hold their entries
  int n_list = 0;
  const int4* vl = nullptr;  // this block's share of pass A's list, when it built one
  if (vc >= 0) {
    // top-k keeps every block: each one also sums its share of the δ̄ bound
    parts = a.policy == ENTMAXKV_POLICY_TOPK ? a.splits : max(1, min(a.splits, (vc + kWarps - 1) / kWarps));
    global_list = true;
    if (vc <= kWarps * a.splits) {  // kWarps pages a block, in list order
      spec_ok = true;
      n_list = max(0, min(kWarps, vc - split * kWarps));
    } else if (split < parts) {
      const int s_lo = (int)(((long long)vc * split) / parts);
      n_list = (int)(((long long)vc * (split + 1)) / parts) - s_lo;
      vl = a.vlist + skv * a.cap_pages + s_lo;
    }
  } else if (!dense && n_sel <= 32 * kThreads) {
    const int per = (n_sel + kThreads - 1) / kThreads;
    const int r0 = tid * per;
    uint32_t mask = 0u;
    for (int k = 0; k < per; ++k) {
      const int r = r0 + k;
      if (r < n_sel) {
        const float* pm = a.pmax + (skv * a.cap_pages + r) * (size_t)G;
        bool need = false;
#pragma unroll
        for (int h = 0; h < GP; ++h)
          if (h < G) need = need || (__ldcg(pm + h) > tau[h]);
        if (need) mask |= 1u << k;
      }
    }
    int nv_all;
    int j = block_exclusive_scan(__popc(mask), scan_sh, nv_all);
    // top-k keeps every block: each one also sums its share of the δ̄ bound
    const int pb = a.policy == ENTMAXKV_POLICY_TOPK
                       ? a.splits
                       : max(1, min(a.splits, (nv_all + kWarps - 1) / kWarps));
    if ((nv_all + pb - 1) / pb <= kListCap) {
      global_list = true;
      parts = pb;
      const int s_lo = split < pb ? (int)(((long long)nv_all * split) / pb) : 0;
      const int s_hi = split < pb ? (int)(((long long)nv_all * (split + 1)) / pb) : 0;
      n_list = s_hi - s_lo;
      while (mask && j < s_hi) {
        const int k = __ffs(mask) - 1;
        mask &= mask - 1u;
        if (j >= s_lo) list_sh[j - s_lo] = r0 + k;
        ++j;
      }
    }
    __syncthreads();
  }
  if (split >= parts) return;  // no pages and no partial (block-uniform)
  const int nb = hi - lo;
  for (int c0 = 0; c0 < (global_list ? 1 : nb); c0 += kListCap) {
    if (!global_list) {  // this chunk of the block's range: 4 ranks a thread
      const int cn = min(kListCap, nb - c0);
      uint32_t mask = 0u;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = 4 * tid + k;
        if (i < cn) {
          bool need = dense;
          const float* pm = a.pmax + (skv * a.cap_pages + lo + c0 + i) * (size_t)G;
#pragma unroll
          for (int h = 0; h < GP; ++h)
            if (h < G) need = need || (__ldcg(pm + h) > tau[h]);
          if (need) mask |= 1u << k;
        }
      }
      int j = block_exclusive_scan(__popc(mask), scan_sh, n_list);
      while (mask) {
        const int k = __ffs(mask) - 1;
        mask &= mask - 1u;
        list_sh[j++] = lo + c0 + 4 * tid + k;
      }
      __syncthreads();
    }
    for (int jj = warp; jj < n_list; jj += kWarps) {
      if (spec_ok) {
        if (spec_e.z >= 0) do_page(spec_e.x, spec_e.y, spec_e.z);
      } else if (vl) {
        const int4 e = __ldcg(vl + jj);
        if (e.z >= 0) do_page(e.x, e.y, e.z);
      } else {
        const int rank = list_sh[jj];
        const int2 pp = __ldcg(&a.sel_pp[skv * a.cap_pages + rank]);
        if (pp.y >= 0) do_page(rank, pp.x, pp.y);
      }
    }
    __syncthreads();  // list_sh is rewritten by the next chunk
  }
  float acc[GP][VEC];
#pragma unroll
  for (int h = 0; h < GP; ++h)
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) f2_unpack(accp[h][i], acc[h][2 * i], acc[h][2 * i + 1]);
  if (stuck) {
    // flag it; the copy still in flight is waited for (bounded) before leaving
    if (lane == 0) {
      raise_flag(a.status, ENTMAXKV_DEV_TIMEOUT);
      mbar_wait_bounded(&vbar[warp], vphase);
    }
    __syncwarp();
  }
  if constexpr (MMA) {
    const int c = lane & 3, r = lane >> 2;
#pragma unroll
    for (int m = 0; m < D / 16; ++m) {
      if (2 * c < GP) {
        red[warp][2 * c][16 * m + r] = cacc[m][0];
        red[warp][2 * c][16 * m + r + 8] = cacc[m][2];
      }
      if (2 * c + 1 < GP) {
        red[warp][2 * c + 1][16 * m + r] = cacc[m][1];
        red[warp][2 * c + 1][16 * m + r + 8] = cacc[m][3];
      }
    }
  } else {
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
      for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[h][j] += __shfl_xor_sync(0xffffffffu, acc[h][j], o);
    if (tg == 0) {
#pragma unroll
      for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int j = 0; j < VEC; ++j) red[warp][h][dc * VEC + j] = acc[h][j];
    }
  }
  // top-k: this block's share of the certified dropped mass
  if (a.policy == ENTMAXKV_POLICY_TOPK) {
    float dd[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) dd[h] = 0.0f;
    const uint32_t* bm = a.bitmap + skv * a.words;
    const int plo = (int)(((long long)n_pages * split) / a.splits);
    const int phi = (int)(((long long)n_pages * (split + 1)) / a.splits);
    // four pages a thread per round, their loads issued together
    for (int p0 = plo + tid; p0 < phi; p0 += 4 * kThreads) {
      uint32_t w[4];
      float u[4][GP];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int p = p0 + j * kThreads;
        w[j] = p < phi ? bm[p >> 5] : 0xffffffffu;
#pragma unroll
        for (int h = 0; h < GP; ++h) u[j][h] = (p < phi && h < G) ? a.bbox_u[(hq0 + h) * a.maxp + p] : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int p = p0 + j * kThreads;
        if (p >= phi || ((w[j] >> (p & 31)) & 1u)) continue;  // kept pages carry no dropped mass
        const float np = (float)(p == n_pages - 1 ? L - p * P : P);
#pragma unroll
        for (int h = 0; h < GP; ++h)
          if (h < G) dd[h] += np * pos_pow(a.a1 * u[j][h] - tau[h], a.beta);
      }
    }
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      const float w = warp_sum(dd[h]);
      if (lane == 0) dsum[warp][h] = w;
    }
  }
  __syncthreads();
  // The block's sums go straight into the output (zeroed by pass A) as
  // vector float additions: no partials, no ticket, no combine. The order of
  // the additions is the order blocks finish in.
  float4* orow = reinterpret_cast<float4*>(a.out + hq0 * D);
  for (int e = tid; e < G * D / 4; e += kThreads) {
    const int h = (4 * e) / D, d = (4 * e) % D;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float4 r = *reinterpret_cast<const float4*>(&red[w][h][d]);
      sum.x += r.x;
      sum.y += r.y;
      sum.z += r.z;
      sum.w += r.w;
    }
    atomicAdd(orow + e, sum);
  }
  if (a.policy != ENTMAXKV_POLICY_TOPK) return;
  // top-k: the last block turns the summed dropped-mass terms into δ̄
  if (tid < G) {
    float sum = 0.0f;
    for (int w = 0; w < kWarps; ++w) sum += dsum[w][tid];
    if (sum != 0.0f) atomicAdd(&a.dbar[hq0 + tid], sum);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last_sh = atomicAdd(&a.cnt_b[skv], 1) == parts - 1;
  __syncthreads();
  if (!last_sh) return;
  __threadfence();
  if (a.delta_out && tid < G)
    a.delta_out[hq0 + tid] = L > 0 ? fminf(1.0f, __ldcg(&a.dbar[hq0 + tid])) : 0.0f;
}

// ---------------------------------------------------------------------------

// Exact dropped mass (summary §3).
// - Softmax over the top-k pages: δ = 1 − exp(lse_kept − lse_full), from the
//   two log-normalisers.
// - Entmax: with τ and z of the full-cache solve in f's workspace and the
//   kept pages of the decode in m's, one block per (sequence, KV head) sums
//   p_i^full = [z_i − τ_full]_+^β over the kept pages' tokens (a warp per
//   page, lanes over tokens) and writes δ = max(0, 1 − Σ kept p_i^full) for
//   every query head of the group.
__global__ void __launch_bounds__(kThreads) exact_delta_kernel(DecodeArgs m, DecodeArgs f) {
  pdl_enter();
  __shared__ float part[kWarps][8];
  const int kvh = blockIdx.x, s = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = m.G, P = m.P;
  const int seq = seq_row(m.seq_ids, s, m.max_seqs, nullptr);
  const int L = seq_len_clamped(m.seq_lens, seq, m.maxp, P, nullptr);
  const int n_pages = (L + P - 1) / P;
  const size_t skv = (size_t)s * m.Hkv + kvh;
  const size_t hq0 = (size_t)s * m.Hq + (size_t)kvh * G;
  const bool bitmap = uses_bitmap(m.policy);
  if (m.policy == ENTMAXKV_POLICY_SOFTMAX_TOPK) {
    // softmax: the kept share of the full normaliser is exp(lse_kept − lse_full)
    if (tid < G && m.delta_out) {
      const double lk = __ldcg(&m.tau_ws[hq0 + tid]), lf = __ldcg(&f.tau_ws[hq0 + tid]);
      m.delta_out[hq0 + tid] = isnan(lf) ? 0.0f : (isnan(lk) ? 1.0f : (float)fmax(0.0, -expm1(lk - lf)));
    }
    return;
  }
  const int n_sel = bitmap ? __ldcg(&m.nsel_ws[skv]) : n_pages;
  double tau[8];
  float acc[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    tau[h] = h < G ? __ldcg(&f.tau_ws[hq0 + h]) : 0.0;
    acc[h] = 0.0f;
  }
  for (int r = warp; r < n_sel; r += kWarps) {
    const int page = bitmap ? __ldcg(&m.sel_list[skv * m.cap_pages + r]) : r;
    const float* zr = f.z + (skv * f.cap_pages + page) * (size_t)P * G;  // full cache: rank = page
    if (lane < P) {
#pragma unroll
      for (int h = 0; h < 8; ++h)
        if (h < G) acc[h] += pos_pow((float)((double)__ldcg(zr + lane * G + h) - tau[h]), f.beta);
    }
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const float w = warp_sum(acc[h]);
    if (lane == 0) part[warp][h] = w;
  }
  __syncthreads();
  if (tid < G && m.delta_out) {
    float kept = 0.0f;
    for (int w = 0; w < kWarps; ++w) kept += part[w][tid];
    m.delta_out[hq0 + tid] = isnan(tau[tid]) ? 0.0f : fmaxf(0.0f, 1.0f - kept);
  }
}

cudaError_t launch_exact_delta(const DecodeArgs& m, const DecodeArgs& f, cudaStream_t st) {
  return launch_k(false, exact_delta_kernel, dim3(m.Hkv, m.S), dim3(kThreads), 0, st, m, f);
}

static int pick_gp(int G) { return G <= 1 ? 1 : (G <= 2 ? 2 : (G <= 4 ? 4 : 8)); }

cudaError_t launch_pass_a(const DecodeArgs& a, int kv_dtype, cudaStream_t st) {
  dim3 grid(a.splits, a.Hkv, a.S);
  if (kv_dtype == ENTMAXKV_BF16) {
    if (a.D == 128) launch_k(false, pass_a_kernel<__nv_bfloat16, 128>, dim3(grid), dim3(kThreads), 0, st, a);
    else launch_k(false, pass_a_kernel<__nv_bfloat16, 64>, dim3(grid), dim3(kThreads), 0, st, a);
  } else {
    if (a.D == 128) launch_k(false, pass_a_kernel<float, 128>, dim3(grid), dim3(kThreads), 0, st, a);
    else launch_k(false, pass_a_kernel<float, 64>, dim3(grid), dim3(kThreads), 0, st, a);
  }
  return cudaGetLastError();
}

template <typename T, int D, int GP>
static cudaError_t pass_b_launch(const DecodeArgs& a, const CUtensorMap& vmap, dim3 grid, cudaStream_t st) {
  // one V slab per warp (bf16: plus the slack that aligns the boxes to 1024 bytes)
  constexpr int slack = sizeof(T) == 2 ? 1024 : 0;
  const int smem = kWarps * a.P * D * (int)sizeof(T) + slack;
  const cudaError_t e =
      ensure_smem((const void*)pass_b_kernel<T, D, GP>, kWarps * 32 * D * (int)sizeof(T) + slack);
  if (e != cudaSuccess) return e;
  launch_k(false, pass_b_kernel<T, D, GP>, dim3(grid), dim3(kThreads), smem, st, a, vmap);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t pass_b_g(const DecodeArgs& a, const CUtensorMap& vmap, dim3 grid, cudaStream_t st) {
  switch (pick_gp(a.G)) {
    case 1: return pass_b_launch<T, D, 1>(a, vmap, grid, st);
    case 2: return pass_b_launch<T, D, 2>(a, vmap, grid, st);
    case 4: return pass_b_launch<T, D, 4>(a, vmap, grid, st);
    default: return pass_b_launch<T, D, 8>(a, vmap, grid, st);
  }
}

cudaError_t launch_pass_b(const DecodeArgs& a, int kv_dtype, cudaStream_t st) {
  dim3 grid(a.splits, a.Hkv, a.S);
  CUtensorMap vmap;
  memset(&vmap, 0, sizeof(vmap));
  if (kv_dtype == ENTMAXKV_BF16) {
    const cudaError_t e = make_v_map(&vmap, a.v_pool, a.nphys, a.Hkv, a.P, a.D);
    if (e != cudaSuccess) return e;
    return a.D == 128 ? pass_b_g<__nv_bfloat16, 128>(a, vmap, grid, st)
                      : pass_b_g<__nv_bfloat16, 64>(a, vmap, grid, st);
  }
  return a.D == 128 ? pass_b_g<float, 128>(a, vmap, grid, st) : pass_b_g<float, 64>(a, vmap, grid, st);
}

}  // namespace ekv
