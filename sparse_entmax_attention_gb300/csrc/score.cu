// score.cu -- query-aware page scoring from per-page metadata.
//
// EntmaxKV (gist.science technical summary, §2A):
//  * bounding box: U_p = Σ_d max(q_d·kmin_d, q_d·kmax_d)/√d bounds every
//    token score of page p. With q⁺ = max(q,0), q⁻ = min(q,0) this is the
//    contraction U_p = (q⁺·kmax_p + q⁻·kmin_p)/√d, exact term by term.
//  * Gaussian statistics: token scores of page p modelled as N(μ_p, σ_p²)
//    with μ_p = q·mean_p/√d and σ_p² = Σ_d q_d²·var_{p,d}/d (diagonal model),
//    reported on the z scale: m_p = (α−1)μ_p, ς_p = (α−1)σ_p.
//
// bf16 metadata (both kinds): 8 pages' metadata rows against the group's
// query heads form m16n8k16 tiles (products of bf16 values are exact in the
// fp32 accumulator), with the pages' rows streamed through a ring of
// shared-memory stages by bulk copies (gauss_mma_kernel).
#include "common.cuh"

namespace ekv {

// Split a bf16 pair into its positive and negative parts (exact).
__device__ __forceinline__ void split_sign(uint32_t w, uint32_t& pos, uint32_t& neg) {
  uint32_t lo = w & 0xffffu, hi = w >> 16;
  uint32_t plo = (lo & 0x8000u) ? 0u : lo, nlo = (lo & 0x8000u) ? lo : 0u;
  uint32_t phi = (hi & 0x8000u) ? 0u : hi, nhi = (hi & 0x8000u) ? hi : 0u;
  pos = plo | (phi << 16);
  neg = nlo | (nhi << 16);
}

// fp32 metadata: one thread per page, q in shared memory.
template <int D>
__global__ void __launch_bounds__(kThreads) bbox_f32_kernel(DecodeArgs a) {
  pdl_enter();
  __shared__ float qs[8][D];
  const int kvh = blockIdx.y, s = blockIdx.z;
  clear_ctrl_slice(a.ctrl, a.ctrl_vec);
  const int seq = seq_row(a.seq_ids, s, a.max_seqs, threadIdx.x == 0 ? a.status : nullptr);
  if (seq < 0) return;
  const int L = seq_len_clamped(a.seq_lens, seq, a.maxp, a.P, threadIdx.x == 0 ? a.status : nullptr);
  const int n_pages = (L + a.P - 1) / a.P;
  for (int i = threadIdx.x; i < a.G * D; i += blockDim.x)
    qs[i / D][i % D] = ((const float*)a.q)[((size_t)s * a.Hq + (size_t)kvh * a.G) * D + i];
  __syncthreads();
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < n_pages; p += gridDim.x * blockDim.x) {
    const int ph = phys_page(a.block_table, seq, p, a.maxp, a.nphys, a.status);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (ph >= 0) {
      const float* lo = (const float*)a.kmin + ((size_t)ph * a.Hkv + kvh) * D;
      const float* hi = (const float*)a.kmax + ((size_t)ph * a.Hkv + kvh) * D;
      for (int d = 0; d < D; d += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(lo + d);
        const float4 h4 = *reinterpret_cast<const float4*>(hi + d);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, hv[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          if (h < a.G) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float qd = qs[h][d + e];
              acc[h] += fmaxf(qd * lv[e], qd * hv[e]);
            }
          }
        }
      }
    }
    float mx = -CUDART_INF_F;
    for (int h = 0; h < a.G; ++h) {
      const float u = ph >= 0 ? acc[h] * a.inv_sqrt_d : -CUDART_INF_F;
      a.bbox_u[((size_t)s * a.Hq + (size_t)kvh * a.G + h) * a.maxp + p] = u;
      mx = fmaxf(mx, u);
    }
    a.bbox_uhat[((size_t)s * a.Hkv + kvh) * a.maxp + p] = mx;
  }
}

// Gaussian page scores, streamed by page slab. A block covers a range of
// pages for up to 8 KV heads at once, so each page's mean and m2 rows for
// those heads are one contiguous run (KH·D floats) in each array: a stage of
// PPS pages is filled by 2·PPS bulk asynchronous copies completing on the
// stage's "full" mbarrier. Warp w scores KV head w of every staged page and
// then arrives on the stage's "empty" mbarrier; the producer (lane 0 of
// warp 0) refills a stage once all warps have released it, keeping NST−1
// stages in flight. Scoring: half-warp h takes pages h and h+2 of a stage;
// lane l of a half covers the 16-byte chunks l and l+16 of a row (conflict-
// free shared loads), with q and q² of those dims in registers as fp32 pairs
// for the paired FMA; a butterfly reduce-scatter over the 16 lanes leaves
// each of the 2·2·GP totals in some lane. GP = group padded to a power of 2.
// TM is the type of the streamed metadata: the fp32 mean and m2, or their
// bf16 copies (half the bytes; twice the stages, so as many bytes in flight).
constexpr int kGaussWarps = 8, kGaussPPS = 4;

template <typename TM>
__host__ __device__ constexpr int gauss_nst() {
  return sizeof(TM) == 4 ? 3 : 6;
}

template <typename TM, int D>
__host__ __device__ constexpr int gauss_smem_bytes() {
  return gauss_nst<TM>() * kGaussPPS * 2 * 8 * D * (int)sizeof(TM) + gauss_nst<TM>() * (16 + kGaussPPS * 4);
}

// The metadata arrays of type TM: mean (which = 0) or m2 (which = 1).
template <typename TM>
__device__ __forceinline__ const TM* gauss_meta(const DecodeArgs& a, int which) {
  if constexpr (sizeof(TM) == 4) return which ? a.m2 : a.mean;
  else return which ? a.m2_lo : a.mean_lo;
}

// N metadata values of one chunk (16 bytes, or 8 for 4 bf16 values) as floats.
template <typename TM, int N>
__device__ __forceinline__ void load_chunk(const TM* p, bool valid, float (&f)[N]) {
  static_assert(N * sizeof(TM) == 16 || N * sizeof(TM) == 8, "16- or 8-byte chunks");
  uint4 r = make_uint4(0u, 0u, 0u, 0u);
  if (valid) {
    if constexpr (N * sizeof(TM) == 16) {
      r = *reinterpret_cast<const uint4*>(p);
    } else {
      const uint2 h = *reinterpret_cast<const uint2*>(p);
      r.x = h.x;
      r.y = h.y;
    }
  }
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if constexpr (sizeof(TM) == 4) f[i] = __uint_as_float(w[i]);
    else f[i] = (i & 1) ? bf_hi(w[i >> 1]) : bf_lo(w[i >> 1]);
  }
}

template <typename TQ, typename TM, int D, int GP>
__global__ void __launch_bounds__(kGaussWarps * 32) gauss_kernel(DecodeArgs a) {
  pdl_enter();
  constexpr int DPL = D / 16;             // dims per lane (a half-warp covers a row)
  // metadata values in one chunk load: 16 bytes, capped at the lane's share of a row
  constexpr int VECM = (int)(16 / sizeof(TM)) < DPL ? (int)(16 / sizeof(TM)) : DPL;
  constexpr int CH = DPL / VECM;          // chunks per lane per row
  constexpr int PPS = kGaussPPS, NST = gauss_nst<TM>();
  constexpr int NV = 2 * 2 * GP;          // totals per half-warp per stage: page × (μ, σ²) × head
  extern __shared__ __align__(128) unsigned char dyn[];
  const int kv0 = blockIdx.y * 8, s = blockIdx.z;
  const int KH = min(8, a.Hkv - kv0);     // KV heads of this block
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, hl = lane & 15;
  const int kvh = kv0 + warp;
  const bool active = warp < KH;
  TM* stages = reinterpret_cast<TM*>(dyn);                               // [NST][PPS][2][KH][D]
  uint64_t* full = reinterpret_cast<uint64_t*>(dyn + NST * PPS * 2 * 8 * D * sizeof(TM));
  uint64_t* empty = full + NST;
  int* phys_sm = reinterpret_cast<int*>(empty + NST);                   // [NST][PPS]
  __shared__ uint32_t smax[8][GP];
  static_assert(NST * PPS <= 32, "warp 0 looks up the first stages' pages at once");
  // every block, with pages or not, clears its slice of the control words
  clear_ctrl_slice(a.ctrl, a.ctrl_vec);
  // this block's slot of the per-head maxima starts as "none"
  for (int i = threadIdx.x; i < KH * a.G; i += blockDim.x)
    a.mslot[((size_t)s * a.Hq + (size_t)kv0 * a.G + i) * a.mslots + blockIdx.x] = 0u;
  const int seq = seq_row(a.seq_ids, s, a.max_seqs, threadIdx.x == 0 ? a.status : nullptr);
  if (seq < 0) return;
  const int L = seq_len_clamped(a.seq_lens, seq, a.maxp, a.P, threadIdx.x == 0 ? a.status : nullptr);
  const int n_pages = (L + a.P - 1) / a.P;
  const int n_groups = (n_pages + PPS - 1) / PPS;
  // contiguous share of page groups for this block
  const int g_lo = (int)(((long long)n_groups * blockIdx.x) / gridDim.x);
  const int g_hi = (int)(((long long)n_groups * (blockIdx.x + 1)) / gridDim.x);
  const int n_mine = g_hi - g_lo;
  if (n_mine <= 0) return;
  const uint32_t row_bytes = (uint32_t)(KH * D * sizeof(TM));
  if (threadIdx.x < 8 * GP) smax[threadIdx.x / GP][threadIdx.x % GP] = 0u;

  // producer (warp 0): copy stage st's pages, whose physical ids are in
  // phys_sm (lanes 0..2·PPS−1 copy one run each: page lane/2, array lane%2)
  auto issue_copies = [&](int st) {
    const int ph = lane < 2 * PPS ? phys_sm[st * PPS + (lane >> 1)] : -1;
    const uint32_t valid = __ballot_sync(0xffffffffu, ph >= 0);
    if (lane == 0) mbar_expect_tx(&full[st], (uint32_t)__popc(valid) * row_bytes);
    __syncwarp();
    if (ph >= 0) {
      const TM* src = gauss_meta<TM>(a, lane & 1) + ((size_t)ph * a.Hkv + kv0) * D;
      TM* dst = stages + (((size_t)st * PPS + (lane >> 1)) * 2 + (lane & 1)) * KH * D;
      bulk_g2s(dst, src, row_bytes, &full[st]);
    }
  };
  // refill stage st with group g: look its pages up, then copy
  int n_issued = 0;  // fills issued so far (warp 0)
  auto issue = [&](int g, int st) {
    if (lane < PPS) {
      const int p = g * PPS + lane;
      phys_sm[st * PPS + lane] = p < n_pages ? phys_page(a.block_table, seq, p, a.maxp, a.nphys, a.status) : -1;
    }
    __syncwarp();
    issue_copies(st);
    ++n_issued;
  };
  if (warp == 0) {
    // The pipeline starts before anything else: barriers, then every page of
    // the first NST stages looked up in one round trip, then their copies.
    if (lane < NST) {
      mbar_init(&full[lane], 1);
      mbar_init(&empty[lane], kGaussWarps);
    }
    mbar_fence_init();
    __syncwarp();
    const int nfill = min(NST, n_mine);
    if (lane < NST * PPS) {
      const int j = lane / PPS, p = (g_lo + j) * PPS + lane % PPS;
      phys_sm[lane] = (j < nfill && p < n_pages)
                          ? phys_page(a.block_table, seq, p, a.maxp, a.nphys, a.status) : -1;
    }
    __syncwarp();
    for (int j = 0; j < nfill; ++j) issue_copies(j);
    n_issued = nfill;
  }

  unsigned long long qp[GP][DPL / 2], q2p[GP][DPL / 2];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    const bool hv = active && h < a.G;
    const TQ* qh = (const TQ*)a.q + ((size_t)s * a.Hq + (size_t)(hv ? kvh : 0) * a.G + (hv ? h : 0)) * D;
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
      for (int e = 0; e < VECM / 2; ++e) {  // dims of lane hl's chunk c, in pairs
        const int d0 = VECM * (hl + 16 * c) + 2 * e;
        const float x0 = hv ? to_f(qh[d0]) : 0.0f, x1 = hv ? to_f(qh[d0 + 1]) : 0.0f;
        qp[h][c * (VECM / 2) + e] = f2_pack(x0, x1);
        q2p[h][c * (VECM / 2) + e] = f2_pack(x0 * x0, x1 * x1);
      }
  }
  int idx = 0, nfin = NV;
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1)
    if (nfin > 1) {
      nfin >>= 1;
      if (hl & o) idx += nfin;
    }
  constexpr int NFIN = NV > 16 ? NV / 16 : 1;
  const int my_i = idx / (2 * GP), my_qty = (idx / GP) & 1, my_h0 = idx % GP;
  const int my_pg = 2 * my_i + half;  // page within the stage
  const bool writer = active && ((NV >= 16) || ((hl & (16 / NV - 1)) == 0));
  float runmax[NFIN];
#pragma unroll
  for (int i = 0; i < NFIN; ++i) runmax[i] = -CUDART_INF_F;
  const float inv_full = 1.0f / ((float)a.P * (float)D);

  __syncthreads();  // barriers initialised, q in registers

  const int wait_limit = (a.flags & ENTMAXKV_FLAG_EXPIRE_WAITS) ? 0 : kPollLimit;
  int stuck = 0;
  for (int j = 0; j < n_mine; ++j) {
    const int st = j % NST;
    const uint32_t par = (uint32_t)((j / NST) & 1);
    const int g = g_lo + j;
    if (!__all_sync(0xffffffffu, mbar_wait_limit(&full[st], par, wait_limit))) {  // warp-uniform
      stuck = 1;
      break;
    }
    float v[NV];
    int my_ph = -1;
    if (active) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int pg = 2 * i + half;
        const bool pv = phys_sm[st * PPS + pg] >= 0;
        const TM* mrow = stages + (((size_t)st * PPS + pg) * 2 * KH + warp) * D;
        const TM* vrow = mrow + (size_t)KH * D;
        unsigned long long mu[GP], sg[GP];
#pragma unroll
        for (int h = 0; h < GP; ++h) mu[h] = sg[h] = 0ull;
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          float mf[VECM], vf[VECM];
          load_chunk<TM, VECM>(mrow + VECM * (hl + 16 * c), pv, mf);
          load_chunk<TM, VECM>(vrow + VECM * (hl + 16 * c), pv, vf);
#pragma unroll
          for (int e = 0; e < VECM / 2; ++e) {
            const unsigned long long mp = f2_pack(mf[2 * e], mf[2 * e + 1]);
            const unsigned long long vp = f2_pack(vf[2 * e], vf[2 * e + 1]);
#pragma unroll
            for (int h = 0; h < GP; ++h) {
              mu[h] = f2_fma(qp[h][c * (VECM / 2) + e], mp, mu[h]);
              sg[h] = f2_fma(q2p[h][c * (VECM / 2) + e], vp, sg[h]);
            }
          }
        }
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          v[(i * 2 + 0) * GP + h] = f2_sum(mu[h]);
          v[(i * 2 + 1) * GP + h] = f2_sum(sg[h]);
        }
      }
      my_ph = phys_sm[st * PPS + my_pg];
    }
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&empty[st])) : "memory");
    if (warp == 0 && j + NST < n_mine) {  // refill once every warp released the stage
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[st], par))) {
        stuck = 1;
        break;
      }
      issue(g + NST, st);
    }
    if (!active) continue;
    int n = NV;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
      if (n > 1) {
        const int hf = n >> 1;
        const bool up = hl & o;
#pragma unroll
        for (int i = 0; i < NV / 2; ++i) {
          if (i < hf) {
            const float send = up ? v[i] : v[i + hf];
            const float keep = up ? v[i + hf] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        n = hf;
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
      }
    }
    const int p = g * PPS + my_pg;
#pragma unroll
    for (int i = 0; i < NFIN; ++i) {
      const int my_h = my_h0 + i;
      if (writer && my_h < a.G && p < n_pages) {
        float* dst = reinterpret_cast<float*>(
            a.gauss_ms + ((size_t)s * a.Hq + (size_t)kvh * a.G + my_h) * a.maxp + p);
        if (my_ph < 0) {  // unreadable page: no mass, never selected
          dst[my_qty] = my_qty == 0 ? -CUDART_INF_F : 0.0f;
        } else if (my_qty == 0) {
          const float m = a.a1 * v[i] * a.inv_sqrt_d;
          dst[0] = m;
          runmax[i] = fmaxf(runmax[i], m);
        } else {
          const int nv = min(a.P, L - p * a.P);
          const float inv_n = nv == a.P ? inv_full : 1.0f / ((float)nv * (float)D);
          dst[1] = a.a1 * sqrtf(fmaxf(v[i], 0.0f) * inv_n);
        }
      }
    }
  }
  if (stuck) {
    // A copy or a stage release never arrived within the bound: flag it and
    // stop. The producer waits (bounded) for the last fill it issued into
    // each stage, so no copy is still landing when the block exits.
    if (lane == 0) raise_flag(a.status, ENTMAXKV_DEV_TIMEOUT);
    if (warp == 0)
      for (int st = 0; st < NST; ++st) {
        const int f = ring_fills(n_issued, st, NST);
        if (f > 0) mbar_wait_bounded(&full[st], (uint32_t)((f - 1) & 1));
      }
  }
#pragma unroll
  for (int i = 0; i < NFIN; ++i)
    if (writer && my_qty == 0 && my_h0 + i < a.G && runmax[i] > -CUDART_INF_F)
      atomicMax(&smax[warp][my_h0 + i], ord_enc(runmax[i]));
  __syncthreads();
  if (threadIdx.x < 8 * GP) {
    const int w = threadIdx.x / GP, h = threadIdx.x % GP;
    if (w < KH && h < a.G)
      a.mslot[((size_t)s * a.Hq + (size_t)(kv0 + w) * a.G + h) * a.mslots + blockIdx.x] = smax[w][h];
  }
}

// Gaussian page scores on the tensor cores, for bf16 queries with the bf16
// metadata copies: μ = q·mean and σ² = Σ_d q_d²·m2_d are a dense contraction
// (pages × dims × heads) on m16n8k16 tiles of 8 pages. The products are exact
// in fp32: q·mean is bf16 × bf16, and q² (at most 16 significant bits) is
// split exactly into bf16 hi + lo, two MMAs whose sums are added. The tile's
// orientation depends on the group (the MODE comment below): up to 4 heads,
// the pages' rows are A and the queries B; larger groups the other way
// round. The streaming is the one of gauss_kernel: stages of 8 pages (for up
// to 8 KV heads) filled by bulk copies on full/empty mbarriers. Page runs sit
// 16 bytes apart modulo 128, so the 8 page rows an ldmatrix reads fall in
// different banks.
constexpr int kGaussMmaPPS = 8, kGaussMmaNST = 3;
constexpr int kGaussMmaPre = 512;  // physical ids of a block's pages looked up at the start

__host__ __device__ constexpr int gauss_mma_stage_bytes(int D) {
  return kGaussMmaPPS * (2 * 8 * D * 2 + 16);
}
__host__ __device__ constexpr int gauss_mma_smem_bytes(int D) {
  return kGaussMmaNST * gauss_mma_stage_bytes(D) + kGaussMmaNST * (16 + kGaussMmaPPS * 4);
}

__device__ __forceinline__ void ldsm_x2(uint32_t& r0, uint32_t& r1, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];\n"
               : "=r"(r0), "=r"(r1)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ uint32_t bf2_pack(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// MODE 0: the Gaussian statistics (μ, σ) from the bf16 mean and m2 copies;
// MODE 1: the bounding box U = (q⁺·kmax + q⁻·kmin)/√d from the bf16 kmax and
// kmin (exact term by term), per query head and as the group's maximum;
// MODE 2: MODE 0 for groups of at most 4 query heads with the operands
// swapped. The stage is A: rows 0-7 the 8 pages' mean, rows 8-15 their m2.
// The queries are B, held in registers for the whole kernel: columns 0-3
// are q and 4-7 q² hi, and a second B has zero and q² lo. Then
// C[mean row][q column] = μ and C[m2 row][q² column] = σ² (hi + lo from the
// two accumulators), and the rest of C is unused. A stage's A fragments fit
// in registers at once, so, as in MODE 1, a warp releases the stage before
// its MMAs and the refill does not wait on them. MODE 0 holds three query
// fragments per 16 dims instead and has no room for that;
// MODE 3: MODE 1 with the same swap. A: rows 0-7 the 8 pages' kmax, rows
// 8-15 their kmin; B: columns 0-3 q⁺ and 4-7 q⁻, so one MMA per 16 dims
// gives q⁺·kmax in C[kmax row][q⁺ column] and q⁻·kmin in C[kmin row][q⁻
// column].
template <int D, int MODE>
__global__ void __launch_bounds__(kGaussWarps * 32) gauss_mma_kernel(DecodeArgs a) {
  pdl_enter();
  constexpr int PPS = kGaussMmaPPS, NST = kGaussMmaNST, KS = D / 16;
  extern __shared__ __align__(128) unsigned char dyn[];
  const int kv0 = blockIdx.y * 8, s = blockIdx.z;
  const int KH = min(8, a.Hkv - kv0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = kv0 + warp;
  const bool active = warp < KH;
  const int run = KH * D * 2;                 // bytes of one (page, array) run: KH rows of D
  const int pstride = 2 * run + 16;           // bytes from one page's runs to the next's
  const int sstride = PPS * pstride;          // bytes of one stage
  uint64_t* full = reinterpret_cast<uint64_t*>(dyn + NST * gauss_mma_stage_bytes(D));
  uint64_t* empty = full + NST;
  int* phys_sm = reinterpret_cast<int*>(empty + NST);  // [NST][PPS]
  __shared__ uint32_t smax[8][8];
  __shared__ int phys_pre[kGaussMmaPre];
  static_assert(NST * PPS <= 32, "warp 0 looks up the first stages' pages at once");
  clear_ctrl_slice(a.ctrl, a.ctrl_vec);
  constexpr bool GAUSS = MODE == 0 || MODE == 2;
  constexpr bool BOX = !GAUSS;
  constexpr bool SWAP = MODE >= 2;  // metadata rows in A, queries in B
  if (GAUSS)
    for (int i = threadIdx.x; i < KH * a.G; i += blockDim.x)
      a.mslot[((size_t)s * a.Hq + (size_t)kv0 * a.G + i) * a.mslots + blockIdx.x] = 0u;
  // MODE 1 and 3: this block's largest bound Û per KV head (the top-k
  // select's lower bound), "no page" until the block has scored its pages;
  // lane 0 of the head's warp writes both, in order
  uint32_t* bslot = BOX && active ? a.mslot + ((size_t)s * a.Hkv + kvh) * a.mslots + blockIdx.x : nullptr;
  if (bslot && lane == 0) *bslot = ord_enc(-CUDART_INF_F);
  const int seq = seq_row(a.seq_ids, s, a.max_seqs, threadIdx.x == 0 ? a.status : nullptr);
  if (seq < 0) return;
  const int L = seq_len_clamped(a.seq_lens, seq, a.maxp, a.P, threadIdx.x == 0 ? a.status : nullptr);
  const int n_pages = (L + a.P - 1) / a.P;
  const int n_groups = (n_pages + PPS - 1) / PPS;
  const int g_lo = (int)(((long long)n_groups * blockIdx.x) / gridDim.x);
  const int g_hi = (int)(((long long)n_groups * (blockIdx.x + 1)) / gridDim.x);
  const int n_mine = g_hi - g_lo;
  if (n_mine <= 0) return;
  if (threadIdx.x < 64) smax[threadIdx.x >> 3][threadIdx.x & 7] = 0u;
  // the block's later pages (after the first NST stages) are looked up now,
  // all at once, so that a refill issues its copies without a dependent load.
  // Warps 1..7 do it: warp 0 goes straight to the first stages' lookups and
  // copies, which would otherwise wait behind these loads (one round trip
  // more before the block's first byte arrives).
  const int n_pre = min(kGaussMmaPre, n_mine * PPS);
  if (warp > 0)
    for (int i = NST * PPS + (int)threadIdx.x - 32; i < n_pre; i += (int)blockDim.x - 32) {
      const int p = g_lo * PPS + i;
      phys_pre[i] = p < n_pages ? phys_page(a.block_table, seq, p, a.maxp, a.nphys, a.status) : -1;
    }

  // producer (warp 0): lanes 0..2·PPS−1 copy one run each (page lane/2, array lane%2)
  auto issue_copies = [&](int st) {
    const int ph = lane < 2 * PPS ? phys_sm[st * PPS + (lane >> 1)] : -1;
    const uint32_t valid = __ballot_sync(0xffffffffu, ph >= 0);
    if (lane == 0) mbar_expect_tx(&full[st], (uint32_t)__popc(valid) * (uint32_t)run);
    __syncwarp();
    if (ph >= 0) {
      const __nv_bfloat16* arr = GAUSS ? ((lane & 1) ? a.m2_lo : a.mean_lo)
                                           : (const __nv_bfloat16*)((lane & 1) ? a.kmin : a.kmax);
      const __nv_bfloat16* src = arr + ((size_t)ph * a.Hkv + kv0) * D;
      bulk_g2s(dyn + st * sstride + (lane >> 1) * pstride + (lane & 1) * run, src, (uint32_t)run, &full[st]);
    }
  };
  int n_issued = 0;  // fills issued so far (warp 0)
  auto issue = [&](int g, int st) {
    if (lane < PPS) {
      const int p = g * PPS + lane, i = p - g_lo * PPS;
      phys_sm[st * PPS + lane] = p >= n_pages ? -1
                                 : i < n_pre ? phys_pre[i]
                                             : phys_page(a.block_table, seq, p, a.maxp, a.nphys, a.status);
    }
    __syncwarp();
    issue_copies(st);
    ++n_issued;
  };
  if (warp == 0) {
    if (lane < NST) {
      mbar_init(&full[lane], 1);
      mbar_init(&empty[lane], kGaussWarps);
    }
    mbar_fence_init();
    __syncwarp();
    const int nfill = min(NST, n_mine);
    if (lane < NST * PPS) {
      const int j = lane / PPS, p = (g_lo + j) * PPS + lane % PPS;
      phys_sm[lane] = (j < nfill && p < n_pages)
                          ? phys_page(a.block_table, seq, p, a.maxp, a.nphys, a.status) : -1;
    }
    __syncwarp();
    for (int j = 0; j < nfill; ++j) issue_copies(j);
    n_issued = nfill;
  }

  // Query fragments, dims 2(lane%4)+{0,1} and +8 of each 16-dim step.
  // MODE 0 and 1 (A): row lane/4 is a query head of the group, rows 8..15
  // are zero; MODE 0 holds q, q² hi, q² lo, MODE 1 q⁺ and q⁻ (in aq and ah;
  // al unused). MODE 2 (B): column lane/4 is head (lane/4)%4; lanes 0-15
  // hold q in aq and zero in ah, lanes 16-31 q² hi in aq and q² lo in ah.
  // MODE 3 (B): lanes 0-15 hold q⁺ in aq, lanes 16-31 q⁻.
  const int r = lane >> 2, cpair = 2 * (lane & 3);
  const int qrow = SWAP ? (r & 3) : r;
  const bool hv = active && r < a.G;
  const bool qv = active && qrow < a.G;
  const __nv_bfloat16* qh = (const __nv_bfloat16*)a.q + ((size_t)s * a.Hq + (size_t)(qv ? kvh : 0) * a.G + (qv ? qrow : 0)) * D;
  uint32_t aq[KS][2], ah[KS][2], al[KS][2];
#pragma unroll
  for (int k = 0; k < KS; ++k)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int d0 = 16 * k + 8 * u + cpair;
      const uint32_t w = qv ? *reinterpret_cast<const uint32_t*>(qh + d0) : 0u;
      if (MODE == 1) {
        split_sign(w, aq[k][u], ah[k][u]);
        al[k][u] = 0u;
        continue;
      }
      if (MODE == 3) {
        uint32_t pos, neg;
        split_sign(w, pos, neg);
        aq[k][u] = lane < 16 ? pos : neg;
        ah[k][u] = 0u;
        al[k][u] = 0u;
        continue;
      }
      if (MODE == 2 && lane < 16) {
        aq[k][u] = w;
        ah[k][u] = 0u;
        al[k][u] = 0u;
        continue;
      }
      aq[k][u] = w;
      const float x0 = bf_lo(w), x1 = bf_hi(w);
      const float s0 = x0 * x0, s1 = x1 * x1;  // exact: at most 16 significant bits
      const float h0 = __bfloat162float(__float2bfloat16_rn(s0)), h1 = __bfloat162float(__float2bfloat16_rn(s1));
      if (MODE == 2) {
        aq[k][u] = bf2_pack(h0, h1);
        ah[k][u] = bf2_pack(s0 - h0, s1 - h1);
        al[k][u] = 0u;
        continue;
      }
      ah[k][u] = bf2_pack(h0, h1);
      al[k][u] = bf2_pack(s0 - h0, s1 - h1);  // the exact remainders, representable in bf16
    }
  __syncthreads();  // barriers initialised

  const float inv_full = 1.0f / ((float)a.P * (float)D);
  float runmax = -CUDART_INF_F;
  const int lrow = lane & 7, lk = ((lane >> 3) & 1) * 16;  // ldmatrix: page row, byte offset in the step
  const int wait_limit = (a.flags & ENTMAXKV_FLAG_EXPIRE_WAITS) ? 0 : kPollLimit;
  int stuck = 0;
  for (int j = 0; j < n_mine; ++j) {
    const int st = j % NST;
    const uint32_t par = (uint32_t)((j / NST) & 1);
    const int g = g_lo + j;
    if (!__all_sync(0xffffffffu, mbar_wait_limit(&full[st], par, wait_limit))) {  // warp-uniform
      stuck = 1;
      break;
    }
    // independent accumulator chains, added at the end, so each chain waits
    // on its own MMAs only: MODE 0 three (μ, σ² hi, σ² lo), MODE 1 two
    // (q⁺·kmax, q⁻·kmin); MODE 2 and 3 deal their steps as their branch says
    float mu[4] = {0.f, 0.f, 0.f, 0.f}, sg[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
    int ph0 = -1, ph1 = -1;
    if constexpr (MODE == 1) {
      // the bounding box's fragments fit in registers at once: the stage is
      // released before the MMA chains run, so its refill does not wait on them
      uint32_t bm[KS][2], bv[KS][2];
      if (active) {
        const unsigned char* rowm = dyn + st * sstride + lrow * pstride + warp * D * 2 + lk;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
          ldsm_x2(bm[k][0], bm[k][1], rowm + 32 * k);
          ldsm_x2(bv[k][0], bv[k][1], rowm + run + 32 * k);
        }
        ph0 = phys_sm[st * PPS + cpair];
        ph1 = phys_sm[st * PPS + cpair + 1];
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&empty[st])) : "memory");
      if (warp == 0 && j + NST < n_mine) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[st], par))) {
          stuck = 1;
          break;
        }
        issue(g + NST, st);
      }
      if (active) {
#pragma unroll
        for (int k = 0; k < KS; ++k) {
          mma_bf16(mu, aq[k][0], 0u, aq[k][1], 0u, bm[k][0], bm[k][1]);  // q⁺·kmax
          mma_bf16(sg, ah[k][0], 0u, ah[k][1], 0u, bv[k][0], bv[k][1]);  // q⁻·kmin
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) mu[i] += sg[i];
      }
    } else if constexpr (SWAP) {
      // lanes 8j..8j+7 address tile j: pages lane%8, mean (j even) or m2
      // (j odd), dims 0-7 (j < 2) or 8-15 of the step
      uint32_t fa[KS][4];
      if (active) {
        const unsigned char* rowa = dyn + st * sstride + lrow * pstride + ((lane >> 3) & 1) * run + warp * D * 2 +
                                    (lane >> 4) * 16;
#pragma unroll
        for (int k = 0; k < KS; ++k) ldsm_x4(fa[k][0], fa[k][1], fa[k][2], fa[k][3], rowa + 32 * k);
        ph0 = phys_sm[st * PPS + r];
      }
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&empty[st])) : "memory");
      if (warp == 0 && j + NST < n_mine) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[st], par))) {
          stuck = 1;
          break;
        }
        issue(g + NST, st);
      }
      if (active) {
        // independent accumulator chains, summed at the end: a chain of
        // dependent MMAs is latency-bound, and the warp's next stage waits
        // for it. MODE 2: four chains of KS/2 (two chains cost 2 µs of the
        // 1M scoring); MODE 3: two chains of KS/2 (four measured 2 µs
        // slower).
        float sh[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < KS; ++k) {
          if (MODE == 2) {
            mma_bf16(k & 1 ? sl : mu, fa[k][0], fa[k][1], fa[k][2], fa[k][3], aq[k][0], aq[k][1]);  // μ; σ² hi
            mma_bf16(k & 1 ? sh : sg, fa[k][0], fa[k][1], fa[k][2], fa[k][3], ah[k][0], ah[k][1]);  // σ² lo
          } else {  // q⁺·kmax; q⁻·kmin, even and odd steps
            mma_bf16(k & 1 ? sg : mu, fa[k][0], fa[k][1], fa[k][2], fa[k][3], aq[k][0], aq[k][1]);
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (MODE == 2) {
            mu[i] += sl[i];
            sg[i] += sh[i];
          } else {
            mu[i] += sg[i];
          }
        }
      }
    } else if (active) {
      const unsigned char* rowm = dyn + st * sstride + lrow * pstride + warp * D * 2 + lk;
      const unsigned char* rowv = rowm + run;
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        uint32_t bm0, bm1, bv0, bv1;
        ldsm_x2(bm0, bm1, rowm + 32 * k);
        ldsm_x2(bv0, bv1, rowv + 32 * k);
        mma_bf16(mu, aq[k][0], 0u, aq[k][1], 0u, bm0, bm1);  // μ: q · mean
        mma_bf16(sg, ah[k][0], 0u, ah[k][1], 0u, bv0, bv1);  // σ²: q² hi · m2
        mma_bf16(sl, al[k][0], 0u, al[k][1], 0u, bv0, bv1);  //   + q² lo · m2
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sg[i] += sl[i];
      ph0 = phys_sm[st * PPS + cpair];
      ph1 = phys_sm[st * PPS + cpair + 1];
    }
    if constexpr (MODE == 0) {
      __syncwarp();
      if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(&empty[st])) : "memory");
      if (warp == 0 && j + NST < n_mine) {
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&empty[st], par))) {
          stuck = 1;
          break;
        }
        issue(g + NST, st);
      }
    }
    if (MODE == 1) {
      // U per query head, and the group's maximum per page (the lanes of one
      // page column differ in bits 2..4: the head)
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int p = g * PPS + cpair + u;
        const int ph = u ? ph1 : ph0;
        const float uv = (hv && ph >= 0) ? mu[u] * a.inv_sqrt_d : -CUDART_INF_F;  // unreadable: no bound mass
        float mx = uv;
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (p < n_pages && active) {
          if (hv) a.bbox_u[((size_t)s * a.Hq + (size_t)kvh * a.G + r) * a.maxp + p] = uv;
          if (r == 0) a.bbox_uhat[((size_t)s * a.Hkv + kvh) * a.maxp + p] = mx;
          runmax = fmaxf(runmax, mx);
        }
      }
      continue;
    }
    if (MODE == 3) {
      // lane l holds page l/4. With c = l%4: c < 2 has q⁺·kmax of heads 2c,
      // 2c+1 (mu[0..1]), c ≥ 2 q⁻·kmin of heads 2c−4, 2c−3 (mu[2..3]); one
      // exchange with lane l^2 gives U of one head: c = 0, 1, 2, 3 → head 0,
      // 2, 1, 3. The group's maximum per page is over the lanes of one page
      // (bits 0..1).
      const int c = lane & 3;
      const bool lowc = c < 2;
      const float got = __shfl_xor_sync(0xffffffffu, lowc ? mu[1] : mu[2], 2);
      const int hh = lowc ? 2 * c : 2 * c - 3;
      const int p = g * PPS + r;
      const bool hok = active && hh < a.G;
      const float uv = (hok && ph0 >= 0) ? ((lowc ? mu[0] : mu[3]) + got) * a.inv_sqrt_d : -CUDART_INF_F;
      float mx = uv;
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (p < n_pages && active) {
        if (hok) a.bbox_u[((size_t)s * a.Hq + (size_t)kvh * a.G + hh) * a.maxp + p] = uv;
        if (c == 0) a.bbox_uhat[((size_t)s * a.Hkv + kvh) * a.maxp + p] = mx;
        runmax = fmaxf(runmax, mx);
      }
      continue;
    }
    if (MODE == 2) {
      // lane l holds page l/4. With c = l%4: c < 2 has μ of heads 2c, 2c+1
      // (mu[0..1]); c ≥ 2 has σ² hi + lo of heads 2c−4, 2c−3 (mu[2..3] +
      // sg[2..3]). One exchange with lane l^2 leaves each lane (μ, σ²) of
      // one head: c = 0, 1, 2, 3 → head 0, 2, 1, 3.
      const int c = lane & 3;
      const bool lowc = c < 2;
      const float sq0 = mu[2] + sg[2], sq1 = mu[3] + sg[3];
      const float got = __shfl_xor_sync(0xffffffffu, lowc ? mu[1] : sq0, 2);
      const int hh = lowc ? 2 * c : 2 * c - 3;
      const float muv = lowc ? mu[0] : got, sgv = lowc ? got : sq1;
      const int p = g * PPS + r;
      if (!active || hh >= a.G || p >= n_pages) continue;
      float2* dst = a.gauss_ms + ((size_t)s * a.Hq + (size_t)kvh * a.G + hh) * a.maxp;
      if (ph0 < 0) {  // unreadable page: no mass, never selected
        dst[p] = make_float2(-CUDART_INF_F, 0.0f);
        continue;
      }
      const int nv = min(a.P, L - p * a.P);
      const float inv_n = nv == a.P ? inv_full : 1.0f / ((float)nv * (float)D);
      const float m = a.a1 * muv * a.inv_sqrt_d;
      dst[p] = make_float2(m, a.a1 * sqrtf(fmaxf(sgv, 0.0f) * inv_n));
      runmax = fmaxf(runmax, m);
      continue;
    }
    if (!hv) continue;
    float2* dst = a.gauss_ms + ((size_t)s * a.Hq + (size_t)kvh * a.G + r) * a.maxp;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int p = g * PPS + cpair + u;
      if (p >= n_pages) continue;
      const int ph = u ? ph1 : ph0;
      if (ph < 0) {  // unreadable page: no mass, never selected
        dst[p] = make_float2(-CUDART_INF_F, 0.0f);
        continue;
      }
      const int nv = min(a.P, L - p * a.P);
      const float inv_n = nv == a.P ? inv_full : 1.0f / ((float)nv * (float)D);
      const float m = a.a1 * mu[u] * a.inv_sqrt_d;
      dst[p] = make_float2(m, a.a1 * sqrtf(fmaxf(sg[u], 0.0f) * inv_n));
      runmax = fmaxf(runmax, m);
    }
  }
  if (stuck) {  // as in gauss_kernel: flag, then let the issued fills land
    if (lane == 0) raise_flag(a.status, ENTMAXKV_DEV_TIMEOUT);
    if (warp == 0)
      for (int st = 0; st < NST; ++st) {
        const int f = ring_fills(n_issued, st, NST);
        if (f > 0) mbar_wait_bounded(&full[st], (uint32_t)((f - 1) & 1));
      }
  }
  if (BOX) {
    runmax = warp_max(runmax);
    if (bslot && lane == 0 && !stuck && runmax > -CUDART_INF_F) *bslot = ord_enc(runmax);
    return;
  }
  if (MODE == 2) {
    // the lanes of one head differ in bits 2..4 (the page)
    runmax = fmaxf(runmax, __shfl_xor_sync(0xffffffffu, runmax, 4));
    runmax = fmaxf(runmax, __shfl_xor_sync(0xffffffffu, runmax, 8));
    runmax = fmaxf(runmax, __shfl_xor_sync(0xffffffffu, runmax, 16));
    const int hh = (lane & 3) < 2 ? 2 * (lane & 3) : 2 * (lane & 3) - 3;
    if (active && lane < 4 && hh < a.G && runmax > -CUDART_INF_F) smax[warp][hh] = ord_enc(runmax);
  } else {
    runmax = fmaxf(runmax, __shfl_xor_sync(0xffffffffu, runmax, 1));
    runmax = fmaxf(runmax, __shfl_xor_sync(0xffffffffu, runmax, 2));
    if (hv && (lane & 3) == 0 && runmax > -CUDART_INF_F) smax[warp][r] = ord_enc(runmax);
  }
  __syncthreads();
  if (threadIdx.x < 64) {
    const int w = threadIdx.x >> 3, h = threadIdx.x & 7;
    if (w < KH && h < a.G)
      a.mslot[((size_t)s * a.Hq + (size_t)(kv0 + w) * a.G + h) * a.mslots + blockIdx.x] = smax[w][h];
  }
}

template <int D, int MODE>
static cudaError_t gauss_mma_launch(const DecodeArgs& a, dim3 grid, cudaStream_t st) {
  constexpr int smem = gauss_mma_smem_bytes(D);
  static_assert(gauss_mma_smem_bytes(D) <= 227 * 1024, "stages exceed shared memory");
  cudaError_t e = ensure_smem((const void*)gauss_mma_kernel<D, MODE>, smem);
  if (e != cudaSuccess) return e;
  return launch_k(false, gauss_mma_kernel<D, MODE>, dim3(grid), dim3(kGaussWarps * 32), smem, st, a);
}

static int grid_x_for(int units, int per_block, int sms, int other_blocks) {
  int need = (units + per_block - 1) / per_block;
  int cap = (sms * 8 + other_blocks - 1) / other_blocks;  // ~8 blocks per SM overall
  if (cap < 1) cap = 1;
  if (need < 1) need = 1;
  return need < cap ? need : cap;
}

cudaError_t launch_bbox(const DecodeArgs& a, int kv_dtype, int sms, cudaStream_t st) {
  const int other = a.Hkv * a.S;
  if (kv_dtype == ENTMAXKV_BF16) {
    // the streamed tensor-core kernel, rows of up to 8 KV heads
    dim3 grid(a.mslots, (a.Hkv + 7) / 8, a.S);  // a.mslots = gauss_grid_x(maxp, Hkv, S, sms)
    const cudaError_t e =
        a.G <= 4 ? (a.D == 128 ? gauss_mma_launch<128, 3>(a, grid, st) : gauss_mma_launch<64, 3>(a, grid, st))
                 : (a.D == 128 ? gauss_mma_launch<128, 1>(a, grid, st) : gauss_mma_launch<64, 1>(a, grid, st));
    if (e != cudaSuccess) return e;
  } else {
    dim3 grid(grid_x_for(a.maxp, kThreads, sms, other), a.Hkv, a.S);
    if (a.D == 128) launch_k(false, bbox_f32_kernel<128>, dim3(grid), dim3(kThreads), 0, st, a);
    else launch_k(false, bbox_f32_kernel<64>, dim3(grid), dim3(kThreads), 0, st, a);
  }
  return cudaGetLastError();
}

template <typename TQ, typename TM, int D, int GP>
static cudaError_t gauss_launch(const DecodeArgs& a, dim3 grid, cudaStream_t st) {
  constexpr int smem = gauss_smem_bytes<TM, D>();
  static_assert(gauss_smem_bytes<TM, D>() <= 227 * 1024, "stages exceed shared memory");
  cudaError_t e = ensure_smem((const void*)gauss_kernel<TQ, TM, D, GP>, smem);
  if (e != cudaSuccess) return e;
  return launch_k(false, gauss_kernel<TQ, TM, D, GP>, dim3(grid), dim3(kGaussWarps * 32), smem, st, a);
}

template <typename TQ, typename TM, int D>
static cudaError_t gauss_dispatch_gm(const DecodeArgs& a, dim3 grid, cudaStream_t st) {
  if (a.G <= 1) return gauss_launch<TQ, TM, D, 1>(a, grid, st);
  if (a.G <= 2) return gauss_launch<TQ, TM, D, 2>(a, grid, st);
  if (a.G <= 4) return gauss_launch<TQ, TM, D, 4>(a, grid, st);
  return gauss_launch<TQ, TM, D, 8>(a, grid, st);
}

template <typename TQ, int D>
static cudaError_t gauss_dispatch_g(const DecodeArgs& a, dim3 grid, cudaStream_t st) {
  return a.mean_lo ? gauss_dispatch_gm<TQ, __nv_bfloat16, D>(a, grid, st)
                   : gauss_dispatch_gm<TQ, float, D>(a, grid, st);
}

// ~2 blocks per SM (96 KiB of stages each) over all (sequence, 8-KV-head)
// rows, at least 8 page groups per block; sms = 0 gives the largest grid any
// device uses (the workspace's count of per-block maxima slots).
int gauss_grid_x(int maxp, int Hkv, int S, int sms) {
  const int groups = (maxp + kGaussPPS - 1) / kGaussPPS;
  const int rows = ((Hkv + 7) / 8) * S;
  int gx = (groups + 7) / 8;
  if (sms > 0) {
    // One sequence: one wave of 2 blocks per SM. Several sequences, whose
    // lengths differ: four waves' worth of blocks, each sequence's split
    // evenly, so that the many blocks of the long ones spread over the SMs
    // that the short ones leave early.
    const int waves = S > 1 ? 8 : 2;
    const int cap = (waves * sms + rows - 1) / rows;
    if (gx > cap) gx = cap;
  }
  return gx < 1 ? 1 : gx;
}

cudaError_t launch_gauss(const DecodeArgs& a, int kv_dtype, int sms, cudaStream_t st) {
  dim3 grid(a.mslots, (a.Hkv + 7) / 8, a.S);
  cudaError_t e;
  if (kv_dtype == ENTMAXKV_BF16 && a.mean_lo)  // bf16 q and metadata: tensor cores
    e = a.G <= 4 ? (a.D == 128 ? gauss_mma_launch<128, 2>(a, grid, st) : gauss_mma_launch<64, 2>(a, grid, st))
                 : (a.D == 128 ? gauss_mma_launch<128, 0>(a, grid, st) : gauss_mma_launch<64, 0>(a, grid, st));
  else if (kv_dtype == ENTMAXKV_BF16)
    e = a.D == 128 ? gauss_dispatch_g<__nv_bfloat16, 128>(a, grid, st)
                   : gauss_dispatch_g<__nv_bfloat16, 64>(a, grid, st);
  else
    e = a.D == 128 ? gauss_dispatch_g<float, 128>(a, grid, st) : gauss_dispatch_g<float, 64>(a, grid, st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ekv
