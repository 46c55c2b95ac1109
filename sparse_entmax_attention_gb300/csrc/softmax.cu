// softmax.cu -- full-cache softmax decode, the FlashDecoding-style baseline
// the EntmaxKV summary compares against (gist.science technical summary, §4
// "Efficiency": speedups over full-cache softmax FlashDecoding).
//
// Split-K over pages: each warp streams its pages once (K then V of the same
// page), keeps an online softmax (running max m, running sum l, accumulator
// Σ 2^{s−m} v) per query head in the base-2 domain, the block merges its warps
// and writes (m, l, acc) as a partial, and the last block to finish merges the
// partials in split order. The "τ" output carries log Σ_i exp(s_i).
// bf16 pages: the scores are m16n8k16 MMAs on K loaded straight into the
// fragments; the page's V arrives by two TMA tensor boxes (128-byte swizzle)
// while they run, and Σ 2^{s−m} v is out^T = V^T·p on the tensor cores (V^T by
// ldmatrix.trans, p split into bf16 hi + lo), the fragments rescaled per head
// when a head's running max grows.
//
// With ENTMAXKV_POLICY_SOFTMAX_TOPK the same kernel runs over the top-k
// selected pages only (the softmax side of the summary's comparison at equal
// budget), and δ is certified: the full normaliser A + B has B, the mass of
// the dropped tokens, at most B̄ = Σ_dropped n_p·e^{U_p} (every token of page
// p scores ≤ U_p), and δ = B/(A + B) grows in B, so δ ≤ D/(1 + D) with
// D = B̄/A. Each block also folds its share of the dropped pages into a
// per-head (max, Σ n_p·e^{U_p − max}) pair that the last block merges.
#include "common.cuh"

#include "page_scores.cuh"

namespace ekv {

template <typename T, int D, int GP>
__global__ void __launch_bounds__(kThreads, 2)
    softmax_kernel(DecodeArgs a, const __grid_constant__ CUtensorMap vmap) {
  pdl_enter();
  constexpr bool MMA = sizeof(T) == 2;  // bf16 pages: p·v on the tensor cores
  constexpr int VEC = 16 / sizeof(T), LPR = D / VEC, TG = 32 / LPR;
  constexpr int MAXT = 32 / TG;                  // tokens per lane in a 32-token page
  constexpr int CH = MAXT < 8 ? MAXT : 8;        // V rows in flight per lane
  // q and the page scores live during the page loop, the per-warp sums after
  // it: one buffer, with a barrier between the two uses
  constexpr int kLoopFloats = 8 * D + kWarps * 32 * GP, kRedFloats = kWarps * GP * D;
  __shared__ __align__(16) float buf_sm[kLoopFloats > kRedFloats ? kLoopFloats : kRedFloats];
  float(*qs)[D] = reinterpret_cast<float(*)[D]>(buf_sm);
  float(*sbuf)[32][GP] = reinterpret_cast<float(*)[32][GP]>(buf_sm + 8 * D);
  float(*red)[GP][D] = reinterpret_cast<float(*)[GP][D]>(buf_sm);
  __shared__ float pmx[kWarps][8];
  __shared__ float wm_sh[kWarps][GP], wl_sh[kWarps][GP];
  __shared__ float4 red4[kThreads];
  __shared__ float Mg_sh[8], Lg_sh[8];
  __shared__ float um_sh[kWarps][8], us_sh[kWarps][8];
  static_assert(sizeof(red4) >= kListCap * sizeof(int), "the page list shares the combine scratch");
  int* list = reinterpret_cast<int*>(red4);  // the page list is done before the combine starts
  __shared__ int sh_scan[32];
  __shared__ int last_sh;
  __shared__ uint64_t vbar[kWarps];
  // bf16: a V slab per warp, [kWarps][D/64][P][128 B] swizzled boxes from a
  // 1024-byte boundary
  extern __shared__ __align__(128) unsigned char vstage_sm[];
  const int split = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G, P = a.P;
  const int dc = lane % LPR, tg = lane / LPR;
  const int seq = seq_row(a.seq_ids, s, a.max_seqs, tid == 0 ? a.status : nullptr);
  const int L = seq_len_clamped(a.seq_lens, seq, a.maxp, P, tid == 0 ? a.status : nullptr);
  const int n_pages = (L + P - 1) / P;
  const bool bitmap = uses_bitmap(a.policy);  // softmax over the top-k pages
  int n_sel, lo, hi;
  block_page_range(a, s, kvh, n_pages, split, list, sh_scan, n_sel, lo, hi);
  const size_t skv = (size_t)s * a.Hkv + kvh;
  const size_t hq0 = (size_t)s * a.Hq + (size_t)kvh * G;
  if (split == 0 && tid == 0 && a.n_sel_out) a.n_sel_out[skv] = n_sel;
  if (a.page_ids)
    for (int i = tid; i < hi - lo; i += kThreads)
      a.page_ids[skv * a.page_ids_stride + lo + i] = bitmap ? list[i] : lo + i;
  const float scale2 = a.inv_sqrt_d * 1.4426950408889634f;  // scores in log2 units
  uint32_t bq[D / 16][2];
  if constexpr (sizeof(T) == 2) {
    load_q_bfrag<D>((const __nv_bfloat16*)a.q + hq0 * D, G, lane, bq);
  } else {
    for (int i = tid; i < G * D; i += kThreads) qs[i / D][i % D] = ((const float*)a.q)[hq0 * D + i];
    __syncthreads();
  }
  float m[GP], l[GP], acc[MMA ? 1 : GP][VEC];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    m[h] = -CUDART_INF_F;
    l[h] = 0.0f;
  }
#pragma unroll
  for (int h = 0; h < (MMA ? 1 : GP); ++h)
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[h][j] = 0.0f;
  // bf16: out^T = V^T·p per m16n8k16 tile (16 dims × 8 heads, 16 tokens deep);
  // lane l holds dims 16m + l/4 (+8) of heads 2(l%4), 2(l%4) + 1, and the
  // running sum of p for head l/4 over its tokens
  float cacc[MMA ? D / 16 : 1][4];
#pragma unroll
  for (int mt = 0; mt < (MMA ? D / 16 : 1); ++mt) cacc[mt][0] = cacc[mt][1] = cacc[mt][2] = cacc[mt][3] = 0.0f;
  float lpart = 0.0f;
  const int cq = lane & 3, rq = lane >> 2;
  // bf16 pages: the V slab is requested by one bulk copy into the warp's
  // buffer before the page's scores are computed, so its transfer overlaps
  // the K loads and the scores, and the weighted sum reads it from shared
  // memory (no V registers in flight)
  const uint32_t vs_base = (smem_u32(vstage_sm) + 1023u) & ~1023u;
  T* vbuf = reinterpret_cast<T*>(vstage_sm + (vs_base - smem_u32(vstage_sm))) + (size_t)warp * P * D;
  uint32_t vphase = 0u;
  bool stuck = false;
  if constexpr (sizeof(T) == 2) {
    if (lane == 0) {
      mbar_init(&vbar[warp], 1);
      mbar_fence_init();
    }
    __syncwarp();
  }
  for (int i = warp; i < hi - lo && !stuck; i += kWarps) {
    const int page = bitmap ? list[i] : lo + i;
    const int ph = phys_page(a.block_table, seq, page, a.maxp, a.nphys, lane == 0 ? a.status : nullptr);
    if (ph < 0) continue;
    const int nv = min(P, L - page * P);
    const size_t slab_off = ((size_t)ph * a.Hkv + kvh) * P * D;
    if constexpr (sizeof(T) == 2) {
      if (lane == 0) {
        const uint32_t bytes = (uint32_t)(P * D * sizeof(T));
        mbar_expect_tx(&vbar[warp], bytes);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tma_load_3d(reinterpret_cast<unsigned char*>(vbuf) + hf * P * 128, &vmap, 64 * hf, kvh * P, ph,
                      &vbar[warp]);
      }
    }
    if constexpr (sizeof(T) == 2) {
      float zf[2][4];
      // one 16-token tile at a time: half the K fragments live at once
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        if (16 * mt >= P) {
          zf[mt][0] = zf[mt][1] = zf[mt][2] = zf[mt][3] = -CUDART_INF_F;
          continue;
        }
        float zt[2][4];
        page_scores_bf16<D>((const __nv_bfloat16*)a.k_pool + slab_off + (size_t)16 * mt * D, 16,
                            nv - 16 * mt, bq, scale2, lane, zt);
#pragma unroll
        for (int e = 0; e < 4; ++e) zf[mt][e] = zt[0][e];
      }
      const int r = lane >> 2, c = lane & 3, h0 = 2 * c, h1 = h0 + 1;
      float pm0 = -CUDART_INF_F, pm1 = -CUDART_INF_F;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        if (16 * mt >= P) break;
        const int t0 = 16 * mt + r, t1 = t0 + 8;
        if (h0 < GP) {
          sbuf[warp][t0][h0] = zf[mt][0];
          sbuf[warp][t1][h0] = zf[mt][2];
        }
        if (h1 < GP) {
          sbuf[warp][t0][h1] = zf[mt][1];
          sbuf[warp][t1][h1] = zf[mt][3];
        }
        pm0 = fmaxf(pm0, fmaxf(zf[mt][0], zf[mt][2]));
        pm1 = fmaxf(pm1, fmaxf(zf[mt][1], zf[mt][3]));
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, o));
        pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, o));
      }
      if (lane < 4) {
        pmx[warp][h0] = pm0;
        pmx[warp][h1] = pm1;
      }
    } else {
      float zt[8];
      page_scores_f32<D>((const float*)a.k_pool + slab_off, nv, qs, G, scale2, lane, zt);
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        if (lane < P) sbuf[warp][lane][h] = zt[h];
        const float mm = warp_max(zt[h]);
        if (lane == 0) pmx[warp][h] = mm;
      }
    }
    __syncwarp();
    if constexpr (MMA) {
      // rescale: the lane's p sum is of head rq, its accumulators of heads 2cq, 2cq + 1
      float s_r = 1.0f, s_0 = 1.0f, s_1 = 1.0f;
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float mn = fmaxf(m[h], h < G ? pmx[warp][h] : -CUDART_INF_F);
        if (mn > m[h]) {
          const float sc = exp2f(m[h] - mn);  // 0 when m was −inf
          if (h == rq) s_r = sc;
          if (h == 2 * cq) s_0 = sc;
          if (h == 2 * cq + 1) s_1 = sc;
          m[h] = mn;
        }
      }
      lpart *= s_r;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        cacc[mt][0] *= s_0;
        cacc[mt][2] *= s_0;
        cacc[mt][1] *= s_1;
        cacc[mt][3] *= s_1;
      }
      float m_r = -CUDART_INF_F;
#pragma unroll
      for (int h = 0; h < GP; ++h)
        if (h == rq) m_r = m[h];
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&vbar[warp], vphase))) {
        stuck = true;
        break;
      }
      vphase ^= 1u;
      unsigned char* vb = reinterpret_cast<unsigned char*>(vbuf);
      if (nv < P) {  // token slots past the sequence's end: zero, so p = 0 meets no NaN
        for (int e = lane; e < (D / 64) * (P - nv) * 8; e += 32) {
          const int hf = e / ((P - nv) * 8), rem = e - hf * (P - nv) * 8;
          *reinterpret_cast<uint4*>(vb + hf * P * 128 + (nv + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
      }
      // p = 2^(s − m) of tokens 16ks + 2cq (+1) and +8 for head rq (0 for
      // padding heads, heads without a finite max and invalid tokens)
      const bool hv = rq < G && m_r > -CUDART_INF_F;
      const uint32_t vb_s = smem_u32(vb);
#pragma unroll
      for (int ks = 0; ks < P / 16; ++ks) {
        const int t0 = 16 * ks + 2 * cq;
        const int hs = rq < GP ? rq : 0;
        const float p0 = hv ? exp2f(sbuf[warp][t0][hs] - m_r) : 0.0f;
        const float p1 = hv ? exp2f(sbuf[warp][t0 + 1][hs] - m_r) : 0.0f;
        const float p2 = hv ? exp2f(sbuf[warp][t0 + 8][hs] - m_r) : 0.0f;
        const float p3 = hv ? exp2f(sbuf[warp][t0 + 9][hs] - m_r) : 0.0f;
        lpart += (p0 + p1) + (p2 + p3);
        uint32_t bh0, bl0, bh1, bl1;
        bf16_split2(p0, p1, bh0, bl0);
        bf16_split2(p2, p3, bh1, bl1);
        const int tr = 16 * ks + (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int ch = 2 * mt + ((lane >> 3) & 1);
          uint32_t a0, a1, a2, a3;
          ldsm_x4_trans(a0, a1, a2, a3, vb_s + (ch >> 3) * P * 128 + swz128(tr, ch & 7));
          mma_bf16(cacc[mt], a0, a1, a2, a3, bh0, bh1);
          mma_bf16(cacc[mt], a0, a1, a2, a3, bl0, bl1);
        }
      }
      __syncwarp();  // the buffer is refilled for the next page
      continue;
    }
    if constexpr (!MMA) {  // fp32 pages: p·v in fp32 on the CUDA cores
  #pragma unroll
      for (int h = 0; h < GP; ++h) {
        const float mn = fmaxf(m[h], h < G ? pmx[warp][h] : -CUDART_INF_F);
        if (mn > m[h]) {
          const float sc = exp2f(m[h] - mn);  // 0 when m was −inf
          l[h] *= sc;
  #pragma unroll
          for (int j = 0; j < VEC; ++j) acc[h][j] *= sc;
          m[h] = mn;
        }
      }
      const T* vs = (const T*)a.v_pool + slab_off + dc * VEC;
      for (int c0 = 0; c0 < MAXT; c0 += CH) {
        uint4 raw[CH];
  #pragma unroll
        for (int u = 0; u < CH; ++u) {
          const int t = tg + TG * (c0 + u);
          raw[u] = t < nv ? ld_stream(vs + (size_t)t * D) : make_uint4(0u, 0u, 0u, 0u);
        }
  #pragma unroll
        for (int u = 0; u < CH; ++u) {
          const int t = tg + TG * (c0 + u);
          if (t < nv) {
            float v[VEC];
            if constexpr (sizeof(T) == 2) {
              v[0] = bf_lo(raw[u].x); v[1] = bf_hi(raw[u].x); v[2] = bf_lo(raw[u].y); v[3] = bf_hi(raw[u].y);
              v[4] = bf_lo(raw[u].z); v[5] = bf_hi(raw[u].z); v[6] = bf_lo(raw[u].w); v[7] = bf_hi(raw[u].w);
            } else {
              v[0] = __uint_as_float(raw[u].x); v[1] = __uint_as_float(raw[u].y);
              v[2] = __uint_as_float(raw[u].z); v[3] = __uint_as_float(raw[u].w);
            }
  #pragma unroll
            for (int h = 0; h < GP; ++h) {
              if (h < G && m[h] > -CUDART_INF_F) {
                const float p = exp2f(sbuf[warp][t][h] - m[h]);
                l[h] += p;
  #pragma unroll
                for (int j = 0; j < VEC; ++j) acc[h][j] = fmaf(p, v[j], acc[h][j]);
              }
            }
          }
        }
      }
      __syncwarp();
    }
  }
  if (stuck) {  // a copy did not arrive within the bound: flag it, let it land, stop
    if (lane == 0) {
      raise_flag(a.status, ENTMAXKV_DEV_TIMEOUT);
      mbar_wait_bounded(&vbar[warp], vphase);
    }
    __syncwarp();
  }
  if constexpr (MMA) {
    // head rq's p sum: over the four lanes of its tokens
    lpart += __shfl_xor_sync(0xffffffffu, lpart, 1);
    lpart += __shfl_xor_sync(0xffffffffu, lpart, 2);
    __syncthreads();  // every warp is done with qs and sbuf
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      if (2 * cq < GP) {
        red[warp][2 * cq][16 * mt + rq] = cacc[mt][0];
        red[warp][2 * cq][16 * mt + rq + 8] = cacc[mt][2];
      }
      if (2 * cq + 1 < GP) {
        red[warp][2 * cq + 1][16 * mt + rq] = cacc[mt][1];
        red[warp][2 * cq + 1][16 * mt + rq + 8] = cacc[mt][3];
      }
    }
    if (cq == 0 && rq < GP) wl_sh[warp][rq] = lpart;
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < GP; ++h) wm_sh[warp][h] = m[h];
    }
  } else {
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        l[h] += __shfl_xor_sync(0xffffffffu, l[h], o);
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[h][j] += __shfl_xor_sync(0xffffffffu, acc[h][j], o);
      }
    __syncthreads();  // every warp is done with qs and sbuf
    if (tg == 0) {
#pragma unroll
      for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int j = 0; j < VEC; ++j) red[warp][h][dc * VEC + j] = acc[h][j];
    }
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        wm_sh[warp][h] = m[h];
        wl_sh[warp][h] = l[h];
      }
    }
  }
  if (bitmap) {  // this block's share of all pages: the dropped ones' Σ n_p·e^{U_p}, online
    float um[GP], us[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      um[h] = -CUDART_INF_F;
      us[h] = 0.0f;
    }
    const uint32_t* bm = a.bitmap + skv * a.words;
    const int plo = (int)(((long long)n_pages * split) / a.splits);
    const int phi = (int)(((long long)n_pages * (split + 1)) / a.splits);
    // four pages a thread per round, their bitmap words and bounds loaded together
    for (int p0 = plo + tid; p0 < phi; p0 += 4 * kThreads) {
      uint32_t w[4];
      float uu[4][GP];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int p = p0 + j * kThreads;
        w[j] = p < phi ? bm[p >> 5] : 0xffffffffu;
#pragma unroll
        for (int h = 0; h < GP; ++h) uu[j][h] = (p < phi && h < G) ? a.bbox_u[(hq0 + h) * a.maxp + p] : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int p = p0 + j * kThreads;
        if (p >= phi || ((w[j] >> (p & 31)) & 1u)) continue;  // kept pages drop nothing
        const float np = (float)min(P, L - p * P);
#pragma unroll
        for (int h = 0; h < GP; ++h) {
          if (h < G) {
            const float u = uu[j][h];
            if (u > um[h]) {
              us[h] = us[h] * expf(um[h] - u) + np;
              um[h] = u;
            } else {
              us[h] += np * expf(u - um[h]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int h = 0; h < GP; ++h) {  // merge the warp's (max, sum) pairs
      float M = warp_max(um[h]);
      const float sw = warp_sum(um[h] > -CUDART_INF_F ? us[h] * expf(um[h] - M) : 0.0f);
      if (lane == 0) {
        um_sh[warp][h] = M;
        us_sh[warp][h] = sw;
      }
    }
  }
  __syncthreads();
  float* part = a.partial + (skv * a.splits + split) * (size_t)a.pstride;
  for (int e = tid; e < G * (D + 1); e += kThreads) {
    const int h = e / (D + 1), d = e % (D + 1);
    float M = -CUDART_INF_F;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm_sh[w][h]);
    float sum = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
      const float wt = wm_sh[w][h] > -CUDART_INF_F ? exp2f(wm_sh[w][h] - M) : 0.0f;
      sum += wt * (d < D ? red[w][h][d] : wl_sh[w][h]);
    }
    if (d < D) {
      part[h * D + d] = sum;
    } else {
      part[G * D + h] = M;
      part[G * D + G + h] = sum;
    }
  }
  if (bitmap && tid < G) {
    float M = -CUDART_INF_F, sum = 0.0f;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, um_sh[w][tid]);
    for (int w = 0; w < kWarps; ++w)
      if (um_sh[w][tid] > -CUDART_INF_F) sum += us_sh[w][tid] * expf(um_sh[w][tid] - M);
    part[G * D + 2 * G + tid] = M;
    part[G * D + 3 * G + tid] = sum;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last_sh = atomicAdd(&a.cnt_b[skv], 1) == a.splits - 1;
  __syncthreads();
  if (!last_sh) return;
  __threadfence();
  // merge the split partials: per-head max and weighted sums, then columns
  const float* base = a.partial + skv * a.splits * (size_t)a.pstride;
  if (warp < G) {
    float M = -CUDART_INF_F;
    for (int sp = lane; sp < a.splits; sp += 32)
      M = fmaxf(M, __ldcg(base + (size_t)sp * a.pstride + G * D + warp));
    M = warp_max(M);
    float Ls = 0.0f;
    for (int sp = lane; sp < a.splits; sp += 32) {
      const float Ms = __ldcg(base + (size_t)sp * a.pstride + G * D + warp);
      if (Ms > -CUDART_INF_F) Ls += exp2f(Ms - M) * __ldcg(base + (size_t)sp * a.pstride + G * D + G + warp);
    }
    Ls = warp_sum(Ls);
    if (lane == 0) {
      Mg_sh[warp] = M;
      Lg_sh[warp] = Ls;
    }
  }
  __syncthreads();
  const int cols = G * D / 4;
  const int groups = kThreads / cols > 0 ? kThreads / cols : 1;
  const int col = tid % cols, grp = tid / cols;
  const int h = (col * 4) / D;
  if (grp < groups) {
    float4 accv = make_float4(0.f, 0.f, 0.f, 0.f);
    const float Mg = Mg_sh[h];
#pragma unroll 4
    for (int sp = grp; sp < a.splits; sp += groups) {
      const float Ms = __ldcg(base + (size_t)sp * a.pstride + G * D + h);
      if (!(Ms > -CUDART_INF_F)) continue;
      const float wt = exp2f(Ms - Mg);
      const float4 v = __ldcg(reinterpret_cast<const float4*>(base + (size_t)sp * a.pstride) + col);
      accv.x += wt * v.x;
      accv.y += wt * v.y;
      accv.z += wt * v.z;
      accv.w += wt * v.w;
    }
    red4[grp * cols + col] = accv;
  }
  __syncthreads();
  if (tid < cols) {
    float4 sum = red4[tid];
    for (int g2 = 1; g2 < groups; ++g2) {
      const float4 v = red4[g2 * cols + tid];
      sum.x += v.x;
      sum.y += v.y;
      sum.z += v.z;
      sum.w += v.w;
    }
    const float Lg = Lg_sh[h];
    const float inv = Lg > 0.0f ? 1.0f / Lg : 0.0f;
    if (a.out)
      reinterpret_cast<float4*>(a.out + hq0 * D)[tid] =
          make_float4(sum.x * inv, sum.y * inv, sum.z * inv, sum.w * inv);
  }
  if (tid < G) {
    const float Lg = Lg_sh[tid], Mg = Mg_sh[tid];
    const float lse = Lg > 0.0f ? (Mg + log2f(Lg)) * 0.6931471805599453f : CUDART_NAN_F;
    a.tau_ws[hq0 + tid] = lse;
    if (a.tau_out) a.tau_out[hq0 + tid] = lse;
    if (a.delta_out) {
      float dl = 0.0f;
      if (bitmap && L > 0) {  // certified D/(1 + D); all dropped when nothing was kept
        double Dd = 0.0;
        for (int sp = 0; sp < a.splits; ++sp) {
          const float um = __ldcg(base + (size_t)sp * a.pstride + G * D + 2 * G + tid);
          if (um > -CUDART_INF_F)
            Dd += (double)__ldcg(base + (size_t)sp * a.pstride + G * D + 3 * G + tid) * exp((double)um - (double)lse);
        }
        dl = Lg > 0.0f ? (float)(Dd / (1.0 + Dd)) : 1.0f;
      }
      a.delta_out[hq0 + tid] = dl;
    }
  }
}

template <typename T, int D, int GP>
static cudaError_t softmax_l(const DecodeArgs& a, const CUtensorMap& vmap, dim3 grid, cudaStream_t st) {
  // bf16: a V slab per warp in dynamic shared memory, plus the slack that
  // aligns the boxes to 1024 bytes
  const int smem = sizeof(T) == 2 ? kWarps * a.P * D * (int)sizeof(T) + 1024 : 0;
  if (smem) {
    const cudaError_t e = ensure_smem((const void*)softmax_kernel<T, D, GP>, smem);
    if (e != cudaSuccess) return e;
  }
  return launch_k(false, softmax_kernel<T, D, GP>, dim3(grid), dim3(kThreads), (size_t)smem, st, a, vmap);
}

template <typename T, int D>
static cudaError_t softmax_g(const DecodeArgs& a, const CUtensorMap& vmap, dim3 grid, cudaStream_t st) {
  if (a.G <= 1) return softmax_l<T, D, 1>(a, vmap, grid, st);
  if (a.G <= 2) return softmax_l<T, D, 2>(a, vmap, grid, st);
  if (a.G <= 4) return softmax_l<T, D, 4>(a, vmap, grid, st);
  return softmax_l<T, D, 8>(a, vmap, grid, st);
}

cudaError_t launch_softmax(const DecodeArgs& a, int kv_dtype, cudaStream_t st) {
  dim3 grid(a.splits, a.Hkv, a.S);
  CUtensorMap vmap;
  memset(&vmap, 0, sizeof(vmap));
  cudaError_t e;
  if (kv_dtype == ENTMAXKV_BF16) {
    e = make_v_map(&vmap, a.v_pool, a.nphys, a.Hkv, a.P, a.D);
    if (e != cudaSuccess) return e;
    e = a.D == 128 ? softmax_g<__nv_bfloat16, 128>(a, vmap, grid, st) : softmax_g<__nv_bfloat16, 64>(a, vmap, grid, st);
  } else {
    e = a.D == 128 ? softmax_g<float, 128>(a, vmap, grid, st) : softmax_g<float, 64>(a, vmap, grid, st);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace ekv
