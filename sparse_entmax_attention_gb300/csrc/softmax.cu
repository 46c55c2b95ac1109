// softmax.cu -- full-cache softmax decode, the FlashDecoding-style baseline
// the EntmaxKV summary compares against (gist.science technical summary, §4
// "Efficiency": speedups over full-cache softmax FlashDecoding).
//
// Split-K over pages: each warp streams its pages once (K then V of the same
// page), keeps an online softmax (running max m, running sum l, accumulator
// Σ 2^{s−m} v) per query head in the base-2 domain, the block merges its warps
// and writes (m, l, acc) as a partial, and the last block to finish merges the
// partials in split order. The "τ" output carries log Σ_i exp(s_i).
#include "common.cuh"

#include "page_scores.cuh"

namespace ekv {

template <typename T, int D, int GP>
__global__ void __launch_bounds__(kThreads) softmax_kernel(DecodeArgs a) {
  constexpr int VEC = 16 / sizeof(T), LPR = D / VEC, TG = 32 / LPR;
  __shared__ float qs[8][D];
  __shared__ float sbuf[kWarps][32][GP];
  __shared__ float pmx[kWarps][8];
  __shared__ float red[kWarps][GP][D];
  __shared__ float wm_sh[kWarps][GP], wl_sh[kWarps][GP];
  __shared__ int last_sh;
  const int split = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G, P = a.P;
  const int dc = lane % LPR, tg = lane / LPR;
  const int seq = seq_row(a.seq_ids, s, a.max_seqs, tid == 0 ? a.status : nullptr);
  const int L = seq_len_clamped(a.seq_lens, seq, a.maxp, P, tid == 0 ? a.status : nullptr);
  const int n_pages = (L + P - 1) / P;
  const int lo = (int)(((long long)n_pages * split) / a.splits);
  const int hi = (int)(((long long)n_pages * (split + 1)) / a.splits);
  const size_t skv = (size_t)s * a.Hkv + kvh;
  const size_t hq0 = (size_t)s * a.Hq + (size_t)kvh * G;
  if (split == 0 && tid == 0 && a.n_sel_out) a.n_sel_out[skv] = n_pages;
  if (a.page_ids)
    for (int p = lo + tid; p < hi; p += kThreads) a.page_ids[skv * a.page_ids_stride + p] = p;
  const float scale2 = a.inv_sqrt_d * 1.4426950408889634f;  // scores in log2 units
  uint32_t bq[D / 16][2];
  if constexpr (sizeof(T) == 2) {
    load_q_bfrag<D>((const __nv_bfloat16*)a.q + hq0 * D, G, lane, bq);
  } else {
    for (int i = tid; i < G * D; i += kThreads) qs[i / D][i % D] = ((const float*)a.q)[hq0 * D + i];
    __syncthreads();
  }
  float m[GP], l[GP], acc[GP][VEC];
#pragma unroll
  for (int h = 0; h < GP; ++h) {
    m[h] = -CUDART_INF_F;
    l[h] = 0.0f;
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[h][j] = 0.0f;
  }
  for (int page = lo + warp; page < hi; page += kWarps) {
    const int ph = phys_page(a.block_table, seq, page, a.maxp, a.nphys, lane == 0 ? a.status : nullptr);
    if (ph < 0) continue;
    const int nv = min(P, L - page * P);
    const size_t slab_off = ((size_t)ph * a.Hkv + kvh) * P * D;
    if constexpr (sizeof(T) == 2) {
      float zf[2][4];
      page_scores_bf16<D>((const __nv_bfloat16*)a.k_pool + slab_off, P, nv, bq, scale2, lane, zf);
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
    for (int t = tg; t < nv; t += TG) {
      const uint4 raw = ld_stream(vs + (size_t)t * D);
      float v[VEC];
      if constexpr (sizeof(T) == 2) {
        v[0] = bf_lo(raw.x); v[1] = bf_hi(raw.x); v[2] = bf_lo(raw.y); v[3] = bf_hi(raw.y);
        v[4] = bf_lo(raw.z); v[5] = bf_hi(raw.z); v[6] = bf_lo(raw.w); v[7] = bf_hi(raw.w);
      } else {
        v[0] = __uint_as_float(raw.x); v[1] = __uint_as_float(raw.y);
        v[2] = __uint_as_float(raw.z); v[3] = __uint_as_float(raw.w);
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
    __syncwarp();
  }
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      l[h] += __shfl_xor_sync(0xffffffffu, l[h], o);
#pragma unroll
      for (int j = 0; j < VEC; ++j) acc[h][j] += __shfl_xor_sync(0xffffffffu, acc[h][j], o);
    }
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
  __syncthreads();
  float* part = a.partial + (skv * a.splits + split) * (size_t)G * (D + 2);
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
      part[h * (D + 2) + d] = sum;
    } else {
      part[h * (D + 2) + D] = M;
      part[h * (D + 2) + D + 1] = sum;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) last_sh = atomicAdd(&a.cnt_b[skv], 1) == a.splits - 1;
  __syncthreads();
  if (!last_sh) return;
  __threadfence();
  for (int e = tid; e < G * (D + 1); e += kThreads) {
    const int h = e / (D + 1), d = e % (D + 1);
    float M = -CUDART_INF_F;
    for (int sp = 0; sp < a.splits; ++sp)
      M = fmaxf(M, __ldcg(a.partial + (skv * a.splits + sp) * (size_t)G * (D + 2) + h * (D + 2) + D));
    float num = 0.0f, den = 0.0f;
    for (int sp = 0; sp < a.splits; ++sp) {
      const float* pp = a.partial + (skv * a.splits + sp) * (size_t)G * (D + 2) + h * (D + 2);
      const float Ms = __ldcg(pp + D);
      if (!(Ms > -CUDART_INF_F)) continue;
      const float wt = exp2f(Ms - M);
      den += wt * __ldcg(pp + D + 1);
      if (d < D) num += wt * __ldcg(pp + d);
    }
    if (d < D) {
      a.out[(hq0 + h) * D + d] = den > 0.0f ? num / den : 0.0f;
    } else {
      const float lse = den > 0.0f ? (M + log2f(den)) * 0.6931471805599453f : CUDART_NAN_F;
      if (a.tau_out) a.tau_out[hq0 + h] = lse;
      if (a.delta_out) a.delta_out[hq0 + h] = 0.0f;
    }
  }
}

template <typename T, int D>
static void softmax_g(const DecodeArgs& a, dim3 grid, cudaStream_t st) {
  if (a.G <= 1) softmax_kernel<T, D, 1><<<grid, kThreads, 0, st>>>(a);
  else if (a.G <= 2) softmax_kernel<T, D, 2><<<grid, kThreads, 0, st>>>(a);
  else if (a.G <= 4) softmax_kernel<T, D, 4><<<grid, kThreads, 0, st>>>(a);
  else softmax_kernel<T, D, 8><<<grid, kThreads, 0, st>>>(a);
}

cudaError_t launch_softmax(const DecodeArgs& a, int kv_dtype, cudaStream_t st) {
  dim3 grid(a.splits, a.Hkv, a.S);
  if (kv_dtype == ENTMAXKV_BF16) {
    if (a.D == 128) softmax_g<__nv_bfloat16, 128>(a, grid, st);
    else softmax_g<__nv_bfloat16, 64>(a, grid, st);
  } else {
    if (a.D == 128) softmax_g<float, 128>(a, grid, st);
    else softmax_g<float, 64>(a, grid, st);
  }
  return cudaGetLastError();
}

}  // namespace ekv
