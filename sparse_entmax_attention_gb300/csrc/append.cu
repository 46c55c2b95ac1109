// append.cu -- write new tokens into their pages and maintain the per-page
// key metadata the scorers read.
//
// EntmaxKV (gist.science technical summary, §2A "Query-Aware Page Scoring"):
// each page keeps the coordinate-wise minimum and maximum key and the first
// and second moments (mean and variance) of its keys. Here kmin/kmax are
// exact element-wise extrema in the KV dtype; mean and m2 (the sum of squared
// deviations, var = m2/n_p) are float32. A page that already holds tokens is
// merged with the new ones by the pairwise update of Chan, Golub & LeVeque:
//   n = na + nb,  δ = mean_b − mean_a,  mean = mean_a + δ·nb/n,
//   m2 = m2_a + m2_b + δ²·na·nb/n.
#include "common.cuh"

namespace ekv {

template <typename T, int N>
struct alignas(N * sizeof(T)) Vec {
  T v[N];
};

// Touched page i of (slot b, KV head kvh) by one warp: lane j covers
// elements [j·D/32, (j+1)·D/32) of every row. L is the sequence's length
// before this append.
template <typename T, int D>
__device__ __forceinline__ void append_page(const AppendArgs& a, int b, int seq, int L, int kvh, int i,
                                            int lane) {
  constexpr int EPL = D / 32;
  using V = Vec<T, EPL>;
  const int P = a.P, T_new = a.n_tokens;
  const int first = L / P, last = (L + T_new - 1) / P;
  const int lp = first + i;
  if (lp > last) return;
  if (lp >= a.maxp) {
    if (lane == 0) raise_flag(a.status, ENTMAXKV_DEV_CAPACITY);
    return;
  }
  const int ph = phys_page(a.block_table, seq, lp, a.maxp, a.nphys, lane == 0 ? a.status : nullptr);
  if (ph < 0) return;
  const int tlo = max(L, lp * P), thi = min(L + T_new, (lp + 1) * P);
  const int n_old = tlo - lp * P, n_new = thi - tlo;

  const size_t src_row0 = (((size_t)b * a.Hkv + kvh) * T_new + (tlo - L)) * D + lane * EPL;
  const size_t dst_row0 = (((size_t)ph * a.Hkv + kvh) * P + n_old) * D + lane * EPL;
  const T* ks = (const T*)a.k + src_row0;
  const T* vs = (const T*)a.v + src_row0;
  T* kd = (T*)a.k_pool + dst_row0;
  T* vd = (T*)a.v_pool + dst_row0;

  float mn[EPL], mx[EPL], sum[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    mn[e] = CUDART_INF_F;
    mx[e] = -CUDART_INF_F;
    sum[e] = 0.0f;
  }
  // U rows at a time, their K and V loads in flight together before the
  // first store (about 256 bytes a lane: 16 rows of bf16, 8 of fp32 at d = 128)
  constexpr int U = sizeof(V) >= 16 ? 8 : 16;
  int t = 0;
  for (; t + U <= n_new; t += U) {
    V kv[U], vv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      kv[u] = *reinterpret_cast<const V*>(ks + (size_t)(t + u) * D);
      vv[u] = *reinterpret_cast<const V*>(vs + (size_t)(t + u) * D);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      *reinterpret_cast<V*>(kd + (size_t)(t + u) * D) = kv[u];
      *reinterpret_cast<V*>(vd + (size_t)(t + u) * D) = vv[u];
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        float x = to_f(kv[u].v[e]);
        mn[e] = fminf(mn[e], x);
        mx[e] = fmaxf(mx[e], x);
        sum[e] += x;
      }
    }
  }
  for (; t < n_new; ++t) {
    V kv = *reinterpret_cast<const V*>(ks + (size_t)t * D);
    V vv = *reinterpret_cast<const V*>(vs + (size_t)t * D);
    *reinterpret_cast<V*>(kd + (size_t)t * D) = kv;
    *reinterpret_cast<V*>(vd + (size_t)t * D) = vv;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      float x = to_f(kv.v[e]);
      mn[e] = fminf(mn[e], x);
      mx[e] = fmaxf(mx[e], x);
      sum[e] += x;
    }
  }
  float mean[EPL], m2[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    mean[e] = sum[e] / (float)n_new;
    m2[e] = 0.0f;
  }
  for (int t = 0; t < n_new; ++t) {  // second pass over the (cached) new rows
    V kv = *reinterpret_cast<const V*>(ks + (size_t)t * D);
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      float dx = to_f(kv.v[e]) - mean[e];
      m2[e] = fmaf(dx, dx, m2[e]);
    }
  }
  const size_t meta = ((size_t)ph * a.Hkv + kvh) * D + lane * EPL;
  V* kminp = reinterpret_cast<V*>((T*)a.kmin + meta);
  V* kmaxp = reinterpret_cast<V*>((T*)a.kmax + meta);
  float* meanp = a.mean + meta;
  float* m2p = a.m2 + meta;
  if (n_old > 0) {
    V omin = *kminp, omax = *kmaxp;
    const float na = (float)n_old, nb = (float)n_new, n = na + nb;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      mn[e] = fminf(mn[e], to_f(omin.v[e]));
      mx[e] = fmaxf(mx[e], to_f(omax.v[e]));
      float om = meanp[e], om2 = m2p[e];
      float dlt = mean[e] - om;
      mean[e] = om + dlt * (nb / n);
      m2[e] = om2 + m2[e] + dlt * dlt * (na * nb / n);
    }
  }
  V vmin, vmax;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    vmin.v[e] = (T)mn[e];  // exact: each extremum is one of the stored values
    vmax.v[e] = (T)mx[e];
    meanp[e] = mean[e];
    m2p[e] = m2[e];
  }
  *kminp = vmin;
  *kmaxp = vmax;
  if (a.mean_lo) {  // the copies the scorer streams: each rounded once from the fp32 values
    using VB = Vec<__nv_bfloat16, EPL>;
    VB ml, vl;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      ml.v[e] = __float2bfloat16_rn(mean[e]);
      vl.v[e] = __float2bfloat16_rn(m2[e]);
    }
    *reinterpret_cast<VB*>(a.mean_lo + meta) = ml;
    *reinterpret_cast<VB*>(a.m2_lo + meta) = vl;
  }
}

// Bulk appends: a warp per (slot, KV head, touched page); the lengths are
// advanced by a second kernel once every page is written.
template <typename T, int D>
__global__ void __launch_bounds__(128) append_kernel(AppendArgs a) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int seq = seq_row(a.seq_ids, b, a.max_seqs, lane == 0 ? a.status : nullptr);
  if (seq < 0) return;
  append_page<T, D>(a, b, seq, max(a.seq_lens[seq], 0), kvh, blockIdx.x * 4 + warp, lane);
}

// Small appends (a decode step's token): one block per slot writes every
// touched page of every KV head, then advances the slot's length itself.
template <typename T, int D>
__global__ void __launch_bounds__(512) append_step_kernel(AppendArgs a, int pages) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int b = blockIdx.x;
  const int seq = seq_row(a.seq_ids, b, a.max_seqs, threadIdx.x == 0 ? a.status : nullptr);
  if (seq < 0) return;  // block-uniform
  const int L = max(a.seq_lens[seq], 0);
  for (int item = warp; item < a.Hkv * pages; item += nw)
    append_page<T, D>(a, b, seq, L, item / pages, item % pages, lane);
  __syncthreads();  // every read of the old length is done
  if (threadIdx.x == 0) a.seq_lens[seq] += a.n_tokens;
}

__global__ void advance_lens_kernel(AppendArgs a) {
  pdl_enter();
  int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= a.n_seqs) return;
  int seq = a.seq_ids ? a.seq_ids[b] : b;
  if (seq < 0 || seq >= a.max_seqs) return;  // flagged by append_kernel
  a.seq_lens[seq] += a.n_tokens;
}

template <typename T, int D>
static cudaError_t launch_append_t(const AppendArgs& a, cudaStream_t st) {
  const int pages = (a.n_tokens + a.P - 1) / a.P + 1;  // pages one append can touch
  if ((long long)a.Hkv * pages <= 64) {
    const int warps = a.Hkv * pages < 16 ? a.Hkv * pages : 16;
    return launch_k(false, append_step_kernel<T, D>, dim3(a.n_seqs), dim3(32 * warps), 0, st, a, pages);
  }
  dim3 grid((pages + 3) / 4, a.Hkv, a.n_seqs);
  cudaError_t e = launch_k(false, append_kernel<T, D>, grid, dim3(128), 0, st, a);
  if (e == cudaSuccess) e = launch_k(false, advance_lens_kernel, dim3((a.n_seqs + 127) / 128), dim3(128), 0, st, a);
  return e;
}

cudaError_t launch_append(const AppendArgs& a, int kv_dtype, cudaStream_t st) {
  if (kv_dtype == ENTMAXKV_BF16)
    return a.D == 128 ? launch_append_t<__nv_bfloat16, 128>(a, st)
                      : launch_append_t<__nv_bfloat16, 64>(a, st);
  return a.D == 128 ? launch_append_t<float, 128>(a, st) : launch_append_t<float, 64>(a, st);
}

}  // namespace ekv
