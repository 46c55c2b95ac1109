// page_scores.cuh -- scores of one KV page for the query heads of a group,
// shared by the entmax decode and the softmax baseline. Internal.
#pragma once

#include "common.cuh"

namespace ekv {

// Page scores. bf16: thread (r = lane/4, c = lane%4) loads 16-byte chunks
// 8c..8c+7 (+32j) of token rows r and r+8 of each 16-token tile; the q
// fragments use the same permuted k order, so the MMA computes q·k exactly as
// the plain dot product (up to fp32 summation order).

template <int D>
__device__ __forceinline__ void load_q_bfrag(const __nv_bfloat16* q_group, int G, int lane,
                                             uint32_t (&bq)[D / 16][2]) {
  const int n = lane >> 2, c = lane & 3;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    if (n < G) {
      const uint2 x = *reinterpret_cast<const uint2*>(q_group + (size_t)n * D + 32 * (ks >> 1) +
                                                      8 * c + 4 * (ks & 1));
      bq[ks][0] = x.x;
      bq[ks][1] = x.y;
    } else {
      bq[ks][0] = bq[ks][1] = 0u;
    }
  }
}

// z for the tokens this thread holds: zf[mt][0..3] = (t0,h0) (t0,h1) (t1,h0) (t1,h1)
// with t0 = 16·mt + lane/4, t1 = t0 + 8, h0 = 2·(lane%4), h1 = h0 + 1.
template <int D>
__device__ __forceinline__ void page_scores_bf16(const __nv_bfloat16* slab, int P, int nv,
                                                 const uint32_t (&bq)[D / 16][2], float scale,
                                                 int lane, float (&zf)[2][4]) {
  constexpr int C16 = D / 32;
  const int r = lane >> 2, c = lane & 3;
  const int ntile = P >> 4;
  uint4 x[2][2][C16];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
    if (mt < ntile)
#pragma unroll
      for (int j = 0; j < C16; ++j) {
        x[mt][0][j] = ld_stream(slab + (size_t)(16 * mt + r) * D + 32 * j + 8 * c);
        x[mt][1][j] = ld_stream(slab + (size_t)(16 * mt + r + 8) * D + 32 * j + 8 * c);
      }
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    if (mt >= ntile) {
      zf[mt][0] = zf[mt][1] = zf[mt][2] = zf[mt][3] = -CUDART_INF_F;
      continue;
    }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const int j = ks >> 1;
      const bool u = ks & 1;
      mma_bf16(acc, u ? x[mt][0][j].z : x[mt][0][j].x, u ? x[mt][1][j].z : x[mt][1][j].x,
               u ? x[mt][0][j].w : x[mt][0][j].y, u ? x[mt][1][j].w : x[mt][1][j].y, bq[ks][0],
               bq[ks][1]);
    }
    const int t0 = 16 * mt + r, t1 = t0 + 8;
    zf[mt][0] = t0 < nv ? acc[0] * scale : -CUDART_INF_F;
    zf[mt][1] = t0 < nv ? acc[1] * scale : -CUDART_INF_F;
    zf[mt][2] = t1 < nv ? acc[2] * scale : -CUDART_INF_F;
    zf[mt][3] = t1 < nv ? acc[3] * scale : -CUDART_INF_F;
  }
}

// fp32 pages: lane t scores token t for every head of the group. The dot
// product is accumulated in double (each fp32 product is exact there), so the
// only rounding is the final one to fp32: fp32 KV is the accuracy path.
template <int D>
__device__ __forceinline__ void page_scores_f32(const float* slab, int nv, const float (*qs)[D],
                                                int G, float scale, int lane, float (&zt)[8]) {
  double acc[8] = {0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0};
  if (lane < nv) {
    const float* row = slab + (size_t)lane * D;
    for (int d = 0; d < D; d += 4) {
      const float4 k4 = *reinterpret_cast<const float4*>(row + d);
#pragma unroll
      for (int h = 0; h < 8; ++h)
        if (h < G) {
          acc[h] = fma((double)qs[h][d], (double)k4.x, acc[h]);
          acc[h] = fma((double)qs[h][d + 1], (double)k4.y, acc[h]);
          acc[h] = fma((double)qs[h][d + 2], (double)k4.z, acc[h]);
          acc[h] = fma((double)qs[h][d + 3], (double)k4.w, acc[h]);
        }
    }
  }
#pragma unroll
  for (int h = 0; h < 8; ++h) zt[h] = lane < nv ? (float)(acc[h] * (double)scale) : -CUDART_INF_F;
}

}  // namespace ekv
