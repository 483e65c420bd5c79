// The fold of a verify's committed window into a block's state rows as
// tensor-core products (dstate or dk 128, rows in blocks of 64, four warps:
// warp w the rows 8w..8w+7 and 32+8w..32+8w+7).
#pragma once
#include "fast_rows.cuh"

namespace rssm {
namespace fastrows {

// h' = P h0 + sum_{k<n} (w_k c_k[r]) R_k for a warp's 16 rows (rl0..rl0+7 and
// rl1..rl1+7), written once to dst (row stride FN), as m16n8k8 tf32 products of
// the transposed update h'^T = P h0^T + R^T (w c)^T: M = 16 state columns per
// tile, N = 8 rows per n-tile (n-tile 0 the rows from rl0, 1 those from rl1),
// K = 8 records per step. Tile m holds the columns 32 (m >> 1) + 4 i + 2 (m & 1)
// + (i >> 3), i < 16, so that a lane's accumulators in tiles 2j and 2j + 1 are
// the four consecutive columns 32 j + 4 qg .. + 3 of its rows: one 16-byte load
// of h0 (shared memory, row stride FN) and one 16-byte store per row and tile
// pair, the 8 lanes of a row on distinct banks. R_k = row(k) is a bf16 row
// (exact in tf32); w_k sits on lane k; w_k c_k[r], c_k[r] = coef(k, r), enters
// as two tf32 parts; records k >= n enter as 0. n <= 32 and uniform over the
// warp; every lane must call this.
template <class Row, class Coef>
__device__ __forceinline__ void fold_rows_mma(const float* h0, float* dst, Row row, Coef coef, int n, float P, float w,
                                              int rl0, int rl1, int lane) {
  const int qg = lane >> 2, qt = lane & 3;
#pragma unroll
  for (int pass = 0; pass < 2; pass++) {  // tile pairs j = 2 pass, 2 pass + 1
    float d[4][2][4];                     // [tile m - 4 pass][n-tile][fragment]
#pragma unroll
    for (int nt = 0; nt < 2; nt++) {
      const int r0 = (nt ? rl1 : rl0) + 2 * qt;
#pragma unroll
      for (int jj = 0; jj < 2; jj++) {
        const int col = 32 * (2 * pass + jj) + 4 * qg;
        const float4 u = ld4(h0 + r0 * FN + col), v = ld4(h0 + (r0 + 1) * FN + col);
        d[2 * jj][nt][0] = P * u.x;
        d[2 * jj][nt][2] = P * u.y;
        d[2 * jj + 1][nt][0] = P * u.z;
        d[2 * jj + 1][nt][2] = P * u.w;
        d[2 * jj][nt][1] = P * v.x;
        d[2 * jj][nt][3] = P * v.y;
        d[2 * jj + 1][nt][1] = P * v.z;
        d[2 * jj + 1][nt][3] = P * v.w;
      }
    }
    for (int k0 = 0; k0 < n; k0 += 8) {
      const int ka = k0 + qt, kb = ka + 4;
      uint2 ba[2] = {make_uint2(0, 0), make_uint2(0, 0)}, bb[2] = {ba[0], ba[0]};
#pragma unroll
      for (int jj = 0; jj < 2; jj++) {
        const int col = 32 * (2 * pass + jj) + 4 * qg;
        if (ka < n) ba[jj] = *reinterpret_cast<const uint2*>(row(ka) + col);
        if (kb < n) bb[jj] = *reinterpret_cast<const uint2*>(row(kb) + col);
      }
      const float wa = __shfl_sync(FULL, w, ka), wb = __shfl_sync(FULL, w, kb);
#pragma unroll
      for (int nt = 0; nt < 2; nt++) {
        const int r = (nt ? rl1 : rl0) + qg;
        const float ca = ka < n ? wa * coef(ka, r) : 0.f, cb = kb < n ? wb * coef(kb, r) : 0.f;
        uint32_t h0a, l0a, h0b, l0b;
        split_tf32(ca, h0a, l0a);
        split_tf32(cb, h0b, l0b);
#pragma unroll
        for (int m = 0; m < 4; m++) {
          const uint32_t pa = (m & 1) ? ba[m >> 1].y : ba[m >> 1].x;  // columns + 2 (m & 1) and + 1
          const uint32_t pb = (m & 1) ? bb[m >> 1].y : bb[m >> 1].x;
          const uint32_t a0 = pa << 16, a1 = pa & 0xffff0000u, a2 = pb << 16, a3 = pb & 0xffff0000u;
          mma_tf32_1688(d[m][nt], a0, a1, a2, a3, h0a, h0b);
          mma_tf32_1688(d[m][nt], a0, a1, a2, a3, l0a, l0b);
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < 2; nt++) {
      const int r0 = (nt ? rl1 : rl0) + 2 * qt;
#pragma unroll
      for (int jj = 0; jj < 2; jj++) {
        float* o = dst + (size_t)r0 * FN + 32 * (2 * pass + jj) + 4 * qg;
        __stcs(reinterpret_cast<float4*>(o),
               make_float4(d[2 * jj][nt][0], d[2 * jj][nt][2], d[2 * jj + 1][nt][0], d[2 * jj + 1][nt][2]));
        __stcs(reinterpret_cast<float4*>(o + FN),
               make_float4(d[2 * jj][nt][1], d[2 * jj][nt][3], d[2 * jj + 1][nt][1], d[2 * jj + 1][nt][3]));
      }
    }
  }
}

}  // namespace fastrows
}  // namespace rssm
