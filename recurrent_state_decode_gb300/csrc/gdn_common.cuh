// Pieces shared by the Gated DeltaNet verify kernels.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace rssm {

// Epilogue of a Gated DeltaNet verify for sequence b, run by a whole block once
// no block of the sequence reads the ring rows it overwrites: on a cursor with
// 0 <= start < L, 0 <= count <= L and pending == 0, append the K new records'
// k, q (rows), g and beta at slots (start + count + j) mod L and set pending =
// K, flags = folded; otherwise report as the cursor checks do and leave the
// cursor with its flags word set to `flags`. The records of batch row b go to
// the ring rows (and cursor) of its state slot sb.
__device__ __forceinline__ void gdn_verify_epilogue(const GdnArgs& a, int b, int sb, int4 c, int flags) {
  const int L = a.L, K = a.K, H = a.H, DK = a.DK, tid = threadIdx.x, nt = blockDim.x;
  c.w = flags;
  int err = 0;
  if (!(c.x >= 0 && c.x < L && c.y >= 0 && c.y <= L))
    err = RSSM_DEV_BAD_CURSOR;
  else if (c.z != 0)
    err = RSSM_DEV_PENDING;
  if (err) {
    if (tid == 0) {
      report(a.status, err);
      *reinterpret_cast<int4*>(a.cursors + 4 * (size_t)sb) = c;
    }
    return;
  }
  const int nv = DK >> 3, pieces = K * H * nv;
  constexpr int U = 4;  // pieces in flight per thread: all loads before the stores
  for (int q0 = tid; q0 < pieces; q0 += U * nt) {
    uint4 kv[U], qv[U];
    size_t dst[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int q = q0 + u * nt;
      if (q < pieces) {
        const int j = q / (H * nv), r = q - j * H * nv, h = r / nv, v = r - h * nv;
        dst[u] = (((size_t)sb * H + h) * L + wrap(wrap(c.x + c.y + j, L), L)) * DK + v * 8;
        const size_t src = (((size_t)b * K + j) * H + h) * DK + v * 8;
        kv[u] = *reinterpret_cast<const uint4*>(a.k + src);
        qv[u] = *reinterpret_cast<const uint4*>(a.q + src);
      }
    }
#pragma unroll
    for (int u = 0; u < U; u++) {
      if (q0 + u * nt < pieces) {
        *reinterpret_cast<uint4*>(a.rk + dst[u]) = kv[u];
        *reinterpret_cast<uint4*>(a.rq + dst[u]) = qv[u];
      }
    }
  }
  for (int q = tid; q < K * H; q += nt) {
    const int j = q / H, h = q - j * H;
    const size_t s = ((size_t)sb * H + h) * pad4(L) + wrap(wrap(c.x + c.y + j, L), L);
    a.rg[s] = a.g[((size_t)b * K + j) * H + h];
    a.rbeta[s] = a.beta[((size_t)b * K + j) * H + h];
  }
  if (tid == 0) {
    c.z = K;
    c.w = (c.y + K > L) ? 1 : 0;
    *reinterpret_cast<int4*>(a.cursors + 4 * (size_t)sb) = c;
  }
}

}  // namespace rssm
