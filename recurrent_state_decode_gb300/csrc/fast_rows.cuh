// Pieces shared by the shape-specialised Mamba-2 kernels (dstate 128, rows in
// blocks of 64): a block of four warps holds a (sequence, head) tile's 64
// checkpoint rows, warp w the rows 8w..8w+7 and 32+8w..32+8w+7, lane l the
// float4 column chunk 4l..4l+3 of each.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace rssm {
namespace fastrows {

constexpr int FN = 128;     // dstate
constexpr int FPB = 64;     // rows per block
constexpr int FW = 4;       // warps
constexpr int FT = 32 * FW;
constexpr int HALF = 32;    // a warp's second row group starts here

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) { return *reinterpret_cast<const uint4*>(p); }

// Every lane must call this (a full-warp shuffle).
__device__ __forceinline__ float4 shfl_f4(float4 v, int src) {
  return make_float4(__shfl_sync(FULL, v.x, src), __shfl_sync(FULL, v.y, src), __shfl_sync(FULL, v.z, src),
                     __shfl_sync(FULL, v.w, src));
}

// y[r] before the gate for 8 rows: sum over lanes of (h . PC) + t[r], where
// t[r] is the lane's window term. The total of row rr ends in lane row_src(rr).
__device__ __forceinline__ float rows8(const float4 (&hv)[8], float4 pc, const float (&t)[8], int lane) {
  float v[8];
#pragma unroll
  for (int rr = 0; rr < 8; rr++)
    v[rr] = fmaf(hv[rr].x, pc.x, fmaf(hv[rr].y, pc.y, fmaf(hv[rr].z, pc.z, fmaf(hv[rr].w, pc.w, t[rr]))));
  return reduce_transpose<8>(v, lane);
}

// Two matvecs of 8 rows at once (the delta-rule kernels' S0 k and S0 q): 16
// partials, [rr] = h[rr] . ka + tk[rr] and [8 + rr] = h[rr] . qa + tq[rr];
// lane l ends with the total of partial l >> 1.
__device__ __forceinline__ float rows8x2(const float4 (&hv)[8], float4 ka, float4 qa, const float (&tk)[8],
                                         const float (&tq)[8], int lane) {
  float v[16];
#pragma unroll
  for (int rr = 0; rr < 8; rr++) {
    v[rr] = fmaf(hv[rr].x, ka.x, fmaf(hv[rr].y, ka.y, fmaf(hv[rr].z, ka.z, fmaf(hv[rr].w, ka.w, tk[rr]))));
    v[8 + rr] = fmaf(hv[rr].x, qa.x, fmaf(hv[rr].y, qa.y, fmaf(hv[rr].z, qa.z, fmaf(hv[rr].w, qa.w, tq[rr]))));
  }
  return reduce_transpose<16>(v, lane);
}

__device__ __forceinline__ int row_src(int rr) {
  return ((rr >> 2) & 1) * 16 + ((rr >> 1) & 1) * 8 + (rr & 1) * 4;
}

// silu(z) = z sigmoid(z)
__device__ __forceinline__ float silu_fast(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// Arrival of one block on its sequence's cursor: the high 16 bits of the
// cursor's flags word count the blocks of this launch that have arrived (the
// low 16 bits are the flags themselves). Taken by one thread once every thread
// of the block is done with what the sequence's last block will overwrite (for
// the AR step: the cursor itself); the ticket is only looked at later, so the
// atomic's round trip overlaps the block's work. Its cursor loads are already
// consumed, so no fence is needed before it: the last block's update is
// ordered after every other block's arrival by the atomic itself.
__device__ __forceinline__ int cursor_ticket(int32_t* cursors, int b) {
  return atomicAdd(cursors + 4 * (size_t)b + 3, 1 << 16);
}

__device__ __forceinline__ bool last_ticket(int ticket, int nblocks) { return (ticket >> 16) == nblocks - 1; }

// AR rule, applied by the sequence's last block (one thread): count + 1 == L ?
// 0 : count + 1 on a cursor with 0 <= start < L, 0 <= count < L and pending ==
// 0, else the same error report as the cursor kernel and no move; the arrival
// count is cleared.
__device__ __forceinline__ void finish_ar_cursor(int32_t* cursors, int b, int4 cur, int ticket, int nblocks, int L,
                                                 int32_t* status) {
  if (!last_ticket(ticket, nblocks)) return;
  int4 c = cur;
  c.w = ticket & 0xffff;
  if (!(c.x >= 0 && c.x < L && c.y >= 0 && c.y <= L && c.z >= 0))
    report(status, RSSM_DEV_BAD_CURSOR);
  else if (c.z != 0)
    report(status, RSSM_DEV_PENDING);
  else if (c.y == L)
    report(status, RSSM_DEV_WINDOW_FULL);
  else
    c.y = (c.y + 1 == L) ? 0 : c.y + 1;
  *reinterpret_cast<int4*>(cursors + 4 * (size_t)b) = c;
}

// gate: silu(z) of row (lane & 7), computed before the rows land
template <bool OUT_BF16>
__device__ __forceinline__ void gate_store(const M2Args& a, size_t obase, float gate, float tot, int lane) {
  const float t = __shfl_sync(FULL, tot, row_src(lane & 7));
  if (lane < 8) store_out<OUT_BF16>(a.y, obase + lane, t * gate);
}

// The read copy (if any) of 8 rows of the state: element offset `off` of row
// 0's float4 at column 4 lane; every lane must call this.
__device__ __forceinline__ void store_read_copy8(const M2Args& a, const float4 (&hv)[8], size_t off, int lane) {
  if (!a.ckpt_read) return;
  if (a.read_f8) {
    uint8_t* q = reinterpret_cast<uint8_t*>(a.ckpt_read);
    float* scales = reinterpret_cast<float*>(q + (size_t)a.Sn * a.H * a.P * FN);
#pragma unroll
    for (int rr = 0; rr < 8; rr++) store_f8_row(q, scales, off / FN + rr, hv[rr], lane);
  } else {
#pragma unroll
    for (int rr = 0; rr < 8; rr++)
      __stcs(reinterpret_cast<uint2*>(a.ckpt_read + off + (size_t)rr * FN), to_rc4(hv[rr], a.read_f16));
  }
}

// h1 = P h0 + sum_k (w_k x_k[r]) B_k for 8 rows, written once (and the read copy);
// the window's B rows are ring group row sg, the current record's is record group row bg.
__device__ __forceinline__ void fold8(const M2Args& a, float4 (&hv)[8], float Pm, float wk, const float (&xl)[8],
                                      int m, int count, int start, int sg, int bg, size_t off, int lane) {
  const int L = a.L;
#pragma unroll
  for (int rr = 0; rr < 8; rr++) hv[rr] = scale4(Pm, hv[rr]);
  const uint16_t* rB = a.rB + (size_t)sg * L * FN + lane * 4;
  for (int k = 0; k < m; k++) {
    const float w = __shfl_sync(FULL, wk, k);
    int s = start + k;
    s = s < L ? s : s - L;
    const float4 bk = load_bf4(k < count ? rB + s * FN : a.B + (size_t)bg * FN + lane * 4);
#pragma unroll
    for (int rr = 0; rr < 8; rr++) hv[rr] = fma4(w * __shfl_sync(FULL, xl[rr], k), bk, hv[rr]);
  }
#pragma unroll
  for (int rr = 0; rr < 8; rr++) __stcs(reinterpret_cast<float4*>(a.ckpt + off + (size_t)rr * FN), hv[rr]);
  store_read_copy8(a, hv, off, lane);
}

}  // namespace fastrows
}  // namespace rssm
