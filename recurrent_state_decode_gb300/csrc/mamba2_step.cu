// ReplaySSM AR decode step for Mamba-2 on sm_103a ("How ReplaySSM works":
// non-flush steps read the checkpoint and the window and store no state; the
// L-th step folds the window into the checkpoint and writes it once).
//
// One CTA of four warps per (sequence, head, row block); each warp owns up to
// 16 rows (8 when dstate > 128) and each lane a float4 column chunk of them.
// The kernel is shaped like a streaming copy: every thread first issues the
// 16-byte loads of its checkpoint rows straight into registers (the bf16
// read copy on non-flush steps when there is one), so a resident CTA keeps its
// whole 32 KiB tile in flight, and only then does the latency-bound window
// work:
//   1. lane k of every warp takes record k's dt and one warp suffix scan gives
//      w_k = dt_k exp(A sum_{j>k} dt_j) and P = exp(A sum_j dt_j);
//   2. warp w forms c_k = B_k . C for records k = w, w+4, ... (per-lane
//      partials over the lane's column chunk, one transposed butterfly
//      reduction for all of them) and shares them through shared memory;
//   3. lane k holds x_k of the warp's rows; per 8-row group each lane adds its
//      record's term (w_k c_k [+ D on the current record]) x_k[r] to its
//      P (h0 . C) partials, so one transposed 8-row reduction gives
//      P (h0 C)[r] + sum_k w_k c_k x_k[r] + D x[r]; the gate silu(z) and the
//      store run on one lane per row;
//   4. on the L-th step the window is folded into the rows held in registers
//      and written once (with the bf16 read copy); otherwise the record is
//      appended to its ring slot.
// The cursor is only read here; a trailing kernel advances it.
#include "common.cuh"
#include "kernels.h"

namespace rssm {

namespace {

constexpr int THREADS = 128;

// Rows [r0, r1) of warp w: R rows (a multiple of 8) in 8-row groups dealt out
// contiguously to the four warps.
__device__ __forceinline__ void warp_rows(int R, int w, int& r0, int& r1) {
  const int ngrp = R >> 3;
  r0 = ((w * ngrp) >> 2) * 8;
  r1 = (((w + 1) * ngrp) >> 2) * 8;
}

template <int LM, int NCH, bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 4) m2_step_kernel(M2Args a) {
  constexpr int G8 = 2 / NCH;   // 8-row groups per warp at most
  constexpr int KW = LM / 4;    // records whose B.C dot one warp forms
  __shared__ float sc[LM];      // c_k = B_k . C
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int blk = blockIdx.x;
  const int pb = blk % a.nPB;
  blk /= a.nPB;
  const int h = blk % a.H, b = blk / a.H;
  const int L = a.L, N = a.N, P = a.P, H = a.H, G = a.G;
  const int g = (h * G) / H;
  const int p0 = pb * a.PB, R = min(a.PB, P - p0);
  const size_t bh = (size_t)b * H + h, bg = (size_t)b * G + g;
  int r0w, r1w;
  warp_rows(R, warp, r0w, r1w);
  const int nrows = r1w - r0w;
  const size_t toff = (bh * P + p0) * N;

  // 0. checkpoint rows into registers first (fp32 unless a read copy is used)
  float4 hv[G8][8][NCH];
  const bool has_copy = a.ckpt_read != nullptr;
  if (!has_copy) {
#pragma unroll
    for (int gg = 0; gg < G8; gg++)
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) {
          const int c = lane + 32 * jj;
          hv[gg][rr][jj] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (gg * 8 < nrows && c * 4 < N)
            hv[gg][rr][jj] =
                __ldcs(reinterpret_cast<const float4*>(a.ckpt + toff + (size_t)(r0w + gg * 8 + rr) * N) + c);
        }
  }
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)b);
  const int start = cur.x, count = cur.y;
  if (start < 0 || start >= L || count < 0 || count >= L || cur.z != 0) return;  // reported by the cursor kernel
  const int m = count + 1;
  const bool flush = (m == L);
  if (has_copy) {
#pragma unroll
    for (int gg = 0; gg < G8; gg++)
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) {
          const int c = lane + 32 * jj;
          const size_t row = toff + (size_t)(r0w + gg * 8 + rr) * N;
          hv[gg][rr][jj] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (gg * 8 < nrows && c * 4 < N)
            hv[gg][rr][jj] = flush ? __ldcs(reinterpret_cast<const float4*>(a.ckpt + row) + c)
                                   : load_bf4(a.ckpt_read + row + c * 4);
        }
  }

  // window record k: ring slot (start + k) mod L for k < count, the input for k == count
  const int kl = lane;
  int sl = start + kl;
  sl = sl < L ? sl : sl - L;
  const float dtk = kl < count ? a.rdt[bh * pad4(L) + sl] : (kl == count ? a.dt[bh] : 0.f);
  const float Ah = a.A[h];
  float4 cm[NCH];
#pragma unroll
  for (int jj = 0; jj < NCH; jj++) {
    const int c = lane + 32 * jj;
    cm[jj] = (c * 4 < N) ? load_bf4(a.C + bg * N + c * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // x_k of this warp's rows, lane k (16 rows: two 16-byte loads)
  float xl[G8][8];
#pragma unroll
  for (int gg = 0; gg < G8; gg++) {
#pragma unroll
    for (int rr = 0; rr < 8; rr++) xl[gg][rr] = 0.f;
    if (kl < m && gg * 8 < nrows) {
      const uint16_t* xs = kl < count ? a.rx + (bh * L + sl) * P : a.x + bh * P;
      const uint4 u = *reinterpret_cast<const uint4*>(xs + p0 + r0w + gg * 8);
      xl[gg][0] = bf_lo(u.x); xl[gg][1] = bf_hi(u.x); xl[gg][2] = bf_lo(u.y); xl[gg][3] = bf_hi(u.y);
      xl[gg][4] = bf_lo(u.z); xl[gg][5] = bf_hi(u.z); xl[gg][6] = bf_lo(u.w); xl[gg][7] = bf_hi(u.w);
    }
  }
  // 2. c_k = B_k . C for k = warp + 4 i
  {
    float pk[KW];
#pragma unroll
    for (int i = 0; i < KW; i++) {
      pk[i] = 0.f;
      const int k = warp + 4 * i;
      if (k < m) {
        int s = start + k;
        s = s < L ? s : s - L;
        const uint16_t* Bk = k < count ? a.rB + (bg * L + s) * N : a.B + bg * N;
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) {
          const int c = lane + 32 * jj;
          if (c * 4 < N) pk[i] += dot4(load_bf4(Bk + c * 4), cm[jj]);
        }
      }
    }
    const float red = reduce_transpose<KW>(pk, lane);
    // lanes whose low bits are zero hold partial index idx(lane) (see reduce_transpose)
    const int idx = KW == 4 ? ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1) : reduce8_row(lane);
    const bool rep = KW == 4 ? (lane & 7) == 0 : (lane & 3) == 0;
    if (rep && warp + 4 * idx < LM) sc[warp + 4 * idx] = red;
  }
  // 1. decay weights (every warp, lane k = record k)
  float sfx = dtk * Ah;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float v = __shfl_down_sync(FULL, sfx, o);
    if (lane + o < 32) sfx += v;
  }
  float ex = __shfl_down_sync(FULL, sfx, 1);
  if (lane == 31) ex = 0.f;
  const float Pm = expf(__shfl_sync(FULL, sfx, 0));
  const float wk = dtk * expf(ex);
  __syncthreads();
  const float coef = kl < m ? fmaf(wk, sc[kl], kl == count ? a.D[h] : 0.f) : 0.f;

  // 3. pre-gate outputs
  float tot[G8];
#pragma unroll
  for (int gg = 0; gg < G8; gg++) {
    float v[8];
#pragma unroll
    for (int rr = 0; rr < 8; rr++) {
      float d = 0.f;
#pragma unroll
      for (int jj = 0; jj < NCH; jj++) d += dot4(hv[gg][rr][jj], cm[jj]);
      v[rr] = fmaf(Pm, d, coef * xl[gg][rr]);
    }
    tot[gg] = reduce_transpose<8>(v, lane);
  }
  {  // lane r < nrows gathers row r's total, gates and stores it
    const int rr = lane & 7;
    const int src = ((rr >> 2) & 1) * 16 + ((rr >> 1) & 1) * 8 + (rr & 1) * 4;
    float mine = __shfl_sync(FULL, tot[0], src);
    if (G8 > 1) {
      const float t1 = __shfl_sync(FULL, tot[G8 - 1], src);
      if (lane & 8) mine = t1;
    }
    if (lane < nrows) {
      const size_t oi = bh * P + p0 + r0w + lane;
      const float zm = bf_to_f(a.z[oi]);
      const float yv = mine * __fdividef(zm, 1.f + __expf(-zm));
      if (OUT_BF16)
        reinterpret_cast<uint16_t*>(a.y)[oi] = f_to_bf(yv);
      else
        reinterpret_cast<float*>(a.y)[oi] = yv;
    }
  }

  if (flush) {  // 4a. fold the window into the rows in registers, write them once
#pragma unroll
    for (int gg = 0; gg < G8; gg++) {
      if (gg * 8 >= nrows) continue;
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) hv[gg][rr][jj] = scale4(Pm, hv[gg][rr][jj]);
      for (int k = 0; k < m; k++) {
        const float w = __shfl_sync(FULL, wk, k);
        float wx[8];
#pragma unroll
        for (int rr = 0; rr < 8; rr++) wx[rr] = w * __shfl_sync(FULL, xl[gg][rr], k);
        int s = start + k;
        s = s < L ? s : s - L;
        const uint16_t* Bk = k < count ? a.rB + (bg * L + s) * N : a.B + bg * N;
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) {
          const int c = lane + 32 * jj;
          if (c * 4 < N) {
            const float4 bk = load_bf4(Bk + c * 4);
#pragma unroll
            for (int rr = 0; rr < 8; rr++) hv[gg][rr][jj] = fma4(wx[rr], bk, hv[gg][rr][jj]);
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) {
          const int c = lane + 32 * jj;
          if (c * 4 < N) {
            const size_t o = toff + (size_t)(r0w + gg * 8 + rr) * N + c * 4;
            __stcs(reinterpret_cast<float4*>(a.ckpt + o), hv[gg][rr][jj]);
            if (has_copy) __stcs(reinterpret_cast<uint2*>(a.ckpt_read + o), f4_to_bf4(hv[gg][rr][jj]));
          }
        }
    }
  } else {  // 4b. append the current record: x, z rows of this warp; dt, B, C once
    const int slot = start + count < L ? start + count : start + count - L;
    const size_t rrow = (bh * L + slot) * P + p0;
    if (lane < 2 * (nrows >> 3)) {
      const int f = lane & 1, r = r0w + (lane >> 1) * 8;
      const uint16_t* src = (f ? a.z : a.x) + bh * P + p0 + r;
      uint16_t* dst = (f ? a.rz : a.rx) + rrow + r;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    }
    if (warp == 0 && pb == 0) {
      if (lane == 0) a.rdt[bh * pad4(L) + slot] = a.dt[bh];
      if (h == g * (H / G)) {  // the group's first head stores the group rows
        const size_t brow = (bg * L + slot) * N;
        for (int i = lane; i < (N >> 3); i += 32) {
          *reinterpret_cast<uint4*>(a.rB + brow + i * 8) = *reinterpret_cast<const uint4*>(a.B + bg * N + i * 8);
          *reinterpret_cast<uint4*>(a.rC + brow + i * 8) = *reinterpret_cast<const uint4*>(a.C + bg * N + i * 8);
        }
      }
    }
  }
}

template <int LM, int NCH, bool OUT_BF16>
cudaError_t launch_step(const M2Args& a, cudaStream_t st) {
  m2_step_kernel<LM, NCH, OUT_BF16><<<a.Bt * a.H * a.nPB, THREADS, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t m2_step_launch(const M2Args& a, int out_bf16, cudaStream_t st) {
  if (a.Bt * a.H * a.nPB == 0) return cudaSuccess;
  const bool small_window = a.L <= 16, narrow = a.N <= 128;
  if (small_window) {
    if (narrow) return out_bf16 ? launch_step<16, 1, true>(a, st) : launch_step<16, 1, false>(a, st);
    return out_bf16 ? launch_step<16, 2, true>(a, st) : launch_step<16, 2, false>(a, st);
  }
  if (narrow) return out_bf16 ? launch_step<32, 1, true>(a, st) : launch_step<32, 1, false>(a, st);
  return out_bf16 ? launch_step<32, 2, true>(a, st) : launch_step<32, 2, false>(a, st);
}

}  // namespace rssm
