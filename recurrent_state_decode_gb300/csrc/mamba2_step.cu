// ReplaySSM AR decode step for Mamba-2 on sm_103a ("How ReplaySSM works":
// non-flush steps read the checkpoint and the window and store no state; the
// L-th step folds the window into the checkpoint and writes it once).
//
// One CTA of eight warps per (sequence, head, row block); each warp owns 8
// rows and each lane a float4 column chunk of them (two when dstate > 128).
// The kernel is shaped like a streaming copy: at launch every thread issues
// the 16-byte loads of its checkpoint rows straight into registers, and, in
// the same breath, lane s loads ring slot s (its dt and its x rows for the
// warp) and the current record, none of which waits on the cursor. Once the
// cursor arrives, lane k takes record k from lane (start + k) mod L by a
// shuffle. Then:
//   1. one warp suffix scan over the window (lane k = record k) gives
//      w_k = dt_k exp(A sum_{j>k} dt_j) and P = exp(A sum_j dt_j);
//   2. the warps form c_s = B_s . C for every ring slot and the current record
//      (per-lane partials over the lane's column chunk, one transposed
//      butterfly reduction per warp) and share them through shared memory;
//   3. each lane adds its record's term (w_k c_k [+ D on the current record])
//      x_k[r] to its P (h0 . C) partials, so one transposed 8-row reduction
//      gives P (h0 C)[r] + sum_k w_k c_k x_k[r] + D x[r]; the gate silu(z)
//      and the store run on one lane per row;
//   4. on the L-th step the window is folded into the rows held in registers
//      and written once (with the bf16 read copy); otherwise the record is
//      appended to its ring slot.
// Loading every ring slot's x rows rather than only the window's costs the
// unused slots' bytes (a few percent of the step) and removes a dependent
// round trip from every block. The cursor is only read; a trailing kernel
// advances it. With a bf16 read copy the checkpoint load waits for the
// cursor, which decides between the copy and the fp32 rows.
#include "common.cuh"
#include "kernels.h"

namespace rssm {

namespace {

constexpr int WARPS = 8;
constexpr int THREADS = 32 * WARPS;

__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
  f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
  f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}

__device__ __forceinline__ uint4 shfl_u4(uint4 v, int src) {
  return make_uint4(__shfl_sync(FULL, v.x, src), __shfl_sync(FULL, v.y, src), __shfl_sync(FULL, v.z, src),
                    __shfl_sync(FULL, v.w, src));
}

// KW = ring slots (plus the current record) whose B.C dot one warp forms:
// warp w takes slots w, w + 8, ...; slot L stands for the current record.
template <int LM, int NCH, bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, NCH == 1 ? 3 : 2) m2_step_kernel(M2Args a) {
  constexpr int KW = LM == 16 ? 4 : 8;  // 8 warps x KW >= L + 1
  __shared__ float sc[WARPS * KW];      // c_s = B_s . C by ring slot; [L] = current record
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int blk = blockIdx.x;
  const int pb = blk % a.nPB;
  blk /= a.nPB;
  const int h = blk % a.H, b = blk / a.H;
  const int L = a.L, N = a.N, P = a.P, H = a.H, G = a.G;
  const int g = (h * G) / H;
  const int p0 = pb * a.PB, R = min(a.PB, P - p0);
  const size_t bh = (size_t)b * H + h, bg = (size_t)b * G + g;
  const int r0 = warp * 8;
  const bool rows = r0 < R;  // R is a multiple of 8
  const size_t toff = (bh * P + p0 + r0) * N;
  const bool has_copy = a.ckpt_read != nullptr;

  // 0. loads that do not depend on the cursor
  float4 hv[8][NCH];
  if (!has_copy) {
#pragma unroll
    for (int rr = 0; rr < 8; rr++)
#pragma unroll
      for (int jj = 0; jj < NCH; jj++) {
        const int c = lane + 32 * jj;
        hv[rr][jj] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (rows && c * 4 < N) hv[rr][jj] = __ldcs(reinterpret_cast<const float4*>(a.ckpt + toff + (size_t)rr * N) + c);
      }
  }
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)b);
  const float dts = lane < L ? a.rdt[bh * pad4(L) + lane] : 0.f;   // ring slot `lane`
  const float dtc = a.dt[bh];                                     // current record
  uint4 xs = make_uint4(0, 0, 0, 0), xc = make_uint4(0, 0, 0, 0);
  if (rows) {
    if (lane < L) xs = *reinterpret_cast<const uint4*>(a.rx + (bh * L + lane) * P + p0 + r0);
    xc = *reinterpret_cast<const uint4*>(a.x + bh * P + p0 + r0);
  }
  float4 cm[NCH];
#pragma unroll
  for (int jj = 0; jj < NCH; jj++) {
    const int c = lane + 32 * jj;
    cm[jj] = (c * 4 < N) ? load_bf4(a.C + bg * N + c * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  {  // 2. c_s = B_s . C for slots s = warp + 8 i (s == L: the current record)
    float pk[KW];
#pragma unroll
    for (int i = 0; i < KW; i++) {
      pk[i] = 0.f;
      const int s = warp + WARPS * i;
      if (s <= L) {
        const uint16_t* Bs = s < L ? a.rB + (bg * L + s) * N : a.B + bg * N;
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) {
          const int c = lane + 32 * jj;
          if (c * 4 < N) pk[i] += dot4(load_bf4(Bs + c * 4), cm[jj]);
        }
      }
    }
    const float red = reduce_transpose<KW>(pk, lane);
    const int idx = KW == 4 ? ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1) : reduce8_row(lane);
    const bool rep = KW == 4 ? (lane & 7) == 0 : (lane & 3) == 0;
    if (rep) sc[warp + WARPS * idx] = red;
  }

  // the cursor decides the window: record k < count is ring slot (start + k) mod L
  const int start = cur.x, count = cur.y;
  if (start < 0 || start >= L || count < 0 || count >= L || cur.z != 0) return;  // reported by the cursor kernel
  const int m = count + 1;
  const bool flush = (m == L);
  if (has_copy) {
#pragma unroll
    for (int rr = 0; rr < 8; rr++)
#pragma unroll
      for (int jj = 0; jj < NCH; jj++) {
        const int c = lane + 32 * jj;
        const size_t row = toff + (size_t)rr * N;
        hv[rr][jj] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (rows && c * 4 < N)
          hv[rr][jj] = flush ? __ldcs(reinterpret_cast<const float4*>(a.ckpt + row) + c)
                             : load_bf4(a.ckpt_read + row + c * 4);
      }
  }
  int sl = start + lane;
  sl = sl < L ? sl : sl - L;
  const int slot_of_lane = lane < count ? sl : L;  // L = the current record
  const float dtr = __shfl_sync(FULL, dts, sl);
  const float dtk = lane < count ? dtr : (lane == count ? dtc : 0.f);
  const uint4 xr = shfl_u4(xs, sl);
  float xl[8];
  unpack8(lane < count ? xr : xc, xl);
  if (lane >= m) {
#pragma unroll
    for (int rr = 0; rr < 8; rr++) xl[rr] = 0.f;
  }
  // 1. decay weights (lane k = record k)
  float sfx = dtk * a.A[h];
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
  const float coef = lane < m ? fmaf(wk, sc[slot_of_lane], lane == count ? a.D[h] : 0.f) : 0.f;
  if (!rows) return;

  // 3. pre-gate outputs of the warp's 8 rows
  float v[8];
#pragma unroll
  for (int rr = 0; rr < 8; rr++) {
    float d = 0.f;
#pragma unroll
    for (int jj = 0; jj < NCH; jj++) d += dot4(hv[rr][jj], cm[jj]);
    v[rr] = fmaf(Pm, d, coef * xl[rr]);
  }
  reduce_transpose<8>(v, lane);
  {
    const int rr = lane & 7;
    const int src = ((rr >> 2) & 1) * 16 + ((rr >> 1) & 1) * 8 + (rr & 1) * 4;
    const float mine = __shfl_sync(FULL, v[0], src);
    if (lane < 8) {
      const size_t oi = bh * P + p0 + r0 + lane;
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
    for (int rr = 0; rr < 8; rr++)
#pragma unroll
      for (int jj = 0; jj < NCH; jj++) hv[rr][jj] = scale4(Pm, hv[rr][jj]);
    for (int k = 0; k < m; k++) {
      const float w = __shfl_sync(FULL, wk, k);
      float wx[8];
#pragma unroll
      for (int rr = 0; rr < 8; rr++) wx[rr] = w * __shfl_sync(FULL, xl[rr], k);
      int s = start + k;
      s = s < L ? s : s - L;
      const uint16_t* Bk = k < count ? a.rB + (bg * L + s) * N : a.B + bg * N;
#pragma unroll
      for (int jj = 0; jj < NCH; jj++) {
        const int c = lane + 32 * jj;
        if (c * 4 < N) {
          const float4 bk = load_bf4(Bk + c * 4);
#pragma unroll
          for (int rr = 0; rr < 8; rr++) hv[rr][jj] = fma4(wx[rr], bk, hv[rr][jj]);
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 8; rr++)
#pragma unroll
      for (int jj = 0; jj < NCH; jj++) {
        const int c = lane + 32 * jj;
        if (c * 4 < N) {
          const size_t o = toff + (size_t)rr * N + c * 4;
          __stcs(reinterpret_cast<float4*>(a.ckpt + o), hv[rr][jj]);
          if (has_copy) __stcs(reinterpret_cast<uint2*>(a.ckpt_read + o), f4_to_bf4(hv[rr][jj]));
        }
      }
  } else {  // 4b. append the current record: x, z rows of this warp; dt, B, C once
    const int slot = start + count < L ? start + count : start + count - L;
    const size_t rrow = (bh * L + slot) * P + p0 + r0;
    if (lane == 0) *reinterpret_cast<uint4*>(a.rx + rrow) = xc;
    if (lane == 1) *reinterpret_cast<uint4*>(a.rz + rrow) = *reinterpret_cast<const uint4*>(a.z + bh * P + p0 + r0);
    if (warp == 0 && pb == 0) {
      if (lane == 2) a.rdt[bh * pad4(L) + slot] = dtc;
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
