// ReplaySSM AR decode step for Mamba-2, shape-specialised fast path:
// dstate = 128 and headdim a multiple of 64 (the serving layers). Same
// algorithm as the generic kernel in mamba2_step.cu ("How ReplaySSM works":
// non-flush steps read the checkpoint and the window and store no state; the
// L-th step folds the window into the checkpoint and writes it once), laid
// out so that almost every instruction is a load, an FMA or a shuffle:
// compile-time row strides, one 64-bit base pointer per stream, no runtime
// shape predicates.
//
// One CTA of four warps per (sequence, head, 64-row block); warp w owns rows
// 16w..16w+15 and lane l the float4 column chunk 4l..4l+3 of each. At launch
// every thread issues its 16 checkpoint-row loads (fp32; the bf16 read copy is
// chosen after the cursor on non-flush steps) and, independently of the
// cursor, lane s loads ring slot s (its dt and its x rows for the warp) and the
// current record; once the cursor arrives lane k takes record k from lane
// (start + k) mod L by a shuffle. Warp w forms the B.C dots of ring slots
// w, w+4, ... and of the current record (slot L) and shares them through
// shared memory. Each lane then adds its record's term (w_k c_k [+ D on the
// current record]) x_k[r] to its P (h0 . C) partials so that one transposed
// 8-row reduction yields P (h0 C)[r] + sum_k w_k c_k x_k[r] + D x[r]; the gate
// and the store run one lane per row. On the L-th step the window is folded
// into the rows in registers and written once; otherwise the record is
// appended to its ring slot. The cursor is only read; a trailing kernel
// advances it.
#include "common.cuh"
#include "kernels.h"

namespace rssm {

namespace {

constexpr int FN = 128;   // dstate
constexpr int FPB = 64;   // rows per block
constexpr int FW = 4;     // warps, 16 rows each
constexpr int FT = 32 * FW;

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void unpack8(uint4 u, float* f) {
  f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
  f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}

__device__ __forceinline__ uint4 shfl_u4(uint4 v, int src) {
  return make_uint4(__shfl_sync(FULL, v.x, src), __shfl_sync(FULL, v.y, src), __shfl_sync(FULL, v.z, src),
                    __shfl_sync(FULL, v.w, src));
}

template <int LM, bool OUT_BF16>
__global__ void __launch_bounds__(FT, 4) m2_step_fast_kernel(M2Args a) {
  constexpr int KW = LM == 16 ? 8 : 16;  // 4 warps x KW >= L + 1 dots
  __shared__ float sc[FW * KW];          // c_s = B_s . C by ring slot; [L] = current record
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.y;
  const int h = blockIdx.x / a.nPB, pb = blockIdx.x - h * a.nPB;
  const int L = a.L, P = a.P, H = a.H;
  const int g = h / (H / a.G);
  const int bh = b * H + h, bg = b * a.G + g;
  const int prow = pb * FPB + warp * 16;  // the warp's first row within the head
  const bool copy = a.ckpt_read != nullptr;
  const size_t hoff = ((size_t)bh * P + prow) * FN + lane * 4;

  // checkpoint rows first
  float4 hv[16];
  if (!copy) {
    const float4* src = reinterpret_cast<const float4*>(a.ckpt + hoff);
#pragma unroll
    for (int r = 0; r < 16; r++) hv[r] = __ldcs(src + r * (FN / 4));
  }
  // cursor-independent records: ring slot `lane`, the current record, the group's C
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * b);
  const float dts = lane < L ? a.rdt[(size_t)bh * pad4(L) + lane] : 0.f;
  const float dtc = a.dt[bh];
  const float Ah = a.A[h], Dh = a.D[h];
  uint4 xs0 = make_uint4(0, 0, 0, 0), xs1 = xs0;
  if (lane < L) {
    const uint16_t* xp = a.rx + ((size_t)bh * L + lane) * P + prow;
    xs0 = ldg16(xp);
    xs1 = ldg16(xp + 8);
  }
  const uint16_t* xcp = a.x + (size_t)bh * P + prow;
  const uint4 xc0 = ldg16(xcp), xc1 = ldg16(xcp + 8);
  const float4 cm = load_bf4(a.C + (size_t)bg * FN + lane * 4);
  {  // c_s = B_s . C for slots s = warp + 4 i (s == L: the current record)
    const uint16_t* rB = a.rB + (size_t)bg * L * FN + lane * 4;
    const float4 bcur = load_bf4(a.B + (size_t)bg * FN + lane * 4);
    float pk[KW];
#pragma unroll
    for (int i = 0; i < KW; i++) {
      const int s = warp + FW * i;
      pk[i] = s < L ? dot4(load_bf4(rB + s * FN), cm) : (s == L ? dot4(bcur, cm) : 0.f);
    }
    const float red = reduce_transpose<KW>(pk, lane);
    const int idx = KW == 8 ? reduce8_row(lane) : (lane >> 1);
    const bool rep = KW == 8 ? (lane & 3) == 0 : (lane & 1) == 0;
    if (rep) sc[warp + FW * idx] = red;
  }

  const int start = cur.x, count = cur.y;
  if (start < 0 || start >= L || count < 0 || count >= L || cur.z != 0) return;  // reported by the cursor kernel
  const int m = count + 1;
  const bool flush = (m == L);
  if (copy) {
    if (flush) {
      const float4* src = reinterpret_cast<const float4*>(a.ckpt + hoff);
#pragma unroll
      for (int r = 0; r < 16; r++) hv[r] = __ldcs(src + r * (FN / 4));
    } else {
      const uint16_t* src = a.ckpt_read + hoff;
#pragma unroll
      for (int r = 0; r < 16; r++) hv[r] = load_bf4(src + r * FN);
    }
  }
  // window: lane k < count is ring slot (start + k) mod L, lane count the current record
  int sl = start + lane;
  sl = sl < L ? sl : sl - L;
  const float dtr = __shfl_sync(FULL, dts, sl);
  const float dtk = lane < count ? dtr : (lane == count ? dtc : 0.f);
  const uint4 xr0 = shfl_u4(xs0, sl), xr1 = shfl_u4(xs1, sl);
  float xl[16];
  unpack8(lane < count ? xr0 : xc0, xl);
  unpack8(lane < count ? xr1 : xc1, xl + 8);
  // decay weights, lane k = record k
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
  const float coef = lane < m ? fmaf(wk, sc[lane < count ? sl : L], lane == count ? Dh : 0.f) : 0.f;

  // pre-gate outputs of the warp's 16 rows
  float tot[2];
#pragma unroll
  for (int gg = 0; gg < 2; gg++) {
    float v[8];
#pragma unroll
    for (int rr = 0; rr < 8; rr++) v[rr] = fmaf(Pm, dot4(hv[gg * 8 + rr], cm), coef * xl[gg * 8 + rr]);
    tot[gg] = reduce_transpose<8>(v, lane);
  }
  {
    const int rr = lane & 7;
    const int src = ((rr >> 2) & 1) * 16 + ((rr >> 1) & 1) * 8 + (rr & 1) * 4;
    const float t0 = __shfl_sync(FULL, tot[0], src), t1 = __shfl_sync(FULL, tot[1], src);
    if (lane < 16) {
      const size_t oi = (size_t)bh * P + prow + lane;
      const float zm = bf_to_f(a.z[oi]);
      const float yv = (lane & 8 ? t1 : t0) * __fdividef(zm, 1.f + __expf(-zm));
      if (OUT_BF16)
        reinterpret_cast<uint16_t*>(a.y)[oi] = f_to_bf(yv);
      else
        reinterpret_cast<float*>(a.y)[oi] = yv;
    }
  }

  if (flush) {  // fold the window into the rows in registers, write them once
#pragma unroll
    for (int r = 0; r < 16; r++) hv[r] = scale4(Pm, hv[r]);
    const uint16_t* rB = a.rB + (size_t)bg * L * FN + lane * 4;
    for (int k = 0; k < m; k++) {
      const float w = __shfl_sync(FULL, wk, k);
      int s = start + k;
      s = s < L ? s : s - L;
      const float4 bk = load_bf4(k < count ? rB + s * FN : a.B + (size_t)bg * FN + lane * 4);
#pragma unroll
      for (int r = 0; r < 16; r++) hv[r] = fma4(w * __shfl_sync(FULL, xl[r], k), bk, hv[r]);
    }
    float4* dst = reinterpret_cast<float4*>(a.ckpt + hoff);
#pragma unroll
    for (int r = 0; r < 16; r++) __stcs(dst + r * (FN / 4), hv[r]);
    if (copy) {
      uint2* d16 = reinterpret_cast<uint2*>(a.ckpt_read + hoff);
#pragma unroll
      for (int r = 0; r < 16; r++) __stcs(d16 + r * (FN / 4), f4_to_bf4(hv[r]));
    }
  } else {  // append the current record: x, z rows of this warp; dt, B, C once
    const int slot = start + count < L ? start + count : start + count - L;
    const size_t rrow = ((size_t)bh * L + slot) * P + prow;
    if (lane < 2) *reinterpret_cast<uint4*>(a.rx + rrow + lane * 8) = lane ? xc1 : xc0;
    if (lane == 2 || lane == 3) {
      const int o = (lane - 2) * 8;
      *reinterpret_cast<uint4*>(a.rz + rrow + o) = ldg16(a.z + (size_t)bh * P + prow + o);
    }
    if (warp == 0 && pb == 0) {
      if (lane == 4) a.rdt[(size_t)bh * pad4(L) + slot] = dtc;
      if (h == g * (H / a.G) && lane < FN / 8) {  // the group's first head stores the group rows
        const size_t brow = ((size_t)bg * L + slot) * FN + lane * 8;
        *reinterpret_cast<uint4*>(a.rB + brow) = ldg16(a.B + (size_t)bg * FN + lane * 8);
        *reinterpret_cast<uint4*>(a.rC + brow) = ldg16(a.C + (size_t)bg * FN + lane * 8);
      }
    }
  }
}

}  // namespace

bool m2_step_fast_applies(const M2Args& a) { return a.N == FN && a.P % FPB == 0 && a.PB == FPB; }

cudaError_t m2_step_fast_launch(const M2Args& a, int out_bf16, cudaStream_t st) {
  const dim3 grid(a.H * a.nPB, a.Bt);
  if (a.L <= 16) {
    if (out_bf16)
      m2_step_fast_kernel<16, true><<<grid, FT, 0, st>>>(a);
    else
      m2_step_fast_kernel<16, false><<<grid, FT, 0, st>>>(a);
  } else {
    if (out_bf16)
      m2_step_fast_kernel<32, true><<<grid, FT, 0, st>>>(a);
    else
      m2_step_fast_kernel<32, false><<<grid, FT, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace rssm
