// ReplaySSM AR decode step for Mamba-2 on sm_103a ("How ReplaySSM works":
// non-flush steps read the checkpoint and the window and store no state; the
// L-th step folds the window into the checkpoint and writes it once).
//
// One CTA of eight warps per (sequence, run of HPC consecutive heads of one
// group, row block). Everything a sequence's heads share is done once per CTA:
// the cursor, the window's slots and the B.C dots (B and C are group rows).
// Each warp owns 8 rows of the row block, each lane a float4 column chunk of
// them (two when dstate > 128). The heads are software-pipelined in
// registers: before a warp computes head i it issues the 16-byte loads of head
// i+1's checkpoint rows and records, so every resident CTA keeps a tile in
// flight the whole time, like a streaming copy. Per head:
//   1. lane k takes record k (ring slot (start + k) mod L, or the current
//      record) by a shuffle from the lane that loaded that slot, and one warp
//      suffix scan gives w_k = dt_k exp(A sum_{j>k} dt_j), P = exp(A sum dt);
//   2. each lane adds its record's term (w_k c_k [+ D on the current record])
//      x_k[r] to its P (h0 . C) partials, so one transposed 8-row reduction
//      gives P (h0 C)[r] + sum_k w_k c_k x_k[r] + D x[r]; the gate silu(z) and
//      the store run on one lane per row;
//   3. on the L-th step the window is folded into the rows in registers and
//      written once (with the bf16 read copy); otherwise the record is
//      appended to its ring slot.
// The B.C dots c_s of every ring slot and of the current record are formed
// at the start by the eight warps together (per-lane partials over the lane's
// column chunk, one transposed butterfly reduction per warp). Fetching every
// ring slot's x rows, not only the window's, costs the unused slots' bytes (a
// few percent of the step) and takes the cursor off the load path. The cursor
// is only read; a trailing kernel advances it.
#include "common.cuh"
#include "kernels.h"

namespace rssm {

namespace {

constexpr int WARPS = 8;
constexpr int THREADS = 32 * WARPS;

// What one head needs besides the dots: its checkpoint rows and records.
template <int NCH>
struct HeadData {
  float4 hv[8][NCH];
  uint4 xs;   // x rows of ring slot `lane`
  uint4 xc;   // x rows of the current record
  float dts;  // dt of ring slot `lane`
  float dtc;  // dt of the current record
};

template <int NCH>
__device__ __forceinline__ void load_head(HeadData<NCH>& d, const M2Args& a, size_t bh, int p0, int r0, bool rows,
                                          bool fp32_rows, int lane) {
  const int L = a.L, N = a.N, P = a.P;
  const size_t toff = (bh * P + p0 + r0) * N;
#pragma unroll
  for (int rr = 0; rr < 8; rr++)
#pragma unroll
    for (int jj = 0; jj < NCH; jj++) {
      const int c = lane + 32 * jj;
      d.hv[rr][jj] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rows && c * 4 < N) {
        const size_t row = toff + (size_t)rr * N;
        d.hv[rr][jj] = fp32_rows ? __ldcs(reinterpret_cast<const float4*>(a.ckpt + row) + c)
                                 : load_rc4(a.ckpt_read + row + c * 4, a.read_f16);
      }
    }
  d.dts = lane < L ? a.rdt[bh * pad4(L) + lane] : 0.f;
  d.dtc = a.dt[bh];
  d.xs = make_uint4(0, 0, 0, 0);
  d.xc = make_uint4(0, 0, 0, 0);
  if (rows) {
    if (lane < L) d.xs = *reinterpret_cast<const uint4*>(a.rx + (bh * L + lane) * P + p0 + r0);
    d.xc = *reinterpret_cast<const uint4*>(a.x + bh * P + p0 + r0);
  }
}

template <int LM, int NCH, bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, NCH == 1 ? 2 : 1) m2_step_kernel(M2Args a, int hpc) {
  constexpr int KW = LM == 16 ? 4 : 8;  // 8 warps x KW >= L + 1 dots
  __shared__ float sc[WARPS * KW];      // c_s = B_s . C by ring slot; [L] = current record
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.y;
  const int pb = blockIdx.x % a.nPB, h0 = (blockIdx.x / a.nPB) * hpc;
  const int L = a.L, N = a.N, P = a.P, H = a.H, G = a.G;
  const int g = (h0 * G) / H;
  const int p0 = pb * a.PB, R = min(a.PB, P - p0);
  const size_t bg = (size_t)b * G + g;
  const int r0 = warp * 8;
  const bool rows = r0 < R;  // R is a multiple of 8
  const bool has_copy = a.ckpt_read != nullptr;

  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)b);
  HeadData<NCH> d;
  if (!has_copy) load_head<NCH>(d, a, (size_t)b * H + h0, p0, r0, rows, true, lane);
  float4 cm[NCH];
#pragma unroll
  for (int jj = 0; jj < NCH; jj++) {
    const int c = lane + 32 * jj;
    cm[jj] = (c * 4 < N) ? load_bf4(a.C + bg * N + c * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  {  // c_s = B_s . C for slots s = warp + 8 i (s == L: the current record), shared by the heads
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
  const bool fp32_rows = !has_copy || flush;
  if (has_copy) load_head<NCH>(d, a, (size_t)b * H + h0, p0, r0, rows, fp32_rows, lane);
  int sl = start + lane;
  sl = sl < L ? sl : sl - L;
  const int appl = start + count < L ? start + count : start + count - L;  // slot the record goes to
  __syncthreads();
  const float ck = lane < m ? sc[lane < count ? sl : L] : 0.f;

  for (int i = 0; i < hpc; i++) {
    const int h = h0 + i;
    const size_t bh = (size_t)b * H + h;
    HeadData<NCH> nx;
    if (i + 1 < hpc) load_head<NCH>(nx, a, bh + 1, p0, r0, rows, fp32_rows, lane);  // next head in flight

    // 1. window of this head, lane k = record k
    const float dtr = __shfl_sync(FULL, d.dts, sl);
    const float dtk = lane < count ? dtr : (lane == count ? d.dtc : 0.f);
    const uint4 xr = shfl_u4(d.xs, sl);
    float xl[8];
    unpack8(lane < count ? xr : d.xc, xl);
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
    const float coef = lane < m ? fmaf(wk, ck, lane == count ? a.D[h] : 0.f) : 0.f;

    if (rows) {
      // 2. pre-gate outputs of the warp's 8 rows
      float v[8];
#pragma unroll
      for (int rr = 0; rr < 8; rr++) {
        float dd = 0.f;
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) dd += dot4(d.hv[rr][jj], cm[jj]);
        v[rr] = fmaf(Pm, dd, coef * xl[rr]);
      }
      reduce_transpose<8>(v, lane);
      const int rr8 = lane & 7;
      const int src = ((rr8 >> 2) & 1) * 16 + ((rr8 >> 1) & 1) * 8 + (rr8 & 1) * 4;
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
      const size_t toff = (bh * P + p0 + r0) * N;
      if (flush) {  // 3a. fold the window into the rows in registers, write them once
#pragma unroll
        for (int r = 0; r < 8; r++)
#pragma unroll
          for (int jj = 0; jj < NCH; jj++) d.hv[r][jj] = scale4(Pm, d.hv[r][jj]);
        for (int k = 0; k < m; k++) {
          const float w = __shfl_sync(FULL, wk, k);
          float wx[8];
#pragma unroll
          for (int r = 0; r < 8; r++) wx[r] = w * __shfl_sync(FULL, xl[r], k);
          int s = start + k;
          s = s < L ? s : s - L;
          const uint16_t* Bk = k < count ? a.rB + (bg * L + s) * N : a.B + bg * N;
#pragma unroll
          for (int jj = 0; jj < NCH; jj++) {
            const int c = lane + 32 * jj;
            if (c * 4 < N) {
              const float4 bk = load_bf4(Bk + c * 4);
#pragma unroll
              for (int r = 0; r < 8; r++) d.hv[r][jj] = fma4(wx[r], bk, d.hv[r][jj]);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < 8; r++)
#pragma unroll
          for (int jj = 0; jj < NCH; jj++) {
            const int c = lane + 32 * jj;
            if (c * 4 < N) {
              const size_t o = toff + (size_t)r * N + c * 4;
              __stcs(reinterpret_cast<float4*>(a.ckpt + o), d.hv[r][jj]);
              if (has_copy) __stcs(reinterpret_cast<uint2*>(a.ckpt_read + o), to_rc4(d.hv[r][jj], a.read_f16));
            }
          }
      } else {  // 3b. append the current record: x, z rows of this warp, dt once per head
        const size_t rrow = (bh * L + appl) * P + p0 + r0;
        if (lane == 0) *reinterpret_cast<uint4*>(a.rx + rrow) = d.xc;
        if (lane == 1)
          *reinterpret_cast<uint4*>(a.rz + rrow) = *reinterpret_cast<const uint4*>(a.z + bh * P + p0 + r0);
        if (lane == 2 && warp == 0 && pb == 0) a.rdt[bh * pad4(L) + appl] = d.dtc;
      }
    }
    if (i + 1 < hpc) d = nx;
  }
  // the group's B and C rows, once per group (by the block holding its first head)
  if (!flush && pb == 0 && h0 == g * (H / G)) {
    const size_t brow = (bg * L + appl) * N;
    for (int i = threadIdx.x; i < (N >> 3); i += THREADS) {
      *reinterpret_cast<uint4*>(a.rB + brow + i * 8) = *reinterpret_cast<const uint4*>(a.B + bg * N + i * 8);
      *reinterpret_cast<uint4*>(a.rC + brow + i * 8) = *reinterpret_cast<const uint4*>(a.C + bg * N + i * 8);
    }
  }
}

template <int LM, int NCH, bool OUT_BF16>
cudaError_t launch_step(const M2Args& a, cudaStream_t st) {
  // heads per block: up to 4 consecutive heads of one group
  const int hpg = a.H / a.G;
  const int hpc = hpg % 4 == 0 ? 4 : (hpg % 2 == 0 ? 2 : 1);
  const dim3 grid((a.H / hpc) * a.nPB, a.Bt);
  m2_step_kernel<LM, NCH, OUT_BF16><<<grid, THREADS, 0, st>>>(a, hpc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t m2_step_launch(const M2Args& a, int out_bf16, cudaStream_t st) {
  if (a.Bt * a.H * a.nPB == 0) return cudaSuccess;
  if (m2_step_fast_applies(a)) return m2_step_fast_launch(a, out_bf16, st);
  const bool small_window = a.L <= 16, narrow = a.N <= 128;
  if (small_window) {
    if (narrow) return out_bf16 ? launch_step<16, 1, true>(a, st) : launch_step<16, 1, false>(a, st);
    return out_bf16 ? launch_step<16, 2, true>(a, st) : launch_step<16, 2, false>(a, st);
  }
  if (narrow) return out_bf16 ? launch_step<32, 1, true>(a, st) : launch_step<32, 1, false>(a, st);
  return out_bf16 ? launch_step<32, 2, true>(a, st) : launch_step<32, 2, false>(a, st);
}

}  // namespace rssm
