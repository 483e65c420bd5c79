// ReplaySSM AR decode step for Mamba-2 reading the bf16 read copy of the
// checkpoint ("ReplaySSM" repository, introduction, "Separate state
// precisions": non-flush steps read a low-precision copy; the flush reads and
// writes the fp32 checkpoint and refreshes the copy). Shape-specialised like
// mamba2_step_fast.cu (dstate 128, headdim a multiple of 64, L <= 31), with two
// heads of one group per block so that a warp moves twice the bytes for its
// fixed per-record work: the read copy halves the bytes of a tile, not the work.
//
// One CTA of four warps per (sequence, pair of heads of a group, 64-row block):
// warp w owns head h0 + (w >> 1), rows 32 (w & 1) .. + 31 (four groups of 8).
// At launch, none waiting on the cursor: bulk copies (TMA, non-tensor; never
// multicast) of both heads' bf16 rows (16 KiB each), of their ring x rows (all
// L slots) and of the current record's x rows into shared memory, all on one
// mbarrier; lane s loads ring slot s's dt, and the warps form the B.C dots of
// the group once for both heads. After the cursor each warp scans its head's
// window (w_k = dt_k exp(A sum_{j>k} dt_j), P = exp(A sum dt)); per 8-row group
// lane k reads record k's x rows from shared memory, and one transposed 8-row
// reduction gives y[r] before the gate. A flushing sequence folds from the
// fp32 rows in global memory and writes fp32 and bf16 once. The last of the
// sequence's blocks advances its cursor.
#include "fast_rows.cuh"
#include "kernels.h"

namespace rssm {

namespace {

using namespace fastrows;

constexpr int RG = 4;   // row groups of 8 per warp
constexpr int KW = 8;   // dot entries per warp: 4 x 8 >= L + 1
constexpr int XST = FPB + 8;  // bf16 elements per staged x slot (144 bytes: a 16-byte multiple, off the bank period)

template <bool OUT_BF16>
__global__ void __launch_bounds__(FT, 6) m2_step_read16_kernel(M2Args a) {
  extern __shared__ __align__(128) uint16_t dsm16[];
  uint16_t* tile = dsm16;                  // [2 heads][64 rows][128] bf16
  uint16_t* xr = dsm16 + 2 * FPB * FN;     // [2 heads][L + 1 slots][XST] bf16 x rows; slot L = current
  __shared__ float sc[FW * KW];            // c_s = B_s . C by ring slot; [L] = current
  __shared__ uint64_t bar;
  __shared__ int4 scur;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pb = blockIdx.x, hp = blockIdx.y, b = blockIdx.z;
  const int L = a.L, P = a.P, H = a.H, N2 = 2;
  const int h0 = 2 * hp, hh = warp >> 1, h = h0 + hh;  // this warp's head
  const int g = h0 >> a.hpg_log2;                      // both heads' group (heads per group >= 2)
  const int bg = b * a.G + g;
  const int p0 = pb * FPB;
  const int XL = L + 1;                                // x slots per head
  const int rw0 = 32 * (warp & 1);                     // the warp's first row (within the block)
  uint16_t* tw = tile + hh * FPB * FN;                 // this warp's head tile
  const uint16_t* xw = xr + hh * XL * XST;             // this warp's head x slots

  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    const uint32_t tbytes = FPB * FN * 2, xbytes = FPB * 2;
    mbar_arrive_expect_tx(&bar, N2 * (tbytes + XL * xbytes));
    for (int u = 0; u < N2; u++) {
      const size_t bhu = (size_t)b * H + h0 + u;
      bulk_load(tile + u * FPB * FN, a.ckpt_read + (bhu * P + p0) * FN, tbytes, &bar);
      for (int s = 0; s < L; s++) bulk_load(xr + (u * XL + s) * XST, a.rx + (bhu * L + s) * P + p0, xbytes, &bar);
      bulk_load(xr + (u * XL + L) * XST, a.x + bhu * P + p0, xbytes, &bar);
    }
  }
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * b);
  const size_t bh = (size_t)b * H + h;
  const float dts = lane < L ? a.rdt[bh * pad4(L) + lane] : 0.f;
  const float dtc = a.dt[bh], Ah = a.A[h], Dh = a.D[h];
  float zg[RG];  // gate z of row (lane & 7) of each group
#pragma unroll
  for (int j = 0; j < RG; j++) zg[j] = bf_to_f(a.z[bh * P + p0 + rw0 + 8 * j + (lane & 7)]);
  // the append's x and z rows: lane j < RG copies group j's 8 values of each
  const uint4 zap = ldg16(a.z + bh * P + p0 + rw0 + 8 * (lane & (RG - 1)));
  const uint4 xap = ldg16(a.x + bh * P + p0 + rw0 + 8 * (lane & (RG - 1)));
  const uint2 craw = *reinterpret_cast<const uint2*>(a.C + (size_t)bg * FN + lane * 4);
  const uint2 braw = *reinterpret_cast<const uint2*>(a.B + (size_t)bg * FN + lane * 4);
  const float4 cm = bf4_to_f4(craw);
  {  // c_s = B_s . C for slots s = warp + 4 i (s == L: the current record), shared by both heads
    const uint16_t* rBp = a.rB + (size_t)bg * L * FN + lane * 4;
    const float4 bc = bf4_to_f4(braw);
    float pk[KW];
#pragma unroll
    for (int i = 0; i < KW; i++) {
      const int s = warp + FW * i;
      pk[i] = s < L ? dot4(load_bf4(rBp + s * FN), cm) : (s == L ? dot4(bc, cm) : 0.f);
    }
    const float red = reduce_transpose<KW>(pk, lane);
    if ((lane & 3) == 0) sc[warp + FW * reduce8_row(lane)] = red;
  }
  const bool valid = cur.x >= 0 && cur.x < L && cur.y >= 0 && cur.y < L && cur.z == 0;
  const int nblocks = (H >> 1) * a.nPB;  // blocks of this sequence
  if (!valid) {  // uniform over the block; the last block of the sequence reports it
    if (threadIdx.x == 0) {
      const int ticket = cursor_ticket(a.cursors, b);
      mbar_wait(&bar, 0);  // the copies land before the block leaves
      finish_ar_cursor(a.cursors, b, cur, ticket, nblocks, L, a.status);
    }
    return;
  }
  const int start = cur.x, count = cur.y, m = count + 1;
  const bool flush = (m == L);
  // window of this warp's head, lane k = record k
  int sl = start + lane;
  sl = sl < L ? sl : sl - L;
  const float dtr = __shfl_sync(FULL, dts, sl);
  const float dtk = lane < count ? dtr : (lane == count ? dtc : 0.f);
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
  const float4 pc = scale4(Pm, cm);
  __syncthreads();  // the dot table
  int ticket = 0;
  if (threadIdx.x == 0) {  // every thread has read the cursor
    ticket = cursor_ticket(a.cursors, b);
    scur = cur;
  }
  const float coef = lane < m ? fmaf(wk, sc[lane < count ? sl : L], lane == count ? Dh : 0.f) : 0.f;
  const int xslot = lane < count ? sl : L;  // staged x slot of record `lane` (the current one past the window)
  // Append the current record now: its slot is outside the window
  if (!flush) {
    const int slot = start + count < L ? start + count : start + count - L;
    const size_t rrow = (bh * L + slot) * P + p0 + rw0;
    if (lane < RG) {
      *reinterpret_cast<uint4*>(a.rx + rrow + 8 * lane) = xap;
      *reinterpret_cast<uint4*>(a.rz + rrow + 8 * lane) = zap;
    }
    if ((warp & 1) == 0 && pb == 0 && lane == RG) a.rdt[bh * pad4(L) + slot] = dtc;
    if (warp == 0 && pb == 0 && (h0 & ((1 << a.hpg_log2) - 1)) == 0) {  // the group's first head
      const size_t brow = ((size_t)bg * L + slot) * FN + lane * 4;
      *reinterpret_cast<uint2*>(a.rB + brow) = braw;
      *reinterpret_cast<uint2*>(a.rC + brow) = craw;
    }
  }
  if (!__all_sync(FULL, mbar_wait(&bar, 0))) {
    if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
    mbar_wait(&bar, 0);
    if (threadIdx.x == 0) finish_ar_cursor(a.cursors, b, scur, ticket, nblocks, L, a.status);
    return;
  }
  const size_t ybase = bh * P + p0;
#pragma unroll
  for (int j = 0; j < RG; j++) {
    const int r0 = rw0 + 8 * j;  // the group's first row (within the block)
    float xl[8], tx[8];
    unpack8(*reinterpret_cast<const uint4*>(xw + xslot * XST + r0), xl);
#pragma unroll
    for (int rr = 0; rr < 8; rr++) tx[rr] = coef * xl[rr];  // coef = 0 off the window; x finite there
    float4 hv[8];
    if (!flush) {
#pragma unroll
      for (int rr = 0; rr < 8; rr++) hv[rr] = load_bf4(tw + (r0 + rr) * FN + lane * 4);
      gate_store<OUT_BF16>(a, ybase + r0, silu_fast(zg[j]), rows8(hv, pc, tx, lane), lane);
    } else {  // a flushing sequence reads and folds the fp32 rows, then writes fp32 and bf16 once
      const size_t off = (bh * P + p0 + r0) * FN + lane * 4;
#pragma unroll
      for (int rr = 0; rr < 8; rr++) hv[rr] = __ldcs(reinterpret_cast<const float4*>(a.ckpt + off + (size_t)rr * FN));
      gate_store<OUT_BF16>(a, ybase + r0, silu_fast(zg[j]), rows8(hv, pc, tx, lane), lane);
      fold8(a, hv, Pm, wk, xl, m, count, start, bg, off, lane);
    }
  }
  if (threadIdx.x == 0) finish_ar_cursor(a.cursors, b, scur, ticket, nblocks, L, a.status);
}

}  // namespace

bool m2_step_read16_applies(const M2Args& a) {
  return a.ckpt_read != nullptr && m2_step_fast_applies(a) && a.hpg_log2 >= 1 &&
         (size_t)2 * (FPB * FN + (a.L + 1) * XST) * 2 <= 48 * 1024 - 256;
}

cudaError_t m2_step_read16_launch(const M2Args& a, int out_bf16, cudaStream_t st) {
  const dim3 grid(a.nPB, a.H / 2, a.Bt);
  auto k = out_bf16 ? m2_step_read16_kernel<true> : m2_step_read16_kernel<false>;
  const int smem = 2 * (FPB * FN + (a.L + 1) * XST) * 2;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<grid, FT, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace rssm
