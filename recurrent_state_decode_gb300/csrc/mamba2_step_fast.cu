// ReplaySSM AR decode step for Mamba-2, shape-specialised fast path:
// dstate = 128 and headdim a multiple of 64 (the serving layers). Same
// algorithm as the generic kernel in mamba2_step.cu ("How ReplaySSM works":
// non-flush steps read the checkpoint and the window and store no state; the
// L-th step folds the window into the checkpoint and writes it once).
//
// One CTA of four warps per (sequence, head, 64-row block). Every global load
// the block needs is issued at launch, none of them waiting on the cursor, so a
// block's life is one memory round trip plus its arithmetic: thread 0 starts one
// bulk copy (TMA, non-tensor; never multicast) of the block's 64 checkpoint rows
// into shared memory (32 KiB fp32, or 16 KiB from the bf16 read copy), and every
// lane loads, for its warp's two 8-row groups, ring slot `lane` (its dt and x
// rows), the current record, the gate z, and the B rows of the ring slots whose
// B.C dots the warp forms (per-lane partials over the lane's column chunk, one
// transposed butterfly reduction; shared through shared memory). Six blocks --
// 192 KiB of checkpoint -- are in flight per SM. Once the cursor is known lane k
// takes record k from lane (start + k) mod L by a shuffle, one warp suffix scan
// gives w_k = dt_k exp(A sum_{j>k} dt_j) and P = exp(A sum dt), and per 8-row
// group each lane's partial (h0 . P C) plus its record's term (w_k c_k [+ D on
// the current record]) x_k[r] goes through one transposed 8-row reduction,
// yielding y[r] before the gate; the gate silu(z) and the store run one lane per
// row. On the L-th step the window is folded into the rows and written once,
// with the bf16 read copy (a block reading the bf16 copy takes its fp32 rows
// from global memory on that step); otherwise the record is appended to its
// ring slot. The last of a sequence's blocks to have read its cursor advances
// it (an arrival count in the high half of the cursor's flags word), so the
// step needs no second kernel.
#include <mutex>
#include <type_traits>

#include "fast_rows.cuh"
#include "kernels.h"

namespace rssm {

namespace {

using namespace fastrows;

constexpr int KW = 8;  // 4 warps x 8 >= L + 1 dots for L <= 31
// With L <= 16 four slots per warp cover the ring, and the current record's
// dot is one warp sum instead: half the dot work and a 4-wide reduction.
constexpr int KW_SHORT = 4;

// Emulated read of 8 rows (a non-flush step of the emulated instantiation):
// every element x becomes Q(x * inv) * s for its row's (or its tile's)
// scale, Q the format's rounding; err and nrm gather (read - x)^2 and x^2.
// With a row scale the rows' maxima come from one transposed max reduction,
// lane row_src(rr) computing row rr's quotients. Every lane must call this.
__device__ __forceinline__ void emu_read8(float4 (&hv)[8], const M2Args& a, const EmuQ& fq, float tinv, float ts,
                                          int lane, float& err, float& nrm) {
  float inv[8], sc[8];
  const bool scaled = a.emu_scale != RSSM_EMU_SCALE_NONE;
  if (a.emu_scale == RSSM_EMU_SCALE_ROW) {
    float m[8];
#pragma unroll
    for (int rr = 0; rr < 8; rr++) m[rr] = abs_max4(hv[rr]);
    const float mm = max_transpose<8>(m, lane);  // the max of row reduce8_row(lane)
    const float qmax = emu_qmax(a.emu_fmt);
    const float my_inv = mm > 0.f ? qmax / mm : 0.f, my_s = mm / qmax;
#pragma unroll
    for (int rr = 0; rr < 8; rr++) {
      inv[rr] = __shfl_sync(FULL, my_inv, row_src(rr));
      sc[rr] = __shfl_sync(FULL, my_s, row_src(rr));
    }
  } else {
#pragma unroll
    for (int rr = 0; rr < 8; rr++) {
      inv[rr] = tinv;
      sc[rr] = ts;
    }
  }
#pragma unroll
  for (int rr = 0; rr < 8; rr++) {
    const float4 x = hv[rr];
    const float4 t = scaled ? make_float4(__fmul_rn(x.x, inv[rr]), __fmul_rn(x.y, inv[rr]), __fmul_rn(x.z, inv[rr]),
                                          __fmul_rn(x.w, inv[rr]))
                            : x;
    const float4 q = emu_quantise4(t, fq);
    const float4 r = scaled ? make_float4(__fmul_rn(q.x, sc[rr]), __fmul_rn(q.y, sc[rr]), __fmul_rn(q.z, sc[rr]),
                                          __fmul_rn(q.w, sc[rr]))
                            : q;
    const float d0 = r.x - x.x, d1 = r.y - x.y, d2 = r.z - x.z, d3 = r.w - x.w;
    err = fmaf(d0, d0, err);
    err = fmaf(d1, d1, err);
    err = fmaf(d2, d2, err);
    err = fmaf(d3, d3, err);
    nrm = fmaf(x.x, x.x, nrm);
    nrm = fmaf(x.y, x.y, nrm);
    nrm = fmaf(x.z, x.z, nrm);
    nrm = fmaf(x.w, x.w, nrm);
    hv[rr] = r;
  }
}

// RD16: the block reads the 16-bit or fp8 read copy (16 KiB tiles, seven blocks
// per SM: at eight the 64-register cap spilled, and seven measured 2% faster).
// SLOTS: batch rows name their state rows through a slot table.
// EMU: non-flush steps read the fp32 tile through an emulated precision and
// each block writes its (error, norm) sums to a.emu_part (fp32 tiles, no slots).
// KWT: dot slots per warp (KW, or KW_SHORT when L <= 16).
template <bool OUT_BF16, bool RD16, bool SLOTS, bool EMU = false, int KWT = KW>
__global__ void __launch_bounds__(FT, RD16 ? 7 : 6) m2_step_fast_kernel(M2Args a) {
  // the block's rows: a static fp32 tile, or the dynamic 16 KiB of a bf16 one
  __shared__ __align__(128) float tile_s[RD16 ? 4 : FPB * FN];
  extern __shared__ __align__(128) float tile_d[];
  float* const tile = RD16 ? tile_d : tile_s;
  __shared__ float sc[FW * KW];                    // c_s = B_s . C by ring slot; [L] = current
  __shared__ uint64_t bar;
  __shared__ int4 scur;  // the cursor as read, for the sequence's last block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int L = a.L, P = a.P, H = a.H;
  const int g = h >> a.hpg_log2;  // H / G heads per group, a power of two on this path
  // the batch row's state slot; a padding row (or a reported bad slot) leaves at once
  const int sb = SLOTS ? state_slot(a.slots, a.Sn, b, a.status, pb == 0 && h == 0 && threadIdx.x == 0) : b;
  if (SLOTS && sb < 0) return;
  const int bh = b * H + h, bg = b * a.G + g;    // the record's rows (x, z, B, C, dt, y)
  const int sh = sb * H + h, sg = sb * a.G + g;  // the state's rows (checkpoint, ring, cursor)
  const int p0 = pb * FPB;
  // a bf16 read copy is present (known at compile time only in the read-copy instantiation; the
  // fp32 one keeps the run-time test, which measured faster there)
  const bool copy = RD16 || a.ckpt_read != nullptr;
  const size_t tbase = ((size_t)sh * P + p0) * FN;  // element offset of the block's row 0

  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (copy && a.read_f8) {  // e4m3 rows, then their 64 scales after them
      const uint8_t* q = reinterpret_cast<const uint8_t*>(a.ckpt_read);
      const float* scales = reinterpret_cast<const float*>(q + (size_t)a.Sn * H * P * FN);
      mbar_arrive_expect_tx(&bar, FPB * FN + FPB * 4);
      bulk_load(tile, q + tbase, FPB * FN, &bar);
      bulk_load(reinterpret_cast<uint8_t*>(tile) + FPB * FN, scales + tbase / FN, FPB * 4, &bar);
    } else {
      const uint32_t bytes = FPB * FN * (copy ? 2 : 4);
      mbar_arrive_expect_tx(&bar, bytes);
      bulk_load(tile, copy ? (const void*)(a.ckpt_read + tbase) : (const void*)(a.ckpt + tbase), bytes, &bar);
    }
  }
  // everything else, at launch: cursor, window records, current record, gate
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * sb);
  const int rl0 = warp * 8, rl1 = HALF + warp * 8;  // the warp's two row groups (within the block)
  const int rA = p0 + rl0, rB2 = p0 + rl1;          // ... within the head
  const size_t xrow = (size_t)bh * P;
  const float dts = lane < L ? a.rdt[(size_t)sh * pad4(L) + lane] : 0.f;
  const float dtc = a.dt[bh], Ah = a.A[h], Dh = a.D[h];
  uint4 xsA = make_uint4(0, 0, 0, 0), xsB = xsA;
  if (lane < L) {
    const uint16_t* xp = a.rx + ((size_t)sh * L + lane) * P;
    xsA = ldg16(xp + rA);
    xsB = ldg16(xp + rB2);
  }
  const uint4 xcA = ldg16(a.x + xrow + rA), xcB = ldg16(a.x + xrow + rB2);
  const float zA = bf_to_f(a.z[xrow + rA + (lane & 7)]), zB = bf_to_f(a.z[xrow + rB2 + (lane & 7)]);
  const uint4 zap = ldg16(a.z + xrow + ((lane & 1) ? rB2 : rA));  // the append's z rows (lanes 2, 3)
  const uint2 craw = *reinterpret_cast<const uint2*>(a.C + (size_t)bg * FN + lane * 4);
  const uint2 braw = *reinterpret_cast<const uint2*>(a.B + (size_t)bg * FN + lane * 4);
  const float4 cm = bf4_to_f4(craw);
  float cdot = 0.f;  // B . C of the current record (with KW_SHORT slots per warp)
  {  // c_s = B_s . C for slots s = warp + 4 i (s == L: the current record, with KW slots per warp)
    const uint16_t* rBp = a.rB + (size_t)sg * L * FN + lane * 4;
    const float4 bc = bf4_to_f4(braw);
    float pk[KWT];
#pragma unroll
    for (int i = 0; i < KWT; i++) {
      const int s = warp + FW * i;
      pk[i] = s < L ? dot4(load_bf4(rBp + s * FN), cm) : (KWT == KW && s == L ? dot4(bc, cm) : 0.f);
    }
    const float red = reduce_transpose<KWT>(pk, lane);
    if (KWT == KW) {
      if ((lane & 3) == 0) sc[warp + FW * reduce8_row(lane)] = red;
    } else {  // 4-wide: lane l holds slot index 2 (l >> 4 & 1) + (l >> 3 & 1)
      if ((lane & 7) == 0) sc[warp + FW * (((lane >> 4) & 1) * 2 + ((lane >> 3) & 1))] = red;
      cdot = warp_sum(dot4(bc, cm));
    }
  }
  const bool valid = cur.x >= 0 && cur.x < L && cur.y >= 0 && cur.y < L && cur.z == 0;
  const int nblocks = a.H * a.nPB;  // blocks of this sequence
  // this block's entry of the emulated read's error sums (every path writes it)
  float2* const emu_slot = EMU ? a.emu_part + ((size_t)bh * a.nPB + pb) : nullptr;
  if (EMU && !valid && threadIdx.x == 0) *emu_slot = make_float2(0.f, 0.f);
  if (!valid) {  // uniform over the block; the last block of the sequence reports it
    if (threadIdx.x == 0) {
      const int ticket = cursor_ticket(a.cursors, sb);
      mbar_wait(&bar, 0);  // the copy lands before the block leaves
      finish_ar_cursor(a.cursors, sb, cur, ticket, nblocks, L, a.status);
    }
    return;
  }
  const int start = cur.x, count = cur.y, m = count + 1;
  const bool flush = (m == L);
  // window, lane k = record k
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
  const uint4 xrA = shfl_u4(xsA, sl), xrB = shfl_u4(xsB, sl);
  __syncthreads();
  int ticket = 0;
  if (threadIdx.x == 0) {  // every thread has read the cursor
    ticket = cursor_ticket(a.cursors, sb);
    scur = cur;
  }
  const float cs = lane < count ? sc[sl] : (KWT == KW ? sc[L] : cdot);
  const float coef = lane < m ? fmaf(wk, cs, lane == count ? Dh : 0.f) : 0.f;
  // the gates do not need the checkpoint rows: computed before waiting for them
  const uint4 xq[2] = {lane < count ? xrA : xcA, lane < count ? xrB : xcB};  // lane k: x_k, both groups
  const float gA = silu_fast(zA), gB = silu_fast(zB);
  // Append the current record now: its slot is outside the window (no block
  // reads it for a result; this block's own loads of it are consumed above).
  if (!flush) {  // x, z rows of this warp's groups; dt, B, C once
    const int slot = start + count < L ? start + count : start + count - L;
    const size_t rrow = ((size_t)sh * L + slot) * P;
    if (lane == 0) *reinterpret_cast<uint4*>(a.rx + rrow + rA) = xcA;
    if (lane == 1) *reinterpret_cast<uint4*>(a.rx + rrow + rB2) = xcB;
    if (lane == 2 || lane == 3) *reinterpret_cast<uint4*>(a.rz + rrow + (lane == 3 ? rB2 : rA)) = zap;
    if (warp == 0 && pb == 0) {
      if (lane == 4) a.rdt[(size_t)sh * pad4(L) + slot] = dtc;
      if (h == (g << a.hpg_log2)) {  // the group's first head
        const size_t brow = ((size_t)sg * L + slot) * FN + lane * 4;
        *reinterpret_cast<uint2*>(a.rB + brow) = braw;
        *reinterpret_cast<uint2*>(a.rC + brow) = craw;
      }
    }
  }
  // (the emulated instantiation makes the outcome block-uniform: it meets a block barrier after the wait)
  if (!(EMU ? __syncthreads_and(mbar_wait(&bar, 0)) : __all_sync(FULL, mbar_wait(&bar, 0)))) {
    if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
    if (EMU && threadIdx.x == 0) *emu_slot = make_float2(0.f, 0.f);
    mbar_wait(&bar, 0);
    if (threadIdx.x == 0) finish_ar_cursor(a.cursors, sb, scur, ticket, nblocks, L, a.status);
    return;
  }
  // Emulated read with one scale per 64-row tile: the maxima of the warps'
  // rows meet in shared memory (the dot table's first entries, consumed by now).
  float emu_tinv = 1.f, emu_ts = 1.f, emu_err = 0.f, emu_nrm = 0.f;
  EmuQ emu_q{};
  if (EMU) emu_q = emu_params(a.emu_fmt);
  if (EMU && !flush && a.emu_scale == RSSM_EMU_SCALE_TILE64) {
    float m = 0.f;
#pragma unroll
    for (int rr = 0; rr < 8; rr++) {
      m = fmaxf(m, abs_max4(reinterpret_cast<const float4*>(tile + (rl0 + rr) * FN)[lane]));
      m = fmaxf(m, abs_max4(reinterpret_cast<const float4*>(tile + (rl1 + rr) * FN)[lane]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
    if (lane == 0) sc[warp] = m;
    __syncthreads();
    m = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
    const float qmax = emu_qmax(a.emu_fmt);
    emu_tinv = m > 0.f ? qmax / m : 0.f;
    emu_ts = m / qmax;
  }
  // A block that reads the bf16 copy folds from the fp32 rows in global memory.
  const bool from_tile = !(copy && flush);
#pragma unroll
  for (int half = 0; half < 2; half++) {
    const int rl = half ? rl1 : rl0;
    float4 hv[8];
    if (!from_tile) {
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
        hv[rr] = __ldcs(reinterpret_cast<const float4*>(a.ckpt + tbase + (size_t)(rl + rr) * FN) + lane);
    } else if (copy) {
      if (a.read_f8) {  // e4m3 values times their row's scale
        const uint8_t* t8 = reinterpret_cast<const uint8_t*>(tile) + lane * 4;
        const float* ts = reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(tile) + FPB * FN);
#pragma unroll
        for (int rr = 0; rr < 8; rr++) hv[rr] = scale4(ts[rl + rr], load_f8x4(t8 + (rl + rr) * FN));
      } else {
        const uint16_t* t16 = reinterpret_cast<const uint16_t*>(tile) + lane * 4;
#pragma unroll
        for (int rr = 0; rr < 8; rr++) hv[rr] = load_rc4(t16 + (rl + rr) * FN, a.read_f16);
      }
    } else {
#pragma unroll
      for (int rr = 0; rr < 8; rr++) hv[rr] = reinterpret_cast<const float4*>(tile + (rl + rr) * FN)[lane];
      if (EMU && !flush) emu_read8(hv, a, emu_q, emu_tinv, emu_ts, lane, emu_err, emu_nrm);
    }
    float xl[8], tx[8];
    unpack8(xq[half], xl);
#pragma unroll
    for (int rr = 0; rr < 8; rr++) tx[rr] = coef * xl[rr];  // coef = 0 off the window; x finite there
    gate_store<OUT_BF16>(a, xrow + p0 + rl, half ? gB : gA, rows8(hv, pc, tx, lane), lane);
    if (flush) {
      fold8(a, hv, Pm, wk, xl, m, count, start, sg, bg, tbase + (size_t)rl * FN + lane * 4, lane);
    }
  }

  if (EMU) {  // the block's sums, warps 0..3 added in order (the outcome of the wait is block-uniform here);
             // entries 16.. of the dot table, apart from the tile maxima's 0..3
    const float e = warp_sum(emu_err), n = warp_sum(emu_nrm);
    float* const red = sc + 16;
    if (lane == 0) red[warp] = e, red[FW + warp] = n;
    __syncthreads();
    if (threadIdx.x == 0)
      *emu_slot = make_float2(((red[0] + red[1]) + red[2]) + red[3], ((red[FW] + red[FW + 1]) + red[FW + 2]) + red[FW + 3]);
  }
  if (threadIdx.x == 0) finish_ar_cursor(a.cursors, sb, scur, ticket, nblocks, L, a.status);
}

// The emulated step's error sums, added in a fixed order in two stages. A
// single block of the whole reduction spent most of its time in fp64 adds on
// one SM (this GPU's fp64 rate is low); spread over one block per 256 pairs
// the adds take a few microseconds.
constexpr int EMU_C = 256;    // pairs per first-stage block (its threads)
constexpr int EMU_RT = 1024;  // threads of the second stage

// (a, b) summed over a warp by a fixed butterfly; every lane ends with the total.
__device__ __forceinline__ void warp_sum2(double& a, double& b) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(FULL, a, o);
    b += __shfl_xor_sync(FULL, b, o);
  }
}

// Stage 1: block j adds pairs [256 j, 256 j + 256) in fp64 (a butterfly per
// warp, then the eight warps in order) and writes the total over the chunk's
// first two pairs (one double2, which needs 16 bytes: a chunk of one pair is
// left as it is and read as a pair by stage 2).
__global__ void __launch_bounds__(EMU_C) emu_reduce1_kernel(float2* part, size_t n) {
  __shared__ double2 w[EMU_C / 32];
  const size_t base = (size_t)blockIdx.x * EMU_C, i = base + threadIdx.x;
  const float2 v = i < n ? part[i] : make_float2(0.f, 0.f);
  double e = v.x, q = v.y;
  warp_sum2(e, q);
  if ((threadIdx.x & 31) == 0) w[threadIdx.x >> 5] = make_double2(e, q);
  __syncthreads();  // every pair of the chunk is read before its first two are overwritten
  if (threadIdx.x == 0 && n - base >= 2) {
    double2 t = w[0];
#pragma unroll
    for (int k = 1; k < EMU_C / 32; k++) t.x += w[k].x, t.y += w[k].y;
    *reinterpret_cast<double2*>(part + base) = t;
  }
}

// Stage 2: one block adds the chunks' totals (thread t chunks t, t + 1024, ...
// in order, then a tree over the block) into err[0..1].
__global__ void __launch_bounds__(EMU_RT) emu_reduce2_kernel(const float2* __restrict__ part, size_t n, double* err) {
  __shared__ double se[EMU_RT], sn[EMU_RT];
  const size_t chunks = (n + EMU_C - 1) / EMU_C;
  double e = 0.0, q = 0.0;
  for (size_t j = threadIdx.x; j < chunks; j += EMU_RT) {
    const size_t base = j * EMU_C;
    if (n - base >= 2) {
      const double2 t = *reinterpret_cast<const double2*>(part + base);
      e += t.x;
      q += t.y;
    } else {
      e += part[base].x;
      q += part[base].y;
    }
  }
  se[threadIdx.x] = e;
  sn[threadIdx.x] = q;
  __syncthreads();
  for (int o = EMU_RT / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      se[threadIdx.x] += se[threadIdx.x + o];
      sn[threadIdx.x] += sn[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    err[0] = se[0];
    err[1] = sn[0];
  }
}

}  // namespace

bool m2_step_fast_applies(const M2Args& a) {
  return a.N == FN && a.P % FPB == 0 && a.PB == FPB && a.L <= FW * KW - 1 && a.H * a.nPB < (1 << 15) &&
         a.hpg_log2 >= 0;
}

cudaError_t m2_step_fast_launch(const M2Args& a, int out_bf16, cudaStream_t st) {
  const dim3 grid(a.nPB, a.H, a.Bt);
  const bool rd16 = a.ckpt_read != nullptr, short_window = a.L <= FW * KW_SHORT;
  auto pick = [&](auto slots, auto kwt) {
    constexpr bool S = decltype(slots)::value;
    constexpr int W = decltype(kwt)::value;
    return rd16 ? (out_bf16 ? m2_step_fast_kernel<true, true, S, false, W> : m2_step_fast_kernel<false, true, S, false, W>)
                : (out_bf16 ? m2_step_fast_kernel<true, false, S, false, W> : m2_step_fast_kernel<false, false, S, false, W>);
  };
  using KS = std::integral_constant<int, KW_SHORT>;
  using KL = std::integral_constant<int, KW>;
  auto k = a.slots ? (short_window ? pick(std::true_type{}, KS{}) : pick(std::true_type{}, KL{}))
                   : (short_window ? pick(std::false_type{}, KS{}) : pick(std::false_type{}, KL{}));
  const int smem = rd16 ? FPB * FN * 2 : 0;
  // six 32 KiB (seven 16 KiB) tiles per SM need the largest shared-memory split of the unified L1
  cudaError_t e = prepare(k, smem, true);
  if (e != cudaSuccess) return e;
  k<<<grid, FT, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t m2_step_emulated_launch(const M2Args& a, int out_bf16, double* err, cudaStream_t st) {
  if (a.Bt == 0) return cudaSuccess;
  const dim3 grid(a.nPB, a.H, a.Bt);
  const bool short_window = a.L <= FW * KW_SHORT;
  auto k = out_bf16 ? (short_window ? m2_step_fast_kernel<true, false, false, true, KW_SHORT>
                                    : m2_step_fast_kernel<true, false, false, true, KW>)
                    : (short_window ? m2_step_fast_kernel<false, false, false, true, KW_SHORT>
                                    : m2_step_fast_kernel<false, false, false, true, KW>);
  cudaError_t e = prepare(k, 0, true);
  if (e != cudaSuccess) return e;
  k<<<grid, FT, 0, st>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const size_t n = m2_emulated_partials(a);
  emu_reduce1_kernel<<<(unsigned)((n + EMU_C - 1) / EMU_C), EMU_C, 0, st>>>(a.emu_part, n);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  emu_reduce2_kernel<<<1, EMU_RT, 0, st>>>(a.emu_part, n, err);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- the no-allocation variant's scratch

// The emulated step's per-warp error sums for callers that cannot hand the
// library a workspace: a static device array, present on every GPU that
// loads the library until the process exits.
static __device__ __align__(256) float2 g_emu_scratch[M2_NOALLOC_PARTIALS];

// Device address of g_emu_scratch on the current device. In host code the
// array's name stands for a host-side shadow, not device memory, so the
// address is looked up once per device with that device current, and kept.
static cudaError_t emu_scratch_address(float2** out) {
  static std::mutex mu;
  static float2* addr[RSSM_NOALLOC_MAX_DEVICES] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= RSSM_NOALLOC_MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_emu_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float2*>(p);
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t m2_step_emulated_noalloc_launch(M2Args a, int out_bf16, double* err, cudaStream_t st) {
  if (m2_emulated_partials(a) > (size_t)M2_NOALLOC_PARTIALS) return cudaErrorInvalidValue;  // checked by the caller
  cudaError_t e = emu_scratch_address(&a.emu_part);
  if (e != cudaSuccess) return e;
  return m2_step_emulated_launch(a, out_bf16, err, st);
}

}  // namespace rssm
