// Speculative verify for Mamba-2, shape-specialised fast path: dstate 128,
// headdim a multiple of 64, at most 4 new records and L + K <= 32 ("How
// ReplaySSM works": drafts go into the buffer instead of a state snapshot and
// are verified output-only; "ReplaySSM" repository, introduction: rollback by
// moving a pointer). Same results as the persistent verify in
// mamba2_verify.cu, built like the AR step's fast path.
//
// One CTA of four warps per (sequence, head, 64-row block); warp w owns rows
// 8w..8w+7 and 32+8w..32+8w+7. Everything is requested at launch, none of it
// waiting on the cursor: thread 0 starts one bulk copy (TMA, non-tensor, never
// multicast) of the block's checkpoint rows into shared memory; lane s loads
// ring slot s (dt, x rows), lane j new record j (dt, x rows), lane 8i + r the
// gate z of new record i at row r, and every lane its column chunk of the new
// records' C. Records are indexed k in [0, count + K): k < count the committed
// window (ring slot (start + k) mod L), then the K new ones. Entry e of the
// B.C table is ring slot e (e < L) or new record e - L; the table [32 x 128] .
// [128 x 4] is a tensor-core product (m16n8k8 tf32, the bf16 inputs exact),
// warp w taking entries 16 (w & 1) .. + 15 over column half w >> 1, and the
// readers add the halves. Warp w then builds row w of the coefficient table.
//
// Once the cursor is known lane k takes record k by a shuffle and one
// inclusive warp scan gives S_k = A sum_{j<=k} dt_j. If count + K > L the
// committed window is folded first, h' = e^{S_{count-1}} h0 + sum_{k<count}
// dt_k e^{S_{count-1}-S_k} x_k B_k^T, written once (with the read copy),
// and output i covers records [count, count+i]; otherwise h' = h0 and output i
// covers [0, count+i]. Output i: y_i[r] = (e^{S_last - S_first-1} (h' . C_i)[r]
// + sum_k dt_k e^{S_last - S_k} (B_k . C_i) x_k[r] + D x_last[r]) silu(z_i[r]),
// last = count + i; h0 . [C_0..C_3] is an m16n8k8 tf32 product per warp (the
// fp32 state split in two tf32 parts on two independent accumulator chains, a
// 16-bit read copy exact in tf32, an fp8 one scaled by its row scales after the
// product), and so is the window term [x_k] . [coefficients] (x bf16, the
// coefficients in two tf32 parts). The fold of an fp32 checkpoint is a
// tensor-core product too; with a read copy it runs in the row layout, from
// the fp32 rows in global memory.
// The new records' x and z rows go to the ring here (these rows are read by
// this block alone); their B, C and dt rows, which other blocks read, are
// appended by the last of the sequence's blocks to finish (an arrival count in
// the high half of the cursor's flags word), which also marks the cursor
// pending: a verify is one kernel.
#include "fast_rows.cuh"
#include "fold_mma.cuh"
#include "kernels.h"

namespace rssm {

namespace {

using namespace fastrows;

constexpr int KMAX = 4;  // new records per verify on this path
constexpr int EW = 8;    // B.C entries per warp: 4 warps x 8 = 32 >= L + K
constexpr int XS = FPB + 8;  // x table row stride (bf16): a record's rows start 16 bytes apart in bank terms

// Epilogue of a verify, run by all threads of the sequence's last block: on a
// cursor with 0 <= start < L, 0 <= count <= L and pending == 0, append the K
// new records' B, C (group rows) and dt to the ring and set pending = K, flags
// = folded; otherwise report as the cursor checks do and leave it (clearing
// the arrival count in the high half of the flags word).
// Batch row b's records go to the ring rows of its state slot sb.
__device__ __forceinline__ void verify_epilogue(const M2Args& a, int b, int sb, int4 cur, int flags) {
  const int L = a.L, H = a.H, G = a.G, K = a.K, tid = threadIdx.x;
  int4 c = cur;
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
  constexpr int NV = FN / 8;  // 16-byte pieces per group row
  constexpr int U = 4;        // pieces in flight per thread: all loads before the stores
  const int pieces = K * G * NV;
  for (int q0 = tid; q0 < pieces; q0 += U * FT) {
    uint4 bv[U], cv[U];
    size_t dst[U];
#pragma unroll
    for (int u = 0; u < U; u++) {
      const int q = q0 + u * FT;
      if (q < pieces) {
        const int i = q / (G * NV), r = q - i * G * NV, g = r / NV, v = r - g * NV;
        const int slot = wrap(wrap(c.x + c.y + i, L), L);
        const size_t src = (((size_t)b * K + i) * G + g) * FN + v * 8;
        dst[u] = (((size_t)sb * G + g) * L + slot) * FN + v * 8;
        bv[u] = ldg16(a.B + src);
        cv[u] = ldg16(a.C + src);
      }
    }
#pragma unroll
    for (int u = 0; u < U; u++) {
      if (q0 + u * FT < pieces) {
        *reinterpret_cast<uint4*>(a.rB + dst[u]) = bv[u];
        *reinterpret_cast<uint4*>(a.rC + dst[u]) = cv[u];
      }
    }
  }
  for (int q = tid; q < K * H; q += FT) {
    const int i = q / H, h = q - i * H;
    int slot = c.x + c.y + i;
    slot = slot < L ? slot : slot - L;
    slot = slot < L ? slot : slot - L;
    a.rdt[((size_t)sb * H + h) * pad4(L) + slot] = a.dt[((size_t)b * K + i) * H + h];
  }
  if (tid == 0) {
    c.z = K;
    c.w = (c.y + K > L) ? 1 : 0;
    *reinterpret_cast<int4*>(a.cursors + 4 * (size_t)sb) = c;
  }
}

// Rows rA, rB of the state at columns col..col+3 as the kernel reads them: the
// fp32 tile, the bf16 read copy in the tile, or (a folding block of the read
// copy) the fp32 rows in global memory.
__device__ __forceinline__ void state_rows(const float* tile, const float* gstate, bool bf16, bool f16, bool f8, int rA,
                                           int rB, int col, float4& r0, float4& r1) {
  if (gstate) {
    r0 = __ldcs(reinterpret_cast<const float4*>(gstate + (size_t)rA * FN + col));
    r1 = __ldcs(reinterpret_cast<const float4*>(gstate + (size_t)rB * FN + col));
  } else if (bf16 && f8) {  // e4m3 values, unscaled (exact in tf32): the caller scales the rows
    const uint8_t* t8 = reinterpret_cast<const uint8_t*>(tile);
    r0 = load_f8x4(t8 + rA * FN + col);
    r1 = load_f8x4(t8 + rB * FN + col);
  } else if (bf16) {
    const uint16_t* t16 = reinterpret_cast<const uint16_t*>(tile);
    r0 = load_rc4(t16 + rA * FN + col, f16);
    r1 = load_rc4(t16 + rB * FN + col, f16);
  } else {
    r0 = *reinterpret_cast<const float4*>(tile + rA * FN + col);
    r1 = *reinterpret_cast<const float4*>(tile + rB * FN + col);
  }
}

// SLOTS: batch rows name their state rows through a slot table.
template <bool OUT_BF16, bool SLOTS>
__global__ void __launch_bounds__(FT, 6) m2_verify_fast_kernel(M2Args a) {
  extern __shared__ __align__(128) float dsm[];
  float* tile = dsm;                                                  // the block's rows (fp32, or bf16)
  uint16_t* xs = reinterpret_cast<uint16_t*>(dsm + FPB * FN);         // x of record k, row r: xs[k * XS + r]
  __shared__ float tbl[2][KMAX][FW * EW];                             // B_e . C_i over column half [0] / [1]
  __shared__ float cf[KMAX][33];                                      // window coefficient of record k, output i
  __shared__ uint64_t bar;
  __shared__ int last_flags;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int L = a.L, P = a.P, H = a.H, G = a.G, K = a.K;
  const int g = h >> a.hpg_log2;  // H / G heads per group, a power of two on this path
  // the batch row's state slot; a padding row (or a reported bad slot) leaves at once
  const int sb = SLOTS ? state_slot(a.slots, a.Sn, b, a.status, pb == 0 && h == 0 && threadIdx.x == 0) : b;
  if (SLOTS && sb < 0) return;
  const int sh = sb * H + h, sg = sb * G + g;  // the state's rows (checkpoint, ring, cursor)
  const int p0 = pb * FPB;
  const bool copy = a.ckpt_read != nullptr;
  const size_t tbase = ((size_t)sh * P + p0) * FN;

  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    const uint32_t bytes = FPB * FN * (copy ? (a.read_f8 ? 1 : 2) : 4);
    mbar_arrive_expect_tx(&bar, bytes);
    const void* src = !copy ? (const void*)(a.ckpt + tbase)
                            : (a.read_f8 ? (const void*)(reinterpret_cast<const uint8_t*>(a.ckpt_read) + tbase)
                                         : (const void*)(a.ckpt_read + tbase));
    bulk_load(tile, src, bytes, &bar);
  }
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * sb);
  const int rl0 = warp * 8, rl1 = HALF + warp * 8;
  const int qg = lane >> 2, qt = lane & 3;  // tensor-core fragment coordinates
  const int rA = rl0 + qg, rB = rl1 + qg;   // rows of this lane's accumulator fragments (within the block)
  // ring slot `lane`
  const float dts = lane < L ? a.rdt[(size_t)sh * pad4(L) + lane] : 0.f;
  uint4 xsA = make_uint4(0, 0, 0, 0), xsB = xsA, xnA = xsA, xnB = xsA;
  if (lane < L) {
    const uint16_t* xp = a.rx + ((size_t)sh * L + lane) * P + p0;
    xsA = ldg16(xp + rl0);
    xsB = ldg16(xp + rl1);
  }
  // new record `lane`
  const size_t nrow = ((size_t)b * K + lane) * H + h;
  float dtn = 0.f;
  if (lane < K) {
    dtn = a.dt[nrow];
    xnA = ldg16(a.x + nrow * P + p0 + rl0);
    xnB = ldg16(a.x + nrow * P + p0 + rl1);
  }
  // gate z of outputs n = 2 qt, 2 qt + 1 at rows rA, rB (lanes qt < 2); the z append rows
  float zg[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int u = 0; u < 2; u++) {
    const int n = 2 * qt + u;
    if (n < K) {
      const size_t zrow = (((size_t)b * K + n) * H + h) * P + p0;
      zg[u][0] = bf_to_f(a.z[zrow + rA]);
      zg[u][1] = bf_to_f(a.z[zrow + rB]);
    }
  }
  const int gi = lane >> 3, gr = lane & 7;
  uint16_t zbA = 0, zbB = 0;
  if (gi < K) {
    const size_t zrow = (((size_t)b * K + gi) * H + h) * P + p0;
    zbA = a.z[zrow + rl0 + gr];
    zbB = a.z[zrow + rl1 + gr];
  }
  const float Ah = a.A[h], Dh = a.D[h];
  // the lane's B-fragment source: C_n, n = qg (zero for n >= K)
  const uint16_t* cvec = qg < K ? a.C + (((size_t)b * K + qg) * G + g) * FN : nullptr;
  // dot table tbl[i][e] = B_e . C_i for entries e < 32 (ring slot e if e < L, new
  // record e - L if e < L + K, else 0): [32 x 128] . [128 x 8] on the tensor
  // cores, warp w taking entries 16 (w & 1) .. 16 (w & 1) + 15 over the column
  // half w >> 1 (bf16 inputs are exact in tf32); the reader adds the halves
  {
    const int e0 = 16 * (warp & 1) + qg, e1 = e0 + 8, ch = warp >> 1;
    auto row_of = [&](int e) -> const uint16_t* {
      if (e < L) return a.rB + ((size_t)sg * L + e) * FN;
      if (e < L + K) return a.B + (((size_t)b * K + (e - L)) * G + g) * FN;
      return nullptr;
    };
    const uint16_t* s0 = row_of(e0);
    const uint16_t* s1 = row_of(e1);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int jb = ch * (FN / 32); jb < (ch + 1) * (FN / 32); jb++) {
      const int col = 16 * jb + 4 * qt;
      const float4 r0 = s0 ? load_bf4(s0 + col) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 r1 = s1 ? load_bf4(s1 + col) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 bv = cvec ? load_bf4(cvec + col) : make_float4(0.f, 0.f, 0.f, 0.f);
      mma_tf32_1688(acc, __float_as_uint(r0.x), __float_as_uint(r1.x), __float_as_uint(r0.y), __float_as_uint(r1.y),
                    __float_as_uint(bv.x), __float_as_uint(bv.y));
      mma_tf32_1688(acc, __float_as_uint(r0.z), __float_as_uint(r1.z), __float_as_uint(r0.w), __float_as_uint(r1.w),
                    __float_as_uint(bv.z), __float_as_uint(bv.w));
    }
    if (qt < 2) {  // columns 2 qt, 2 qt + 1 are outputs 0..3
      tbl[ch][2 * qt][e0] = acc[0];
      tbl[ch][2 * qt + 1][e0] = acc[1];
      tbl[ch][2 * qt][e1] = acc[2];
      tbl[ch][2 * qt + 1][e1] = acc[3];
    }
  }
  // An invalid cursor (reported by the epilogue below) runs as an empty window
  // with every store masked.
  const bool valid = cur.x >= 0 && cur.x < L && cur.y >= 0 && cur.y <= L && cur.z == 0;
  const int start = valid ? cur.x : 0, count = valid ? cur.y : 0, total = count + K;
  const bool fold = total > L;
  // record k on lane k: committed (ring slot sl) or new (record jn)
  int sl = start + lane;
  sl = sl < L ? sl : sl - L;
  const int jn = (lane - count) & 31;
  const float dtr = __shfl_sync(FULL, dts, sl), dtw = __shfl_sync(FULL, dtn, jn);
  const float dtk = lane < count ? dtr : (lane < total ? dtw : 0.f);
  float S = dtk * Ah;  // inclusive scan: S_k = A sum_{j<=k} dt_j
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float v = __shfl_up_sync(FULL, S, o);
    if (lane >= o) S += v;
  }
  const float Sf = __shfl_sync(FULL, S, (count - 1) & 31);
  const float Pf = expf(Sf);                                // fold: e^{S_{count-1}}
  const float wf = lane < count ? dtk * expf(Sf - S) : 0.f;  // fold weights
  const int ek = lane < count ? sl : (lane < total ? L + jn : 0);
  const uint4 xar = shfl_u4(xsA, sl), xbr = shfl_u4(xsB, sl), xan = shfl_u4(xnA, jn), xbn = shfl_u4(xnB, jn);
  const uint4 xq[2] = {lane < count ? xar : xan, lane < count ? xbr : xbn};
  if (lane < total) {  // this warp's rows of every record's x, in record order
    *reinterpret_cast<uint4*>(xs + lane * XS + rl0) = xq[0];
    *reinterpret_cast<uint4*>(xs + lane * XS + rl1) = xq[1];
  }
  __syncthreads();  // the dot table (and each warp's x rows)
  // Without a fold the epilogue writes free ring slots only: this block is done
  // with what it overwrites (dots, dt) and arrives now; a folding block arrives
  // after its fold.
  int ticket = (threadIdx.x == 0 && !fold) ? cursor_ticket(a.cursors, sb) : 0;
  // Outputs come from the checkpoint and every record since it (the fold only
  // writes the checkpoint): output i = e^{S_a} (h0 . C_i) + sum_{k<=a} cf[i][k] x_k,
  // a = count + i, cf = dt_k e^{S_a - S_k} (B_k . C_i) (+ D on record a).
  {  // warp w builds row i = w (KMAX = 4 warps; every warp holds S, dtk and ek)
    const int i = warp;
    const float Sa = __shfl_sync(FULL, S, (count + i) & 31);
    cf[i][lane] = (i < K && lane <= count + i) ? fmaf(dtk * expf(Sa - S), tbl[0][i][ek] + tbl[1][i][ek],
                                                    lane == count + i ? Dh : 0.f)
                                               : 0.f;
  }
  // Append the new records' x and z rows of this block now: its committed x
  // rows are in registers and shared memory already.
  auto slot_of = [&](int j) {
    int s = start + count + j;
    s = s < L ? s : s - L;
    return s < L ? s : s - L;
  };
  if (valid && lane < K) {
    const size_t rrow = ((size_t)sh * L + slot_of(lane)) * P + p0;
    *reinterpret_cast<uint4*>(a.rx + rrow + rl0) = xnA;
    *reinterpret_cast<uint4*>(a.rx + rrow + rl1) = xnB;
  }
  if (valid && gi < K) {
    const size_t rrow = ((size_t)sh * L + slot_of(gi)) * P + p0;
    a.rz[rrow + rl0 + gr] = zbA;
    a.rz[rrow + rl1 + gr] = zbB;
  }
#pragma unroll
  for (int u = 0; u < 2; u++) {  // the gates, silu(z)
    zg[u][0] = silu_fast(zg[u][0]);
    zg[u][1] = silu_fast(zg[u][1]);
  }
  const float Pn0 = expf(__shfl_sync(FULL, S, (count + 2 * qt) & 31));
  const float Pn1 = expf(__shfl_sync(FULL, S, (count + 2 * qt + 1) & 31));
  // this lane's columns of C_qg (the mma's B fragments), requested before the wait
  uint2 cv[FN / 16];
#pragma unroll
  for (int jb = 0; jb < FN / 16; jb++)
    cv[jb] = cvec ? *reinterpret_cast<const uint2*>(cvec + 16 * jb + 4 * qt) : make_uint2(0, 0);
  __syncthreads();  // the coefficient table
  // window term W[r][n] = sum_k x_k[r] cf[n][k] at rows (rA, rB), outputs n < 4: m16n8k8
  // tf32 products over blocks of 8 records in acc's fragment layout (x is bf16, exact
  // in tf32; cf enters as two tf32 parts; records past the window enter as 0), before the rows land
  float wd[2][4] = {};
  for (int k0 = 0; k0 < total; k0 += 8) {
    const int ka = k0 + qt, kb = ka + 4;
    const uint32_t a0 = ka < total ? (uint32_t)xs[ka * XS + rA] << 16 : 0u;
    const uint32_t a1 = ka < total ? (uint32_t)xs[ka * XS + rB] << 16 : 0u;
    const uint32_t a2 = kb < total ? (uint32_t)xs[kb * XS + rA] << 16 : 0u;
    const uint32_t a3 = kb < total ? (uint32_t)xs[kb * XS + rB] << 16 : 0u;
    uint32_t h0 = 0, l0 = 0, h1 = 0, l1 = 0;
    if (qg < KMAX) {  // cf[n][k] = 0 past output n's window
      split_tf32(cf[qg][ka], h0, l0);
      split_tf32(cf[qg][kb], h1, l1);
    }
    mma_tf32_1688(wd[0], a0, a1, a2, a3, h0, h1);
    mma_tf32_1688(wd[1], a0, a1, a2, a3, l0, l1);
  }
  const bool landed = __all_sync(FULL, mbar_wait(&bar, 0));  // uniform over the warp
  if (!landed) {
    if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
    mbar_wait(&bar, 0);
  }
  // A block that reads the bf16 copy folds (and, on that step, outputs) from the
  // fp32 rows in global memory.
  const float* gstate = (copy && fold) ? a.ckpt + tbase : nullptr;
  const bool t16 = copy && !fold;
  if (landed) {
    // h0 . [C_0..C_3] for rows (rA, rB) as m16n8k8 tf32 mma; an fp32 state is
    // split into two tf32 parts, the bf16 or fp16 read copy is exact in tf32
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    float ch[2][4] = {};
#pragma unroll
    for (int jb = 0; jb < FN / 16; jb++) {
      const int col = 16 * jb + 4 * qt;
      float4 r0, r1;
      state_rows(tile, gstate, t16, a.read_f16, a.read_f8, rA, rB, col, r0, r1);
      const float4 bv = bf4_to_f4(cv[jb]);
      if (t16) {  // uniform
        mma_tf32_1688(ch[0], __float_as_uint(r0.x), __float_as_uint(r1.x), __float_as_uint(r0.y),
                      __float_as_uint(r1.y), __float_as_uint(bv.x), __float_as_uint(bv.y));
        mma_tf32_1688(ch[1], __float_as_uint(r0.z), __float_as_uint(r1.z), __float_as_uint(r0.w),
                      __float_as_uint(r1.w), __float_as_uint(bv.z), __float_as_uint(bv.w));
      } else {
        uint32_t h0, l0, h1, l1, h2, l2, h3, l3;
        split_tf32(r0.x, h0, l0);
        split_tf32(r1.x, h1, l1);
        split_tf32(r0.y, h2, l2);
        split_tf32(r1.y, h3, l3);
        mma_tf32_1688(ch[0], h0, h1, h2, h3, __float_as_uint(bv.x), __float_as_uint(bv.y));
        mma_tf32_1688(ch[1], l0, l1, l2, l3, __float_as_uint(bv.x), __float_as_uint(bv.y));
        split_tf32(r0.z, h0, l0);
        split_tf32(r1.z, h1, l1);
        split_tf32(r0.w, h2, l2);
        split_tf32(r1.w, h3, l3);
        mma_tf32_1688(ch[0], h0, h1, h2, h3, __float_as_uint(bv.z), __float_as_uint(bv.w));
        mma_tf32_1688(ch[1], l0, l1, l2, l3, __float_as_uint(bv.z), __float_as_uint(bv.w));
      }
    }
#pragma unroll
    for (int q = 0; q < 4; q++) acc[q] = ch[0][q] + ch[1][q];
    if (t16 && a.read_f8) {  // e4m3 rows times their scales (the scale of a row factors out of its dots)
      const float* scales = reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(a.ckpt_read) +
                                                           (size_t)a.Sn * H * P * FN);
      const float sA = scales[tbase / FN + rA], sB = scales[tbase / FN + rB];
      acc[0] *= sA;
      acc[1] *= sA;
      acc[2] *= sB;
      acc[3] *= sB;
    }
    if (qt < 2) {  // outputs n0 = 2 qt, n1 = n0 + 1 at rows rA, rB
      const int n0 = 2 * qt, n1 = n0 + 1;
      const float w00 = wd[0][0] + wd[1][0], w01 = wd[0][1] + wd[1][1];
      const float w10 = wd[0][2] + wd[1][2], w11 = wd[0][3] + wd[1][3];
      if (valid) {
        const size_t y0 = (((size_t)b * K + n0) * H + h) * P + p0;
        if (n0 < K) {
          store_out<OUT_BF16>(a.y, y0 + rA, fmaf(Pn0, acc[0], w00) * zg[0][0]);
          store_out<OUT_BF16>(a.y, y0 + rB, fmaf(Pn0, acc[2], w10) * zg[0][1]);
        }
        if (n1 < K) {
          store_out<OUT_BF16>(a.y, y0 + (size_t)H * P + rA, fmaf(Pn1, acc[1], w01) * zg[1][0]);
          store_out<OUT_BF16>(a.y, y0 + (size_t)H * P + rB, fmaf(Pn1, acc[3], w11) * zg[1][1]);
        }
      }
    }
    if (fold && !copy) {  // h' = Pf h0 + sum_{k<count} wf_k x_k[r] B_k, written once (tensor cores)
      const uint16_t* rBg = a.rB + (size_t)sg * L * FN;
      fold_rows_mma(
          tile, a.ckpt + tbase, [&](int k) { return rBg + wrap(start + k, L) * FN; },
          [&](int k, int r) { return bf_to_f(xs[k * XS + r]); }, count, Pf, wf, rl0, rl1, lane);
    } else if (fold) {  // the read copy: row layout, from the fp32 rows in global memory (with the copy)
#pragma unroll
      for (int half = 0; half < 2; half++) {
        const int rl = half ? rl1 : rl0;
        float4 hv[8];
        if (gstate) {
#pragma unroll
          for (int rr = 0; rr < 8; rr++)
            hv[rr] = __ldcs(reinterpret_cast<const float4*>(gstate + (size_t)(rl + rr) * FN) + lane);
        } else {
#pragma unroll
          for (int rr = 0; rr < 8; rr++) hv[rr] = reinterpret_cast<const float4*>(tile + (rl + rr) * FN)[lane];
        }
        float xl[8];
        unpack8(xq[half], xl);
#pragma unroll
        for (int rr = 0; rr < 8; rr++) hv[rr] = scale4(Pf, hv[rr]);
        const uint16_t* rBp = a.rB + (size_t)sg * L * FN + lane * 4;
        for (int k0 = 0; k0 < count; k0 += 4) {
          float4 bk[4];
#pragma unroll
          for (int u = 0; u < 4; u++) {
            int s = start + k0 + u;
            s = s < L ? s : s - L;
            bk[u] = k0 + u < count ? load_bf4(rBp + s * FN) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 4; u++) {
            const int k = (k0 + u) & 31;
            const float w = __shfl_sync(FULL, wf, k);  // 0 for k >= count
#pragma unroll
            for (int rr = 0; rr < 8; rr++) hv[rr] = fma4(w * __shfl_sync(FULL, xl[rr], k), bk[u], hv[rr]);
          }
        }
        const size_t off = tbase + (size_t)rl * FN + lane * 4;
#pragma unroll
        for (int rr = 0; rr < 8; rr++) __stcs(reinterpret_cast<float4*>(a.ckpt + off + (size_t)rr * FN), hv[rr]);
        store_read_copy8(a, hv, off, lane);
      }
    }
  }
  // The last of the sequence's blocks to arrive (all of them are done with the
  // ring rows the append overwrites) appends the new records' B, C and dt and
  // marks the cursor pending.
  if (fold) {  // uniform: the committed B rows were read by the fold until here
    __syncthreads();
    if (threadIdx.x == 0) ticket = cursor_ticket(a.cursors, sb);
  }
  if (threadIdx.x == 0) last_flags = last_ticket(ticket, a.H * a.nPB) ? (ticket & 0xffff) : -1;
  __syncthreads();  // every thread is done; last_flags is visible
  if (last_flags >= 0) verify_epilogue(a, b, sb, cur, last_flags);
}

}  // namespace

bool m2_verify_fast_applies(const M2Args& a) {
  return a.N == FN && a.P % FPB == 0 && a.PB == FPB && a.K <= KMAX && a.L + a.K <= FW * EW &&
         a.H * a.nPB < (1 << 15) &&
         a.hpg_log2 >= 0;
}

cudaError_t m2_verify_fast_launch(const M2Args& a, int out_bf16, cudaStream_t st) {
  const dim3 grid(a.nPB, a.H, a.Bt);
  auto k = a.slots ? (out_bf16 ? m2_verify_fast_kernel<true, true> : m2_verify_fast_kernel<false, true>)
                   : (out_bf16 ? m2_verify_fast_kernel<true, false> : m2_verify_fast_kernel<false, false>);
  const int smem = FPB * FN * 4 + (a.L + a.K) * XS * 2;  // tile + the records' x rows
  cudaError_t e = prepare(k, smem, true);
  if (e != cudaSuccess) return e;
  k<<<grid, FT, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace rssm
