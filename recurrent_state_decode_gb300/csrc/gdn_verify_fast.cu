// Speculative verify for Gated DeltaNet, shape-specialised fast path: dk = dv =
// 128, at most 4 new records and L + K <= 32. Same algebra as the generic
// kernel in gdn_verify.cu (records t < count + K relative to the checkpoint S0,
// G_t = sum_{j<=t} g_j, D(a, t) = exp(G_a - G_t); the committed records' e_t
// come from the ring, the new ones are solved in order), built like the AR
// fast step.
//
// One CTA of four warps per (sequence, head, 64 state rows); warp w owns rows
// 8w..8w+7 and 32+8w..32+8w+7, lane l the float4 column chunk 4l..4l+3. At
// launch, none of it waiting on another: one bulk copy (TMA, non-tensor; never
// multicast) of the 64 rows; lane s ring slot s (g); lane j new record j (g,
// beta); lane 4g + t the v of new record t at rows 8w + g and 32 + 8w + g; each
// lane its fragments of the dot tables' operands and of the new records' k and
// q (bf16, in registers). Entry e of the dot tables is ring slot e (e < L) or
// new record e - L; (k_e . k_j) and (k_e . q_i) for all 32 entries come from
// tensor-core products [32 x 128] . [128 x 8], warp w taking entries 16 (w & 1)
// .. + 15 over column half w >> 1 (readers add the halves), taken once thread
// 0 has requested the window records' e rows (one 256-byte bulk copy each,
// second mbarrier), which it does as soon as the cursor arrives. Then one
// inclusive warp scan of g and a per-block table of the committed records'
// coefficients D (k_t . vec), warp w building rows w and w + 4. Each warp then
// forms S0 . [k_0..k_3, q_0..q_3] for its 16 rows as m16n8k8 tf32 mma (the fp32
// state split into two tf32 parts, two independent accumulator chains), adds
// the committed window's terms, solves the new records' e in order within each
// quad and completes the outputs. If count + K > L the committed window is
// folded into the rows on the tensor cores, written once. The new records' v
// and e rows go to the ring here; their k, q, g, beta (read by the other block
// of the head) are appended by the sequence's last block to arrive, which also
// marks the cursor pending.
#include "fast_rows.cuh"
#include "fold_mma.cuh"
#include "gdn_common.cuh"

namespace rssm {

namespace {

using namespace fastrows;

constexpr int GD = 128;      // dk = dv
constexpr int KMAX = 4;      // new records per verify on this path
constexpr int EW = 8;        // dot entries per warp: 4 x 8 = 32 >= L + K
constexpr int ES = FPB + 4;  // floats per staged e row (padded; 16-byte multiple)

// SLOTS: batch rows name their state rows through a slot table.
template <bool OUT_BF16, bool SLOTS>
__global__ void __launch_bounds__(FT, 5) gdn_verify_fast_kernel(GdnArgs a) {
  extern __shared__ __align__(128) float dsm[];
  float* tile = dsm;                 // the block's 64 rows
  float* es = dsm + FPB * GD;        // e of committed record t at es + t * ES
  __shared__ float tbl[2][2 * KMAX][FW * EW];  // [half][n][e]: k_e . vec_n over column half `half`;
                                                // vec 0..3 = new k_j, 4..7 = new q_i
  __shared__ float cf[2 * KMAX][33];        // [n][t]: D(a_n, t) (k_t . vec_n) of committed record t (padded rows)
  __shared__ uint64_t bar[2];
  __shared__ int4 cur_s;
  __shared__ int last_flags;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int L = a.L, H = a.H, K = a.K;
  // the batch row's state slot; a padding row (or a reported bad slot) leaves at once
  const int sb = SLOTS ? state_slot(a.slots, a.Sn, b, a.status, pb == 0 && h == 0 && threadIdx.x == 0) : b;
  if (SLOTS && sb < 0) return;
  const size_t sh = (size_t)sb * H + h;  // the state's rows (S, ring, cursor)
  const int p0 = pb * FPB;
  const size_t tbase = (sh * GD + p0) * GD;

  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar[0], FPB * GD * 4);
    bulk_load(tile, a.S + tbase, FPB * GD * 4, &bar[0]);
  }
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)sb);
  const int rl0 = warp * 8, rl1 = HALF + warp * 8;
  const int qg = lane >> 2, qt = lane & 3;   // tensor-core fragment coordinates
  const int rA = rl0 + qg, rB = rl1 + qg;    // the rows of this lane's accumulator fragments
  const float gs = lane < L ? a.rg[sh * pad4(L) + lane] : 0.f;
  float gn = 0.f, bn = 0.f;
  if (lane < K) {
    gn = a.g[((size_t)b * K + lane) * H + h];
    bn = a.beta[((size_t)b * K + lane) * H + h];
  }
  uint32_t vtA = 0, vtB = 0;  // v of new record qt at rows rA, rB (bf16 bits)
  if (qt < K) {
    const size_t vrow = (((size_t)b * K + qt) * H + h) * GD + p0;
    vtA = a.v[vrow + rA];
    vtB = a.v[vrow + rB];
  }
  // the products' B fragments: vector n = qg (new k_n for n < 4, new q_{n-4} from 4 on) at
  // columns 16 jb + 4 qt .. + 3, bf16 (exact in tf32), zero past the K new records
  uint2 cv[GD / 16];
  {
    const int j = qg & (KMAX - 1);
    const uint16_t* vp = (qg < KMAX ? a.k : a.q) + (((size_t)b * K + j) * H + h) * GD + 4 * qt;
#pragma unroll
    for (int jb = 0; jb < GD / 16; jb++)
      cv[jb] = j < K ? *reinterpret_cast<const uint2*>(vp + 16 * jb) : make_uint2(0, 0);
  }
  // dot tables tbl[n][e] = k_e . vec_n for entries e < 32 (ring slot e if e < L,
  // new record e - L if e < L + K, else 0): [32 x 128] . [128 x 8] on the
  // tensor cores, warp w taking entries 16 (w & 1) .. 16 (w & 1) + 15 over the
  // column half w >> 1 (bf16 inputs are exact in tf32, so one mma per k-step);
  // readers add the two halves. The rows are requested here, the products
  // taken once the e rows are on their way.
  const int e0 = 16 * (warp & 1) + qg, e1 = e0 + 8, ch = warp >> 1;
  uint2 da[GD / 32], db[GD / 32];
  {
    auto row_of = [&](int e) -> const uint16_t* {
      if (e < L) return a.rk + (sh * L + e) * GD;
      if (e < L + K) return a.k + (((size_t)b * K + (e - L)) * H + h) * GD;
      return nullptr;
    };
    const uint16_t* g0 = row_of(e0);
    const uint16_t* g1 = row_of(e1);
#pragma unroll
    for (int j = 0; j < GD / 32; j++) {
      const int col = 16 * (ch * (GD / 32) + j) + 4 * qt;
      da[j] = g0 ? *reinterpret_cast<const uint2*>(g0 + col) : make_uint2(0, 0);
      db[j] = g1 ? *reinterpret_cast<const uint2*>(g1 + col) : make_uint2(0, 0);
    }
  }
  // An invalid cursor (reported by the epilogue) runs as an empty window with
  // every store masked.
  const bool valid = cur.x >= 0 && cur.x < L && cur.y >= 0 && cur.y <= L && cur.z == 0;
  const int start = valid ? cur.x : 0, count = valid ? cur.y : 0, total = count + K;
  const bool fold = valid && total > L;
  if (threadIdx.x == 0) {  // committed records' e rows of this block, in record order
    cur_s = cur;
    mbar_arrive_expect_tx(&bar[1], (uint32_t)count * FPB * 4);
    for (int t = 0; t < count; t++)
      bulk_load(es + t * ES, a.re + (sh * L + wrap(start + t, L)) * GD + p0, FPB * 4, &bar[1]);
  }
  {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < GD / 32; j++) {
      const float4 r0 = bf4_to_f4(da[j]), r1 = bf4_to_f4(db[j]);
      const float4 bv = bf4_to_f4(ch ? cv[GD / 32 + j] : cv[j]);
      mma_tf32_1688(acc, __float_as_uint(r0.x), __float_as_uint(r1.x), __float_as_uint(r0.y), __float_as_uint(r1.y),
                    __float_as_uint(bv.x), __float_as_uint(bv.y));
      mma_tf32_1688(acc, __float_as_uint(r0.z), __float_as_uint(r1.z), __float_as_uint(r0.w), __float_as_uint(r1.w),
                    __float_as_uint(bv.z), __float_as_uint(bv.w));
    }
    tbl[ch][2 * qt][e0] = acc[0];
    tbl[ch][2 * qt + 1][e0] = acc[1];
    tbl[ch][2 * qt][e1] = acc[2];
    tbl[ch][2 * qt + 1][e1] = acc[3];
  }
  // record t on lane t: committed (ring slot sl) or new (record jn)
  int sl = start + lane;
  sl = sl < L ? sl : sl - L;
  const int jn = (lane - count) & 31;
  const float g_ring = __shfl_sync(FULL, gs, sl), g_new = __shfl_sync(FULL, gn, jn);
  float G = lane < count ? g_ring : (lane < total ? g_new : 0.f);  // inclusive scan: G_t
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float v = __shfl_up_sync(FULL, G, o);
    if (lane >= o) G += v;
  }
  const float Gc = __shfl_sync(FULL, G, (count - 1) & 31);
  const float Pf = expf(Gc);                                 // fold: e^{G_{count-1}}
  const float wf = lane < count ? expf(Gc - G) : 0.f;        // fold weight of record `lane`
  // lane-distributed couplings among the new records: lane 4 j + j' holds
  // D(a_j, a_j') (k_j' . k_j) (j' < j); lane 16 + 4 i + j holds D(a_i, a_j) (k_j . q_i) (j <= i)
  const int cj = (lane >> 2) & 3, cj2 = lane & 3;
  const float Gx = __shfl_sync(FULL, G, (count + cj) & 31), Gy = __shfl_sync(FULL, G, (count + cj2) & 31);
  __syncthreads();  // the dot tables
  int ticket = 0;
  if (threadIdx.x == 0 && !fold) ticket = cursor_ticket(a.cursors, sb);  // done with the ring's k and g
  {  // window coefficients of committed record `lane`: warp w builds rows w and w + 4 (vectors k_w, q_w)
    const float Gw = __shfl_sync(FULL, G, (count + warp) & 31);
    const float d = lane < count ? expf(Gw - G) : 0.f;
    cf[warp][lane] = d * (tbl[0][warp][sl] + tbl[1][warp][sl]);
    cf[warp + KMAX][lane] = d * (tbl[0][warp + KMAX][sl] + tbl[1][warp + KMAX][sl]);
  }
  __syncthreads();  // the coefficient table
  float cpl = 0.f;
  if (lane < 16) {
    if (cj2 < cj && cj < K) cpl = expf(Gx - Gy) * (tbl[0][cj][L + cj2] + tbl[1][cj][L + cj2]);
  } else {
    if (cj2 <= cj && cj < K) cpl = expf(Gx - Gy) * (tbl[0][KMAX + cj][L + cj2] + tbl[1][KMAX + cj][L + cj2]);
  }
  const bool ok0 = mbar_wait(&bar[0], 0), ok1 = mbar_wait(&bar[1], 0);
  const bool landed = __all_sync(FULL, ok0 && ok1);  // uniform over the warp
  if (!landed) {
    if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
    mbar_wait(&bar[0], 0);
    mbar_wait(&bar[1], 0);
  }
  if (landed) {
    // S0 . [k_0..k_3, q_0..q_3] for rows (rA, rB) on the tensor cores: per 16
    // columns two k-steps of m16n8k8 (lane t takes the float4 at column 4t, so
    // the k order is permuted alike in A and B), S0 split into two tf32 parts.
    float acc[4], ch[2][4] = {};  // the hi and lo parts' products, two independent chains
#pragma unroll
    for (int jb = 0; jb < GD / 16; jb++) {
      const int col = 16 * jb + 4 * qt;
      const float4 r0 = ld4(tile + rA * GD + col), r1 = ld4(tile + rB * GD + col);
      const float4 bv = bf4_to_f4(cv[jb]);
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
#pragma unroll
    for (int q = 0; q < 4; q++) acc[q] = ch[0][q] + ch[1][q];
    // + the committed window: sum_t D(a_n, t) (k_t . vec_n) e_t[row]
    const int n0 = 2 * qt, n1 = n0 + 1;
    float w00 = 0.f, w01 = 0.f, w10 = 0.f, w11 = 0.f;
    for (int t = 0; t < count; t++) {
      const float c0 = cf[n0][t], c1 = cf[n1][t];
      const float eA = es[t * ES + rA], eB = es[t * ES + rB];
      w00 = fmaf(c0, eA, w00);
      w01 = fmaf(c1, eA, w01);
      w10 = fmaf(c0, eB, w10);
      w11 = fmaf(c1, eB, w11);
    }
    const float ga0 = expf(__shfl_sync(FULL, G, (count + (n0 & 3)) & 31));
    const float ga1 = expf(__shfl_sync(FULL, G, (count + (n1 & 3)) & 31));
    // X (vectors 0..3, lanes t = 0, 1) or Y (vectors 4..7, lanes t = 2, 3), rows rA / rB
    const float x00 = fmaf(ga0, acc[0], w00), x01 = fmaf(ga1, acc[1], w01);
    const float x10 = fmaf(ga0, acc[2], w10), x11 = fmaf(ga1, acc[3], w11);
    // the new records' e, solved in order (every lane of the quad, rows rA and rB)
    const int qb = lane & ~3;
    float XA[KMAX], XB[KMAX], vA[KMAX], vB[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; j++) {
      XA[j] = __shfl_sync(FULL, (j & 1) ? x01 : x00, qb + (j >> 1));
      XB[j] = __shfl_sync(FULL, (j & 1) ? x11 : x10, qb + (j >> 1));
      vA[j] = bf_to_f((uint16_t)__shfl_sync(FULL, vtA, qb + j));
      vB[j] = bf_to_f((uint16_t)__shfl_sync(FULL, vtB, qb + j));
    }
    float eA[KMAX], eB[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; j++) {
      const float bj = __shfl_sync(FULL, bn, j);  // 0 for j >= K
      float ra = vA[j] - XA[j], rb = vB[j] - XB[j];
#pragma unroll
      for (int j2 = 0; j2 < j; j2++) {
        const float m = __shfl_sync(FULL, cpl, 4 * j + j2);
        ra = fmaf(-m, eA[j2], ra);
        rb = fmaf(-m, eB[j2], rb);
      }
      eA[j] = bj * ra;
      eB[j] = bj * rb;
    }
    // outputs i0, i0 + 1 on lanes t = 2, 3: Y + sum_{j<=i} D(a_i, a_j) (k_j . q_i) e_j
    const int i0 = (2 * qt) & 3;
    float oA0 = x00, oA1 = x01, oB0 = x10, oB1 = x11;
#pragma unroll
    for (int j = 0; j < KMAX; j++) {
      const float c0 = __shfl_sync(FULL, cpl, (16 + 4 * i0 + j) & 31);
      const float c1 = __shfl_sync(FULL, cpl, (16 + 4 * (i0 + 1) + j) & 31);
      oA0 = fmaf(c0, eA[j], oA0);
      oA1 = fmaf(c1, eA[j], oA1);
      oB0 = fmaf(c0, eB[j], oB0);
      oB1 = fmaf(c1, eB[j], oB1);
    }
    if (valid && qt >= 2) {
      const size_t o0 = (((size_t)b * K + i0) * H + h) * GD + p0;
      if (i0 < K) {
        store_out<OUT_BF16>(a.o, o0 + rA, oA0);
        store_out<OUT_BF16>(a.o, o0 + rB, oB0);
      }
      if (i0 + 1 < K) {
        store_out<OUT_BF16>(a.o, o0 + (size_t)H * GD + rA, oA1);
        store_out<OUT_BF16>(a.o, o0 + (size_t)H * GD + rB, oB1);
      }
    }
    if (valid && qt < K) {  // the new record qt's e and v rows, at rows rA, rB
      float ma = eA[0], mb = eB[0];
#pragma unroll
      for (int j = 1; j < KMAX; j++) {
        ma = qt == j ? eA[j] : ma;
        mb = qt == j ? eB[j] : mb;
      }
      const size_t slot = sh * L + wrap(wrap(start + count + qt, L), L);
      a.re[slot * GD + p0 + rA] = ma;
      a.re[slot * GD + p0 + rB] = mb;
      a.rv[slot * GD + p0 + rA] = (uint16_t)vtA;
      a.rv[slot * GD + p0 + rB] = (uint16_t)vtB;
    }
    if (fold) {  // S0' = e^{G_{c-1}} S0 + sum_{t<c} D(c-1, t) e_t k_t^T, written once (tensor cores)
      const uint16_t* rk0 = a.rk + sh * L * GD;
      fold_rows_mma(
          tile, a.S + tbase, [&](int t) { return rk0 + wrap(start + t, L) * GD; },
          [&](int t, int r) { return es[t * ES + r]; }, count, Pf, wf, rl0, rl1, lane);
    }
  }
  if (fold) {  // uniform: the fold read the ring's k rows until here
    __syncthreads();
    if (threadIdx.x == 0) ticket = cursor_ticket(a.cursors, sb);
  }
  __syncthreads();
  if (threadIdx.x == 0) last_flags = last_ticket(ticket, 2 * H) ? (ticket & 0xffff) : -1;
  __syncthreads();
  if (last_flags >= 0) gdn_verify_epilogue(a, b, sb, cur_s, last_flags);
}

}  // namespace

bool gdn_verify_fast_applies(const GdnArgs& a) {
  return a.DK == GD && a.DV == GD && a.K <= KMAX && a.L + a.K <= FW * EW && 2 * a.H < (1 << 15) && a.H <= 65535 &&
         a.Bt <= 65535 && a.Sn <= 65535;
}

cudaError_t gdn_verify_fast_launch(const GdnArgs& a, int out_bf16, cudaStream_t st) {
  if (a.Bt == 0) return cudaSuccess;
  auto k = a.slots ? (out_bf16 ? gdn_verify_fast_kernel<true, true> : gdn_verify_fast_kernel<false, true>)
                   : (out_bf16 ? gdn_verify_fast_kernel<true, false> : gdn_verify_fast_kernel<false, false>);
  const int smem = (FPB * GD + a.L * ES) * 4;
  cudaError_t e = prepare(k, smem, true);
  if (e != cudaSuccess) return e;
  k<<<dim3(2, a.H, a.Bt), FT, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace rssm
