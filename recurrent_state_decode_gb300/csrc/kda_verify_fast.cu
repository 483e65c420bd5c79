// Speculative verify for Kimi Delta Attention (KDA), shape-specialised: dk =
// dv = 128, at most 4 new records and L + K <= 32 ("How ReplaySSM works":
// drafts go into the buffer and are verified output-only; "ReplaySSM"
// repository, "Adoption": ReplaySSM added to a KDA decode kernel). Built on
// the Gated DeltaNet verify's structure, with the decay taken per key channel.
//
// Algebra. Records t < count + K since the checkpoint S0 (t < count the
// committed window, ring slot (start + t) mod L; then the K new ones, a_j =
// count + j), G_t the channel-wise prefix sums of g, * the channel-wise
// product. Split every decay at the window's end W = count - 1:
//   f_t = exp(G_W - G_t)           committed record t to the window's end
//   w_j = exp(G_{a_j} - G_W)       the window's end to new record j
//   E   = exp(G_W)                 the checkpoint to the window's end
// each a product of later-minus-earlier decays, so no exponential of a
// positive sum is formed. With k~_j = w_j * k_j, q~_i = w_i * q_i:
//   e_j = beta_j (v_j - S0 (E * k~_j) - sum_{t<count} ((f_t * k_t) . k~_j) e_t
//                    - sum_{j'<j} ((exp(G_{a_j} - G_{a_j'}) * k_j') . k_j) e_j')
//   o_i = S0 (E * q~_i) + sum_{t<count} ((f_t * k_t) . q~_i) e_t
//                       + sum_{j<=i} ((exp(G_{a_i} - G_{a_j}) * k_j) . q_i) e_j
// and a fold (count + K > L) writes S0 Diag(E) + sum_{t<count} e_t (f_t * k_t)^T.
// The committed records' e come from the ring (fixed from their append).
//
// One CTA of eight warps per (sequence, head), so that the work per head --
// the couplings, the decays, the dot table -- is done once: warp w owns state
// rows 8w..8w+7 and 64+8w..64+8w+7. At launch: the head's 128 rows by two
// bulk copies (TMA, non-tensor; never multicast) into shared memory; threads
// c < 128 take channel c of the new records (g, k, q), form w_j, k~_j, q~_i
// into shared memory and their channel's share of the sixteen couplings among
// new records (one transposed reduction per warp, summed over the warps in
// shared memory); lane j the new record j's beta, lane 4 j + t the v of new
// record t at the lane's rows, as in the Gated DeltaNet verify. The last warp
// (idle in the channel phase) requests the rows and, before the cursor is
// known, every ring slot's e, g and k rows (one slot per lane, second
// mbarrier), so that nothing later waits on global memory. Then thread c
// turns its channel of the window's g rows into f_t in place and E; each warp forms the
// dots (f_t * k_t) . [k~, q~] of two committed records per round (one 16-value
// transposed reduction). The S0 product with the eight vectors E * k~_j,
// E * q~_i is an m16n8k8 tf32 mma per warp with both operands split into two
// tf32 parts (three products per k-step); the new records' e are solved within
// each quad, the outputs completed, the new e and v rows appended, the fold
// written if any. The block then appends its head's new k, q, g rows and beta
// (no other block reads them), and the sequence's last block to arrive marks
// the cursor pending.
#include "fast_rows.cuh"
#include "kernels.h"

namespace rssm {

namespace {

using namespace fastrows;

constexpr int GD = 128;      // dk = dv
constexpr int KMAX = 4;      // new records per verify on this path
constexpr int WMAX = 32;     // records since the checkpoint: L + K <= 32
constexpr int VW = 8;        // warps per block: one block per (sequence, head), warp w rows 8w.. and 64 + 8w..
constexpr int VT = 32 * VW;  // threads per block
constexpr int VHALF = 64;    // a warp's second row group starts here
constexpr int ES = GD + 4;   // floats per staged e row (padded; 16-byte multiple)

// The new records' k, q, g rows and beta of head h at ring slots (start +
// count + j) mod L (cursor c, already checked), by the whole block. One block
// per (sequence, head) reads that head's ring rows, so it appends them itself
// once it is done reading.
__device__ __forceinline__ void append_head(const GdnArgs& a, int b, int sb, int h, int4 c) {
  const int L = a.L, K = a.K, H = a.H, tid = threadIdx.x;
  constexpr int NB = GD / 8, NG = GD / 4;  // 16-byte pieces of a bf16 row, of an fp32 row
  constexpr int PER = 2 * NB + NG;         // pieces of one record: k, q, g
  for (int q = tid; q < K * PER; q += VT) {
    const int j = q / PER, piece = q - j * PER;
    const size_t ring = ((size_t)sb * H + h) * L + wrap(wrap(c.x + c.y + j, L), L);
    const size_t rec = ((size_t)b * K + j) * H + h;
    if (piece < NB) {
      *reinterpret_cast<uint4*>(a.rk + ring * GD + piece * 8) = *reinterpret_cast<const uint4*>(a.k + rec * GD + piece * 8);
    } else if (piece < 2 * NB) {
      const int v = piece - NB;
      *reinterpret_cast<uint4*>(a.rq + ring * GD + v * 8) = *reinterpret_cast<const uint4*>(a.q + rec * GD + v * 8);
    } else {
      const int v = piece - 2 * NB;
      *reinterpret_cast<uint4*>(a.rg + ring * GD + v * 4) = *reinterpret_cast<const uint4*>(a.g + rec * GD + v * 4);
    }
  }
  if (tid < K)
    a.rbeta[((size_t)sb * H + h) * pad4(L) + wrap(wrap(c.x + c.y + tid, L), L)] = a.beta[((size_t)b * K + tid) * H + h];
}

// The cursor rule of a verify, applied by the sequence's last block to arrive
// (one thread): on a cursor with 0 <= start < L, 0 <= count <= L and pending
// == 0, pending = K and flags = folded; otherwise the same report as the
// cursor checks and no move. The arrival count is cleared.
__device__ __forceinline__ void finish_verify_cursor(int32_t* cursors, int b, int4 c, int ticket, int nblocks, int L,
                                                     int K, int32_t* status) {
  if (!last_ticket(ticket, nblocks)) return;
  c.w = ticket & 0xffff;
  if (!(c.x >= 0 && c.x < L && c.y >= 0 && c.y <= L)) {
    report(status, RSSM_DEV_BAD_CURSOR);
  } else if (c.z != 0) {
    report(status, RSSM_DEV_PENDING);
  } else {
    c.z = K;
    c.w = (c.y + K > L) ? 1 : 0;
  }
  *reinterpret_cast<int4*>(cursors + 4 * (size_t)b) = c;
}

// SLOTS: batch rows name their state rows through a slot table.
template <bool OUT_BF16, bool SLOTS>
__global__ void __launch_bounds__(VT, 2) kda_verify_fast_kernel(GdnArgs a) {
  extern __shared__ __align__(128) float dsm[];
  const int L = a.L, H = a.H, K = a.K;
  float* tile = dsm;                 // the head's 128 rows
  float* vt = tile + GD * GD;        // [0..3] k~_j, [4..7] q~_i (fp32, all channels)
  float* ew = vt + 2 * KMAX * GD;    // E by channel
  float* fd = ew + GD;               // g, then f, of ring slot s at fd + s * GD
  float* es = fd + L * GD;           // e of ring slot s at es + s * ES (all rows)
  uint16_t* ks = reinterpret_cast<uint16_t*>(es + L * ES);  // k of ring slot s at ks + s * GD
  __shared__ float cf[2 * KMAX][WMAX + 1];  // [n][t]: (f_t * k_t) . vec_n
  __shared__ float cred[4][32];             // the couplings' per-warp sums (warps 0..3; lane layout of cpl)
  __shared__ uint64_t bar[2];               // [0] the rows, [1] the window's e and g rows
  __shared__ int4 cur_s;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, c = threadIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  // the batch row's state slot; a padding row (or a reported bad slot) leaves at once
  const int sb = SLOTS ? state_slot(a.slots, a.Sn, b, a.status, h == 0 && threadIdx.x == 0) : b;
  if (SLOTS && sb < 0) return;
  const size_t sh = (size_t)sb * H + h;  // the state's rows (S, ring, cursor); the records' are b's
  const size_t tbase = sh * GD * GD;

  if (warp == VW - 1) {  // the last warp (idle in the channel phase below): the rows, and every ring slot's e, g, k
    if (lane == 0) {
      mbar_init(&bar[0], 1);
      mbar_init(&bar[1], 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&bar[0], GD * GD * 4);
      bulk_load(tile, a.S + tbase, GD * GD * 2, &bar[0]);
      bulk_load(tile + GD * GD / 2, a.S + tbase + GD * GD / 2, GD * GD * 2, &bar[0]);
      mbar_arrive_expect_tx(&bar[1], (uint32_t)L * (2 * GD * 4 + GD * 2));
    }
    __syncwarp();
    if (lane < L) {  // lane s: ring slot s, requested before the cursor is known
      const size_t row = sh * L + lane;
      bulk_load(es + lane * ES, a.re + row * GD, GD * 4, &bar[1]);
      bulk_load(fd + lane * GD, a.rg + row * GD, GD * 4, &bar[1]);
      bulk_load(ks + lane * GD, a.rk + row * GD, GD * 2, &bar[1]);
    }
  }
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)sb);
  if (threadIdx.x == 0) cur_s = cur;
  // An invalid cursor (reported by the sequence's last block) runs as an empty
  // window with every store masked.
  const bool valid = cur.x >= 0 && cur.x < L && cur.y >= 0 && cur.y <= L && cur.z == 0;
  const int start = valid ? cur.x : 0, count = valid ? cur.y : 0, total = count + K;
  const bool fold = valid && total > L;
  const int rl0 = warp * 8, rl1 = VHALF + warp * 8;
  const int qg = lane >> 2, qt = lane & 3;  // tensor-core fragment coordinates
  const int rA = rl0 + qg, rB = rl1 + qg;   // the rows of this lane's accumulator fragments
  float bn = 0.f;
  if (lane < K) bn = a.beta[((size_t)b * K + lane) * H + h];
  uint32_t vtA = 0, vtB = 0;  // v of new record qt at rows rA, rB (bf16 bits)
  if (qt < K) {
    const size_t vrow = (((size_t)b * K + qt) * H + h) * GD;
    vtA = a.v[vrow + rA];
    vtB = a.v[vrow + rB];
  }
  if (warp < 4) {  // thread c: channel c of the new records -> w_j, k~_j, q~_i and the couplings among them
    float gn[KMAX], kn[KMAX], qn[KMAX], Gn[KMAX];
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < KMAX; j++) {
      const size_t row = (((size_t)b * K + j) * H + h) * GD + c;
      gn[j] = j < K ? a.g[row] : 0.f;
      kn[j] = j < K ? bf_to_f(a.k[row]) : 0.f;
      qn[j] = j < K ? bf_to_f(a.q[row]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < KMAX; j++) {
      acc += gn[j];
      Gn[j] = acc;
      const float w = expf(acc);
      vt[j * GD + c] = j < K ? w * kn[j] : 0.f;
      vt[(KMAX + j) * GD + c] = j < K ? w * qn[j] : 0.f;
    }
    // lane 4 j + j' (j' < j): (exp(G_{a_j} - G_{a_j'}) * k_j') . k_j; lane 16 + 4 i + j (j <= i):
    // (exp(G_{a_i} - G_{a_j}) * k_j) . q_i -- this thread's channel
    float p[32];
#pragma unroll
    for (int j = 0; j < KMAX; j++) {
#pragma unroll
      for (int j2 = 0; j2 < KMAX; j2++) {
        const float d = j2 < j ? expf(Gn[j] - Gn[j2]) : 1.f;
        p[4 * j + j2] = (j2 < j && j < K) ? d * kn[j2] * kn[j] : 0.f;
        p[16 + 4 * j + j2] = (j2 <= j && j < K) ? d * kn[j2] * qn[j] : 0.f;
      }
    }
    cred[warp][lane] = reduce_transpose<32>(p, lane);  // lane l: this warp's sum of index l
  }
  __syncthreads();  // k~, q~ and the couplings' partial sums; the barriers' initialisation
  const float cpl = cred[0][lane] + cred[1][lane] + cred[2][lane] + cred[3][lane];
  const bool staged = __syncthreads_and(mbar_wait(&bar[1], 0));
  int ticket = 0;
  if (threadIdx.x == 0 && !staged) {
    report(a.status, RSSM_DEV_TIMEOUT);
    mbar_wait(&bar[1], 0);  // the copies land before the block can leave
  }
  const bool live = valid && staged;
  const int cnt = staged ? count : 0;
  if (c < GD) {  // channel c: f_t = exp(G_W - G_t) in place of g_t, backwards over the window, then E = exp(G_W)
    float s = 0.f;
    for (int t = cnt - 1; t >= 0; t--) {
      const int sl = wrap(start + t, L);
      const float x = fd[sl * GD + c];
      fd[sl * GD + c] = expf(s);
      s += x;
    }
    ew[c] = expf(s);
  }
  __syncthreads();  // f_t and E
  if (threadIdx.x == 0) ticket = cursor_ticket(a.cursors, sb);  // every thread has read the cursor
  // window coefficients cf[n][t] = (f_t * k_t) . vec_n: warp w takes records 16 r + 2 w + i (i < 2)
  for (int base = 0; base < cnt; base += 2 * VW) {  // uniform
    float4 kh[2];
#pragma unroll
    for (int i = 0; i < 2; i++) {
      const int t = base + 2 * warp + i;
      const int sl = wrap(start + t, L);
      kh[i] = t < cnt ? mul4(ld4(fd + sl * GD + lane * 4), load_bf4(ks + sl * GD + lane * 4))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float pk[16];
#pragma unroll
    for (int n = 0; n < 2 * KMAX; n++) {
      const float4 v = ld4(vt + n * GD + lane * 4);
      pk[n] = dot4(kh[0], v);
      pk[8 + n] = dot4(kh[1], v);
    }
    const float red = reduce_transpose<16>(pk, lane);  // lane l: index l >> 1 = record 2 w + (l >> 4), vector (l >> 1) & 7
    const int t = base + 2 * warp + (lane >> 4);
    if ((lane & 1) == 0 && t < cnt) cf[(lane >> 1) & 7][t] = red;
  }
  __syncthreads();  // the coefficient table
  const bool landed = __all_sync(FULL, mbar_wait(&bar[0], 0));  // uniform over the warp
  if (!landed) {
    if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
    mbar_wait(&bar[0], 0);
  }
  if (landed) {
    // S0 . [E * k~_0..3, E * q~_0..3] for rows (rA, rB): m16n8k8 tf32 with both operands split
    // (hi hi + lo hi + hi lo); lane t takes the float4 at column 4 t, the k order permuted alike in A and B
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int jb = 0; jb < GD / 16; jb++) {
      const int col = 16 * jb + 4 * qt;
      const float4 r0 = ld4(tile + rA * GD + col), r1 = ld4(tile + rB * GD + col);
      const float4 bv = mul4(ld4(ew + col), ld4(vt + qg * GD + col));
      uint32_t ah[4], al[4], bh[2], bl[2];
      split_tf32(r0.x, ah[0], al[0]);
      split_tf32(r1.x, ah[1], al[1]);
      split_tf32(r0.y, ah[2], al[2]);
      split_tf32(r1.y, ah[3], al[3]);
      split_tf32(bv.x, bh[0], bl[0]);
      split_tf32(bv.y, bh[1], bl[1]);
      mma_tf32_1688(acc, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
      mma_tf32_1688(acc, al[0], al[1], al[2], al[3], bh[0], bh[1]);
      mma_tf32_1688(acc, ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
      split_tf32(r0.z, ah[0], al[0]);
      split_tf32(r1.z, ah[1], al[1]);
      split_tf32(r0.w, ah[2], al[2]);
      split_tf32(r1.w, ah[3], al[3]);
      split_tf32(bv.z, bh[0], bl[0]);
      split_tf32(bv.w, bh[1], bl[1]);
      mma_tf32_1688(acc, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
      mma_tf32_1688(acc, al[0], al[1], al[2], al[3], bh[0], bh[1]);
      mma_tf32_1688(acc, ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
    }
    // + the committed window: sum_t cf[n][t] e_t[row]
    const int n0 = 2 * qt, n1 = n0 + 1;
    float w00 = 0.f, w01 = 0.f, w10 = 0.f, w11 = 0.f;
    for (int t = 0; t < cnt; t++) {
      const int sl = wrap(start + t, L);
      const float c0 = cf[n0][t], c1 = cf[n1][t];
      const float eA = es[sl * ES + rA], eB = es[sl * ES + rB];
      w00 = fmaf(c0, eA, w00);
      w01 = fmaf(c1, eA, w01);
      w10 = fmaf(c0, eB, w10);
      w11 = fmaf(c1, eB, w11);
    }
    // X (vectors 0..3, lanes t = 0, 1) or Y (vectors 4..7, lanes t = 2, 3), rows rA / rB
    const float x00 = acc[0] + w00, x01 = acc[1] + w01;
    const float x10 = acc[2] + w10, x11 = acc[3] + w11;
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
    // outputs i0, i0 + 1 on lanes t = 2, 3: Y + sum_{j<=i} coupling(i, j) e_j
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
    if (live && qt >= 2) {
      const size_t o0 = (((size_t)b * K + i0) * H + h) * GD;
      if (i0 < K) {
        store_out<OUT_BF16>(a.o, o0 + rA, oA0);
        store_out<OUT_BF16>(a.o, o0 + rB, oB0);
      }
      if (i0 + 1 < K) {
        store_out<OUT_BF16>(a.o, o0 + (size_t)H * GD + rA, oA1);
        store_out<OUT_BF16>(a.o, o0 + (size_t)H * GD + rB, oB1);
      }
    }
    if (live && qt < K) {  // the new record qt's e and v rows, at rows rA, rB
      float ma = eA[0], mb = eB[0];
#pragma unroll
      for (int j = 1; j < KMAX; j++) {
        ma = qt == j ? eA[j] : ma;
        mb = qt == j ? eB[j] : mb;
      }
      const size_t slot = sh * L + wrap(wrap(start + count + qt, L), L);
      a.re[slot * GD + rA] = ma;
      a.re[slot * GD + rB] = mb;
      a.rv[slot * GD + rA] = (uint16_t)vtA;
      a.rv[slot * GD + rB] = (uint16_t)vtB;
    }
    if (fold && staged) {  // S0 Diag(E) + sum_{t<count} e_t (f_t * k_t)^T, written once
      const float4 e4 = ld4(ew + lane * 4);
#pragma unroll
      for (int half = 0; half < 2; half++) {
        const int rl = half ? rl1 : rl0;
        float4 hv[8];
#pragma unroll
        for (int rr = 0; rr < 8; rr++) hv[rr] = mul4(e4, ld4(tile + (rl + rr) * GD + lane * 4));
        for (int t0 = 0; t0 < cnt; t0 += 2) {
          float4 kt[2];
#pragma unroll
          for (int u = 0; u < 2; u++) {
            const int t = t0 + u, sl = wrap(start + t, L);
            kt[u] = t < cnt ? mul4(ld4(fd + sl * GD + lane * 4), load_bf4(ks + sl * GD + lane * 4))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int u = 0; u < 2; u++) {
            const int t = t0 + u;
            if (t < cnt) {  // uniform
              const int sl = wrap(start + t, L);
              const float4 ea2 = ld4(es + sl * ES + rl), eb2 = ld4(es + sl * ES + rl + 4);
              const float et[8] = {ea2.x, ea2.y, ea2.z, ea2.w, eb2.x, eb2.y, eb2.z, eb2.w};
#pragma unroll
              for (int rr = 0; rr < 8; rr++) hv[rr] = fma4(et[rr], kt[u], hv[rr]);
            }
          }
        }
#pragma unroll
        for (int rr = 0; rr < 8; rr++)
          __stcs(reinterpret_cast<float4*>(a.S + tbase + (size_t)(rl + rr) * GD) + lane, hv[rr]);
      }
    }
  }
  // this head's new k, q, g rows and beta, after every warp is done with the ring rows they may overwrite
  __syncthreads();
  if (live) append_head(a, b, sb, h, cur_s);
  if (threadIdx.x == 0) finish_verify_cursor(a.cursors, sb, cur_s, ticket, H, L, K, a.status);
}

}  // namespace

bool kda_verify_applies(const GdnArgs& a) {
  return a.DK == GD && a.DV == GD && a.K <= KMAX && a.L + a.K <= WMAX && a.H < (1 << 15) && a.H <= 65535 &&
         a.Bt <= 65535 && a.Sn <= 65535;
}

size_t kda_verify_fast_smem(int L) { return (size_t)(GD * GD + 2 * KMAX * GD + GD + L * GD + L * ES) * 4 + (size_t)L * GD * 2; }

cudaError_t kda_verify_launch(const GdnArgs& a, int out_bf16, cudaStream_t st) {
  if (a.Bt == 0) return cudaSuccess;
  auto k = a.slots ? (out_bf16 ? kda_verify_fast_kernel<true, true> : kda_verify_fast_kernel<false, true>)
                   : (out_bf16 ? kda_verify_fast_kernel<true, false> : kda_verify_fast_kernel<false, false>);
  const size_t smem = kda_verify_fast_smem(a.L);
  cudaError_t e = prepare(k, smem, true);
  if (e != cudaSuccess) return e;
  k<<<dim3(1, a.H, a.Bt), VT, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace rssm
