// Speculative verify for Gated DeltaNet, shape-specialised fast path: dk = dv =
// 128, at most 4 new records and L + K <= 32. Same algebra as the generic
// kernel in gdn_verify.cu (records t < count + K relative to the checkpoint S0,
// G_t = sum_{j<=t} g_j, D(a, t) = exp(G_a - G_t); the committed records' e_t
// come from the ring, the new ones are solved in order), built like the AR
// fast step.
//
// One CTA of four warps per (sequence, head, 64 state rows); warp w owns rows
// 8w..8w+7 and 32+8w..32+8w+7, lane l the float4 column chunk 4l..4l+3. At
// launch: one bulk copy (TMA, non-tensor; never multicast) of the 64 rows;
// lane s ring slot s (g); lane j new record j (g, beta); lane 8j + r the v of
// new record j at row r of each group; the new records' k and q into shared
// memory (fp32). Entry e of the dot tables is ring slot e (e < L) or new
// record e - L; warp w forms (k_e . k_j) and (k_e . q_i) for entries w, w+4, ...
// (two transposed 32-value reductions). After the cursor: the window records'
// e rows by one 256-byte bulk copy each (second mbarrier) and one inclusive
// warp scan of g. Per 8-row group two transposed 32-value reductions give, for
// each (new record j, row r), e^{G_a} S0 k_j + the committed window's k-term
// and e^{G_a} S0 q_i + its q-term; the new records' e are then solved in
// order (one shuffle each) and the outputs completed. If count + K > L the
// committed window is folded into the rows, written once. The new records'
// v and e rows go to the ring here; their k, q, g, beta (read by the other
// block of the head) are appended by the sequence's last block to arrive,
// which also marks the cursor pending.
#include "fast_rows.cuh"
#include "gdn_common.cuh"

namespace rssm {

namespace {

using namespace fastrows;

constexpr int GD = 128;      // dk = dv
constexpr int KMAX = 4;      // new records per verify on this path
constexpr int EW = 8;        // dot entries per warp: 4 x 8 = 32 >= L + K
constexpr int ES = FPB + 4;  // floats per staged e row (padded; 16-byte multiple)

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// 32 partials for 8 rows x 4 vectors: [j * 8 + rr] = h[rr] . vec_j + cf[j] * el[rr].
// Lane l ends with partial l (vector l >> 3, row l & 7).
__device__ __forceinline__ float rows8x4(const float4 (&hv)[8], const float* vecs, const float (&gam)[KMAX],
                                         const float (&cf)[KMAX], const float (&el)[8], int lane) {
  float v[32];
#pragma unroll
  for (int j = 0; j < KMAX; j++) {
    const float4 c = scale4(gam[j], lds4(vecs + j * GD + lane * 4));
#pragma unroll
    for (int rr = 0; rr < 8; rr++)
      v[j * 8 + rr] = fmaf(hv[rr].x, c.x, fmaf(hv[rr].y, c.y, fmaf(hv[rr].z, c.z, fmaf(hv[rr].w, c.w, cf[j] * el[rr]))));
  }
  return reduce_transpose<32>(v, lane);
}

template <bool OUT_BF16>
__global__ void __launch_bounds__(FT, 5) gdn_verify_fast_kernel(GdnArgs a) {
  extern __shared__ __align__(128) float dsm[];
  float* tile = dsm;                 // the block's 64 rows
  float* vecs = dsm + FPB * GD;      // [0..3] new k_j, [4..7] new q_i (fp32)
  float* es = vecs + 2 * KMAX * GD;  // e of committed record t at es + t * ES
  __shared__ float skk[KMAX][FW * EW], skq[KMAX][FW * EW];  // k_e . k_j, k_e . q_i
  __shared__ uint64_t bar[2];
  __shared__ int4 cur_s;
  __shared__ int last_flags;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int pb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int L = a.L, H = a.H, K = a.K;
  const size_t bh = (size_t)b * H + h;
  const int p0 = pb * FPB;
  const size_t tbase = (bh * GD + p0) * GD;

  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar[0], FPB * GD * 4);
    bulk_load(tile, a.S + tbase, FPB * GD * 4, &bar[0]);
  }
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)b);
  const int rl0 = warp * 8, rl1 = HALF + warp * 8;
  const int gj = lane >> 3, gr = lane & 7;  // (new record, row) this lane finishes
  const float gs = lane < L ? a.rg[bh * pad4(L) + lane] : 0.f;
  float gn = 0.f, bn = 0.f;
  if (lane < K) {
    gn = a.g[((size_t)b * K + lane) * H + h];
    bn = a.beta[((size_t)b * K + lane) * H + h];
  }
  uint16_t vbA = 0, vbB = 0;
  if (gj < K) {
    const size_t vrow = (((size_t)b * K + gj) * H + h) * GD + p0 + gr;
    vbA = a.v[vrow + rl0];
    vbB = a.v[vrow + rl1];
  }
  // the new records' k and q, fp32, in shared memory (each warp its own rows of the table)
  for (int v = warp; v < 2 * KMAX; v += FW) {
    const int j = v & (KMAX - 1);
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < K) f = load_bf4((v < KMAX ? a.k : a.q) + (((size_t)b * K + j) * H + h) * GD + lane * 4);
    reinterpret_cast<float4*>(vecs + v * GD)[lane] = f;
  }
  __syncthreads();
  // dot tables for entries e = warp + 4 m: ring slot e (e < L) or new record e - L
  const uint16_t* rkp = a.rk + bh * L * GD + lane * 4;
#pragma unroll
  for (int pass = 0; pass < 2; pass++) {
    float4 vv[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; j++) vv[j] = lds4(vecs + (pass * KMAX + j) * GD + lane * 4);
    float pk[EW * KMAX];
#pragma unroll
    for (int m = 0; m < EW; m++) {
      const int e = warp + FW * m;
      float4 ke = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e < L)
        ke = load_bf4(rkp + e * GD);
      else if (e < L + K)
        ke = lds4(vecs + (e - L) * GD + lane * 4);
#pragma unroll
      for (int j = 0; j < KMAX; j++) pk[m * KMAX + j] = dot4(ke, vv[j]);
    }
    const float red = reduce_transpose<EW * KMAX>(pk, lane);  // lane l: entry warp + 4 (l >> 2), vector l & 3
    (pass ? skq : skk)[lane & 3][warp + FW * (lane >> 2)] = red;
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
      bulk_load(es + t * ES, a.re + (bh * L + wrap(start + t, L)) * GD + p0, FPB * 4, &bar[1]);
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
  float Ga[KMAX], gam[KMAX];  // G at record count + j; e^{G_a}
#pragma unroll
  for (int j = 0; j < KMAX; j++) {
    Ga[j] = __shfl_sync(FULL, G, (count + j) & 31);
    gam[j] = expf(Ga[j]);
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
  if (threadIdx.x == 0 && !fold) ticket = cursor_ticket(a.cursors, b);  // done with the ring's k and g
  float cK[KMAX], cQ[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; j++) {
    const float d = lane < count ? expf(Ga[j] - G) : 0.f;
    cK[j] = d * skk[j][sl];
    cQ[j] = d * skq[j][sl];
  }
  float cpl = 0.f;
  if (lane < 16) {
    if (cj2 < cj && cj < K) cpl = expf(Gx - Gy) * skk[cj][L + cj2];
  } else {
    if (cj2 <= cj && cj < K) cpl = expf(Gx - Gy) * skq[cj][L + cj2];
  }
  const bool ok0 = mbar_wait(&bar[0], 0), ok1 = mbar_wait(&bar[1], 0);
  const bool landed = __all_sync(FULL, ok0 && ok1);  // uniform over the warp
  if (!landed) {
    if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
    mbar_wait(&bar[0], 0);
    mbar_wait(&bar[1], 0);
  }
  if (landed) {
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int rl = half ? rl1 : rl0;
      float4 hv[8];
#pragma unroll
      for (int rr = 0; rr < 8; rr++) hv[rr] = lds4(tile + (rl + rr) * GD + lane * 4);
      float el[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // e of committed record `lane`, the 8 rows
      if (lane < count) {
        const float4 ea = lds4(es + lane * ES + rl), eb = lds4(es + lane * ES + rl + 4);
        el[0] = ea.x; el[1] = ea.y; el[2] = ea.z; el[3] = ea.w;
        el[4] = eb.x; el[5] = eb.y; el[6] = eb.z; el[7] = eb.w;
      }
      // lane (j, r): e^{G_a} S0 k_j + sum over the committed window of D (k_t . k_j) e_t
      const float X = rows8x4(hv, vecs, gam, cK, el, lane);
      const float vm = bf_to_f(half ? vbB : vbA);
      float en[KMAX];  // e of new record j at this lane's row
#pragma unroll
      for (int j = 0; j < KMAX; j++) {
        float rhs = vm - X;
#pragma unroll
        for (int j2 = 0; j2 < j; j2++) rhs = fmaf(-__shfl_sync(FULL, cpl, 4 * j + j2), en[j2], rhs);
        en[j] = __shfl_sync(FULL, __shfl_sync(FULL, bn, j) * rhs, 8 * j + gr);
      }
      const float Y = rows8x4(hv, vecs + KMAX * GD, gam, cQ, el, lane);
      float o = Y;
#pragma unroll
      for (int j = 0; j < KMAX; j++) {
        const float c = __shfl_sync(FULL, cpl, (16 + 4 * gj + j) & 31);
        o = fmaf(c, en[j], o);  // c = 0 unless j <= gj < K
      }
      if (valid && gj < K) {
        float my = en[0];
#pragma unroll
        for (int j = 1; j < KMAX; j++) my = gj == j ? en[j] : my;
        store_y<OUT_BF16>(a.o, (((size_t)b * K + gj) * H + h) * GD + p0 + rl + gr, o);
        const size_t slot = bh * L + wrap(wrap(start + count + gj, L), L);
        a.re[slot * GD + p0 + rl + gr] = my;
        a.rv[slot * GD + p0 + rl + gr] = half ? vbB : vbA;
      }
      if (fold) {  // S0' = e^{G_{c-1}} S0 + sum_{t<c} D(c-1, t) e_t k_t^T, written once
#pragma unroll
        for (int rr = 0; rr < 8; rr++) hv[rr] = scale4(Pf, hv[rr]);
        for (int t0 = 0; t0 < count; t0 += 2) {
          float4 kt[2];
#pragma unroll
          for (int u = 0; u < 2; u++)
            kt[u] = t0 + u < count ? load_bf4(rkp + wrap(start + t0 + u, L) * GD) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int u = 0; u < 2; u++) {
            const int t = t0 + u;
            const float c = __shfl_sync(FULL, wf, t & 31);
            if (t < count) {  // uniform
              const float4 ea2 = lds4(es + t * ES + rl), eb2 = lds4(es + t * ES + rl + 4);
              const float et[8] = {ea2.x, ea2.y, ea2.z, ea2.w, eb2.x, eb2.y, eb2.z, eb2.w};
#pragma unroll
              for (int rr = 0; rr < 8; rr++) hv[rr] = fma4(c * et[rr], kt[u], hv[rr]);
            }
          }
        }
#pragma unroll
        for (int rr = 0; rr < 8; rr++)
          __stcs(reinterpret_cast<float4*>(a.S + tbase + (size_t)(rl + rr) * GD) + lane, hv[rr]);
      }
    }
  }
  if (fold) {  // uniform: the fold read the ring's k rows until here
    __syncthreads();
    if (threadIdx.x == 0) ticket = cursor_ticket(a.cursors, b);
  }
  __syncthreads();
  if (threadIdx.x == 0) last_flags = last_ticket(ticket, 2 * H) ? (ticket & 0xffff) : -1;
  __syncthreads();
  if (last_flags >= 0) gdn_verify_epilogue(a, b, cur_s, last_flags);
}

}  // namespace

bool gdn_verify_fast_applies(const GdnArgs& a) {
  return a.DK == GD && a.DV == GD && a.K <= KMAX && a.L + a.K <= FW * EW && 2 * a.H < (1 << 15) && a.H <= 65535 &&
         a.Bt <= 65535;
}

cudaError_t gdn_verify_fast_launch(const GdnArgs& a, int out_bf16, cudaStream_t st) {
  if (a.Bt == 0) return cudaSuccess;
  auto k = out_bf16 ? gdn_verify_fast_kernel<true> : gdn_verify_fast_kernel<false>;
  const int smem = (FPB * GD + 2 * KMAX * GD + a.L * ES) * 4;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<dim3(2, a.H, a.Bt), FT, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace rssm
