// ReplaySSM AR decode step for Gated DeltaNet, shape-specialised fast path:
// dk = dv = 128, L <= 31 ("How ReplaySSM works": non-flush steps read the
// checkpoint and the window and write no state; the L-th step folds the window
// and writes the state once).
//
// Algebra (the gated delta rule S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T)
// + beta_t v_t k_t^T rewritten as S_t = alpha_t S_{t-1} + e_t k_t^T with
// e_t = beta_t (v_t - alpha_t S_{t-1} k_t)). Window records t = 0..m-1 (the
// last is the current one), D(t, s) = exp(sum_{s<j<=t} g_j), gamma = D(m-1, -1):
//   e_cur = beta (v - gamma S0 k - sum_{t<m-1} D(m-1,t) (k_t . k) e_t)
//   o     = gamma S0 q + sum_{t<m-1} D(m-1,t) (k_t . q) e_t + (k . q) e_cur
//   S_m   = gamma S0 + sum_{t<=m-1} D(m-1,t) e_t k_t^T             (flush only)
// e_t of a committed record depends on S0 and earlier records only, so it is
// read from the ring (written when the record was current) instead of being
// solved again: a step costs two matvecs of the checkpoint (S0 k, S0 q).
//
// One CTA of four warps per (sequence, head, 64 state rows); warp w owns rows
// 8w..8w+7 and 32+8w..32+8w+7, lane l the float4 column chunk 4l..4l+3. Every
// load is issued at launch, none waiting on the cursor: the 64 rows by one bulk
// copy (TMA, non-tensor; never multicast) into shared memory; lane s ring slot
// s (g); the current record. Once the cursor is known the block's threads also
// copy the window records' e rows of this block (16-byte asynchronous copies,
// spread over the threads), so that only the window's corrections are read. Warp w forms the dots
// k_s . k and k_s . q of ring slots w, w+4, ... (slot L: the current k), one
// transposed reduction, shared through shared memory. After the cursor, lane t
// takes record t by a shuffle and one suffix scan gives every D(m-1, t). Per
// 8-row group one transposed 16-value reduction yields, for each row,
// gamma S0 k + the window's k-term and gamma S0 q + the window's q-term (the
// window terms are each lane's partials, added before the reduction). The last
// of a sequence's blocks to have read its cursor advances it (an arrival count
// in the high half of the cursor's flags word), so the step is one kernel.
#include <type_traits>

#include "fast_rows.cuh"
#include "kernels.h"

namespace rssm {

namespace {

using namespace fastrows;

constexpr int GD = 128;  // dk = dv
constexpr int KW = 8;    // dot entries per warp: 4 x 8 >= L + 1
// With L <= 16 four ring slots per warp cover the window, and the current
// record's k . q is one warp sum instead: half the dot work, an 8-wide reduction.
constexpr int KW_SHORT = 4;
constexpr int ES = FPB + 4;  // floats per staged e row (padded against bank conflicts; 16-byte multiple)

// SLOTS: batch rows name their state rows through a slot table.
// KWT: ring slots per warp in the dot table (KW, or KW_SHORT when L <= 16).
template <bool OUT_BF16, bool SLOTS, int KWT = KW>
__global__ void __launch_bounds__(FT, 6) gdn_step_fast_kernel(GdnArgs a) {
  extern __shared__ __align__(128) float dsm[];
  float* tile = dsm;               // the block's 64 rows
  float* es = dsm + FPB * GD;      // e of window record t at es + t * ES (the block's rows)
  __shared__ float skk[FW * KW], skq[FW * KW];  // k_s . k, k_s . q by ring slot; [L] = current
  __shared__ uint64_t bar;         // the rows
  __shared__ int4 cur_s;           // the cursor as read, for the sequence's last block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int L = a.L, H = a.H;
  const int pb = blockIdx.x, b = blockIdx.z;
  // the batch row's state slot; a padding row (or a reported bad slot) leaves at once
  const int sb = SLOTS ? state_slot(a.slots, a.Sn, b, a.status, pb == 0 && blockIdx.y == 0 && threadIdx.x == 0) : b;
  if (SLOTS && sb < 0) return;
  const size_t bh = (size_t)b * H + blockIdx.y;   // the record's rows (q, k, v, g, beta, o)
  const size_t sh = (size_t)sb * H + blockIdx.y;  // the state's rows (S, ring, cursor)
  const int p0 = pb * FPB;
  const size_t tbase = (sh * GD + p0) * GD;

  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, FPB * GD * 4);
    bulk_load(tile, a.S + tbase, FPB * GD * 4, &bar);
  }
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * sb);
  const bool valid = cur.x >= 0 && cur.x < L && cur.y >= 0 && cur.y < L && cur.z == 0;
  // An invalid cursor (reported by the cursor kernel) runs as an empty window
  // with every store masked, so that no lane leaves before the shuffles below.
  const int start = valid ? cur.x : 0, count = valid ? cur.y : 0, m = count + 1;
  const int rl0 = warp * 8, rl1 = HALF + warp * 8;  // the warp's row groups (within the block)
  // ring slot `lane`: g
  const float gs = lane < L ? a.rg[sh * pad4(L) + lane] : 0.f;
  // the current record
  const uint2 kraw = *reinterpret_cast<const uint2*>(a.k + bh * GD + lane * 4);
  const uint2 qraw = *reinterpret_cast<const uint2*>(a.q + bh * GD + lane * 4);
  const float gm = a.g[bh], bm = a.beta[bh];
  const int vr = (lane >> 1) & 7;  // the row this lane finishes (lanes 0..15)
  const uint16_t vbA = a.v[bh * GD + p0 + rl0 + vr], vbB = a.v[bh * GD + p0 + rl1 + vr];
  float kq_cur;  // k . q of the current record
  {  // k_s . k and k_s . q for ring slots s = warp + 4 j (s == L: the current k, with KW slots per warp)
    const uint16_t* rkp = a.rk + sh * L * GD + lane * 4;
    float pk[2 * KWT];
#pragma unroll
    for (int j = 0; j < KWT; j++) {
      const int s = warp + FW * j;
      const float4 ks = s < L ? load_bf4(rkp + s * GD)
                              : (KWT == KW && s == L ? bf4_to_f4(kraw) : make_float4(0.f, 0.f, 0.f, 0.f));
      pk[2 * j] = dot4(ks, bf4_to_f4(kraw));
      pk[2 * j + 1] = dot4(ks, bf4_to_f4(qraw));
    }
    const float red = reduce_transpose<2 * KWT>(pk, lane);
    if (KWT == KW) {  // lane l: partial l >> 1 = (slot j = l >> 2, k or q)
      if ((lane & 1) == 0) ((lane & 2) ? skq : skk)[warp + FW * (lane >> 2)] = red;
      kq_cur = 0.f;
    } else {  // lane l: partial reduce8_row(l) = (slot j = index >> 1, k or q)
      const int idx = reduce8_row(lane);
      if ((lane & 3) == 0) ((idx & 1) ? skq : skk)[warp + FW * (idx >> 1)] = red;
      kq_cur = warp_sum(dot4(bf4_to_f4(kraw), bf4_to_f4(qraw)));
    }
  }
  // the window's e rows of this block, in record order: 16-byte asynchronous copies spread over the threads
  for (int c = threadIdx.x; c < count * (FPB / 4); c += FT) {
    const int t = c / (FPB / 4), j = c - t * (FPB / 4);
    const int s = start + t < L ? start + t : start + t - L;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(es + t * ES + 4 * j)),
                 "l"(a.re + (sh * L + s) * GD + p0 + 4 * j)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  const bool flush = valid && m == L;
  const int scur = start + count < L ? start + count : start + count - L;  // the current record's slot
  // window, lane t = record t
  int sl = start + lane;
  sl = sl < L ? sl : sl - L;
  const float gr = __shfl_sync(FULL, gs, sl);
  const float gt = lane < count ? gr : (lane == count ? gm : 0.f);
  float sfx = gt;  // sum_{t<=j<=m-1} g_j
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float v = __shfl_down_sync(FULL, sfx, o);
    if (lane + o < 32) sfx += v;
  }
  float ex = __shfl_down_sync(FULL, sfx, 1);  // sum_{t<j<=m-1} g_j
  if (lane == 31) ex = 0.f;
  const float gamma = expf(__shfl_sync(FULL, sfx, 0));
  const float Dt = expf(ex);  // D(m-1, t)
  __syncthreads();
  int ticket = 0;
  if (threadIdx.x == 0) {  // every thread has read the cursor
    ticket = cursor_ticket(a.cursors, sb);
    cur_s = cur;
  }
  const int ent = lane < count ? sl : L;
  const float cK = lane < count ? Dt * skk[ent] : 0.f;
  const float cQ = lane < count ? Dt * skq[ent] : 0.f;
  if (KWT == KW) kq_cur = skq[L];
  const float4 ka = scale4(gamma, bf4_to_f4(kraw)), qa = scale4(gamma, bf4_to_f4(qraw));
  // Append the current record now (its e follows below): its slot is outside
  // the window, so no block reads it for a result.
  if (valid && !flush) {
    const size_t vrow = (sh * L + scur) * GD + p0 + vr;
    if (lane < 16 && (lane & 1) == 0) {
      a.rv[vrow + rl0] = vbA;
      a.rv[vrow + rl1] = vbB;
    }
    if (pb == 0 && warp == 0) {
      const size_t krow = (sh * L + scur) * GD + lane * 4;
      *reinterpret_cast<uint2*>(a.rk + krow) = kraw;
      *reinterpret_cast<uint2*>(a.rq + krow) = qraw;
      if (lane == 0) {
        a.rg[sh * pad4(L) + scur] = gm;
        a.rbeta[sh * pad4(L) + scur] = bm;
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();  // every thread's e chunks
  if (!__all_sync(FULL, mbar_wait(&bar, 0))) {
    if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
    mbar_wait(&bar, 0);
    if (threadIdx.x == 0) finish_ar_cursor(a.cursors, sb, cur_s, ticket, a.H * 2, L, a.status);
    return;
  }
#pragma unroll
  for (int half = 0; half < 2; half++) {
    const int rl = half ? rl1 : rl0;
    float4 ea = make_float4(0.f, 0.f, 0.f, 0.f), eb = ea;  // e_t of the 8 rows (lane t)
    if (lane < count) {
      ea = ld4(es + lane * ES + rl);
      eb = ld4(es + lane * ES + rl + 4);
    }
    const float el[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
    float4 hv[8];
#pragma unroll
    for (int rr = 0; rr < 8; rr++) hv[rr] = reinterpret_cast<const float4*>(tile + (rl + rr) * GD)[lane];
    float tk[8], tq[8];
#pragma unroll
    for (int rr = 0; rr < 8; rr++) {
      tk[rr] = cK * el[rr];
      tq[rr] = cQ * el[rr];
    }
    // lanes 0..15: gamma S0 k + k-term of row vr; lanes 16..31: the q counterpart
    const float tot = rows8x2(hv, ka, qa, tk, tq, lane);
    const float yq = __shfl_down_sync(FULL, tot, 16);
    const float ec = bm * (bf_to_f(half ? vbB : vbA) - tot);  // e of the current record, row vr (lanes < 16)
    const size_t row = bh * GD + p0 + rl + vr;
    if (valid && lane < 16 && (lane & 1) == 0) {
      store_out<OUT_BF16>(a.o, row, fmaf(kq_cur, ec, yq));
      if (!flush) a.re[(sh * L + scur) * GD + p0 + rl + vr] = ec;
    }
    if (flush) {  // S_m = gamma S0 + sum_t D(m-1,t) e_t k_t^T, written once
#pragma unroll
      for (int rr = 0; rr < 8; rr++) hv[rr] = scale4(gamma, hv[rr]);
      const uint16_t* rkp = a.rk + sh * L * GD + lane * 4;
      for (int t0 = 0; t0 < count; t0 += 2) {  // e_t rows from shared memory (a broadcast read)
        float4 kt[2];
#pragma unroll
        for (int u = 0; u < 2; u++) {
          int s = start + t0 + u;
          s = s < L ? s : s - L;
          kt[u] = t0 + u < count ? load_bf4(rkp + s * GD) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 2; u++) {
          const int t = t0 + u;
          const float c = __shfl_sync(FULL, Dt, t & 31);
          if (t < count) {  // uniform
            const float4 ea2 = ld4(es + t * ES + rl), eb2 = ld4(es + t * ES + rl + 4);
            const float et[8] = {ea2.x, ea2.y, ea2.z, ea2.w, eb2.x, eb2.y, eb2.z, eb2.w};
#pragma unroll
            for (int rr = 0; rr < 8; rr++) hv[rr] = fma4(c * et[rr], kt[u], hv[rr]);
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < 8; rr++) hv[rr] = fma4(__shfl_sync(FULL, ec, 2 * rr), bf4_to_f4(kraw), hv[rr]);  // current, D = 1
#pragma unroll
      for (int rr = 0; rr < 8; rr++) __stcs(reinterpret_cast<float4*>(a.S + tbase + (size_t)(rl + rr) * GD) + lane, hv[rr]);
    }
  }
  if (threadIdx.x == 0) finish_ar_cursor(a.cursors, sb, cur_s, ticket, a.H * 2, L, a.status);
}

}  // namespace

bool gdn_step_fast_applies(const GdnArgs& a) {
  return a.DK == GD && a.DV == GD && a.L <= FW * KW - 1 && a.H * 2 < (1 << 15) && a.H <= 65535 &&
         a.Bt <= 65535 && a.Sn <= 65535;
}

cudaError_t gdn_step_fast_launch(const GdnArgs& a, int out_bf16, cudaStream_t st) {
  if (a.Bt == 0) return cudaSuccess;
  auto pick = [&](auto kwt) {
    constexpr int W = decltype(kwt)::value;
    return a.slots ? (out_bf16 ? gdn_step_fast_kernel<true, true, W> : gdn_step_fast_kernel<false, true, W>)
                   : (out_bf16 ? gdn_step_fast_kernel<true, false, W> : gdn_step_fast_kernel<false, false, W>);
  };
  auto k = a.L <= FW * KW_SHORT ? pick(std::integral_constant<int, KW_SHORT>{}) : pick(std::integral_constant<int, KW>{});
  const int smem = (FPB * GD + a.L * ES) * 4;
  cudaError_t e = prepare(k, smem, true);
  if (e != cudaSuccess) return e;
  k<<<dim3(2, a.H, a.Bt), FT, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace rssm
