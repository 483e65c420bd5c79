// ReplaySSM AR decode step for Kimi Delta Attention (KDA), shape-specialised:
// dk = dv = 128, L <= 31 ("How ReplaySSM works": non-flush steps read the
// checkpoint and the window and write no state; the L-th step folds the window
// and writes the state once). KDA is the gated delta rule with one decay per
// key channel, alpha = exp(g), g [dk].
//
// Algebra (S_t = S_{t-1} Diag(alpha_t) + e_t k_t^T with e_t = beta_t (v_t -
// S_{t-1} (alpha_t * k_t)), * channel-wise). Window records t = 0..m-1 (the
// last is the current one); f_t = exp(sum_{t<j<=m-1} g_j), a vector over the
// channels (f_{m-1} = 1), and Gamma = exp(sum_{j<=m-1} g_j):
//   e_cur = beta (v - S0 (Gamma * k) - sum_{t<m-1} ((f_t * k_t) . k) e_t)
//   o     = S0 (Gamma * q) + sum_{t<m-1} ((f_t * k_t) . q) e_t + (k . q) e_cur
//   S_m   = S0 Diag(Gamma) + sum_{t<=m-1} e_t (f_t * k_t)^T          (flush only)
// e_t of a committed record depends on S0 and earlier records only, so it is
// read from the ring (written when the record was current).
//
// One CTA of four warps per (sequence, head, 64 state rows), laid out as the
// Gated DeltaNet step: warp w owns rows 8w..8w+7 and 32+8w..32+8w+7, lane l
// the column chunk 4l..4l+3. At launch: the 64 rows by one bulk copy (TMA,
// non-tensor; never multicast) into shared memory, the current record, and
// the ring keys of the slots whose dots the warp forms. As soon as the cursor
// arrives, the block's threads copy the window records' e rows of this block
// and their g rows (16-byte asynchronous copies spread over the threads); thread c then
// runs the suffix sums of channel c backwards over the window, leaving f_t in
// place of g_t, and Gamma. Warp w forms (f_s * k_s) . k and (f_s * k_s) . q
// for ring slots w, w+4, ... (slot L: the current k), one transposed
// reduction. Per 8-row group one transposed 16-value reduction gives
// S0 (Gamma * k) and S0 (Gamma * q) plus the window terms. The last of a
// sequence's blocks to have read its cursor advances it.
#include <type_traits>

#include "fast_rows.cuh"
#include "kernels.h"

namespace rssm {

namespace {

using namespace fastrows;

constexpr int GD = 128;      // dk = dv
constexpr int KW = 8;        // dot entries per warp: 4 x 8 >= L + 1
// With L <= 16 four ring slots per warp cover the window, and the current
// record's k . q is one warp sum instead: half the dot work, an 8-wide reduction.
constexpr int KW_SHORT = 4;
constexpr int ES = FPB + 4;  // floats per staged e row (padded against bank conflicts; 16-byte multiple)

// SLOTS: batch rows name their state rows through a slot table.
// KWT: ring slots per warp in the dot table (KW, or KW_SHORT when L <= 16).
template <bool OUT_BF16, bool SLOTS, int KWT = KW>
__global__ void __launch_bounds__(FT, 5) kda_step_fast_kernel(GdnArgs a) {
  extern __shared__ __align__(128) float dsm[];
  const int L = a.L, H = a.H;
  // a step's window holds at most L - 1 committed records: staging for that many
  float* tile = dsm;                 // the block's 64 rows
  float* es = dsm + FPB * GD;        // e of window record t at es + t * ES (the block's rows)
  float* fd = es + (L - 1) * ES;     // g, then f, of window record t at fd + t * GD (all channels)
  __shared__ float skk[FW * KW], skq[FW * KW];  // (f_s * k_s) . k and . q by ring slot; [L] = current
  __shared__ __align__(16) float gam[GD];       // Gamma by channel
  __shared__ uint64_t bar;                      // the rows
  __shared__ int4 cur_s;                        // the cursor as read, for the sequence's last block
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
  // An invalid cursor (reported by the sequence's last block) runs as an empty
  // window with every store masked, so that no thread leaves before a barrier.
  const bool valid = cur.x >= 0 && cur.x < L && cur.y >= 0 && cur.y < L && cur.z == 0;
  const int start = valid ? cur.x : 0, count = valid ? cur.y : 0;
  // the window's e rows (this block's) and g rows, in record order, as soon as the cursor is known: 16-byte
  // asynchronous copies spread over the threads
  for (int c = threadIdx.x; c < count * ((FPB + GD) / 4); c += FT) {
    const int t = c / ((FPB + GD) / 4), j = c - t * ((FPB + GD) / 4);
    const size_t row = sh * L + wrap(start + t, L);
    float* dst = j < FPB / 4 ? es + t * ES + 4 * j : fd + t * GD + 4 * (j - FPB / 4);
    const float* src = j < FPB / 4 ? a.re + row * GD + p0 + 4 * j : a.rg + row * GD + 4 * (j - FPB / 4);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  const int rl0 = warp * 8, rl1 = HALF + warp * 8;  // the warp's row groups (within the block)
  // the current record; thread c holds channel c of its log decay
  const uint2 kraw = *reinterpret_cast<const uint2*>(a.k + bh * GD + lane * 4);
  const uint2 qraw = *reinterpret_cast<const uint2*>(a.q + bh * GD + lane * 4);
  const float gc = a.g[bh * GD + threadIdx.x], bm = a.beta[bh];
  const int vr = (lane >> 1) & 7;  // the row this lane finishes (lanes 0..15)
  const uint16_t vbA = a.v[bh * GD + p0 + rl0 + vr], vbB = a.v[bh * GD + p0 + rl1 + vr];
  // ring keys of slots s = warp + 4 j (their decays are known once the cursor is)
  uint2 kr[KWT];
#pragma unroll
  for (int j = 0; j < KWT; j++) {
    const int s = warp + FW * j;
    kr[j] = s < L ? *reinterpret_cast<const uint2*>(a.rk + (sh * L + s) * GD + lane * 4) : make_uint2(0, 0);
  }
  int ticket = 0;
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();  // the barrier's initialisation is visible; every thread has read the cursor; the window's rows
  if (threadIdx.x == 0) {
    ticket = cursor_ticket(a.cursors, sb);
    cur_s = cur;
  }
  const int cnt = count;
  const bool live = valid;
  const int m = cnt + 1;
  const bool flush = live && m == L;
  const int scur = wrap(start + count, L);  // the current record's slot
  {  // channel suffix sums, backwards over the window: f_t = exp(sum_{t<j<=m-1} g_j)
    const int c = threadIdx.x;
    float acc = gc;
    for (int t = cnt - 1; t >= 0; t--) {
      const float x = fd[t * GD + c];
      fd[t * GD + c] = expf(acc);
      acc += x;
    }
    gam[c] = expf(acc);
  }
  __syncthreads();
  const float4 kc = bf4_to_f4(kraw), qc = bf4_to_f4(qraw);
  float kq_cur;  // k . q of the current record
  {  // (f_s * k_s) . k and (f_s * k_s) . q for ring slots s = warp + 4 j (s == L: the current k, with KW slots per warp)
    float pk[2 * KWT];
#pragma unroll
    for (int j = 0; j < KWT; j++) {
      const int s = warp + FW * j;
      int pos = s - start;
      pos = pos < 0 ? pos + L : pos;  // the slot's record index in the window
      float4 ks = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s < L && pos < cnt)
        ks = mul4(bf4_to_f4(kr[j]), ld4(fd + pos * GD + lane * 4));
      else if (KWT == KW && s == L)
        ks = kc;
      pk[2 * j] = dot4(ks, kc);
      pk[2 * j + 1] = dot4(ks, qc);
    }
    const float red = reduce_transpose<2 * KWT>(pk, lane);
    if (KWT == KW) {  // lane l: partial l >> 1 = (slot j = l >> 2, k or q)
      if ((lane & 1) == 0) ((lane & 2) ? skq : skk)[warp + FW * (lane >> 2)] = red;
      kq_cur = 0.f;
    } else {  // lane l: partial reduce8_row(l) = (slot j = index >> 1, k or q)
      const int idx = reduce8_row(lane);
      if ((lane & 3) == 0) ((idx & 1) ? skq : skk)[warp + FW * (idx >> 1)] = red;
      kq_cur = warp_sum(dot4(kc, qc));
    }
  }
  __syncthreads();
  int sl = start + lane;
  sl = sl < L ? sl : sl - L;
  const float cK = lane < cnt ? skk[sl] : 0.f;  // lane t: record t's coefficients
  const float cQ = lane < cnt ? skq[sl] : 0.f;
  if (KWT == KW) kq_cur = skq[L];
  const float4 gm4 = ld4(gam + lane * 4);
  const float4 ka = mul4(gm4, kc), qa = mul4(gm4, qc);
  // Append the current record now (its e follows below): its slot is outside
  // the window, so no block reads it for a result.
  if (live && !flush) {
    const size_t vrow = (sh * L + scur) * GD + p0 + vr;
    if (lane < 16 && (lane & 1) == 0) {
      a.rv[vrow + rl0] = vbA;
      a.rv[vrow + rl1] = vbB;
    }
    if (pb == 0) {
      a.rg[(sh * L + scur) * GD + threadIdx.x] = gc;
      if (warp == 0) {
        const size_t krow = (sh * L + scur) * GD + lane * 4;
        *reinterpret_cast<uint2*>(a.rk + krow) = kraw;
        *reinterpret_cast<uint2*>(a.rq + krow) = qraw;
        if (lane == 0) a.rbeta[sh * pad4(L) + scur] = bm;
      }
    }
  }
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
    if (lane < cnt) {
      ea = ld4(es + lane * ES + rl);
      eb = ld4(es + lane * ES + rl + 4);
    }
    const float el[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
    float4 hv[8];
#pragma unroll
    for (int rr = 0; rr < 8; rr++) hv[rr] = ld4(tile + (rl + rr) * GD + lane * 4);
    float tk[8], tq[8];
#pragma unroll
    for (int rr = 0; rr < 8; rr++) {
      tk[rr] = cK * el[rr];
      tq[rr] = cQ * el[rr];
    }
    // lanes 0..15: S0 (Gamma * k) + k-term of row vr; lanes 16..31: the q counterpart
    const float tot = rows8x2(hv, ka, qa, tk, tq, lane);
    const float yq = __shfl_down_sync(FULL, tot, 16);
    const float ec = bm * (bf_to_f(half ? vbB : vbA) - tot);  // e of the current record, row vr (lanes < 16)
    if (live && lane < 16 && (lane & 1) == 0) {
      store_out<OUT_BF16>(a.o, bh * GD + p0 + rl + vr, fmaf(kq_cur, ec, yq));
      if (!flush) a.re[(sh * L + scur) * GD + p0 + rl + vr] = ec;
    }
    if (flush) {  // S_m = S0 Diag(Gamma) + sum_t e_t (f_t * k_t)^T, written once
#pragma unroll
      for (int rr = 0; rr < 8; rr++) hv[rr] = mul4(gm4, hv[rr]);
      const uint16_t* rkp = a.rk + sh * L * GD + lane * 4;
      for (int t0 = 0; t0 < cnt; t0 += 2) {
        float4 kt[2];
#pragma unroll
        for (int u = 0; u < 2; u++) {
          const int t = t0 + u;
          kt[u] = t < cnt ? mul4(load_bf4(rkp + wrap(start + t, L) * GD), ld4(fd + t * GD + lane * 4))
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 2; u++) {
          const int t = t0 + u;
          if (t < cnt) {  // uniform
            const float4 ea2 = ld4(es + t * ES + rl), eb2 = ld4(es + t * ES + rl + 4);
            const float et[8] = {ea2.x, ea2.y, ea2.z, ea2.w, eb2.x, eb2.y, eb2.z, eb2.w};
#pragma unroll
            for (int rr = 0; rr < 8; rr++) hv[rr] = fma4(et[rr], kt[u], hv[rr]);
          }
        }
      }
#pragma unroll
      for (int rr = 0; rr < 8; rr++) hv[rr] = fma4(__shfl_sync(FULL, ec, 2 * rr), kc, hv[rr]);  // current, f = 1
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
        __stcs(reinterpret_cast<float4*>(a.S + tbase + (size_t)(rl + rr) * GD) + lane, hv[rr]);
    }
  }
  if (threadIdx.x == 0) finish_ar_cursor(a.cursors, sb, cur_s, ticket, a.H * 2, L, a.status);
}

}  // namespace

bool kda_step_fast_applies(const GdnArgs& a) {
  return a.DK == GD && a.DV == GD && a.L <= FW * KW - 1 && a.H * 2 < (1 << 15) && a.H <= 65535 &&
         a.Bt <= 65535 && a.Sn <= 65535;
}

cudaError_t kda_step_fast_launch(const GdnArgs& a, int out_bf16, cudaStream_t st) {
  if (a.Bt == 0) return cudaSuccess;
  auto pick = [&](auto slots, auto kwt) {
    constexpr bool S = decltype(slots)::value;
    constexpr int W = decltype(kwt)::value;
    return out_bf16 ? kda_step_fast_kernel<true, S, W> : kda_step_fast_kernel<false, S, W>;
  };
  const bool short_window = a.L <= FW * KW_SHORT;
  auto k = a.slots ? (short_window ? pick(std::true_type{}, std::integral_constant<int, KW_SHORT>{})
                                   : pick(std::true_type{}, std::integral_constant<int, KW>{}))
                   : (short_window ? pick(std::false_type{}, std::integral_constant<int, KW_SHORT>{})
                                   : pick(std::false_type{}, std::integral_constant<int, KW>{}));
  const int smem = (FPB * GD + (a.L - 1) * (ES + GD)) * 4;  // five blocks per SM at L = 16
  cudaError_t e = prepare(k, smem, true);
  if (e != cudaSuccess) return e;
  k<<<dim3(2, a.H, a.Bt), FT, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace rssm
