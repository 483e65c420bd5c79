// Gated DeltaNet decode kernels for sm_103a: conventional step (comparison
// point), ReplaySSM AR step with the fused flush, standalone flush.
//
// Replay algebra (from S_t = alpha_t S_{t-1} + e_t k_t^T with
// e_t = beta_t (v_t - alpha_t S_{t-1} k_t); "How ReplaySSM works"): window
// records t = 0..m-1 (the last is current), D(t, s) = exp(sum_{s<j<=t} g_j),
// gamma_t = exp(sum_{j<=t} g_j), u_t = S0 k_t:
//   e_t = beta_t v_t - beta_t gamma_t u_t - sum_{s<t} beta_t D(t,s) (k_s . k_t) e_s
//   o   = gamma_{m-1} S0 q + sum_t D(m-1, t) (k_t . q) e_t
//   S_m = gamma_{m-1} S0 + sum_t D(m-1, t) e_t k_t^T          (flush only)
// Every D(t, s) is a sum of the g terms it spans (no prefix differences).
//
// Work unit: one CTA of 256 threads per (sequence, head, block of 64 state
// rows). Thread (warp w, lane l) owns row 8w + l/4 and the column quarter
// q = l%4: float4 chunks c = 4j + q, j < NJ. The rows of each warp arrive by
// their own bulk copy (TMA, non-tensor) on their own mbarrier.
#include "common.cuh"
#include "kernels.h"

namespace rssm {

constexpr int GDN_THREADS = 256;
constexpr int GDN_RB = 64;  // state rows per block

struct GdnSmem {
  float* tile;  // [RB, DK]
  float* ks;    // [L, DK]
  float* qv;    // [DK]
  float* vs;    // [L, RB]
  float* es;    // [L, RB]
  float* sg;    // [L]
  float* sb;    // [L]
  float* kk;    // [L, L]  kk[s*L + t] = k_s . k_t (s < t)
  float* kq;    // [L]
  float* Mts;   // [L, L]  Mts[t*L + s] = beta_t D(t,s) kk(s,t)
  float* bg;    // [L]     beta_t gamma_t
  float* oc;    // [L]     D(m-1,t) (k_t . q)
  float* fc;    // [L]     D(m-1,t)
  float* misc;  // [4]     gamma_{m-1}
  uint64_t* bars;  // [8]
};

__host__ __device__ inline size_t gdn_smem_layout(int RB, int DK, int L, unsigned char* base, GdnSmem* s) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align16(off + bytes);
    return o;
  };
  size_t o_tile = take((size_t)RB * DK * 4), o_ks = take((size_t)L * DK * 4), o_q = take((size_t)DK * 4);
  size_t o_vs = take((size_t)L * RB * 4), o_es = take((size_t)L * RB * 4);
  size_t o_g = take(L * 4), o_b = take(L * 4), o_kk = take(L * L * 4), o_kq = take(L * 4);
  size_t o_M = take(L * L * 4), o_bg = take(L * 4), o_oc = take(L * 4), o_fc = take(L * 4), o_misc = take(16);
  size_t o_bar = take(8 * 8);
  if (s) {
    s->tile = (float*)(base + o_tile);
    s->ks = (float*)(base + o_ks);
    s->qv = (float*)(base + o_q);
    s->vs = (float*)(base + o_vs);
    s->es = (float*)(base + o_es);
    s->sg = (float*)(base + o_g);
    s->sb = (float*)(base + o_b);
    s->kk = (float*)(base + o_kk);
    s->kq = (float*)(base + o_kq);
    s->Mts = (float*)(base + o_M);
    s->bg = (float*)(base + o_bg);
    s->oc = (float*)(base + o_oc);
    s->fc = (float*)(base + o_fc);
    s->misc = (float*)(base + o_misc);
    s->bars = (uint64_t*)(base + o_bar);
  }
  return off;
}

__device__ __forceinline__ void bf_row_to_smem(float* dst, const uint16_t* src, int n, int tid, int nthreads) {
  for (int i = tid; i < (n >> 3); i += nthreads) {
    const uint4 u = *reinterpret_cast<const uint4*>(src + i * 8);
    reinterpret_cast<float4*>(dst + i * 8)[0] = make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
    reinterpret_cast<float4*>(dst + i * 8)[1] = make_float4(bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w));
  }
}

// ------------------------------------------------------------------ conventional

template <int NJ, bool OUT_BF16>
__global__ void __launch_bounds__(GDN_THREADS) gdn_conventional_kernel(GdnArgs a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nRB = (a.DV + GDN_RB - 1) / GDN_RB;
  int blk = blockIdx.x;
  const int rb = blk % nRB;
  blk /= nRB;
  const int h = blk % a.H, b = blk / a.H;
  const int DK = a.DK, DV = a.DV, NC = DK >> 2;
  const int row = rb * GDN_RB + warp * 8 + (lane >> 2), q4 = lane & 3;
  const bool active = row < DV;  // whole quads share `active`
  const size_t bh = (size_t)b * a.H + h;
  const float alpha = expf(a.g[bh]), beta = a.beta[bh];
  float* Srow = a.S + (bh * DV + (active ? row : 0)) * DK;
  const uint16_t* kp = a.k + bh * DK;
  const uint16_t* qp = a.q + bh * DK;

  float4 sv[NJ];
  float u = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; j++) {
    const int c = 4 * j + q4;
    sv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active && c < NC) {
      sv[j] = __ldcs(reinterpret_cast<const float4*>(Srow) + c);
      u += dot4(sv[j], load_bf4(kp + c * 4));
    }
  }
  u = quad_sum(u);
  const float vi = active ? bf_to_f(a.v[bh * DV + row]) : 0.f;
  const float e = beta * (vi - alpha * u);
  float o = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; j++) {
    const int c = 4 * j + q4;
    if (active && c < NC) {
      const float4 kc = load_bf4(kp + c * 4);
      const float4 sn = fma4(e, kc, scale4(alpha, sv[j]));
      __stcs(reinterpret_cast<float4*>(Srow) + c, sn);
      o += dot4(sn, load_bf4(qp + c * 4));
    }
  }
  o = quad_sum(o);
  if (active && q4 == 0) store_out<OUT_BF16>(a.o, bh * DV + row, o);
}

// ------------------------------------------------------------------ replay step / flush

// MODE GDN_STEP: the AR step (window = committed + current; the current
// record's e_t goes to the ring unless the step flushes). GDN_FLUSH: the
// standalone flush (window = the count committed records, no output, no
// append). GDN_PRIME: e_t of the count committed records into the ring, no
// output, no state written.
template <int NJ, bool OUT_BF16, int MODE>
__global__ void __launch_bounds__(GDN_THREADS) gdn_replay_kernel(GdnArgs a) {
  constexpr bool FLUSH_ONLY = MODE != GDN_STEP;  // window without a current record
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nRB = (a.DV + GDN_RB - 1) / GDN_RB;
  int blk = blockIdx.x;
  const int rb = blk % nRB;
  blk /= nRB;
  const int h = blk % a.H, b = blk / a.H;
  const int DK = a.DK, DV = a.DV, L = a.L, NC = DK >> 2;
  const int i0 = rb * GDN_RB, R = min(GDN_RB, DV - i0);
  const size_t bh = (size_t)b * a.H + h;

  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)b);
  const int start = cur.x, count = cur.y;
  int m;
  bool flush;
  if (FLUSH_ONLY) {
    if (start < 0 || start >= L || count <= 0 || count > L || cur.z != 0) return;
    m = count;
    flush = MODE == GDN_FLUSH;
  } else {
    if (start < 0 || start >= L || count < 0 || count >= L || cur.z != 0) return;
    m = count + 1;
    flush = (m == L);
  }

  GdnSmem s;
  gdn_smem_layout(GDN_RB, DK, L, smem_raw, &s);
  if (tid == 0) {
    for (int w = 0; w < 8; w++) mbar_init(&s.bars[w], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const size_t tile_off = (bh * DV + i0) * DK;
  if (tid == 0) {
    for (int w = 0; w < 8; w++) {
      const int r0 = w * 8, r1 = min(R, r0 + 8);
      if (r1 > r0) {
        const uint32_t bytes = (uint32_t)((r1 - r0) * DK * 4);
        mbar_arrive_expect_tx(&s.bars[w], bytes);
        bulk_load(s.tile + (size_t)r0 * DK, a.S + tile_off + (size_t)r0 * DK, bytes, &s.bars[w]);
      }
    }
  }

  // window records
  for (int t = 0; t < m; t++) {
    const bool ring = t < count;
    const size_t slot = bh * L + (start + t) % L;
    bf_row_to_smem(s.ks + (size_t)t * DK, ring ? a.rk + slot * DK : a.k + bh * DK, DK, tid, GDN_THREADS);
    bf_row_to_smem(s.vs + (size_t)t * GDN_RB, (ring ? a.rv + slot * DV : a.v + bh * DV) + i0, R, tid,
                   GDN_THREADS);
  }
  if (!FLUSH_ONLY) bf_row_to_smem(s.qv, a.q + bh * DK, DK, tid, GDN_THREADS);
  if (tid < m) {
    const bool ring = tid < count;
    const size_t sslot = bh * pad4(L) + (start + tid) % L;
    s.sg[tid] = ring ? a.rg[sslot] : a.g[bh];
    s.sb[tid] = ring ? a.rbeta[sslot] : a.beta[bh];
  }
  if (!FLUSH_ONLY && !flush) {  // append the current record
    const size_t slot = bh * L + (start + count) % L;
    for (int i = tid; i < (R >> 3); i += GDN_THREADS)
      *reinterpret_cast<uint4*>(a.rv + slot * DV + i0 + i * 8) =
          *reinterpret_cast<const uint4*>(a.v + bh * DV + i0 + i * 8);
    if (rb == 0) {
      for (int i = tid; i < (DK >> 3); i += GDN_THREADS) {
        *reinterpret_cast<uint4*>(a.rk + slot * DK + i * 8) = *reinterpret_cast<const uint4*>(a.k + bh * DK + i * 8);
        *reinterpret_cast<uint4*>(a.rq + slot * DK + i * 8) = *reinterpret_cast<const uint4*>(a.q + bh * DK + i * 8);
      }
      if (tid == 0) {
        const size_t sslot = bh * pad4(L) + (start + count) % L;
        a.rg[sslot] = a.g[bh];
        a.rbeta[sslot] = a.beta[bh];
      }
    }
  }
  __syncthreads();

  // Gram entries k_s . k_t (s < t) and k_t . q: item (s, t), s == m meaning q
  for (int it = tid; it < (m + 1) * m; it += GDN_THREADS) {
    const int sidx = it / m, t = it - sidx * m;
    if (sidx >= t && sidx != m) continue;
    if (FLUSH_ONLY && sidx == m) continue;
    const float* x0 = (sidx == m) ? s.qv : s.ks + (size_t)sidx * DK;
    const float* x1 = s.ks + (size_t)t * DK;
    float acc = 0.f;
    for (int i = 0; i < NC; i++) {
      const int c = (i + lane) % NC;  // stagger lanes across banks
      acc += dot4(reinterpret_cast<const float4*>(x0)[c], reinterpret_cast<const float4*>(x1)[c]);
    }
    if (sidx == m)
      s.kq[t] = acc;
    else
      s.kk[sidx * L + t] = acc;
  }
  __syncthreads();
  // coefficients; thread t < m owns record t
  if (tid < m) {
    const int t = tid;
    const float bt = s.sb[t];
    float acc = 0.f;  // sum_{s<j<=t} g_j, growing as s goes down
    for (int sidx = t - 1; sidx >= 0; sidx--) {
      acc += s.sg[sidx + 1];
      s.Mts[t * L + sidx] = bt * expf(acc) * s.kk[sidx * L + t];
    }
    acc += s.sg[0];  // now sum_{j<=t} g_j
    s.bg[t] = bt * expf(acc);
    float tail = 0.f;  // sum_{t<j<=m-1} g_j
    for (int j = t + 1; j < m; j++) tail += s.sg[j];
    const float d = expf(tail);
    s.fc[t] = d;
    if (!FLUSH_ONLY) s.oc[t] = d * s.kq[t];
    if (t == m - 1) s.misc[0] = expf(acc);
  }
  __syncthreads();

  const int rloc = warp * 8 + (lane >> 2), q4 = lane & 3;
  if (warp * 8 >= R) return;  // whole warp idle (R is a multiple of 8)
  if (!mbar_wait_or_report(&s.bars[warp], 0, a.status)) return;
  float4 sv[NJ];
#pragma unroll
  for (int j = 0; j < NJ; j++) {
    const int c = 4 * j + q4;
    sv[j] = (c < NC) ? reinterpret_cast<const float4*>(s.tile + (size_t)rloc * DK)[c] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float* es_row = s.es + rloc;
  for (int t = 0; t < m; t++) {
    float u = 0.f;
    const float4* kt = reinterpret_cast<const float4*>(s.ks + (size_t)t * DK);
#pragma unroll
    for (int j = 0; j < NJ; j++) {
      const int c = 4 * j + q4;
      if (c < NC) u += dot4(sv[j], kt[c]);
    }
    u = quad_sum(u);
    float e = s.sb[t] * s.vs[(size_t)t * GDN_RB + rloc] - s.bg[t] * u;
    for (int sidx = 0; sidx < t; sidx++) e = fmaf(-s.Mts[t * L + sidx], es_row[(size_t)sidx * GDN_RB], e);
    __syncwarp();
    if (q4 == 0) {
      es_row[(size_t)t * GDN_RB] = e;
      // the ring keeps e of every record it holds: all of them when priming,
      // the current one on a non-flush step
      if (MODE == GDN_PRIME || (MODE == GDN_STEP && !flush && t == m - 1))
        a.re[(bh * L + (start + t) % L) * DV + i0 + rloc] = e;
    }
    __syncwarp();
  }
  const float gm = s.misc[0];
  if (!FLUSH_ONLY) {
    float w = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; j++) {
      const int c = 4 * j + q4;
      if (c < NC) w += dot4(sv[j], reinterpret_cast<const float4*>(s.qv)[c]);
    }
    w = quad_sum(w);
    float o = gm * w;
    for (int t = 0; t < m; t++) o = fmaf(s.oc[t], es_row[(size_t)t * GDN_RB], o);
    if (q4 == 0) store_out<OUT_BF16>(a.o, bh * DV + i0 + rloc, o);
  }
  if (flush) {
#pragma unroll
    for (int j = 0; j < NJ; j++) sv[j] = scale4(gm, sv[j]);
    for (int t = 0; t < m; t++) {
      const float ce = s.fc[t] * es_row[(size_t)t * GDN_RB];
      const float4* kt = reinterpret_cast<const float4*>(s.ks + (size_t)t * DK);
#pragma unroll
      for (int j = 0; j < NJ; j++) {
        const int c = 4 * j + q4;
        if (c < NC) sv[j] = fma4(ce, kt[c], sv[j]);
      }
    }
    float* dst = a.S + tile_off + (size_t)rloc * DK;
#pragma unroll
    for (int j = 0; j < NJ; j++) {
      const int c = 4 * j + q4;
      if (c < NC) __stcs(reinterpret_cast<float4*>(dst) + c, sv[j]);
    }
  }
}

namespace {
template <typename Kern>
cudaError_t launch_gdn(Kern k, int grid, size_t smem, cudaStream_t st, const GdnArgs& a) {
  cudaError_t e = prepare(k, smem, false);
  if (e != cudaSuccess) return e;
  k<<<grid, GDN_THREADS, smem, st>>>(a);
  return cudaGetLastError();
}
}  // namespace

#define RSSM_DISPATCH_NJ(NJ_, ...) \
  if (a.DK <= 128) {               \
    constexpr int NJ_ = 8;         \
    __VA_ARGS__                    \
  } else {                         \
    constexpr int NJ_ = 16;        \
    __VA_ARGS__                    \
  }

cudaError_t gdn_launch(int kind, const GdnArgs& a, int out_bf16, cudaStream_t st) {
  const int nRB = (a.DV + GDN_RB - 1) / GDN_RB;
  const int grid = a.Bt * a.H * nRB;
  if (grid == 0) return cudaSuccess;
  const size_t smem = gdn_smem_layout(GDN_RB, a.DK, a.L, nullptr, nullptr);
  cudaError_t e = cudaSuccess;
  switch (kind) {
    case GDN_CONVENTIONAL:
      RSSM_DISPATCH_NJ(NJ, {
        e = out_bf16 ? launch_gdn(gdn_conventional_kernel<NJ, true>, grid, 0, st, a)
                     : launch_gdn(gdn_conventional_kernel<NJ, false>, grid, 0, st, a);
      })
      return e;
    case GDN_STEP:
      if (gdn_step_fast_applies(a)) return gdn_step_fast_launch(a, out_bf16, st);
      RSSM_DISPATCH_NJ(NJ, {
        e = out_bf16 ? launch_gdn(gdn_replay_kernel<NJ, true, GDN_STEP>, grid, smem, st, a)
                     : launch_gdn(gdn_replay_kernel<NJ, false, GDN_STEP>, grid, smem, st, a);
      })
      return e;
    case GDN_FLUSH:
      RSSM_DISPATCH_NJ(NJ, { e = launch_gdn(gdn_replay_kernel<NJ, false, GDN_FLUSH>, grid, smem, st, a); })
      return e;
    case GDN_PRIME:
      RSSM_DISPATCH_NJ(NJ, { e = launch_gdn(gdn_replay_kernel<NJ, false, GDN_PRIME>, grid, smem, st, a); })
      return e;
  }
  return cudaErrorInvalidValue;
}

}  // namespace rssm
