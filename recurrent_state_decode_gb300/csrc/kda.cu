// Kimi Delta Attention (KDA) kernels besides the AR step: the conventional
// step (comparison point) and the window kernel behind the standalone flush
// and the prime. KDA is the gated delta rule with one decay per key channel:
// S <- S Diag(alpha) (I - beta k k^T) + beta v k^T, o = S q, alpha = exp(g).
//
// Window algebra ("How ReplaySSM works"; S_t = S_{t-1} Diag(alpha_t) + e_t k_t^T,
// e_t = beta_t (v_t - S_{t-1} (alpha_t * k_t))). For the count committed records
// t = 0..c-1 with channel-wise prefix sums G_t = sum_{j<=t} g_j:
//   e_t = beta_t (v_t - S0 (exp(G_t) * k_t) - sum_{i<t} ((exp(G_t - G_i) * k_i) . k_t) e_i)   (prime)
//   S_c = S0 Diag(exp(G_{c-1})) + sum_t e_t (exp(G_{c-1} - G_t) * k_t)^T                     (flush)
// Every exponent is a sum of g's over a later-minus-earlier range, so no
// exponential of a positive sum is taken.
#include "fast_rows.cuh"
#include "kernels.h"

namespace rssm {

namespace {

using namespace fastrows;

constexpr int KD = 128;           // dk = dv on the window kernel
constexpr int CONV_THREADS = 256;
constexpr int CONV_RB = 64;       // state rows per conventional block
constexpr int WMAX = 32;          // records in a window

__device__ __forceinline__ float4 exp4(float4 a) { return make_float4(expf(a.x), expf(a.y), expf(a.z), expf(a.w)); }

__device__ __forceinline__ float4 sub4(float4 a, float4 b) { return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w); }

// ------------------------------------------------------------------ conventional

// One block of 256 threads per (sequence, head, 64 state rows); thread (warp w,
// lane l) owns row 8w + l/4 and the column chunks c = 4j + l%4. The block's
// decays alpha = exp(g) are computed once into shared memory.
template <int NJ, bool OUT_BF16>
__global__ void __launch_bounds__(CONV_THREADS) kda_conventional_kernel(GdnArgs a) {
  __shared__ __align__(16) float alpha[2 * KD];  // dk <= 256
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nRB = (a.DV + CONV_RB - 1) / CONV_RB;
  int blk = blockIdx.x;
  const int rb = blk % nRB;
  blk /= nRB;
  const int h = blk % a.H, b = blk / a.H;
  const int DK = a.DK, DV = a.DV, NC = DK >> 2;
  const size_t bh = (size_t)b * a.H + h;
  for (int c = threadIdx.x; c < DK; c += CONV_THREADS) alpha[c] = expf(a.g[bh * DK + c]);
  __syncthreads();
  const int row = rb * CONV_RB + warp * 8 + (lane >> 2), q4 = lane & 3;
  const bool active = row < DV;  // whole quads share `active`
  const float beta = a.beta[bh];
  float* Srow = a.S + (bh * DV + (active ? row : 0)) * DK;
  const uint16_t* kp = a.k + bh * DK;
  const uint16_t* qp = a.q + bh * DK;
  float4 sv[NJ];  // S Diag(alpha), this thread's chunks
  float u = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; j++) {
    const int c = 4 * j + q4;
    sv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active && c < NC) {
      sv[j] = mul4(__ldcs(reinterpret_cast<const float4*>(Srow) + c), ld4(alpha + 4 * c));
      u += dot4(sv[j], load_bf4(kp + c * 4));
    }
  }
  u = quad_sum(u);
  const float vi = active ? bf_to_f(a.v[bh * DV + row]) : 0.f;
  const float e = beta * (vi - u);
  float o = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; j++) {
    const int c = 4 * j + q4;
    if (active && c < NC) {
      const float4 sn = fma4(e, load_bf4(kp + c * 4), sv[j]);
      __stcs(reinterpret_cast<float4*>(Srow) + c, sn);
      o += dot4(sn, load_bf4(qp + c * 4));
    }
  }
  o = quad_sum(o);
  if (active && q4 == 0) store_out<OUT_BF16>(a.o, bh * DV + row, o);
}

// ------------------------------------------------------------------ window: flush / prime

struct KdaWinSmem {
  float tile[FPB * KD];      // the block's 64 state rows
  float kw[WMAX * KD];       // window keys (fp32), record order
  float G[WMAX * KD];        // channel prefix sums of g, record order
  float es[WMAX * FPB];      // e of the block's rows, record order
  float us[WMAX * FPB];      // prime: S0 (exp(G_t) * k_t) of the block's rows
  float M[WMAX * WMAX];      // prime: M[t][i] = (exp(G_t - G_i) * k_i) . k_t, i < t
  uint64_t bar;
};

// One CTA of four warps per (sequence, head, 64 state rows), laid out as the
// shape-specialised step. MODE GDN_FLUSH folds the count committed records
// (their e from the ring) into S; GDN_PRIME solves their e and writes the ring.
template <int MODE>
__global__ void __launch_bounds__(FT) kda_window_kernel(GdnArgs a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  KdaWinSmem& s = *reinterpret_cast<KdaWinSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = a.L, pb = blockIdx.x, b = blockIdx.z;
  const size_t sh = (size_t)b * a.H + blockIdx.y;
  const int p0 = pb * FPB;
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)b);
  // uniform over the block; a bad cursor is reported by the flush's cursor kernel
  if (!(cur.x >= 0 && cur.x < L && cur.y > 0 && cur.y <= L && cur.z == 0)) return;
  const int start = cur.x, cnt = cur.y;
  auto slot = [&](int t) { return (start + t) % L; };
  const size_t tbase = (sh * KD + p0) * KD;
  if (tid == 0) {
    mbar_init(&s.bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&s.bar, FPB * KD * 4);
    bulk_load(s.tile, a.S + tbase, FPB * KD * 4, &s.bar);
  }
  {  // thread c: channel c of every window key and of the decay prefix sums
    const int c = tid;
    float acc = 0.f;
    for (int t = 0; t < cnt; t++) {
      const size_t row = sh * L + slot(t);
      acc += a.rg[row * KD + c];
      s.G[t * KD + c] = acc;
      s.kw[t * KD + c] = bf_to_f(a.rk[row * KD + c]);
    }
  }
  if (MODE == GDN_FLUSH)
    for (int i = tid; i < cnt * FPB; i += FT) {
      const int t = i / FPB, r = i - t * FPB;
      s.es[i] = a.re[(sh * L + slot(t)) * KD + p0 + r];
    }
  __syncthreads();
  const int rl0 = warp * 8, rl1 = HALF + warp * 8;
  if (MODE == GDN_PRIME) {
    // coupling table, one warp per (t, i) pair
    for (int it = warp; it < cnt * cnt; it += FW) {
      const int t = it / cnt, i = it - t * cnt;
      if (i >= t) continue;  // uniform over the warp
      const float4 kd = mul4(exp4(sub4(ld4(s.G + t * KD + 4 * lane), ld4(s.G + i * KD + 4 * lane))),
                             ld4(s.kw + i * KD + 4 * lane));
      const float p = warp_sum(dot4(kd, ld4(s.kw + t * KD + 4 * lane)));
      if (lane == 0) s.M[t * WMAX + i] = p;
    }
  }
  if (!__syncthreads_and(mbar_wait(&s.bar, 0))) {  // uniform over the block
    if (tid == 0) {
      report(a.status, RSSM_DEV_TIMEOUT);
      mbar_wait(&s.bar, 0);  // the copy lands before the block leaves
    }
    return;
  }
  if (MODE == GDN_FLUSH) {
    const float4 Gl = ld4(s.G + (cnt - 1) * KD + 4 * lane);
    const float4 gl = exp4(Gl);
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int rl = half ? rl1 : rl0;
      float4 hv[8];
#pragma unroll
      for (int rr = 0; rr < 8; rr++) hv[rr] = mul4(gl, ld4(s.tile + (rl + rr) * KD + 4 * lane));
      for (int t = 0; t < cnt; t++) {
        const float4 kt = mul4(exp4(sub4(Gl, ld4(s.G + t * KD + 4 * lane))), ld4(s.kw + t * KD + 4 * lane));
#pragma unroll
        for (int rr = 0; rr < 8; rr++) hv[rr] = fma4(s.es[t * FPB + rl + rr], kt, hv[rr]);
      }
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
        __stcs(reinterpret_cast<float4*>(a.S + tbase + (size_t)(rl + rr) * KD) + lane, hv[rr]);
    }
    return;
  }
  // prime: u_t = S0 (exp(G_t) * k_t) for the warp's rows
  for (int t = 0; t < cnt; t++) {
    const float4 kd = mul4(exp4(ld4(s.G + t * KD + 4 * lane)), ld4(s.kw + t * KD + 4 * lane));
#pragma unroll
    for (int half = 0; half < 2; half++) {
      const int rl = half ? rl1 : rl0;
      float v[8];
#pragma unroll
      for (int rr = 0; rr < 8; rr++) v[rr] = dot4(ld4(s.tile + (rl + rr) * KD + 4 * lane), kd);
      reduce8(v, lane);
      if ((lane & 3) == 0) s.us[t * FPB + rl + reduce8_row(lane)] = v[0];
    }
  }
  __syncthreads();
  // the corrections in record order, thread r < 64 owning row r
  if (tid < FPB) {
    const int r = tid;
    for (int t = 0; t < cnt; t++) {
      const size_t row = sh * L + slot(t);
      float rhs = bf_to_f(a.rv[row * KD + p0 + r]) - s.us[t * FPB + r];
      for (int i = 0; i < t; i++) rhs = fmaf(-s.M[t * WMAX + i], s.es[i * FPB + r], rhs);
      const float e = a.rbeta[sh * pad4(L) + slot(t)] * rhs;
      s.es[t * FPB + r] = e;
      a.re[row * KD + p0 + r] = e;
    }
  }
}

template <typename Kern>
cudaError_t launch_smem(Kern k, dim3 grid, int threads, size_t smem, cudaStream_t st, const GdnArgs& a) {
  cudaError_t e = prepare(k, smem, false);
  if (e != cudaSuccess) return e;
  k<<<grid, threads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool kda_window_applies(const GdnArgs& a) { return a.DK == KD && a.DV == KD && a.Bt <= 65535 && a.H <= 65535; }

cudaError_t kda_launch(int kind, const GdnArgs& a, int out_bf16, cudaStream_t st) {
  if (a.Bt == 0) return cudaSuccess;
  switch (kind) {
    case GDN_CONVENTIONAL: {
      const int nRB = (a.DV + CONV_RB - 1) / CONV_RB;
      const dim3 grid(a.Bt * a.H * nRB);
      if (a.DK <= 128)
        return out_bf16 ? launch_smem(kda_conventional_kernel<8, true>, grid, CONV_THREADS, 0, st, a)
                        : launch_smem(kda_conventional_kernel<8, false>, grid, CONV_THREADS, 0, st, a);
      return out_bf16 ? launch_smem(kda_conventional_kernel<16, true>, grid, CONV_THREADS, 0, st, a)
                      : launch_smem(kda_conventional_kernel<16, false>, grid, CONV_THREADS, 0, st, a);
    }
    case GDN_STEP:
      return kda_step_fast_launch(a, out_bf16, st);
    case GDN_FLUSH:
      return launch_smem(kda_window_kernel<GDN_FLUSH>, dim3(2, a.H, a.Bt), FT, sizeof(KdaWinSmem), st, a);
    case GDN_PRIME:
      return launch_smem(kda_window_kernel<GDN_PRIME>, dim3(2, a.H, a.Bt), FT, sizeof(KdaWinSmem), st, a);
  }
  return cudaErrorInvalidValue;
}

}  // namespace rssm
