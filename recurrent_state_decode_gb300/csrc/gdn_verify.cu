// Speculative verify for Gated DeltaNet ("How ReplaySSM works": drafts are
// appended to the buffer and verified output-only; "ReplaySSM" repository,
// introduction: rollback by moving a pointer). Generic kernel for any
// dk, dv <= 256; the epilogue kernel appends the new records' shared fields.
//
// Records of a verify are indexed t in [0, count + K): t < count the committed
// window (ring slot (start + t) mod L), then the K new ones. With G_t = sum_{j<=t}
// g_j and D(a, t) = exp(G_a - G_t), relative to the checkpoint S0:
//   e_t   = beta_t (v_t - e^{G_t} S0 k_t - sum_{s<t} D(t, s) (k_s . k_t) e_s)
//   o_i   = e^{G_a} S0 q_i + sum_{t<=a} D(a, t) (k_t . q_i) e_t,   a = count + i
// The committed records' e_t are read from the ring (they do not change until
// their flush); the new records' are solved here and appended. If count + K > L
// the committed window is folded first, S0' = e^{G_{c-1}} S0 + sum_{t<c}
// D(c-1, t) e_t k_t^T (c = count), written once; the outputs are the same
// whether computed from S0 with every record or from S0' with the new ones.
#include "gdn_common.cuh"
#include "kernels.h"

namespace rssm {

namespace {

constexpr int GV_THREADS = 128;
constexpr int GV_MAXR = 64;  // records in view: L + K <= 2 * RSSM_MAX_BUF_LEN

// Row `r` of record t's key (t < count: ring slot; else new record t - count).
__device__ __forceinline__ const uint16_t* key_of(const GdnArgs& a, size_t bh, int b, int h, int t, int start,
                                                  int count) {
  if (t < count) return a.rk + (bh * a.L + wrap(start + t, a.L)) * a.DK;
  return a.k + (((size_t)b * a.K + (t - count)) * a.H + h) * a.DK;
}

}  // namespace

// One block per (sequence, head); thread i owns state rows i, i + 128, ...
template <bool OUT_BF16>
__global__ void __launch_bounds__(GV_THREADS) gdn_verify_kernel(GdnArgs a) {
  __shared__ float Gs[GV_MAXR];            // G_t
  __shared__ float kk[GV_MAXR * 32];       // (k_t . k_j), [t * K + j], j < K
  __shared__ float kq[GV_MAXR * 32];       // (k_t . q_i), [t * K + i]
  __shared__ float bs[32];                 // beta of the new records
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x % a.H, b = blockIdx.x / a.H;
  const int L = a.L, K = a.K, DK = a.DK, DV = a.DV;
  const size_t bh = (size_t)b * a.H + h;
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)b);
  if (!(cur.x >= 0 && cur.x < L && cur.y >= 0 && cur.y <= L && cur.z == 0)) return;  // reported by the epilogue
  const int start = cur.x, count = cur.y, total = count + K;
  const bool fold = total > L;
  if (tid == 0) {
    float acc = 0.f;
    for (int t = 0; t < total; t++) {
      acc += t < count ? a.rg[bh * pad4(L) + wrap(start + t, L)] : a.g[((size_t)b * K + (t - count)) * a.H + h];
      Gs[t] = acc;
    }
  }
  if (tid < K) bs[tid] = a.beta[((size_t)b * K + tid) * a.H + h];
  // dots: one warp per (t, j) pair, lanes over dk
  for (int it = warp; it < total * K; it += GV_THREADS / 32) {
    const int t = it / K, j = it - t * K;
    const uint16_t* kt = key_of(a, bh, b, h, t, start, count);
    const uint16_t* kj = a.k + (((size_t)b * K + j) * a.H + h) * DK;
    const uint16_t* qj = a.q + (((size_t)b * K + j) * a.H + h) * DK;
    float sk = 0.f, sq = 0.f;
    for (int c = lane; c < DK; c += 32) {
      const float x = bf_to_f(kt[c]);
      sk = fmaf(x, bf_to_f(kj[c]), sk);
      sq = fmaf(x, bf_to_f(qj[c]), sq);
    }
    sk = warp_sum(sk);
    sq = warp_sum(sq);
    if (lane == 0) {
      kk[t * K + j] = sk;
      kq[t * K + j] = sq;
    }
  }
  __syncthreads();
  const float* S0 = a.S + bh * DV * DK;
  for (int r = tid; r < DV; r += GV_THREADS) {
    const float* row = S0 + (size_t)r * DK;
    float e[GV_MAXR];
    for (int t = 0; t < count; t++) e[t] = a.re[(bh * L + wrap(start + t, L)) * DV + r];
    // new records in order
    for (int j = 0; j < K; j++) {
      const int t = count + j;
      const uint16_t* kj = a.k + (((size_t)b * K + j) * a.H + h) * DK;
      float u = 0.f;
      for (int c = 0; c < DK; c++) u = fmaf(row[c], bf_to_f(kj[c]), u);
      float rhs = bf_to_f(a.v[(((size_t)b * K + j) * a.H + h) * DV + r]) - expf(Gs[t]) * u;
      for (int s = 0; s < t; s++) rhs -= expf(Gs[t] - Gs[s]) * kk[s * K + j] * e[s];
      e[t] = bs[j] * rhs;
    }
    for (int i = 0; i < K; i++) {
      const int t = count + i;
      const uint16_t* qi = a.q + (((size_t)b * K + i) * a.H + h) * DK;
      float w = 0.f;
      for (int c = 0; c < DK; c++) w = fmaf(row[c], bf_to_f(qi[c]), w);
      float o = expf(Gs[t]) * w;
      for (int s = 0; s <= t; s++) o = fmaf(expf(Gs[t] - Gs[s]) * kq[s * K + i], e[s], o);
      const size_t oi = (((size_t)b * K + i) * a.H + h) * DV + r;
      if (OUT_BF16)
        reinterpret_cast<uint16_t*>(a.o)[oi] = f_to_bf(o);
      else
        reinterpret_cast<float*>(a.o)[oi] = o;
    }
    if (fold) {  // committed window into the checkpoint, this row, written once
      const float Pf = expf(Gs[count - 1]);
      float* orow = a.S + (bh * DV + r) * DK;
      for (int c = 0; c < DK; c++) {
        float acc = Pf * row[c];
        for (int t = 0; t < count; t++)
          acc = fmaf(expf(Gs[count - 1] - Gs[t]) * e[t], bf_to_f(key_of(a, bh, b, h, t, start, count)[c]), acc);
        orow[c] = acc;  // each element read above by this thread only
      }
    }
    // the new records' e and v rows of this row
    for (int j = 0; j < K; j++) {
      const size_t slot = bh * L + wrap(wrap(start + count + j, L), L);
      a.re[slot * DV + r] = e[count + j];
      a.rv[slot * DV + r] = a.v[(((size_t)b * K + j) * a.H + h) * DV + r];
    }
  }
}

// One block per sequence, after the verify in stream order.
__global__ void __launch_bounds__(GV_THREADS) gdn_verify_epilogue_kernel(GdnArgs a) {
  const int4 c = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)blockIdx.x);
  gdn_verify_epilogue(a, blockIdx.x, blockIdx.x, c, c.w);
}

cudaError_t gdn_verify_launch(const GdnArgs& a, int out_bf16, cudaStream_t st) {
  if (a.Bt == 0) return cudaSuccess;
  if (gdn_verify_fast_applies(a)) return gdn_verify_fast_launch(a, out_bf16, st);
  if (out_bf16)
    gdn_verify_kernel<true><<<a.Bt * a.H, GV_THREADS, 0, st>>>(a);
  else
    gdn_verify_kernel<false><<<a.Bt * a.H, GV_THREADS, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  gdn_verify_epilogue_kernel<<<a.Bt, GV_THREADS, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace rssm
