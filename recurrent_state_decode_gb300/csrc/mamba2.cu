// Mamba-2 decode kernels for sm_103a: the conventional read-modify-write step
// (comparison point), the standalone flush and the speculative verify. The
// AR step with its fused flush lives in mamba2_step.cu.
//
// Work unit: one CTA of 128 threads per (sequence b, head h, row block) of the
// [headdim, dstate] state tile; a row block holds PB rows (PB*dstate*4 <= 32
// KiB, so one block is the whole tile for headdim 64 / dstate 128). Each warp
// owns a contiguous run of 8-row groups. In the replay kernels the tile is
// streamed into shared memory by bulk copies (one per warp, each on its own
// mbarrier) issued before anything else, so the HBM stream starts at once and
// every warp starts on its rows as soon as they land; the window records are
// read and reduced meanwhile.
//
// Replay algebra ("ReplaySSM Caches Inputs Instead of State...", "How
// ReplaySSM works"), window records k = 0..m-1 (the last is the current one),
// a_k = dt_k * A:
//   P_m = exp(sum_k a_k);  w_k = dt_k * exp(sum_{j>k} a_j)
//   y   = (P_m (h0 C_m) + sum_k w_k (B_k . C_m) x_k + D x_m) * silu(z_m)
//   h_m = P_m h0 + sum_k (w_k x_k) B_k^T            (flush only)
// The suffix sums come from one warp scan over the <= 32 records, so a decay
// weight is a sum of the exact terms it spans, not a difference of prefixes.

#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace rssm {

// ------------------------------------------------------------------ shared layout

struct M2Smem {
  float* tile;   // [PB, N] fp32 (or [PB, N] bf16 for a read-copy tile)
  float* Bs;     // [Lf, N]  B rows of the folded records (fp32)
  float* xs;     // [W, PB]  x rows of the window records (fp32), scaled by w_k before a fold
  float* xsum;   // [K, PB]  sum_k coef_k x_k per output
  float* sdt;    // [W]
  float* sc;     // [K, W]  B_k . C_i
  float* sw;     // [K+1, W] decay weights (row K = fold weights)
  float* scoef;  // [K, W]
  float* sP;     // [K+1]   P_m per output (+ fold)
  uint64_t* bars;  // [4]
};


// W = records held in shared memory, Lf = records folded, K = outputs.
__host__ __device__ inline size_t m2_smem_layout(int PB, int N, int W, int Lf, int K, unsigned char* base,
                                                 M2Smem* s) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align16(off + bytes);
    return o;
  };
  size_t o_tile = take((size_t)PB * N * 4);
  size_t o_Bs = take((size_t)Lf * N * 4);
  size_t o_xs = take((size_t)W * PB * 4);
  size_t o_xsum = take((size_t)K * PB * 4);
  size_t o_dt = take((size_t)W * 4);
  size_t o_sc = take((size_t)K * W * 4);
  size_t o_sw = take((size_t)(K + 1) * W * 4);
  size_t o_coef = take((size_t)K * W * 4);
  size_t o_P = take((size_t)(K + 1) * 4);
  size_t o_bar = take(4 * 8);
  if (s) {
    s->tile = (float*)(base + o_tile);
    s->Bs = (float*)(base + o_Bs);
    s->xs = (float*)(base + o_xs);
    s->xsum = (float*)(base + o_xsum);
    s->sdt = (float*)(base + o_dt);
    s->sc = (float*)(base + o_sc);
    s->sw = (float*)(base + o_sw);
    s->scoef = (float*)(base + o_coef);
    s->sP = (float*)(base + o_P);
    s->bars = (uint64_t*)(base + o_bar);
  }
  return off;
}

// ------------------------------------------------------------------ small device pieces

__device__ __forceinline__ int4 load_cursor(const int32_t* cursors, int b) {
  return *reinterpret_cast<const int4*>(cursors + 4 * (size_t)b);
}

// Rows [r0, r1) of warp w when the R rows of a block are split into 8-row
// groups dealt out contiguously to the four warps.
__device__ __forceinline__ void warp_rows(int R, int w, int& r0, int& r1) {
  const int ngrp = R >> 3;
  r0 = ((w * ngrp) >> 2) * 8;
  r1 = (((w + 1) * ngrp) >> 2) * 8;
}

// Issue the bulk copies of a row block (esz = 2 for bf16, 4 for fp32):
// one copy per warp's rows, each completing on that warp's barrier.
__device__ __forceinline__ void issue_tile(const M2Smem& s, const char* src, int R, int N, int esz) {
  for (int w = 0; w < 4; w++) {
    int r0, r1;
    warp_rows(R, w, r0, r1);
    if (r1 > r0) {
      const uint32_t bytes = (uint32_t)((r1 - r0) * N * esz);
      mbar_arrive_expect_tx(&s.bars[w], bytes);
      bulk_load((char*)s.tile + (size_t)r0 * N * esz, src + (size_t)r0 * N * esz, bytes, &s.bars[w]);
    }
  }
}

__device__ __forceinline__ void init_bars(const M2Smem& s) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < 4; i++) mbar_init(&s.bars[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
}

// Warp-wide decay weights of a window of m <= 32 records whose dt values are
// dts[0..m): w[k] = dts[k] * exp(A * sum_{j>k} dts[j]) and P = exp(A * sum dts).
// If c != nullptr, coef[k] = w[k] * c[k] as well.
__device__ __forceinline__ void window_weights(const float* dts, int m, float A, int lane, float* w,
                                               const float* c, float* coef, float* P) {
  const float dtk = (lane < m) ? dts[lane] : 0.f;
  float sfx = dtk * A;  // inclusive suffix sum over lanes lane..31
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_down_sync(FULL, sfx, o);
    if (lane + o < 32) sfx += t;
  }
  float ex = __shfl_down_sync(FULL, sfx, 1);
  if (lane == 31) ex = 0.f;
  const float tot = __shfl_sync(FULL, sfx, 0);
  if (lane < m) {
    const float wk = dtk * expf(ex);
    w[lane] = wk;
    if (c) coef[lane] = wk * c[lane];
  }
  if (lane == 0) *P = expf(tot);
}

// Load 8 consecutive bf16 as fp32 into shared memory.
__device__ __forceinline__ void bf8_to_smem(float* dst, const uint16_t* src) {
  const uint4 u = *reinterpret_cast<const uint4*>(src);
  float4 a = make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
  float4 b = make_float4(bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w));
  reinterpret_cast<float4*>(dst)[0] = a;
  reinterpret_cast<float4*>(dst)[1] = b;
}

__device__ __forceinline__ void copy8(uint16_t* dst, const uint16_t* src) {
  *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
}

template <int NCH>
__device__ __forceinline__ float4 tile_chunk(const M2Smem& s, bool rd16, int row, int N, int c) {
  if (rd16) return load_bf4(reinterpret_cast<const uint16_t*>(s.tile) + (size_t)row * N + c * 4);
  return reinterpret_cast<const float4*>(s.tile + (size_t)row * N)[c];
}

// Fold one 8-row group: h1 = P h0 + sum_k wx[k][r] B_k, for the lane's column
// chunks; h0 is given in registers. Writes fp32 (and bf16) rows to global and,
// if back != nullptr, the fp32 rows back to shared memory.
template <int NCH>
__device__ __forceinline__ void fold_group(float4 (&hv)[8][NCH], const M2Smem& s, int r0, int PB, int N, int m,
                                           float P, int lane, float* g32, uint16_t* g16, bool f16, float* back,
                                           uint8_t* q8 = nullptr, float* sc8 = nullptr, size_t row0 = 0) {
#pragma unroll
  for (int rr = 0; rr < 8; rr++)
#pragma unroll
    for (int j = 0; j < NCH; j++) hv[rr][j] = scale4(P, hv[rr][j]);
  for (int k = 0; k < m; k++) {
    const float4 wa = *reinterpret_cast<const float4*>(s.xs + (size_t)k * PB + r0);
    const float4 wb = *reinterpret_cast<const float4*>(s.xs + (size_t)k * PB + r0 + 4);
    const float wx[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int j = 0; j < NCH; j++) {
      const int c = lane + 32 * j;
      if (c * 4 < N) {
        const float4 bk = reinterpret_cast<const float4*>(s.Bs + (size_t)k * N)[c];
#pragma unroll
        for (int rr = 0; rr < 8; rr++) hv[rr][j] = fma4(wx[rr], bk, hv[rr][j]);
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < 8; rr++)
#pragma unroll
    for (int j = 0; j < NCH; j++) {
      const int c = lane + 32 * j;
      if (c * 4 < N) {
        const size_t o = (size_t)(r0 + rr) * N + c * 4;
        __stcs(reinterpret_cast<float4*>(g32 + o), hv[rr][j]);
        if (g16) __stcs(reinterpret_cast<uint2*>(g16 + o), to_rc4(hv[rr][j], f16));
        if (back) *reinterpret_cast<float4*>(back + o) = hv[rr][j];
      }
    }
  if (NCH == 1 && q8) {  // fp8 read copy: rows of 128 values, one float4 per lane
#pragma unroll
    for (int rr = 0; rr < 8; rr++) store_f8_row(q8, sc8, row0 + r0 + rr, hv[rr][0], lane);
  }
}

// ------------------------------------------------------------------ conventional step

template <int NCH, bool OUT_BF16>
__global__ void __launch_bounds__(128) m2_conventional_kernel(M2Args a) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int blk = blockIdx.x;
  const int pb = blk % a.nPB;
  blk /= a.nPB;
  const int h = blk % a.H, b = blk / a.H;
  const int g = (h * a.G) / a.H;
  const int N = a.N, P = a.P;
  const int p0 = pb * a.PB, R = min(a.PB, P - p0);
  const size_t bh = (size_t)b * a.H + h, bg = (size_t)b * a.G + g;

  const float dt = a.dt[bh];
  const float dA = expf(dt * a.A[h]);
  const float Dh = a.D[h];
  float4 cm[NCH], bm[NCH];
#pragma unroll
  for (int j = 0; j < NCH; j++) {
    const int c = lane + 32 * j;
    cm[j] = bm[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c * 4 < N) {
      cm[j] = load_bf4(a.C + bg * N + c * 4);
      bm[j] = scale4(dt, load_bf4(a.B + bg * N + c * 4));
    }
  }
  int r0w, r1w;
  warp_rows(R, warp, r0w, r1w);
  float* st = a.ckpt + (bh * P + p0) * N;
  for (int r0 = r0w; r0 < r1w; r0 += 8) {
    float4 hv[8][NCH];
#pragma unroll
    for (int rr = 0; rr < 8; rr++)
#pragma unroll
      for (int j = 0; j < NCH; j++) {
        const int c = lane + 32 * j;
        hv[rr][j] = (c * 4 < N) ? __ldcs(reinterpret_cast<const float4*>(st + (size_t)(r0 + rr) * N) + c)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    const uint4 xu = *reinterpret_cast<const uint4*>(a.x + bh * P + p0 + r0);
    const float xr[8] = {bf_lo(xu.x), bf_hi(xu.x), bf_lo(xu.y), bf_hi(xu.y),
                         bf_lo(xu.z), bf_hi(xu.z), bf_lo(xu.w), bf_hi(xu.w)};
    float v[8];
#pragma unroll
    for (int rr = 0; rr < 8; rr++) {
      v[rr] = 0.f;
#pragma unroll
      for (int j = 0; j < NCH; j++) {
        const int c = lane + 32 * j;
        if (c * 4 < N) {
          float4 hn = fma4(xr[rr], bm[j], scale4(dA, hv[rr][j]));
          __stcs(reinterpret_cast<float4*>(st + (size_t)(r0 + rr) * N) + c, hn);
          v[rr] += dot4(hn, cm[j]);
        }
      }
    }
    reduce8(v, lane);
    if ((lane & 3) == 0) {
      const int r = r0 + reduce8_row(lane);
      const size_t oi = bh * P + p0 + r;
      const float xm = bf_to_f(a.x[oi]), zm = bf_to_f(a.z[oi]);
      store_out<OUT_BF16>(a.y, oi, (v[0] + Dh * xm) * silu(zm));
    }
  }
}

// ------------------------------------------------------------------ standalone flush

template <int NCH>
__global__ void __launch_bounds__(128) m2_flush_kernel(M2Args a) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int blk = blockIdx.x;
  const int pb = blk % a.nPB;
  blk /= a.nPB;
  const int h = blk % a.H, b = blk / a.H;
  const int g = (h * a.G) / a.H;
  const int L = a.L, N = a.N, P = a.P, PB = a.PB, H = a.H;
  const int p0 = pb * PB, R = min(PB, P - p0);
  const size_t bh = (size_t)b * H + h, bg = (size_t)b * a.G + g;

  const int4 cur = load_cursor(a.cursors, b);
  const int start = cur.x, m = cur.y;
  if (start < 0 || start >= L || m < 0 || m > L || cur.z != 0 || m == 0) return;

  M2Smem s;
  m2_smem_layout(PB, N, L, L, 1, smem_raw, &s);
  init_bars(s);
  const size_t tile_off = (bh * P + p0) * N;
  if (tid == 0) issue_tile(s, (const char*)(a.ckpt + tile_off), R, N, 4);

  if (tid < m) s.sdt[tid] = a.rdt[bh * pad4(L) + (start + tid) % L];
  const int xv = R >> 3;
  for (int i = tid; i < m * xv; i += 128) {
    const int k = i / xv, v = i - k * xv;
    bf8_to_smem(s.xs + (size_t)k * PB + v * 8, a.rx + (bh * L + (start + k) % L) * P + p0 + v * 8);
  }
  for (int i = tid; i < m * (N >> 3); i += 128) {
    const int k = i / (N >> 3), v = i - k * (N >> 3);
    bf8_to_smem(s.Bs + (size_t)k * N + v * 8, a.rB + (bg * L + (start + k) % L) * N + v * 8);
  }
  __syncthreads();
  if (warp == 0) window_weights(s.sdt, m, a.A[h], lane, s.sw, nullptr, nullptr, &s.sP[0]);
  __syncthreads();
  for (int i = tid; i < m * R; i += 128) {
    const int k = i / R, r = i - k * R;
    s.xs[(size_t)k * PB + r] *= s.sw[k];
  }
  __syncthreads();
  const float Pm = s.sP[0];
  int r0w, r1w;
  warp_rows(R, warp, r0w, r1w);
  if (r1w <= r0w) return;
  if (!mbar_wait_or_report(&s.bars[warp], 0, a.status)) return;
  for (int r0 = r0w; r0 < r1w; r0 += 8) {
    float4 hv[8][NCH];
#pragma unroll
    for (int rr = 0; rr < 8; rr++)
#pragma unroll
      for (int j = 0; j < NCH; j++) {
        const int c = lane + 32 * j;
        hv[rr][j] = (c * 4 < N) ? tile_chunk<NCH>(s, false, r0 + rr, N, c) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    uint8_t* q8 = (a.ckpt_read && a.read_f8) ? reinterpret_cast<uint8_t*>(a.ckpt_read) : nullptr;
    float* sc8 = q8 ? reinterpret_cast<float*>(q8 + (size_t)a.Bt * a.H * a.P * a.N) : nullptr;
    fold_group<NCH>(hv, s, r0, PB, N, m, Pm, lane, a.ckpt + tile_off,
                    (a.ckpt_read && !a.read_f8) ? a.ckpt_read + tile_off : nullptr, a.read_f16, nullptr, q8, sc8,
                    tile_off / N);
  }
}

// ------------------------------------------------------------------ speculative verify epilogue

// Verify epilogue, one block per sequence (runs after the verify kernel in
// stream order): checks the cursor as the verify did, appends the group rows
// (B, C) and dt of the K new records, then marks pending = K and the fold flag.
__global__ void __launch_bounds__(128) m2_verify_epilogue_kernel(M2Args a) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int L = a.L, N = a.N, H = a.H, G = a.G, K = a.K;
  const int4 cur = load_cursor(a.cursors, b);
  const int start = cur.x, count = cur.y;
  if (start < 0 || start >= L || count < 0 || count > L) {
    if (tid == 0) report(a.status, RSSM_DEV_BAD_CURSOR);
    return;
  }
  if (cur.z != 0) {
    if (tid == 0) report(a.status, RSSM_DEV_PENDING);
    return;
  }
  const int nv = N >> 3;
  for (int q = tid; q < K * G * nv; q += 128) {
    const int i = q / (G * nv), r = q - i * G * nv, g = r / nv, v = r - g * nv;
    const int slot = (start + count + i) % L;
    const size_t src = (((size_t)b * K + i) * G + g) * N + v * 8;
    const size_t dst = (((size_t)b * G + g) * L + slot) * N + v * 8;
    copy8(a.rB + dst, a.B + src);
    copy8(a.rC + dst, a.C + src);
  }
  for (int q = tid; q < K * H; q += 128) {
    const int i = q / H, h = q - i * H;
    const int slot = (start + count + i) % L;
    a.rdt[((size_t)b * H + h) * pad4(L) + slot] = a.dt[((size_t)b * K + i) * H + h];
  }
  if (tid == 0) {
    int4 nc = cur;
    nc.z = K;
    nc.w = (count + K > L) ? 1 : 0;
    *reinterpret_cast<int4*>(a.cursors + 4 * (size_t)b) = nc;
  }
}

// ------------------------------------------------------------------ launchers

namespace {

template <typename Kern>
cudaError_t launch(Kern k, int grid, size_t smem, cudaStream_t st, const M2Args& a) {
  cudaError_t e = prepare(k, smem, false);
  if (e != cudaSuccess) return e;
  k<<<grid, 128, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t m2_smem_bytes(int kind, const M2Args& a) {
  return kind == M2_FLUSH ? m2_smem_layout(a.PB, a.N, a.L, a.L, 1, nullptr, nullptr) : 0;
}

#define RSSM_DISPATCH_NCH(NCH_, ...)       \
  if (a.N <= 128) {                        \
    constexpr int NCH_ = 1;                \
    __VA_ARGS__                            \
  } else {                                 \
    constexpr int NCH_ = 2;                \
    __VA_ARGS__                            \
  }

cudaError_t m2_launch(int kind, const M2Args& a, int out_bf16, cudaStream_t st) {
  const int grid = a.Bt * a.H * a.nPB;
  if (grid == 0) return cudaSuccess;
  const size_t smem = m2_smem_bytes(kind, a);
  cudaError_t e = cudaSuccess;
  switch (kind) {
    case M2_CONVENTIONAL:
      RSSM_DISPATCH_NCH(NCH, {
        e = out_bf16 ? launch(m2_conventional_kernel<NCH, true>, grid, 0, st, a)
                     : launch(m2_conventional_kernel<NCH, false>, grid, 0, st, a);
      })
      return e;
    case M2_STEP:
      return m2_step_launch(a, out_bf16, st);
    case M2_FLUSH:
      RSSM_DISPATCH_NCH(NCH, { e = launch(m2_flush_kernel<NCH>, grid, smem, st, a); })
      return e;
    case M2_VERIFY:
      if (m2_verify_fast_applies(a)) return m2_verify_fast_launch(a, out_bf16, st);  // includes the epilogue
      if ((e = m2_verify_launch(a, out_bf16, st)) != cudaSuccess) return e;
      m2_verify_epilogue_kernel<<<a.Bt, 128, 0, st>>>(a);
      return cudaGetLastError();
  }
  return cudaErrorInvalidValue;
}

}  // namespace rssm
