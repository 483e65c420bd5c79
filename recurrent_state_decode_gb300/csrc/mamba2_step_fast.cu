// ReplaySSM AR decode step for Mamba-2, shape-specialised fast path:
// dstate = 128 and headdim a multiple of 64 (the serving layers). Same
// algorithm as the generic kernel in mamba2_step.cu ("How ReplaySSM works":
// non-flush steps read the checkpoint and the window and store no state; the
// L-th step folds the window into the checkpoint and writes it once).
//
// Persistent warps, each working alone: warp gw of the grid takes the
// (sequence, head, 64-row block) tiles gw, gw + W, ... (W = warps in the grid),
// so the tiles of a flushing sequence spread over all warps. A tile streams
// through the warp in four slabs of 16 rows (8 KiB fp32, 4 KiB from the bf16
// read copy), each one bulk copy (TMA, non-tensor; never multicast) into the
// warp's double buffer on the warp's own mbarriers: while the warp computes
// slab n the copy of slab n+1 -- possibly the first slab of its next tile -- is
// in flight. The next tile's cursor, dts, A and D are loaded a tile ahead and
// each slab's x records a slab ahead, so no warp ever waits on them. Nothing is
// shared between warps.
//
// Per tile (lane k = window record k; ring slots are fetched by slot and the
// window picked by shuffles once the cursor is known):
//   * one warp suffix scan: w_k = dt_k exp(A sum_{j>k} dt_j), P = exp(A sum dt);
//   * c_k = B_k . C for all ring slots by per-lane partials over the lane's
//     float4 column chunk and one transposed butterfly reduction, plus the
//     current record's dot;
//   * coef_k = w_k c_k (+ D on the current record).
// Per 8-row group of a slab: lane l holds the float4 chunk 4l..4l+3 of each
// row; its partial P (h0 . C) plus coef_l x_l[r] goes through one transposed
// 8-row reduction, giving y[r] before the gate; the gate silu(z) and the store
// run one lane per row. On the L-th step the window is folded into each row
// (re-read from the buffer) and written once, with the bf16 read copy;
// otherwise the record is appended to its ring slot. The cursor is only read;
// a trailing kernel advances it.
#include "common.cuh"
#include "kernels.h"

namespace rssm {

namespace {

constexpr int FN = 128;                   // dstate
constexpr int FPB = 64;                   // rows per tile
constexpr int SR = 16;                    // rows per slab
constexpr int NSLAB = FPB / SR;
constexpr int WPC = 4;                    // warps per block
constexpr int FT = 32 * WPC;
constexpr int CPS = 3;                    // blocks per SM
constexpr int SLAB = SR * FN;             // floats of one slab
constexpr int SMEM = WPC * 2 * SLAB * 4;  // per-warp double buffer: 64 KiB per block

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void unpack8(uint4 u, float* f) {
  f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
  f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}

__device__ __forceinline__ uint4 shfl_u4(uint4 v, int src) {
  return make_uint4(__shfl_sync(FULL, v.x, src), __shfl_sync(FULL, v.y, src), __shfl_sync(FULL, v.z, src),
                    __shfl_sync(FULL, v.w, src));
}

// What a tile needs before its first slab: where it is, its cursor, its scalars.
struct TileHead {
  int t;          // tile index, >= ntiles when there is none
  int bh, h, pb;  // bh = b * H + h
  int b, g;
  int4 cur;
  float dts, dtc, A, D;  // dt of ring slot `lane`, current dt, A[h], D[h]
};

__device__ __forceinline__ void load_head(TileHead& th, const M2Args& a, int t, int ntiles, int lane) {
  th.t = t;
  if (t >= ntiles) return;
  const int pb = t % a.nPB, bh = t / a.nPB;
  th.pb = pb;
  th.bh = bh;
  th.h = bh % a.H;
  th.b = bh / a.H;
  th.g = th.h / (a.H / a.G);
  th.cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)th.b);
  th.dts = lane < a.L ? a.rdt[(size_t)bh * pad4(a.L) + lane] : 0.f;
  th.dtc = a.dt[bh];
  th.A = a.A[th.h];
  th.D = a.D[th.h];
}

__device__ __forceinline__ bool head_valid(const TileHead& th, int L) {
  const int4 c = th.cur;
  return c.x >= 0 && c.x < L && c.y >= 0 && c.y < L && c.z == 0;
}

// x rows of one slab: ring slot `lane` and the current record.
struct SlabRec {
  uint4 xs0, xs1, xc0, xc1;
};

__device__ __forceinline__ void load_slab_rec(SlabRec& r, const M2Args& a, int bh, int row0, int lane) {
  const int L = a.L, P = a.P;
  r.xs0 = r.xs1 = make_uint4(0, 0, 0, 0);
  if (lane < L) {
    const uint16_t* xp = a.rx + ((size_t)bh * L + lane) * P + row0;
    r.xs0 = ldg16(xp);
    r.xs1 = ldg16(xp + 8);
  }
  const uint16_t* xcp = a.x + (size_t)bh * P + row0;
  r.xc0 = ldg16(xcp);
  r.xc1 = ldg16(xcp + 8);
}

template <int LM, bool OUT_BF16>
__global__ void __launch_bounds__(FT, CPS) m2_step_fast_kernel(M2Args a, int ntiles) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t bars[WPC * 2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int L = a.L, P = a.P, H = a.H;
  const int W = gridDim.x * WPC;
  float* buf = reinterpret_cast<float*>(smem) + warp * 2 * SLAB;
  uint64_t* bar = bars + warp * 2;
  const bool copy = a.ckpt_read != nullptr;
  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncwarp();

  // slab q of a tile into buffer n & 1
  auto issue = [&](const TileHead& th, int q, uint32_t n) {
    if (lane != 0) return;
    const bool rd16 = copy && (th.cur.y + 1 < L);
    const size_t off = ((size_t)th.bh * P + th.pb * FPB + q * SR) * FN;
    const uint32_t bytes = rd16 ? SLAB * 2 : SLAB * 4;
    fence_proxy_async();
    mbar_arrive_expect_tx(&bar[n & 1], bytes);
    bulk_load(buf + (n & 1) * SLAB, rd16 ? (const void*)(a.ckpt_read + off) : (const void*)(a.ckpt + off), bytes,
              &bar[n & 1]);
  };
  // the next valid tile from t on (invalid cursors are skipped and reported by the cursor kernel)
  auto next_valid = [&](TileHead& th, int t) {
    load_head(th, a, t, ntiles, lane);
    while (th.t < ntiles && !head_valid(th, L)) load_head(th, a, th.t + W, ntiles, lane);
  };

  TileHead cur;
  next_valid(cur, blockIdx.x * WPC + warp);
  if (cur.t >= ntiles) return;
  uint32_t n = 0;  // slabs consumed by this warp
  issue(cur, 0, n);
  SlabRec rec;
  load_slab_rec(rec, a, cur.bh, cur.pb * FPB, lane);

  while (cur.t < ntiles) {
    TileHead nxt;
    next_valid(nxt, cur.t + W);  // a whole tile ahead

    // ---- per-tile setup
    const int start = cur.cur.x, count = cur.cur.y, m = count + 1;
    const bool flush = (m == L), rd16 = copy && !flush;
    const int bg = cur.b * a.G + cur.g;
    int sl = start + lane;
    sl = sl < L ? sl : sl - L;
    const float dtr = __shfl_sync(FULL, cur.dts, sl);
    const float dtk = lane < count ? dtr : (lane == count ? cur.dtc : 0.f);
    float sfx = dtk * cur.A;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_down_sync(FULL, sfx, o);
      if (lane + o < 32) sfx += v;
    }
    float ex = __shfl_down_sync(FULL, sfx, 1);
    if (lane == 31) ex = 0.f;
    const float Pm = expf(__shfl_sync(FULL, sfx, 0));
    const float wk = dtk * expf(ex);
    const float4 cm = load_bf4(a.C + (size_t)bg * FN + lane * 4);
    float coef;
    {
      const uint16_t* rB = a.rB + (size_t)bg * L * FN + lane * 4;
      float pk[LM];
#pragma unroll
      for (int s = 0; s < LM; s++) pk[s] = s < L ? dot4(load_bf4(rB + s * FN), cm) : 0.f;
      const float cc = warp_sum(dot4(load_bf4(a.B + (size_t)bg * FN + lane * 4), cm));
      const float red = reduce_transpose<LM>(pk, lane);  // slot s at lane idx^-1(s)
      const float cs = __shfl_sync(FULL, red, LM == 16 ? (2 * sl) & 31 : sl);
      coef = lane < count ? wk * cs : (lane == count ? fmaf(wk, cc, cur.D) : 0.f);
    }
    const int appl = start + count < L ? start + count : start + count - L;

    for (int q = 0; q < NSLAB; q++, n++) {
      const int row0 = cur.pb * FPB + q * SR;  // first row of the slab within the head
      // next slab in flight, its records into registers
      SlabRec nrec;
      if (q + 1 < NSLAB) {
        issue(cur, q + 1, n + 1);
        load_slab_rec(nrec, a, cur.bh, row0 + SR, lane);
      } else if (nxt.t < ntiles) {
        issue(nxt, 0, n + 1);
        load_slab_rec(nrec, a, nxt.bh, nxt.pb * FPB, lane);
      }
      // this slab's window x rows, lane k = record k
      float xl[SR];
      // every lane takes part in the shuffles; the choice comes after
      const uint4 xr0 = shfl_u4(rec.xs0, sl), xr1 = shfl_u4(rec.xs1, sl);
      unpack8(lane < count ? xr0 : rec.xc0, xl);
      unpack8(lane < count ? xr1 : rec.xc1, xl + 8);
      if (lane >= m) {
#pragma unroll
        for (int r = 0; r < SR; r++) xl[r] = 0.f;
      }
      if (!__all_sync(FULL, mbar_wait(&bar[n & 1], (n >> 1) & 1))) {
        if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
        mbar_wait(&bar[(n + 1) & 1], ((n + 1) >> 1) & 1);  // let the next copy land before leaving
        return;
      }
      const float* s32 = buf + (n & 1) * SLAB;
      const uint16_t* s16 = reinterpret_cast<const uint16_t*>(s32);
      auto row_chunk = [&](int r) -> float4 {
        return rd16 ? load_bf4(s16 + r * FN + lane * 4) : reinterpret_cast<const float4*>(s32 + r * FN)[lane];
      };
      float tot[2];
#pragma unroll
      for (int gg = 0; gg < 2; gg++) {
        float v[8];
#pragma unroll
        for (int rr = 0; rr < 8; rr++) v[rr] = fmaf(Pm, dot4(row_chunk(gg * 8 + rr), cm), coef * xl[gg * 8 + rr]);
        tot[gg] = reduce_transpose<8>(v, lane);
      }
      {
        const int rr = lane & 7;
        const int src = ((rr >> 2) & 1) * 16 + ((rr >> 1) & 1) * 8 + (rr & 1) * 4;
        const float t0 = __shfl_sync(FULL, tot[0], src), t1 = __shfl_sync(FULL, tot[1], src);
        if (lane < SR) {
          const size_t oi = (size_t)cur.bh * P + row0 + lane;
          const float zm = bf_to_f(a.z[oi]);
          const float yv = (lane & 8 ? t1 : t0) * __fdividef(zm, 1.f + __expf(-zm));
          if (OUT_BF16)
            reinterpret_cast<uint16_t*>(a.y)[oi] = f_to_bf(yv);
          else
            reinterpret_cast<float*>(a.y)[oi] = yv;
        }
      }
      const size_t soff = ((size_t)cur.bh * P + row0) * FN + lane * 4;
      if (flush) {  // fold the window into the slab's rows, write them once
        const uint16_t* rB = a.rB + (size_t)bg * L * FN + lane * 4;
#pragma unroll
        for (int gg = 0; gg < 2; gg++) {
          float4 hv[8];
#pragma unroll
          for (int rr = 0; rr < 8; rr++) hv[rr] = scale4(Pm, row_chunk(gg * 8 + rr));
          for (int k = 0; k < m; k++) {
            const float w = __shfl_sync(FULL, wk, k);
            int s = start + k;
            s = s < L ? s : s - L;
            const float4 bk = load_bf4(k < count ? rB + s * FN : a.B + (size_t)bg * FN + lane * 4);
#pragma unroll
            for (int rr = 0; rr < 8; rr++) hv[rr] = fma4(w * __shfl_sync(FULL, xl[gg * 8 + rr], k), bk, hv[rr]);
          }
#pragma unroll
          for (int rr = 0; rr < 8; rr++) {
            const size_t o = soff + (size_t)(gg * 8 + rr) * FN;
            __stcs(reinterpret_cast<float4*>(a.ckpt + o), hv[rr]);
            if (copy) __stcs(reinterpret_cast<uint2*>(a.ckpt_read + o), f4_to_bf4(hv[rr]));
          }
        }
      } else {  // append the current record's x, z rows of this slab (dt, B, C once per tile)
        const size_t rrow = ((size_t)cur.bh * L + appl) * P + row0;
        if (lane < 2) *reinterpret_cast<uint4*>(a.rx + rrow + lane * 8) = lane ? rec.xc1 : rec.xc0;
        if (lane == 2 || lane == 3) {
          const int o = (lane - 2) * 8;
          *reinterpret_cast<uint4*>(a.rz + rrow + o) = ldg16(a.z + (size_t)cur.bh * P + row0 + o);
        }
        if (q == 0 && cur.pb == 0) {
          if (lane == 4) a.rdt[(size_t)cur.bh * pad4(L) + appl] = cur.dtc;
          if (cur.h == cur.g * (H / a.G) && lane >= 8 && lane < 8 + FN / 8) {  // the group's first head
            const int c8 = (lane - 8) * 8;
            const size_t brow = ((size_t)bg * L + appl) * FN + c8;
            *reinterpret_cast<uint4*>(a.rB + brow) = ldg16(a.B + (size_t)bg * FN + c8);
            *reinterpret_cast<uint4*>(a.rC + brow) = ldg16(a.C + (size_t)bg * FN + c8);
          }
        }
      }
      __syncwarp();  // the buffer may be refilled from here on
      rec = nrec;
    }
    cur = nxt;
  }
}

struct DeviceSMs {
  int sms = 0;
};

int sm_count() {
  static DeviceSMs cache[64];
  int dev = 0;
  cudaGetDevice(&dev);
  DeviceSMs& d = cache[dev & 63];
  if (d.sms == 0) cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  return d.sms;
}

template <int LM, bool OUT_BF16>
cudaError_t launch_fast(const M2Args& a, cudaStream_t st) {
  auto k = m2_step_fast_kernel<LM, OUT_BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  const int ntiles = a.Bt * a.H * a.nPB;
  int grid = sm_count() * CPS;
  const int need = (ntiles + WPC - 1) / WPC;
  if (grid > need) grid = need;
  k<<<grid, FT, SMEM, st>>>(a, ntiles);
  return cudaGetLastError();
}

}  // namespace

bool m2_step_fast_applies(const M2Args& a) { return a.N == FN && a.P % FPB == 0 && a.PB == FPB; }

cudaError_t m2_step_fast_launch(const M2Args& a, int out_bf16, cudaStream_t st) {
  if (a.L <= 16) return out_bf16 ? launch_fast<16, true>(a, st) : launch_fast<16, false>(a, st);
  return out_bf16 ? launch_fast<32, true>(a, st) : launch_fast<32, false>(a, st);
}

}  // namespace rssm
