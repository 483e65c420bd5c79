// ReplaySSM AR decode step for Mamba-2, shape-specialised fast path:
// dstate = 128 and headdim a multiple of 64 (the serving layers). Same
// algorithm as the generic kernel in mamba2_step.cu ("How ReplaySSM works":
// non-flush steps read the checkpoint and the window and store no state; the
// L-th step folds the window into the checkpoint and writes it once), laid
// out so that almost every instruction is a load, an FMA or a shuffle:
// compile-time row strides, one 64-bit base pointer per stream, no runtime
// shape predicates.
//
// One CTA of four warps per (sequence, run of HPC consecutive heads of one
// group, 64-row block). Warp w owns rows 16w..16w+15 of each head and lane l
// the float4 column chunk 4l..4l+3 of each row. The heads are pipelined: each
// warp streams its 8 KiB slab of the NEXT head into its own shared-memory
// double buffer with one bulk copy (TMA, non-tensor, on a per-warp mbarrier;
// never multicast) and prefetches that head's records into registers, while it
// computes the current head from registers. What the heads share is done once
// per CTA: the cursor (hence the window's slots and the flush decision) and the
// group's B.C dots of every ring slot and of the current record (warp w forms
// slots w, w+4, ... by per-lane partials and one transposed butterfly
// reduction; shared through shared memory).
//
// Per head, ring slot s and the current record are loaded without waiting on
// the cursor; lane k takes record k from lane (start + k) mod L by a shuffle.
// One warp suffix scan gives w_k = dt_k exp(A sum_{j>k} dt_j) and
// P = exp(A sum dt). Each lane adds its record's term (w_k c_k [+ D on the
// current record]) x_k[r] to its P (h0 . C) partials so that one transposed
// 8-row reduction yields P (h0 C)[r] + sum_k w_k c_k x_k[r] + D x[r]; the gate
// and the store run one lane per row. On the L-th step the window is folded
// into the rows in registers and written once (with the bf16 read copy);
// otherwise the record is appended to its ring slot. The cursor is only read;
// a trailing kernel advances it.
#include "common.cuh"
#include "kernels.h"

namespace rssm {

namespace {

constexpr int FN = 128;                     // dstate
constexpr int FPB = 64;                     // rows per block
constexpr int FW = 4;                       // warps, 16 rows each
constexpr int FT = 32 * FW;
constexpr int SLAB = 16 * FN;               // floats of one warp's rows of one head
constexpr int SMEM = FW * 2 * SLAB * 4;     // per-warp double buffer: 64 KiB

__device__ __forceinline__ uint4 ldg16(const uint16_t* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void unpack8(uint4 u, float* f) {
  f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
  f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}

__device__ __forceinline__ uint4 shfl_u4(uint4 v, int src) {
  return make_uint4(__shfl_sync(FULL, v.x, src), __shfl_sync(FULL, v.y, src), __shfl_sync(FULL, v.z, src),
                    __shfl_sync(FULL, v.w, src));
}

// A head's records: ring slot `lane` and the current record, for the warp's rows.
struct Rec {
  uint4 xs0, xs1;  // x rows of ring slot `lane`
  uint4 xc0, xc1;  // x rows of the current record
  float dts, dtc, A, D;
};

__device__ __forceinline__ void load_rec(Rec& r, const M2Args& a, int bh, int h, int prow, int lane) {
  const int L = a.L, P = a.P;
  r.dts = lane < L ? a.rdt[(size_t)bh * pad4(L) + lane] : 0.f;
  r.dtc = a.dt[bh];
  r.A = a.A[h];
  r.D = a.D[h];
  r.xs0 = r.xs1 = make_uint4(0, 0, 0, 0);
  if (lane < L) {
    const uint16_t* xp = a.rx + ((size_t)bh * L + lane) * P + prow;
    r.xs0 = ldg16(xp);
    r.xs1 = ldg16(xp + 8);
  }
  const uint16_t* xcp = a.x + (size_t)bh * P + prow;
  r.xc0 = ldg16(xcp);
  r.xc1 = ldg16(xcp + 8);
}

template <int LM, bool OUT_BF16>
__global__ void __launch_bounds__(FT, 3) m2_step_fast_kernel(M2Args a, int hpc) {
  constexpr int KW = LM == 16 ? 8 : 16;  // 4 warps x KW >= L + 1 dots
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float sc[FW * KW];           // c_s = B_s . C by ring slot; [L] = current record
  __shared__ uint64_t bars[FW * 2];       // per warp, per buffer
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.y;
  const int run = blockIdx.x / a.nPB, pb = blockIdx.x - run * a.nPB;
  const int h0 = run * hpc;
  const int L = a.L, P = a.P, H = a.H;
  const int g = h0 / (H / a.G);
  const int bg = b * a.G + g;
  const int prow = pb * FPB + warp * 16;  // the warp's first row within a head
  const bool copy = a.ckpt_read != nullptr;
  float* buf = reinterpret_cast<float*>(smem) + warp * 2 * SLAB;
  uint64_t* bar = bars + warp * 2;
  const uint32_t slab_bytes_f32 = SLAB * 4;

  if (lane == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const int4 cur = *reinterpret_cast<const int4*>(a.cursors + 4 * b);
  const int start = cur.x, count = cur.y;
  const bool valid = start >= 0 && start < L && count >= 0 && count < L && cur.z == 0;
  if (!valid) return;  // reported by the cursor kernel (uniform over the CTA)
  const int m = count + 1;
  const bool flush = (m == L);
  const bool rd16 = copy && !flush;  // non-flush steps read the bf16 read copy
  const uint32_t slab_bytes = rd16 ? slab_bytes_f32 / 2 : slab_bytes_f32;

  // issue the first head's slab
  auto slab_src = [&](int h) -> const void* {
    const size_t off = ((size_t)(b * H + h) * P + prow) * FN;
    return rd16 ? (const void*)(a.ckpt_read + off) : (const void*)(a.ckpt + off);
  };
  if (lane == 0) {
    mbar_arrive_expect_tx(&bar[0], slab_bytes);
    bulk_load(buf, slab_src(h0), slab_bytes, &bar[0]);
  }
  Rec rc;
  load_rec(rc, a, b * H + h0, h0, prow, lane);
  const float4 cm = load_bf4(a.C + (size_t)bg * FN + lane * 4);
  {  // c_s = B_s . C for slots s = warp + 4 i (s == L: the current record), shared by the heads
    const uint16_t* rB = a.rB + (size_t)bg * L * FN + lane * 4;
    const float4 bcur = load_bf4(a.B + (size_t)bg * FN + lane * 4);
    float pk[KW];
#pragma unroll
    for (int i = 0; i < KW; i++) {
      const int s = warp + FW * i;
      pk[i] = s < L ? dot4(load_bf4(rB + s * FN), cm) : (s == L ? dot4(bcur, cm) : 0.f);
    }
    const float red = reduce_transpose<KW>(pk, lane);
    const int idx = KW == 8 ? reduce8_row(lane) : (lane >> 1);
    const bool rep = KW == 8 ? (lane & 3) == 0 : (lane & 1) == 0;
    if (rep) sc[warp + FW * idx] = red;
  }
  int sl = start + lane;
  sl = sl < L ? sl : sl - L;
  const int appl = start + count < L ? start + count : start + count - L;  // slot the record goes to
  __syncthreads();
  const float ck = lane < m ? sc[lane < count ? sl : L] : 0.f;

  for (int i = 0; i < hpc; i++) {
    const int h = h0 + i;
    const int bh = b * H + h;
    Rec nx;
    if (i + 1 < hpc) {  // next head in flight: slab into the other buffer, records into registers
      if (lane == 0) {
        fence_proxy_async();
        mbar_arrive_expect_tx(&bar[(i + 1) & 1], slab_bytes);
        bulk_load(buf + ((i + 1) & 1) * SLAB, slab_src(h + 1), slab_bytes, &bar[(i + 1) & 1]);
      }
      load_rec(nx, a, bh + 1, h + 1, prow, lane);
    }
    // this head's window, lane k = record k
    const float dtr = __shfl_sync(FULL, rc.dts, sl);
    const float dtk = lane < count ? dtr : (lane == count ? rc.dtc : 0.f);
    const uint4 xr0 = shfl_u4(rc.xs0, sl), xr1 = shfl_u4(rc.xs1, sl);
    float xl[16];
    unpack8(lane < count ? xr0 : rc.xc0, xl);
    unpack8(lane < count ? xr1 : rc.xc1, xl + 8);
    float sfx = dtk * rc.A;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_down_sync(FULL, sfx, o);
      if (lane + o < 32) sfx += v;
    }
    float ex = __shfl_down_sync(FULL, sfx, 1);
    if (lane == 31) ex = 0.f;
    const float Pm = expf(__shfl_sync(FULL, sfx, 0));
    const float wk = dtk * expf(ex);
    const float coef = lane < m ? fmaf(wk, ck, lane == count ? rc.D : 0.f) : 0.f;

    // this head's slab: shared memory -> registers
    if (!__all_sync(FULL, mbar_wait(&bar[i & 1], (i >> 1) & 1))) {
      // give the copies in flight a second bounded wait before the block exits
      if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
      mbar_wait(&bar[i & 1], (i >> 1) & 1);
      if (i + 1 < hpc) mbar_wait(&bar[(i + 1) & 1], ((i + 1) >> 1) & 1);
      return;
    }
    float4 hv[16];
    if (rd16) {
      const uint16_t* s16 = reinterpret_cast<const uint16_t*>(buf + (i & 1) * SLAB) + lane * 4;
#pragma unroll
      for (int r = 0; r < 16; r++) hv[r] = load_bf4(s16 + r * FN);
    } else {
      const float4* s32 = reinterpret_cast<const float4*>(buf + (i & 1) * SLAB) + lane;
#pragma unroll
      for (int r = 0; r < 16; r++) hv[r] = s32[r * (FN / 4)];
    }
    __syncwarp();  // the buffer may be refilled from here on

    // pre-gate outputs of the warp's 16 rows
    float tot[2];
#pragma unroll
    for (int gg = 0; gg < 2; gg++) {
      float v[8];
#pragma unroll
      for (int rr = 0; rr < 8; rr++) v[rr] = fmaf(Pm, dot4(hv[gg * 8 + rr], cm), coef * xl[gg * 8 + rr]);
      tot[gg] = reduce_transpose<8>(v, lane);
    }
    {
      const int rr = lane & 7;
      const int src = ((rr >> 2) & 1) * 16 + ((rr >> 1) & 1) * 8 + (rr & 1) * 4;
      const float t0 = __shfl_sync(FULL, tot[0], src), t1 = __shfl_sync(FULL, tot[1], src);
      if (lane < 16) {
        const size_t oi = (size_t)bh * P + prow + lane;
        const float zm = bf_to_f(a.z[oi]);
        const float yv = (lane & 8 ? t1 : t0) * __fdividef(zm, 1.f + __expf(-zm));
        if (OUT_BF16)
          reinterpret_cast<uint16_t*>(a.y)[oi] = f_to_bf(yv);
        else
          reinterpret_cast<float*>(a.y)[oi] = yv;
      }
    }
    const size_t hoff = ((size_t)bh * P + prow) * FN + lane * 4;
    if (flush) {  // fold the window into the rows in registers, write them once
#pragma unroll
      for (int r = 0; r < 16; r++) hv[r] = scale4(Pm, hv[r]);
      const uint16_t* rB = a.rB + (size_t)bg * L * FN + lane * 4;
      for (int k = 0; k < m; k++) {
        const float w = __shfl_sync(FULL, wk, k);
        int s = start + k;
        s = s < L ? s : s - L;
        const float4 bk = load_bf4(k < count ? rB + s * FN : a.B + (size_t)bg * FN + lane * 4);
#pragma unroll
        for (int r = 0; r < 16; r++) hv[r] = fma4(w * __shfl_sync(FULL, xl[r], k), bk, hv[r]);
      }
      float4* dst = reinterpret_cast<float4*>(a.ckpt + hoff);
#pragma unroll
      for (int r = 0; r < 16; r++) __stcs(dst + r * (FN / 4), hv[r]);
      if (copy) {
        uint2* d16 = reinterpret_cast<uint2*>(a.ckpt_read + hoff);
#pragma unroll
        for (int r = 0; r < 16; r++) __stcs(d16 + r * (FN / 4), f4_to_bf4(hv[r]));
      }
    } else {  // append the current record: x, z rows of this warp, dt once per head
      const size_t rrow = ((size_t)bh * L + appl) * P + prow;
      if (lane < 2) *reinterpret_cast<uint4*>(a.rx + rrow + lane * 8) = lane ? rc.xc1 : rc.xc0;
      if (lane == 2 || lane == 3) {
        const int o = (lane - 2) * 8;
        *reinterpret_cast<uint4*>(a.rz + rrow + o) = ldg16(a.z + (size_t)bh * P + prow + o);
      }
      if (lane == 4 && warp == 0 && pb == 0) a.rdt[(size_t)bh * pad4(L) + appl] = rc.dtc;
    }
    if (i + 1 < hpc) rc = nx;
  }
  // the group's B and C rows, once per group (by the block holding its first head)
  if (!flush && pb == 0 && h0 == g * (H / a.G) && threadIdx.x < FN / 8) {
    const size_t brow = ((size_t)bg * L + appl) * FN + threadIdx.x * 8;
    *reinterpret_cast<uint4*>(a.rB + brow) = ldg16(a.B + (size_t)bg * FN + threadIdx.x * 8);
    *reinterpret_cast<uint4*>(a.rC + brow) = ldg16(a.C + (size_t)bg * FN + threadIdx.x * 8);
  }
}

template <int LM, bool OUT_BF16>
cudaError_t launch_fast(const M2Args& a, int hpc, cudaStream_t st) {
  auto k = m2_step_fast_kernel<LM, OUT_BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid((a.H / hpc) * a.nPB, a.Bt);
  k<<<grid, FT, SMEM, st>>>(a, hpc);
  return cudaGetLastError();
}

}  // namespace

bool m2_step_fast_applies(const M2Args& a) { return a.N == FN && a.P % FPB == 0 && a.PB == FPB; }

cudaError_t m2_step_fast_launch(const M2Args& a, int out_bf16, cudaStream_t st) {
  // heads per block: up to 4 consecutive heads of one group
  const int hpg = a.H / a.G;
  const int hpc = hpg % 4 == 0 ? 4 : (hpg % 2 == 0 ? 2 : 1);
  if (a.L <= 16) return out_bf16 ? launch_fast<16, true>(a, hpc, st) : launch_fast<16, false>(a, hpc, st);
  return out_bf16 ? launch_fast<32, true>(a, hpc, st) : launch_fast<32, false>(a, hpc, st);
}

}  // namespace rssm
