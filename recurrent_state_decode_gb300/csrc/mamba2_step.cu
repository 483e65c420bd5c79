// ReplaySSM AR decode step for Mamba-2 on sm_103a: a persistent,
// warp-specialised kernel ("How ReplaySSM works": non-flush steps read the
// checkpoint and the window and store no state; the L-th step folds the window
// into the checkpoint and writes it once).
//
// One CTA per SM walks the (sequence, head, row block) items of the layer in
// a static round-robin. Shared memory holds two rings: T tile buffers (the
// fp32 checkpoint rows, or the bf16 read copy on a non-flush step) and R small
// record buffers (x rows and B rows of the window records and of the current
// record, z, C, the dt ring row and the item's metadata), each guarded by
// `full` and `empty` mbarriers. The last warp is the producer: it prefetches
// cursors, dt, A and D of the next 32 items one lane per item, then per item
// fills a record buffer and a tile buffer with bulk copies (TMA, non-tensor;
// never multicast). Record rows land with a 16-byte pad per row so the
// lane-per-record reads and the ldmatrix reads below are bank-conflict free.
//
// Three consumer groups of four warps take items in turn; each warp owns a
// quarter of the item's rows:
//   1. decay weights of the m <= 32 window records by one warp suffix scan
//      (lane k = record k): w_k = dt_k exp(A sum_{j>k} dt_j), P = exp(A sum dt);
//   2. c_k = B_k . C for all records on the tensor cores (mma.sync m16n8k16,
//      bf16 in, fp32 accumulate: records x dstate times C) when dstate is a
//      multiple of 16, else by lane partials and one transposed reduction;
//   3. pulls its rows of the tile into registers and releases the tile buffer
//      at once, so the producer can refill it while the warp computes;
//   4. per 8-row group adds lane k's term (w_k c_k [+ D on the current
//      record]) x_k[r] to the P (h0 . C) partials, so one transposed 8-row
//      reduction yields P (h0 C)[r] + sum_k w_k c_k x_k[r] + D x[r]; the gate
//      silu(z) and the store run on one lane per row;
//   5. on a flush folds h1 = P h0 + sum_k (w_k x_k) B_k^T from the rows in
//      registers and streams them out (with the bf16 read copy), otherwise
//      appends the current record to its ring slot;
// then releases the record buffer. Every wait is bounded.
#include "persistent.cuh"

namespace rssm {

namespace {

using persistent::Carver;
using persistent::NCONS;
using persistent::consumer_rows;
using persistent::decode_tile;
using persistent::device_info;
using persistent::DeviceInfo;

constexpr int NG = 3;                    // consumer groups
constexpr int NW = NG * NCONS;           // consumer warps
constexpr int THREADS = 32 * (NW + 1);   // + one producer warp
constexpr int MAXB = 8;                  // tile / record buffers at most
constexpr uint32_t BAR_BYTES = 4 * MAXB * 8;  // full_t, empty_t, full_r, empty_r

struct Meta {
  int start, count, b, h;
  int g, pb, skip, rd16;
  float dt, A, D, pad;
};

struct Layout {
  uint32_t xw, zc, Bw, Cc, dtr, meta, rec_bytes;  // record buffer offsets
  uint32_t tile_bytes;
  int XS, BS;  // shared-memory row strides (elements) of the x rows and B rows
  int T, R;    // tile and record buffers
};

inline Layout make_layout(int PB, int N, int L, int LM, int smem_optin) {
  Layout s{};
  s.XS = PB + 8;
  s.BS = N + 8;
  Carver c;
  s.xw = c.take(L * s.XS * 2);       // x rows of window records k (record k at row k)
  s.zc = c.take(PB * 2);             // z rows of the current record
  s.Bw = c.take(LM * s.BS * 2);      // B rows of window records (LM >= L rows for the mma tiles)
  s.Cc = c.take(N * 2);              // C of the current record
  s.dtr = c.take(pad4(L) * 4);       // dt ring row, slot order
  s.meta = c.take(sizeof(Meta));
  s.rec_bytes = c.off;
  s.tile_bytes = (PB * N * 4 + 127u) & ~127u;
  s.R = 2 * NG + 2 < MAXB ? 2 * NG + 2 : MAXB;
  const int avail = smem_optin - (int)BAR_BYTES - s.R * (int)s.rec_bytes;
  s.T = avail / (int)s.tile_bytes;
  if (s.T > MAXB) s.T = MAXB;
  return s;
}

// Record copy q of an item; false if it moves nothing.
__device__ __forceinline__ bool record_copy(const M2Args& a, const Layout& lay, unsigned char* rb, int q, int b,
                                            int h, int g, int pb, int start, int count, void*& dst,
                                            const void*& src, uint32_t& bytes) {
  const int L = a.L, N = a.N, P = a.P, PB = a.PB;
  const int p0 = pb * PB, R = min(PB, P - p0);
  const size_t bh = (size_t)b * a.H + h, bg = (size_t)b * a.G + g;
  bytes = 0;
  switch (q) {
    case 0: dst = rb + lay.xw + (size_t)count * lay.XS * 2; src = a.x + bh * P + p0; bytes = R * 2; break;
    case 1: dst = rb + lay.zc; src = a.z + bh * P + p0; bytes = R * 2; break;
    case 2: dst = rb + lay.Bw + (size_t)count * lay.BS * 2; src = a.B + bg * N; bytes = N * 2; break;
    case 3: dst = rb + lay.Cc; src = a.C + bg * N; bytes = N * 2; break;
    case 4:
      dst = rb + lay.dtr;
      src = a.rdt + bh * pad4(L);
      bytes = count > 0 ? pad4(L) * 4 : 0;
      break;
    default: {
      int k = q - 5;
      if (k < count) {  // x row of window record k
        const int slot = start + k < L ? start + k : start + k - L;
        dst = rb + lay.xw + (size_t)k * lay.XS * 2;
        src = a.rx + (bh * L + slot) * P + p0;
        bytes = R * 2;
      } else if ((k -= count) < count) {  // B row of window record k
        const int slot = start + k < L ? start + k : start + k - L;
        dst = rb + lay.Bw + (size_t)k * lay.BS * 2;
        src = a.rB + (bg * L + slot) * N;
        bytes = N * 2;
      }
    }
  }
  return bytes != 0;
}

__device__ void producer(const M2Args& a, const Layout& lay, unsigned char* tiles, unsigned char* recs,
                         uint64_t* bars, int ntiles, int lane) {
  uint64_t* full_t = bars;
  uint64_t* empty_t = bars + MAXB;
  uint64_t* full_r = bars + 2 * MAXB;
  uint64_t* empty_r = bars + 3 * MAXB;
  const int G = gridDim.x, L = a.L, T = lay.T, RB = lay.R;
  int j = 0;
  for (int base = blockIdx.x; base < ntiles; base += 32 * G) {
    // lane i prefetches what item base + i*G needs before its copies can be issued
    const int tl = base + lane * G;
    int4 cur = make_int4(-1, 0, 0, 0);
    float dtl = 0.f, Al = 0.f, Dl = 0.f;
    if (tl < ntiles) {
      int b, h, pb;
      decode_tile(a, tl, b, h, pb);
      cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)b);
      dtl = a.dt[(size_t)b * a.H + h];
      Al = a.A[h];
      Dl = a.D[h];
    }
    const int nb = min(32, (ntiles - base + G - 1) / G);
    for (int i = 0; i < nb; i++, j++) {
      const int jr = j % RB, jt = j % T;
      bool ok = true;
      if (j >= RB) ok = mbar_wait(&empty_r[jr], ((j / RB) - 1) & 1);
      if (j >= T) ok = ok && mbar_wait(&empty_t[jt], ((j / T) - 1) & 1);
      if (!__all_sync(FULL, ok)) {
        if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
        return;
      }
      unsigned char* rb = recs + (size_t)jr * lay.rec_bytes;
      const int start = __shfl_sync(FULL, cur.x, i), count = __shfl_sync(FULL, cur.y, i);
      const int pending = __shfl_sync(FULL, cur.z, i);
      const float dtt = __shfl_sync(FULL, dtl, i), At = __shfl_sync(FULL, Al, i), Dt = __shfl_sync(FULL, Dl, i);
      int b, h, pb;
      decode_tile(a, base + i * G, b, h, pb);
      const int g = (h * a.G) / a.H;
      // invalid cursors are skipped here and reported by the cursor kernel
      const bool valid = start >= 0 && start < L && count >= 0 && count < L && pending == 0;
      const bool rd16 = valid && (count + 1 < L) && a.ckpt_read != nullptr;
      if (lane == 0) {
        *reinterpret_cast<Meta*>(rb + lay.meta) =
            Meta{start, count, b, h, g, pb, valid ? 0 : 1, rd16 ? 1 : 0, dtt, At, Dt, 0.f};
      }
      if (!valid) {
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full_r[jr]);
          mbar_arrive(&full_t[jt]);
        }
        continue;
      }
      const int ncopies = 5 + 2 * count;
      uint32_t mine = 0;
      for (int q = lane; q < ncopies; q += 32) {
        void* d;
        const void* s;
        uint32_t n;
        if (record_copy(a, lay, rb, q, b, h, g, pb, start, count, d, s, n)) mine += n;
      }
      const uint32_t total = __reduce_add_sync(FULL, mine);
      if (lane == 0) mbar_arrive_expect_tx(&full_r[jr], total);
      __syncwarp();
      for (int q = lane; q < ncopies; q += 32) {
        void* d;
        const void* s;
        uint32_t n;
        if (record_copy(a, lay, rb, q, b, h, g, pb, start, count, d, s, n)) bulk_load(d, s, n, &full_r[jr]);
      }
      if (lane == 0) {
        const int p0 = pb * a.PB, R = min(a.PB, a.P - p0);
        const size_t off = (((size_t)b * a.H + h) * a.P + p0) * a.N;
        const uint32_t tb = (uint32_t)(R * a.N * (rd16 ? 2 : 4));
        mbar_arrive_expect_tx(&full_t[jt], tb);
        bulk_load(tiles + (size_t)jt * lay.tile_bytes,
                  rd16 ? (const void*)(a.ckpt_read + off) : (const void*)(a.ckpt + off), tb, &full_t[jt]);
      }
    }
  }
}

// c_k = B_k . C for records k = 0..LM-1 (rows of Bw), returned at lane k.
// Tensor-core path: A = B rows (records x dstate), B operand column 0 = C.
template <int LM>
__device__ __forceinline__ float dots_mma(const uint16_t* Bw, int BS, const uint16_t* Cc, int N, int lane) {
  float d[LM / 16][4];
#pragma unroll
  for (int t = 0; t < LM / 16; t++) d[t][0] = d[t][1] = d[t][2] = d[t][3] = 0.f;
  const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;
  for (int k0 = 0; k0 < N; k0 += 16) {
    uint32_t b0 = 0, b1 = 0;
    if (lane < 4) {
      b0 = *reinterpret_cast<const uint32_t*>(Cc + k0 + 2 * lane);
      b1 = *reinterpret_cast<const uint32_t*>(Cc + k0 + 8 + 2 * lane);
    }
#pragma unroll
    for (int t = 0; t < LM / 16; t++) {
      uint32_t af[4];
      ldmatrix_x4(af, Bw + (size_t)(t * 16 + arow) * BS + k0 + acol);
      mma_bf16_16816(d[t], af, b0, b1);
    }
  }
  // D[row][0] sits in lane 4*(row & 7), register 0 (rows 0-7) or 2 (rows 8-15)
  const int src = (lane & 7) * 4;
  const float r0 = __shfl_sync(FULL, d[0][0], src), r1 = __shfl_sync(FULL, d[0][2], src);
  float ck = (lane & 8) ? r1 : r0;
  if (LM == 32) {
    const float r2 = __shfl_sync(FULL, d[LM / 16 - 1][0], src), r3 = __shfl_sync(FULL, d[LM / 16 - 1][2], src);
    if (lane & 16) ck = (lane & 8) ? r3 : r2;
  }
  return ck;
}

// Same dots without tensor cores (dstate not a multiple of 16).
template <int LM, int NCH>
__device__ __forceinline__ float dots_fma(const uint16_t* Bw, int BS, const float4 (&cm)[NCH], int m, int N,
                                          int lane) {
  float pk[LM];
#pragma unroll
  for (int k = 0; k < LM; k++) {
    pk[k] = 0.f;
    if (k < m) {
#pragma unroll
      for (int jj = 0; jj < NCH; jj++) {
        const int c = lane + 32 * jj;
        if (c * 4 < N) pk[k] += dot4(load_bf4(Bw + (size_t)k * BS + c * 4), cm[jj]);
      }
    }
  }
  const float red = reduce_transpose<LM>(pk, lane);
  return __shfl_sync(FULL, red, LM == 16 ? (2 * lane) & 31 : lane);
}

template <int LM, int NCH, bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 1) m2_step_kernel(M2Args a, Layout lay, int ntiles) {
  constexpr int G8 = 2 / NCH;  // 8-row groups a consumer warp holds at most
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* full_t = bars;
  uint64_t* empty_t = bars + MAXB;
  uint64_t* full_r = bars + 2 * MAXB;
  uint64_t* empty_r = bars + 3 * MAXB;
  unsigned char* tiles = smem + BAR_BYTES;
  unsigned char* recs = tiles + (size_t)lay.T * lay.tile_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < MAXB; s++) {
      mbar_init(&full_t[s], 1);
      mbar_init(&empty_t[s], NCONS);
      mbar_init(&full_r[s], 1);
      mbar_init(&empty_r[s], NCONS);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == NW) {
    producer(a, lay, tiles, recs, bars, ntiles, lane);
    return;
  }
  const int group = warp / NCONS, wg = warp % NCONS;
  const int L = a.L, N = a.N, P = a.P, PB = a.PB, H = a.H, T = lay.T, RB = lay.R;
  for (int j = group, t = blockIdx.x + group * gridDim.x; t < ntiles; j += NG, t += NG * gridDim.x) {
    const int jr = j % RB, jt = j % T;
    const unsigned char* rb = recs + (size_t)jr * lay.rec_bytes;
    const unsigned char* tb = tiles + (size_t)jt * lay.tile_bytes;
    if (!__all_sync(FULL, mbar_wait(&full_r[jr], (j / RB) & 1))) {
      if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
      return;
    }
    const Meta mt = *reinterpret_cast<const Meta*>(rb + lay.meta);
    if (mt.skip) {
      const bool ok = __all_sync(FULL, mbar_wait(&full_t[jt], (j / T) & 1));
      if (lane == 0) {
        if (!ok) report(a.status, RSSM_DEV_TIMEOUT);
        mbar_arrive(&empty_t[jt]);
        mbar_arrive(&empty_r[jr]);
      }
      continue;
    }
    const int start = mt.start, count = mt.count, m = count + 1;
    const bool flush = (m == L), rd16 = mt.rd16 != 0;
    const int p0 = mt.pb * PB, R = min(PB, P - p0);
    const size_t bh = (size_t)mt.b * H + mt.h, bg = (size_t)mt.b * a.G + mt.g;
    const uint16_t* xw = reinterpret_cast<const uint16_t*>(rb + lay.xw);
    const uint16_t* zc = reinterpret_cast<const uint16_t*>(rb + lay.zc);
    const uint16_t* Bw = reinterpret_cast<const uint16_t*>(rb + lay.Bw);
    const uint16_t* Cc = reinterpret_cast<const uint16_t*>(rb + lay.Cc);
    const float* dtr = reinterpret_cast<const float*>(rb + lay.dtr);

    // 1. decay weights, lane k = window record k
    int sl = start + lane;
    sl = sl < L ? sl : sl - L;
    const float dtk = (lane < count) ? dtr[sl] : (lane == count ? mt.dt : 0.f);
    float sfx = dtk * mt.A;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float v = __shfl_down_sync(FULL, sfx, o);
      if (lane + o < 32) sfx += v;
    }
    float ex = __shfl_down_sync(FULL, sfx, 1);
    if (lane == 31) ex = 0.f;
    const float Pm = expf(__shfl_sync(FULL, sfx, 0));
    const float wk = dtk * expf(ex);
    // 2. c_k = B_k . C
    float4 cm[NCH];
#pragma unroll
    for (int jj = 0; jj < NCH; jj++) {
      const int c = lane + 32 * jj;
      cm[jj] = (c * 4 < N) ? load_bf4(Cc + c * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float ck = (N % 16 == 0) ? dots_mma<LM>(Bw, lay.BS, Cc, N, lane)
                                   : dots_fma<LM, NCH>(Bw, lay.BS, cm, m, N, lane);
    const float coef = (lane < m) ? fmaf(wk, ck, lane == count ? mt.D : 0.f) : 0.f;

    // 3. this warp's rows of the tile into registers, then release the tile buffer
    int r0w, r1w;
    consumer_rows(R, wg, r0w, r1w);
    const int nrows = r1w - r0w;
    if (!__all_sync(FULL, mbar_wait(&full_t[jt], (j / T) & 1))) {
      if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
      return;
    }
    const float* t32 = reinterpret_cast<const float*>(tb);
    const uint16_t* t16 = reinterpret_cast<const uint16_t*>(tb);
    float4 hv[G8][8][NCH];
#pragma unroll
    for (int gg = 0; gg < G8; gg++)
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) {
          const int c = lane + 32 * jj, row = r0w + gg * 8 + rr;
          hv[gg][rr][jj] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (gg * 8 < nrows && c * 4 < N)
            hv[gg][rr][jj] = rd16 ? load_bf4(t16 + (size_t)row * N + c * 4)
                                  : reinterpret_cast<const float4*>(t32 + (size_t)row * N)[c];
        }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_t[jt]);

    // 4. pre-gate outputs: P (h0 . C)[r] + sum_k coef_k x_k[r]
    float tot[G8];
#pragma unroll
    for (int gg = 0; gg < G8; gg++) {
      tot[gg] = 0.f;
      if (gg * 8 < nrows) {
        float xl[8];
        if (lane < m) {
          const uint4 u = *reinterpret_cast<const uint4*>(xw + (size_t)lane * lay.XS + r0w + gg * 8);
          xl[0] = bf_lo(u.x); xl[1] = bf_hi(u.x); xl[2] = bf_lo(u.y); xl[3] = bf_hi(u.y);
          xl[4] = bf_lo(u.z); xl[5] = bf_hi(u.z); xl[6] = bf_lo(u.w); xl[7] = bf_hi(u.w);
        } else {
#pragma unroll
          for (int rr = 0; rr < 8; rr++) xl[rr] = 0.f;
        }
        float v[8];
#pragma unroll
        for (int rr = 0; rr < 8; rr++) {
          float d = 0.f;
#pragma unroll
          for (int jj = 0; jj < NCH; jj++) d += dot4(hv[gg][rr][jj], cm[jj]);
          v[rr] = fmaf(Pm, d, coef * xl[rr]);
        }
        tot[gg] = reduce_transpose<8>(v, lane);
      }
    }
    {  // lane r < nrows gathers row r's total, gates and stores it
      const int rr = lane & 7;
      const int src = ((rr >> 2) & 1) * 16 + ((rr >> 1) & 1) * 8 + (rr & 1) * 4;
      float mine = __shfl_sync(FULL, tot[0], src);
      if (G8 > 1) {
        const float t1 = __shfl_sync(FULL, tot[G8 - 1], src);
        if (lane & 8) mine = t1;
      }
      if (lane < nrows) {
        const int r = r0w + lane;
        const float zm = bf_to_f(zc[r]);
        const float yv = mine * __fdividef(zm, 1.f + __expf(-zm));
        const size_t oi = bh * P + p0 + r;
        if (OUT_BF16)
          reinterpret_cast<uint16_t*>(a.y)[oi] = f_to_bf(yv);
        else
          reinterpret_cast<float*>(a.y)[oi] = yv;
      }
    }
    if (flush) {  // 5a. fold the window into the rows held in registers, write them once
#pragma unroll
      for (int gg = 0; gg < G8; gg++) {
        if (gg * 8 >= nrows) continue;
        const int r0 = r0w + gg * 8;
#pragma unroll
        for (int rr = 0; rr < 8; rr++)
#pragma unroll
          for (int jj = 0; jj < NCH; jj++) hv[gg][rr][jj] = scale4(Pm, hv[gg][rr][jj]);
        for (int k = 0; k < m; k++) {
          const float w = __shfl_sync(FULL, wk, k);
          const uint4 u = *reinterpret_cast<const uint4*>(xw + (size_t)k * lay.XS + r0);
          const float wx[8] = {w * bf_lo(u.x), w * bf_hi(u.x), w * bf_lo(u.y), w * bf_hi(u.y),
                               w * bf_lo(u.z), w * bf_hi(u.z), w * bf_lo(u.w), w * bf_hi(u.w)};
#pragma unroll
          for (int jj = 0; jj < NCH; jj++) {
            const int c = lane + 32 * jj;
            if (c * 4 < N) {
              const float4 bk = load_bf4(Bw + (size_t)k * lay.BS + c * 4);
#pragma unroll
              for (int rr = 0; rr < 8; rr++) hv[gg][rr][jj] = fma4(wx[rr], bk, hv[gg][rr][jj]);
            }
          }
        }
        const size_t toff = (bh * P + p0 + r0) * N;
#pragma unroll
        for (int rr = 0; rr < 8; rr++)
#pragma unroll
          for (int jj = 0; jj < NCH; jj++) {
            const int c = lane + 32 * jj;
            if (c * 4 < N) {
              const size_t o = toff + (size_t)rr * N + c * 4;
              __stcs(reinterpret_cast<float4*>(a.ckpt + o), hv[gg][rr][jj]);
              if (a.ckpt_read) __stcs(reinterpret_cast<uint2*>(a.ckpt_read + o), f4_to_bf4(hv[gg][rr][jj]));
            }
          }
      }
    } else {  // 5b. append the current record: x, z rows of this warp; dt, B, C once
      const int slot = start + count < L ? start + count : start + count - L;
      const size_t rrow = (bh * L + slot) * P + p0;
      if (lane < (nrows >> 3)) {
        const int r = r0w + lane * 8;
        *reinterpret_cast<uint4*>(a.rx + rrow + r) =
            *reinterpret_cast<const uint4*>(xw + (size_t)count * lay.XS + r);
        *reinterpret_cast<uint4*>(a.rz + rrow + r) = *reinterpret_cast<const uint4*>(zc + r);
      }
      if (wg == 0 && mt.pb == 0) {
        if (lane == 0) a.rdt[bh * pad4(L) + slot] = mt.dt;
        if (mt.h == mt.g * (H / a.G)) {  // the group's first head stores the group rows
          const size_t brow = (bg * L + slot) * N;
          for (int i = lane; i < (N >> 3); i += 32) {
            *reinterpret_cast<uint4*>(a.rB + brow + i * 8) =
                *reinterpret_cast<const uint4*>(Bw + (size_t)count * lay.BS + i * 8);
            *reinterpret_cast<uint4*>(a.rC + brow + i * 8) = *reinterpret_cast<const uint4*>(Cc + i * 8);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_r[jr]);
  }
}

template <int LM, int NCH, bool OUT_BF16>
cudaError_t launch_step(const M2Args& a, cudaStream_t st) {
  const DeviceInfo di = device_info();
  const Layout lay = make_layout(a.PB, a.N, a.L, LM, di.smem_optin);
  if (lay.T < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = BAR_BYTES + (size_t)lay.T * lay.tile_bytes + (size_t)lay.R * lay.rec_bytes;
  const int ntiles = a.Bt * a.H * a.nPB;
  const int grid = ntiles < di.sms ? ntiles : di.sms;
  auto k = m2_step_kernel<LM, NCH, OUT_BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<grid, THREADS, smem, st>>>(a, lay, ntiles);
  return cudaGetLastError();
}

}  // namespace

cudaError_t m2_step_launch(const M2Args& a, int out_bf16, cudaStream_t st) {
  if (a.Bt * a.H * a.nPB == 0) return cudaSuccess;
  const bool small_window = a.L <= 16, narrow = a.N <= 128;
  if (small_window) {
    if (narrow) return out_bf16 ? launch_step<16, 1, true>(a, st) : launch_step<16, 1, false>(a, st);
    return out_bf16 ? launch_step<16, 2, true>(a, st) : launch_step<16, 2, false>(a, st);
  }
  if (narrow) return out_bf16 ? launch_step<32, 1, true>(a, st) : launch_step<32, 1, false>(a, st);
  return out_bf16 ? launch_step<32, 2, true>(a, st) : launch_step<32, 2, false>(a, st);
}

}  // namespace rssm
