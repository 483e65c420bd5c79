// ReplaySSM AR decode step for Mamba-2 on sm_103a: a persistent,
// warp-specialised kernel ("How ReplaySSM works": non-flush steps read the
// checkpoint and the window and store no state; the L-th step folds the window
// into the checkpoint and writes it once).
//
// One CTA per SM walks the (sequence, head, row block) tiles of the layer in
// a static round-robin. Warp 4 is the producer: for each tile it fills one
// stage of an S-deep shared-memory ring with bulk copies (TMA, non-tensor;
// never multicast) of the checkpoint rows (fp32, or the bf16 read copy on a
// non-flush step), the window records of that (sequence, head) in window order
// (x rows, group B rows, the dt ring row) and the current record, all
// completing on the stage's `full` mbarrier. Cursors, dt, A and D of the next
// 32 tiles are prefetched one lane per tile, so the producer's critical path is
// a few shuffles and copy issues per tile. Warps 0-3 consume: each owns a
// quarter of the tile's rows and
//   1. takes the decay weights of the m <= 32 window records from one warp
//      suffix scan (lane k = record k): w_k = dt_k exp(A sum_{j>k} dt_j),
//      P = exp(A sum_j dt_j);
//   2. forms c_k = B_k . C for every record at once (per-lane partials over
//      the lane's column chunks, then one transposed butterfly reduction);
//   3. for each 8-row group, adds lane k's term (w_k c_k [+ D if k is the
//      current record]) x_k[r] to P * (h0 . C) partials, so a single 8-row
//      transposed reduction yields y[r] = P (h0 C)[r] + sum_k w_k c_k x_k[r]
//      + D x[r], then gates it by silu(z[r]);
//   4. on a flush, folds h1 = P h0 + sum_k (w_k x_k) B_k^T from the rows it
//      holds in registers and streams them out (and the bf16 read copy);
//   5. otherwise appends the current record to its ring slot;
// and releases the stage on its `empty` mbarrier. All waits are bounded.
#include "persistent.cuh"

namespace rssm {

namespace {

using namespace persistent;

struct Meta {
  int start, count, b, h;
  int pb, skip, rd16, pad0;
  float dt, A, D, pad1;
};

struct Layout {  // byte offsets inside one stage, 128-byte aligned
  uint32_t tile, xw, zc, Bw, Cc, dtr, meta, bytes;
};

inline Layout make_layout(int PB, int N, int L) {
  Layout s{};
  Carver c;
  s.tile = c.take(PB * N * 4);     // checkpoint rows (fp32; bf16 uses the first half)
  s.xw = c.take(L * PB * 2);       // x rows of the window records, window order (bf16)
  s.zc = c.take(PB * 2);           // z rows of the current record
  s.Bw = c.take(L * N * 2);        // B rows of the window records, window order
  s.Cc = c.take(N * 2);            // C of the current record
  s.dtr = c.take(pad4(L) * 4);     // dt ring row (slot order)
  s.meta = c.take(sizeof(Meta));
  s.bytes = c.off;
  return s;
}

// Copy q of a stage fill; returns false if copy q moves nothing.
__device__ __forceinline__ bool stage_copy(const M2Args& a, const Layout& lay, unsigned char* st, int q, int b, int h,
                                           int pb, int start, int count, bool rd16, void*& dst, const void*& src,
                                           uint32_t& bytes) {
  const int L = a.L, N = a.N, P = a.P, PB = a.PB, H = a.H;
  const int g = (h * a.G) / H;
  const int p0 = pb * PB, R = min(PB, P - p0);
  const size_t bh = (size_t)b * H + h, bg = (size_t)b * a.G + g;
  const int n1 = min(count, L - start), n2 = count - n1;
  bytes = 0;
  switch (q) {
    case 0: {
      const size_t off = (bh * P + p0) * N;
      dst = st + lay.tile;
      src = rd16 ? (const void*)(a.ckpt_read + off) : (const void*)(a.ckpt + off);
      bytes = (uint32_t)(R * N * (rd16 ? 2 : 4));
      break;
    }
    case 1: dst = st + lay.xw + (size_t)count * PB * 2; src = a.x + bh * P + p0; bytes = R * 2; break;
    case 2: dst = st + lay.zc; src = a.z + bh * P + p0; bytes = R * 2; break;
    case 3: dst = st + lay.Bw + (size_t)count * N * 2; src = a.B + bg * N; bytes = N * 2; break;
    case 4: dst = st + lay.Cc; src = a.C + bg * N; bytes = N * 2; break;
    case 5:
      dst = st + lay.dtr;
      src = a.rdt + bh * pad4(L);
      bytes = count > 0 ? pad4(L) * 4 : 0;
      break;
    case 6: dst = st + lay.Bw; src = a.rB + (bg * L + start) * N; bytes = n1 * N * 2; break;
    case 7: dst = st + lay.Bw + (size_t)n1 * N * 2; src = a.rB + bg * L * N; bytes = n2 * N * 2; break;
    default:
      if (a.nPB == 1) {  // whole rows: the window's slots are 1 or 2 contiguous runs
        if (q == 8) {
          dst = st + lay.xw;
          src = a.rx + (bh * L + start) * P;
          bytes = n1 * P * 2;
        } else if (q == 9) {
          dst = st + lay.xw + (size_t)n1 * PB * 2;
          src = a.rx + bh * L * P;
          bytes = n2 * P * 2;
        }
      } else {  // row blocks: one copy per window slot
        const int k = q - 8;
        if (k < count) {
          dst = st + lay.xw + (size_t)k * PB * 2;
          src = a.rx + (bh * L + (start + k) % L) * P + p0;
          bytes = R * 2;
        }
      }
  }
  return bytes != 0;
}

__device__ void producer(const M2Args& a, const Layout& lay, int S, unsigned char* stages, uint64_t* full,
                         uint64_t* empty, int ntiles, int lane) {
  const int G = gridDim.x, L = a.L;
  const int ncopies = a.nPB == 1 ? 10 : 8 + L;
  int j = 0;
  for (int base = blockIdx.x; base < ntiles; base += 32 * G) {
    // lane i prefetches what tile base + i*G needs before its copies can be issued
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
      const int stage = j % S;
      unsigned char* st = stages + (size_t)stage * lay.bytes;
      if (j >= S && !__all_sync(FULL, mbar_wait(&empty[stage], ((j / S) - 1) & 1))) {
        if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
        return;
      }
      const int start = __shfl_sync(FULL, cur.x, i), count = __shfl_sync(FULL, cur.y, i);
      const int pending = __shfl_sync(FULL, cur.z, i);
      const float dtt = __shfl_sync(FULL, dtl, i), At = __shfl_sync(FULL, Al, i), Dt = __shfl_sync(FULL, Dl, i);
      int b, h, pb;
      decode_tile(a, base + i * G, b, h, pb);
      // invalid cursors are skipped here and reported by the cursor kernel
      const bool valid = start >= 0 && start < L && count >= 0 && count < L && pending == 0;
      const bool rd16 = valid && (count + 1 < L) && a.ckpt_read != nullptr;
      if (lane == 0) {
        Meta* mt = reinterpret_cast<Meta*>(st + lay.meta);
        *mt = Meta{start, count, b, h, pb, valid ? 0 : 1, rd16 ? 1 : 0, 0, dtt, At, Dt, 0.f};
      }
      if (!valid) {
        if (lane == 0) mbar_arrive(&full[stage]);
        __syncwarp();
        continue;
      }
      uint32_t mine = 0;
      for (int q = lane; q < ncopies; q += 32) {
        void* d;
        const void* s;
        uint32_t n;
        if (stage_copy(a, lay, st, q, b, h, pb, start, count, rd16, d, s, n)) mine += n;
      }
      const uint32_t total = __reduce_add_sync(FULL, mine);
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], total);
      __syncwarp();
      for (int q = lane; q < ncopies; q += 32) {
        void* d;
        const void* s;
        uint32_t n;
        if (stage_copy(a, lay, st, q, b, h, pb, start, count, rd16, d, s, n)) bulk_load(d, s, n, &full[stage]);
      }
    }
  }
}

template <int LM, int NCH, bool OUT_BF16>
__device__ __forceinline__ void consume_tile(const M2Args& a, const Layout& lay, const unsigned char* st,
                                             const Meta& mt, int warp, int lane) {
  const int L = a.L, N = a.N, P = a.P, PB = a.PB, H = a.H;
  const int b = mt.b, h = mt.h, pb = mt.pb, start = mt.start, count = mt.count, m = count + 1;
  const int g = (h * a.G) / H;
  const int p0 = pb * PB, R = min(PB, P - p0);
  const bool flush = (m == L), rd16 = mt.rd16 != 0;
  const size_t bh = (size_t)b * H + h, bg = (size_t)b * a.G + g;
  const uint16_t* xw = reinterpret_cast<const uint16_t*>(st + lay.xw);
  const uint16_t* zc = reinterpret_cast<const uint16_t*>(st + lay.zc);
  const uint16_t* Bw = reinterpret_cast<const uint16_t*>(st + lay.Bw);
  const uint16_t* Cc = reinterpret_cast<const uint16_t*>(st + lay.Cc);
  const float* dtr = reinterpret_cast<const float*>(st + lay.dtr);
  const float* t32 = reinterpret_cast<const float*>(st + lay.tile);
  const uint16_t* t16 = reinterpret_cast<const uint16_t*>(st + lay.tile);

  float4 cm[NCH];
#pragma unroll
  for (int j = 0; j < NCH; j++) {
    const int c = lane + 32 * j;
    cm[j] = (c * 4 < N) ? load_bf4(Cc + c * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // 1. decay weights, lane k = window record k
  const float dtk = (lane < count) ? dtr[(start + lane) % L] : (lane == count ? mt.dt : 0.f);
  float sfx = dtk * mt.A;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_down_sync(FULL, sfx, o);
    if (lane + o < 32) sfx += t;
  }
  float ex = __shfl_down_sync(FULL, sfx, 1);
  if (lane == 31) ex = 0.f;
  const float Pm = expf(__shfl_sync(FULL, sfx, 0));
  const float wk = dtk * expf(ex);
  // 2. c_k = B_k . C for all records: lane partials, transposed reduction
  float pk[LM];
#pragma unroll
  for (int k = 0; k < LM; k++) {
    pk[k] = 0.f;
    if (k < m) {
#pragma unroll
      for (int j = 0; j < NCH; j++) {
        const int c = lane + 32 * j;
        if (c * 4 < N) pk[k] += dot4(load_bf4(Bw + (size_t)k * N + c * 4), cm[j]);
      }
    }
  }
  const float red = reduce_transpose<LM>(pk, lane);
  const float ck = __shfl_sync(FULL, red, LM == 16 ? (2 * lane) & 31 : lane);
  const float coef = (lane < m) ? wk * ck + (lane == count ? mt.D : 0.f) : 0.f;

  int r0w, r1w;
  consumer_rows(R, warp, r0w, r1w);
  for (int r0 = r0w; r0 < r1w; r0 += 8) {
    // 3. outputs of rows r0..r0+7
    float xl[8];
    if (lane < m) {
      const uint4 u = *reinterpret_cast<const uint4*>(xw + (size_t)lane * PB + r0);
      xl[0] = bf_lo(u.x); xl[1] = bf_hi(u.x); xl[2] = bf_lo(u.y); xl[3] = bf_hi(u.y);
      xl[4] = bf_lo(u.z); xl[5] = bf_hi(u.z); xl[6] = bf_lo(u.w); xl[7] = bf_hi(u.w);
    } else {
#pragma unroll
      for (int rr = 0; rr < 8; rr++) xl[rr] = 0.f;
    }
    float4 hv[8][NCH];
    float v[8];
#pragma unroll
    for (int rr = 0; rr < 8; rr++) {
      float d = 0.f;
#pragma unroll
      for (int j = 0; j < NCH; j++) {
        const int c = lane + 32 * j;
        if (c * 4 < N) {
          hv[rr][j] = rd16 ? load_bf4(t16 + (size_t)(r0 + rr) * N + c * 4)
                           : reinterpret_cast<const float4*>(t32 + (size_t)(r0 + rr) * N)[c];
        } else {
          hv[rr][j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        d += dot4(hv[rr][j], cm[j]);
      }
      v[rr] = fmaf(Pm, d, coef * xl[rr]);
    }
    reduce_transpose<8>(v, lane);
    if ((lane & 3) == 0) {
      const int r = r0 + reduce8_row(lane);
      const float zm = bf_to_f(zc[r]);
      const size_t oi = bh * P + p0 + r;
      const float yv = v[0] * silu(zm);
      if (OUT_BF16)
        reinterpret_cast<uint16_t*>(a.y)[oi] = f_to_bf(yv);
      else
        reinterpret_cast<float*>(a.y)[oi] = yv;
    }
    // 4. flush: fold the window into the rows held in registers
    if (flush) {
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
#pragma unroll
        for (int j = 0; j < NCH; j++) hv[rr][j] = scale4(Pm, hv[rr][j]);
      for (int k = 0; k < m; k++) {
        const float w = __shfl_sync(FULL, wk, k);
        const uint4 u = *reinterpret_cast<const uint4*>(xw + (size_t)k * PB + r0);
        const float wx[8] = {w * bf_lo(u.x), w * bf_hi(u.x), w * bf_lo(u.y), w * bf_hi(u.y),
                             w * bf_lo(u.z), w * bf_hi(u.z), w * bf_lo(u.w), w * bf_hi(u.w)};
#pragma unroll
        for (int j = 0; j < NCH; j++) {
          const int c = lane + 32 * j;
          if (c * 4 < N) {
            const float4 bk = load_bf4(Bw + (size_t)k * N + c * 4);
#pragma unroll
            for (int rr = 0; rr < 8; rr++) hv[rr][j] = fma4(wx[rr], bk, hv[rr][j]);
          }
        }
      }
      const size_t toff = (bh * P + p0 + r0) * N;
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
#pragma unroll
        for (int j = 0; j < NCH; j++) {
          const int c = lane + 32 * j;
          if (c * 4 < N) {
            const size_t o = toff + (size_t)rr * N + c * 4;
            __stcs(reinterpret_cast<float4*>(a.ckpt + o), hv[rr][j]);
            if (a.ckpt_read) __stcs(reinterpret_cast<uint2*>(a.ckpt_read + o), f4_to_bf4(hv[rr][j]));
          }
        }
    }
  }
  // 5. non-flush: append the current record (x, z rows of this warp; dt, B, C once)
  if (!flush) {
    const int slot = (start + count) % L;
    const size_t rrow = (bh * L + slot) * P + p0;
    for (int i = lane; i < ((r1w - r0w) >> 3); i += 32) {
      const int r = r0w + i * 8;
      *reinterpret_cast<uint4*>(a.rx + rrow + r) = *reinterpret_cast<const uint4*>(xw + (size_t)count * PB + r);
      *reinterpret_cast<uint4*>(a.rz + rrow + r) = *reinterpret_cast<const uint4*>(zc + r);
    }
    if (warp == 0 && pb == 0) {
      if (lane == 0) a.rdt[bh * pad4(L) + slot] = mt.dt;
      if (h == g * (H / a.G)) {  // the group's first head stores the group rows
        const size_t brow = (bg * L + slot) * N;
        for (int i = lane; i < (N >> 3); i += 32) {
          *reinterpret_cast<uint4*>(a.rB + brow + i * 8) =
              *reinterpret_cast<const uint4*>(Bw + (size_t)count * N + i * 8);
          *reinterpret_cast<uint4*>(a.rC + brow + i * 8) = *reinterpret_cast<const uint4*>(Cc + i * 8);
        }
      }
    }
  }
}

template <int LM, int NCH, bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 1) m2_step_kernel(M2Args a, Layout lay, int S, int ntiles) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + MAX_STAGES;
  unsigned char* stages = smem + BAR_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  init_ring(full, S);
  if (warp == NCW) {
    producer(a, lay, S, stages, full, empty, ntiles, lane);
    return;
  }
  const int group = warp / NCONS, wg = warp % NCONS;
  for (int j = group, t = blockIdx.x + group * gridDim.x; t < ntiles; j += NGROUPS, t += NGROUPS * gridDim.x) {
    const int stage = j % S;
    const unsigned char* st = stages + (size_t)stage * lay.bytes;
    if (!__all_sync(FULL, mbar_wait(&full[stage], (j / S) & 1))) {
      if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
      return;
    }
    const Meta mt = *reinterpret_cast<const Meta*>(st + lay.meta);
    if (!mt.skip) consume_tile<LM, NCH, OUT_BF16>(a, lay, st, mt, wg, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
}

template <int LM, int NCH, bool OUT_BF16>
cudaError_t launch_step(const M2Args& a, cudaStream_t st) {
  const DeviceInfo di = device_info();
  const Layout lay = make_layout(a.PB, a.N, a.L);
  const int S = stages_for(lay.bytes);
  if (S == 0) return cudaErrorInvalidConfiguration;
  const size_t smem = BAR_BYTES + (size_t)S * lay.bytes;
  const int ntiles = a.Bt * a.H * a.nPB;
  const int grid = ntiles < di.sms ? ntiles : di.sms;
  auto k = m2_step_kernel<LM, NCH, OUT_BF16>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k<<<grid, THREADS, smem, st>>>(a, lay, S, ntiles);
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
