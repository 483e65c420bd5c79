// Speculative verify for Mamba-2 on sm_103a, persistent and warp-specialised
// like the AR step ("How ReplaySSM works": drafts are appended to the buffer
// instead of snapshotting state; "ReplaySSM" repository, introduction:
// output-only verification, rollback by moving a pointer).
//
// Tile = (sequence, head, row block). Records of a verify are indexed
// k in [0, count + K): k < count are the committed window records (ring slot
// (start + k) mod L), k >= count the K new ones. If count + K > L the committed
// window is folded first (h' = P h0 + sum_{k<count} w_k x_k B_k^T, written
// once with its bf16 copy) and output i covers records [count, count + i];
// otherwise h' = h0 and output i covers [0, count + i].
//
// The producer warp fills a stage with the checkpoint rows (bf16 read copy
// when there is one and no fold), the x and B rows of every record in record
// order, the z and C rows of the new records and the dt ring row; the new
// records' dt values (strided in memory) are prefetched one lane per tile and
// stored by the producer. Consumer warp w computes the decay weights and
// B.C dots of outputs w, w+4, ... (one warp scan and one transposed
// reduction each) and publishes them in the stage; once the group's four
// warps have arrived on the stage's aux mbarrier each warp folds (if needed)
// and produces all K outputs of its rows,
// adding lane j's term coef_j x_{first+j}[r] into the P (h' C_i) partials of a
// single 8-row reduction per output. x and z rows of the new records go to
// the ring here; B, C and dt rows (shared by other blocks that may still read
// the committed slots a fold overwrites) go in the epilogue kernel.
#include "persistent.cuh"

namespace rssm {

namespace {

using namespace persistent;

constexpr int KPRE = 8;  // new-record dt values prefetched per tile

struct VMeta {
  int start, count, b, h;
  int pb, skip, rd16, fold;
  float A, D, pad0, pad1;
};

struct VLayout {
  uint32_t tile, xw, zn, Bw, Cn, dtr, dtn, coef, meta, bytes;
};

inline VLayout make_vlayout(int PB, int N, int L, int K) {
  VLayout s{};
  Carver c;
  s.tile = c.take(PB * N * 4);        // checkpoint rows
  s.xw = c.take((L + K) * PB * 2);    // x rows of records 0 .. count+K-1
  s.zn = c.take(K * PB * 2);          // z rows of the new records
  s.Bw = c.take((L + K) * N * 2);     // B rows of records 0 .. count+K-1
  s.Cn = c.take(K * N * 2);           // C rows of the new records
  s.dtr = c.take(pad4(L) * 4);        // dt ring row
  s.dtn = c.take(32 * 4);             // dt of the new records
  s.coef = c.take(K * 33 * 4);        // per output: 32 window coefficients + P
  s.meta = c.take(sizeof(VMeta));
  s.bytes = c.off;
  return s;
}

// Copy q of a stage fill (see the header comment); false if it moves nothing.
__device__ __forceinline__ bool vstage_copy(const M2Args& a, const VLayout& lay, unsigned char* st, int q, int b,
                                            int h, int pb, int start, int count, bool rd16, void*& dst,
                                            const void*& src, uint32_t& bytes) {
  const int L = a.L, N = a.N, P = a.P, PB = a.PB, H = a.H, K = a.K, G = a.G;
  const int g = (h * G) / H;
  const int p0 = pb * PB, R = min(PB, P - p0);
  const size_t bh = (size_t)b * H + h, bg = (size_t)b * G + g;
  const int n1 = min(count, L - start), n2 = count - n1;
  bytes = 0;
  if (q < 6) {
    switch (q) {
      case 0: {
        const size_t off = (bh * P + p0) * N;
        dst = st + lay.tile;
        src = rd16 ? (const void*)(a.ckpt_read + off) : (const void*)(a.ckpt + off);
        bytes = (uint32_t)(R * N * (rd16 ? 2 : 4));
        break;
      }
      case 1:
        if (a.nPB == 1) { dst = st + lay.xw; src = a.rx + (bh * L + start) * P; bytes = n1 * P * 2; }
        break;
      case 2:
        if (a.nPB == 1) {
          dst = st + lay.xw + (size_t)n1 * PB * 2;
          src = a.rx + bh * L * P;
          bytes = n2 * P * 2;
        }
        break;
      case 3: dst = st + lay.Bw; src = a.rB + (bg * L + start) * N; bytes = n1 * N * 2; break;
      case 4: dst = st + lay.Bw + (size_t)n1 * N * 2; src = a.rB + bg * L * N; bytes = n2 * N * 2; break;
      case 5: dst = st + lay.dtr; src = a.rdt + bh * pad4(L); bytes = count > 0 ? pad4(L) * 4 : 0; break;
    }
    return bytes != 0;
  }
  q -= 6;
  if (q < 4 * K) {  // new record i: x, z, B, C rows
    const int i = q >> 2, f = q & 3;
    const size_t ih = ((size_t)b * K + i) * H + h, ig = ((size_t)b * K + i) * G + g;
    switch (f) {
      case 0: dst = st + lay.xw + (size_t)(count + i) * PB * 2; src = a.x + ih * P + p0; bytes = R * 2; break;
      case 1: dst = st + lay.zn + (size_t)i * PB * 2; src = a.z + ih * P + p0; bytes = R * 2; break;
      case 2: dst = st + lay.Bw + (size_t)(count + i) * N * 2; src = a.B + ig * N; bytes = N * 2; break;
      case 3: dst = st + lay.Cn + (size_t)i * N * 2; src = a.C + ig * N; bytes = N * 2; break;
    }
    return true;
  }
  q -= 4 * K;
  if (a.nPB > 1 && q < count) {  // row blocks: x rows slot by slot
    dst = st + lay.xw + (size_t)q * PB * 2;
    src = a.rx + (bh * L + (start + q) % L) * P + p0;
    bytes = R * 2;
  }
  return bytes != 0;
}

__device__ void vproducer(const M2Args& a, const VLayout& lay, int S, unsigned char* stages, uint64_t* full,
                          uint64_t* empty, int ntiles, int lane) {
  const int G = gridDim.x, L = a.L, K = a.K, H = a.H;
  const int ncopies = 6 + 4 * K + (a.nPB > 1 ? L : 0);
  int j = 0;
  for (int base = blockIdx.x; base < ntiles; base += 32 * G) {
    const int tl = base + lane * G;
    int4 cur = make_int4(-1, 0, 0, 0);
    float Al = 0.f, Dl = 0.f, dtp[KPRE];
#pragma unroll
    for (int i = 0; i < KPRE; i++) dtp[i] = 0.f;
    if (tl < ntiles) {
      int b, h, pb;
      decode_tile(a, tl, b, h, pb);
      cur = *reinterpret_cast<const int4*>(a.cursors + 4 * (size_t)b);
      Al = a.A[h];
      Dl = a.D[h];
#pragma unroll
      for (int i = 0; i < KPRE; i++)
        if (i < K) dtp[i] = a.dt[((size_t)b * K + i) * H + h];
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
      const float At = __shfl_sync(FULL, Al, i), Dt = __shfl_sync(FULL, Dl, i);
      int b, h, pb;
      decode_tile(a, base + i * G, b, h, pb);
      const bool valid = start >= 0 && start < L && count >= 0 && count <= L && pending == 0;
      const bool fold = count + K > L;
      const bool rd16 = valid && !fold && a.ckpt_read != nullptr;
      // dt of the new records: lane r holds record r's
      float mydt = 0.f;
#pragma unroll
      for (int r = 0; r < KPRE; r++) {
        const float v = __shfl_sync(FULL, dtp[r], i);
        if (lane == r) mydt = v;
      }
      if (valid) {
        float* dtn = reinterpret_cast<float*>(st + lay.dtn);
        if (lane < K) dtn[lane] = lane < KPRE ? mydt : a.dt[((size_t)b * K + lane) * H + h];
      }
      if (lane == 0) {
        VMeta* mt = reinterpret_cast<VMeta*>(st + lay.meta);
        *mt = VMeta{start, count, b, h, pb, valid ? 0 : 1, rd16 ? 1 : 0, fold ? 1 : 0, At, Dt, 0.f, 0.f};
      }
      __syncwarp();  // every lane's dt store happens before lane 0's arrive
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
        if (vstage_copy(a, lay, st, q, b, h, pb, start, count, rd16, d, s, n)) mine += n;
      }
      const uint32_t total = __reduce_add_sync(FULL, mine);
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], total);
      __syncwarp();
      for (int q = lane; q < ncopies; q += 32) {
        void* d;
        const void* s;
        uint32_t n;
        if (vstage_copy(a, lay, st, q, b, h, pb, start, count, rd16, d, s, n)) bulk_load(d, s, n, &full[stage]);
      }
    }
  }
}

// Suffix-scan decay weights of the window whose lane-j dt is `dtj` (0 beyond
// the window): returns w_j; *P = exp(A * sum).
__device__ __forceinline__ float lane_weights(float dtj, float A, int lane, float* P) {
  float sfx = dtj * A;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_down_sync(FULL, sfx, o);
    if (lane + o < 32) sfx += t;
  }
  float ex = __shfl_down_sync(FULL, sfx, 1);
  if (lane == 31) ex = 0.f;
  *P = expf(__shfl_sync(FULL, sfx, 0));
  return dtj * expf(ex);
}

template <int LM, int NCH, bool OUT_BF16>
__device__ __forceinline__ void vconsume_tile(const M2Args& a, const VLayout& lay, unsigned char* st,
                                              const VMeta& mt, int warp, int lane, uint64_t* aux,
                                              uint32_t parity) {
  const int L = a.L, N = a.N, P = a.P, PB = a.PB, H = a.H, K = a.K;
  const int b = mt.b, h = mt.h, pb = mt.pb, start = mt.start, count = mt.count;
  const bool fold = mt.fold != 0, rd16 = mt.rd16 != 0;
  const int first = fold ? count : 0;
  const int p0 = pb * PB, R = min(PB, P - p0);
  const size_t bh = (size_t)b * H + h;
  const uint16_t* xw = reinterpret_cast<const uint16_t*>(st + lay.xw);
  const uint16_t* zn = reinterpret_cast<const uint16_t*>(st + lay.zn);
  const uint16_t* Bw = reinterpret_cast<const uint16_t*>(st + lay.Bw);
  const uint16_t* Cn = reinterpret_cast<const uint16_t*>(st + lay.Cn);
  const float* dtr = reinterpret_cast<const float*>(st + lay.dtr);
  const float* dtn = reinterpret_cast<const float*>(st + lay.dtn);
  float* coef = reinterpret_cast<float*>(st + lay.coef);
  const float* t32 = reinterpret_cast<const float*>(st + lay.tile);
  const uint16_t* t16 = reinterpret_cast<const uint16_t*>(st + lay.tile);

  // 1. coefficients of outputs warp, warp + NCONS, ... published in the stage
  for (int i = warp; i < K; i += NCONS) {
    const int mi = count + i + 1 - first;  // records of output i's window
    const int r = first + lane;            // record of lane
    float dtj = 0.f;
    if (lane < mi) dtj = r < count ? dtr[(start + r) % L] : dtn[r - count];
    float Pi;
    const float wj = lane_weights(dtj, mt.A, lane, &Pi);
    float4 ci[NCH];
#pragma unroll
    for (int jj = 0; jj < NCH; jj++) {
      const int c = lane + 32 * jj;
      ci[jj] = (c * 4 < N) ? load_bf4(Cn + (size_t)i * N + c * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float pk[LM];
#pragma unroll
    for (int k = 0; k < LM; k++) {
      pk[k] = 0.f;
      if (k < mi) {
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) {
          const int c = lane + 32 * jj;
          if (c * 4 < N) pk[k] += dot4(load_bf4(Bw + (size_t)(first + k) * N + c * 4), ci[jj]);
        }
      }
    }
    const float red = reduce_transpose<LM>(pk, lane);
    const float cj = __shfl_sync(FULL, red, LM == 16 ? (2 * lane) & 31 : lane);
    coef[i * 33 + lane] = (lane < mi) ? wj * cj + (lane == mi - 1 ? mt.D : 0.f) : 0.f;
    if (lane == 0) coef[i * 33 + 32] = Pi;
  }
  // fold weights (every warp: lane k = committed record k)
  float wf = 0.f, Pf = 1.f;
  if (fold) wf = lane_weights(lane < count ? dtr[(start + lane) % L] : 0.f, mt.A, lane, &Pf);
  __syncwarp();
  if (lane == 0) mbar_arrive(aux);
  if (!__all_sync(FULL, mbar_wait(aux, parity)) && lane == 0) report(a.status, RSSM_DEV_TIMEOUT);

  int r0w, r1w;
  consumer_rows(R, warp, r0w, r1w);
  const int mlast = count + K - first;  // lanes carrying a record in the widest window
  for (int r0 = r0w; r0 < r1w; r0 += 8) {
    float4 hv[8][NCH];
#pragma unroll
    for (int rr = 0; rr < 8; rr++)
#pragma unroll
      for (int jj = 0; jj < NCH; jj++) {
        const int c = lane + 32 * jj;
        hv[rr][jj] = (c * 4 < N) ? (rd16 ? load_rc4(t16 + (size_t)(r0 + rr) * N + c * 4, a.read_f16)
                                         : reinterpret_cast<const float4*>(t32 + (size_t)(r0 + rr) * N)[c])
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    if (fold) {  // h' = P h0 + sum_{k<count} (w_k x_k) B_k^T, written once
#pragma unroll
      for (int rr = 0; rr < 8; rr++)
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) hv[rr][jj] = scale4(Pf, hv[rr][jj]);
      for (int k = 0; k < count; k++) {
        const float w = __shfl_sync(FULL, wf, k);
        const uint4 u = *reinterpret_cast<const uint4*>(xw + (size_t)k * PB + r0);
        const float wx[8] = {w * bf_lo(u.x), w * bf_hi(u.x), w * bf_lo(u.y), w * bf_hi(u.y),
                             w * bf_lo(u.z), w * bf_hi(u.z), w * bf_lo(u.w), w * bf_hi(u.w)};
#pragma unroll
        for (int jj = 0; jj < NCH; jj++) {
          const int c = lane + 32 * jj;
          if (c * 4 < N) {
            const float4 bk = load_bf4(Bw + (size_t)k * N + c * 4);
#pragma unroll
            for (int rr = 0; rr < 8; rr++) hv[rr][jj] = fma4(wx[rr], bk, hv[rr][jj]);
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
            __stcs(reinterpret_cast<float4*>(a.ckpt + o), hv[rr][jj]);
            if (a.ckpt_read) __stcs(reinterpret_cast<uint2*>(a.ckpt_read + o), to_rc4(hv[rr][jj], a.read_f16));
          }
        }
    }
    // x rows of the lane's record (first + lane)
    float xl[8];
    if (lane < mlast) {
      const uint4 u = *reinterpret_cast<const uint4*>(xw + (size_t)(first + lane) * PB + r0);
      xl[0] = bf_lo(u.x); xl[1] = bf_hi(u.x); xl[2] = bf_lo(u.y); xl[3] = bf_hi(u.y);
      xl[4] = bf_lo(u.z); xl[5] = bf_hi(u.z); xl[6] = bf_lo(u.w); xl[7] = bf_hi(u.w);
    } else {
#pragma unroll
      for (int rr = 0; rr < 8; rr++) xl[rr] = 0.f;
    }
    for (int i = 0; i < K; i++) {
      const float cj = coef[i * 33 + lane], Pi = coef[i * 33 + 32];
      float v[8];
#pragma unroll
      for (int rr = 0; rr < 8; rr++) v[rr] = 0.f;
#pragma unroll
      for (int jj = 0; jj < NCH; jj++) {
        const int c = lane + 32 * jj;
        if (c * 4 < N) {
          const float4 ci = load_bf4(Cn + (size_t)i * N + c * 4);
#pragma unroll
          for (int rr = 0; rr < 8; rr++) v[rr] += dot4(hv[rr][jj], ci);
        }
      }
#pragma unroll
      for (int rr = 0; rr < 8; rr++) v[rr] = fmaf(Pi, v[rr], cj * xl[rr]);
      reduce_transpose<8>(v, lane);
      if ((lane & 3) == 0) {
        const int r = r0 + reduce8_row(lane);
        const float zm = bf_to_f(zn[(size_t)i * PB + r]);
        const size_t oi = (((size_t)b * K + i) * H + h) * P + p0 + r;
        const float yv = v[0] * silu(zm);
        if (OUT_BF16)
          reinterpret_cast<uint16_t*>(a.y)[oi] = f_to_bf(yv);
        else
          reinterpret_cast<float*>(a.y)[oi] = yv;
      }
    }
  }
  // x and z rows of the new records into their ring slots (this warp's rows)
  for (int q = lane; q < K * ((r1w - r0w) >> 3); q += 32) {
    const int i = q / ((r1w - r0w) >> 3), r = r0w + (q % ((r1w - r0w) >> 3)) * 8;
    const int slot = (start + count + i) % L;
    const size_t rrow = (bh * L + slot) * P + p0;
    *reinterpret_cast<uint4*>(a.rx + rrow + r) =
        *reinterpret_cast<const uint4*>(xw + (size_t)(count + i) * PB + r);
    *reinterpret_cast<uint4*>(a.rz + rrow + r) = *reinterpret_cast<const uint4*>(zn + (size_t)i * PB + r);
  }
}

template <int LM, int NCH, bool OUT_BF16>
__global__ void __launch_bounds__(THREADS, 1) m2_verify_kernel(M2Args a, VLayout lay, int S, int ntiles) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* aux = full + 2 * MAX_STAGES;
  unsigned char* stages = smem + BAR_BYTES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  init_ring(full, S);
  if (warp == NCW) {
    vproducer(a, lay, S, stages, full, empty, ntiles, lane);
    return;
  }
  const int group = warp / NCONS, wg = warp % NCONS;
  for (int j = group, t = blockIdx.x + group * gridDim.x; t < ntiles; j += NGROUPS, t += NGROUPS * gridDim.x) {
    const int stage = j % S;
    unsigned char* st = stages + (size_t)stage * lay.bytes;
    if (!__all_sync(FULL, mbar_wait(&full[stage], (j / S) & 1))) {
      if (lane == 0) report(a.status, RSSM_DEV_TIMEOUT);
      return;
    }
    const VMeta mt = *reinterpret_cast<const VMeta*>(st + lay.meta);
    if (!mt.skip) {
      vconsume_tile<LM, NCH, OUT_BF16>(a, lay, st, mt, wg, lane, &aux[stage], (j / S) & 1);
    } else {  // keep the aux barrier's phases in step with the stage's uses
      __syncwarp();
      if (lane == 0) mbar_arrive(&aux[stage]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }
}

template <int LM, int NCH, bool OUT_BF16>
cudaError_t launch_verify(const M2Args& a, cudaStream_t st) {
  const DeviceInfo di = device_info();
  const VLayout lay = make_vlayout(a.PB, a.N, a.L, a.K);
  const int S = stages_for(lay.bytes);
  if (S == 0) return cudaErrorInvalidConfiguration;
  const size_t smem = BAR_BYTES + (size_t)S * lay.bytes;
  const int ntiles = a.Bt * a.H * a.nPB;
  const int grid = ntiles < di.sms ? ntiles : di.sms;
  auto k = m2_verify_kernel<LM, NCH, OUT_BF16>;
  cudaError_t e = prepare(k, smem, false);
  if (e != cudaSuccess) return e;
  k<<<grid, THREADS, smem, st>>>(a, lay, S, ntiles);
  return cudaGetLastError();
}

}  // namespace

cudaError_t m2_verify_launch(const M2Args& a, int out_bf16, cudaStream_t st) {
  if (a.Bt * a.H * a.nPB == 0) return cudaSuccess;
  const bool small_window = a.L <= 16, narrow = a.N <= 128;
  if (small_window) {
    if (narrow) return out_bf16 ? launch_verify<16, 1, true>(a, st) : launch_verify<16, 1, false>(a, st);
    return out_bf16 ? launch_verify<16, 2, true>(a, st) : launch_verify<16, 2, false>(a, st);
  }
  if (narrow) return out_bf16 ? launch_verify<32, 1, true>(a, st) : launch_verify<32, 1, false>(a, st);
  return out_bf16 ? launch_verify<32, 2, true>(a, st) : launch_verify<32, 2, false>(a, st);
}

}  // namespace rssm
