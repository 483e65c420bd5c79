// Device helpers shared by the librssm kernels: bf16 packing, warp
// reductions, mbarrier + bulk-copy (TMA, non-tensor) wrappers and the
// bounded waits every kernel uses on them.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rssm.h"

namespace rssm {

constexpr unsigned FULL = 0xffffffffu;
// A bounded wait gives up after this many nanoseconds and reports
// RSSM_DEV_TIMEOUT; a healthy bulk copy lands in microseconds.
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

// ---------------------------------------------------------------- bf16 packing

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ float4 bf4_to_f4(uint2 u) {
  return make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
}

__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // RNE, a in the low half
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint2 f4_to_bf4(float4 v) {
  return make_uint2(pack_bf2(v.x, v.y), pack_bf2(v.z, v.w));
}

__device__ __forceinline__ uint16_t f_to_bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ float bf_to_f(uint16_t v) { return __uint_as_float(((uint32_t)v) << 16); }

__device__ __forceinline__ float4 load_bf4(const uint16_t* p) {
  return bf4_to_f4(*reinterpret_cast<const uint2*>(p));
}

// fp16 <-> fp32 (the read copy's other element type), through the CUDA half intrinsics.
__device__ __forceinline__ float4 load_h4(const uint16_t* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ uint2 f4_to_h4(float4 v) {
  const __half2 lo = __floats2half2_rn(v.x, v.y), hi = __floats2half2_rn(v.z, v.w);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

// The read copy's four elements at p as fp32, and four fp32 rounded (RNE) to
// it; f16 selects fp16 over bf16 (uniform over a launch).
__device__ __forceinline__ float4 load_rc4(const uint16_t* p, bool f16) { return f16 ? load_h4(p) : load_bf4(p); }
__device__ __forceinline__ uint2 to_rc4(float4 v, bool f16) { return f16 ? f4_to_h4(v) : f4_to_bf4(v); }

// fp8 e4m3 read copy: four values at p (unscaled), and four fp32 rounded to
// e4m3 (nearest even, saturating at +-448) packed in one word, through the
// CUDA fp8 conversion intrinsics.
__device__ __forceinline__ float4 load_f8x4(const uint8_t* p) {
  const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
  const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(u & 0xffffu), __NV_E4M3);
  const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(u >> 16), __NV_E4M3);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ uint32_t f4_to_f8x4(float4 v) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v.x, v.y), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v.z, v.w), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// Largest magnitude e4m3 represents; an fp8 read-copy row is stored as
// value / scale with scale = max|row| / E4M3_MAX.
constexpr float E4M3_MAX = 448.f;

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

__device__ __forceinline__ float4 fma4(float s, float4 a, float4 c) {
  return make_float4(fmaf(s, a.x, c.x), fmaf(s, a.y, c.y), fmaf(s, a.z, c.z), fmaf(s, a.w, c.w));
}

__device__ __forceinline__ float4 scale4(float s, float4 a) {
  return make_float4(s * a.x, s * a.y, s * a.z, s * a.w);
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

// A 16-byte aligned float4 (shared or global memory).
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
  return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w);
}

// Eight bf16 values (one uint4) to fp32.
__device__ __forceinline__ void unpack8(uint4 u, float* f) {
  f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
  f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
}

// Ring slot of s in [0, 2L).
__device__ __forceinline__ int wrap(int s, int L) { return s < L ? s : s - L; }

// An output element, fp32 or bf16 (round to nearest even).
template <bool OUT_BF16>
__device__ __forceinline__ void store_out(void* y, size_t i, float v) {
  if (OUT_BF16)
    reinterpret_cast<uint16_t*>(y)[i] = f_to_bf(v);
  else
    reinterpret_cast<float*>(y)[i] = v;
}

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

// ---------------------------------------------------------------- reductions

// Every lane must call these (full-warp shuffles).
__device__ __forceinline__ uint4 shfl_u4(uint4 v, int src) {
  return make_uint4(__shfl_sync(FULL, v.x, src), __shfl_sync(FULL, v.y, src), __shfl_sync(FULL, v.z, src),
                    __shfl_sync(FULL, v.w, src));
}

// Sum over the four lanes of a quad.
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(FULL, v, 1);
  v += __shfl_xor_sync(FULL, v, 2);
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

// Sum eight per-lane partials v[0..7] over the warp. Afterwards v[0] of a
// lane holds the total of partial index reduce8_row(lane); the four lanes
// that share bits 4..2 of the lane id hold the same total. 9 shuffles
// instead of 40 for eight separate butterflies.
__device__ __forceinline__ int reduce8_row(int lane) {
  return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}

__device__ __forceinline__ void reduce8(float (&v)[8], int lane) {
  const bool b16 = lane & 16;
#pragma unroll
  for (int i = 0; i < 4; i++) {
    float send = b16 ? v[i] : v[i + 4];
    float keep = b16 ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(FULL, send, 16);
  }
  const bool b8 = lane & 8;
#pragma unroll
  for (int i = 0; i < 2; i++) {
    float send = b8 ? v[i] : v[i + 2];
    float keep = b8 ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(FULL, send, 8);
  }
  const bool b4 = lane & 4;
  {
    float send = b4 ? v[0] : v[1];
    float keep = b4 ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(FULL, send, 4);
  }
  v[0] += __shfl_xor_sync(FULL, v[0], 2);
  v[0] += __shfl_xor_sync(FULL, v[0], 1);
}

// Sum V per-lane partials p[0..V) (V = 8, 16 or 32) over the warp by a
// transposed butterfly: V-1 shuffles in all instead of 5V. Afterwards p[0] of
// lane l holds the total of partial index idx(l): for V = 32, idx(l) = l; for
// V = 16, idx(l) = l >> 1; for V = 8, idx(l) = reduce8_row(l).
template <int V>
__device__ __forceinline__ float reduce_transpose(float (&p)[V], int lane) {
#pragma unroll
  for (int lvl = 0; lvl < 5; lvl++) {
    const int off = 16 >> lvl;
    const int n = V >> lvl;  // partials still held before this level
    if (n > 1) {
      const bool hi = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; i++) {
        const float send = hi ? p[i] : p[i + n / 2];
        const float keep = hi ? p[i + n / 2] : p[i];
        p[i] = keep + __shfl_xor_sync(FULL, send, off);
      }
    } else {
      p[0] += __shfl_xor_sync(FULL, p[0], off);
    }
  }
  return p[0];
}

// One row of 128 fp32 values (lane: the float4 at column 4 lane) into the fp8
// read copy: stored as value * (448 / max|row|), nearest even, with the row's
// scale max|row| / 448 in scales[row] (0 for a row of zeros). Every lane must
// call this.
__device__ __forceinline__ void store_f8_row(uint8_t* q, float* scales, size_t row, float4 v, int lane) {
  float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
  const float inv = m > 0.f ? E4M3_MAX / m : 0.f;
  *reinterpret_cast<uint32_t*>(q + row * 128 + lane * 4) = f4_to_f8x4(scale4(inv, v));
  if (lane == 0) scales[row] = m / E4M3_MAX;
}

// ---------------------------------------------------------------- emulated read precisions

// Largest code magnitude of a scaled emulated format (RSSM_EMU_E4M3, _E5M2,
// _INT8); 1 for the unscaled ones.
__device__ __forceinline__ float emu_qmax(int fmt) {
  return fmt == RSSM_EMU_E4M3 ? 448.f : fmt == RSSM_EMU_E5M2 ? 57344.f : fmt == RSSM_EMU_INT8 ? 127.f : 1.f;
}

// An emulated format, taken once per thread (see emu_quantise4).
struct EmuQ {
  int fmt;     // RSSM_EMU_*
  float vmax;  // the largest finite value
};

__device__ __forceinline__ EmuQ emu_params(int fmt) {
  EmuQ q;
  q.fmt = fmt;
  q.vmax = fmt == RSSM_EMU_BF16 ? 0x1.fep127f : fmt == RSSM_EMU_F16 ? 65504.f : emu_qmax(fmt);
  return q;
}

// Four values rounded to nearest, ties to even, into an emulated format and
// back to fp32, saturating at the format's largest finite value, through
// CUDA's conversions: e4m3 and e5m2 by the saturating fp8 conversion; bf16
// and fp16 by the round-to-nearest conversions after a clamp to the largest
// finite value (so that nothing rounds to infinity); int8 by rintf (half to
// even), clamped to [-127, 127]. The format is uniform over the launch.
__device__ __forceinline__ float4 emu_quantise4(float4 t, const EmuQ& q) {
  auto clamp = [&](float x) { return fminf(fmaxf(x, -q.vmax), q.vmax); };
  auto fp8 = [](float a, float b, __nv_fp8_interpretation_t k) {
    const __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, k);
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(p, k);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
  };
  float2 lo, hi;
  switch (q.fmt) {
    case RSSM_EMU_BF16:
      lo = __bfloat1622float2(__floats2bfloat162_rn(clamp(t.x), clamp(t.y)));
      hi = __bfloat1622float2(__floats2bfloat162_rn(clamp(t.z), clamp(t.w)));
      break;
    case RSSM_EMU_F16:
      lo = __half22float2(__floats2half2_rn(clamp(t.x), clamp(t.y)));
      hi = __half22float2(__floats2half2_rn(clamp(t.z), clamp(t.w)));
      break;
    case RSSM_EMU_E4M3:
      lo = fp8(t.x, t.y, __NV_E4M3);
      hi = fp8(t.z, t.w, __NV_E4M3);
      break;
    case RSSM_EMU_E5M2:
      lo = fp8(t.x, t.y, __NV_E5M2);
      hi = fp8(t.z, t.w, __NV_E5M2);
      break;
    default:  // int8
      lo = make_float2(fminf(fmaxf(rintf(t.x), -127.f), 127.f), fminf(fmaxf(rintf(t.y), -127.f), 127.f));
      hi = make_float2(fminf(fmaxf(rintf(t.z), -127.f), 127.f), fminf(fmaxf(rintf(t.w), -127.f), 127.f));
  }
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// Maxima of V per-lane values over the warp, transposed like
// reduce_transpose: afterwards m[0] of lane l is the maximum of index idx(l).
template <int V>
__device__ __forceinline__ float max_transpose(float (&m)[V], int lane) {
#pragma unroll
  for (int lvl = 0; lvl < 5; lvl++) {
    const int off = 16 >> lvl;
    const int n = V >> lvl;
    if (n > 1) {
      const bool hi = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; i++) {
        const float send = hi ? m[i] : m[i + n / 2];
        const float keep = hi ? m[i + n / 2] : m[i];
        m[i] = fmaxf(keep, __shfl_xor_sync(FULL, send, off));
      }
    } else {
      m[0] = fmaxf(m[0], __shfl_xor_sync(FULL, m[0], off));
    }
  }
  return m[0];
}

__device__ __forceinline__ float abs_max4(float4 v) {
  return fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
}

// ---------------------------------------------------------------- warp-level tensor-core pieces

// Four 8x8 bf16 matrices from shared memory; lane l gives the address of row
// (l & 7) of matrix (l >> 3). Rows are 16 bytes, 16-byte aligned.
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* smem_row) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_row))));
}

// d += A (16x16 bf16, row-major fragment) * B (16x8 bf16, column fragment), fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// d += A (16x8 tf32, row-major fragment: a0 (g, t), a1 (g+8, t), a2 (g, t+4),
// a3 (g+8, t+4)) * B (8x8 tf32, column fragment: b0 (t, g), b1 (t+4, g)), fp32
// accumulate; d0, d1 = (g, 2t), (g, 2t+1), d2, d3 = (g+8, 2t), (g+8, 2t+1);
// g = lane / 4, t = lane % 4.
__device__ __forceinline__ void mma_tf32_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp32 x = hi + lo with hi exactly representable in tf32 (the top 11
// significand bits) and lo = x - hi exact in fp32; a tf32 mma reads only the
// top 19 bits of each operand, so lo enters truncated to 11 significant bits.
// Two tf32 products with an operand that is exact in tf32 (a bf16 or fp16
// value) then recover x * y to within 2^-20 relative.
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
  hi = __float_as_uint(x) & 0xffffe000u;
  lo = __float_as_uint(x - __uint_as_float(hi));
}

// ---------------------------------------------------------------- status

__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// State row of batch row b: b itself, or slots[b] of n state rows when a slot
// table is given. A padding row (slot -1) and a slot outside [0, n) both give
// -1; the latter is reported (RSSM_DEV_BAD_SLOT) by the threads for which
// `reporter` holds (one per row is enough).
__device__ __forceinline__ int state_slot(const int32_t* slots, int n, int b, int32_t* status, bool reporter) {
  if (!slots) return b;
  const int s = __ldg(slots + b);
  if (s >= 0 && s < n) return s;
  if (s != -1 && reporter) report(status, RSSM_DEV_BAD_SLOT);
  return -1;
}

// ---------------------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// Global -> shared bulk copy (TMA, non-tensor form) completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses, e.g. before refilling a buffer.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or the hint (ns) runs out, so a waiting warp takes no issue slots.
__device__ __forceinline__ bool mbar_test_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(20000u)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete; false after WAIT_LIMIT_NS.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_test_sleep(bar, parity)) return true;
    if (global_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
}

// Wait for a bulk copy; on timeout report it, wait once more (bounded) so the
// copy is not left writing into shared memory of an exited block, and
// return false so the caller can skip the tile.
__device__ __forceinline__ bool mbar_wait_or_report(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_wait(bar, parity)) return true;
  report(status, RSSM_DEV_TIMEOUT);
  mbar_wait(bar, parity);
  return false;
}

}  // namespace rssm
