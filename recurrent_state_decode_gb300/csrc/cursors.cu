// Cursor kernels (integer, one thread per sequence) and the fp32 -> bf16
// checkpoint downcast. Rules ("ReplaySSM Caches Inputs Instead of State...",
// "How ReplaySSM works"; "ReplaySSM", introduction, "Cheap rollback"):
//   AR step   needs count < L, pending == 0: count + 1 == L ? count = 0 : count += 1
//   flush     needs pending == 0: start = (start + count) mod L, count = 0
//   commit    needs 0 <= kept <= pending: if folded {start += count mod L; count = 0};
//             count += kept; pending = 0; flags = 0
//   reset     cursor = {0, 0, 0, 0}
// With a slot table, batch row b's cursor is the one of its state slot.
// The compute kernels only read cursors; these run after them in stream
// order, so no block ever sees a cursor another block of the same launch moved.
#include "common.cuh"
#include "kernels.h"

namespace rssm {

__global__ void cursor_kernel(int mode, int32_t* cursors, const int32_t* kept, int batch, int L, int32_t* status,
                              const int32_t* slots, int n_state) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int s = state_slot(slots, n_state, b, status, true);
  if (s < 0) return;
  int4 c = *reinterpret_cast<int4*>(cursors + 4 * (size_t)s);
  const bool range_ok = c.x >= 0 && c.x < L && c.y >= 0 && c.y <= L && c.z >= 0;
  if (!range_ok) {
    report(status, RSSM_DEV_BAD_CURSOR);
    return;
  }
  if (mode == CUR_AR) {
    if (c.z != 0) { report(status, RSSM_DEV_PENDING); return; }
    if (c.y == L) { report(status, RSSM_DEV_WINDOW_FULL); return; }
    c.y = (c.y + 1 == L) ? 0 : c.y + 1;
  } else if (mode == CUR_FLUSH) {
    if (c.z != 0) { report(status, RSSM_DEV_PENDING); return; }
    c.x = (c.x + c.y) % L;
    c.y = 0;
  } else {  // CUR_COMMIT
    const int kb = kept[b];
    if (kb < 0 || kb > c.z) { report(status, RSSM_DEV_BAD_KEPT); return; }
    if (c.w & 1) {
      c.x = (c.x + c.y) % L;
      c.y = 0;
    }
    c.y += kb;
    c.z = 0;
    c.w = 0;
  }
  *reinterpret_cast<int4*>(cursors + 4 * (size_t)s) = c;
}

__global__ void reset_kernel(int32_t* cursors, const int32_t* slots, int n, int batch, int32_t* status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int s = slots[i];
  if (s < 0 || s >= batch) {
    report(status, RSSM_DEV_BAD_SLOT);
    return;
  }
  *reinterpret_cast<int4*>(cursors + 4 * (size_t)s) = make_int4(0, 0, 0, 0);
}

__global__ void downcast_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst, size_t n, bool f16) {
  const size_t n4 = n >> 2;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(src) + i);
    __stcs(reinterpret_cast<uint2*>(dst) + i, to_rc4(v, f16));
  }
  if (blockIdx.x == 0 && threadIdx.x < (n & 3)) {
    const size_t i = (n4 << 2) + threadIdx.x;
    dst[i] = f16 ? __half_as_ushort(__float2half_rn(src[i])) : f_to_bf(src[i]);
  }
}

// fp8 read copy, one warp per row of 128 values; the row scales follow the
// rows * 128 bytes of e4m3 values.
__global__ void downcast_f8_kernel(const float* __restrict__ src, uint8_t* __restrict__ dst, size_t rows) {
  const int lane = threadIdx.x & 31;
  const size_t row = (size_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;  // uniform over the warp
  const float4 v = __ldcs(reinterpret_cast<const float4*>(src + row * 128) + lane);
  store_f8_row(dst, reinterpret_cast<float*>(dst + rows * 128), row, v, lane);
}

// Self-test of the bounded wait every kernel uses for its bulk copies: one
// thread arms an mbarrier for 16 bytes that no copy delivers, so its wait gives
// up after the limit and reports RSSM_DEV_TIMEOUT. No copy is in flight, so
// nothing writes into the block's shared memory after it leaves.
__global__ void bounded_wait_selftest_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_arrive_expect_tx(&bar, 16);
  mbar_wait_or_report(&bar, 0, status);
}

cudaError_t bounded_wait_selftest_launch(int32_t* status, cudaStream_t st) {
  bounded_wait_selftest_kernel<<<1, 1, 0, st>>>(status);
  return cudaGetLastError();
}

cudaError_t cursor_launch(int mode, int32_t* cursors, const int32_t* kept, int batch, int L, int32_t* status,
                          cudaStream_t st, const int32_t* slots, int n_state) {
  if (batch <= 0) return cudaSuccess;
  cursor_kernel<<<(batch + 127) / 128, 128, 0, st>>>(mode, cursors, kept, batch, L, status, slots, n_state);
  return cudaGetLastError();
}

cudaError_t reset_launch(int32_t* cursors, const int32_t* slots, int n_slots, int batch, int32_t* status,
                         cudaStream_t st) {
  if (n_slots <= 0) return cudaSuccess;
  reset_kernel<<<(n_slots + 127) / 128, 128, 0, st>>>(cursors, slots, n_slots, batch, status);
  return cudaGetLastError();
}

cudaError_t downcast_launch(const float* src, uint16_t* dst, size_t n, bool f16, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  size_t blocks = ((n >> 2) + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks == 0) blocks = 1;
  downcast_kernel<<<(unsigned)blocks, 256, 0, st>>>(src, dst, n, f16);
  return cudaGetLastError();
}

cudaError_t downcast_f8_launch(const float* src, uint8_t* dst, size_t rows, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  downcast_f8_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, st>>>(src, dst, rows);
  return cudaGetLastError();
}

}  // namespace rssm
