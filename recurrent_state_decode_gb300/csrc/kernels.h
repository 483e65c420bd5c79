// Internal interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "rssm.h"

namespace rssm {

// Mamba-2 launch arguments (device pointers, dense row-major layouts of rssm.h).
struct M2Args {
  int Bt, H, P, N, G, L;
  int PB, nPB;  // rows per block, row blocks per (sequence, head) tile
  int K;        // records per verify (1 for the AR step)
  int hpg_log2;  // log2(H / G) when H / G is a power of two, else -1
  int read_f16;  // the read copy ckpt_read holds fp16 (else bf16)
  int read_f8;   // the read copy holds e4m3 values, then one fp32 scale per state row
  float* ckpt;
  uint16_t* ckpt_read;
  uint16_t *rx, *rz, *rB, *rC;
  float* rdt;
  int32_t* cursors;
  const uint16_t *x, *z, *B, *C;
  const float *dt, *A, *D;
  void* y;
  int32_t* status;
  const int32_t* slots;  // [Bt] state row of each batch row (-1: padding), or null: row b uses state row b
  int Sn;                // state rows (the leading dimension of ckpt, ckpt_read, the ring and the cursors)
  int emu_fmt, emu_scale;  // emulated read precision (RSSM_EMU_*; 0: none)
  float2* emu_part;        // [blocks] per-block (sum of squared read errors, sum of squares)
};

enum { M2_CONVENTIONAL = 0, M2_STEP = 1, M2_FLUSH = 2, M2_VERIFY = 3 };

cudaError_t m2_launch(int kind, const M2Args& a, int out_bf16, cudaStream_t st);
// The persistent, warp-specialised AR step (mamba2_step.cu).
cudaError_t m2_step_launch(const M2Args& a, int out_bf16, cudaStream_t st);
// Shape-specialised AR step (dstate 128, headdim a multiple of 64; mamba2_step_fast.cu).
bool m2_step_fast_applies(const M2Args& a);
cudaError_t m2_step_fast_launch(const M2Args& a, int out_bf16, cudaStream_t st);
// The same kernel with an emulated read precision (a.emu_fmt, a.emu_scale), writing per-block error
// sums to a.emu_part, then their fixed-order reduction into err[2].
cudaError_t m2_step_emulated_launch(const M2Args& a, int out_bf16, double* err, cudaStream_t st);
// Entries of a.emu_part an emulated step of these arguments writes.
inline size_t m2_emulated_partials(const M2Args& a) { return (size_t)a.Bt * a.H * a.nPB; }
// The same step with its error sums in the library's static device array (mamba2_step_fast.cu), which holds
// M2_NOALLOC_PARTIALS pairs: a.emu_part is ignored; a larger launch returns cudaErrorInvalidValue.
constexpr int M2_NOALLOC_PARTIALS = RSSM_NOALLOC_MAX_WARPS / 4;  // one pair per block of four warps
cudaError_t m2_step_emulated_noalloc_launch(M2Args a, int out_bf16, double* err, cudaStream_t st);
// The persistent speculative verify (mamba2_verify.cu); its epilogue kernel is in mamba2.cu.
cudaError_t m2_verify_launch(const M2Args& a, int out_bf16, cudaStream_t st);
// Shape-specialised verify (dstate 128, headdim a multiple of 64, K <= 4; mamba2_verify_fast.cu).
bool m2_verify_fast_applies(const M2Args& a);
cudaError_t m2_verify_fast_launch(const M2Args& a, int out_bf16, cudaStream_t st);
size_t m2_smem_bytes(int kind, const M2Args& a);

// Gated DeltaNet launch arguments.
struct GdnArgs {
  int Bt, H, DK, DV, L;
  float* S;
  uint16_t *rq, *rk, *rv;
  float *rg, *rbeta;
  float* re;  // cached corrections e_t [Bt, H, L, DV]
  int K;      // records per verify (1 for the AR step)
  int32_t* cursors;
  const uint16_t *q, *k, *v;
  const float *g, *beta;
  void* o;
  int32_t* status;
  const int32_t* slots;  // as in M2Args
  int Sn;
};

enum { GDN_CONVENTIONAL = 0, GDN_STEP = 1, GDN_FLUSH = 2, GDN_PRIME = 3 };

// Speculative verify for Gated DeltaNet (gdn_verify.cu): K new records per sequence.
cudaError_t gdn_verify_launch(const GdnArgs& a, int out_bf16, cudaStream_t st);
// Shape-specialised verify (dk = dv = 128, K <= 4, L + K <= 32; gdn_verify_fast.cu), epilogue included.
bool gdn_verify_fast_applies(const GdnArgs& a);
cudaError_t gdn_verify_fast_launch(const GdnArgs& a, int out_bf16, cudaStream_t st);

cudaError_t gdn_launch(int kind, const GdnArgs& a, int out_bf16, cudaStream_t st);
// Shape-specialised AR step (dk = dv = 128, L <= 31; gdn_step_fast.cu).
bool gdn_step_fast_applies(const GdnArgs& a);
cudaError_t gdn_step_fast_launch(const GdnArgs& a, int out_bf16, cudaStream_t st);

// One block whose bulk-copy wait expires (cursors.cu): the timeout path's self-test.
cudaError_t bounded_wait_selftest_launch(int32_t* status, cudaStream_t st);

// Kimi Delta Attention (kda.cu, kda_step_fast.cu) takes GdnArgs with g, rg
// holding one log decay per key channel: g [Bt, H, DK], rg [Bt, H, L, DK].
// GDN_CONVENTIONAL, GDN_STEP, GDN_FLUSH and GDN_PRIME name its kernels too.
cudaError_t kda_launch(int kind, const GdnArgs& a, int out_bf16, cudaStream_t st);
// The replay kernels' shapes: dk = dv = 128 (the step also L <= 31).
bool kda_window_applies(const GdnArgs& a);
bool kda_step_fast_applies(const GdnArgs& a);
// Speculative verify (kda_verify_fast.cu: dk = dv = 128, K <= 4, L + K <= 32, state slots honoured); the
// sequence's last block appends the shared fields and marks the cursor, so a verify is one kernel.
bool kda_verify_applies(const GdnArgs& a);
cudaError_t kda_verify_launch(const GdnArgs& a, int out_bf16, cudaStream_t st);
cudaError_t kda_step_fast_launch(const GdnArgs& a, int out_bf16, cudaStream_t st);

// Cursor kernels (one thread per sequence).
enum { CUR_AR = 0, CUR_FLUSH = 1, CUR_COMMIT = 2 };

// `slots` (or null): cursor of batch row b is slots[b] of n_state (-1 skipped).
cudaError_t cursor_launch(int mode, int32_t* cursors, const int32_t* kept, int batch, int L, int32_t* status,
                          cudaStream_t st, const int32_t* slots = nullptr, int n_state = 0);
cudaError_t reset_launch(int32_t* cursors, const int32_t* slots, int n_slots, int batch, int32_t* status,
                         cudaStream_t st);
cudaError_t downcast_launch(const float* src, uint16_t* dst, size_t n, bool f16, cudaStream_t st);
// fp8 read copy of `rows` rows of 128 fp32 values, with one scale per row after the bytes.
cudaError_t downcast_f8_launch(const float* src, uint8_t* dst, size_t rows, cudaStream_t st);

// Launch attributes of a kernel on the current device, set the first time a
// launch needs them rather than on every launch: the largest shared-memory
// carveout of the unified L1 (when max_carveout) and a dynamic shared-memory
// limit of at least dyn_smem bytes (when above the 48 KiB default). Later
// calls that need no more are a table lookup under a mutex.
cudaError_t prepare_kernel(const void* fn, size_t dyn_smem, bool max_carveout);
template <typename Kern>
inline cudaError_t prepare(Kern* k, size_t dyn_smem, bool max_carveout) {
  return prepare_kernel(reinterpret_cast<const void*>(k), dyn_smem, max_carveout);
}

// Row stride of the per-record scalar rings (dt; g, beta): L rounded up to a
// multiple of 4 slots, so that a row is a whole number of 16-byte units.
inline __host__ __device__ int pad4(int L) { return (L + 3) & ~3; }

// Rows per block of a Mamba-2 state tile of `rows` (headdim) x `cols` (dstate)
// fp32 elements: 64 rows when a row fits one float4 per lane (dstate <= 128),
// 32 rows otherwise, so a block is at most 32 KiB and a consumer warp holds its
// quarter of the rows in 64 registers.
inline int rows_per_block(int rows, int cols) {
  const int pb = cols <= 128 ? 64 : 32;
  return pb < rows ? pb : rows;
}

}  // namespace rssm
