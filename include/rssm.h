/*
 * rssm.h -- C ABI of librssm, ReplaySSM decode kernels for GB300 (sm_103a).
 *
 * ReplaySSM keeps each sequence's SSM state as a high-precision checkpoint
 * plus a ring buffer of the last L input records ("ReplaySSM Caches Inputs
 * Instead of State to Speed Up Hybrid-Model Decoding", section "How ReplaySSM
 * works"). A non-flush step appends the current record and computes the
 * output from the read-only checkpoint and the window, storing no state; the
 * L-th step folds the window into the checkpoint and writes it once.
 * Speculative decoding appends draft records and rolls rejected ones back by
 * moving a cursor ("ReplaySSM", code repository, introduction: "Cheap
 * rollback").
 *
 * Conventions shared by every call:
 *  - All tensor arguments are DEVICE pointers to memory the caller owns.
 *    Tensors are dense, row-major (C order) with the shapes given below, and
 *    every base pointer must be 16-byte aligned (RSSM_ERR_MISALIGNED).
 *  - bf16 tensors hold IEEE bfloat16 bit patterns (rssm_bf16).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream). The library allocates no memory and never
 *    synchronises.
 *  - Host-side checks run first; on failure the call returns a negative
 *    RSSM_ERR_* code and launches nothing. RSSM_ERR_CUDA reports a launch
 *    error (cudaGetLastError after the launch).
 *  - Errors that depend on device data (a cursor out of range, a commit of
 *    more drafts than are pending) are written to the optional device word
 *    `dev_status` (int32, caller-zeroed; the first error code wins). The
 *    affected sequence is skipped: its checkpoint, ring and cursor are left
 *    as they were and its outputs are not written. Pass NULL to ignore them.
 *  - batch == 0 is a valid empty call: nothing is launched.
 *  - State slots (the descriptors' state_slots): by default batch row b of a
 *    call's records and outputs uses state row b (checkpoint, read copy, ring
 *    and cursor). Given state_slots [batch] int32, row b uses state row
 *    state_slots[b] of state arrays holding n_slots rows, so a serving engine
 *    keeps its states in fixed slots and gathers no state. A slot of -1 marks
 *    a padding row: it is skipped (its outputs are not written, no state is
 *    touched). Any other slot outside [0, n_slots) is reported as
 *    RSSM_DEV_BAD_SLOT and its row skipped. Two rows of one call must not
 *    name the same slot (their state updates would race). State slots are
 *    honoured by the decode calls on the shape-specialised kernels -- the
 *    Mamba-2 step and spec_verify (dstate 128, headdim a multiple of 64, a
 *    power-of-two nheads / ngroups), the Gated DeltaNet step and spec_verify
 *    and the KDA step and spec_verify (dk = dv = 128) -- and by
 *    rssm_commit_cursors_slots;
 *    elsewhere a non-NULL state_slots returns RSSM_ERR_UNSUPPORTED. Calls on whole state arrays (flush, prime,
 *    downcast, conventional steps) take state_slots = NULL with batch = the
 *    number of state rows.
 *
 * Cursor: int32 [batch, 4] = {start, count, pending, flags} per sequence.
 *  start   ring slot of the oldest record since the checkpoint, [0, L)
 *  count   committed records in the window, [0, L]
 *  pending draft records appended by the last verify, not yet committed
 *  flags   bit 0: that verify folded the committed window into the checkpoint
 * Record j of the window (j = 0 oldest) lives in ring slot (start + j) mod L.
 */
#ifndef RSSM_H
#define RSSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define RSSM_API __attribute__((visibility("default")))
#else
#define RSSM_API
#endif

typedef struct CUstream_st* rssm_stream_t; /* identical to cudaStream_t */
typedef uint16_t rssm_bf16;                /* bfloat16 bit pattern */

/* Return codes of every call. */
enum {
  RSSM_OK = 0,
  RSSM_ERR_INVALID_ARG = -1, /* null pointer, bad dimension, bad n_new */
  RSSM_ERR_UNSUPPORTED = -2, /* valid but outside the library's limits */
  RSSM_ERR_MISALIGNED = -3,  /* a base pointer is not 16-byte aligned */
  RSSM_ERR_CUDA = -4         /* a CUDA launch failed */
};

/* Codes written to dev_status. */
enum {
  RSSM_DEV_OK = 0,
  RSSM_DEV_BAD_CURSOR = 1,  /* start or count out of range */
  RSSM_DEV_WINDOW_FULL = 2, /* AR step on a window holding L records */
  RSSM_DEV_PENDING = 3,     /* step, verify or flush before the last verify was committed */
  RSSM_DEV_BAD_KEPT = 4,    /* commit with kept < 0 or kept > pending */
  RSSM_DEV_BAD_SLOT = 5,    /* a state slot outside its range (reset: [0, batch);
                             * state_slots: -1 or [0, n_slots)) */
  RSSM_DEV_TIMEOUT = 6      /* a bounded wait for an asynchronous copy expired */
};

/* Element types: of outputs (RSSM_F32, RSSM_BF16) and of the checkpoint's
 * read copy (RSSM_BF16, RSSM_F16, RSSM_FP8_E4M3). */
enum { RSSM_F32 = 0, RSSM_BF16 = 1, RSSM_F16 = 2, RSSM_FP8_E4M3 = 3 };

/* Limits of the library. */
#define RSSM_MAX_BUF_LEN 32 /* L in [1, 32] */
#define RSSM_MAX_BATCH 65535 /* Mamba-2 batch (RSSM_ERR_UNSUPPORTED above) */
#define RSSM_MAX_DIM 256    /* headdim, dstate, dk, dv: multiples of 8 in [8, 256] */

/* ----------------------------------------------------------------------------
 * Mamba-2
 *
 * Recurrence per (sequence b, head h), group g = floor(h * ngroups / nheads),
 * state h[headdim, dstate] (the published selective_state_update decode step;
 * the pages name the Mamba-2 layer in "Why SSM layers slow down hybrid models"):
 *   dA = exp(dt * A[h]);  h = dA * h + dt * x B^T;  y = (h C + D[h] x) * silu(z)
 * A record is (x, z [headdim] bf16; B, C [dstate] bf16 per group; dt fp32 > 0).
 */
typedef struct {
  int batch, nheads, headdim, dstate, ngroups;
  int buf_len;   /* L, the window length */
  int out_dtype; /* RSSM_F32 or RSSM_BF16: element type of y */
  int read_dtype; /* element type of the read copy ckpt_read, when one is
                   * passed: RSSM_BF16 (0 reads as RSSM_BF16), RSSM_F16, or
                   * RSSM_FP8_E4M3 -- then ckpt_read holds S * nheads *
                   * headdim * dstate e4m3 bytes (S state rows: batch, or
                   * n_slots) followed by one fp32 scale per state row
                   * ([S, nheads, headdim]); a value reads
                   * as e4m3 * scale, scale = max|row| / 448. FP8 needs
                   * dstate 128, headdim a multiple of 64, buf_len <= 31 and
                   * a power-of-two nheads / ngroups (else
                   * RSSM_ERR_UNSUPPORTED). */
  const int32_t* state_slots; /* [batch] state row of each batch row (-1:
                               * padding), or NULL: row b uses state row b */
  int n_slots;                /* state rows when state_slots is given: the
                               * leading dimension of ckpt, ckpt_read, the
                               * ring and the cursors (else batch) */
} rssm_mamba2_desc;

/* Ring buffer of window records, head- (or group-) major so that one
 * (sequence, head) tile's history is contiguous. Each step stores the whole
 * record of its token. */
typedef struct {
  rssm_bf16* x;  /* [batch, nheads, buf_len, headdim] */
  rssm_bf16* z;  /* [batch, nheads, buf_len, headdim] */
  rssm_bf16* B;  /* [batch, ngroups, buf_len, dstate] */
  rssm_bf16* C;  /* [batch, ngroups, buf_len, dstate] */
  float* dt;     /* [batch, nheads, Lp], Lp = buf_len rounded up to a
                    multiple of 4 (slots >= buf_len unused) */
} rssm_mamba2_ring;

/* Bytes of each ring field, in the order x, z, B, C, dt. Returns RSSM_OK or
 * RSSM_ERR_INVALID_ARG. */
RSSM_API int rssm_mamba2_ring_bytes(const rssm_mamba2_desc* desc, size_t bytes[5]);

/* Conventional decode step (the comparison point): reads and writes the full
 * state every step ("Why SSM layers slow down hybrid models", first cause).
 *  state [batch, nheads, headdim, dstate] fp32, updated in place
 *  x, z [batch, nheads, headdim]; B, C [batch, ngroups, dstate] (bf16)
 *  dt [batch, nheads] fp32; A, D [nheads] fp32
 *  y [batch, nheads, headdim] of desc->out_dtype (written) */
RSSM_API int rssm_mamba2_conventional_step(const rssm_mamba2_desc* desc, float* state,
                                  const rssm_bf16* x, const rssm_bf16* z,
                                  const rssm_bf16* B, const rssm_bf16* C,
                                  const float* dt, const float* A,
                                  const float* D, void* y,
                                  rssm_stream_t stream);

/* One ReplaySSM AR decode step ("How ReplaySSM works"). For each sequence
 * with window count c (needs c < L and pending == 0):
 *  - c + 1 < L (non-flush): stores the record in ring slot (start + c) mod L
 *    and computes y from the checkpoint and the c + 1 window records without
 *    writing any state; count becomes c + 1.
 *  - c + 1 == L (flush): folds the L records into the checkpoint, writes it
 *    (and ckpt_read, if given) once, computes y; count becomes 0.
 *  ckpt      [batch, nheads, headdim, dstate] fp32 recurrence checkpoint
 *  ckpt_read same shape in desc->read_dtype (bf16 or fp16), or NULL. When given, non-flush steps read
 *            it instead of ckpt (the low-precision read copy of "ReplaySSM",
 *            introduction, "Separate state precisions"); flushes read ckpt
 *            and write both.
 *  ring      window records (see rssm_mamba2_ring), cursors [batch, 4]
 *  x .. D, y as in rssm_mamba2_conventional_step.
 * The cursors advance within the call, in stream order (count + 1, or 0 on
 * the flushing step); while a call runs, the high 16 bits of a cursor's flags
 * word are in use. */
RSSM_API int rssm_mamba2_step(const rssm_mamba2_desc* desc, float* ckpt,
                     rssm_bf16* ckpt_read, const rssm_mamba2_ring* ring,
                     int32_t* cursors, const rssm_bf16* x, const rssm_bf16* z,
                     const rssm_bf16* B, const rssm_bf16* C, const float* dt,
                     const float* A, const float* D, void* y,
                     int32_t* dev_status, rssm_stream_t stream);

/* Standalone flush: for every sequence with count > 0 and pending == 0,
 * folds its window into ckpt (and ckpt_read, if given); start moves past the
 * folded records and count becomes 0. Produces no output. */
RSSM_API int rssm_mamba2_flush(const rssm_mamba2_desc* desc, float* ckpt,
                      rssm_bf16* ckpt_read, const rssm_mamba2_ring* ring,
                      int32_t* cursors, const float* A, int32_t* dev_status,
                      rssm_stream_t stream);

/* Speculative verify ("How ReplaySSM works": drafts are appended to the
 * buffer instead of snapshotting state; "Core implementation files":
 * speculative decode on a circular buffer). Appends n_new = K records per
 * sequence (the bonus token and K-1 drafts) at ring slots
 * (start + count + i) mod L and computes, output-only, y_i for i < K: the
 * output after committed records plus new records 0..i. If count + K > L the
 * committed window is first folded into the checkpoint (written once).
 * Needs pending == 0; sets pending = K and flags = folded. Must be followed
 * by one rssm_commit_cursors.
 *  x, z [batch, K, nheads, headdim]; B, C [batch, K, ngroups, dstate] (bf16)
 *  dt [batch, K, nheads] fp32; y [batch, K, nheads, headdim]
 *  1 <= n_new <= buf_len (else RSSM_ERR_INVALID_ARG). */
RSSM_API int rssm_mamba2_spec_verify(const rssm_mamba2_desc* desc, int n_new,
                            float* ckpt, rssm_bf16* ckpt_read,
                            const rssm_mamba2_ring* ring, int32_t* cursors,
                            const rssm_bf16* x, const rssm_bf16* z,
                            const rssm_bf16* B, const rssm_bf16* C,
                            const float* dt, const float* A, const float* D,
                            void* y, int32_t* dev_status,
                            rssm_stream_t stream);

/* Emulated read precision ("ReplaySSM", code repository, introduction: the
 * emulation kernels implement separate read and recurrence precision and
 * expose their quantization behavior). Nothing low-precision is stored: a
 * non-flush step reads each checkpoint element through a quantise-dequantise
 * in the chosen format, computed in fp32 registers, while a flushing step
 * reads and folds the exact fp32 checkpoint. Formats saturate at their
 * largest finite value; rounding is to nearest, ties to even:
 *   RSSM_EMU_BF16, RSSM_EMU_F16   8 / 11 significant bits (IEEE exponent
 *                                 ranges), no scale;
 *   RSSM_EMU_E4M3, RSSM_EMU_E5M2  OCP FP8 (4 / 3 significant bits, largest
 *                                 448 / 57344, subnormals), with a scale;
 *   RSSM_EMU_INT8                 symmetric 8-bit integers in [-127, 127],
 *                                 with a scale.
 * A scale s = max|group| / qmax (qmax = 448, 57344 or 127) covers one state
 * row of dstate values (RSSM_EMU_SCALE_ROW) or one 64-row block of a
 * (sequence, head) tile (RSSM_EMU_SCALE_TILE64); an element x reads as
 * Q(x * (qmax / max|group|)) * s, both quotients and both products in fp32. */
enum { RSSM_EMU_BF16 = 1, RSSM_EMU_F16 = 2, RSSM_EMU_E4M3 = 3, RSSM_EMU_E5M2 = 4, RSSM_EMU_INT8 = 5 };
enum { RSSM_EMU_SCALE_NONE = 0, RSSM_EMU_SCALE_ROW = 1, RSSM_EMU_SCALE_TILE64 = 2 };
typedef struct {
  int format; /* RSSM_EMU_* */
  int scale;  /* RSSM_EMU_SCALE_NONE for bf16 / fp16; ROW or TILE64 for e4m3, e5m2, int8 */
} rssm_emulation;

/* Bytes of device workspace rssm_mamba2_step_emulated needs for desc: one
 * pair of fp32 partial sums per block of the launch (desc->batch * nheads *
 * headdim / 64 pairs of 8 bytes). 0 with RSSM_ERR_INVALID_ARG or _UNSUPPORTED in *rc
 * (if rc is non-NULL) for a descriptor the call rejects. */
RSSM_API size_t rssm_mamba2_emulated_workspace_bytes(const rssm_mamba2_desc* desc, int* rc);

/* rssm_mamba2_step with an emulated read precision (see rssm_emulation):
 * the same protocol (append, output-only non-flush steps, the fused flush
 * on the L-th step from the exact checkpoint, cursors advanced within the
 * call), and the quantisation behaviour of what the call read:
 *  err        [2] double, device, written: the sum over every element that a
 *             non-flush step of this call read of (read value - fp32 value)^2,
 *             and of (fp32 value)^2 -- so sqrt(err[0] / err[1]) is the
 *             relative L2 error of the emulated read. Summed in a fixed order
 *             (fp32 within each block's 8192 elements, then fp64): the same
 *             inputs give the same bits.
 *  workspace  device scratch of at least
 *             rssm_mamba2_emulated_workspace_bytes(desc) bytes (else
 *             RSSM_ERR_INVALID_ARG), 16-byte aligned, owned by the caller;
 *             its contents need no initialisation and are overwritten.
 * Needs the shape-specialised kernel's shapes (dstate 128, headdim a
 * multiple of 64, buf_len <= 31, a power-of-two nheads / ngroups) and no
 * state slots (else RSSM_ERR_UNSUPPORTED); desc->read_dtype is ignored.
 * A format / scale pair other than those listed: RSSM_ERR_INVALID_ARG. */
RSSM_API int rssm_mamba2_step_emulated(const rssm_mamba2_desc* desc, const rssm_emulation* emu, float* ckpt,
                                       const rssm_mamba2_ring* ring, int32_t* cursors, const rssm_bf16* x,
                                       const rssm_bf16* z, const rssm_bf16* B, const rssm_bf16* C,
                                       const float* dt, const float* A, const float* D, void* y, double* err,
                                       void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                       rssm_stream_t stream);

/* rssm_mamba2_step_emulated for callers that cannot allocate device memory
 * when they decode. The pages have no counterpart of this call. Some hosts
 * reserve nearly all of the GPU's memory for their own pools before decoding
 * starts, or hand a kernel library a stream but no allocator, and cudaMalloc
 * itself may synchronise the device in the middle of a decode loop. This
 * variant takes no workspace: its per-block error sums go to a static device
 * array inside librssm of RSSM_NOALLOC_MAX_WARPS / 4 (error, norm) fp32
 * pairs -- 512 KiB on every GPU that loads the library, held until the
 * process exits -- and it never calls cudaMalloc, cudaFree or any routine
 * that allocates.
 *  - Arguments, protocol, limits and results are those of
 *    rssm_mamba2_step_emulated, without workspace and workspace_bytes.
 *  - A launch of more than RSSM_NOALLOC_MAX_WARPS warps (batch * nheads *
 *    headdim / 16; the serving layer of batch 256, 128 heads of 64 rows has
 *    131072) returns RSSM_ERR_UNSUPPORTED and launches nothing.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and keeps it; make that
 *    first call before any stream capture. Devices 0..RSSM_NOALLOC_MAX_DEVICES-1.
 *  - Every call on a device uses the same array, which keeps the last call's
 *    sums. Nothing in it needs clearing (each call writes every entry it reads
 *    before reading it), but two calls whose kernels overlap on the GPU --
 *    on different streams without an ordering between them -- race on it:
 *    order them (one stream, or events). */
#define RSSM_NOALLOC_MAX_WARPS 262144
#define RSSM_NOALLOC_MAX_DEVICES 64
RSSM_API int rssm_mamba2_step_emulated_noalloc(const rssm_mamba2_desc* desc, const rssm_emulation* emu, float* ckpt,
                                               const rssm_mamba2_ring* ring, int32_t* cursors, const rssm_bf16* x,
                                               const rssm_bf16* z, const rssm_bf16* B, const rssm_bf16* C,
                                               const float* dt, const float* A, const float* D, void* y,
                                               double* err, int32_t* dev_status, rssm_stream_t stream);

/* ----------------------------------------------------------------------------
 * Cursors (shared by Mamba-2, Gated DeltaNet and KDA)
 */

/* Commit after a verify ("ReplaySSM", introduction, "Cheap rollback";
 * "Core implementation files": the commit call of the speculative path).
 * kept [batch] int32: records of the last verify to keep, 0 <= kept <=
 * pending. If that verify folded: start += count (mod L), count = 0. Then
 * count += kept, pending = 0, flags = 0. Rejected drafts are dropped by this
 * cursor move alone. */
RSSM_API int rssm_commit_cursors(int32_t* cursors, const int32_t* kept, int batch,
                        int buf_len, int32_t* dev_status,
                        rssm_stream_t stream);

/* rssm_commit_cursors for a call made with state slots: kept [batch] is per
 * batch row and applies to cursor state_slots[b] of n_slots; rows whose slot is
 * -1 are skipped, other slots outside [0, n_slots) reported as
 * RSSM_DEV_BAD_SLOT. */
RSSM_API int rssm_commit_cursors_slots(int32_t* cursors, const int32_t* kept, const int32_t* state_slots,
                              int batch, int n_slots, int buf_len, int32_t* dev_status,
                              rssm_stream_t stream);

/* Reset the cursors of the listed sequences to {0, 0, 0, 0} (a new request in
 * that slot; "Core implementation files": the reset call). slots [n_slots]
 * int32 in [0, batch). The checkpoint is not touched: the caller writes it,
 * then calls rssm_checkpoint_downcast if it keeps a read copy. */
RSSM_API int rssm_reset_cursors(int32_t* cursors, const int32_t* slots, int n_slots,
                       int batch, int32_t* dev_status, rssm_stream_t stream);

/* fp32 -> low-precision read copy, round to nearest even ("ReplaySSM",
 * introduction, "Separate state precisions"). src [n] fp32, dst [n] of dtype
 * RSSM_BF16 or RSSM_F16 (16-bit elements; fp16 saturates to +-inf above its
 * range). Any other dtype: RSSM_ERR_INVALID_ARG. */
RSSM_API int rssm_checkpoint_downcast(const float* src, rssm_bf16* dst, size_t n, int dtype,
                             rssm_stream_t stream);

/* The read copy of a whole Mamba-2 checkpoint in desc->read_dtype ("ReplaySSM",
 * introduction, "Separate state precisions"), for a checkpoint written by the
 * caller (a new request, a reset slot): ckpt [batch, nheads, headdim, dstate]
 * fp32; ckpt_read laid out as rssm_mamba2_desc.read_dtype says. Round to
 * nearest even; fp8 rows are scaled by their own max|row| / 448. */
RSSM_API int rssm_mamba2_downcast(const rssm_mamba2_desc* desc, const float* ckpt, void* ckpt_read,
                         rssm_stream_t stream);

/* ----------------------------------------------------------------------------
 * Gated DeltaNet
 *
 * Recurrence per (sequence, head), state S[dv, dk], alpha = exp(g) (the
 * published gated delta rule; Gated DeltaNet is named in "Why SSM layers slow
 * down hybrid models"):
 *   S = alpha * S (I - beta k k^T) + beta v k^T;   o = S q
 * A record is (q, k [dk] bf16; v [dv] bf16; g, beta fp32).
 */
typedef struct {
  int batch, nheads, dk, dv;
  int buf_len;
  int out_dtype; /* element type of o */
  const int32_t* state_slots; /* as in rssm_mamba2_desc */
  int n_slots;
} rssm_gdn_desc;

typedef struct {
  rssm_bf16* q;  /* [batch, nheads, buf_len, dk] */
  rssm_bf16* k;  /* [batch, nheads, buf_len, dk] */
  rssm_bf16* v;  /* [batch, nheads, buf_len, dv] */
  float* g;      /* [batch, nheads, Lp], Lp as in rssm_mamba2_ring.dt */
  float* beta;   /* [batch, nheads, Lp] */
  float* e;      /* [batch, nheads, buf_len, dv]: each window record's
                  * correction e_t = beta_t (v_t - alpha_t S_{t-1} k_t), kept
                  * next to the record (see rssm_gdn_step) */
} rssm_gdn_ring;

/* Bytes of each ring field, in the order q, k, v, g, beta, e. */
RSSM_API int rssm_gdn_ring_bytes(const rssm_gdn_desc* desc, size_t bytes[6]);

/* Conventional step: S [batch, nheads, dv, dk] fp32 updated in place;
 * q, k [batch, nheads, dk], v [batch, nheads, dv] bf16; g, beta
 * [batch, nheads] fp32; o [batch, nheads, dv] of desc->out_dtype. */
RSSM_API int rssm_gdn_conventional_step(const rssm_gdn_desc* desc, float* S,
                               const rssm_bf16* q, const rssm_bf16* k,
                               const rssm_bf16* v, const float* g,
                               const float* beta, void* o,
                               rssm_stream_t stream);

/* ReplaySSM AR step for Gated DeltaNet: same protocol as rssm_mamba2_step
 * (non-flush steps write no state; the L-th step folds and writes S once).
 * A record's correction e_t depends only on the checkpoint and the records
 * before it, so it is fixed from the step that appends the record until the
 * flush that folds it: the step computes e for the current record only,
 * reads the window's e from ring->e and appends the new one there. The
 * checkpoint is still never written outside a flush. */
RSSM_API int rssm_gdn_step(const rssm_gdn_desc* desc, float* S, const rssm_gdn_ring* ring,
                  int32_t* cursors, const rssm_bf16* q, const rssm_bf16* k,
                  const rssm_bf16* v, const float* g, const float* beta,
                  void* o, int32_t* dev_status, rssm_stream_t stream);

/* Standalone flush for Gated DeltaNet (as rssm_mamba2_flush). */
RSSM_API int rssm_gdn_flush(const rssm_gdn_desc* desc, float* S, const rssm_gdn_ring* ring,
                   int32_t* cursors, int32_t* dev_status, rssm_stream_t stream);

/* Speculative verify for Gated DeltaNet (as rssm_mamba2_spec_verify: "How
 * ReplaySSM works", drafts appended to the buffer; "ReplaySSM" repository,
 * introduction, output-only verification and rollback by moving a pointer).
 * Appends n_new = K records per sequence at ring slots (start + count + i)
 * mod L, with their corrections e, and computes, output-only, o_i for i < K:
 * the output after the committed records plus new records 0..i. If count + K
 * > L the committed window is first folded into S (written once). Needs
 * pending == 0; sets pending = K and flags = folded. Must be followed by one
 * rssm_commit_cursors.
 *  q, k [batch, K, nheads, dk]; v [batch, K, nheads, dv] (bf16);
 *  g, beta [batch, K, nheads] fp32; o [batch, K, nheads, dv] of out_dtype.
 *  1 <= n_new <= buf_len (else RSSM_ERR_INVALID_ARG). */
RSSM_API int rssm_gdn_spec_verify(const rssm_gdn_desc* desc, int n_new, float* S,
                         const rssm_gdn_ring* ring, int32_t* cursors,
                         const rssm_bf16* q, const rssm_bf16* k, const rssm_bf16* v,
                         const float* g, const float* beta, void* o,
                         int32_t* dev_status, rssm_stream_t stream);

/* Fills ring->e for the records already in each sequence's window (count of
 * them, from its checkpoint S), for windows whose records were written into
 * the ring directly rather than appended by rssm_gdn_step. The pages have no
 * counterpart (their windows are only filled by decode steps). Writes ring->e
 * only; sequences with count == 0 or pending != 0 are skipped. */
RSSM_API int rssm_gdn_prime(const rssm_gdn_desc* desc, const float* S, const rssm_gdn_ring* ring,
                   const int32_t* cursors, int32_t* dev_status, rssm_stream_t stream);

/* ----------------------------------------------------------------------------
 * Kimi Delta Attention (KDA)
 *
 * The gated delta rule with a decay per key channel (the pages name KDA as an
 * SSM layer in "Why SSM layers slow down hybrid models" and report ReplaySSM
 * added to a KDA decode kernel in the "ReplaySSM" repository page, section
 * "Adoption"; the recurrence is the published KDA one). Per (sequence, head),
 * state S[dv, dk], alpha = exp(g) with g [dk] (g <= 0):
 *   S = S Diag(alpha) (I - beta k k^T) + beta v k^T;   o = S q
 * A record is (q, k [dk] bf16; v [dv] bf16; g [dk] fp32; beta fp32). The
 * descriptor is the Gated DeltaNet one (state slots included).
 * The replay calls (step, flush, prime) need dk = dv = 128 (else
 * RSSM_ERR_UNSUPPORTED); the step also needs buf_len <= 31.
 */
typedef rssm_gdn_desc rssm_kda_desc;

typedef struct {
  rssm_bf16* q;  /* [batch, nheads, buf_len, dk] */
  rssm_bf16* k;  /* [batch, nheads, buf_len, dk] */
  rssm_bf16* v;  /* [batch, nheads, buf_len, dv] */
  float* g;      /* [batch, nheads, buf_len, dk]: each record's log decay per channel */
  float* beta;   /* [batch, nheads, Lp], Lp as in rssm_mamba2_ring.dt */
  float* e;      /* [batch, nheads, buf_len, dv]: each window record's correction
                  * e_t = beta_t (v_t - S_{t-1} (alpha_t * k_t)) (see rssm_kda_step) */
} rssm_kda_ring;

/* Bytes of each ring field, in the order q, k, v, g, beta, e. */
RSSM_API int rssm_kda_ring_bytes(const rssm_kda_desc* desc, size_t bytes[6]);

/* Conventional step: S [batch, nheads, dv, dk] fp32 updated in place;
 * q, k [batch, nheads, dk], v [batch, nheads, dv] bf16; g [batch, nheads, dk]
 * and beta [batch, nheads] fp32; o [batch, nheads, dv] of desc->out_dtype.
 * Any dk, dv the descriptor allows. */
RSSM_API int rssm_kda_conventional_step(const rssm_kda_desc* desc, float* S,
                               const rssm_bf16* q, const rssm_bf16* k,
                               const rssm_bf16* v, const float* g,
                               const float* beta, void* o,
                               rssm_stream_t stream);

/* ReplaySSM AR step for KDA: the protocol of rssm_gdn_step (non-flush steps
 * write no state; the L-th step folds the window and writes S once; the
 * cursors advance within the call). With G the per-channel sum of the log
 * decays from a window record to the current one, a window record's key
 * enters as k * exp(G) (channel-wise); its correction e_t is fixed from the
 * step that appends it until the flush that folds it, so the step reads the
 * window's e from ring->e and appends the current record's.
 * Records as in rssm_kda_conventional_step. */
RSSM_API int rssm_kda_step(const rssm_kda_desc* desc, float* S, const rssm_kda_ring* ring,
                  int32_t* cursors, const rssm_bf16* q, const rssm_bf16* k,
                  const rssm_bf16* v, const float* g, const float* beta,
                  void* o, int32_t* dev_status, rssm_stream_t stream);

/* Standalone flush for KDA (as rssm_gdn_flush); folds each window with the
 * corrections kept in ring->e. */
RSSM_API int rssm_kda_flush(const rssm_kda_desc* desc, float* S, const rssm_kda_ring* ring,
                   int32_t* cursors, int32_t* dev_status, rssm_stream_t stream);

/* Speculative verify for KDA (as rssm_gdn_spec_verify: K = n_new records
 * appended at ring slots (start + count + i) mod L with their corrections,
 * outputs o_i after the committed records plus new records 0..i, the
 * committed window folded into S first if count + K > L; pending = K, flags =
 * folded; followed by one rssm_commit_cursors).
 *  q, k [batch, K, nheads, dk], v [batch, K, nheads, dv] (bf16);
 *  g [batch, K, nheads, dk], beta [batch, K, nheads] fp32;
 *  o [batch, K, nheads, dv] of out_dtype.
 *  1 <= n_new <= buf_len (else RSSM_ERR_INVALID_ARG); dk = dv = 128, n_new <= 4
 *  and buf_len + n_new <= 32 (else RSSM_ERR_UNSUPPORTED). State slots are
 *  honoured (records and outputs by batch row, state rows by slot). */
RSSM_API int rssm_kda_spec_verify(const rssm_kda_desc* desc, int n_new, float* S, const rssm_kda_ring* ring,
                         int32_t* cursors, const rssm_bf16* q, const rssm_bf16* k, const rssm_bf16* v,
                         const float* g, const float* beta, void* o, int32_t* dev_status,
                         rssm_stream_t stream);

/* Fills ring->e for windows written into the ring directly (as
 * rssm_gdn_prime). Writes ring->e only. */
RSSM_API int rssm_kda_prime(const rssm_kda_desc* desc, const float* S, const rssm_kda_ring* ring,
                   const int32_t* cursors, int32_t* dev_status, rssm_stream_t stream);

/* ----------------------------------------------------------------------------
 * Misc
 */
RSSM_API const char* rssm_status_string(int code); /* text for RSSM_* and RSSM_DEV_* codes */
RSSM_API int rssm_version(void);                   /* major * 10000 + minor * 100 + patch */

/* Self-test of the kernels' bounded waits: launches one block that waits for
 * a copy nothing delivers. The wait gives up after its limit (about one
 * second; the block waits once more, bounded, before it leaves) and writes
 * RSSM_DEV_TIMEOUT to dev_status (non-NULL, 16-byte aligned, caller-zeroed).
 * The context stays usable. Takes about two seconds of one block. */
RSSM_API int rssm_selftest_bounded_wait(int32_t* dev_status, rssm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RSSM_H */
