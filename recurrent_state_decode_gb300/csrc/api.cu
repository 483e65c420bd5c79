// C ABI of librssm: host-side argument checks, then kernel launches on the
// caller's stream. Nothing here allocates, synchronises or reads device data.
#include <climits>
#include <cstdint>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "rssm.h"

using namespace rssm;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dim_ok(int v) { return v >= 8 && v <= RSSM_MAX_DIM && v % 8 == 0; }

// All pointers non-null and 16-byte aligned.
int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p) return RSSM_ERR_INVALID_ARG;
  for (const void* p : ps)
    if (!aligned16(p)) return RSSM_ERR_MISALIGNED;
  return RSSM_OK;
}

int check_opt(const void* p) { return (p && !aligned16(p)) ? RSSM_ERR_MISALIGNED : RSSM_OK; }

// A state-slot table needs 0 <= n_slots <= RSSM_MAX_BATCH.
int check_slots(const int32_t* slots, int n_slots) {
  if (!slots) return RSSM_OK;
  if (n_slots < 0) return RSSM_ERR_INVALID_ARG;
  return n_slots > RSSM_MAX_BATCH ? RSSM_ERR_UNSUPPORTED : RSSM_OK;
}

// State rows of the arrays a call addresses.
template <typename Desc>
size_t state_rows(const Desc* d) {
  return d->state_slots ? (size_t)d->n_slots : (size_t)d->batch;
}

int check_m2(const rssm_mamba2_desc* d) {
  if (!d) return RSSM_ERR_INVALID_ARG;
  if (d->batch < 0 || d->nheads < 1 || d->ngroups < 1 || d->nheads % d->ngroups != 0) return RSSM_ERR_INVALID_ARG;
  if (!dim_ok(d->headdim) || !dim_ok(d->dstate)) return RSSM_ERR_INVALID_ARG;
  if (d->buf_len < 1 || d->buf_len > RSSM_MAX_BUF_LEN) return RSSM_ERR_INVALID_ARG;
  if (d->out_dtype != RSSM_F32 && d->out_dtype != RSSM_BF16) return RSSM_ERR_INVALID_ARG;
  if (d->read_dtype != 0 && d->read_dtype != RSSM_BF16 && d->read_dtype != RSSM_F16 && d->read_dtype != RSSM_FP8_E4M3)
    return RSSM_ERR_INVALID_ARG;
  const int pb = rows_per_block(d->headdim, d->dstate);
  const long long grid = (long long)d->batch * d->nheads * ((d->headdim + pb - 1) / pb);
  if (grid > INT_MAX || d->batch > RSSM_MAX_BATCH) return RSSM_ERR_UNSUPPORTED;
  if (int rc = check_slots(d->state_slots, d->n_slots)) return rc;
  if (d->read_dtype == RSSM_FP8_E4M3) {  // the fp8 read copy lives on the shape-specialised kernels only
    const int hpg = d->nheads / d->ngroups;
    if (d->dstate != 128 || d->headdim % 64 != 0 || d->buf_len > 31 || (hpg & (hpg - 1)) != 0 ||
        (long long)d->nheads * (d->headdim / 64) >= (1 << 15))
      return RSSM_ERR_UNSUPPORTED;
  }
  return RSSM_OK;
}

int check_gdn(const rssm_gdn_desc* d) {
  if (!d) return RSSM_ERR_INVALID_ARG;
  if (d->batch < 0 || d->nheads < 1) return RSSM_ERR_INVALID_ARG;
  if (!dim_ok(d->dk) || !dim_ok(d->dv)) return RSSM_ERR_INVALID_ARG;
  if (d->buf_len < 1 || d->buf_len > RSSM_MAX_BUF_LEN) return RSSM_ERR_INVALID_ARG;
  if (d->out_dtype != RSSM_F32 && d->out_dtype != RSSM_BF16) return RSSM_ERR_INVALID_ARG;
  const long long grid = (long long)d->batch * d->nheads * ((d->dv + 63) / 64);
  if (grid > INT_MAX) return RSSM_ERR_UNSUPPORTED;
  return check_slots(d->state_slots, d->n_slots);
}

M2Args m2_args(const rssm_mamba2_desc* d) {
  M2Args a{};
  a.Bt = d->batch;
  a.H = d->nheads;
  a.P = d->headdim;
  a.N = d->dstate;
  a.G = d->ngroups;
  a.L = d->buf_len;
  a.PB = rows_per_block(a.P, a.N);
  a.nPB = (a.P + a.PB - 1) / a.PB;
  a.K = 1;
  a.read_f16 = d->read_dtype == RSSM_F16;
  a.read_f8 = d->read_dtype == RSSM_FP8_E4M3;
  const int hpg = a.H / a.G;
  a.hpg_log2 = (hpg & (hpg - 1)) == 0 ? __builtin_ctz(hpg) : -1;
  a.slots = d->state_slots;
  a.Sn = (int)state_rows(d);
  return a;
}

void set_ring(M2Args& a, const rssm_mamba2_ring* r) {
  a.rx = r->x;
  a.rz = r->z;
  a.rB = r->B;
  a.rC = r->C;
  a.rdt = r->dt;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? RSSM_OK : RSSM_ERR_CUDA; }

// The KDA ring: the GDN fields, g holding one log decay per key channel.
void set_kda_ring(GdnArgs& a, const rssm_kda_ring* r) {
  a.rq = r->q;
  a.rk = r->k;
  a.rv = r->v;
  a.rg = r->g;
  a.rbeta = r->beta;
  a.re = r->e;
}

GdnArgs gdn_args(const rssm_gdn_desc* d) {
  GdnArgs a{};
  a.Bt = d->batch;
  a.H = d->nheads;
  a.DK = d->dk;
  a.DV = d->dv;
  a.L = d->buf_len;
  a.K = 1;
  a.slots = d->state_slots;
  a.Sn = (int)state_rows(d);
  return a;
}

}  // namespace

extern "C" {

int rssm_version(void) { return 200; }

int rssm_selftest_bounded_wait(int32_t* dev_status, rssm_stream_t stream) {
  int rc;
  if (!dev_status) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_opt(dev_status))) return rc;
  return cuda_rc(bounded_wait_selftest_launch(dev_status, (cudaStream_t)stream));
}

const char* rssm_status_string(int code) {
  switch (code) {
    case RSSM_OK: return "ok";
    case RSSM_ERR_INVALID_ARG: return "invalid argument (null pointer, bad dimension or bad count)";
    case RSSM_ERR_UNSUPPORTED: return "unsupported by the library (shape or size limit)";
    case RSSM_ERR_MISALIGNED: return "a base pointer is not 16-byte aligned";
    case RSSM_ERR_CUDA: return "CUDA launch error";
    case RSSM_DEV_BAD_CURSOR: return "device: cursor start/count out of range";
    case RSSM_DEV_WINDOW_FULL: return "device: AR step on a full window (flush or commit first)";
    case RSSM_DEV_PENDING: return "device: previous verify not committed";
    case RSSM_DEV_BAD_KEPT: return "device: kept outside [0, pending]";
    case RSSM_DEV_BAD_SLOT: return "device: state slot out of range";
    case RSSM_DEV_TIMEOUT: return "device: bounded wait for a bulk copy expired";
    default: return "unknown status code";
  }
}

int rssm_mamba2_ring_bytes(const rssm_mamba2_desc* d, size_t bytes[5]) {
  int rc = check_m2(d);
  if (rc) return rc;
  if (!bytes) return RSSM_ERR_INVALID_ARG;
  const size_t Bt = state_rows(d), H = d->nheads, L = d->buf_len, G = d->ngroups;
  bytes[0] = bytes[1] = Bt * H * L * d->headdim * 2;
  bytes[2] = bytes[3] = Bt * G * L * d->dstate * 2;
  bytes[4] = Bt * H * pad4(d->buf_len) * 4;
  return RSSM_OK;
}

int rssm_gdn_ring_bytes(const rssm_gdn_desc* d, size_t bytes[6]) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (!bytes) return RSSM_ERR_INVALID_ARG;
  const size_t Bt = state_rows(d), H = d->nheads, L = d->buf_len;
  bytes[0] = bytes[1] = Bt * H * L * d->dk * 2;
  bytes[2] = Bt * H * L * d->dv * 2;
  bytes[3] = bytes[4] = Bt * H * pad4(d->buf_len) * 4;
  bytes[5] = Bt * H * L * d->dv * 4;
  return RSSM_OK;
}

int rssm_mamba2_conventional_step(const rssm_mamba2_desc* d, float* state, const rssm_bf16* x, const rssm_bf16* z,
                                  const rssm_bf16* B, const rssm_bf16* C, const float* dt, const float* A,
                                  const float* D, void* y, rssm_stream_t stream) {
  int rc = check_m2(d);
  if (rc) return rc;
  if (d->state_slots) return RSSM_ERR_UNSUPPORTED;
  if (d->batch == 0) return RSSM_OK;
  if ((rc = check_ptrs({state, x, z, B, C, dt, A, D, y}))) return rc;
  M2Args a = m2_args(d);
  a.ckpt = state;
  a.x = x;
  a.z = z;
  a.B = B;
  a.C = C;
  a.dt = dt;
  a.A = A;
  a.D = D;
  a.y = y;
  return cuda_rc(m2_launch(M2_CONVENTIONAL, a, d->out_dtype == RSSM_BF16, (cudaStream_t)stream));
}

int rssm_mamba2_step(const rssm_mamba2_desc* d, float* ckpt, rssm_bf16* ckpt_read, const rssm_mamba2_ring* ring,
                     int32_t* cursors, const rssm_bf16* x, const rssm_bf16* z, const rssm_bf16* B,
                     const rssm_bf16* C, const float* dt, const float* A, const float* D, void* y,
                     int32_t* dev_status, rssm_stream_t stream) {
  int rc = check_m2(d);
  if (rc) return rc;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({ckpt, ring->x, ring->z, ring->B, ring->C, ring->dt, cursors, x, z, B, C, dt, A, D, y})))
    return rc;
  if ((rc = check_opt(ckpt_read)) || (rc = check_opt(dev_status))) return rc;
  M2Args a = m2_args(d);
  a.ckpt = ckpt;
  a.ckpt_read = ckpt_read;
  set_ring(a, ring);
  a.cursors = cursors;
  a.x = x;
  a.z = z;
  a.B = B;
  a.C = C;
  a.dt = dt;
  a.A = A;
  a.D = D;
  a.y = y;
  a.status = dev_status;
  cudaStream_t st = (cudaStream_t)stream;
  if (a.slots && !m2_step_fast_applies(a)) return RSSM_ERR_UNSUPPORTED;  // state slots: shape-specialised path
  if ((rc = cuda_rc(m2_launch(M2_STEP, a, d->out_dtype == RSSM_BF16, st)))) return rc;
  if (m2_step_fast_applies(a)) return RSSM_OK;  // that kernel advanced the cursors itself
  return cuda_rc(cursor_launch(CUR_AR, cursors, nullptr, d->batch, d->buf_len, dev_status, st));
}

// An emulated step's descriptor and format: the shape-specialised kernel's shapes, no slots, a listed
// format / scale pair. Fills the launch arguments' shape fields.
static int check_emulated(const rssm_mamba2_desc* d, const rssm_emulation* emu, M2Args& a) {
  int rc = check_m2(d);
  if (rc) return rc;
  if (!emu) return RSSM_ERR_INVALID_ARG;
  const bool unscaled = emu->format == RSSM_EMU_BF16 || emu->format == RSSM_EMU_F16;
  const bool scaled = emu->format == RSSM_EMU_E4M3 || emu->format == RSSM_EMU_E5M2 || emu->format == RSSM_EMU_INT8;
  if (!(unscaled && emu->scale == RSSM_EMU_SCALE_NONE) &&
      !(scaled && (emu->scale == RSSM_EMU_SCALE_ROW || emu->scale == RSSM_EMU_SCALE_TILE64)))
    return RSSM_ERR_INVALID_ARG;
  if (d->state_slots) return RSSM_ERR_UNSUPPORTED;
  a = m2_args(d);
  a.emu_fmt = emu->format;
  a.emu_scale = emu->scale;
  return m2_step_fast_applies(a) ? RSSM_OK : RSSM_ERR_UNSUPPORTED;
}

size_t rssm_mamba2_emulated_workspace_bytes(const rssm_mamba2_desc* d, int* rc_out) {
  // any listed format: the workspace depends on the shape alone
  const rssm_emulation probe = {RSSM_EMU_BF16, RSSM_EMU_SCALE_NONE};
  M2Args a{};
  const int rc = check_emulated(d, &probe, a);
  if (rc_out) *rc_out = rc;
  return rc ? 0 : m2_emulated_partials(a) * sizeof(float2);
}

int rssm_mamba2_step_emulated(const rssm_mamba2_desc* d, const rssm_emulation* emu, float* ckpt,
                              const rssm_mamba2_ring* ring, int32_t* cursors, const rssm_bf16* x, const rssm_bf16* z,
                              const rssm_bf16* B, const rssm_bf16* C, const float* dt, const float* A, const float* D,
                              void* y, double* err, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              rssm_stream_t stream) {
  M2Args a{};
  int rc = check_emulated(d, emu, a);
  if (rc) return rc;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({ckpt, ring->x, ring->z, ring->B, ring->C, ring->dt, cursors, x, z, B, C, dt, A, D, y, err,
                        workspace})))
    return rc;
  if ((rc = check_opt(dev_status))) return rc;
  if (workspace_bytes < m2_emulated_partials(a) * sizeof(float2)) return RSSM_ERR_INVALID_ARG;
  a.ckpt = ckpt;
  set_ring(a, ring);
  a.cursors = cursors;
  a.x = x;
  a.z = z;
  a.B = B;
  a.C = C;
  a.dt = dt;
  a.A = A;
  a.D = D;
  a.y = y;
  a.status = dev_status;
  a.emu_part = static_cast<float2*>(workspace);
  return cuda_rc(m2_step_emulated_launch(a, d->out_dtype == RSSM_BF16, err, (cudaStream_t)stream));
}

int rssm_mamba2_step_emulated_noalloc(const rssm_mamba2_desc* d, const rssm_emulation* emu, float* ckpt,
                                      const rssm_mamba2_ring* ring, int32_t* cursors, const rssm_bf16* x,
                                      const rssm_bf16* z, const rssm_bf16* B, const rssm_bf16* C, const float* dt,
                                      const float* A, const float* D, void* y, double* err, int32_t* dev_status,
                                      rssm_stream_t stream) {
  M2Args a{};
  int rc = check_emulated(d, emu, a);
  if (rc) return rc;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({ckpt, ring->x, ring->z, ring->B, ring->C, ring->dt, cursors, x, z, B, C, dt, A, D, y, err})))
    return rc;
  if ((rc = check_opt(dev_status))) return rc;
  if (m2_emulated_partials(a) > (size_t)M2_NOALLOC_PARTIALS) return RSSM_ERR_UNSUPPORTED;  // beyond the static array
  a.ckpt = ckpt;
  set_ring(a, ring);
  a.cursors = cursors;
  a.x = x;
  a.z = z;
  a.B = B;
  a.C = C;
  a.dt = dt;
  a.A = A;
  a.D = D;
  a.y = y;
  a.status = dev_status;
  return cuda_rc(m2_step_emulated_noalloc_launch(a, d->out_dtype == RSSM_BF16, err, (cudaStream_t)stream));
}

int rssm_mamba2_flush(const rssm_mamba2_desc* d, float* ckpt, rssm_bf16* ckpt_read, const rssm_mamba2_ring* ring,
                      int32_t* cursors, const float* A, int32_t* dev_status, rssm_stream_t stream) {
  int rc = check_m2(d);
  if (rc) return rc;
  if (d->state_slots) return RSSM_ERR_UNSUPPORTED;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({ckpt, ring->x, ring->B, ring->dt, cursors, A}))) return rc;
  if ((rc = check_opt(ckpt_read)) || (rc = check_opt(dev_status))) return rc;
  M2Args a = m2_args(d);
  a.ckpt = ckpt;
  a.ckpt_read = ckpt_read;
  set_ring(a, ring);
  a.cursors = cursors;
  a.A = A;
  a.status = dev_status;
  cudaStream_t st = (cudaStream_t)stream;
  if ((rc = cuda_rc(m2_launch(M2_FLUSH, a, 0, st)))) return rc;
  return cuda_rc(cursor_launch(CUR_FLUSH, cursors, nullptr, d->batch, d->buf_len, dev_status, st));
}

int rssm_mamba2_spec_verify(const rssm_mamba2_desc* d, int n_new, float* ckpt, rssm_bf16* ckpt_read,
                            const rssm_mamba2_ring* ring, int32_t* cursors, const rssm_bf16* x, const rssm_bf16* z,
                            const rssm_bf16* B, const rssm_bf16* C, const float* dt, const float* A,
                            const float* D, void* y, int32_t* dev_status, rssm_stream_t stream) {
  int rc = check_m2(d);
  if (rc) return rc;
  if (n_new < 1 || n_new > d->buf_len) return RSSM_ERR_INVALID_ARG;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({ckpt, ring->x, ring->z, ring->B, ring->C, ring->dt, cursors, x, z, B, C, dt, A, D, y})))
    return rc;
  if ((rc = check_opt(ckpt_read)) || (rc = check_opt(dev_status))) return rc;
  M2Args a = m2_args(d);
  a.K = n_new;
  a.ckpt = ckpt;
  a.ckpt_read = ckpt_read;
  set_ring(a, ring);
  a.cursors = cursors;
  a.x = x;
  a.z = z;
  a.B = B;
  a.C = C;
  a.dt = dt;
  a.A = A;
  a.D = D;
  a.y = y;
  a.status = dev_status;
  // fp8 read copies and state slots: the shape-specialised path only (K <= 4, L + K <= 32)
  if (((a.read_f8 && a.ckpt_read) || a.slots) && !m2_verify_fast_applies(a)) return RSSM_ERR_UNSUPPORTED;
  return cuda_rc(m2_launch(M2_VERIFY, a, d->out_dtype == RSSM_BF16, (cudaStream_t)stream));
}

int rssm_commit_cursors(int32_t* cursors, const int32_t* kept, int batch, int buf_len, int32_t* dev_status,
                        rssm_stream_t stream) {
  if (batch < 0 || buf_len < 1 || buf_len > RSSM_MAX_BUF_LEN) return RSSM_ERR_INVALID_ARG;
  if (batch == 0) return RSSM_OK;
  int rc;
  if ((rc = check_ptrs({cursors, kept})) || (rc = check_opt(dev_status))) return rc;
  return cuda_rc(cursor_launch(CUR_COMMIT, cursors, kept, batch, buf_len, dev_status, (cudaStream_t)stream));
}

int rssm_commit_cursors_slots(int32_t* cursors, const int32_t* kept, const int32_t* state_slots, int batch,
                              int n_slots, int buf_len, int32_t* dev_status, rssm_stream_t stream) {
  if (batch < 0 || n_slots < 0 || buf_len < 1 || buf_len > RSSM_MAX_BUF_LEN) return RSSM_ERR_INVALID_ARG;
  if (batch == 0) return RSSM_OK;
  int rc;
  if ((rc = check_ptrs({cursors, kept})) || (rc = check_opt(dev_status))) return rc;
  if (!state_slots) return RSSM_ERR_INVALID_ARG;
  return cuda_rc(cursor_launch(CUR_COMMIT, cursors, kept, batch, buf_len, dev_status, (cudaStream_t)stream,
                               state_slots, n_slots));
}

int rssm_reset_cursors(int32_t* cursors, const int32_t* slots, int n_slots, int batch, int32_t* dev_status,
                       rssm_stream_t stream) {
  if (n_slots < 0 || batch < 0) return RSSM_ERR_INVALID_ARG;
  if (n_slots == 0) return RSSM_OK;
  int rc;
  if ((rc = check_ptrs({cursors, slots})) || (rc = check_opt(dev_status))) return rc;
  return cuda_rc(reset_launch(cursors, slots, n_slots, batch, dev_status, (cudaStream_t)stream));
}

int rssm_checkpoint_downcast(const float* src, rssm_bf16* dst, size_t n, int dtype, rssm_stream_t stream) {
  if (dtype != RSSM_BF16 && dtype != RSSM_F16) return RSSM_ERR_INVALID_ARG;
  if (n == 0) return RSSM_OK;
  int rc;
  if ((rc = check_ptrs({src, dst}))) return rc;
  return cuda_rc(downcast_launch(src, dst, n, dtype == RSSM_F16, (cudaStream_t)stream));
}

int rssm_mamba2_downcast(const rssm_mamba2_desc* d, const float* ckpt, void* ckpt_read, rssm_stream_t stream) {
  int rc = check_m2(d);
  if (rc) return rc;
  if (d->state_slots) return RSSM_ERR_UNSUPPORTED;
  if (d->batch == 0) return RSSM_OK;
  if ((rc = check_ptrs({ckpt, ckpt_read}))) return rc;
  const size_t rows = (size_t)d->batch * d->nheads * d->headdim;
  if (d->read_dtype == RSSM_FP8_E4M3)
    return cuda_rc(downcast_f8_launch(ckpt, static_cast<uint8_t*>(ckpt_read), rows, (cudaStream_t)stream));
  return cuda_rc(downcast_launch(ckpt, static_cast<uint16_t*>(ckpt_read), rows * d->dstate, d->read_dtype == RSSM_F16,
                                 (cudaStream_t)stream));
}

int rssm_gdn_conventional_step(const rssm_gdn_desc* d, float* S, const rssm_bf16* q, const rssm_bf16* k,
                               const rssm_bf16* v, const float* g, const float* beta, void* o,
                               rssm_stream_t stream) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (d->state_slots) return RSSM_ERR_UNSUPPORTED;
  if (d->batch == 0) return RSSM_OK;
  if ((rc = check_ptrs({S, q, k, v, g, beta, o}))) return rc;
  GdnArgs a = gdn_args(d);
  a.S = S;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.o = o;
  return cuda_rc(gdn_launch(GDN_CONVENTIONAL, a, d->out_dtype == RSSM_BF16, (cudaStream_t)stream));
}

int rssm_gdn_step(const rssm_gdn_desc* d, float* S, const rssm_gdn_ring* ring, int32_t* cursors, const rssm_bf16* q,
                  const rssm_bf16* k, const rssm_bf16* v, const float* g, const float* beta, void* o,
                  int32_t* dev_status, rssm_stream_t stream) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({S, ring->q, ring->k, ring->v, ring->g, ring->beta, ring->e, cursors, q, k, v, g, beta, o})))
    return rc;
  if ((rc = check_opt(dev_status))) return rc;
  GdnArgs a = gdn_args(d);
  a.S = S;
  a.rq = ring->q;
  a.rk = ring->k;
  a.rv = ring->v;
  a.rg = ring->g;
  a.rbeta = ring->beta;
  a.re = ring->e;
  a.cursors = cursors;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.o = o;
  a.status = dev_status;
  cudaStream_t st = (cudaStream_t)stream;
  if (a.slots && !gdn_step_fast_applies(a)) return RSSM_ERR_UNSUPPORTED;  // state slots: shape-specialised path
  if ((rc = cuda_rc(gdn_launch(GDN_STEP, a, d->out_dtype == RSSM_BF16, st)))) return rc;
  if (gdn_step_fast_applies(a)) return RSSM_OK;  // that kernel advanced the cursors itself
  return cuda_rc(cursor_launch(CUR_AR, cursors, nullptr, d->batch, d->buf_len, dev_status, st));
}

int rssm_gdn_flush(const rssm_gdn_desc* d, float* S, const rssm_gdn_ring* ring, int32_t* cursors, int32_t* dev_status,
                   rssm_stream_t stream) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (d->state_slots) return RSSM_ERR_UNSUPPORTED;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({S, ring->k, ring->v, ring->g, ring->beta, cursors}))) return rc;
  if ((rc = check_opt(dev_status))) return rc;
  GdnArgs a = gdn_args(d);
  a.S = S;
  a.rq = ring->q;
  a.rk = ring->k;
  a.rv = ring->v;
  a.rg = ring->g;
  a.rbeta = ring->beta;
  a.re = ring->e;
  a.cursors = cursors;
  a.status = dev_status;
  cudaStream_t st = (cudaStream_t)stream;
  if ((rc = cuda_rc(gdn_launch(GDN_FLUSH, a, 0, st)))) return rc;
  return cuda_rc(cursor_launch(CUR_FLUSH, cursors, nullptr, d->batch, d->buf_len, dev_status, st));
}

int rssm_gdn_spec_verify(const rssm_gdn_desc* d, int n_new, float* S, const rssm_gdn_ring* ring, int32_t* cursors,
                         const rssm_bf16* q, const rssm_bf16* k, const rssm_bf16* v, const float* g,
                         const float* beta, void* o, int32_t* dev_status, rssm_stream_t stream) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (n_new < 1 || n_new > d->buf_len) return RSSM_ERR_INVALID_ARG;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({S, ring->q, ring->k, ring->v, ring->g, ring->beta, ring->e, cursors, q, k, v, g, beta, o})))
    return rc;
  if ((rc = check_opt(dev_status))) return rc;
  GdnArgs a = gdn_args(d);
  a.K = n_new;
  a.S = S;
  a.rq = ring->q;
  a.rk = ring->k;
  a.rv = ring->v;
  a.rg = ring->g;
  a.rbeta = ring->beta;
  a.re = ring->e;
  a.cursors = cursors;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.o = o;
  a.status = dev_status;
  if (a.slots && !gdn_verify_fast_applies(a)) return RSSM_ERR_UNSUPPORTED;  // state slots: shape-specialised path
  return cuda_rc(gdn_verify_launch(a, d->out_dtype == RSSM_BF16, (cudaStream_t)stream));
}

int rssm_gdn_prime(const rssm_gdn_desc* d, const float* S, const rssm_gdn_ring* ring, const int32_t* cursors,
                   int32_t* dev_status, rssm_stream_t stream) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (d->state_slots) return RSSM_ERR_UNSUPPORTED;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({S, ring->k, ring->v, ring->g, ring->beta, ring->e, cursors}))) return rc;
  if ((rc = check_opt(dev_status))) return rc;
  GdnArgs a = gdn_args(d);
  a.S = const_cast<float*>(S);  // read only in this mode
  a.rq = ring->q;
  a.rk = ring->k;
  a.rv = ring->v;
  a.rg = ring->g;
  a.rbeta = ring->beta;
  a.re = ring->e;
  a.cursors = const_cast<int32_t*>(cursors);  // read only in this mode
  a.status = dev_status;
  return cuda_rc(gdn_launch(GDN_PRIME, a, 0, (cudaStream_t)stream));
}

// ---------------------------------------------------------------- Kimi Delta Attention

int rssm_kda_ring_bytes(const rssm_kda_desc* d, size_t bytes[6]) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (!bytes) return RSSM_ERR_INVALID_ARG;
  const size_t Bt = state_rows(d), H = d->nheads, L = d->buf_len;
  bytes[0] = bytes[1] = Bt * H * L * d->dk * 2;
  bytes[2] = Bt * H * L * d->dv * 2;
  bytes[3] = Bt * H * L * d->dk * 4;
  bytes[4] = Bt * H * pad4(d->buf_len) * 4;
  bytes[5] = Bt * H * L * d->dv * 4;
  return RSSM_OK;
}

int rssm_kda_conventional_step(const rssm_kda_desc* d, float* S, const rssm_bf16* q, const rssm_bf16* k,
                               const rssm_bf16* v, const float* g, const float* beta, void* o,
                               rssm_stream_t stream) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (d->state_slots) return RSSM_ERR_UNSUPPORTED;
  if (d->batch == 0) return RSSM_OK;
  if ((rc = check_ptrs({S, q, k, v, g, beta, o}))) return rc;
  GdnArgs a = gdn_args(d);
  a.S = S;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.o = o;
  return cuda_rc(kda_launch(GDN_CONVENTIONAL, a, d->out_dtype == RSSM_BF16, (cudaStream_t)stream));
}

int rssm_kda_step(const rssm_kda_desc* d, float* S, const rssm_kda_ring* ring, int32_t* cursors, const rssm_bf16* q,
                  const rssm_bf16* k, const rssm_bf16* v, const float* g, const float* beta, void* o,
                  int32_t* dev_status, rssm_stream_t stream) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({S, ring->q, ring->k, ring->v, ring->g, ring->beta, ring->e, cursors, q, k, v, g, beta, o})))
    return rc;
  if ((rc = check_opt(dev_status))) return rc;
  GdnArgs a = gdn_args(d);
  if (!kda_step_fast_applies(a)) return RSSM_ERR_UNSUPPORTED;  // dk = dv = 128, L <= 31
  a.S = S;
  set_kda_ring(a, ring);
  a.cursors = cursors;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.o = o;
  a.status = dev_status;
  return cuda_rc(kda_launch(GDN_STEP, a, d->out_dtype == RSSM_BF16, (cudaStream_t)stream));  // cursors advance inside
}

int rssm_kda_flush(const rssm_kda_desc* d, float* S, const rssm_kda_ring* ring, int32_t* cursors, int32_t* dev_status,
                   rssm_stream_t stream) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (d->state_slots) return RSSM_ERR_UNSUPPORTED;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({S, ring->k, ring->g, ring->e, cursors}))) return rc;
  if ((rc = check_opt(dev_status))) return rc;
  GdnArgs a = gdn_args(d);
  if (!kda_window_applies(a)) return RSSM_ERR_UNSUPPORTED;
  a.S = S;
  set_kda_ring(a, ring);
  a.cursors = cursors;
  a.status = dev_status;
  cudaStream_t st = (cudaStream_t)stream;
  if ((rc = cuda_rc(kda_launch(GDN_FLUSH, a, 0, st)))) return rc;
  return cuda_rc(cursor_launch(CUR_FLUSH, cursors, nullptr, d->batch, d->buf_len, dev_status, st));
}

int rssm_kda_spec_verify(const rssm_kda_desc* d, int n_new, float* S, const rssm_kda_ring* ring, int32_t* cursors,
                         const rssm_bf16* q, const rssm_bf16* k, const rssm_bf16* v, const float* g,
                         const float* beta, void* o, int32_t* dev_status, rssm_stream_t stream) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (n_new < 1 || n_new > d->buf_len) return RSSM_ERR_INVALID_ARG;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({S, ring->q, ring->k, ring->v, ring->g, ring->beta, ring->e, cursors, q, k, v, g, beta, o})))
    return rc;
  if ((rc = check_opt(dev_status))) return rc;
  GdnArgs a = gdn_args(d);
  a.K = n_new;
  if (!kda_verify_applies(a)) return RSSM_ERR_UNSUPPORTED;  // dk = dv = 128, K <= 4, L + K <= 32
  a.S = S;
  set_kda_ring(a, ring);
  a.cursors = cursors;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = g;
  a.beta = beta;
  a.o = o;
  a.status = dev_status;
  return cuda_rc(kda_verify_launch(a, d->out_dtype == RSSM_BF16, (cudaStream_t)stream));
}

int rssm_kda_prime(const rssm_kda_desc* d, const float* S, const rssm_kda_ring* ring, const int32_t* cursors,
                   int32_t* dev_status, rssm_stream_t stream) {
  int rc = check_gdn(d);
  if (rc) return rc;
  if (d->state_slots) return RSSM_ERR_UNSUPPORTED;
  if (d->batch == 0) return RSSM_OK;
  if (!ring) return RSSM_ERR_INVALID_ARG;
  if ((rc = check_ptrs({S, ring->k, ring->v, ring->g, ring->beta, ring->e, cursors}))) return rc;
  if ((rc = check_opt(dev_status))) return rc;
  GdnArgs a = gdn_args(d);
  if (!kda_window_applies(a)) return RSSM_ERR_UNSUPPORTED;
  a.S = const_cast<float*>(S);  // read only in this mode
  set_kda_ring(a, ring);
  a.cursors = const_cast<int32_t*>(cursors);  // read only in this mode
  a.status = dev_status;
  return cuda_rc(kda_launch(GDN_PRIME, a, 0, (cudaStream_t)stream));
}

}  // extern "C"

namespace rssm {

cudaError_t prepare_kernel(const void* fn, size_t dyn_smem, bool max_carveout) {
  struct Entry {
    const void* fn;
    int device;
    size_t smem;  // dynamic shared-memory limit set so far (0: the default)
    bool carveout;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const size_t need = dyn_smem > 48 * 1024 ? dyn_smem : 0;
  std::lock_guard<std::mutex> lock(mu);
  Entry* ent = nullptr;
  for (Entry& d : done)
    if (d.fn == fn && d.device == dev) ent = &d;
  if (!ent) {
    done.push_back(Entry{fn, dev, 0, false});
    ent = &done.back();
  }
  if (max_carveout && !ent->carveout) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    ent->carveout = true;
  }
  if (need > ent->smem) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)need);
    if (e != cudaSuccess) return e;
    ent->smem = need;
  }
  return cudaSuccess;
}

}  // namespace rssm
