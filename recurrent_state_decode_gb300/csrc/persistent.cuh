// Pieces shared by the persistent, warp-specialised kernels: one CTA per SM,
// NGROUPS groups of NCONS consumer warps plus one producer warp, an S-deep ring
// of shared-memory stages guarded by `full` (bulk copies landed) and `empty`
// (the consuming group is done) mbarriers. Tiles are dealt out round-robin
// over the grid; inside a CTA its j-th tile goes to stage j mod S and to
// consumer group j mod NGROUPS, so two tiles are computed at a time while the
// other stages load, and every scheduler holds two consumer warps to hide
// latency with.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace rssm {
namespace persistent {

constexpr int NCONS = 4;                    // consumer warps per group (one tile each)
constexpr int NGROUPS = 2;                  // consumer groups
constexpr int NCW = NCONS * NGROUPS;        // consumer warps
constexpr int THREADS = 32 * (NCW + 1);     // + one producer warp
constexpr int MAX_STAGES = 8;
constexpr uint32_t BAR_BYTES = 3 * MAX_STAGES * 8;  // full, empty, aux [MAX_STAGES]

// Stage-relative byte offsets are handed out 128-byte aligned.
struct Carver {
  uint32_t off = 0;
  uint32_t take(uint32_t bytes) {
    const uint32_t o = off;
    off = (off + bytes + 127u) & ~127u;
    return o;
  }
};

__device__ __forceinline__ void decode_tile(const M2Args& a, int t, int& b, int& h, int& pb) {
  pb = t % a.nPB;
  t /= a.nPB;
  h = t % a.H;
  b = t / a.H;
}

// Rows [r0, r1) of consumer warp w: the R rows (a multiple of 8) in 8-row
// groups dealt out contiguously to the NCONS consumers.
__device__ __forceinline__ void consumer_rows(int R, int w, int& r0, int& r1) {
  const int ngrp = R >> 3;
  r0 = ((w * ngrp) / NCONS) * 8;
  r1 = (((w + 1) * ngrp) / NCONS) * 8;
}

// full[s]: one producer arrival + the stage's bulk-copy bytes; empty[s] and
// aux[s]: one arrival per warp of the consuming group.
__device__ __forceinline__ void init_ring(uint64_t* bars, int S) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; s++) {
      mbar_init(&bars[s], 1);
      mbar_init(&bars[MAX_STAGES + s], NCONS);
      mbar_init(&bars[2 * MAX_STAGES + s], NCONS);
    }
    fence_mbar_init();
  }
  __syncthreads();
}

struct DeviceInfo {
  int sms = 0, smem_optin = 0;
};

inline DeviceInfo device_info() {
  static DeviceInfo cache[64];
  int dev = 0;
  cudaGetDevice(&dev);
  DeviceInfo& d = cache[dev & 63];
  if (d.sms == 0) {
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  }
  return d;
}

// Stages that fit the opt-in shared memory of one CTA (0 if fewer than 2).
inline int stages_for(uint32_t stage_bytes) {
  const DeviceInfo di = device_info();
  int S = (int)((di.smem_optin - (int)BAR_BYTES) / (int)stage_bytes);
  if (S > MAX_STAGES) S = MAX_STAGES;
  return S < 2 ? 0 : S;
}

}  // namespace persistent
}  // namespace rssm
