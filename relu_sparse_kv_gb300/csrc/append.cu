// Appending the decode step's token to the caches: row `pos` of every (batch, KV head)
// plane of a cache is copied from a packed array holding one row per plane.  The decode
// calls read the caches as they lie; this is how the current token's K and V (and, for
// 8-bit caches, their per-token scales) get there without a copy kernel of the caller's
// between the step's kernels, which would hold up the launch of the full-layer kernels
// behind it ("The Architecture of Embla 1", "Three kinds of attention": the full layers
// keep a cache of every token).
#include "internal.h"
#include "ptx.cuh"

namespace embla {
namespace {

// Up to four arrays in one launch; every thread walks the pieces of all of them.
__global__ void __launch_bounds__(256) append_rows_kernel(const AppendParams p) {
  // The kernel after this one may launch now: it waits for this kernel to finish before it
  // reads anything, so it sees the appended rows.
  pdl_launch_dependents();
  pdl_wait_primary();  // the packed rows have been written
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int j = 0; j < p.njobs; ++j) {
    const AppendJob &a = p.job[j];
    const int64_t per = a.row_bytes / a.vec;  // pieces of a row
    const int64_t total = p.units * per;
    for (int64_t e = t0; e < total; e += stride) {
      const int64_t u = e / per, k = e - u * per;
      const uint8_t *s = a.src + u * a.row_bytes + k * a.vec;
      uint8_t *d = a.dst + (u * a.cache_stride + p.pos) * a.row_bytes + k * a.vec;
      if (a.vec == 16)
        *reinterpret_cast<uint4 *>(d) = *reinterpret_cast<const uint4 *>(s);
      else if (a.vec == 4)
        *reinterpret_cast<uint32_t *>(d) = *reinterpret_cast<const uint32_t *>(s);
      else
        *d = *s;
    }
  }
}

// The widest piece (16, 4 or 1 bytes) that every source and destination address is a
// multiple of.
int piece_bytes(const AppendJob &a, int64_t pos) {
  const uint64_t addr = reinterpret_cast<uintptr_t>(a.src) | reinterpret_cast<uintptr_t>(a.dst);
  const uint64_t steps = static_cast<uint64_t>(a.row_bytes) |
                         static_cast<uint64_t>(a.cache_stride * a.row_bytes) |
                         static_cast<uint64_t>(pos * a.row_bytes);
  const uint64_t all = addr | steps;
  if ((all & 15u) == 0) return 16;
  if ((all & 3u) == 0) return 4;
  return 1;
}

}  // namespace

cudaError_t launch_append_rows(const AppendJob *jobs, int njobs, int64_t units, int64_t pos,
                               cudaStream_t stream) {
  if (njobs < 1 || njobs > kAppendMaxJobs) return cudaErrorInvalidValue;
  if (units == 0) return cudaSuccess;
  AppendParams p = {};
  p.njobs = njobs;
  p.units = units;
  p.pos = pos;
  int64_t most = 0;
  for (int j = 0; j < njobs; ++j) {
    p.job[j] = jobs[j];
    p.job[j].vec = piece_bytes(jobs[j], pos);
    const int64_t pieces = units * (jobs[j].row_bytes / p.job[j].vec);
    if (pieces > most) most = pieces;
  }
  const int64_t blocks = (most + 255) / 256;
  return launch_pdl(append_rows_kernel, dim3(static_cast<unsigned>(blocks < 64 ? blocks : 64)),
                    dim3(256), 0, stream, 0u, p);
}

}  // namespace embla
