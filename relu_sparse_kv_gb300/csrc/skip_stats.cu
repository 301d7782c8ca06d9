// V-read accounting at a chosen granularity.
//
// Source: "The Architecture of Embla 1", section "Skipping V": a value row is read only
// when some query head of the KV group gives its key a weight above zero, i.e. when the
// selection score sigma_j = max_h s_hj is above zero; the page's own kernel checks keys
// in groups of 8 at a time.
//
// One CTA per (batch, KV head) unit.  A warp takes one block of max(chunk, 32) keys at a
// time: each lane tests one key per 32-key word, the ballot is that word's survivor mask,
// and a chunk of up to 32 keys is needed when its field of the mask is non-zero (a longer
// chunk when any of its words is).
#include "internal.h"
#include "ptx.cuh"

namespace embla {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct StatsParams {
  const float *sel;
  int64_t n, ncap;
  int chunk;  // a power of two, 1..1024
  int32_t *keys_needed, *chunks_needed;
};

// Lowest bit of every chunk-wide field of a 32-bit word (chunk <= 32).
__device__ __forceinline__ uint32_t field_starts(int chunk) {
  switch (chunk) {
    case 1: return 0xFFFFFFFFu;
    case 2: return 0x55555555u;
    case 4: return 0x11111111u;
    case 8: return 0x01010101u;
    case 16: return 0x00010001u;
    default: return 0x00000001u;
  }
}

__global__ void __launch_bounds__(kThreads) skip_stats_kernel(const StatsParams p) {
  pdl_wait_primary();  // the selection scores are complete
  pdl_launch_dependents();
  __shared__ int32_t s_keys, s_chunks;
  if (threadIdx.x == 0) {
    s_keys = 0;
    s_chunks = 0;
  }
  __syncthreads();
  const int64_t u = blockIdx.x;
  const float *sel = p.sel + u * p.ncap;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int block = p.chunk > 32 ? p.chunk : 32;  // keys a warp takes at a time
  const int words = block / 32;
  const uint32_t starts = field_starts(p.chunk);
  int keys = 0, chunks = 0;
  for (int64_t b0 = static_cast<int64_t>(warp) * block; b0 < p.n; b0 += static_cast<int64_t>(kWarps) * block) {
    uint32_t any = 0u;
    for (int w = 0; w < words; ++w) {
      const int64_t j = b0 + 32 * w + lane;
      const uint32_t m = __ballot_sync(0xffffffffu, j < p.n && sel[j] > 0.0f);
      keys += __popc(m);
      if (p.chunk <= 32) {
        // fold each field onto its lowest bit, then count the fields that are set
        uint32_t f = m;
        for (int k = 1; k < p.chunk; k <<= 1) f |= f >> k;
        chunks += __popc(f & starts);
      } else {
        any |= m;
      }
    }
    if (p.chunk > 32 && any) ++chunks;
  }
  if (lane == 0) {
    atomicAdd(&s_keys, keys);
    atomicAdd(&s_chunks, chunks);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    p.keys_needed[u] = s_keys;
    p.chunks_needed[u] = s_chunks;
  }
}

}  // namespace

cudaError_t launch_skip_stats(const float *sel_scores, int64_t units, int64_t n, int64_t ncap,
                              int chunk, int32_t *keys_needed, int32_t *chunks_needed,
                              cudaStream_t stream) {
  if (units == 0) return cudaSuccess;
  StatsParams p;
  p.sel = sel_scores;
  p.n = n;
  p.ncap = ncap;
  p.chunk = chunk;
  p.keys_needed = keys_needed;
  p.chunks_needed = chunks_needed;
  return launch_pdl(skip_stats_kernel, dim3(static_cast<unsigned>(units)), dim3(kThreads), 0,
                    stream, 0u, p);
}

}  // namespace embla
