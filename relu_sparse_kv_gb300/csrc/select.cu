// Sparse-layer selection: the top-k keys by the full layer's selection score among
// the non-recent keys, plus the `recent` newest keys, in ascending index order.
//
// Source: "The Architecture of Embla 1", section "Three kinds of attention" (Sparse):
// the sparse layers reuse the 1,024 keys the full layer scored highest together with
// the 128 newest, chosen by score whether or not the key survived ReLU^2.
//
// Exact radix select on the order-preserving 32-bit key of each fp32 score, with the
// key index as a tie-break (equal scores: smaller index first), i.e. on the unique
// 64-bit key (order_key(sigma) << 32) | (2^32 - 1 - j).  The top 11 bits were
// histogrammed by the full-layer decode.
//
// Contexts up to 8 x 32768 keys (select_fast_kernel): a cluster of one to eight CTAs of
// 1024 threads per (batch, KV head), each holding the order keys of 32768 keys and its
// selection bitmap in shared memory:
//   1  the scores load (coalesced, 32 per thread) while the histogram, minus the recent
//      keys, gives the boundary bin b* and the count `above` of keys above it;
//   2  one pass marks the keys above b* (and the recent keys) as selected and those in
//      b* as candidates, straight from the warp ballots;
//   3  while the unit has more than kRankMax candidates, an 8-bit digit of the 64-bit
//      key below the bin is histogrammed over the cluster and the candidates above /
//      below the boundary digit are decided; the last few are ranked pairwise;
//   4  each CTA writes the indices of its words in order after those of lower ranks.
//
// Longer contexts (select_kernel): one cluster of 8 CTAs per (batch, KV head):
//   A  every CTA finds the boundary bin from the histogram minus the recent keys, while
//      its chunk of scores is already loading;
//   B  it classifies its chunk: bitmap words for keys above the bin (and recent keys),
//      a list of the keys inside it;
//   C  the boundary bin is resolved exactly: each CTA ranks its own boundary keys against
//      all of the unit's (read through distributed shared memory) and sets its chosen
//      keys' bits; if the bin is very full the leader does it instead (bitonic sort in
//      shared memory after 8-bit radix passes);
//   D  each CTA counts its bits, takes the counts of the CTAs before it through
//      distributed shared memory, and writes its indices in ascending order.
#include <cooperative_groups.h>

#include "internal.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace embla {
namespace {

constexpr int kCl = 8;             // CTAs per unit
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 16;           // keys a thread classifies per pass
constexpr int kSortCap = 2048;     // boundary-bin keys sorted in shared memory at once
constexpr int kLocalCap = 512;     // boundary-bin keys a CTA keeps for the ranking path
constexpr int kRankCap = kLocalCap * kCl;  // boundary-bin keys of a unit the fast path handles

struct SelLayout {
  int64_t words;  // bitmap words per unit
  int64_t chunk;  // keys per CTA (a multiple of 32)
  size_t bitmap_off, cand_off, bufa_off, bufb_off, total;
};

SelLayout sel_layout(int64_t units, int64_t n) {
  SelLayout L;
  L.chunk = ((n + kCl - 1) / kCl + 31) / 32 * 32;
  L.words = (n + 31) / 32;
  const int64_t cand_per_unit = L.chunk * kCl;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return o;
  };
  L.bitmap_off = take(static_cast<size_t>(units * (L.words + kCl)) * 4);
  L.cand_off = take(static_cast<size_t>(units * cand_per_unit) * 4);
  L.bufa_off = take(static_cast<size_t>(units * cand_per_unit) * 4);
  L.bufb_off = take(static_cast<size_t>(units * cand_per_unit) * 4);
  L.total = off;
  return L;
}

struct SelParams {
  const float *sel;
  const uint32_t *hist;
  int64_t n, ncap, words, chunk;
  int topk, recent;
  uint32_t *bitmap;   // [U][words + kCl]
  int32_t *cand;      // [U][kCl][chunk]
  int32_t *bufa, *bufb;
  int32_t *idx;
  int idx_stride;
  int32_t *count;
};

struct Shared {
  uint32_t h[kHistBins];
  uint64_t keys[kSortCap];
  uint64_t local[kLocalCap];  // this CTA's boundary-bin keys
  uint64_t local2[kLocalCap]; // its keys tied at the second-level boundary digit
  uint32_t dh[256];
  int32_t warp_sum[kWarps];
  int32_t bin, above;        // boundary bin, candidates strictly above it
  int32_t ncand;             // boundary-bin keys listed by this CTA
  int32_t bits;              // selected keys in this CTA's chunk (after C)
  int32_t added[kCl];        // leader: boundary keys it selected per CTA chunk
  int32_t len, dstar, dabove;
  int32_t mine_added;        // boundary keys this CTA selected itself (ranking path)
  int32_t n2;                // entries of local2
  int32_t d2, above2;        // second-level boundary digit, keys above it
};

__device__ __forceinline__ uint64_t select_key(float s, int64_t j) {
  return (static_cast<uint64_t>(order_key(s)) << 32) |
         static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(j));
}

__device__ __forceinline__ uint64_t select_key_ok(uint32_t okey, int64_t j) {
  return (static_cast<uint64_t>(okey) << 32) |
         static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(j));
}

// Exclusive block scan of one int per thread; returns the prefix and sets *total.
__device__ int block_exclusive_scan(int v, int *total, int32_t *warp_sum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sum[warp] = x;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int s = warp_sum[w];
    before += w < warp ? s : 0;
    all += s;
  }
  __syncthreads();
  *total = all;
  return before + x - v;
}

// Sort keys[0, m) descending in shared memory (bitonic network over the next power of two).
__device__ void bitonic_desc(uint64_t *keys, int m) {
  int m2 = 1;
  while (m2 < m) m2 <<= 1;
  for (int i = m + threadIdx.x; i < m2; i += blockDim.x) keys[i] = 0ull;
  __syncthreads();
  for (int k = 2; k <= m2; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = threadIdx.x; i < m2; i += blockDim.x) {
        const int l = i ^ jj;
        if (l > i) {
          const uint64_t a = keys[i], b = keys[l];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            keys[i] = b;
            keys[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kThreads)
    select_kernel(const SelParams p) {
  pdl_wait_primary();  // the scores and histogram are complete
  pdl_launch_dependents();
  __shared__ Shared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t u = blockIdx.x / kCl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = p.n;
  const int64_t j0 = rank * p.chunk;
  const int64_t j1 = min(n, j0 + p.chunk);
  int32_t *idx = p.idx + u * p.idx_stride;

  if (n <= static_cast<int64_t>(p.topk) + p.recent) {
    for (int64_t j = j0 + tid; j < j1; j += kThreads) idx[j] = static_cast<int32_t>(j);
    if (rank == 0 && tid == 0) p.count[u] = static_cast<int32_t>(n);
    return;
  }
  const float *sel = p.sel + u * p.ncap;
  uint32_t *bitmap = p.bitmap + u * (p.words + kCl);
  int32_t *cand = p.cand + (u * kCl + rank) * p.chunk;
  const int64_t first_recent = n - p.recent;

  // ---- A: boundary bin (the first pass of this CTA's scores is loading meanwhile)
  float pre[kPer];
  {
    const int64_t base = j0 + warp * 32 * kPer + lane;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int64_t j = base + 32 * k;
      pre[k] = j < j1 ? sel[j] : 0.0f;
    }
  }
  // the recent keys' scores load together with the histogram (one round trip)
  float rsig = 0.0f;
  const bool has_recent = tid < p.recent;
  if (has_recent) rsig = sel[first_recent + tid];
  for (int i = tid; i < kHistBins; i += kThreads) sh.h[i] = p.hist[u * kHistBins + i];
  for (int i = tid; i < 256; i += kThreads) sh.dh[i] = 0u;
  if (tid == 0) {
    sh.ncand = 0;
    sh.n2 = 0;
  }
  __syncthreads();
  for (int64_t j = first_recent + kThreads + tid; j < n; j += kThreads)  // recent > kThreads
    atomicSub(&sh.h[order_key(sel[j]) >> 21], 1u);
  {
    // one shared-memory atomic per distinct bin in the warp
    const uint32_t rmask = __ballot_sync(0xffffffffu, has_recent);
    if (has_recent) {
      const uint32_t bin = order_key(rsig) >> 21;
      const uint32_t peers = __match_any_sync(rmask, bin);
      if (lane == __ffs(peers) - 1) atomicSub(&sh.h[bin], static_cast<uint32_t>(__popc(peers)));
    }
  }
  __syncthreads();
  {
    // thread t owns bins 2047-8t .. 2040-8t (descending)
    constexpr int kBins = kHistBins / kThreads;
    uint32_t mine = 0;
#pragma unroll
    for (int k = 0; k < kBins; ++k) mine += sh.h[kHistBins - 1 - kBins * tid - k];
    int total;
    uint32_t above = static_cast<uint32_t>(block_exclusive_scan(static_cast<int>(mine), &total, sh.warp_sum));
    const uint32_t topk = static_cast<uint32_t>(p.topk);
#pragma unroll
    for (int k = 0; k < kBins; ++k) {
      const int b = kHistBins - 1 - kBins * tid - k;
      const uint32_t c = sh.h[b];
      if (above < topk && above + c >= topk) {
        sh.bin = b;
        sh.above = static_cast<int>(above);
      }
      above += c;
    }
  }
  __syncthreads();
  const uint32_t bstar = static_cast<uint32_t>(sh.bin);

  // ---- B: classify this CTA's chunk (32 consecutive keys per warp step)
  int my_bits = 0;
  const uint32_t lanemask_lt = (1u << lane) - 1u;
  for (int64_t pass = j0; pass < j1; pass += static_cast<int64_t>(kThreads) * kPer) {
    const int64_t base = pass + warp * 32 * kPer;
    float cur[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int64_t j = base + 32 * k + lane;
      cur[k] = pass == j0 ? pre[k] : (j < j1 ? sel[j] : 0.0f);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int64_t wbase = base + 32 * k;
      if (wbase >= j1) break;
      const int64_t j = wbase + lane;
      bool take = false, maybe = false;
      if (j < j1) {
        if (j >= first_recent) {
          take = true;
        } else {
          const uint32_t b = order_key(cur[k]) >> 21;
          take = b > bstar;
          maybe = b == bstar;
        }
      }
      const uint32_t word = __ballot_sync(0xffffffffu, take);
      if (lane == 0) bitmap[wbase / 32] = word;
      my_bits += lane == 0 ? __popc(word) : 0;
      const uint32_t mb = __ballot_sync(0xffffffffu, maybe);
      if (mb) {
        int pos0 = 0;
        if (lane == 0) pos0 = atomicAdd(&sh.ncand, __popc(mb));
        pos0 = __shfl_sync(0xffffffffu, pos0, 0);
        if (maybe) {
          const int pos = pos0 + __popc(mb & lanemask_lt);
          cand[pos] = static_cast<int32_t>(j);
          if (pos < kLocalCap) sh.local[pos] = select_key(cur[k], j);
        }
      }
    }
  }
  {
    int total;
    block_exclusive_scan(my_bits, &total, sh.warp_sum);
    if (tid == 0) {
      sh.bits = total;
      sh.mine_added = 0;
      for (int c = 0; c < kCl; ++c) sh.added[c] = 0;
    }
  }
  cluster.sync();

  // ---- C: resolve the boundary bin
  int cnts[kCl], m = 0;
  bool spill = false;
#pragma unroll
  for (int c = 0; c < kCl; ++c) {
    cnts[c] = cluster.map_shared_rank(&sh, c)->ncand;
    m += cnts[c];
    spill |= cnts[c] > kLocalCap;
  }
  const bool ranking = !spill && m <= kRankCap;
  if (ranking) {
    // second radix level on the next 8 key bits (bits 45..52 of the 64-bit key)
    const int need = p.topk - sh.above;
    for (int k = tid; k < cnts[rank]; k += kThreads)
      atomicAdd(&sh.dh[(sh.local[k] >> 45) & 0xFFu], 1u);
    cluster.sync();
    {
      // digit 255 - tid: its count over the cluster, then a descending exclusive scan
      const int d = 255 - tid;
      int v = 0;
      if (tid < 256) {
#pragma unroll
        for (int c = 0; c < kCl; ++c) v += static_cast<int>(cluster.map_shared_rank(sh.dh, c)[d]);
      }
      int total;
      const int above = block_exclusive_scan(v, &total, sh.warp_sum);
      if (tid < 256 && above < need && above + v >= need) {
        sh.d2 = d;
        sh.above2 = above;
      }
      __syncthreads();
    }
    const uint64_t d2 = static_cast<uint64_t>(sh.d2);
    const int need2 = need - sh.above2;
    int added = 0;
    for (int k = tid; k < cnts[rank]; k += kThreads) {
      const uint64_t key = sh.local[k];
      const uint64_t dg = (key >> 45) & 0xFFu;
      if (dg > d2) {
        const uint32_t j = 0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull);
        atomicOr(&bitmap[j >> 5], 1u << (j & 31));
        ++added;
      } else if (dg == d2) {
        sh.local2[atomicAdd(&sh.n2, 1)] = key;
      }
    }
    cluster.sync();
    // the keys tied at the boundary digit: rank this CTA's against all of them
    int n2s[kCl], start[kCl], m2 = 0;
#pragma unroll
    for (int c = 0; c < kCl; ++c) {
      n2s[c] = cluster.map_shared_rank(&sh, c)->n2;
      start[c] = m2;
      m2 += n2s[c];
    }
    const bool local_copy = m2 <= kSortCap;
    if (local_copy) {
#pragma unroll
      for (int c = 0; c < kCl; ++c) {
        const uint64_t *list = cluster.map_shared_rank(sh.local2, c);
        for (int i = tid; i < n2s[c]; i += kThreads) sh.keys[start[c] + i] = list[i];
      }
    }
    __syncthreads();
    for (int k = warp; k < n2s[rank]; k += kWarps) {
      const uint64_t key = sh.local2[k];
      int greater = 0;
      if (local_copy) {
        for (int i = lane; i < m2; i += 32) greater += sh.keys[i] > key ? 1 : 0;
      } else {
        // very many ties in the top 19 key bits: compare against the lists in place
#pragma unroll
        for (int c = 0; c < kCl; ++c) {
          const uint64_t *list = cluster.map_shared_rank(sh.local2, c);
          for (int i = lane; i < n2s[c]; i += 32) greater += list[i] > key ? 1 : 0;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) greater += __shfl_xor_sync(0xffffffffu, greater, o);
      if (greater < need2 && lane == 0) {
        const uint32_t j = 0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull);
        atomicOr(&bitmap[j >> 5], 1u << (j & 31));
        ++added;
      }
    }
    if (added) atomicAdd(&sh.mine_added, added);  // every thread may have selected keys
  } else if (rank == 0) {
    // fallback (a crowded bin): the leader resolves every boundary key
    int need = p.topk - sh.above;
    const int32_t *cand_u = p.cand + u * kCl * p.chunk;
    int len = m;
    if (m <= kSortCap) {
      int off = 0;
      for (int c = 0; c < kCl; ++c) {
        for (int i = tid; i < cnts[c]; i += kThreads) {
          const int32_t j = cand_u[c * p.chunk + i];
          sh.keys[off + i] = select_key(sel[j], j);
        }
        off += cnts[c];
      }
      __syncthreads();
    } else {
      // crowded bin: 8-bit radix passes over the 53 key bits below the shared top 11
      int32_t *list = p.bufa + u * kCl * p.chunk;
      int32_t *other = p.bufb + u * kCl * p.chunk;
      int off = 0;
      for (int c = 0; c < kCl; ++c) {
        for (int i = tid; i < cnts[c]; i += kThreads) list[off + i] = cand_u[c * p.chunk + i];
        off += cnts[c];
      }
      __syncthreads();
      int hi = 52;
      while (len > kSortCap && hi >= 0) {
        const int lo = hi >= 7 ? hi - 7 : 0;
        const uint64_t mask = (1ull << (hi - lo + 1)) - 1ull;
        for (int i = tid; i < 256; i += kThreads) sh.dh[i] = 0u;
        if (tid == 0) sh.len = 0;
        __syncthreads();
        for (int i = tid; i < len; i += kThreads) {
          const int32_t j = list[i];
          atomicAdd(&sh.dh[(select_key(sel[j], j) >> lo) & mask], 1u);
        }
        __syncthreads();
        if (tid == 0) {
          uint32_t acc = 0;
          for (int d = 255; d >= 0; --d) {
            if (acc + sh.dh[d] >= static_cast<uint32_t>(need)) {
              sh.dstar = d;
              sh.dabove = static_cast<int>(acc);
              break;
            }
            acc += sh.dh[d];
          }
        }
        __syncthreads();
        const uint64_t dstar = static_cast<uint64_t>(sh.dstar);
        for (int i = tid; i < len; i += kThreads) {
          const int32_t j = list[i];
          const uint64_t d = (select_key(sel[j], j) >> lo) & mask;
          if (d > dstar) {
            atomicOr(&bitmap[j >> 5], 1u << (j & 31));
            atomicAdd(&sh.added[j / p.chunk], 1);
          } else if (d == dstar) {
            other[atomicAdd(&sh.len, 1)] = j;
          }
        }
        __syncthreads();
        need -= sh.dabove;
        len = sh.len;
        int32_t *t = list;
        list = other;
        other = t;
        hi = lo - 1;
        __syncthreads();
      }
      for (int i = tid; i < len; i += kThreads) {
        const int32_t j = list[i];
        sh.keys[i] = select_key(sel[j], j);
      }
      __syncthreads();
    }
    bitonic_desc(sh.keys, len);
    for (int i = tid; i < need; i += kThreads) {
      const uint32_t j = 0xFFFFFFFFu - static_cast<uint32_t>(sh.keys[i] & 0xFFFFFFFFull);
      atomicOr(&bitmap[j >> 5], 1u << (j & 31));
      atomicAdd(&sh.added[j / p.chunk], 1);
    }
  }
  cluster.sync();

  // ---- D: ascending indices
  int before = 0, all = 0;
#pragma unroll
  for (int c = 0; c < kCl; ++c) {
    const Shared *o = cluster.map_shared_rank(&sh, c);
    const int t = o->bits + (ranking ? o->mine_added : cluster.map_shared_rank(&sh, 0)->added[c]);
    before += c < rank ? t : 0;
    all += t;
  }
  const int64_t w0 = j0 / 32, w1 = (j1 + 31) / 32;
  const int64_t nw = w1 - w0;
  // each thread takes a run of consecutive words
  const int64_t per = (nw + kThreads - 1) / kThreads;
  const int64_t lo_w = static_cast<int64_t>(tid) * per, hi_w = static_cast<int64_t>(tid + 1) * per;
  const int64_t a0 = w0 + (lo_w < nw ? lo_w : nw), a1 = w0 + (hi_w < nw ? hi_w : nw);
  int mine = 0;
  for (int64_t w = a0; w < a1; ++w) mine += __popc(bitmap[w]);
  int total;
  int64_t pos = before + block_exclusive_scan(mine, &total, sh.warp_sum);
  for (int64_t w = a0; w < a1; ++w) {
    uint32_t bits = bitmap[w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      if (pos < p.idx_stride) idx[pos] = static_cast<int32_t>(w * 32 + b);
      ++pos;
    }
  }
  if (rank == 0 && tid == 0) p.count[u] = all;
  cluster.sync();  // the leader's shared memory is read by the others above
}


// ----------------------------------------------------------------------------- fast path

constexpr int kFThreads = 512;
constexpr int kFWarps = kFThreads / 32;
constexpr int kFKeys = 32768;               // keys a CTA can hold
#ifndef EMBLA_SEL_CHUNK
#define EMBLA_SEL_CHUNK 8192
#endif
constexpr int kFChunk = EMBLA_SEL_CHUNK;    // keys per CTA aimed for (at most 8 CTAs a unit)
constexpr int kFWords = kFKeys / 32;
constexpr int kRankMax = 256;               // candidates ranked pairwise
constexpr int kMaxCluster = 8;              // CTAs per unit: contexts up to 262144 keys

// Shared memory of a CTA: this struct, then the chunk's scores (turned into order keys in
// place), chunk + 4 entries, sized at launch.
struct __align__(16) FastShared {
  uint32_t sel[kFWords];      // selected
  uint32_t cand[kFWords];     // still undecided (in the boundary bin)
  uint32_t h[kHistBins];
  uint64_t list[kRankMax];    // every candidate of the unit (ranking step)
  uint64_t mine[kRankMax];    // this CTA's candidates
  uint32_t dh[256];           // digit histogram of this CTA's candidates
  int32_t warp_sum[kFWarps];
  int32_t picked[kMaxCluster];  // candidates chosen per CTA of the cluster
  int32_t info_mine[kMaxCluster], info_sel[kMaxCluster], info_off[kMaxCluster + 1];
  int32_t bin, above, ncand, nmine, nsel, dstar, dabove, overflow;
  uint64_t bar;
};
static_assert(sizeof(FastShared) % 16 == 0, "the scores that follow start 16-byte aligned");

struct FastParams {
  const float *sel;
  const uint32_t *hist;
  int64_t n, ncap, chunk;     // chunk: keys per CTA (a multiple of 32)
  int topk, recent, cl;       // cl: CTAs per unit
  int32_t *idx;
  int idx_stride;
  int32_t *count;
  uint32_t *flags;
};

__device__ __forceinline__ int fast_scan(int v, int *total, int32_t *warp_sum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sum[warp] = x;
  __syncthreads();
  const int ws = lane < kFWarps ? warp_sum[lane] : 0;
  int incl = ws;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int before = __shfl_sync(0xffffffffu, incl - ws, warp);
  *total = __shfl_sync(0xffffffffu, incl, kFWarps - 1);
  __syncthreads();
  return before + x - v;
}

__global__ void __launch_bounds__(kFThreads, 1) select_fast_kernel(const FastParams p) {
  pdl_wait_primary();  // the scores and histogram are complete
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t smem_raw[];
  FastShared &sh = *reinterpret_cast<FastShared *>(smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const int cl = p.cl;
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t u = blockIdx.x / cl;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t n = p.n;
  const int64_t j0 = rank * p.chunk;
  const int64_t j1 = min(n, j0 + p.chunk);
  const int nloc = j1 > j0 ? static_cast<int>(j1 - j0) : 0;  // keys of this CTA
  const int nwords = (nloc + 31) >> 5;
  int32_t *idx = p.idx + u * p.idx_stride;

  if (n <= static_cast<int64_t>(p.topk) + p.recent) {
    for (int64_t j = j0 + tid; j < j1; j += kFThreads) idx[j] = static_cast<int32_t>(j);
    if (rank == 0 && tid == 0) p.count[u] = static_cast<int32_t>(n);
    return;
  }
  const float *sel = p.sel + u * p.ncap;
  const int64_t first_recent = n - p.recent;

  // 1: this CTA's scores stream in with one bulk copy (the 16-byte aligned middle; the
  // few keys before and after it load directly) while the histogram, minus the recent
  // keys, gives the boundary bin.  Key k of the chunk sits at entry phase + k, so the
  // copied middle starts on a 16-byte boundary of shared memory as it does in global.
  const uint64_t gbeg = reinterpret_cast<uint64_t>(sel + j0);
  const uint64_t gend = reinterpret_cast<uint64_t>(sel + j1);
  const uint64_t abeg = (gbeg + 15u) & ~15ull, aend = gend & ~15ull;
  const bool bulk = nloc > 0 && aend > abeg;
  const int phase = static_cast<int>((gbeg >> 2) & 3u);
  const int head = bulk ? static_cast<int>((abeg - gbeg) / 4) : nloc;   // keys before it
  const int mid_end = bulk ? static_cast<int>((aend - gbeg) / 4) : nloc;
  uint32_t *okey = reinterpret_cast<uint32_t *>(smem_raw + sizeof(FastShared)) + phase;
  float *sf = reinterpret_cast<float *>(okey);
  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    fence_barrier_init();
    if (bulk) {
      mbar_arrive_expect_tx(&sh.bar, static_cast<uint32_t>(aend - abeg));
      // the shared destination keeps the same 16-byte phase as the source
      bulk_load(sf + head, reinterpret_cast<const void *>(abeg), static_cast<uint32_t>(aend - abeg), &sh.bar);
    }
    sh.ncand = 0;
    sh.nmine = 0;
    sh.nsel = 0;
    sh.overflow = 0;
    sh.bin = kHistBins;  // topk == 0: no bin holds a selected key
    sh.above = 0;
  }
  for (int k = tid; k < head; k += kFThreads) sf[k] = sel[j0 + k];
  for (int k = mid_end + tid; k < nloc; k += kFThreads) sf[k] = sel[j0 + k];
  // the recent keys' scores load together with the histogram (one round trip)
  const bool has_recent = tid < p.recent;
  const float rsig = has_recent ? sel[first_recent + tid] : 0.0f;
  for (int b = tid; b < kHistBins; b += kFThreads) sh.h[b] = p.hist[u * kHistBins + b];
  if (tid < 256) sh.dh[tid] = 0u;
  if (tid < kMaxCluster) sh.picked[tid] = 0;
  __syncthreads();
  if (has_recent) atomicSub(&sh.h[order_key(rsig) >> 21], 1u);
  for (int64_t j = first_recent + kFThreads + tid; j < n; j += kFThreads)
    atomicSub(&sh.h[order_key(sel[j]) >> 21], 1u);
  __syncthreads();
  {
    // thread t owns bins 2047 - 4t .. 2044 - 4t (descending)
    uint32_t c[4], tot = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      c[k] = sh.h[kHistBins - 1 - 4 * tid - k];
      tot += c[k];
    }
    int total;
    uint32_t before = static_cast<uint32_t>(fast_scan(static_cast<int>(tot), &total, sh.warp_sum));
    const uint32_t topk = static_cast<uint32_t>(p.topk);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (before < topk && before + c[k] >= topk) {
        sh.bin = kHistBins - 1 - 4 * tid - k;
        sh.above = static_cast<int>(before);
      }
      before += c[k];
    }
  }
  const bool landed = !bulk || mbar_wait(&sh.bar, 0);
  if (!landed && tid == 0) atomicOr(p.flags, kFlagWaitTimeout);
  __syncthreads();
  const uint32_t bstar = static_cast<uint32_t>(sh.bin);
  int need = p.topk - sh.above;

  // 2: classify, four steps of kFThreads keys at a time; the ballot of warp w in step i
  // is bitmap word 16 i + w
  int nsel = 0;
  for (int base = 0; base < nwords * 32; base += 4 * kFThreads) {
    uint32_t ok[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int jl = base + r * kFThreads + tid;
      ok[r] = jl < nloc ? order_key(sf[jl]) : 0u;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int jl = base + r * kFThreads + tid;
      const int64_t j = j0 + jl;
      const bool valid = jl < nloc && landed;
      if (jl < nloc) okey[jl] = ok[r];  // in place: the same thread read this entry
      const bool recent = valid && j >= first_recent;
      const uint32_t b = ok[r] >> 21;
      const bool take = recent || (valid && b > bstar);
      const bool maybe = valid && !recent && b == bstar;
      const uint32_t wsel = __ballot_sync(0xffffffffu, take);
      const uint32_t wcand = __ballot_sync(0xffffffffu, maybe);
      // one atomic per warp for its candidates' places in the list
      int cbase = 0;
      if (lane == 0) {
        if ((jl >> 5) < kFWords) {
          sh.sel[jl >> 5] = wsel;
          sh.cand[jl >> 5] = wcand;
          nsel += __popc(wsel);
        }
        if (wcand) cbase = atomicAdd(&sh.nmine, __popc(wcand));
      }
      cbase = __shfl_sync(0xffffffffu, cbase, 0);
      if (maybe) {
        const int pos = cbase + __popc(wcand & ((1u << lane) - 1u));
        if (pos < kRankMax) sh.mine[pos] = select_key_ok(ok[r], j);
      }
    }
  }
  if (lane == 0 && nsel) atomicAdd(&sh.nsel, nsel);
  __syncthreads();
  if (tid == 0) {
    sh.ncand = sh.nmine;
    sh.overflow = sh.nmine > kRankMax;
  }
  cluster.sync();
  int m = 0;
  bool overflow = false;
  for (int c = 0; c < cl; ++c) {
    const FastShared *o = cluster.map_shared_rank(&sh, c);
    m += o->ncand;
    overflow |= o->overflow != 0;
  }

  if (m > kRankMax || overflow) {
    // 3a (crowded boundary bin): decide the candidates digit by digit until few are left
    int lo = 53;  // 64-bit key bits [lo, 64) are decided
    while (m > kRankMax && lo > 0) {
      const int nlo = lo >= 8 ? lo - 8 : 0;
      const uint64_t mask = (1ull << (lo - nlo)) - 1ull;
      for (int w = tid; w < nwords; w += kFThreads) {
        uint32_t cw = sh.cand[w];
        while (cw) {
          const int bb = __ffs(cw) - 1;
          cw &= cw - 1u;
          const int jl = 32 * w + bb;
          atomicAdd(&sh.dh[(select_key_ok(okey[jl], j0 + jl) >> nlo) & mask], 1u);
        }
      }
      cluster.sync();
      {
        // thread t < 256: digit 255 - t summed over the cluster; a descending scan finds
        // the digit holding the need-th candidate
        const int d = 255 - tid;
        int v = 0;
        if (tid < 256)
          for (int c = 0; c < cl; ++c) v += static_cast<int>(cluster.map_shared_rank(sh.dh, c)[d]);
        int total;
        const int above = fast_scan(v, &total, sh.warp_sum);
        if (tid < 256 && above < need && above + v >= need) {
          sh.dstar = d;
          sh.dabove = above;
          sh.ncand = v;
        }
      }
      cluster.sync();  // every CTA has read the others' digit counts
      const uint64_t dstar = static_cast<uint64_t>(sh.dstar);
      for (int w = tid; w < nwords; w += kFThreads) {
        uint32_t cw = sh.cand[w], keep = 0u, take = 0u;
        while (cw) {
          const int bb = __ffs(cw) - 1;
          cw &= cw - 1u;
          const int jl = 32 * w + bb;
          const uint64_t d = (select_key_ok(okey[jl], j0 + jl) >> nlo) & mask;
          if (d > dstar) take |= 1u << bb;
          if (d == dstar) keep |= 1u << bb;
        }
        sh.sel[w] |= take;
        sh.cand[w] = keep;
      }
      if (tid < 256) sh.dh[tid] = 0u;
      need -= sh.dabove;
      m = sh.ncand;
      lo = nlo;
      __syncthreads();
    }
    // the selected counts changed: recount, then list the remaining candidates
    int cnt = 0;
    for (int w = tid; w < nwords; w += kFThreads) cnt += __popc(sh.sel[w]);
    int total;
    fast_scan(cnt, &total, sh.warp_sum);
    if (tid == 0) {
      sh.nsel = total;
      sh.nmine = 0;
    }
    __syncthreads();
    for (int w = tid; w < nwords; w += kFThreads) {
      uint32_t cw = sh.cand[w];
      while (cw) {
        const int bb = __ffs(cw) - 1;
        cw &= cw - 1u;
        const int jl = 32 * w + bb;
        const int pos = atomicAdd(&sh.nmine, 1);
        if (pos < kRankMax) sh.mine[pos] = select_key_ok(okey[jl], j0 + jl);
      }
    }
    cluster.sync();
  }

  // 3: every CTA ranks all of the unit's candidates (so it also knows how many of each
  // CTA's are chosen) and marks its own chosen keys.  Remote reads are issued together:
  // thread c reads CTA c's counts, then every thread fetches its share of the lists.
  if (tid < cl) {
    const FastShared *o = cluster.map_shared_rank(&sh, tid);
    sh.info_mine[tid] = min(o->nmine, kRankMax);
    sh.info_sel[tid] = o->nsel;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int c = 0; c < cl; ++c) {
      sh.info_off[c] = acc;
      acc += sh.info_mine[c];
    }
    sh.info_off[cl] = acc;
  }
  __syncthreads();
  const int ml = min(sh.info_off[cl], kRankMax);
  for (int i = tid; i < ml; i += kFThreads) {
    int c = 0;
    while (i >= sh.info_off[c + 1]) ++c;
    sh.list[i] = cluster.map_shared_rank(sh.mine, c)[i - sh.info_off[c]];
  }
  __syncthreads();
  cluster_arrive();  // no more reads of the other CTAs' shared memory
  // T consecutive threads share a key, each comparing it with every T-th entry
  int T = 1;
  while (T < 32 && T * 2 * ml <= kFThreads) T *= 2;
  const int sub = tid & (T - 1);
  const int per_round = kFThreads / T;
  const int rounds = (ml + per_round - 1) / per_round;
  for (int r = 0; r < rounds; ++r) {
    const int k = r * per_round + tid / T;
    const bool real = k < ml;
    const uint64_t key = real ? sh.list[k] : 0ull;
    int greater = 0;
#pragma unroll 4
    for (int i = sub; i < ml; i += T) greater += sh.list[i] > key ? 1 : 0;
    for (int o = 1; o < T; o <<= 1) greater += __shfl_xor_sync(0xffffffffu, greater, o);
    if (real && sub == 0 && greater < need) {
      const int64_t j = 0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull);
      const int owner = static_cast<int>(j / p.chunk);
      atomicAdd(&sh.picked[owner], 1);
      if (owner == rank) {
        const int jl = static_cast<int>(j - j0);
        atomicOr(&sh.sel[jl >> 5], 1u << (jl & 31));
      }
    }
  }
  __syncthreads();

  // 4: ascending indices, after the lower ranks' keys
  int before = 0, all = 0;
  for (int c = 0; c < cl; ++c) {
    const int t = sh.info_sel[c] + sh.picked[c];
    before += c < rank ? t : 0;
    all += t;
  }
  // thread t owns words 2t and 2t + 1
  const uint32_t w0 = 2 * tid < nwords ? sh.sel[2 * tid] : 0u;
  const uint32_t w1 = 2 * tid + 1 < nwords ? sh.sel[2 * tid + 1] : 0u;
  int total;
  const int pre = fast_scan(__popc(w0) + __popc(w1), &total, sh.warp_sum);
  int64_t pos = before + pre;
  uint32_t w = w0;
  for (int half = 0; half < 2; ++half) {
    const int64_t kbase = j0 + 32 * (2 * tid + half);
    while (w) {
      const int bb = __ffs(w) - 1;
      w &= w - 1u;
      if (pos < p.idx_stride) idx[pos] = static_cast<int32_t>(kbase + bb);
      ++pos;
    }
    w = w1;
  }
  if (rank == 0 && tid == 0) p.count[u] = all;
  cluster_wait();  // the others are done reading this CTA's shared memory
}
}  // namespace

size_t select_workspace_bytes(int64_t units, int64_t ctx_len) {
  // contexts the shared-memory path handles need no workspace
  if (ctx_len <= static_cast<int64_t>(kMaxCluster) * kFKeys) return 0;
  return sel_layout(units, ctx_len).total;
}

cudaError_t launch_select(const float *sel_scores, const uint32_t *sel_hist, int64_t units,
                          int64_t n, int64_t ncap, int topk, int recent, int32_t *idx,
                          int idx_stride, int32_t *count, void *workspace, uint32_t *flags,
                          int sm_count, cudaStream_t stream) {
  if (units == 0) return cudaSuccess;
  if (n <= static_cast<int64_t>(kMaxCluster) * kFKeys) {
    // about kFChunk keys per CTA, but no more CTAs than two per SM over all units (one
    // wave), and never more than kFKeys keys in one CTA
    int64_t cl = (n + kFChunk - 1) / kFChunk;
    const int64_t wave = units > 0 ? (2 * static_cast<int64_t>(sm_count)) / units : 1;
    if (cl > wave) cl = wave;
    const int64_t least = (n + kFKeys - 1) / kFKeys;
    if (cl < least) cl = least;
    cl = cl < 1 ? 1 : (cl > kMaxCluster ? kMaxCluster : cl);
    FastParams f;
    f.sel = sel_scores;
    f.hist = sel_hist;
    f.n = n;
    f.ncap = ncap;
    f.topk = topk;
    f.recent = recent;
    f.cl = static_cast<int>(cl);
    f.chunk = ((n + cl - 1) / cl + 31) / 32 * 32;
    f.flags = flags;
    f.idx = idx;
    f.idx_stride = idx_stride;
    f.count = count;
    const int bytes = static_cast<int>(sizeof(FastShared) + (f.chunk + 4) * sizeof(uint32_t));
    cudaError_t e = cudaFuncSetAttribute(select_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sizeof(FastShared) + (kFKeys + 4) * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    return launch_pdl(select_fast_kernel, dim3(static_cast<unsigned>(units * f.cl)), dim3(kFThreads),
                      static_cast<size_t>(bytes), stream, static_cast<unsigned>(f.cl), f);
  }
  const SelLayout L = sel_layout(units, n);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  SelParams p;
  p.sel = sel_scores;
  p.hist = sel_hist;
  p.n = n;
  p.ncap = ncap;
  p.words = L.words;
  p.chunk = L.chunk;
  p.topk = topk;
  p.recent = recent;
  p.bitmap = reinterpret_cast<uint32_t *>(ws + L.bitmap_off);
  p.cand = reinterpret_cast<int32_t *>(ws + L.cand_off);
  p.bufa = reinterpret_cast<int32_t *>(ws + L.bufa_off);
  p.bufb = reinterpret_cast<int32_t *>(ws + L.bufb_off);
  p.idx = idx;
  p.idx_stride = idx_stride;
  p.count = count;
  return launch_pdl(select_kernel, dim3(static_cast<unsigned>(units * kCl)), dim3(kThreads), 0,
                    stream, 0u, p);
}

namespace {

// hist[u][b] = number of keys j < n of unit u whose score's order key has top 11 bits b.
__global__ void __launch_bounds__(512) score_hist_kernel(const float *scores, int64_t n, int64_t ncap,
                                                         uint32_t *hist) {
  pdl_wait_primary();  // the scores are complete
  pdl_launch_dependents();
  __shared__ uint32_t s_h[kHistBins];
  for (int b = threadIdx.x; b < kHistBins; b += blockDim.x) s_h[b] = 0u;
  __syncthreads();
  const int64_t u = blockIdx.x;
  const float *su = scores + u * ncap;
  for (int64_t j = threadIdx.x; j < n; j += blockDim.x) atomicAdd(&s_h[order_key(su[j]) >> 21], 1u);
  __syncthreads();
  for (int b = threadIdx.x; b < kHistBins; b += blockDim.x) hist[u * kHistBins + b] = s_h[b];
}

}  // namespace

cudaError_t launch_score_hist(const float *scores, int64_t units, int64_t n, int64_t ncap,
                              uint32_t *hist, cudaStream_t stream) {
  if (units == 0) return cudaSuccess;
  return launch_pdl(score_hist_kernel, dim3(static_cast<unsigned>(units)), dim3(512), 0, stream, 0u,
                    scores, n, ncap, hist);
}

}  // namespace embla
