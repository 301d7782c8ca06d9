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
// Contexts up to 8 x 65536 keys: a cluster of two to eight CTAs of 1024 threads per (batch,
// KV head) (select_cluster_kernel), each holding up to 32768 scores at a time and its
// selection bitmap in shared memory, or one such CTA (select_single_kernel) for contexts of
// one pass or when a cluster per unit would not fit in one wave (the steps are described
// with the kernels).
//
// Longer contexts (select_kernel): one cluster of 8 CTAs per (batch, KV head), the bitmap
// and candidate lists in the workspace:
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


// Parameters of the cluster path (below).
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

// ----------------------------------------------------------------------------- cluster path
//
// Contexts up to 8 x kUPasses x 32768 keys: a cluster of C (1, 2, 4 or 8) CTAs of 1024
// threads per unit, CTA r owning keys [r chunk, (r + 1) chunk), chunk a multiple of 32.
//   1  a pass's (up to 32768) scores land in shared memory by bulk copies (the 16-byte
//      aligned middle; the few keys before and after it load directly) while the
//      histogram, minus the recent keys, gives the boundary bin b* (every CTA finds it);
//   2  thread t classifies keys 32t .. 32t + 31 of the pass (read in a rotated order, so a
//      warp's reads hit 32 banks), comparing each score as a float against the edges of b*
//      (exact for non-NaN scores): one bitmap word of keys above b* (and recent keys) and
//      one of keys in b*, which are also listed with their 64-bit order keys and counted
//      by their next 8-bit digit;
//   3  after one cluster barrier every CTA reads all CTAs' candidate lists, digit counts
//      and selected counts (distributed shared memory) and narrows the candidates by 8-bit
//      digits of the 64-bit key below the bin until at most 32 are left, which one warp
//      ranks pairwise.  Every CTA reaches the same winners, so each knows how many keys
//      every CTA keeps without a second barrier.  More than kUListMax candidates in b*
//      are first narrowed over the bitmaps, a cluster barrier per digit;
//   4  each CTA writes its keys' indices after those of lower ranks.

constexpr int kUThreads = 1024;
constexpr int kUWarps = kUThreads / 32;
constexpr int kUPassKeys = 32 * kUThreads;    // keys per pass: 32 per thread
#ifndef EMBLA_SEL_UNIT_PASSES
#define EMBLA_SEL_UNIT_PASSES 2
#endif
constexpr int kUPasses = EMBLA_SEL_UNIT_PASSES;  // contexts up to kUPasses x 32768 keys
constexpr int kUWords = kUPasses * kUThreads;    // bitmap words (32 keys each)
constexpr int kUListMax = kUThreads;             // listed candidates: one per thread
#ifndef EMBLA_SEL_BULK_PIECES
#define EMBLA_SEL_BULK_PIECES 16
#endif
constexpr int kUBulkPieces = EMBLA_SEL_BULK_PIECES;

// The float whose order key is k (k the key of a non-NaN float other than -0).
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

constexpr int kUMaxCluster = 8;
#ifndef EMBLA_SEL_CHUNK_TARGET
#define EMBLA_SEL_CHUNK_TARGET 8192
#endif
constexpr int kUChunkTarget = EMBLA_SEL_CHUNK_TARGET;  // keys per CTA aimed for

struct __align__(16) UnitShared {
  uint32_t h[kHistBins];       // recent keys per bin
  uint32_t sel[kUWords];       // selected (this CTA's keys)
  uint32_t cand[kUWords];      // in the boundary bin, undecided (this CTA's keys)
  uint64_t mine[kUListMax];    // this CTA's candidates
  uint64_t list[2][kUListMax]; // the unit's candidates (current, next)
  uint32_t dh[256];            // this CTA's candidates per digit
  uint32_t gdh[256];           // the unit's candidates per digit
  int32_t warp_sum[2][kUWarps];
  int32_t off[kUMaxCluster + 1];  // list offsets of the CTAs' candidates
  int32_t kept[kUMaxCluster];     // keys each CTA keeps (selected + winners)
  int32_t nnext[2];
  int32_t bin, above, nlist, nsure, dstar, dabove, dcount, pad_;
  uint64_t bar;
};
static_assert(sizeof(UnitShared) % 16 == 0, "the scores that follow start 16-byte aligned");

// Exclusive scan of one int per thread over the 1024 threads (one barrier; `ws` must not be
// reused until after the next barrier); sets *total.
__device__ __forceinline__ int unit_scan(int v, int *total, int32_t *ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  const int w = ws[lane];
  int incl = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int before = __shfl_sync(0xffffffffu, incl - w, warp);
  *total = __shfl_sync(0xffffffffu, incl, 31);
  return before + x - v;
}

// One warp: the boundary digit of the 256-bin digit histogram dh (descending) for the need-th
// key; writes dstar, dabove (keys in higher digits) and dcount (keys in it).
__device__ __forceinline__ void unit_digit_boundary(UnitShared &sh, const uint32_t *dh, int need) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8], tot = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    c[k] = dh[255 - 8 * lane - k];  // lane l: digits 255 - 8l .. 248 - 8l
    tot += c[k];
  }
  uint32_t x = tot;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  uint32_t before = x - tot;
  const uint32_t nd = static_cast<uint32_t>(need);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (before < nd && before + c[k] >= nd) {
      sh.dstar = 255 - 8 * lane - k;
      sh.dabove = static_cast<int>(before);
      sh.dcount = static_cast<int>(c[k]);
    }
    before += c[k];
  }
}

// Start loading the scores of keys [0, nloc) from src into sf[k] (sf = buf + the source's
// 16-byte phase): the aligned middle goes as kUBulkPieces bulk copies on `bar` (threads
// 0 .. kUBulkPieces - 1 issue one each, so they are in flight together), every thread loads
// its share of the few keys around it.  *bulk says whether a bulk copy was issued.
__device__ __forceinline__ float *unit_pass_load(float *buf, const float *src, int nloc,
                                                 uint64_t *bar, bool *bulk) {
  const uint64_t gbeg = reinterpret_cast<uint64_t>(src);
  const uint64_t gend = reinterpret_cast<uint64_t>(src + nloc);
  const uint64_t abeg = (gbeg + 15u) & ~15ull, aend = gend & ~15ull;
  *bulk = nloc > 0 && aend > abeg;
  const int phase = static_cast<int>((gbeg >> 2) & 3u);
  const int head = *bulk ? static_cast<int>((abeg - gbeg) / 4) : nloc;
  const int mid_end = *bulk ? static_cast<int>((aend - gbeg) / 4) : nloc;
  float *sf = buf + phase;
  const int t = threadIdx.x;
  if (*bulk) {
    const uint32_t len = static_cast<uint32_t>(aend - abeg);
    // the expected bytes may be posted after some pieces land: the phase also waits for
    // thread 0's arrival, which comes with them
    if (t == 0) mbar_arrive_expect_tx(bar, len);
    const uint32_t piece = ((len + kUBulkPieces - 1) / kUBulkPieces + 15u) & ~15u;
    const uint32_t off = static_cast<uint32_t>(t) * piece;
    if (t < kUBulkPieces && off < len) {
      fence_proxy_async_smem();  // earlier generic reads of the buffer come first
      bulk_load(reinterpret_cast<uint8_t *>(sf + head) + off,
                reinterpret_cast<const uint8_t *>(abeg) + off, min(piece, len - off), bar);
    }
  }
  if (t < head) sf[t] = __ldcg(src + t);
  if (mid_end + t < nloc) sf[mid_end + t] = __ldcg(src + mid_end + t);
  return sf;
}

// Mask of the bits [a, b) of a 32-bit word (0 <= a, b <= 32 after clamping).
__device__ __forceinline__ uint32_t bit_range(int a, int b) {
  a = a < 0 ? 0 : (a > 32 ? 32 : a);
  b = b < 0 ? 0 : (b > 32 ? 32 : b);
  if (b <= a) return 0u;
  const uint32_t hi = b >= 32 ? 0xFFFFFFFFu : ((1u << b) - 1u);
  const uint32_t lo = (1u << a) - 1u;  // a < 32 here
  return hi & ~lo;
}

// Thread t classifies KP = 32 / S keys of bitmap word w = t / S of a pass (part t % S of it):
// keys 32w + KP part + i, read in an order rotated by w so that a warp's reads hit 32 banks.
// Every lane of the word's S lanes ends with the word's masks: scores at or above f_take
// (tm) and those at or above f_lo (cm).
template <int KP>
__device__ __forceinline__ void unit_classify(const float *sf, float f_take, float f_lo,
                                              uint32_t &tm, uint32_t &cm) {
  constexpr int S = 32 / KP;
  const int w = threadIdx.x / S, part = threadIdx.x % S;
  const float *mine = sf + 32 * w + KP * part;
  const int rot = w & (KP - 1);
  uint32_t a = 0u, c = 0u;
#pragma unroll
  for (int k = 0; k < KP; ++k) {
    const float s = mine[(k + rot) & (KP - 1)];
    a |= (s >= f_take ? 1u : 0u) << k;
    c |= (s >= f_lo ? 1u : 0u) << k;
  }
  // bit k belongs to key (k + rot) mod KP
  if constexpr (KP == 32) {
    a = __funnelshift_l(a, a, rot);
    c = __funnelshift_l(c, c, rot);
  } else {
    constexpr uint32_t full = (1u << KP) - 1u;
    a = ((a << rot) | (a >> (KP - rot))) & full;
    c = ((c << rot) | (c >> (KP - rot))) & full;
  }
  a <<= KP * part;
  c <<= KP * part;
#pragma unroll
  for (int o = 1; o < S; o <<= 1) {
    a |= __shfl_xor_sync(0xffffffffu, a, o);
    c |= __shfl_xor_sync(0xffffffffu, c, o);
  }
  tm = a;
  cm = c;
}

// The same masks read four scores per load when the scores start 16-byte aligned in shared
// memory: the thread's KP / 4 chunks in an order rotated by w (a quarter-warp's loads hit
// 32 different banks), each chunk's four compares making a nibble at its place.
template <int KP>
__device__ __forceinline__ void unit_classify4(const float *sf, float f_take, float f_lo,
                                               uint32_t &tm, uint32_t &cm) {
  constexpr int S = 32 / KP, NC = KP / 4;
  const int w = threadIdx.x / S, part = threadIdx.x % S;
  const float4 *mine = reinterpret_cast<const float4 *>(sf + 32 * w + KP * part);
  uint32_t a = 0u, c = 0u;
#pragma unroll
  for (int k = 0; k < NC; ++k) {
    const int ch = (k + w) & (NC - 1);
    const float4 v = mine[ch];
    const uint32_t na = (v.x >= f_take ? 1u : 0u) | (v.y >= f_take ? 2u : 0u) |
                        (v.z >= f_take ? 4u : 0u) | (v.w >= f_take ? 8u : 0u);
    const uint32_t nc = (v.x >= f_lo ? 1u : 0u) | (v.y >= f_lo ? 2u : 0u) |
                        (v.z >= f_lo ? 4u : 0u) | (v.w >= f_lo ? 8u : 0u);
    a |= na << (4 * ch);
    c |= nc << (4 * ch);
  }
  a <<= KP * part;
  c <<= KP * part;
#pragma unroll
  for (int o = 1; o < S; o <<= 1) {
    a |= __shfl_xor_sync(0xffffffffu, a, o);
    c |= __shfl_xor_sync(0xffffffffu, c, o);
  }
  tm = a;
  cm = c;
}

// Either form, for KP keys per thread.
template <int KP>
__device__ __forceinline__ void unit_classify_any(const float *sf, float f_take, float f_lo,
                                                  uint32_t &tm, uint32_t &cm) {
  if ((reinterpret_cast<uintptr_t>(sf) & 15u) == 0u)
    unit_classify4<KP>(sf, f_take, f_lo, tm, cm);
  else
    unit_classify<KP>(sf, f_take, f_lo, tm, cm);
}

// One CTA per unit (contexts up to kUPasses x 32768 keys when a cluster would not fit in
// one wave, and every context of one pass): the steps of the cluster path with every
// exchange a block barrier, the candidates listed and counted by digit straight into the
// unit's list.
__global__ void __launch_bounds__(kUThreads, 1) select_single_kernel(const FastParams p) {
  pdl_wait_primary();  // the scores and histogram are complete
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t smem_raw[];
  UnitShared &sh = *reinterpret_cast<UnitShared *>(smem_raw);
  float *buf = reinterpret_cast<float *>(smem_raw + sizeof(UnitShared));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = blockIdx.x;
  const int n = static_cast<int>(p.n);
  int32_t *idx = p.idx + u * p.idx_stride;
  if (static_cast<int64_t>(n) <= static_cast<int64_t>(p.topk) + p.recent || p.topk == 0) {
    // every key, or (no top-k) just the newest `recent`
    const int j0 = p.topk == 0 && n > p.recent ? n - p.recent : 0;
    for (int j = j0 + tid; j < n; j += kUThreads) idx[j - j0] = j;
    if (tid == 0) p.count[u] = n - j0;
    return;
  }
  const float *sel = p.sel + u * p.ncap;
  const int first_recent = n - p.recent;
  const int npass = (n + kUPassKeys - 1) / kUPassKeys;

  // 1: pass 0's scores stream in while the boundary bin is found.  The histogram (thread t
  // owns bins 2047 - 2t and 2046 - 2t, descending: one 8-byte load) and the recent keys'
  // scores are requested first, so they do not queue behind the bulk copies.
  const uint2 hv = __ldcg(reinterpret_cast<const uint2 *>(p.hist + u * kHistBins) + (1023 - tid));
  const float rs = tid < p.recent ? __ldcg(sel + first_recent + tid) : 0.0f;
  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    fence_barrier_init();
    sh.nlist = 0;
    sh.nnext[0] = 0;
  }
  sh.h[2 * tid] = 0u;
  sh.h[2 * tid + 1] = 0u;
  if (tid < 256) sh.dh[tid] = 0u;
  __syncthreads();
  bool bulk;
  float *sf = unit_pass_load(buf, sel, min(n, kUPassKeys), &sh.bar, &bulk);
  if (tid < p.recent) atomicAdd(&sh.h[order_key(rs) >> 21], 1u);
  for (int t = kUThreads + tid; t < p.recent; t += kUThreads)
    atomicAdd(&sh.h[order_key(__ldcg(sel + first_recent + t)) >> 21], 1u);
  __syncthreads();
  {
    const uint32_t c0 = hv.y - sh.h[kHistBins - 1 - 2 * tid];
    const uint32_t c1 = hv.x - sh.h[kHistBins - 2 - 2 * tid];
    int total;
    const uint32_t before =
        static_cast<uint32_t>(unit_scan(static_cast<int>(c0 + c1), &total, sh.warp_sum[0]));
    const uint32_t topk = static_cast<uint32_t>(p.topk);
    if (before < topk && before + c0 >= topk) {
      sh.bin = kHistBins - 1 - 2 * tid;
      sh.above = static_cast<int>(before);
    } else if (before + c0 < topk && before + c0 + c1 >= topk) {
      sh.bin = kHistBins - 2 - 2 * tid;
      sh.above = static_cast<int>(before + c0);
    }
  }
  __syncthreads();
  // order keys of b* are [b* << 21, (b* + 1) << 21): a score at or above f_take is selected,
  // one at or above f_lo and below f_take is a candidate
  const uint32_t bstar = static_cast<uint32_t>(sh.bin);
  const float f_lo = key_float(bstar << 21);
  const float f_take = bstar + 1 < kHistBins ? key_float((bstar + 1) << 21) : __uint_as_float(0x7FC00000u);
  int need = p.topk - sh.above;

  // 2: classify, one pass of 32768 keys at a time
  bool landed = true;
  uint32_t copies = 0;  // bulk copies waited for (the barrier's phase)
  for (int pass = 0; pass < npass; ++pass) {
    if (pass > 0) {
      __syncthreads();  // every thread is done with the previous pass's scores
      if (landed)
        sf = unit_pass_load(buf, sel + pass * kUPassKeys, min(n - pass * kUPassKeys, kUPassKeys),
                            &sh.bar, &bulk);
      __syncthreads();  // the keys around the bulk copies are stored
    }
    if (landed && bulk && !mbar_wait(&sh.bar, copies++ & 1u)) {
      landed = false;
      if (tid == 0) atomicOr(p.flags, kFlagWaitTimeout);
    }
    const float *mine = sf + 32 * tid;
    uint32_t tm, cm;
    unit_classify_any<32>(sf, f_take, f_lo, tm, cm);
    cm &= ~tm;
    const int k0 = pass * kUPassKeys + 32 * tid;  // this thread's first key
    if (k0 + 32 > first_recent || !landed) {
      const uint32_t valid = landed ? bit_range(0, n - k0) : 0u;
      const uint32_t recent = bit_range(first_recent - k0, n - k0);
      tm = (tm & valid) | recent;
      cm &= valid & ~recent;
    }
    sh.sel[pass * kUThreads + tid] = tm;
    sh.cand[pass * kUThreads + tid] = cm;
    // list the candidates (one shared atomic per warp)
    const int c = __popc(cm);
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    int base = 0;
    if (lane == 31 && x > 0) base = atomicAdd(&sh.nlist, x);
    base = __shfl_sync(0xffffffffu, base, 31) + x - c;
    while (cm) {
      const int b = __ffs(cm) - 1;
      cm &= cm - 1u;
      const uint64_t key = select_key(mine[b], k0 + b);
      atomicAdd(&sh.dh[(key >> 45) & 0xFFu], 1u);  // the first narrowing digit
      if (base < kUListMax) sh.list[0][base] = key;
      ++base;
    }
  }
  __syncthreads();
  int m = sh.nlist;
  int lo = 53;  // bits [lo, 64) of the 64-bit key are decided for the candidates
  const int nwords = npass * kUThreads;
  bool dh_ready = true;  // dh holds every candidate's digit of bits [45, 53)

  if (m > kUListMax) {
    // 3a (crowded boundary bin): decide 8-bit digits over the candidates' bits until the
    // list can hold them, then list them
    while (m > kUListMax && lo > 0) {
      const int nlo = lo >= 8 ? lo - 8 : 0;
      const uint64_t mask = (1ull << (lo - nlo)) - 1ull;
      if (!dh_ready) {
        for (int k = tid; k < nwords; k += kUThreads) {
          uint32_t cw = sh.cand[k];
          while (cw) {
            const int b = __ffs(cw) - 1;
            cw &= cw - 1u;
            const int j = 32 * k + b;
            atomicAdd(&sh.dh[(select_key(__ldcg(sel + j), j) >> nlo) & mask], 1u);
          }
        }
        __syncthreads();
      }
      dh_ready = false;
      if (warp == 0) unit_digit_boundary(sh, sh.dh, need);
      __syncthreads();
      const uint64_t dstar = static_cast<uint64_t>(sh.dstar);
      for (int k = tid; k < nwords; k += kUThreads) {
        uint32_t cw = sh.cand[k], keep = 0u, take = 0u;
        while (cw) {
          const int b = __ffs(cw) - 1;
          cw &= cw - 1u;
          const int j = 32 * k + b;
          const uint64_t d = (select_key(__ldcg(sel + j), j) >> nlo) & mask;
          if (d > dstar) take |= 1u << b;
          if (d == dstar) keep |= 1u << b;
        }
        sh.sel[k] |= take;
        sh.cand[k] = keep;
      }
      need -= sh.dabove;
      m = sh.dcount;
      lo = nlo;
      if (tid < 256) sh.dh[tid] = 0u;
      if (tid == 0) sh.nlist = 0;
      __syncthreads();  // dstar is read by all before the next round rewrites it
    }
    for (int k = tid; k < nwords; k += kUThreads) {
      uint32_t cw = sh.cand[k];
      while (cw) {
        const int b = __ffs(cw) - 1;
        cw &= cw - 1u;
        const int j = 32 * k + b;
        const int pos = atomicAdd(&sh.nlist, 1);
        if (pos < kUListMax) sh.list[0][pos] = select_key(__ldcg(sel + j), j);
      }
    }
    __syncthreads();
    m = min(sh.nlist, kUListMax);
  }

  // 3: narrow the listed candidates digit by digit (one candidate per thread); dh holds the
  // first round's digits or is zero
  int cur = 0;
  while (m > 32 && lo > 0) {
    const int nlo = lo >= 8 ? lo - 8 : 0;
    const uint64_t mask = (1ull << (lo - nlo)) - 1ull;
    const uint64_t key = tid < m ? sh.list[cur][tid] : 0ull;
    const uint32_t dg = static_cast<uint32_t>((key >> nlo) & mask);
    if (tid == 0) sh.nnext[cur ^ 1] = 0;  // last used two rounds ago
    if (!dh_ready) {
      if (tid < m) atomicAdd(&sh.dh[dg], 1u);
      __syncthreads();
    }
    dh_ready = false;
    if (warp == 0) unit_digit_boundary(sh, sh.dh, need);
    __syncthreads();
    const uint32_t dstar = static_cast<uint32_t>(sh.dstar);
    if (tid < m) {
      if (dg > dstar) {
        const int j = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull));
        atomicOr(&sh.sel[j >> 5], 1u << (j & 31));
      } else if (dg == dstar) {
        sh.list[cur ^ 1][atomicAdd(&sh.nnext[cur], 1)] = key;
      }
    }
    need -= sh.dabove;
    m = sh.dcount;
    cur ^= 1;
    lo = nlo;
    if (tid < 256) sh.dh[tid] = 0u;
    __syncthreads();  // the next list is complete; dstar is read by all
  }
  if (warp == 0) {
    // at most 32 left: the need highest of them are selected
    const uint64_t key = lane < m ? sh.list[cur][lane] : 0ull;
    int greater = 0;
    for (int i = 0; i < m; ++i) greater += __shfl_sync(0xffffffffu, key, i) > key ? 1 : 0;
    if (lane < m && greater < need) {
      const int j = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull));
      atomicOr(&sh.sel[j >> 5], 1u << (j & 31));
    }
  }
  __syncthreads();

  // 4: ascending indices; thread t takes words t*npass .. t*npass + npass - 1
  uint32_t wv[kUPasses];
  int mine = 0;
#pragma unroll
  for (int q = 0; q < kUPasses; ++q) {
    wv[q] = q < npass ? sh.sel[tid * npass + q] : 0u;
    mine += __popc(wv[q]);
  }
  int total;
  int pos = unit_scan(mine, &total, sh.warp_sum[1]);
#pragma unroll
  for (int q = 0; q < kUPasses; ++q) {
    uint32_t w = wv[q];
    const int kbase = 32 * (tid * npass + q);
    while (w) {
      const int b = __ffs(w) - 1;
      w &= w - 1u;
      if (pos < p.idx_stride) idx[pos] = kbase + b;
      ++pos;
    }
  }
  if (tid == 0) p.count[u] = total;
}
__global__ void __launch_bounds__(kUThreads, 1) select_cluster_kernel(const FastParams p) {
  pdl_wait_primary();  // the scores and histogram are complete
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t smem_raw[];
  UnitShared &sh = *reinterpret_cast<UnitShared *>(smem_raw);
  float *buf = reinterpret_cast<float *>(smem_raw + sizeof(UnitShared));
  cg::cluster_group cluster = cg::this_cluster();
  const int C = p.cl;
  const int rank = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t u = blockIdx.x / C;
  const int n = static_cast<int>(p.n);
  const int chunk = static_cast<int>(p.chunk);
  const int j0 = min(n, rank * chunk), j1 = min(n, j0 + chunk);  // this CTA's keys
  const int nloc = j1 - j0;
  int32_t *idx = p.idx + u * p.idx_stride;
  if (static_cast<int64_t>(n) <= static_cast<int64_t>(p.topk) + p.recent || p.topk == 0) {
    // every key, or (no top-k) just the newest `recent`
    const int start = p.topk == 0 && n > p.recent ? n - p.recent : 0;
    for (int j = max(start, j0) + tid; j < j1; j += kUThreads) idx[j - start] = j;
    if (rank == 0 && tid == 0) p.count[u] = n - start;
    return;
  }
  const float *sel = p.sel + u * p.ncap;
  const int first_recent = n - p.recent;
  // keys per thread: 8, 16 or 32 (passes of 8192, 16384 or 32768 keys)
  const int kp = nloc <= kUPassKeys / 4 ? 8 : (nloc <= kUPassKeys / 2 ? 16 : 32);
  const int npass = (nloc + kUPassKeys - 1) / kUPassKeys;  // one unless kp is 32
  const int nwords = (nloc + 31) / 32;                   // bitmap words of this CTA
  const int spt = 32 / kp;                               // threads per word

  // 1: pass 0's scores stream in while the boundary bin is found.  The histogram (thread t
  // owns bins 2047 - 2t and 2046 - 2t, descending: one 8-byte load) and the recent keys'
  // scores are requested first, so they do not queue behind the bulk copies.
  const uint2 hv = __ldcg(reinterpret_cast<const uint2 *>(p.hist + u * kHistBins) + (1023 - tid));
  const float rs = tid < p.recent ? __ldcg(sel + first_recent + tid) : 0.0f;
  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    fence_barrier_init();
    sh.nlist = 0;
    sh.nsure = 0;
    sh.nnext[0] = 0;
  }
  sh.h[2 * tid] = 0u;
  sh.h[2 * tid + 1] = 0u;
  if (tid < 256) {
    sh.dh[tid] = 0u;
    sh.gdh[tid] = 0u;
  }
  if (tid < kUMaxCluster) sh.kept[tid] = 0;

  __syncthreads();
  bool bulk;
  float *sf = unit_pass_load(buf, sel + j0, min(nloc, kUPassKeys), &sh.bar, &bulk);
  if (tid < p.recent) atomicAdd(&sh.h[order_key(rs) >> 21], 1u);
  for (int t = kUThreads + tid; t < p.recent; t += kUThreads)
    atomicAdd(&sh.h[order_key(__ldcg(sel + first_recent + t)) >> 21], 1u);
  __syncthreads();
  {
    const uint32_t c0 = hv.y - sh.h[kHistBins - 1 - 2 * tid];
    const uint32_t c1 = hv.x - sh.h[kHistBins - 2 - 2 * tid];
    int total;
    const uint32_t before =
        static_cast<uint32_t>(unit_scan(static_cast<int>(c0 + c1), &total, sh.warp_sum[0]));
    const uint32_t topk = static_cast<uint32_t>(p.topk);
    if (before < topk && before + c0 >= topk) {
      sh.bin = kHistBins - 1 - 2 * tid;
      sh.above = static_cast<int>(before);
    } else if (before + c0 < topk && before + c0 + c1 >= topk) {
      sh.bin = kHistBins - 2 - 2 * tid;
      sh.above = static_cast<int>(before + c0);
    }
  }
  __syncthreads();
  // order keys of b* are [b* << 21, (b* + 1) << 21): a score at or above f_take is selected,
  // one at or above f_lo and below f_take is a candidate
  const uint32_t bstar = static_cast<uint32_t>(sh.bin);
  const float f_lo = key_float(bstar << 21);
  const float f_take = bstar + 1 < kHistBins ? key_float((bstar + 1) << 21) : __uint_as_float(0x7FC00000u);
  int need = p.topk - sh.above;

  // 2: classify, one pass of 32768 keys at a time
  bool landed = true;
  uint32_t copies = 0;  // bulk copies waited for (the barrier's phase)
  int sure = 0;         // keys this thread selected
  for (int pass = 0; pass < npass; ++pass) {
    if (pass > 0) {
      __syncthreads();  // every thread is done with the previous pass's scores
      if (landed)
        sf = unit_pass_load(buf, sel + j0 + pass * kUPassKeys, min(nloc - pass * kUPassKeys, kUPassKeys),
                            &sh.bar, &bulk);
      __syncthreads();  // the keys around the bulk copies are stored
    }
    if (landed && bulk && !mbar_wait(&sh.bar, copies++ & 1u)) {
      landed = false;
      if (tid == 0) atomicOr(p.flags, kFlagWaitTimeout);
    }
    uint32_t tm, cm;
    if (kp == 8)
      unit_classify_any<8>(sf, f_take, f_lo, tm, cm);
    else if (kp == 16)
      unit_classify_any<16>(sf, f_take, f_lo, tm, cm);
    else
      unit_classify_any<32>(sf, f_take, f_lo, tm, cm);
    cm &= ~tm;
    const int wp = tid / spt;                           // the word within the pass
    const int wk = pass * (kUPassKeys / 32) + wp;       // and within this CTA
    const int k0 = j0 + 32 * wk;                        // its first key
    if (k0 + 32 > first_recent || k0 + 32 > j1 || !landed) {
      const uint32_t valid = landed ? bit_range(0, j1 - k0) : 0u;
      const uint32_t recent = bit_range(first_recent - k0, j1 - k0);
      tm = (tm & valid) | recent;
      cm &= valid & ~recent;
    }
    if (tid % spt != 0) tm = cm = 0u;  // one lane of the word keeps it
    if (tid % spt == 0 && wk < nwords) {
      sh.sel[wk] = tm;
      sh.cand[wk] = cm;
    }
    sure += __popc(tm);
    // list the candidates (one shared atomic per warp) and count their next digit
    const int c = __popc(cm);
    int x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    int base = 0;
    if (lane == 31 && x > 0) base = atomicAdd(&sh.nlist, x);
    base = __shfl_sync(0xffffffffu, base, 31) + x - c;
    while (cm) {
      const int b = __ffs(cm) - 1;
      cm &= cm - 1u;
      const uint64_t key = select_key(sf[32 * wp + b], k0 + b);
      atomicAdd(&sh.dh[(key >> 45) & 0xFFu], 1u);  // the first narrowing digit
      if (base < kUListMax) sh.mine[base] = key;
      ++base;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sure += __shfl_xor_sync(0xffffffffu, sure, o);
  if (lane == 0 && sure) atomicAdd(&sh.nsure, sure);
  cluster.sync();  // every CTA's candidates, digit counts and selected counts

  // 3: every CTA's candidate and selected counts, and the unit's first-digit counts
  if (tid < C) {
    const UnitShared *o = cluster.map_shared_rank(&sh, tid);
    sh.off[tid] = o->nlist;
    sh.kept[tid] = o->nsure;
  }
  if (tid < 256) {
    uint32_t v = 0u;
#pragma unroll
    for (int c = 0; c < kUMaxCluster; ++c)
      if (c < C) v += cluster.map_shared_rank(sh.dh, c)[tid];
    sh.gdh[tid] = v;
  }
  __syncthreads();
  int m = 0;
#pragma unroll
  for (int c = 0; c < kUMaxCluster; ++c) m += c < C ? sh.off[c] : 0;
  int lo = 53;            // bits [lo, 64) of the 64-bit key are decided for the candidates
  bool gdh_ready = true;  // gdh counts the unit's candidates by their digit of bits [45, 53)

  if (m > kUListMax) {
    // 3a (crowded boundary bin): decide 8-bit digits over the CTAs' bitmaps, a cluster
    // barrier per digit, until the list can hold the unit's candidates
    while (m > kUListMax && lo > 0) {
      const int nlo = lo >= 8 ? lo - 8 : 0;
      const uint64_t mask = (1ull << (lo - nlo)) - 1ull;
      if (!gdh_ready) {
        for (int k = tid; k < nwords; k += kUThreads) {
          uint32_t cw = sh.cand[k];
          while (cw) {
            const int b = __ffs(cw) - 1;
            cw &= cw - 1u;
            const int j = j0 + 32 * k + b;
            atomicAdd(&sh.dh[(select_key(__ldcg(sel + j), j) >> nlo) & mask], 1u);
          }
        }
        cluster.sync();
        if (tid < 256) {
          uint32_t v = 0u;
#pragma unroll
          for (int c = 0; c < kUMaxCluster; ++c)
            if (c < C) v += cluster.map_shared_rank(sh.dh, c)[tid];
          sh.gdh[tid] = v;
        }
        __syncthreads();
      }
      gdh_ready = false;
      if (warp == 0) unit_digit_boundary(sh, sh.gdh, need);
      __syncthreads();
      const uint64_t dstar = static_cast<uint64_t>(sh.dstar);
      for (int k = tid; k < nwords; k += kUThreads) {
        uint32_t cw = sh.cand[k], keep = 0u, take = 0u;
        while (cw) {
          const int b = __ffs(cw) - 1;
          cw &= cw - 1u;
          const int j = j0 + 32 * k + b;
          const uint64_t d = (select_key(__ldcg(sel + j), j) >> nlo) & mask;
          if (d > dstar) take |= 1u << b;
          if (d == dstar) keep |= 1u << b;
        }
        sh.sel[k] |= take;
        sh.cand[k] = keep;
      }
      need -= sh.dabove;
      m = sh.dcount;
      lo = nlo;
      cluster.sync();  // every CTA has read the others' digit counts
      if (tid < 256) sh.dh[tid] = 0u;
      __syncthreads();
    }
    // list what is left of this CTA's candidates; count its selected keys again
    if (tid == 0) {
      sh.nlist = 0;
      sh.nsure = 0;
    }
    __syncthreads();
    int cnt = 0;
    for (int k = tid; k < nwords; k += kUThreads) {
      cnt += __popc(sh.sel[k]);
      uint32_t cw = sh.cand[k];
      while (cw) {
        const int b = __ffs(cw) - 1;
        cw &= cw - 1u;
        const int j = j0 + 32 * k + b;
        const int pos = atomicAdd(&sh.nlist, 1);
        if (pos < kUListMax) sh.mine[pos] = select_key(__ldcg(sel + j), j);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (lane == 0 && cnt) atomicAdd(&sh.nsure, cnt);
    cluster.sync();
    if (tid < C) {
      const UnitShared *o = cluster.map_shared_rank(&sh, tid);
      sh.off[tid] = o->nlist;
      sh.kept[tid] = o->nsure;
    }
    if (tid < 256) sh.gdh[tid] = 0u;
    __syncthreads();
  }

  // gather the unit's candidates
  int start[kUMaxCluster + 1];
  start[0] = 0;
#pragma unroll
  for (int c = 0; c < kUMaxCluster; ++c) start[c + 1] = start[c] + (c < C ? min(sh.off[c], kUListMax) : 0);
  m = min(start[kUMaxCluster], kUListMax);
  for (int i = tid; i < m; i += kUThreads) {
    int c = 0, sc = 0;
#pragma unroll
    for (int cc = 1; cc < kUMaxCluster; ++cc)
      if (cc < C && i >= start[cc]) {
        c = cc;
        sc = start[cc];
      }
    sh.list[0][i] = cluster.map_shared_rank(sh.mine, c)[i - sc];
  }
  __syncthreads();
  cluster_arrive();  // no more reads of the other CTAs' shared memory

  // 3b: narrow the unit's candidates digit by digit (one candidate per thread; every CTA the
  // same); gdh holds the first round's digits or is zero.  A winner is counted for the CTA
  // that owns it and, if that is this one, marked.
  auto win = [&](uint64_t key) {
    const int j = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull));
    const int owner = j / chunk;
    atomicAdd(&sh.kept[owner], 1);
    if (owner == rank) atomicOr(&sh.sel[(j - j0) >> 5], 1u << ((j - j0) & 31));
  };
  int cur = 0;
  while (m > 32 && lo > 0) {
    const int nlo = lo >= 8 ? lo - 8 : 0;
    const uint64_t mask = (1ull << (lo - nlo)) - 1ull;
    const uint64_t key = tid < m ? sh.list[cur][tid] : 0ull;
    const uint32_t dg = static_cast<uint32_t>((key >> nlo) & mask);
    if (tid == 0) sh.nnext[cur ^ 1] = 0;  // last used two rounds ago
    if (!gdh_ready) {
      if (tid < m) atomicAdd(&sh.gdh[dg], 1u);
      __syncthreads();
    }
    gdh_ready = false;
    if (warp == 0) unit_digit_boundary(sh, sh.gdh, need);
    __syncthreads();
    const uint32_t dstar = static_cast<uint32_t>(sh.dstar);
    if (tid < m) {
      if (dg > dstar)
        win(key);
      else if (dg == dstar)
        sh.list[cur ^ 1][atomicAdd(&sh.nnext[cur], 1)] = key;
    }
    need -= sh.dabove;
    m = sh.dcount;
    cur ^= 1;
    lo = nlo;
    if (tid < 256) sh.gdh[tid] = 0u;
    __syncthreads();  // the next list is complete; dstar is read by all
  }
  if (warp == 0) {
    // at most 32 left: the need highest of them are selected
    const uint64_t key = lane < m ? sh.list[cur][lane] : 0ull;
    int greater = 0;
    for (int i = 0; i < m; ++i) greater += __shfl_sync(0xffffffffu, key, i) > key ? 1 : 0;
    if (lane < m && greater < need) win(key);
  }
  __syncthreads();

  // 4: ascending indices after the lower ranks' keys; thread t takes this CTA's words
  // t*wpt .. t*wpt + wpt - 1
  int before = 0, all = 0;
#pragma unroll
  for (int c = 0; c < kUMaxCluster; ++c) {
    const int k = c < C ? sh.kept[c] : 0;
    before += c < rank ? k : 0;
    all += k;
  }
  const int wpt = (nwords + kUThreads - 1) / kUThreads;  // at most kUPasses
  uint32_t wv[kUPasses];
  int cnt = 0;
#pragma unroll
  for (int q = 0; q < kUPasses; ++q) {
    wv[q] = q < wpt && tid * wpt + q < nwords ? sh.sel[tid * wpt + q] : 0u;
    cnt += __popc(wv[q]);
  }
  int total;
  int pos = before + unit_scan(cnt, &total, sh.warp_sum[1]);
#pragma unroll
  for (int q = 0; q < kUPasses; ++q) {
    uint32_t w = wv[q];
    const int kbase = j0 + 32 * (tid * wpt + q);
    while (w) {
      const int b = __ffs(w) - 1;
      w &= w - 1u;
      if (pos < p.idx_stride) idx[pos] = kbase + b;
      ++pos;
    }
  }
  if (rank == 0 && tid == 0) p.count[u] = all;
  cluster_wait();  // the other CTAs are done reading this one's shared memory
}

}  // namespace

size_t select_workspace_bytes(int64_t units, int64_t ctx_len) {
  // contexts the shared-memory path handles need no workspace
  if (ctx_len <= static_cast<int64_t>(kUMaxCluster) * kUPasses * kUPassKeys) return 0;
  return sel_layout(units, ctx_len).total;
}

cudaError_t launch_select(const float *sel_scores, const uint32_t *sel_hist, int64_t units,
                          int64_t n, int64_t ncap, int topk, int recent, int32_t *idx,
                          int idx_stride, int32_t *count, void *workspace, uint32_t *flags,
                          int sm_count, cudaStream_t stream) {
  if (units == 0) return cudaSuccess;
  if (n <= static_cast<int64_t>(kUMaxCluster) * kUPasses * kUPassKeys) {
    // about kUChunkTarget keys per CTA, but no more CTAs over all units than SMs (one CTA
    // per SM, one wave), and never more than kUPasses x 32768 keys in one CTA
    // (one pass of one CTA is faster than any cluster: its exchanges cost more than they save)
    int64_t want = n <= kUPassKeys ? 1 : (n + kUChunkTarget - 1) / kUChunkTarget;
    const int64_t wave = units > 0 ? static_cast<int64_t>(sm_count) / units : 1;
    if (want > wave) want = wave;
    const int64_t least = (n + kUPasses * kUPassKeys - 1) / (kUPasses * kUPassKeys);
    if (want < least) want = least;
    int cl = 1;
    while (cl < kUMaxCluster && cl < want) cl <<= 1;
    FastParams f = {};
    f.sel = sel_scores;
    f.hist = sel_hist;
    f.n = n;
    f.ncap = ncap;
    f.topk = topk;
    f.recent = recent;
    f.cl = cl;
    f.chunk = ((n + cl - 1) / cl + 31) / 32 * 32;
    f.flags = flags;
    f.idx = idx;
    f.idx_stride = idx_stride;
    f.count = count;
    const int bytes = static_cast<int>(sizeof(UnitShared) + (kUPassKeys + 4) * sizeof(float));
    auto kernel = cl > 1 ? select_cluster_kernel : select_single_kernel;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, dim3(static_cast<unsigned>(units * cl)), dim3(kUThreads),
                      static_cast<size_t>(bytes), stream, cl > 1 ? static_cast<unsigned>(cl) : 0u, f);
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
