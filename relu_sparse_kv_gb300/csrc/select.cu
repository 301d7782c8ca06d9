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
// histogrammed by the full-layer decode.  One cluster of 8 CTAs per (batch, KV head):
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

}  // namespace

size_t select_workspace_bytes(int64_t units, int64_t ctx_len) {
  return sel_layout(units, ctx_len).total;
}

cudaError_t launch_select(const float *sel_scores, const uint32_t *sel_hist, int64_t units,
                          int64_t n, int64_t ncap, int topk, int recent, int32_t *idx,
                          int idx_stride, int32_t *count, void *workspace, cudaStream_t stream) {
  if (units == 0) return cudaSuccess;
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
  select_kernel<<<static_cast<unsigned>(units * kCl), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace embla
