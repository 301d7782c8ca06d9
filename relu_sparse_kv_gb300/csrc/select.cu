// Sparse-layer selection: the top-k keys by the full layer's selection score among
// the non-recent keys, plus the `recent` newest keys, in ascending index order.
//
// Source: "The Architecture of Embla 1", section "Three kinds of attention" (Sparse):
// the sparse layers reuse the 1,024 keys the full layer scored highest together with
// the 128 newest, chosen by score whether or not the key survived ReLU^2.
//
// Exact radix select on the order-preserving 32-bit key of each fp32 score, with the
// key index as a tie-break (equal scores: smaller index first), i.e. on the unique
// 64-bit key (order_key(sigma) << 32) | (2^32 - 1 - j):
//   pass 1  (fused into the full-layer decode) histogram of the top 11 bits;
//   scan    every CTA finds the boundary bin from the histogram (minus the recent
//           keys), writes the selection bitmap for keys strictly above it and lists
//           the keys inside it;
//   finish  one CTA per unit resolves the boundary bin exactly (bitonic sort in
//           shared memory, after 8-bit radix passes if the bin is very full), then
//           turns the bitmap into ascending indices.
#include "internal.h"
#include "ptx.cuh"

namespace embla {
namespace {

constexpr int kChunk = 4096;  // keys per scan CTA (a multiple of 32)
constexpr int kScanThreads = 256;
constexpr int kFinishThreads = 1024;
constexpr int kSortCap = 4096;

struct SelLayout {
  int64_t words;    // bitmap words per unit
  int64_t nchunks;  // scan chunks per unit
  size_t bitmap_off, cand_off, cnt_off, thr_off, bufa_off, bufb_off, total;
};

SelLayout sel_layout(int64_t units, int64_t n) {
  SelLayout L;
  L.words = (n + 31) / 32;
  L.nchunks = (n + kChunk - 1) / kChunk;
  const int64_t cand_per_unit = L.nchunks * kChunk;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return o;
  };
  L.bitmap_off = take(static_cast<size_t>(units * L.words) * 4);
  L.cand_off = take(static_cast<size_t>(units * cand_per_unit) * 4);
  L.cnt_off = take(static_cast<size_t>(units * L.nchunks) * 4);
  L.thr_off = take(static_cast<size_t>(units) * 8);
  L.bufa_off = take(static_cast<size_t>(units * cand_per_unit) * 4);
  L.bufb_off = take(static_cast<size_t>(units * cand_per_unit) * 4);
  L.total = off;
  return L;
}

struct SelParams {
  const float *sel;
  const uint32_t *hist;
  int64_t n, ncap, words, nchunks;
  int topk, recent;
  uint32_t *bitmap;
  int32_t *cand;      // [U][nchunks*kChunk]
  int32_t *cand_cnt;  // [U][nchunks]
  int32_t *thr;       // [U][2]: boundary bin, keys above it
  int32_t *bufa, *bufb;
  int32_t *idx;
  int idx_stride;
  int32_t *count;
};

__device__ __forceinline__ uint64_t select_key(float s, int64_t j) {
  return (static_cast<uint64_t>(order_key(s)) << 32) |
         static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(j));
}

__global__ void __launch_bounds__(kScanThreads) select_scan_kernel(const SelParams p) {
  const int64_t u = blockIdx.y;
  const int64_t chunk = blockIdx.x;
  const int64_t n = p.n;
  if (n <= static_cast<int64_t>(p.topk) + p.recent) return;
  __shared__ uint32_t h[kHistBins];
  __shared__ uint32_t s_part[kScanThreads];
  __shared__ int s_bin, s_above, s_cnt;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float *sel = p.sel + u * p.ncap;

  for (int i = tid; i < kHistBins; i += kScanThreads) h[i] = p.hist[u * kHistBins + i];
  if (tid == 0) s_cnt = 0;
  __syncthreads();
  for (int64_t j = n - p.recent + tid; j < n; j += kScanThreads)
    atomicSub(&h[order_key(sel[j]) >> 21], 1u);
  __syncthreads();
  // thread t owns bins 2047-8t .. 2040-8t (descending); exclusive scan over threads
  constexpr int kPer = kHistBins / kScanThreads;
  uint32_t mine = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) mine += h[kHistBins - 1 - kPer * tid - k];
  s_part[tid] = mine;
  __syncthreads();
  for (int o = 1; o < kScanThreads; o <<= 1) {
    const uint32_t v = tid >= o ? s_part[tid - o] : 0u;
    __syncthreads();
    s_part[tid] += v;
    __syncthreads();
  }
  uint32_t above = s_part[tid] - mine;
  const uint32_t topk = static_cast<uint32_t>(p.topk);
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int b = kHistBins - 1 - kPer * tid - k;
    const uint32_t c = h[b];
    if (above < topk && above + c >= topk) {
      s_bin = b;
      s_above = static_cast<int>(above);
    }
    above += c;
  }
  __syncthreads();
  const uint32_t bstar = static_cast<uint32_t>(s_bin);
  if (chunk == 0 && tid == 0) {
    p.thr[u * 2] = s_bin;
    p.thr[u * 2 + 1] = s_above;
  }
  const int64_t j0 = chunk * kChunk;
  const int64_t j1 = min(n, j0 + kChunk);
  const int64_t first_recent = n - p.recent;
  int32_t *cand = p.cand + u * p.nchunks * kChunk + j0;
  const uint32_t lanemask_lt = (1u << lane) - 1u;
  for (int64_t base = j0 + warp * 32; base < j1; base += kScanThreads) {
    const int64_t j = base + lane;
    bool take = false, maybe = false;
    if (j < j1) {
      if (j >= first_recent) {
        take = true;
      } else {
        const uint32_t b = order_key(sel[j]) >> 21;
        take = b > bstar;
        maybe = b == bstar;
      }
    }
    const uint32_t word = __ballot_sync(0xffffffffu, take);
    if (lane == 0) p.bitmap[u * p.words + base / 32] = word;
    const uint32_t mb = __ballot_sync(0xffffffffu, maybe);
    if (mb) {
      int pos0 = 0;
      if (lane == 0) pos0 = atomicAdd(&s_cnt, __popc(mb));
      pos0 = __shfl_sync(0xffffffffu, pos0, 0);
      if (maybe) cand[pos0 + __popc(mb & lanemask_lt)] = static_cast<int32_t>(j);
    }
  }
  __syncthreads();
  if (tid == 0) p.cand_cnt[u * p.nchunks + chunk] = s_cnt;
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

__global__ void __launch_bounds__(kFinishThreads) select_finish_kernel(const SelParams p) {
  const int64_t u = blockIdx.x;
  const int64_t n = p.n;
  const int tid = threadIdx.x;
  int32_t *idx = p.idx + u * p.idx_stride;
  if (n <= static_cast<int64_t>(p.topk) + p.recent) {
    for (int64_t j = tid; j < n; j += kFinishThreads) idx[j] = static_cast<int32_t>(j);
    if (tid == 0) p.count[u] = static_cast<int32_t>(n);
    return;
  }
  __shared__ uint64_t keys[kSortCap];
  __shared__ uint32_t dh[256];
  __shared__ int s_m, s_len, s_dstar, s_above;
  __shared__ uint32_t s_part[kFinishThreads];
  const float *sel = p.sel + u * p.ncap;
  uint32_t *bitmap = p.bitmap + u * p.words;
  const int32_t *cand = p.cand + u * p.nchunks * kChunk;
  const int32_t *cnt = p.cand_cnt + u * p.nchunks;
  int need = p.topk - p.thr[u * 2 + 1];

  if (tid == 0) {
    int m = 0;
    for (int64_t c = 0; c < p.nchunks; ++c) m += cnt[c];
    s_m = m;
  }
  __syncthreads();
  const int m = s_m;
  const bool small = m <= kSortCap;
  // gather the boundary-bin candidates: into shared keys when few, else into bufa
  int32_t *list = p.bufa + u * p.nchunks * kChunk;
  int32_t *other = p.bufb + u * p.nchunks * kChunk;
  {
    int off = 0;
    for (int64_t c = 0; c < p.nchunks; ++c) {
      const int cc = cnt[c];
      for (int i = tid; i < cc; i += kFinishThreads) {
        const int32_t j = cand[c * kChunk + i];
        if (small)
          keys[off + i] = select_key(sel[j], j);
        else
          list[off + i] = j;
      }
      off += cc;
    }
  }
  __syncthreads();
  int len = m;
  if (!small) {
    // 8-bit radix passes over the 53 key bits below the shared top 11 bits
    int hi = 52;
    while (len > kSortCap && hi >= 0) {
      const int lo = hi >= 7 ? hi - 7 : 0;
      const uint64_t mask = (1ull << (hi - lo + 1)) - 1ull;
      for (int i = tid; i < 256; i += kFinishThreads) dh[i] = 0u;
      if (tid == 0) s_len = 0;
      __syncthreads();
      for (int i = tid; i < len; i += kFinishThreads) {
        const int32_t j = list[i];
        atomicAdd(&dh[(select_key(sel[j], j) >> lo) & mask], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t acc = 0;
        for (int d = 255; d >= 0; --d) {
          if (acc + dh[d] >= static_cast<uint32_t>(need)) {
            s_dstar = d;
            s_above = static_cast<int>(acc);
            break;
          }
          acc += dh[d];
        }
      }
      __syncthreads();
      const uint64_t dstar = static_cast<uint64_t>(s_dstar);
      for (int i = tid; i < len; i += kFinishThreads) {
        const int32_t j = list[i];
        const uint64_t d = (select_key(sel[j], j) >> lo) & mask;
        if (d > dstar) {
          atomicOr(&bitmap[j >> 5], 1u << (j & 31));
        } else if (d == dstar) {
          other[atomicAdd(&s_len, 1)] = j;
        }
      }
      __syncthreads();
      need -= s_above;
      len = s_len;
      int32_t *t = list;
      list = other;
      other = t;
      hi = lo - 1;
      __syncthreads();
    }
    for (int i = tid; i < len; i += kFinishThreads) {
      const int32_t j = list[i];
      keys[i] = select_key(sel[j], j);
    }
    __syncthreads();
  }
  bitonic_desc(keys, len);
  for (int i = tid; i < need; i += kFinishThreads) {
    const uint32_t j = 0xFFFFFFFFu - static_cast<uint32_t>(keys[i] & 0xFFFFFFFFull);
    atomicOr(&bitmap[j >> 5], 1u << (j & 31));
  }
  __syncthreads();
  // bitmap -> ascending indices
  const int64_t W = p.words;
  const int64_t w0 = (W * tid) / kFinishThreads, w1 = (W * (tid + 1)) / kFinishThreads;
  uint32_t mine = 0;
  for (int64_t w = w0; w < w1; ++w) mine += __popc(bitmap[w]);
  s_part[tid] = mine;
  __syncthreads();
  for (int o = 1; o < kFinishThreads; o <<= 1) {
    const uint32_t v = tid >= o ? s_part[tid - o] : 0u;
    __syncthreads();
    s_part[tid] += v;
    __syncthreads();
  }
  int64_t pos = s_part[tid] - mine;
  for (int64_t w = w0; w < w1; ++w) {
    uint32_t bits = bitmap[w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      if (pos < p.idx_stride) idx[pos] = static_cast<int32_t>(w * 32 + b);
      ++pos;
    }
  }
  if (tid == kFinishThreads - 1) p.count[u] = static_cast<int32_t>(s_part[tid]);
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
  p.nchunks = L.nchunks;
  p.topk = topk;
  p.recent = recent;
  p.bitmap = reinterpret_cast<uint32_t *>(ws + L.bitmap_off);
  p.cand = reinterpret_cast<int32_t *>(ws + L.cand_off);
  p.cand_cnt = reinterpret_cast<int32_t *>(ws + L.cnt_off);
  p.thr = reinterpret_cast<int32_t *>(ws + L.thr_off);
  p.bufa = reinterpret_cast<int32_t *>(ws + L.bufa_off);
  p.bufb = reinterpret_cast<int32_t *>(ws + L.bufb_off);
  p.idx = idx;
  p.idx_stride = idx_stride;
  p.count = count;
  if (n > static_cast<int64_t>(topk) + recent) {
    const dim3 grid(static_cast<unsigned>(L.nchunks), static_cast<unsigned>(units));
    select_scan_kernel<<<grid, kScanThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  select_finish_kernel<<<static_cast<unsigned>(units), kFinishThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace embla
