// Softmax decode over a list of cache rows: the sparse layers (rows chosen by the
// selection) and the sliding-window layers (the newest `window` rows of a ring).
//
// Source: "The Architecture of Embla 1", section "Three kinds of attention":
//   Sparse  — the block's full-layer cache restricted to the selected keys, its own
//             softmax, no position encoding;
//   Sliding window — the newest 128 keys, ordinary softmax, rotary position
//             embedding (the query is rotated here; keys were rotated when written).
//
// Each warp folds chunks of 8 rows; a row is read by 16 lanes (8 dims each, one
// 16-byte load of K and of V), so a warp's two lane groups take 4 rows each.  The
// group's 4 x G partial dot products are summed by a reduce-scatter over its 16 lanes
// and gathered back, then every lane updates its group's running max m, sum l and its
// 8-dim slice of the unnormalised output, rescaling once per chunk.  Warps merge in shared memory by rescaling with exp(m_w - M).
// A sparse layer spreads each (batch, KV-head) unit over a cluster of 8 CTAs that merge
// through distributed shared memory; a window layer uses one CTA per unit.
#include <cooperative_groups.h>

#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace embla {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kCluster = 8;        // CTAs per sparse unit
constexpr int kIdxChunk = 512;     // selected rows a sparse CTA stages at a time
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRowBytes = kHeadDim * 2;

// Lane layout of a warp: two groups of 16 lanes; lane sl of a group holds dims
// 8*sl .. 8*sl+7 of a row (one 16-byte load of K and one of V).  A chunk is 8 rows:
// group 0 takes rows 0-3, group 1 rows 4-7.  Each group keeps its own running state
// (the two are merged with the other warps at the end).
constexpr int kChunk = 8;

template <int G>
struct Soft {
  float m[G], l[G], acc[G][8];
  __device__ void init() {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;
#pragma unroll
      for (int d = 0; d < 8; ++d) acc[h][d] = 0.0f;
    }
  }
};

struct Chunk {
  uint4 k[4], v[4];
  uint32_t present;  // bit r: row r of this lane's group exists
};

// rows[r]: row index of K/V for this lane's group's row r, or -1
__device__ __forceinline__ void load_chunk(Chunk &c, const uint8_t *K, const uint8_t *V,
                                           const int32_t (&rows)[4], int sl) {
  c.present = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    if (rows[r] >= 0) {
      const int64_t off = static_cast<int64_t>(rows[r]) * kRowBytes;
      c.k[r] = __ldg(reinterpret_cast<const uint4 *>(K + off) + sl);
      c.v[r] = __ldg(reinterpret_cast<const uint4 *>(V + off) + sl);
      c.present |= 1u << r;
    } else {
      c.k[r] = make_uint4(0u, 0u, 0u, 0u);
      c.v[r] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// acc += a . b over the 8 bf16 pairs of two uint4 (bf16 products are exact in fp32)
__device__ __forceinline__ float dot8_bf16(const uint4 &a, const uint4 &b) {
  float s0 = 0.0f, s1 = 0.0f;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\tmov.b32 {bl, bh}, %6;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %1, ah, bh, %1;\n\t"
      "mov.b32 {al, ah}, %3;\n\tmov.b32 {bl, bh}, %7;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %1, ah, bh, %1;\n\t"
      "mov.b32 {al, ah}, %4;\n\tmov.b32 {bl, bh}, %8;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %1, ah, bh, %1;\n\t"
      "mov.b32 {al, ah}, %5;\n\tmov.b32 {bl, bh}, %9;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %0;\n\tfma.rn.f32.bf16 %1, ah, bh, %1;\n\t}"
      : "+f"(s0), "+f"(s1)
      : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w));
  return s0 + s1;
}

// Fold one chunk into the group's running softmax state.  Scores are kept in base 2:
// tau2 = tau * log2(e), so exp(tau * s - m) = exp2(tau2 * s - m2).
template <int G, class Dots>
__device__ __forceinline__ void fold_chunk(Soft<G> &st, const Dots &dots, float tau2,
                                           const Chunk &c, int sl) {
  constexpr int NV = 4 * G;    // values r*G + h of this lane's group
  constexpr int R = NV / 16;   // values per lane after the reduce-scatter
  float v[NV];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    float d[G];
    dots(c.k[r], d);
#pragma unroll
    for (int h = 0; h < G; ++h) v[r * G + h] = d[h];
  }
  // reduce-scatter over the 16 lanes of the group (offsets 8, 4, 2, 1 stay in the group)
#pragma unroll
  for (int o = 8, half = NV / 2; o >= 1; o >>= 1, half >>= 1) {
    const bool upper = (sl & o) != 0;
#pragma unroll
    for (int k = 0; k < half; ++k) {
      const float send = upper ? v[k] : v[k + half];
      const float keep = upper ? v[k + half] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  // lane sl holds values sl*R .. sl*R+R-1; gather the group's 4 x G scores to every lane
  const int gbase = (threadIdx.x & 31) & 16;
  float z[4][G];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int i = r * G + h;
      const float s = __shfl_sync(0xffffffffu, v[i % R], gbase + i / R);
      z[r][h] = (c.present >> r) & 1u ? tau2 * s : -INFINITY;
    }
  float vv[4][8];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    vv[r][0] = bf16lo(c.v[r].x); vv[r][1] = bf16hi(c.v[r].x);
    vv[r][2] = bf16lo(c.v[r].y); vv[r][3] = bf16hi(c.v[r].y);
    vv[r][4] = bf16lo(c.v[r].z); vv[r][5] = bf16hi(c.v[r].z);
    vv[r][6] = bf16lo(c.v[r].w); vv[r][7] = bf16hi(c.v[r].w);
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float bm = fmaxf(fmaxf(z[0][h], z[1][h]), fmaxf(z[2][h], z[3][h]));
    const float mn = fmaxf(st.m[h], bm);
    if (mn == -INFINITY) continue;          // nothing seen yet and no row in this chunk
    const float sc = exp2f(st.m[h] - mn);  // 0 while nothing has been seen
    float p[4], sum = 0.0f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      p[r] = exp2f(z[r][h] - mn);          // 0 for absent rows
      sum += p[r];
    }
    st.m[h] = mn;
    st.l[h] = fmaf(st.l[h], sc, sum);
#pragma unroll
    for (int d = 0; d < 8; ++d) {
      float a = st.acc[h][d] * sc;
#pragma unroll
      for (int r = 0; r < 4; ++r) a = fmaf(p[r], vv[r][d], a);
      st.acc[h][d] = a;
    }
  }
}

template <int G>
struct Merge {
  float m[kWarps][G], l[kWarps][G];
  float acc[kWarps][G][kHeadDim];
  float cm[G], cl[G];          // the CTA's merged state
  float ca[G][kHeadDim];
};

// Merge the warps' states (two groups per warp) into the CTA state (cm, cl, ca); ends
// with __syncthreads.
template <int G>
__device__ void merge_warps(Merge<G> &mg, Soft<G> &st, int warp, int lane) {
  // the two lane groups first: lane sl and lane sl+16 hold the same dims
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float m2 = __shfl_xor_sync(0xffffffffu, st.m[h], 16);
    const float l2 = __shfl_xor_sync(0xffffffffu, st.l[h], 16);
    const float M = fmaxf(st.m[h], m2);
    const float s1 = M == -INFINITY ? 0.0f : exp2f(st.m[h] - M);
    const float s2 = M == -INFINITY ? 0.0f : exp2f(m2 - M);
    st.m[h] = M;
    st.l[h] = st.l[h] * s1 + l2 * s2;
#pragma unroll
    for (int d = 0; d < 8; ++d) {
      const float a2 = __shfl_xor_sync(0xffffffffu, st.acc[h][d], 16);
      st.acc[h][d] = st.acc[h][d] * s1 + a2 * s2;
    }
  }
  const int sl = lane & 15;
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      mg.m[warp][h] = st.m[h];
      mg.l[warp][h] = st.l[h];
    }
  }
  if (lane < 16) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      *reinterpret_cast<float4 *>(&mg.acc[warp][h][sl * 8]) =
          make_float4(st.acc[h][0], st.acc[h][1], st.acc[h][2], st.acc[h][3]);
      *reinterpret_cast<float4 *>(&mg.acc[warp][h][sl * 8 + 4]) =
          make_float4(st.acc[h][4], st.acc[h][5], st.acc[h][6], st.acc[h][7]);
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * kHeadDim; i += kThreads) {
    const int h = i / kHeadDim, d = i % kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mg.m[w][h]);
    float L = 0.0f, A = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float sc = exp2f(mg.m[w][h] - M);
        L = fmaf(mg.l[w][h], sc, L);
        A = fmaf(mg.acc[w][h][d], sc, A);
      }
    }
    mg.ca[h][d] = A;
    if (d == 0) {
      mg.cm[h] = M;
      mg.cl[h] = L;
    }
  }
  __syncthreads();
}

// Partial dot products of this lane's 8 dims of a key row with every head's query.
// Sparse layers use the raw bf16 query (exact bf16 products, fp32 sums).
template <int G>
struct DotsBf16 {
  uint4 q[G];
  __device__ void load(const uint16_t *qrow, int sl) {
#pragma unroll
    for (int h = 0; h < G; ++h) q[h] = *reinterpret_cast<const uint4 *>(qrow + h * kHeadDim + sl * 8);
  }
  __device__ __forceinline__ void operator()(const uint4 &k, float (&d)[G]) const {
#pragma unroll
    for (int h = 0; h < G; ++h) d[h] = dot8_bf16(q[h], k);
  }
};

// Window layers use the rotated query, kept in fp32.
template <int G>
struct DotsF32 {
  float q[G][8];
  __device__ __forceinline__ void operator()(const uint4 &k, float (&d)[G]) const {
    const float k0 = bf16lo(k.x), k1 = bf16hi(k.x), k2 = bf16lo(k.y), k3 = bf16hi(k.y),
                k4 = bf16lo(k.z), k5 = bf16hi(k.z), k6 = bf16lo(k.w), k7 = bf16hi(k.w);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float a = q[h][0] * k0;
      float b = q[h][1] * k1;
      a = fmaf(q[h][2], k2, a);
      b = fmaf(q[h][3], k3, b);
      a = fmaf(q[h][4], k4, a);
      b = fmaf(q[h][5], k5, b);
      a = fmaf(q[h][6], k6, a);
      b = fmaf(q[h][7], k7, b);
      d[h] = a + b;
    }
  }
};


// ----------------------------------------------------------------------------- sparse

struct SparseParams {
  const uint16_t *q;
  const uint8_t *K, *V;
  const int32_t *idx, *count;
  float *out;
  uint32_t *flags;
  int64_t n, ncap;
  int idx_stride, rows_per_cta;
  float tau;
};

template <int G>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads, 2)
    sparse_decode_kernel(const SparseParams p) {
  __shared__ Merge<G> mg;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t u = blockIdx.x / kCluster;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int cnt = p.count[u];
  cnt = cnt < 0 ? 0 : (cnt > p.idx_stride ? p.idx_stride : cnt);
  const int grp = lane >> 4, sl = lane & 15;
  DotsBf16<G> dots;
  dots.load(p.q + u * G * kHeadDim, sl);
  Soft<G> st;
  st.init();
  const int32_t *idx = p.idx + u * p.idx_stride;
  const uint8_t *Ku = p.K + u * p.ncap * kRowBytes;
  const uint8_t *Vu = p.V + u * p.ncap * kRowBytes;
  __shared__ int32_t s_rows[kIdxChunk];
  const float tau2 = p.tau * kLog2e;
  const int r0 = rank * p.rows_per_cta;
  const int r1 = min(cnt, r0 + p.rows_per_cta);
  for (int c0 = r0; c0 < r1; c0 += kIdxChunk) {
    const int c1 = min(r1, c0 + kIdxChunk);
    // one round trip for the chunk's indices; out-of-range entries are skipped and flagged
    for (int r = c0 + threadIdx.x; r < c1; r += kThreads) {
      const int32_t j = idx[r];
      const bool bad = j < 0 || static_cast<int64_t>(j) >= p.n;
      if (bad) atomicOr(p.flags, kFlagIndexRange);
      s_rows[r - c0] = bad ? -1 : j;
    }
    __syncthreads();
    for (int cb = c0 + warp * kChunk; cb < c1; cb += kWarps * kChunk) {
      int32_t rows[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int i = cb + grp * 4 + r;
        rows[r] = i < c1 ? s_rows[i - c0] : -1;
      }
      Chunk ch;
      load_chunk(ch, Ku, Vu, rows, sl);
      fold_chunk<G>(st, dots, tau2, ch, sl);
    }
    __syncthreads();
  }
  merge_warps<G>(mg, st, warp, lane);
  cluster.sync();
  if (rank == 0) {
    for (int i = threadIdx.x; i < G * kHeadDim; i += kThreads) {
      const int h = i / kHeadDim, d = i % kHeadDim;
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < kCluster; ++c) M = fmaxf(M, cluster.map_shared_rank(&mg, c)->cm[h]);
      float L = 0.0f, A = 0.0f;
      if (M != -INFINITY) {
#pragma unroll
        for (int c = 0; c < kCluster; ++c) {
          const Merge<G> *o = cluster.map_shared_rank(&mg, c);
          const float sc = exp2f(o->cm[h] - M);
          L = fmaf(o->cl[h], sc, L);
          A = fmaf(o->ca[h][d], sc, A);
        }
      }
      p.out[u * G * kHeadDim + i] = L > 0.0f ? A / L : 0.0f;
    }
  }
  cluster.sync();  // the other CTAs' shared memory stays alive until the leader is done
}

// ----------------------------------------------------------------------------- window

struct WindowParams {
  const uint16_t *q;
  const uint8_t *K, *V;
  float *out;
  int64_t pos;
  int window;
  float rope_base, tau;
};

template <int G>
__global__ void __launch_bounds__(kThreads, 2) window_decode_kernel(const WindowParams p) {
  __shared__ Merge<G> mg;
  const int64_t u = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 4, sl = lane & 15;
  DotsF32<G> dots;
  // this lane's dims 8sl..8sl+7 are rotary pairs 4sl..4sl+3; pair i turns by
  // pos * base^(-2i/D), the angle formed in double so large positions keep their phase
  {
    const uint16_t *qrow = p.q + u * G * kHeadDim + sl * 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = 4 * sl + k;
      const double inv = pow(static_cast<double>(p.rope_base), -2.0 * i / kHeadDim);
      double sn, cs;
      sincos(static_cast<double>(p.pos) * inv, &sn, &cs);
      const float c = static_cast<float>(cs), s = static_cast<float>(sn);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(qrow + h * kHeadDim + 2 * k);
        const float a = bf16lo(w), b = bf16hi(w);
        dots.q[h][2 * k] = a * c - b * s;
        dots.q[h][2 * k + 1] = a * s + b * c;
      }
    }
  }
  Soft<G> st;
  st.init();
  const int64_t first = p.pos - p.window + 1 > 0 ? p.pos - p.window + 1 : 0;
  const int nv = static_cast<int>(p.pos - first + 1);
  const uint8_t *Ku = p.K + u * p.window * kRowBytes;
  const uint8_t *Vu = p.V + u * p.window * kRowBytes;
  const float tau2 = p.tau * kLog2e;
  for (int cb = warp * kChunk; cb < nv; cb += kWarps * kChunk) {
    int32_t rows[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = cb + grp * 4 + r;
      rows[r] = i < nv ? static_cast<int32_t>((first + i) % p.window) : -1;
    }
    Chunk ch;
    load_chunk(ch, Ku, Vu, rows, sl);
    fold_chunk<G>(st, dots, tau2, ch, sl);
  }
  merge_warps<G>(mg, st, warp, lane);
  for (int i = threadIdx.x; i < G * kHeadDim; i += kThreads) {
    const int h = i / kHeadDim;
    p.out[u * G * kHeadDim + i] = mg.cl[h] > 0.0f ? mg.ca[h][i % kHeadDim] / mg.cl[h] : 0.0f;
  }
}

}  // namespace

size_t sparse_workspace_bytes(int64_t units, int G, int idx_stride) {
  (void)units;
  (void)G;
  (void)idx_stride;
  return 0;
}

cudaError_t launch_sparse_decode(int G, const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *idx, int idx_stride, const int32_t *count,
                                 int64_t units, int Hkv, int64_t n, int64_t ncap, float tau,
                                 float *out, void *workspace, uint32_t *flags,
                                 cudaStream_t stream) {
  (void)Hkv;
  (void)workspace;
  if (units == 0) return cudaSuccess;
  SparseParams p;
  p.q = static_cast<const uint16_t *>(q);
  p.K = static_cast<const uint8_t *>(k_cache);
  p.V = static_cast<const uint8_t *>(v_cache);
  p.idx = idx;
  p.count = count;
  p.out = out;
  p.flags = flags;
  p.n = n;
  p.ncap = ncap;
  p.idx_stride = idx_stride;
  p.rows_per_cta = (idx_stride + kCluster - 1) / kCluster;
  p.tau = tau;
  const dim3 grid(static_cast<unsigned>(units * kCluster));
  if (G == 4)
    sparse_decode_kernel<4><<<grid, kThreads, 0, stream>>>(p);
  else if (G == 8)
    sparse_decode_kernel<8><<<grid, kThreads, 0, stream>>>(p);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_window_decode(int G, const void *q, const void *k_win, const void *v_win,
                                 int64_t units, int window, int64_t pos, float rope_base,
                                 float tau, float *out, cudaStream_t stream) {
  if (units == 0) return cudaSuccess;
  WindowParams p;
  p.q = static_cast<const uint16_t *>(q);
  p.K = static_cast<const uint8_t *>(k_win);
  p.V = static_cast<const uint8_t *>(v_win);
  p.out = out;
  p.pos = pos;
  p.window = window;
  p.rope_base = rope_base;
  p.tau = tau;
  if (G == 4)
    window_decode_kernel<4><<<static_cast<unsigned>(units), kThreads, 0, stream>>>(p);
  else if (G == 8)
    window_decode_kernel<8><<<static_cast<unsigned>(units), kThreads, 0, stream>>>(p);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace embla
