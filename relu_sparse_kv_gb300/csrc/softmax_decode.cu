// Softmax decode over a list of cache rows: the sparse layers (rows chosen by the
// selection) and the sliding-window layers (the newest `window` rows of a ring).
//
// Source: "The Architecture of Embla 1", section "Three kinds of attention":
//   Sparse  — the block's full-layer cache restricted to the selected keys, its own
//             softmax, no position encoding;
//   Sliding window — the newest 128 keys, ordinary softmax, rotary position
//             embedding (the query is rotated here; keys were rotated when written).
//
// One warp walks rows; lane l holds dims 4l..4l+3 of every row (a 256-byte row is one
// coalesced warp load).  Eight rows are loaded before any is used so each lane keeps
// sixteen 8-byte loads in flight.  Per head the warp keeps a running max m, a running
// sum l and an unnormalised accumulator; warps and CTAs merge these by rescaling with
// exp(m_i - M).
#include <cmath>

#include "internal.h"
#include "ptx.cuh"

namespace embla {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerSplit = 128;  // sparse decode: selected rows per CTA
constexpr int kBatch = 8;           // rows loaded together per warp

template <int G>
struct SoftState {
  float m[G], l[G], acc[G][4];
  __device__ void init() {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.0f;
      acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.0f;
    }
  }
};

// Fold rows[0..cnt) (row byte offsets into K/V, -1 = skip) into the warp's state.
template <int G>
__device__ __forceinline__ void fold_rows(SoftState<G> &st, const float (&q)[G][4], float tau,
                                          const uint8_t *K, const uint8_t *V,
                                          const int64_t (&off)[kBatch], int cnt, int lane) {
  uint2 kr[kBatch], vr[kBatch];
#pragma unroll
  for (int r = 0; r < kBatch; ++r) {
    if (r < cnt && off[r] >= 0) {
      kr[r] = __ldg(reinterpret_cast<const uint2 *>(K + off[r]) + lane);
      vr[r] = __ldg(reinterpret_cast<const uint2 *>(V + off[r]) + lane);
    } else {
      kr[r] = make_uint2(0u, 0u);
      vr[r] = make_uint2(0u, 0u);
    }
  }
#pragma unroll
  for (int r = 0; r < kBatch; ++r) {
    if (r >= cnt || off[r] < 0) continue;
    const float k0 = bf16lo(kr[r].x), k1 = bf16hi(kr[r].x), k2 = bf16lo(kr[r].y),
                k3 = bf16hi(kr[r].y);
    const float v0 = bf16lo(vr[r].x), v1 = bf16hi(vr[r].x), v2 = bf16lo(vr[r].y),
                v3 = bf16hi(vr[r].y);
    float z[G];
#pragma unroll
    for (int h = 0; h < G; ++h)
      z[h] = fmaf(q[h][0], k0, fmaf(q[h][1], k1, fmaf(q[h][2], k2, q[h][3] * k3)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) z[h] += __shfl_xor_sync(0xffffffffu, z[h], o);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float zz = tau * z[h];
      const float mn = fmaxf(st.m[h], zz);
      const float scale = expf(st.m[h] - mn);  // 0 on the first row (m = -inf)
      const float pz = expf(zz - mn);
      st.m[h] = mn;
      st.l[h] = fmaf(st.l[h], scale, pz);
      st.acc[h][0] = fmaf(st.acc[h][0], scale, pz * v0);
      st.acc[h][1] = fmaf(st.acc[h][1], scale, pz * v1);
      st.acc[h][2] = fmaf(st.acc[h][2], scale, pz * v2);
      st.acc[h][3] = fmaf(st.acc[h][3], scale, pz * v3);
    }
  }
}

// Merge the warps' states of this CTA; warp 0 ends with the CTA's state.
template <int G>
__device__ void merge_warps(SoftState<G> &st, int warp, int lane) {
  __shared__ float s_m[kWarps][G], s_l[kWarps][G];
  __shared__ float s_acc[kWarps][G][kHeadDim];
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      s_m[warp][h] = st.m[h];
      s_l[warp][h] = st.l[h];
    }
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
    *reinterpret_cast<float4 *>(&s_acc[warp][h][lane * 4]) =
        make_float4(st.acc[h][0], st.acc[h][1], st.acc[h][2], st.acc[h][3]);
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w][h]);
      float L = 0.0f, a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float sc = (s_m[w][h] == -INFINITY) ? 0.0f : expf(s_m[w][h] - M);
        L = fmaf(s_l[w][h], sc, L);
        const float4 a = *reinterpret_cast<const float4 *>(&s_acc[w][h][lane * 4]);
        a0 = fmaf(a.x, sc, a0);
        a1 = fmaf(a.y, sc, a1);
        a2 = fmaf(a.z, sc, a2);
        a3 = fmaf(a.w, sc, a3);
      }
      st.m[h] = M;
      st.l[h] = L;
      st.acc[h][0] = a0;
      st.acc[h][1] = a1;
      st.acc[h][2] = a2;
      st.acc[h][3] = a3;
    }
  }
}

template <int G>
__device__ __forceinline__ void load_q(float (&q)[G][4], const uint16_t *qrow, int lane) {
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint2 r = *reinterpret_cast<const uint2 *>(qrow + h * kHeadDim + lane * 4);
    q[h][0] = bf16lo(r.x);
    q[h][1] = bf16hi(r.x);
    q[h][2] = bf16lo(r.y);
    q[h][3] = bf16hi(r.y);
  }
}

// ----------------------------------------------------------------------------- sparse

struct SparseParams {
  const uint16_t *q;
  const uint8_t *K, *V;
  const int32_t *idx, *count;
  float *part;  // [U][S][2G + G*D]
  uint32_t *flags;
  int64_t n, ncap;
  int idx_stride, splits;
  float tau;
};

template <int G>
__global__ void __launch_bounds__(kThreads) sparse_decode_kernel(const SparseParams p) {
  const int64_t u = blockIdx.y;
  const int split = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int cnt = p.count[u];
  cnt = cnt < 0 ? 0 : (cnt > p.idx_stride ? p.idx_stride : cnt);
  float q[G][4];
  load_q<G>(q, p.q + u * G * kHeadDim, lane);
  SoftState<G> st;
  st.init();
  const int32_t *idx = p.idx + u * p.idx_stride;
  const uint8_t *Ku = p.K + u * p.ncap * (kHeadDim * 2);
  const uint8_t *Vu = p.V + u * p.ncap * (kHeadDim * 2);
  const int r0 = split * kRowsPerSplit + warp * (kRowsPerSplit / kWarps);
  const int r1 = min(cnt, r0 + kRowsPerSplit / kWarps);
  for (int rb = r0; rb < r1; rb += kBatch) {
    const int nr = min(kBatch, r1 - rb);
    const int32_t mine = lane < nr ? idx[rb + lane] : 0;
    const bool bad = lane < nr && (mine < 0 || static_cast<int64_t>(mine) >= p.n);
    if (__any_sync(0xffffffffu, bad) && bad) atomicOr(p.flags, kFlagIndexRange);
    int64_t off[kBatch];
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      const int32_t j = __shfl_sync(0xffffffffu, mine, r);
      off[r] = (j < 0 || static_cast<int64_t>(j) >= p.n) ? -1 : static_cast<int64_t>(j) * (kHeadDim * 2);
    }
    fold_rows<G>(st, q, p.tau, Ku, Vu, off, nr, lane);
  }
  merge_warps<G>(st, warp, lane);
  if (warp == 0) {
    float *rec = p.part + (u * p.splits + split) * (2 * G + G * kHeadDim);
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        rec[h] = st.m[h];
        rec[G + h] = st.l[h];
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
      *reinterpret_cast<float4 *>(rec + 2 * G + h * kHeadDim + lane * 4) =
          make_float4(st.acc[h][0], st.acc[h][1], st.acc[h][2], st.acc[h][3]);
  }
}

template <int G>
__global__ void __launch_bounds__(256) sparse_combine_kernel(const float *__restrict__ part,
                                                            int splits, float *__restrict__ out) {
  const int64_t u = blockIdx.x;
  const int stride = 2 * G + G * kHeadDim;
  const float *pu = part + u * splits * stride;
  for (int i = threadIdx.x; i < G * kHeadDim; i += blockDim.x) {
    const int h = i / kHeadDim;
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, pu[s * stride + h]);
    float L = 0.0f, A = 0.0f;
    if (M != -INFINITY) {
      for (int s = 0; s < splits; ++s) {
        const float ms = pu[s * stride + h];
        if (ms == -INFINITY) continue;
        const float sc = expf(ms - M);
        L = fmaf(pu[s * stride + G + h], sc, L);
        A = fmaf(pu[s * stride + 2 * G + i], sc, A);
      }
    }
    out[u * G * kHeadDim + i] = L > 0.0f ? A / L : 0.0f;
  }
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
__global__ void __launch_bounds__(kThreads) window_decode_kernel(const WindowParams p) {
  const int64_t u = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float q[G][4];
  load_q<G>(q, p.q + u * G * kHeadDim, lane);
  // rotate pairs (4l, 4l+1) and (4l+2, 4l+3): pair index i turns by pos * base^(-2i/D);
  // the angle is formed in double so large positions keep their phase
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = 2 * lane + k;
    const double inv = pow(static_cast<double>(p.rope_base), -2.0 * i / kHeadDim);
    double sn, cs;
    sincos(static_cast<double>(p.pos) * inv, &sn, &cs);
    const float c = static_cast<float>(cs), s = static_cast<float>(sn);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float a = q[h][2 * k], b = q[h][2 * k + 1];
      q[h][2 * k] = a * c - b * s;
      q[h][2 * k + 1] = a * s + b * c;
    }
  }
  SoftState<G> st;
  st.init();
  const int64_t first = p.pos - p.window + 1 > 0 ? p.pos - p.window + 1 : 0;
  const int nv = static_cast<int>(p.pos - first + 1);
  const uint8_t *Ku = p.K + u * p.window * (kHeadDim * 2);
  const uint8_t *Vu = p.V + u * p.window * (kHeadDim * 2);
  // warp w takes valid positions w, w+4, w+8, ... (softmax does not depend on order)
  for (int rb = warp; rb < nv; rb += kWarps * kBatch) {
    int64_t off[kBatch];
    int nr = 0;
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
      const int i = rb + r * kWarps;
      if (i < nv) {
        off[r] = ((first + i) % p.window) * (kHeadDim * 2);
        nr = r + 1;
      } else {
        off[r] = -1;
      }
    }
    fold_rows<G>(st, q, p.tau, Ku, Vu, off, nr, lane);
  }
  merge_warps<G>(st, warp, lane);
  if (warp == 0) {
    float *o = p.out + u * G * kHeadDim;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float inv = st.l[h] > 0.0f ? 1.0f / st.l[h] : 0.0f;
      *reinterpret_cast<float4 *>(o + h * kHeadDim + lane * 4) =
          make_float4(st.acc[h][0] * inv, st.acc[h][1] * inv, st.acc[h][2] * inv,
                      st.acc[h][3] * inv);
    }
  }
}

}  // namespace

size_t sparse_workspace_bytes(int64_t units, int G, int idx_stride) {
  const int splits = (idx_stride + kRowsPerSplit - 1) / kRowsPerSplit;
  return static_cast<size_t>(units) * (splits > 0 ? splits : 1) * (2 * G + G * kHeadDim) *
         sizeof(float);
}

cudaError_t launch_sparse_decode(int G, const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *idx, int idx_stride, const int32_t *count,
                                 int64_t units, int Hkv, int64_t n, int64_t ncap, float tau,
                                 float *out, void *workspace, uint32_t *flags,
                                 cudaStream_t stream) {
  (void)Hkv;
  if (units == 0) return cudaSuccess;
  SparseParams p;
  p.q = static_cast<const uint16_t *>(q);
  p.K = static_cast<const uint8_t *>(k_cache);
  p.V = static_cast<const uint8_t *>(v_cache);
  p.idx = idx;
  p.count = count;
  p.part = static_cast<float *>(workspace);
  p.flags = flags;
  p.n = n;
  p.ncap = ncap;
  p.idx_stride = idx_stride;
  p.splits = (idx_stride + kRowsPerSplit - 1) / kRowsPerSplit;
  if (p.splits < 1) p.splits = 1;
  p.tau = tau;
  const dim3 grid(static_cast<unsigned>(p.splits), static_cast<unsigned>(units));
  if (G == 4) {
    sparse_decode_kernel<4><<<grid, kThreads, 0, stream>>>(p);
    sparse_combine_kernel<4><<<static_cast<unsigned>(units), 256, 0, stream>>>(p.part, p.splits, out);
  } else if (G == 8) {
    sparse_decode_kernel<8><<<grid, kThreads, 0, stream>>>(p);
    sparse_combine_kernel<8><<<static_cast<unsigned>(units), 256, 0, stream>>>(p.part, p.splits, out);
  } else {
    return cudaErrorInvalidValue;
  }
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
