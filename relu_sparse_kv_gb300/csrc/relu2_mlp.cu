// ReLU^2 MLP of one token, reading only the down-projection rows of neurons that fired.
//
// Source: "The Architecture of Embla 1", section "ReLU^2 activation": a negative
// pre-activation becomes zero and a positive one is squared; a zero neuron's row of the
// down projection contributes nothing, so at batch size 1 a kernel reads only the rows of
// the neurons that fired.
//
// relu2_mlp_kernel: one CTA per SM over a contiguous range of neurons, 16 warps.
//   phase 1  each warp takes neurons in turn, two rows in flight: h_i = max(w_up_i . x, 0)^2
//            with exact bf16 products summed in fp32 (the token x stays in registers);
//   phase 2  the CTA's neurons with h_i > 0 are listed in ascending order; warp w owns
//            columns d/16 w .. d/16 (w+1) - 1 of y and, for every listed neuron, reads its
//            d/8 bytes of that neuron's down-projection row (eight rows in flight per lane):
//            y += h_i w_down_i in fp32; the CTA's partial y goes to the workspace.
// relu2_mlp_combine_kernel: y = the CTAs' partials summed in CTA order (eight threads per
//            column, then a fixed-order sum of their parts), and the live-neuron count.
#include "internal.h"
#include "ptx.cuh"

namespace embla {
namespace {

constexpr int kMlpWarps = 16;
constexpr int kMlpThreads = kMlpWarps * 32;

struct MlpParams {
  const uint16_t *x, *w_up, *w_down;
  float *part;       // [ctas][d]
  int32_t *live;     // [ctas]
  int64_t d, f, per_cta;
};

// acc0 += lo(w) lo(x), acc1 += hi(w) hi(x): exact bf16 products, fp32 sums.
__device__ __forceinline__ void dot_acc_bf16x2(uint32_t w, uint32_t x, float &acc0, float &acc1) {
  asm("{\n\t.reg .b16 wl, wh, xl, xh;\n\t"
      "mov.b32 {wl, wh}, %2;\n\t"
      "mov.b32 {xl, xh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, wl, xl, %0;\n\t"
      "fma.rn.f32.bf16 %1, wh, xh, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(w), "r"(x));
}

__device__ __forceinline__ float dot_chunk(const uint4 &w, const uint4 &x, float a) {
  float a0 = a, a1 = 0.0f;
  dot_acc_bf16x2(w.x, x.x, a0, a1);
  dot_acc_bf16x2(w.y, x.y, a0, a1);
  dot_acc_bf16x2(w.z, x.z, a0, a1);
  dot_acc_bf16x2(w.w, x.w, a0, a1);
  return a0 + a1;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// KC = d / 256: the 16-byte chunks of a row per lane in phase 1; phase 2 gives each lane
// KC / 2 columns of y (d / 16 per warp).
template <int KC>
__global__ void __launch_bounds__(kMlpThreads, 1) relu2_mlp_kernel(const MlpParams p) {
  pdl_wait_primary();  // the token is complete
  pdl_launch_dependents();
  __shared__ float s_h[kMlpMaxNeuronsPerCta];
  __shared__ int32_t s_idx[kMlpMaxNeuronsPerCta];
  __shared__ float s_hl[kMlpMaxNeuronsPerCta];
  __shared__ int32_t s_nlive;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * p.per_cta;
  const int64_t i1 = i0 + p.per_cta < p.f ? i0 + p.per_cta : p.f;
  const int nn = i1 > i0 ? static_cast<int>(i1 - i0) : 0;

  // ---- phase 1: pre-activations of this CTA's neurons
  uint4 xr[KC];
#pragma unroll
  for (int k = 0; k < KC; ++k) xr[k] = reinterpret_cast<const uint4 *>(p.x)[lane + 32 * k];
  for (int a = warp; a < nn; a += 2 * kMlpWarps) {
    const int b = a + kMlpWarps;  // a second row in flight
    const uint4 *ra = reinterpret_cast<const uint4 *>(p.w_up + (i0 + a) * p.d);
    const uint4 *rb = reinterpret_cast<const uint4 *>(p.w_up + (i0 + (b < nn ? b : a)) * p.d);
    uint4 wa[KC], wb[KC];
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      wa[k] = __ldcs(ra + lane + 32 * k);
      wb[k] = __ldcs(rb + lane + 32 * k);
    }
    float sa = 0.0f, sb = 0.0f;
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      sa = dot_chunk(wa[k], xr[k], sa);
      sb = dot_chunk(wb[k], xr[k], sb);
    }
    sa = warp_sum(sa);
    sb = warp_sum(sb);
    if (lane == 0) {
      s_h[a] = sa > 0.0f ? sa * sa : 0.0f;
      if (b < nn) s_h[b] = sb > 0.0f ? sb * sb : 0.0f;
    }
  }
  __syncthreads();
  // ---- the neurons that fired, in ascending order
  if (warp == 0) {
    int cnt = 0;
    for (int base = 0; base < nn; base += 32) {
      const int i = base + lane;
      const float hv = i < nn ? s_h[i] : 0.0f;
      const uint32_t m = __ballot_sync(0xffffffffu, hv > 0.0f);
      if (hv > 0.0f) {
        const int e = cnt + __popc(m & ((1u << lane) - 1u));
        s_idx[e] = i;
        s_hl[e] = hv;
      }
      cnt += __popc(m);
    }
    if (lane == 0) s_nlive = cnt;
  }
  __syncthreads();
  // ---- phase 2: this warp's columns of y over the listed rows
  const int nlive = s_nlive;
  constexpr int NC = KC / 2;  // columns per lane
  const int64_t c0 = static_cast<int64_t>(warp) * (32 * NC) + static_cast<int64_t>(lane) * NC;
  float y[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) y[c] = 0.0f;
  for (int e0 = 0; e0 < nlive; e0 += 8) {
    uint32_t raw[8][(NC + 1) / 2];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
#pragma unroll
      for (int k = 0; k < (NC + 1) / 2; ++k) raw[r][k] = 0u;
      if (e0 + r < nlive) {
        const uint16_t *row = p.w_down + (i0 + s_idx[e0 + r]) * p.d + c0;
        if constexpr (NC == 4) {
          const uint2 v = __ldcs(reinterpret_cast<const uint2 *>(row));
          raw[r][0] = v.x;
          raw[r][1] = v.y;
        } else if constexpr (NC == 2) {
          raw[r][0] = __ldcs(reinterpret_cast<const unsigned int *>(row));
        } else {
          raw[r][0] = __ldcs(reinterpret_cast<const unsigned short *>(row));
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const float hv = e0 + r < nlive ? s_hl[e0 + r] : 0.0f;
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const uint32_t wv = raw[r][c >> 1];
        const float v = (c & 1) ? bf16hi(wv) : bf16lo(wv);
        y[c] = fmaf(hv, v, y[c]);
      }
    }
  }
  float *dst = p.part + static_cast<int64_t>(blockIdx.x) * p.d + c0;
#pragma unroll
  for (int c = 0; c < NC; ++c) dst[c] = y[c];
  if (threadIdx.x == 0) p.live[blockIdx.x] = nlive;
}

// y[col] = sum over CTAs in order of part[cta][col]: thread (s, c) sums CTAs s, s + 8, ...
// of column c, then the eight parts are added in order of s.
__global__ void __launch_bounds__(256) relu2_mlp_combine_kernel(const float *part, const int32_t *live,
                                                                int ctas, int64_t d, float *y,
                                                                int32_t *n_live) {
  pdl_wait_primary();  // every partial is written
  pdl_launch_dependents();
  __shared__ float s_part[8][33];
  const int c = threadIdx.x & 31, s = threadIdx.x >> 5;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * 32 + c;
  float acc = 0.0f;
  if (col < d) {
    for (int k0 = s; k0 < ctas; k0 += 64) {
      float v[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int k = k0 + 8 * t;
        v[t] = k < ctas ? part[static_cast<int64_t>(k) * d + col] : 0.0f;
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) acc += v[t];
    }
  }
  s_part[s][c] = acc;
  __syncthreads();
  if (s == 0 && col < d) {
    float t = 0.0f;
#pragma unroll
    for (int k = 0; k < 8; ++k) t += s_part[k][c];
    y[col] = t;
  }
  if (blockIdx.x == 0 && s == 1) {
    int32_t tot = 0;
    for (int k = c; k < ctas; k += 32) tot += live[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (c == 0) *n_live = tot;
  }
}

}  // namespace

int mlp_ctas(int64_t f, int sm_count) {
  int64_t ctas = sm_count;
  const int64_t need = (f + kMlpMaxNeuronsPerCta - 1) / kMlpMaxNeuronsPerCta;
  if (ctas < need) ctas = need;
  if (ctas > f) ctas = f;
  return static_cast<int>(ctas < 1 ? 1 : ctas);
}

size_t mlp_workspace_bytes(int64_t d, int64_t f, int sm_count) {
  const int ctas = mlp_ctas(f, sm_count);
  return (static_cast<size_t>(ctas) * static_cast<size_t>(d) * 4 + static_cast<size_t>(ctas) * 4 + 255) &
         ~static_cast<size_t>(255);
}

cudaError_t launch_relu2_mlp(const void *x, const void *w_up, const void *w_down, int64_t d,
                             int64_t f, float *y, int32_t *n_live, void *workspace, int sm_count,
                             cudaStream_t stream) {
  const int ctas = mlp_ctas(f, sm_count);
  MlpParams p;
  p.x = static_cast<const uint16_t *>(x);
  p.w_up = static_cast<const uint16_t *>(w_up);
  p.w_down = static_cast<const uint16_t *>(w_down);
  p.part = static_cast<float *>(workspace);
  p.live = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) +
                                       static_cast<size_t>(ctas) * static_cast<size_t>(d) * 4);
  p.d = d;
  p.f = f;
  p.per_cta = (f + ctas - 1) / ctas;
  cudaError_t e;
  switch (d) {
    case 512: e = launch_pdl(relu2_mlp_kernel<2>, dim3(ctas), dim3(kMlpThreads), 0, stream, 0u, p); break;
    case 1024: e = launch_pdl(relu2_mlp_kernel<4>, dim3(ctas), dim3(kMlpThreads), 0, stream, 0u, p); break;
    case 2048: e = launch_pdl(relu2_mlp_kernel<8>, dim3(ctas), dim3(kMlpThreads), 0, stream, 0u, p); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return launch_pdl(relu2_mlp_combine_kernel, dim3(static_cast<unsigned>((d + 31) / 32)), dim3(256),
                    0, stream, 0u, static_cast<const float *>(p.part),
                    static_cast<const int32_t *>(p.live), ctas, d, y, n_live);
}

}  // namespace embla
