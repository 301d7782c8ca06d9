// ReLU^2 MLP of one token, reading only the down-projection rows of neurons that fired.
//
// Source: "The Architecture of Embla 1", section "ReLU^2 activation": a negative
// pre-activation becomes zero and a positive one is squared; a zero neuron's row of the
// down projection contributes nothing, so at batch size 1 a kernel reads only the rows of
// the neurons that fired.
//
// relu2_mlp_kernel: one CTA per SM over a contiguous range of neurons, 16 warps.
//   phase 1  each warp takes neurons in turn, two rows in flight: h_i = max(w_up_i . x, 0)^2
//            with exact bf16 products summed in fp32 (the token x in shared memory);
//   phase 2  the CTA's neurons with h_i > 0 are listed in ascending order; each thread owns
//            8 columns of y and a class of listed rows (every listed row is read once, 16
//            bytes to a thread, all of a thread's rows in flight together): y += h_i w_down_i
//            in fp32, the classes' sums added in class order; the CTA's partial y goes to
//            the workspace.  Every up-projection row of the CTA is prefetched into L2 when
//            the CTA starts, and a neuron's down-projection row as soon as it fires.
// relu2_mlp_combine_kernel: y = the CTAs' partials summed in a fixed order (8 threads per
//            column, then their sums in order), and the live-neuron count.
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
  __shared__ float s_h[kMlpMaxNeuronsPerCta];
  __shared__ int32_t s_idx[kMlpMaxNeuronsPerCta];
  __shared__ float s_hl[kMlpMaxNeuronsPerCta];
  __shared__ int32_t s_nlive;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * p.per_cta;
  const int64_t i1 = i0 + p.per_cta < p.f ? i0 + p.per_cta : p.f;
  const int nn = i1 > i0 ? static_cast<int>(i1 - i0) : 0;
  // The CTA's up-projection rows start moving into L2 before the wait for the kernel before
  // this one (a prefetch reads nothing into the SM, so it is safe whatever that kernel does);
  // the loads after the wait then find them there.
  const uint32_t row_bytes = static_cast<uint32_t>(p.d * 2);
  for (int a = threadIdx.x; a < nn; a += kMlpThreads) prefetch_l2_bulk(p.w_up + (i0 + a) * p.d, row_bytes);
  pdl_wait_primary();  // the token is complete
  pdl_launch_dependents();

  // ---- phase 1: pre-activations of this CTA's neurons (the token in shared memory)
  __shared__ uint4 s_x[KC * 32];
  for (int k = threadIdx.x; k < KC * 32; k += kMlpThreads) s_x[k] = reinterpret_cast<const uint4 *>(p.x)[k];
  __syncthreads();
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
      const uint4 xk = s_x[lane + 32 * k];
      sa = dot_chunk(wa[k], xk, sa);
      sb = dot_chunk(wb[k], xk, sb);
    }
    sa = warp_sum(sa);
    sb = warp_sum(sb);
    if (lane == 0) {
      s_h[a] = sa > 0.0f ? sa * sa : 0.0f;
      if (b < nn) s_h[b] = sb > 0.0f ? sb * sb : 0.0f;
      // a neuron that fired: its down-projection row starts moving into L2 now
      if (sa > 0.0f) prefetch_l2_bulk(p.w_down + (i0 + a) * p.d, row_bytes);
      if (b < nn && sb > 0.0f) prefetch_l2_bulk(p.w_down + (i0 + b) * p.d, row_bytes);
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
  // ---- phase 2: y over the listed rows.  Thread t owns the 8 columns of 16-byte piece
  // t % (d / 8) of a row and every listed row e with e % R == t / (d / 8), R = 512 / (d / 8)
  // row classes; all of its rows' pieces are requested before any is used (up to 8 in
  // flight, then the next 8), and the R class sums are added in class order.
  const int nlive = s_nlive;
  constexpr int kPieces = KC * 32;          // 16-byte pieces of a row: d / 8
  constexpr int kClasses = kMlpThreads / kPieces;
  const int piece = threadIdx.x % kPieces, cls = threadIdx.x / kPieces;
  float y[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) y[c] = 0.0f;
  for (int e0 = cls; e0 < nlive; e0 += 8 * kClasses) {
    uint4 raw[8];
    float hv[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int e = e0 + r * kClasses;
      raw[r] = make_uint4(0u, 0u, 0u, 0u);
      hv[r] = 0.0f;
      if (e < nlive) {
        raw[r] = __ldcs(reinterpret_cast<const uint4 *>(p.w_down + (i0 + s_idx[e]) * p.d) + piece);
        hv[r] = s_hl[e];
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t w4[4] = {raw[r].x, raw[r].y, raw[r].z, raw[r].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        y[2 * c] = fmaf(hv[r], bf16lo(w4[c]), y[2 * c]);
        y[2 * c + 1] = fmaf(hv[r], bf16hi(w4[c]), y[2 * c + 1]);
      }
    }
  }
  // the class sums, added in class order
  __shared__ float s_y[(kClasses - 1) * kPieces * 8 + 1];
  if (cls > 0) {
#pragma unroll
    for (int c = 0; c < 8; ++c) s_y[(cls - 1) * kPieces * 8 + piece * 8 + c] = y[c];
  }
  __syncthreads();
  if (cls == 0) {
#pragma unroll
    for (int k = 1; k < kClasses; ++k) {
#pragma unroll
      for (int c = 0; c < 8; ++c) y[c] += s_y[(k - 1) * kPieces * 8 + piece * 8 + c];
    }
    float4 *dst = reinterpret_cast<float4 *>(p.part + static_cast<int64_t>(blockIdx.x) * p.d + piece * 8);
    dst[0] = make_float4(y[0], y[1], y[2], y[3]);
    dst[1] = make_float4(y[4], y[5], y[6], y[7]);
  }
  if (threadIdx.x == 0) p.live[blockIdx.x] = nlive;
}

// y[col] = the CTAs' partials of column col summed in a fixed order: thread (s, c) of a CTA
// (32 columns x 8 slices) sums CTAs s, s + 8, ... of column c (all of its loads in flight
// together), then the 8 slice sums are added in slice order.  256 threads of few registers,
// so a CTA fits beside one of the next call's relu2_mlp_kernel on an SM.
constexpr int kCombSlices = 8;
constexpr int kCombLoads = 20;  // loads in flight per thread: 160 CTAs per pass
__global__ void __launch_bounds__(32 * kCombSlices) relu2_mlp_combine_kernel(const float *part,
                                                                             const int32_t *live,
                                                                             int ctas, int64_t d, float *y,
                                                                             int32_t *n_live) {
  __shared__ float s_part[kCombSlices][33];
  const int c = threadIdx.x & 31, s = threadIdx.x >> 5;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * 32 + c;
  // The CTA is launched while the main kernel runs; its partials' lines go to L2 (with their
  // address translations) before the wait: a prefetch reads nothing into the SM.
  if (col < d && c == 0)
    for (int k = s; k < ctas; k += kCombSlices)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(part + static_cast<int64_t>(k) * d + col));
  pdl_wait_primary();  // every partial is written
  pdl_launch_dependents();
  float acc = 0.0f;
  if (col < d) {
    for (int k0 = s; k0 < ctas; k0 += kCombSlices * kCombLoads) {
      float v[kCombLoads];
#pragma unroll
      for (int t = 0; t < kCombLoads; ++t) {
        const int k = k0 + kCombSlices * t;
        v[t] = k < ctas ? part[static_cast<int64_t>(k) * d + col] : 0.0f;
      }
#pragma unroll
      for (int t = 0; t < kCombLoads; ++t) acc += v[t];
    }
  }
  s_part[s][c] = acc;
  __syncthreads();
  if (s == 0 && col < d) {
    float v = s_part[0][c];
#pragma unroll
    for (int k = 1; k < kCombSlices; ++k) v += s_part[k][c];
    y[col] = v;
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
  return launch_pdl(relu2_mlp_combine_kernel, dim3(static_cast<unsigned>((d + 31) / 32)), dim3(32 * kCombSlices),
                    0, stream, 0u, static_cast<const float *>(p.part),
                    static_cast<const int32_t *>(p.live), ctas, d, y, n_live);
}

}  // namespace embla
