// Launchers shared between the translation units of the library (not part of the ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

namespace embla {

// Launch a kernel of this library so that it may be scheduled while the kernel before it
// in the stream is still running (programmatic dependent launch).  Every such kernel
// waits for its predecessor to finish (griddepcontrol.wait) before it reads an input or
// writes an output, and only then lets its own successor launch, so stream order holds
// for data; what overlaps is the launch itself.  `cluster` > 0 sets the cluster size of
// kernels that do not fix it at compile time.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, unsigned cluster, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster > 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(na);
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

constexpr int kHeadDim = 128;
constexpr int kTileKeys = 128;     // keys per full-decode tile (the MMA's M)
constexpr int kHistBins = 2048;    // selection histogram: top 11 bits of the order key

// Work split of the full-layer decode: the T tiles (TU per unit, units one after another)
// are cut into Q = K * P pieces, piece q holding tiles [floor(q*T/Q), floor((q+1)*T/Q)), and
// persistent CTA c of P takes pieces c, c + P, ..., c + (K-1)P in that order.  With K > 1 a
// CTA's tiles come from K places spread over the batch, so sequences whose keys survive
// more often (more V rows to fetch) do not all land on the same CTAs; K is odd, so a
// power-of-two period in the batch (sequences x heads) does not line a CTA's pieces up with
// it.  The partial record of the stretch of unit u inside piece q lives in slot q + u.
struct FullSplit {
  int64_t units;      // B * Hkv
  int64_t tiles_per_unit;
  int64_t tiles;      // units * tiles_per_unit
  int32_t ctas;       // P
  int32_t pieces;     // Q = K * P
};

constexpr int kMaxPiecesPerCta = 5;
static_assert(kMaxPiecesPerCta % 2 == 1, "K is odd");
constexpr int kMinPieceTiles = 20;  // a CTA's share is cut into pieces of at least this many

__host__ __device__ inline int64_t split_piece_start(int64_t q, int64_t T, int64_t Q) {
  return (q * T) / Q;
}
// The piece that holds tile t.
__host__ __device__ inline int64_t split_piece_of_tile(int64_t t, int64_t T, int64_t Q) {
  return ((t + 1) * Q - 1) / T;
}

// max_pieces (odd, >= 1) caps K.
FullSplit full_split(int64_t units, int64_t ctx_len, int sm_count,
                     int max_pieces = kMaxPiecesPerCta);
int full_record_floats(int G);
size_t full_workspace_bytes(const FullSplit &sp, int G);

// The selection launched between the decode and its combining kernel (launch_select's
// arguments beyond the scores and histogram): the combining kernel then runs beside it.
struct SelectJob {
  int topk, recent;
  int32_t *idx;
  int idx_stride;
  int32_t *count;
  void *workspace;
  int sm_count;
};

// kv8: 8-bit E4M3 caches; tm_ks / tm_vs then map the K and V scales as [units, ncap] fp32.
// sj (needs sel_scores): also select each unit's keys from the decode's scores.
cudaError_t launch_full_decode(int G, bool kv8, const CUtensorMap &tm_k, const CUtensorMap &tm_q,
                               const CUtensorMap *tm_ks, const CUtensorMap *tm_vs,
                               const void *v_cache, float *sel_scores, float *head_scores,
                               uint32_t *sel_hist, void *workspace,
                               float *out, int32_t *n_surv, float c, uint32_t *flags,
                               const FullSplit &sp, int64_t n,
                               int64_t ncap, int Hq, int Hkv, float alpha, float eps,
                               cudaStream_t stream, const SelectJob *sj = nullptr);

size_t select_workspace_bytes(int64_t units, int64_t ctx_len);
// hist[u] = 2048-bin counts of the order keys' top 11 bits of scores[u][0..n) (every unit).
cudaError_t launch_score_hist(const float *scores, int64_t units, int64_t n, int64_t ncap,
                              uint32_t *hist, cudaStream_t stream);
cudaError_t launch_select(const float *sel_scores, const uint32_t *sel_hist, int64_t units,
                          int64_t n, int64_t ncap, int topk, int recent, int32_t *idx,
                          int idx_stride, int32_t *count, void *workspace, uint32_t *flags,
                          int sm_count, cudaStream_t stream);

// Appending a token's rows: for each plane u < units, row_bytes bytes from
// src + u * row_bytes to dst + (u * cache_stride + pos) * row_bytes.  vec (the copy width,
// 16, 4 or 1 bytes) is set by the launcher.
struct AppendJob {
  const uint8_t *src;
  uint8_t *dst;
  int64_t row_bytes;
  int64_t cache_stride;
  int vec;
};
constexpr int kAppendMaxJobs = 4;
struct AppendParams {
  AppendJob job[kAppendMaxJobs];
  int njobs;
  int64_t units, pos;
};
cudaError_t launch_append_rows(const AppendJob *jobs, int njobs, int64_t units, int64_t pos,
                               cudaStream_t stream);

size_t sparse_workspace_bytes(int64_t units, int G, int idx_stride);
// k_scales / v_scales: per-token scales of 8-bit E4M3 caches, or both null for bf16 caches.
// per_head: one unit per (sequence, query head) with its own selection (G then 1, the
// cache plane of unit u is (u / Hq) * Hkv + (u % Hq) / (Hq / Hkv)).
cudaError_t launch_sparse_decode(int G, bool per_head, int Hq, const void *q, const void *k_cache,
                                 const void *v_cache,
                                 const float *k_scales, const float *v_scales, const int32_t *idx, int idx_stride, const int32_t *count,
                                 int64_t units, int Hkv, int64_t n, int64_t ncap, float tau,
                                 float *out, void *workspace, uint32_t *flags, int sm_count,
                                 cudaStream_t stream);

cudaError_t launch_skip_stats(const float *sel_scores, int64_t units, int64_t n, int64_t ncap,
                              int chunk, int32_t *keys_needed, int32_t *chunks_needed,
                              cudaStream_t stream);

// Prefill (causal full-layer attention over the last T of n keys): key-norm workspace and
// launch (a key-norm kernel, then the attention kernel).
int64_t prefill_rk_stride(int64_t n);
size_t prefill_workspace_bytes(int64_t units, int64_t n);
cudaError_t launch_prefill(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                           const CUtensorMap &tm_rk, const void *k_cache, float *rk, float *out,
                           uint32_t *flags, int B, int Hq, int Hkv, int64_t n, int64_t T,
                           int64_t ncap, float alpha, float c, float eps, int sm_count,
                           cudaStream_t stream);

// ReLU^2 MLP of one token (d in {512, 1024, 2048}; at most kMlpMaxNeuronsPerCta neurons
// per CTA): the fused kernel's partials and live counts in the workspace, then a combine.
constexpr int kMlpMaxNeuronsPerCta = 1024;
int mlp_ctas(int64_t f, int sm_count);
size_t mlp_workspace_bytes(int64_t d, int64_t f, int sm_count);
cudaError_t launch_relu2_mlp(const void *x, const void *w_up, const void *w_down, int64_t d,
                             int64_t f, float *y, int32_t *n_live, void *workspace, int sm_count,
                             cudaStream_t stream);

cudaError_t launch_window_decode(int G, const void *q, const void *k_win, const void *v_win,
                                 int64_t units, int window, int64_t pos, float rope_base,
                                 float tau, float *out, cudaStream_t stream);

}  // namespace embla
