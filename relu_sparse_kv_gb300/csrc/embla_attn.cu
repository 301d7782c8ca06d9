// C ABI of the library: host-side argument checks, workspace sizing, TMA descriptor
// encoding and the launches of the kernels in this directory.  Declarations and the
// meaning of every argument are in include/embla_attn.h.
#include <atomic>
#include <cstring>
#include <mutex>

#include "embla_attn.h"
#include "internal.h"
#include "ptx.cuh"

using namespace embla;

// Scratch of embla_full_decode_static_scratch: one fixed array per device, so that
// call needs no workspace from its caller and allocates nothing itself.
static __device__ __align__(256) unsigned char g_full_scratch[EMBLA_FULL_DECODE_SCRATCH_BYTES];

namespace {

// Device-side check word (flag bits, see embla_device_check).
__device__ uint32_t g_check_flags;

constexpr int kMaxDevices = 64;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

// Per-device values looked up once and kept.  Every slot is an atomic, filled at most
// once per device (a look-up that fails leaves the slot empty, so the next call retries);
// two host threads making their first call on a device at the same time may both look the
// value up, and both store the same value.
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<void *> g_flags_addr[kMaxDevices];
std::atomic<void *> g_scratch_addr[kMaxDevices];

int sm_count_of(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return 0;
  int v = g_sm_count[dev].load(std::memory_order_acquire);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev].store(v, std::memory_order_release);
  }
  return v;
}

// Device address of a __device__ symbol on the current device, cached in `slot`.
template <typename T>
void *symbol_address(std::atomic<void *> (&slot)[kMaxDevices], const T &symbol) {
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  void *p = slot[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
    slot[dev].store(p, std::memory_order_release);
  }
  return p;
}

uint32_t *flags_ptr() { return static_cast<uint32_t *>(symbol_address(g_flags_addr, g_check_flags)); }

// One thread waits, through the kernels' bounded wait, on a shared-memory barrier that
// nothing arrives at; when the limit runs out it records a timed-out wait in the check
// word, as a kernel's pipeline wait does, and returns.  If `arrive` is set the thread
// arrives first, so the wait succeeds at once and nothing is recorded.
__global__ void wait_limit_kernel(uint32_t *flags, uint64_t limit_ns, int arrive) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (arrive) mbar_arrive(&bar);
  if (!mbar_wait(&bar, 0u, limit_ns)) atomicOr(flags, kFlagWaitTimeout);
}

// Device address of g_full_scratch on the current device, looked up on the first
// call for that device and kept; nullptr if the look-up fails.
void *full_scratch_ptr() { return symbol_address(g_scratch_addr, g_full_scratch); }

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D bf16 tensor [rows, 128] with 256-byte rows, boxes of {64 columns, box_rows}, 128B swizzle.
bool encode_rows(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows,
                 CUtensorMapL2promotion promo) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim * 2)};
  const cuuint32_t box[2] = {64u, box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, promo,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D uint8 tensor [rows, 128] of E4M3 codes (128-byte rows), boxes of {128 columns,
// box_rows}, 128B swizzle.
bool encode_rows_e4m3(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kHeadDim), box_rows};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D fp32 tensor [units, ncap] of per-token scales, boxes of {128 tokens, 1 unit}; tokens
// past ncap read as 0.
bool encode_scales(CUtensorMap *map, const float *base, uint64_t units, uint64_t ncap) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {ncap, units};
  const cuuint64_t strides[1] = {ncap * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileKeys), 1u};
  const cuuint32_t estr[2] = {1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 tensor [planes][rows][128] (256-byte rows, planes `plane_rows` rows apart),
// boxes of {64 columns, 128 rows, 1 plane}, 128B swizzle; rows past `rows` read as zeros.
bool encode_planes(CUtensorMap *map, const void *base, uint64_t rows, uint64_t plane_rows,
                   uint64_t planes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), rows, planes};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim * 2), plane_rows * kHeadDim * 2};
  const cuuint32_t box[3] = {64u, 128u, 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite(float x) { return x == x && x - x == 0.0f; }

// Common shape checks; sets *G.  ctx_checks: also validate ctx_len / cache_stride.
embla_status check_shape(const embla_shape *s, int *G, bool ctx_checks) {
  if (!s) return EMBLA_ERR_INVALID_ARG;
  if (s->batch < 0 || s->n_q_heads < 1 || s->n_kv_heads < 1) return EMBLA_ERR_INVALID_ARG;
  if (s->n_q_heads % s->n_kv_heads) return EMBLA_ERR_INVALID_ARG;
  if (s->head_dim < 1) return EMBLA_ERR_INVALID_ARG;
  if (ctx_checks) {
    if (s->ctx_len < 0 || s->ctx_len > INT32_MAX) return EMBLA_ERR_INVALID_ARG;
    if (s->cache_stride < s->ctx_len) return EMBLA_ERR_INVALID_ARG;
  }
  *G = s->n_q_heads / s->n_kv_heads;
  if (s->head_dim != kHeadDim) return EMBLA_ERR_UNSUPPORTED;
  if (*G != 4 && *G != 8) return EMBLA_ERR_UNSUPPORTED;
  return EMBLA_OK;
}

embla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? EMBLA_OK : EMBLA_ERR_CUDA; }

}  // namespace

extern "C" {

const char *embla_status_string(embla_status status) {
  switch (status) {
    case EMBLA_OK: return "ok";
    case EMBLA_ERR_INVALID_ARG: return "invalid argument";
    case EMBLA_ERR_UNSUPPORTED: return "unsupported shape (head_dim must be 128, G in {4, 8})";
    case EMBLA_ERR_WORKSPACE: return "workspace too small";
    case EMBLA_ERR_CUDA: return "CUDA error";
    case EMBLA_ERR_DEVICE_CHECK: return "device-side check failed";
  }
  return "unknown status";
}

int embla_device_sm_count(void) { return sm_count_of(current_device()); }

size_t embla_full_decode_workspace_size(const embla_shape *shape) {
  int G = 0;
  if (check_shape(shape, &G, true) != EMBLA_OK) return 0;
  const int sms = sm_count_of(current_device());
  if (sms <= 0) return 0;
  return full_workspace_bytes(
      full_split(static_cast<int64_t>(shape->batch) * shape->n_kv_heads, shape->ctx_len, sms), G);
}

}  // extern "C"

namespace {

// The selection requested together with a full-layer decode.
struct SelectArgs {
  int32_t topk, recent;
  int32_t *idx;
  int32_t idx_stride;
  int32_t *count;
};

// The full-layer decode for bf16 caches (k_scales and v_scales null) or 8-bit E4M3 caches
// with per-token scales; with sa, followed by the selection over its scores (the workspace
// then holds the decode's records, then the selection's workspace).
embla_status full_decode_impl(const embla_shape *shape, const void *q, const void *k_cache,
                              const float *k_scales, const void *v_cache, const float *v_scales,
                              bool kv8, float alpha, float c, float eps, float *out,
                              int32_t *n_surv, float *sel_scores, uint32_t *sel_hist,
                              void *workspace, size_t workspace_bytes, void *stream,
                              float *head_scores = nullptr, uint32_t *head_hist = nullptr,
                              int max_pieces = kMaxPiecesPerCta,
                              const SelectArgs *sa = nullptr) {
  int G = 0;
  embla_status st = check_shape(shape, &G, true);
  if (st != EMBLA_OK) return st;
  if (!(finite(alpha) && alpha > 0.0f) || !(finite(c) && c >= 0.0f) ||
      !(finite(eps) && eps >= 0.0f))
    return EMBLA_ERR_INVALID_ARG;
  // the scale arrays are read as [units, cache_stride] with 16-byte aligned rows
  if (kv8 && shape->cache_stride % 4 != 0) return EMBLA_ERR_INVALID_ARG;
  const int64_t units = static_cast<int64_t>(shape->batch) * shape->n_kv_heads;
  if (units == 0) return EMBLA_OK;
  if (!q || !k_cache || !v_cache || !out || !n_surv || !workspace) return EMBLA_ERR_INVALID_ARG;
  if (kv8 && (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales)))
    return EMBLA_ERR_INVALID_ARG;
  if ((sel_scores == nullptr) != (sel_hist == nullptr)) return EMBLA_ERR_INVALID_ARG;
  if (sa && (!sel_scores || sa->topk < 0 || sa->recent < 0 ||
             static_cast<int64_t>(sa->topk) + sa->recent > INT32_MAX ||
             sa->idx_stride < sa->topk + sa->recent || !sa->idx || !sa->count ||
             !aligned16(sa->idx) || !aligned16(sa->count)))
    return EMBLA_ERR_INVALID_ARG;
  if ((head_scores == nullptr) != (head_hist == nullptr)) return EMBLA_ERR_INVALID_ARG;
  if (head_scores && (!aligned16(head_scores) || !aligned16(head_hist)))
    return EMBLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(workspace) || (sel_scores && (!aligned16(sel_scores) || !aligned16(sel_hist))))
    return EMBLA_ERR_INVALID_ARG;
  // TMA row coordinates are 32-bit
  if (units * shape->cache_stride + kTileKeys > INT32_MAX) return EMBLA_ERR_UNSUPPORTED;
  const int dev = current_device();
  const int sms = sm_count_of(dev);
  if (sms <= 0) return EMBLA_ERR_CUDA;
  const FullSplit sp = full_split(units, shape->ctx_len, sms, max_pieces);
  const size_t rec_bytes = full_workspace_bytes(sp, G);
  const size_t sel_bytes = sa ? select_workspace_bytes(units, shape->ctx_len) : 0;
  if (workspace_bytes < rec_bytes + sel_bytes) return EMBLA_ERR_WORKSPACE;
  uint32_t *flags = flags_ptr();
  if (!flags) return EMBLA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (sp.tiles == 0) {
    // no keys: every output is 0, nothing survives, the histogram is empty
    if (sel_scores)
      st = cuda_status(cudaMemsetAsync(sel_hist, 0, static_cast<size_t>(units) * kHistBins * 4, s));
    if (st == EMBLA_OK && head_scores)
      st = cuda_status(cudaMemsetAsync(head_hist, 0,
                                       static_cast<size_t>(shape->batch) * shape->n_q_heads * kHistBins * 4, s));
    if (st == EMBLA_OK)
      st = cuda_status(cudaMemsetAsync(out, 0, static_cast<size_t>(units) * G * kHeadDim * 4, s));
    if (st == EMBLA_OK) st = cuda_status(cudaMemsetAsync(n_surv, 0, static_cast<size_t>(units) * 4, s));
    if (st == EMBLA_OK && sa)  // no keys to select
      st = cuda_status(cudaMemsetAsync(sa->count, 0, static_cast<size_t>(units) * 4, s));
    return st;
  }
  // the launch zeroes the histogram and the survivor counts itself
  const uint64_t rows = static_cast<uint64_t>(units * shape->cache_stride);
  CUtensorMap tm_k, tm_q, tm_ks, tm_vs;
  const bool kmap = kv8 ? encode_rows_e4m3(&tm_k, k_cache, rows, kTileKeys)
                        : encode_rows(&tm_k, k_cache, rows, kTileKeys,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
  if (!kmap ||
      !encode_rows(&tm_q, q, static_cast<uint64_t>(shape->batch) * shape->n_q_heads,
                   static_cast<uint32_t>(G), CU_TENSOR_MAP_L2_PROMOTION_NONE))
    return EMBLA_ERR_CUDA;
  if (kv8 && (!encode_scales(&tm_ks, k_scales, static_cast<uint64_t>(units),
                             static_cast<uint64_t>(shape->cache_stride)) ||
              !encode_scales(&tm_vs, v_scales, static_cast<uint64_t>(units),
                             static_cast<uint64_t>(shape->cache_stride))))
    return EMBLA_ERR_CUDA;
  SelectJob sj = {};
  if (sa) {
    sj.topk = sa->topk;
    sj.recent = sa->recent;
    sj.idx = sa->idx;
    sj.idx_stride = sa->idx_stride;
    sj.count = sa->count;
    sj.workspace = sel_bytes ? static_cast<uint8_t *>(workspace) + rec_bytes : nullptr;
    sj.sm_count = sms;
  }
  st = cuda_status(launch_full_decode(G, kv8, tm_k, tm_q, kv8 ? &tm_ks : nullptr,
                                      kv8 ? &tm_vs : nullptr, v_cache, sel_scores, head_scores,
                                      sel_hist, workspace, out, n_surv, c, flags, sp,
                                      shape->ctx_len, shape->cache_stride, shape->n_q_heads,
                                      shape->n_kv_heads, alpha, eps, s, sa ? &sj : nullptr));
  if (st == EMBLA_OK && head_scores)
    st = cuda_status(launch_score_hist(head_scores,
                                       static_cast<int64_t>(shape->batch) * shape->n_q_heads,
                                       shape->ctx_len, shape->cache_stride, head_hist, s));
  return st;
}

}  // namespace

extern "C" {

embla_status embla_full_decode(const embla_shape *shape, const void *q, const void *k_cache,
                               const void *v_cache, float alpha, float c, float eps, float *out,
                               int32_t *n_surv, float *sel_scores, uint32_t *sel_hist,
                               void *workspace, size_t workspace_bytes, void *stream) {
  return full_decode_impl(shape, q, k_cache, nullptr, v_cache, nullptr, false, alpha, c, eps,
                          out, n_surv, sel_scores, sel_hist, workspace, workspace_bytes, stream);
}

embla_status embla_full_decode_head_scores(const embla_shape *shape, const void *q,
                                           const void *k_cache, const void *v_cache, float alpha,
                                           float c, float eps, float *out, int32_t *n_surv,
                                           float *head_scores, uint32_t *head_hist,
                                           void *workspace, size_t workspace_bytes, void *stream) {
  if (!head_scores || !head_hist) return EMBLA_ERR_INVALID_ARG;
  return full_decode_impl(shape, q, k_cache, nullptr, v_cache, nullptr, false, alpha, c, eps,
                          out, n_surv, nullptr, nullptr, workspace, workspace_bytes, stream,
                          head_scores, head_hist);
}

embla_status embla_full_decode_e4m3(const embla_shape *shape, const void *q,
                                    const uint8_t *k_codes, const float *k_scales,
                                    const uint8_t *v_codes, const float *v_scales, float alpha,
                                    float c, float eps, float *out, int32_t *n_surv,
                                    float *sel_scores, uint32_t *sel_hist, void *workspace,
                                    size_t workspace_bytes, void *stream) {
  return full_decode_impl(shape, q, k_codes, k_scales, v_codes, v_scales, true, alpha, c, eps,
                          out, n_surv, sel_scores, sel_hist, workspace, workspace_bytes, stream);
}

size_t embla_full_decode_select_workspace_size(const embla_shape *shape, int32_t topk,
                                               int32_t recent) {
  int G = 0;
  if (check_shape(shape, &G, true) != EMBLA_OK || topk < 0 || recent < 0) return 0;
  const int sms = sm_count_of(current_device());
  if (sms <= 0) return 0;
  const int64_t units = static_cast<int64_t>(shape->batch) * shape->n_kv_heads;
  return full_workspace_bytes(full_split(units, shape->ctx_len, sms), G) +
         select_workspace_bytes(units, shape->ctx_len);
}

embla_status embla_full_decode_select(const embla_shape *shape, const void *q, const void *k_cache,
                                      const void *v_cache, float alpha, float c, float eps,
                                      float *out, int32_t *n_surv, float *sel_scores,
                                      uint32_t *sel_hist, int32_t topk, int32_t recent,
                                      int32_t *idx, int32_t idx_stride, int32_t *count,
                                      void *workspace, size_t workspace_bytes, void *stream) {
  const SelectArgs sa = {topk, recent, idx, idx_stride, count};
  return full_decode_impl(shape, q, k_cache, nullptr, v_cache, nullptr, false, alpha, c, eps, out,
                          n_surv, sel_scores, sel_hist, workspace, workspace_bytes, stream, nullptr,
                          nullptr, kMaxPiecesPerCta, &sa);
}

embla_status embla_full_decode_e4m3_select(const embla_shape *shape, const void *q,
                                           const uint8_t *k_codes, const float *k_scales,
                                           const uint8_t *v_codes, const float *v_scales,
                                           float alpha, float c, float eps, float *out,
                                           int32_t *n_surv, float *sel_scores, uint32_t *sel_hist,
                                           int32_t topk, int32_t recent, int32_t *idx,
                                           int32_t idx_stride, int32_t *count, void *workspace,
                                           size_t workspace_bytes, void *stream) {
  const SelectArgs sa = {topk, recent, idx, idx_stride, count};
  return full_decode_impl(shape, q, k_codes, k_scales, v_codes, v_scales, true, alpha, c, eps, out,
                          n_surv, sel_scores, sel_hist, workspace, workspace_bytes, stream, nullptr,
                          nullptr, kMaxPiecesPerCta, &sa);
}

embla_status embla_full_decode_static_scratch(const embla_shape *shape, const void *q,
                                              const void *k_cache, const void *v_cache,
                                              float alpha, float c, float eps, float *out,
                                              int32_t *n_surv, float *sel_scores,
                                              uint32_t *sel_hist, void *stream) {
  int G = 0;
  embla_status st = check_shape(shape, &G, true);
  if (st != EMBLA_OK) return st;
  const int64_t units = static_cast<int64_t>(shape->batch) * shape->n_kv_heads;
  const int sms = sm_count_of(current_device());
  if (sms <= 0) return EMBLA_ERR_CUDA;
  // fewer pieces per CTA (fewer records) where the usual split's records do not fit
  int max_pieces = kMaxPiecesPerCta;
  size_t need = full_workspace_bytes(full_split(units, shape->ctx_len, sms, max_pieces), G);
  while (need > EMBLA_FULL_DECODE_SCRATCH_BYTES && max_pieces > 1) {
    max_pieces -= 2;
    need = full_workspace_bytes(full_split(units, shape->ctx_len, sms, max_pieces), G);
  }
  if (need > EMBLA_FULL_DECODE_SCRATCH_BYTES) return EMBLA_ERR_WORKSPACE;
  void *scratch = full_scratch_ptr();
  if (!scratch) return EMBLA_ERR_CUDA;
  return full_decode_impl(shape, q, k_cache, nullptr, v_cache, nullptr, false, alpha, c, eps, out,
                          n_surv, sel_scores, sel_hist, scratch, need, stream, nullptr, nullptr,
                          max_pieces);
}

size_t embla_select_topk_workspace_size(const embla_shape *shape, int32_t topk, int32_t recent) {
  int G = 0;
  if (check_shape(shape, &G, true) != EMBLA_OK || topk < 0 || recent < 0) return 0;
  return select_workspace_bytes(static_cast<int64_t>(shape->batch) * shape->n_kv_heads,
                                shape->ctx_len);
}

embla_status embla_select_topk(const embla_shape *shape, const float *sel_scores,
                               const uint32_t *sel_hist, int32_t topk, int32_t recent,
                               int32_t *idx, int32_t idx_stride, int32_t *count, void *workspace,
                               size_t workspace_bytes, void *stream) {
  int G = 0;
  embla_status st = check_shape(shape, &G, true);
  if (st != EMBLA_OK) return st;
  if (topk < 0 || recent < 0 || static_cast<int64_t>(topk) + recent > INT32_MAX ||
      idx_stride < topk + recent)
    return EMBLA_ERR_INVALID_ARG;
  const int64_t units = static_cast<int64_t>(shape->batch) * shape->n_kv_heads;
  if (units == 0) return EMBLA_OK;
  const size_t ws_need = select_workspace_bytes(units, shape->ctx_len);
  if (!sel_scores || !sel_hist || !idx || !count || (ws_need && !workspace))
    return EMBLA_ERR_INVALID_ARG;
  if (!aligned16(sel_scores) || !aligned16(sel_hist) || !aligned16(idx) || !aligned16(count) ||
      (workspace && !aligned16(workspace)))
    return EMBLA_ERR_INVALID_ARG;
  if (workspace_bytes < ws_need) return EMBLA_ERR_WORKSPACE;
  uint32_t *flags = flags_ptr();
  if (!flags) return EMBLA_ERR_CUDA;
  const int sms = sm_count_of(current_device());
  if (sms <= 0) return EMBLA_ERR_CUDA;
  return cuda_status(launch_select(sel_scores, sel_hist, units, shape->ctx_len,
                                   shape->cache_stride, topk, recent, idx, idx_stride, count,
                                   workspace, flags, sms, static_cast<cudaStream_t>(stream)));
}

size_t embla_select_topk_per_head_workspace_size(const embla_shape *shape, int32_t topk,
                                                  int32_t recent) {
  int G = 0;
  if (check_shape(shape, &G, true) != EMBLA_OK || topk < 0 || recent < 0) return 0;
  return select_workspace_bytes(static_cast<int64_t>(shape->batch) * shape->n_q_heads,
                                shape->ctx_len);
}

embla_status embla_select_topk_per_head(const embla_shape *shape, const float *head_scores,
                                        const uint32_t *head_hist, int32_t topk, int32_t recent,
                                        int32_t *idx, int32_t idx_stride, int32_t *count,
                                        void *workspace, size_t workspace_bytes, void *stream) {
  int G = 0;
  embla_status st = check_shape(shape, &G, true);
  if (st != EMBLA_OK) return st;
  if (topk < 0 || recent < 0 || static_cast<int64_t>(topk) + recent > INT32_MAX ||
      idx_stride < topk + recent)
    return EMBLA_ERR_INVALID_ARG;
  const int64_t units = static_cast<int64_t>(shape->batch) * shape->n_q_heads;
  if (units == 0) return EMBLA_OK;
  const size_t ws_need = select_workspace_bytes(units, shape->ctx_len);
  if (!head_scores || !head_hist || !idx || !count || (ws_need && !workspace))
    return EMBLA_ERR_INVALID_ARG;
  if (!aligned16(head_scores) || !aligned16(head_hist) || !aligned16(idx) || !aligned16(count) ||
      (workspace && !aligned16(workspace)))
    return EMBLA_ERR_INVALID_ARG;
  if (workspace_bytes < ws_need) return EMBLA_ERR_WORKSPACE;
  uint32_t *flags = flags_ptr();
  if (!flags) return EMBLA_ERR_CUDA;
  const int sms = sm_count_of(current_device());
  if (sms <= 0) return EMBLA_ERR_CUDA;
  return cuda_status(launch_select(head_scores, head_hist, units, shape->ctx_len,
                                   shape->cache_stride, topk, recent, idx, idx_stride, count,
                                   workspace, flags, sms, static_cast<cudaStream_t>(stream)));
}

size_t embla_sparse_decode_workspace_size(const embla_shape *shape, int32_t idx_stride) {
  int G = 0;
  if (check_shape(shape, &G, true) != EMBLA_OK || idx_stride < 0) return 0;
  return sparse_workspace_bytes(static_cast<int64_t>(shape->batch) * shape->n_kv_heads, G,
                                idx_stride);
}

}  // extern "C"

namespace {

embla_status sparse_decode_impl(const embla_shape *shape, const void *q, const void *k_cache,
                                const float *k_scales, const void *v_cache,
                                const float *v_scales, bool kv8, const int32_t *idx,
                                int32_t idx_stride, const int32_t *count, float tau, float *out,
                                void *workspace, size_t workspace_bytes, void *stream,
                                bool per_head = false) {
  int G = 0;
  embla_status st = check_shape(shape, &G, true);
  if (st != EMBLA_OK) return st;
  if (!finite(tau) || idx_stride < 0) return EMBLA_ERR_INVALID_ARG;
  const int64_t units = static_cast<int64_t>(shape->batch) *
                       (per_head ? shape->n_q_heads : shape->n_kv_heads);
  if (units == 0) return EMBLA_OK;
  if (!q || !k_cache || !v_cache || !idx || !count || !out || !workspace)
    return EMBLA_ERR_INVALID_ARG;
  if (kv8 && (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales)))
    return EMBLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(workspace) || !aligned16(idx) || !aligned16(count))
    return EMBLA_ERR_INVALID_ARG;
  if (workspace_bytes < sparse_workspace_bytes(units, G, idx_stride)) return EMBLA_ERR_WORKSPACE;
  uint32_t *flags = flags_ptr();
  if (!flags) return EMBLA_ERR_CUDA;
  const int sms = sm_count_of(current_device());
  if (sms <= 0) return EMBLA_ERR_CUDA;
  return cuda_status(launch_sparse_decode(G, per_head, shape->n_q_heads, q, k_cache, v_cache,
                                          kv8 ? k_scales : nullptr,
                                          kv8 ? v_scales : nullptr, idx, idx_stride, count,
                                          units, shape->n_kv_heads, shape->ctx_len,
                                          shape->cache_stride, tau, out, workspace, flags, sms,
                                          static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

embla_status embla_sparse_decode(const embla_shape *shape, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *idx, int32_t idx_stride,
                                 const int32_t *count, float tau, float *out, void *workspace,
                                 size_t workspace_bytes, void *stream) {
  return sparse_decode_impl(shape, q, k_cache, nullptr, v_cache, nullptr, false, idx, idx_stride,
                            count, tau, out, workspace, workspace_bytes, stream);
}

embla_status embla_sparse_decode_per_head(const embla_shape *shape, const void *q,
                                          const void *k_cache, const void *v_cache,
                                          const int32_t *idx, int32_t idx_stride,
                                          const int32_t *count, float tau, float *out,
                                          void *workspace, size_t workspace_bytes, void *stream) {
  return sparse_decode_impl(shape, q, k_cache, nullptr, v_cache, nullptr, false, idx, idx_stride,
                            count, tau, out, workspace, workspace_bytes, stream, true);
}

embla_status embla_sparse_decode_e4m3(const embla_shape *shape, const void *q,
                                      const uint8_t *k_codes, const float *k_scales,
                                      const uint8_t *v_codes, const float *v_scales,
                                      const int32_t *idx, int32_t idx_stride,
                                      const int32_t *count, float tau, float *out,
                                      void *workspace, size_t workspace_bytes, void *stream) {
  return sparse_decode_impl(shape, q, k_codes, k_scales, v_codes, v_scales, true, idx,
                            idx_stride, count, tau, out, workspace, workspace_bytes, stream);
}

size_t embla_prefill_workspace_size(const embla_shape *shape) {
  int G = 0;
  if (check_shape(shape, &G, true) != EMBLA_OK) return 0;
  return prefill_workspace_bytes(static_cast<int64_t>(shape->batch) * shape->n_kv_heads,
                                 shape->ctx_len);
}

embla_status embla_prefill(const embla_shape *shape, int64_t n_new, const void *q,
                           const void *k_cache, const void *v_cache, float alpha, float c,
                           float eps, float *out, void *workspace, size_t workspace_bytes,
                           void *stream) {
  int G = 0;
  embla_status st = check_shape(shape, &G, true);
  if (st != EMBLA_OK) return st;
  if (n_new < 0 || n_new > shape->ctx_len) return EMBLA_ERR_INVALID_ARG;
  if (!(finite(alpha) && alpha > 0.0f) || !(finite(c) && c >= 0.0f) ||
      !(finite(eps) && eps >= 0.0f))
    return EMBLA_ERR_INVALID_ARG;
  const int64_t units = static_cast<int64_t>(shape->batch) * shape->n_kv_heads;
  if (units == 0 || n_new == 0) return EMBLA_OK;
  if (!q || !k_cache || !v_cache || !out || !workspace) return EMBLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      !aligned16(workspace))
    return EMBLA_ERR_INVALID_ARG;
  // TMA coordinates are 32-bit; one CTA per (sequence, head, 128 prompt tokens)
  const int64_t bh = static_cast<int64_t>(shape->batch) * shape->n_q_heads;
  if (shape->ctx_len > INT32_MAX - 256 || bh > INT32_MAX || bh * ((n_new + 127) / 128) > INT32_MAX)
    return EMBLA_ERR_UNSUPPORTED;
  if (workspace_bytes < prefill_workspace_bytes(units, shape->ctx_len)) return EMBLA_ERR_WORKSPACE;
  uint32_t *flags = flags_ptr();
  if (!flags) return EMBLA_ERR_CUDA;
  float *rk = static_cast<float *>(workspace);
  CUtensorMap tm_q, tm_k, tm_v, tm_rk;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return EMBLA_ERR_CUDA;
  const cuuint64_t rdims[2] = {static_cast<cuuint64_t>(shape->ctx_len), static_cast<cuuint64_t>(units)};
  const cuuint64_t rstrides[1] = {static_cast<cuuint64_t>(prefill_rk_stride(shape->ctx_len)) * 4};
  const cuuint32_t rbox[2] = {128u, 1u};
  const cuuint32_t restr[2] = {1u, 1u};
  if (!encode_planes(&tm_q, q, static_cast<uint64_t>(n_new), static_cast<uint64_t>(n_new),
                     static_cast<uint64_t>(bh)) ||
      !encode_planes(&tm_k, k_cache, static_cast<uint64_t>(shape->ctx_len),
                     static_cast<uint64_t>(shape->cache_stride), static_cast<uint64_t>(units)) ||
      !encode_planes(&tm_v, v_cache, static_cast<uint64_t>(shape->ctx_len),
                     static_cast<uint64_t>(shape->cache_stride), static_cast<uint64_t>(units)) ||
      fn(&tm_rk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, rk, rdims, rstrides, rbox, restr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return EMBLA_ERR_CUDA;
  const int sms = sm_count_of(current_device());
  if (sms <= 0) return EMBLA_ERR_CUDA;
  return cuda_status(launch_prefill(tm_q, tm_k, tm_v, tm_rk, k_cache, rk, out, flags, shape->batch,
                                    shape->n_q_heads, shape->n_kv_heads, shape->ctx_len, n_new,
                                    shape->cache_stride, alpha, c, eps, sms,
                                    static_cast<cudaStream_t>(stream)));
}

size_t embla_relu2_mlp_workspace_size(int64_t d, int64_t f) {
  const int sms = sm_count_of(current_device());
  if (sms <= 0 || d < 1 || f < 1) return 0;
  return mlp_workspace_bytes(d, f, sms);
}

embla_status embla_relu2_mlp(int64_t d, int64_t f, const void *x, const void *w_up,
                             const void *w_down, float *y, int32_t *n_live, void *workspace,
                             size_t workspace_bytes, void *stream) {
  if (d != 512 && d != 1024 && d != 2048) return d < 1 ? EMBLA_ERR_INVALID_ARG : EMBLA_ERR_UNSUPPORTED;
  if (f < 1 || f > (static_cast<int64_t>(1) << 30)) return EMBLA_ERR_INVALID_ARG;
  if (!x || !w_up || !w_down || !y || !n_live || !workspace) return EMBLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(y) ||
      !aligned16(n_live) || !aligned16(workspace))
    return EMBLA_ERR_INVALID_ARG;
  const int sms = sm_count_of(current_device());
  if (sms <= 0) return EMBLA_ERR_CUDA;
  if (workspace_bytes < mlp_workspace_bytes(d, f, sms)) return EMBLA_ERR_WORKSPACE;
  return cuda_status(launch_relu2_mlp(x, w_up, w_down, d, f, y, n_live, workspace, sms,
                                      static_cast<cudaStream_t>(stream)));
}

size_t embla_window_decode_workspace_size(const embla_shape *shape, int32_t window) {
  (void)shape;
  (void)window;
  return 0;
}

embla_status embla_window_decode(const embla_shape *shape, const void *q, const void *k_win,
                                 const void *v_win, int32_t window, int64_t pos, float rope_base,
                                 float tau, float *out, void *workspace, size_t workspace_bytes,
                                 void *stream) {
  (void)workspace;
  (void)workspace_bytes;
  int G = 0;
  embla_status st = check_shape(shape, &G, false);
  if (st != EMBLA_OK) return st;
  if (window < 1 || window > 1024 || pos < 0 || !(finite(rope_base) && rope_base > 0.0f) ||
      !finite(tau))
    return EMBLA_ERR_INVALID_ARG;
  const int64_t units = static_cast<int64_t>(shape->batch) * shape->n_kv_heads;
  if (units == 0) return EMBLA_OK;
  if (!q || !k_win || !v_win || !out) return EMBLA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_win) || !aligned16(v_win) || !aligned16(out))
    return EMBLA_ERR_INVALID_ARG;
  return cuda_status(launch_window_decode(G, q, k_win, v_win, units, window, pos, rope_base, tau,
                                          out, static_cast<cudaStream_t>(stream)));
}

embla_status embla_skip_stats(const embla_shape *shape, const float *sel_scores, int32_t chunk,
                              int32_t *keys_needed, int32_t *chunks_needed, void *stream) {
  int G = 0;
  embla_status st = check_shape(shape, &G, true);
  if (st != EMBLA_OK) return st;
  if (chunk < 1 || chunk > 1024 || (chunk & (chunk - 1)) != 0) return EMBLA_ERR_INVALID_ARG;
  const int64_t units = static_cast<int64_t>(shape->batch) * shape->n_kv_heads;
  if (units == 0) return EMBLA_OK;
  if (!sel_scores || !keys_needed || !chunks_needed) return EMBLA_ERR_INVALID_ARG;
  if (!aligned16(sel_scores) || !aligned16(keys_needed) || !aligned16(chunks_needed))
    return EMBLA_ERR_INVALID_ARG;
  return cuda_status(launch_skip_stats(sel_scores, units, shape->ctx_len, shape->cache_stride,
                                       chunk, keys_needed, chunks_needed,
                                       static_cast<cudaStream_t>(stream)));
}

embla_status embla_append_kv(const embla_shape *shape, int64_t pos, const void *k_rows,
                             const void *v_rows, void *k_cache, void *v_cache, void *stream) {
  int G = 0;
  embla_status st = check_shape(shape, &G, false);
  if (st != EMBLA_OK) return st;
  if (shape->cache_stride < 1 || pos < 0 || pos >= shape->cache_stride)
    return EMBLA_ERR_INVALID_ARG;
  const int64_t units = static_cast<int64_t>(shape->batch) * shape->n_kv_heads;
  if (units == 0) return EMBLA_OK;
  if (!k_rows || !v_rows || !k_cache || !v_cache) return EMBLA_ERR_INVALID_ARG;
  const int64_t rb = 2 * kHeadDim;
  const AppendJob jobs[2] = {
      {static_cast<const uint8_t *>(k_rows), static_cast<uint8_t *>(k_cache), rb, shape->cache_stride, 0},
      {static_cast<const uint8_t *>(v_rows), static_cast<uint8_t *>(v_cache), rb, shape->cache_stride, 0}};
  return cuda_status(launch_append_rows(jobs, 2, units, pos, static_cast<cudaStream_t>(stream)));
}

embla_status embla_append_kv_e4m3(const embla_shape *shape, int64_t pos, const uint8_t *k_code_rows,
                                  const float *k_scale_rows, const uint8_t *v_code_rows,
                                  const float *v_scale_rows, uint8_t *k_codes, float *k_scales,
                                  uint8_t *v_codes, float *v_scales, void *stream) {
  int G = 0;
  embla_status st = check_shape(shape, &G, false);
  if (st != EMBLA_OK) return st;
  if (shape->cache_stride < 1 || pos < 0 || pos >= shape->cache_stride)
    return EMBLA_ERR_INVALID_ARG;
  const int64_t units = static_cast<int64_t>(shape->batch) * shape->n_kv_heads;
  if (units == 0) return EMBLA_OK;
  if (!k_code_rows || !k_scale_rows || !v_code_rows || !v_scale_rows || !k_codes || !k_scales ||
      !v_codes || !v_scales)
    return EMBLA_ERR_INVALID_ARG;
  const int64_t ncap = shape->cache_stride;
  const AppendJob jobs[4] = {
      {k_code_rows, k_codes, kHeadDim, ncap, 0},
      {v_code_rows, v_codes, kHeadDim, ncap, 0},
      {reinterpret_cast<const uint8_t *>(k_scale_rows), reinterpret_cast<uint8_t *>(k_scales), 4, ncap, 0},
      {reinterpret_cast<const uint8_t *>(v_scale_rows), reinterpret_cast<uint8_t *>(v_scales), 4, ncap, 0}};
  return cuda_status(launch_append_rows(jobs, 4, units, pos, static_cast<cudaStream_t>(stream)));
}

embla_status embla_self_test_wait_limit(uint32_t limit_us, int arrive, void *stream) {
  if (limit_us == 0 || limit_us > 1000000u) return EMBLA_ERR_INVALID_ARG;
  uint32_t *d = flags_ptr();
  if (!d) return EMBLA_ERR_CUDA;
  wait_limit_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      d, static_cast<uint64_t>(limit_us) * 1000ull, arrive);
  return cuda_status(cudaGetLastError());
}

embla_status embla_device_check(uint32_t *flags, int clear, void *stream) {
  uint32_t *d = flags_ptr();
  if (!d || !flags) return d ? EMBLA_ERR_INVALID_ARG : EMBLA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, d, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return EMBLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return EMBLA_ERR_CUDA;
  if (clear && v) {
    if (cudaMemsetAsync(d, 0, sizeof(uint32_t), s) != cudaSuccess) return EMBLA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return EMBLA_ERR_CUDA;
  }
  *flags = v;
  return v ? EMBLA_ERR_DEVICE_CHECK : EMBLA_OK;
}

}  // extern "C"
