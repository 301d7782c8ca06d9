// Full (ReLU^2) layer decode for one decode token per sequence.
//
// Source: "The Architecture of Embla 1", sections "Sevren Sparse Attention learns
// to be sparse" (weights ReLU(s)^2 of scores between RMS-normalised query and key,
// divided by a constant plus the sum of weights) and "Skipping V" (a value row is
// read only when some query head of the KV group gives its key a weight above zero).
//
// One persistent CTA per SM walks a contiguous run of 128-key tiles of the
// flattened (unit, tile) sequence, unit = (batch, KV head).  Warp roles:
//   warp 0   TMA producer: 32 KB K tiles (two 64-column boxes, 128-byte swizzle)
//            into a 4-stage ring; the unit's G query rows when the unit changes.
//   warp 1   tcgen05 issuer: D[128 keys x 16] = K_tile . Q^T (raw bf16 operands,
//            fp32 accumulation in tensor memory, double-buffered columns).
//   warps 2-5  epilogue, one thread per key: reads its G dot products from tensor
//            memory and its key row from shared memory (sum of squares), forms
//            s_h = dot_h * alpha*rq_h * rk, sigma = max_h s_h, writes sigma and the
//            2048-bin histogram of its order key, compacts the keys with sigma > 0
//            and fetches only their V rows with bulk copies.
//   warps 6-9  V accumulators: num_h += w_h v, den_h += w_h over the fetched rows;
//            at the end of each stretch of a unit they write a partial record.
// A second kernel sums the partial records of each unit and divides.
#include "internal.h"
#include "ptx.cuh"

namespace embla {
namespace {

constexpr int kStages = 4;
constexpr int kVSlots = 4;
constexpr int kVRows = 32;                         // V rows per batch
constexpr int kRowBytes = kHeadDim * 2;            // 256
constexpr int kTileBytes = kTileKeys * kRowBytes;  // 32 KB
constexpr int kHalfBytes = kTileBytes / 2;         // 128 rows x 64 dims
constexpr int kQBufBytes = 4096;                   // 16 rows x 128 dims (MMA N = 16)
constexpr int kQHalfBytes = kQBufBytes / 2;
constexpr int kThreads = 320;
constexpr int kMmaN = 16;
constexpr uint32_t kIdesc = idesc_bf16_f32(128, kMmaN);
constexpr int kFlagFlush = 1, kFlagDone = 2;
constexpr int kEpiBarrier = 1;

template <int G>
struct VMeta {
  int32_t cnt, flags, unit, rec;
  int32_t seg_surv, pad0, pad1, pad2;
  int32_t key[kVRows];
  float w[kVRows][G];
};

template <int G>
struct Smem {
  static constexpr int k_off = 0;
  static constexpr int q_off = k_off + kStages * kTileBytes;
  static constexpr int v_off = q_off + 2 * kQBufBytes;
  static constexpr int meta_off = v_off + kVSlots * kVRows * kRowBytes;
  static constexpr int hist_off = meta_off + kVSlots * static_cast<int>(sizeof(VMeta<G>));
  static constexpr int aq_off = hist_off + kHistBins * 4;
  static constexpr int misc_off = aq_off + 2 * 16 * 4;
  static constexpr int bar_off = misc_off + 64;
  static constexpr int n_bars = 2 * kStages + 8 + 2 * kVSlots;
  static constexpr int total = bar_off + n_bars * 8;
  static constexpr int alloc = total + 1024;  // room to align the base to 1024
};

struct FullParams {
  const uint8_t *v;  // V cache
  float *sel;        // selection scores or null
  uint32_t *hist;    // selection histogram or null
  float *rec;        // partial records
  uint32_t *flags;
  int64_t T, TU, n, ncap;
  int32_t P, Hq, Hkv, rec_stride;
  float alpha, eps;
};

__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float sumsq8(const uint4 &v) {
  float s = 0.0f;
  s = fmaf(bf16lo(v.x), bf16lo(v.x), s);
  s = fmaf(bf16hi(v.x), bf16hi(v.x), s);
  s = fmaf(bf16lo(v.y), bf16lo(v.y), s);
  s = fmaf(bf16hi(v.y), bf16hi(v.y), s);
  s = fmaf(bf16lo(v.z), bf16lo(v.z), s);
  s = fmaf(bf16hi(v.z), bf16hi(v.z), s);
  s = fmaf(bf16lo(v.w), bf16lo(v.w), s);
  s = fmaf(bf16hi(v.w), bf16hi(v.w), s);
  return s;
}

__device__ __forceinline__ void set_abort(volatile int *abort_flag, uint32_t *flags) {
  *abort_flag = 1;
  atomicOr(flags, kFlagWaitTimeout);
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    full_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_q, const FullParams p) {
  using L = Smem<G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sK = smem + L::k_off;
  uint8_t *sQ = smem + L::q_off;
  uint8_t *sV = smem + L::v_off;
  VMeta<G> *meta = reinterpret_cast<VMeta<G> *>(smem + L::meta_off);
  uint32_t *s_hist = reinterpret_cast<uint32_t *>(smem + L::hist_off);
  float *s_aq = reinterpret_cast<float *>(smem + L::aq_off);
  int *misc = reinterpret_cast<int *>(smem + L::misc_off);
  int *s_wcnt = misc;                                   // [4] survivors per TMEM quarter
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(misc + 4);
  volatile int *s_abort = misc + 5;
  volatile int *s_k_issued = misc + 6;
  volatile int *s_vb_total = misc + 7;
  volatile int *s_q_issued = misc + 8;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off);
  uint64_t *full = bars;
  uint64_t *empty = full + kStages;
  uint64_t *accf = empty + kStages;
  uint64_t *acce = accf + 2;
  uint64_t *qfull = acce + 2;
  uint64_t *qempty = qfull + 2;
  uint64_t *vfull = qempty + 2;
  uint64_t *vempty = vfull + kVSlots;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t cta = blockIdx.x;
  const int64_t tb = split_first_tile(cta, p.T, p.P);
  const int64_t te = split_first_tile(cta + 1, p.T, p.P);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf[a], 1);
      mbar_init(&acce[a], 4);
      mbar_init(&qfull[a], 1);
      mbar_init(&qempty[a], 2);
    }
    for (int v = 0; v < kVSlots; ++v) {
      mbar_init(&vfull[v], 1);
      mbar_init(&vempty[v], 4);
    }
    *s_abort = 0;
    *s_k_issued = 0;
    *s_vb_total = 0;
    *s_q_issued = 0;
    fence_barrier_init();
  }
  // Rows G..15 of the query operand feed only MMA columns that are never read; zero
  // them anyway so no stale bits reach the tensor core.
  for (int i = threadIdx.x; i < 2 * kQBufBytes / 16; i += kThreads)
    reinterpret_cast<uint4 *>(sQ)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < kHistBins; i += kThreads) s_hist[i] = 0u;
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(s_tmem, 32);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(s_tmem);

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_q);
      const uint64_t policy = policy_evict_first();
      int64_t cur_u = -1;
      int seg = -1;
      int64_t i = 0;
      for (int64_t t = tb; t < te; ++t, ++i) {
        if (*s_abort) break;
        const int64_t u = t / p.TU;
        const int64_t tl = t - u * p.TU;
        if (u != cur_u) {
          cur_u = u;
          ++seg;
          const int qb = seg & 1;
          if (seg >= 2 && !mbar_wait(&qempty[qb], ((seg >> 1) - 1) & 1)) {
            set_abort(s_abort, p.flags);
            break;
          }
          mbar_arrive_expect_tx(&qfull[qb], 2 * G * 128);
          const int32_t qrow = static_cast<int32_t>((u / p.Hkv) * p.Hq + (u % p.Hkv) * G);
          tma_load_2d(sQ + qb * kQBufBytes, &tm_q, &qfull[qb], 0, qrow);
          tma_load_2d(sQ + qb * kQBufBytes + kQHalfBytes, &tm_q, &qfull[qb], 64, qrow);
          *s_q_issued = seg + 1;
        }
        const int s = static_cast<int>(i % kStages);
        if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) - 1) & 1)) {
          set_abort(s_abort, p.flags);
          break;
        }
        mbar_arrive_expect_tx(&full[s], kTileBytes);
        const int32_t row = static_cast<int32_t>(u * p.ncap + tl * kTileKeys);
        tma_load_2d_hint(sK + s * kTileBytes, &tm_k, &full[s], 0, row, policy);
        tma_load_2d_hint(sK + s * kTileBytes + kHalfBytes, &tm_k, &full[s], 64, row, policy);
        *s_k_issued = static_cast<int>(i + 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int64_t cur_u = -1;
      int seg = -1, qb = 0;
      int64_t i = 0, issued = 0;
      for (int64_t t = tb; t < te; ++t, ++i) {
        if (*s_abort) break;
        const int64_t u = t / p.TU;
        if (u != cur_u) {
          cur_u = u;
          ++seg;
          qb = seg & 1;
          if (!mbar_wait(&qfull[qb], (seg >> 1) & 1)) {
            set_abort(s_abort, p.flags);
            break;
          }
        }
        const int s = static_cast<int>(i % kStages);
        const int a = static_cast<int>(i & 1);
        if (!mbar_wait(&full[s], (i / kStages) & 1) ||
            (i >= 2 && !mbar_wait(&acce[a], ((i >> 1) - 1) & 1))) {
          set_abort(s_abort, p.flags);
          break;
        }
        tc_fence_after_sync();
        const uint32_t kaddr = smem_u32(sK + s * kTileBytes);
        const uint32_t qaddr = smem_u32(sQ + qb * kQBufBytes);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint64_t adesc = smem_desc_sw128(kaddr + (kk >> 2) * kHalfBytes + (kk & 3) * 32);
          const uint64_t bdesc = smem_desc_sw128(qaddr + (kk >> 2) * kQHalfBytes + (kk & 3) * 32);
          tc_mma_bf16(tmem + a * kMmaN, adesc, bdesc, kIdesc, kk > 0 ? 1u : 0u);
        }
        tc_commit(&accf[a]);
        issued = i + 1;
        const bool seg_end = (t + 1 == te) || ((t + 1) / p.TU != u);
        if (seg_end) tc_commit(&qempty[qb]);
      }
      // the accumulator must be idle before the tensor memory is released
      if (issued > 0) mbar_wait(&accf[(issued - 1) & 1], ((issued - 1) >> 1) & 1);
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;  // 0..127
    const int ew = warp - 2;          // epilogue warp 0..3
    const int quarter = warp & 3;     // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;
    const uint32_t lanemask_lt = (1u << lane) - 1u;
    float aq[G];
#pragma unroll
    for (int h = 0; h < G; ++h) aq[h] = 0.0f;
    int64_t cur_u = -1;
    int seg = -1;
    int64_t i = 0, vb = 0;
    int seg_surv = 0;
    for (int64_t t = tb; t < te; ++t, ++i) {
      const int64_t u = t / p.TU;
      const int64_t tl = t - u * p.TU;
      if (u != cur_u) {
        cur_u = u;
        ++seg;
        seg_surv = 0;
        const int qb = seg & 1;
        bool ok = mbar_wait(&qfull[qb], (seg >> 1) & 1);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) {
          for (int h = ew; h < G; h += 4) {
            float ss = 0.0f;
            if (lane < 16) {
              const uint4 v = *reinterpret_cast<const uint4 *>(
                  sQ + qb * kQBufBytes + (lane >> 3) * kQHalfBytes + h * 128 + (lane & 7) * 16);
              ss = sumsq8(v);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) s_aq[qb * 16 + h] = p.alpha * rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
          }
        }
        if (bar_red_or(kEpiBarrier, 128, !ok || *s_abort)) {
          if (!ok) set_abort(s_abort, p.flags);
          break;
        }
#pragma unroll
        for (int h = 0; h < G; ++h) aq[h] = s_aq[qb * 16 + h];
        if (et == 0) mbar_arrive(&qempty[qb]);
      }
      const int s = static_cast<int>(i % kStages);
      const int a = static_cast<int>(i & 1);
      bool ok = mbar_wait(&accf[a], (i >> 1) & 1) && mbar_wait(&full[s], (i / kStages) & 1);
      ok = __all_sync(0xffffffffu, ok);
      float dot[G];
      float ss = 0.0f;
#pragma unroll
      for (int h = 0; h < G; ++h) dot[h] = 0.0f;
      if (ok) {
        tc_fence_after_sync();
        const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + a * kMmaN;
        if constexpr (G == 4) {
          uint32_t r[4];
          tmem_load_x4(taddr, r);
          tmem_wait_ld(r);
#pragma unroll
          for (int h = 0; h < 4; ++h) dot[h] = __uint_as_float(r[h]);
        } else {
          uint32_t r[8];
          tmem_load_x8(taddr, r);
          tmem_wait_ld(r);
#pragma unroll
          for (int h = 0; h < 8; ++h) dot[h] = __uint_as_float(r[h]);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acce[a]);
        // this key's sum of squares; chunk order rotated by row so 8 neighbouring
        // rows hit 8 different bank groups (the swizzle permutes chunks within a row)
        const uint8_t *rowp = sK + s * kTileBytes + row * 128;
        float ss0 = 0.0f, ss1 = 0.0f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int pc = (c ^ (row & 7)) * 16;
          ss0 += sumsq8(*reinterpret_cast<const uint4 *>(rowp + pc));
          ss1 += sumsq8(*reinterpret_cast<const uint4 *>(rowp + kHalfBytes + pc));
        }
        ss = ss0 + ss1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
      const int64_t j = tl * kTileKeys + row;
      const bool valid = ok && j < p.n;
      const float rk = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
      float sc[G];
      float sigma = -INFINITY;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        sc[h] = dot[h] * aq[h] * rk;
        sigma = fmaxf(sigma, sc[h]);
      }
      if (valid && p.sel != nullptr) {
        p.sel[u * p.ncap + j] = sigma;
        atomicAdd(&s_hist[order_key(sigma) >> 21], 1u);
      }
      const bool surv = valid && sigma > 0.0f;
      const uint32_t bal = __ballot_sync(0xffffffffu, surv);
      if (lane == 0) s_wcnt[quarter] = __popc(bal);
      if (bar_red_or(kEpiBarrier, 128, !ok || *s_abort)) {
        if (!ok) set_abort(s_abort, p.flags);
        break;
      }
      int off = 0, m = 0;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int cq = s_wcnt[q4];
        off += (q4 < quarter) ? cq : 0;
        m += cq;
      }
      seg_surv += m;
      const bool seg_end = (t + 1 == te) || ((t + 1) / p.TU != u);
      const bool last = (t + 1 == te);
      int nb = (m + kVRows - 1) / kVRows;
      if (seg_end && nb == 0) nb = 1;
      bool ok2 = true;
      for (int k = 0; k < nb; ++k) {
        const int64_t vbk = vb + k;
        if (vbk >= kVSlots)
          ok2 = ok2 && mbar_wait(&vempty[vbk % kVSlots], ((vbk / kVSlots) - 1) & 1);
      }
      if (ok2 && surv) {
        const int pos = off + __popc(bal & lanemask_lt);
        VMeta<G> &mt = meta[(vb + pos / kVRows) % kVSlots];
        const int e = pos % kVRows;
        mt.key[e] = static_cast<int32_t>(j);
#pragma unroll
        for (int h = 0; h < G; ++h) mt.w[e][h] = sc[h] > 0.0f ? sc[h] * sc[h] : 0.0f;
      }
      if (bar_red_or(kEpiBarrier, 128, !ok2 || *s_abort)) {
        if (!ok2) set_abort(s_abort, p.flags);
        break;
      }
      if (ew < nb) {
        const int slot = static_cast<int>((vb + ew) % kVSlots);
        VMeta<G> &mt = meta[slot];
        const int cnt = min(kVRows, max(0, m - ew * kVRows));
        if (lane == 0) {
          mt.cnt = cnt;
          mt.flags = (ew == nb - 1) ? ((seg_end ? kFlagFlush : 0) | (last ? kFlagDone : 0)) : 0;
          mt.unit = static_cast<int32_t>(u);
          mt.rec = static_cast<int32_t>(cta + u);
          mt.seg_surv = seg_surv;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(&vfull[slot], cnt * kRowBytes);
        __syncwarp();
        if (lane < cnt) {
          const int64_t jj = mt.key[lane];
          bulk_load(sV + slot * (kVRows * kRowBytes) + lane * kRowBytes,
                    p.v + (u * p.ncap + jj) * kRowBytes, kRowBytes, &vfull[slot]);
        }
      }
      vb += nb;
      if (et == 0) *s_vb_total = static_cast<int>(vb);
      if (seg_end && p.sel != nullptr) {
        for (int bin = et; bin < kHistBins; bin += 128) {
          const uint32_t cnt = s_hist[bin];
          if (cnt) {
            atomicAdd(&p.hist[u * kHistBins + bin], cnt);
            s_hist[bin] = 0u;
          }
        }
        named_bar_sync(kEpiBarrier, 128);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ V accumulators
    constexpr int HPW = G / 4;  // heads per warp
    const int vw = warp - 6;
    const int d0 = lane * 4;
    float acc[HPW][4];
    float den[HPW];
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
      den[hh] = 0.0f;
#pragma unroll
      for (int d = 0; d < 4; ++d) acc[hh][d] = 0.0f;
    }
    for (int64_t vb = 0;; ++vb) {
      const int slot = static_cast<int>(vb % kVSlots);
      bool ok = !*s_abort && mbar_wait(&vfull[slot], (vb / kVSlots) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        set_abort(s_abort, p.flags);
        break;
      }
      const VMeta<G> &mt = meta[slot];
      const int cnt = mt.cnt, flags = mt.flags, rec = mt.rec, seg_surv = mt.seg_surv;
      const uint8_t *vd = sV + slot * (kVRows * kRowBytes) + lane * 8;
      for (int e = 0; e < cnt; ++e) {
        const uint2 raw = *reinterpret_cast<const uint2 *>(vd + e * kRowBytes);
        const float v0 = bf16lo(raw.x), v1 = bf16hi(raw.x), v2 = bf16lo(raw.y),
                    v3 = bf16hi(raw.y);
#pragma unroll
        for (int hh = 0; hh < HPW; ++hh) {
          const float w = mt.w[e][vw + 4 * hh];
          acc[hh][0] = fmaf(w, v0, acc[hh][0]);
          acc[hh][1] = fmaf(w, v1, acc[hh][1]);
          acc[hh][2] = fmaf(w, v2, acc[hh][2]);
          acc[hh][3] = fmaf(w, v3, acc[hh][3]);
          den[hh] += w;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&vempty[slot]);
      if (flags & kFlagFlush) {
        float *r = p.rec + static_cast<int64_t>(rec) * p.rec_stride;
#pragma unroll
        for (int hh = 0; hh < HPW; ++hh) {
          const int h = vw + 4 * hh;
          *reinterpret_cast<float4 *>(r + h * kHeadDim + d0) =
              make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
          if (lane == 0) r[G * kHeadDim + h] = den[hh];
          den[hh] = 0.0f;
          acc[hh][0] = acc[hh][1] = acc[hh][2] = acc[hh][3] = 0.0f;
        }
        if (vw == 0 && lane == 0) reinterpret_cast<int32_t *>(r)[G * kHeadDim + G] = seg_surv;
      }
      if (flags & kFlagDone) break;
    }
    __syncwarp();
  }

  __syncthreads();
  if (threadIdx.x == 0) {
    // No copy may still be landing in shared memory when the CTA leaves: wait (bounded)
    // for the last armed phase of every barrier that a copy completes.
    const int k_issued = *s_k_issued, vb_total = *s_vb_total, q_issued = *s_q_issued;
    for (int s = 0; s < kStages; ++s) {
      const int uses = k_issued > s ? (k_issued - 1 - s) / kStages + 1 : 0;
      if (uses) mbar_wait(&full[s], (uses - 1) & 1);
    }
    for (int v = 0; v < kVSlots; ++v) {
      const int uses = vb_total > v ? (vb_total - 1 - v) / kVSlots + 1 : 0;
      if (uses) mbar_wait(&vfull[v], (uses - 1) & 1);
    }
    for (int q = 0; q < 2; ++q) {
      const int uses = q_issued > q ? (q_issued - 1 - q) / 2 + 1 : 0;
      if (uses) mbar_wait(&qfull[q], (uses - 1) & 1);
    }
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 32);
  }
}

template <int G>
__global__ void __launch_bounds__(256)
    full_combine_kernel(const float *__restrict__ rec, int rec_stride, int64_t T, int32_t P,
                        int64_t TU, float c, float *__restrict__ out, int32_t *__restrict__ n_surv) {
  const int64_t u = blockIdx.x;
  float *o = out + u * G * kHeadDim;
  if (TU == 0) {
    for (int i = threadIdx.x; i < G * kHeadDim; i += blockDim.x) o[i] = 0.0f;
    if (threadIdx.x == 0) n_surv[u] = 0;
    return;
  }
  const int64_t c0 = split_cta_of_tile(u * TU, T, P);
  const int64_t c1 = split_cta_of_tile(u * TU + TU - 1, T, P);
  for (int i = threadIdx.x; i < G * kHeadDim; i += blockDim.x) {
    const int h = i / kHeadDim;
    float num = 0.0f, den = 0.0f;
    for (int64_t cc = c0; cc <= c1; ++cc) {
      const float *r = rec + (cc + u) * rec_stride;
      num += r[i];
      den += r[G * kHeadDim + h];
    }
    const float z = c + den;
    o[i] = (z != 0.0f) ? num / z : 0.0f;
  }
  if (threadIdx.x == 0) {
    int32_t s = 0;
    for (int64_t cc = c0; cc <= c1; ++cc)
      s += reinterpret_cast<const int32_t *>(rec + (cc + u) * rec_stride)[G * kHeadDim + G];
    n_surv[u] = s;
  }
}

template <int G>
cudaError_t launch_full_decode_t(const CUtensorMap &tm_k, const CUtensorMap &tm_q,
                                 const FullParams &p, cudaStream_t stream) {
  const int smem = Smem<G>::alloc;
  cudaError_t e = cudaFuncSetAttribute(full_decode_kernel<G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  full_decode_kernel<G><<<p.P, kThreads, smem, stream>>>(tm_k, tm_q, p);
  return cudaGetLastError();
}

}  // namespace

FullSplit full_split(int64_t units, int64_t ctx_len, int sm_count) {
  FullSplit sp;
  sp.units = units;
  sp.tiles_per_unit = (ctx_len + kTileKeys - 1) / kTileKeys;
  sp.tiles = units * sp.tiles_per_unit;
  sp.ctas = static_cast<int32_t>(sp.tiles < sm_count ? sp.tiles : sm_count);
  return sp;
}

int full_record_floats(int G) {
  const int f = G * kHeadDim + G + 1;
  return (f + 3) & ~3;
}

size_t full_workspace_bytes(int64_t units, int G, int sm_count) {
  return static_cast<size_t>(units + sm_count) * full_record_floats(G) * sizeof(float);
}

cudaError_t launch_full_decode(int G, const CUtensorMap &tm_k, const CUtensorMap &tm_q,
                               const void *v_cache, float *sel_scores, uint32_t *sel_hist,
                               float *records, uint32_t *flags, const FullSplit &sp, int64_t n,
                               int64_t ncap, int Hq, int Hkv, float alpha, float eps,
                               cudaStream_t stream) {
  if (sp.tiles == 0) return cudaSuccess;
  FullParams p;
  p.v = static_cast<const uint8_t *>(v_cache);
  p.sel = sel_scores;
  p.hist = sel_hist;
  p.rec = records;
  p.flags = flags;
  p.T = sp.tiles;
  p.TU = sp.tiles_per_unit;
  p.n = n;
  p.ncap = ncap;
  p.P = sp.ctas;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.rec_stride = full_record_floats(G);
  p.alpha = alpha;
  p.eps = eps;
  if (G == 4) return launch_full_decode_t<4>(tm_k, tm_q, p, stream);
  if (G == 8) return launch_full_decode_t<8>(tm_k, tm_q, p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_full_combine(int G, const float *records, const FullSplit &sp, float c,
                                float *out, int32_t *n_surv, cudaStream_t stream) {
  if (sp.units == 0) return cudaSuccess;
  const int stride = full_record_floats(G);
  const dim3 grid(static_cast<unsigned>(sp.units));
  if (G == 4)
    full_combine_kernel<4><<<grid, 256, 0, stream>>>(records, stride, sp.tiles, sp.ctas,
                                                     sp.tiles_per_unit, c, out, n_surv);
  else if (G == 8)
    full_combine_kernel<8><<<grid, 256, 0, stream>>>(records, stride, sp.tiles, sp.ctas,
                                                     sp.tiles_per_unit, c, out, n_surv);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace embla
