// Causal full-layer (ReLU^2) attention over a prompt: the prefill of a full layer.
//
// Source: "The Architecture of Embla 1", sections "KV bridge, KV reuse, and prefill" (the
// early layers run on every prompt token) and "Sevren Sparse Attention learns to be sparse"
// (weights ReLU(s)^2 of scores between RMS-normalised query and key, divided by a constant
// plus the sum of weights).  A full layer has no position encoding, so the prompt token at
// position p (the T prompt tokens are keys n-T .. n-1 of the cache) sees keys 0 .. p.
//
// prefill_knorm_kernel: rk2[u][j] = 1 / (mean(k_j^2) + eps) for every key of every unit.
//
// prefill_kernel: one CTA per (sequence, query head, 128 prompt tokens), the tiles with the
// most keys first.  Warp roles:
//   warp 0     TMA producer: the 128 query rows once; per 128-key tile the K rows (two
//              64-column boxes, 128-byte swizzle), the tile's 128 key norms and the V rows,
//              each in a ring of 3.  Rows past n (and query rows past T) read as zeros.
//   warp 1     tcgen05 issuer of S = Q K^T (M 128 queries x N 128 keys, K 16 per step, fp32
//              in one of three tensor-memory buffers); S of tile t reuses the buffer of tile
//              t - 3 once its P V is done.
//   last warp  tcgen05 issuer of O += P V with P read from tensor memory (the same buffer,
//              where the epilogue wrote it over S) and V as an MN-major operand (the cached
//              rows as they lie), fp32 in tensor memory.  Two issuers, one commit per tile
//              each: S runs ahead of P V, and every commit costs the tensor pipe time.
//   warps 2..  epilogue, one thread per (query row, half of the tile's keys).  With
//              s = alpha rq rk dot, w = max(s, 0)^2 = a2 * w' where a2 = alpha^2 rq^2 is the
//              row's factor and w' = max(dot, 0)^2 * rk^2 (rq, rk > 0), so the row factor
//              is applied once at the end: out = a2 O' / (c + a2 den'), O' = sum w' v,
//              den' = sum w' over keys j <= p.  P = w' is written over the thread's own S
//              columns as two bf16 matrices hi = rn(w'), lo = rn(w' - hi), both multiplied
//              into O', so the weights keep about 16 bits, in the first key tile; as hi
//              alone (den' then sums hi) in the tiles after it.
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace embla {
namespace {

#ifndef EMBLA_PREFILL_EPI_WARPS
#define EMBLA_PREFILL_EPI_WARPS 8
#endif
constexpr int kEpiWarps = EMBLA_PREFILL_EPI_WARPS;  // a multiple of 4 (the lane quarters)
// P goes to the tensor cores as bf16 hi + lo for the first kLoTiles key tiles of a row
// block and as hi alone after them.  A row that reaches past the first tile has at least 128
// keys behind it, over which the rounding errors of hi (2^-9 of each weight, either sign)
// average out; the first tile's rows can have a handful of keys, where they would not.
#ifndef EMBLA_PREFILL_LO_TILES
#define EMBLA_PREFILL_LO_TILES 1
#endif
constexpr int kLoTiles = EMBLA_PREFILL_LO_TILES;
constexpr int kEpiParts = kEpiWarps / 4;          // threads per query row
constexpr int kEpiCols = 128 / kEpiParts;         // keys of a tile per epilogue thread
static_assert(kEpiWarps % 4 == 0 && (kEpiCols == 32 || kEpiCols == 64), "epilogue split");
constexpr int kWarpPV = 2 + kEpiWarps;           // the P V issuer (after the epilogue warps)
constexpr int kPThreads = (3 + kEpiWarps) * 32;
constexpr int kRing = 3;                 // K, V, key-norm stages and S/P buffers
constexpr int kBox = 128 * 128;          // one [128 rows][64 bf16] box, 16 KB
constexpr int kTileB = 2 * kBox;         // a 128 x 128 bf16 tile
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileB;
constexpr int kOffV = kOffK + kRing * kTileB;
constexpr int kOffRK = kOffV + kRing * kTileB;
constexpr int kOffBar = kOffRK + kRing * 128 * 4;
constexpr int kNBars = 1 + 7 * kRing + 3;
constexpr int kOffMisc = kOffBar + kNBars * 8;
constexpr int kPSmem = kOffMisc + 16 + 1024;  // + room to align the base to 1024
static_assert(kPSmem <= 227 * 1024, "shared memory per CTA");
constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128) | (1u << 16);  // B (V) MN-major
constexpr int kColO = kRing * 128, kPTmemCols = 512;
static_assert(kColO + 128 <= kPTmemCols, "tensor memory");

// Two fp32 lanes at once (Blackwell's paired fp32 pipe): a *= b, a += b, each lane rounded
// as the scalar operation would be.
__device__ __forceinline__ void mul_f32x2(float &a0, float &a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y;\n\t"
      "mov.b64 x, {%0, %1};\n\t"
      "mov.b64 y, {%2, %3};\n\t"
      "mul.rn.f32x2 x, x, y;\n\t"
      "mov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}
__device__ __forceinline__ void add_f32x2(float &a0, float &a1, float b0, float b1) {
  asm("{\n\t.reg .b64 x, y;\n\t"
      "mov.b64 x, {%0, %1};\n\t"
      "mov.b64 y, {%2, %3};\n\t"
      "add.rn.f32x2 x, x, y;\n\t"
      "mov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

struct PrefillParams {
  float *out;      // [B, Hq, T, D]
  uint32_t *flags;
  int64_t n, T;
  int32_t Hq, Hkv, BH, nqt, items;  // items = BH * nqt row blocks
  int32_t out32;                     // out is 32-byte aligned (32-byte stores)
  float alpha, c, eps;
};

// Row block number idx of the list ordered by key tiles, the most first: the last query
// tile of every (sequence, head), then the one before it, ...
struct RowBlock {
  int qt, bh, u, nkt;
  int64_t p0;  // position of query row 0
};
__device__ __forceinline__ RowBlock row_block(const PrefillParams &p, int idx) {
  RowBlock r;
  r.qt = p.nqt - 1 - idx / p.BH;
  r.bh = idx % p.BH;
  const int b = r.bh / p.Hq, h = r.bh % p.Hq;
  r.u = b * p.Hkv + h / (p.Hq / p.Hkv);
  r.p0 = p.n - p.T + static_cast<int64_t>(r.qt) * 128;
  const int64_t rows = p.T - static_cast<int64_t>(r.qt) * 128 < 128 ? p.T - static_cast<int64_t>(r.qt) * 128 : 128;
  r.nkt = static_cast<int>((r.p0 + rows - 1) / 128) + 1;  // key tiles up to the last row
  return r;
}

// The k-th row block of CTA c among G: the list taken a round of G at a time, alternate
// rounds in reverse order, so the CTAs' sums of key tiles stay close.  -1 past the end.
__device__ __forceinline__ int block_of(const PrefillParams &p, int k, int c, int G) {
  const int idx = k * G + ((k & 1) ? G - 1 - c : c);
  return idx < p.items ? idx : -1;
}

__device__ __forceinline__ void set_abort_p(volatile int *abort_flag, uint32_t *flags) {
  *abort_flag = 1;
  atomicOr(flags, kFlagWaitTimeout);
}

__global__ void __launch_bounds__(kPThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_rk,
                   const PrefillParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *sQ = smem + kOffQ;
  uint8_t *sK = smem + kOffK;
  uint8_t *sV = smem + kOffV;
  float *sRK = reinterpret_cast<float *>(smem + kOffRK);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint64_t *qfull = bars;
  // A K stage is free once its tile's S is done (sfull), a V stage once its P V is done
  // (pvdone): each MMA issuer commits once per tile.
  uint64_t *kfull = bars + 1;
  uint64_t *rkfull = kfull + kRing, *rkempty = rkfull + kRing;
  uint64_t *vfull = rkempty + kRing;
  uint64_t *sfull = vfull + kRing;    // S of a tile in tensor memory; its K stage free
  uint64_t *pfull = sfull + kRing;    // its P written over it
  uint64_t *pvdone = pfull + kRing;   // its P V done: the S/P buffer and the V stage are free
  uint64_t *ofull = pvdone + kRing;  // a row block's P V all done
  uint64_t *qempty = ofull + 1;      // its query rows no longer needed (S done, row norms read)
  uint64_t *ofree = qempty + 1;      // its O read out of tensor memory
  uint32_t *misc = reinterpret_cast<uint32_t *>(smem + kOffMisc);
  uint32_t *s_tmem = misc;
  volatile int *s_abort = reinterpret_cast<volatile int *>(misc + 1);
  volatile int *s_issued = reinterpret_cast<volatile int *>(misc + 2);   // tile loads issued
  volatile int *s_qissued = reinterpret_cast<volatile int *>(misc + 3);  // query loads issued

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);

  if (warp == 0) {
    // the barriers, by the warp's lanes side by side
    static_assert(kRing <= 32, "one stage per lane");
    if (lane < kRing) {
      mbar_init(&kfull[lane], 1);
      mbar_init(&rkfull[lane], 1);
      mbar_init(&rkempty[lane], kEpiWarps);
      mbar_init(&vfull[lane], 1);
      mbar_init(&sfull[lane], 1);
      mbar_init(&pfull[lane], kEpiWarps);
      mbar_init(&pvdone[lane], 1);
    }
    if (lane == 0) {
      mbar_init(qfull, 1);
      mbar_init(ofull, 1);
      mbar_init(qempty, 1 + kEpiWarps);  // the S issuer's commit + every epilogue warp
      mbar_init(ofree, kEpiWarps);
      *s_abort = 0;
      *s_issued = 0;
      *s_qissued = 0;
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kPTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(s_tmem);
  pdl_wait_primary();  // the key norms (and everything before) are complete
  pdl_launch_dependents();

  // Every role walks the CTA's row blocks in the same order (block_of), and their key tiles
  // through the rings by a running tile count g: stage g % kRing, phase (g / kRing) & 1.
  // Row block k's query and output barriers take phase k & 1.
  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_rk);
      int g = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = block_of(p, k, cta, G);
        if (idx < 0) break;
        const RowBlock rb = row_block(p, idx);
        // the query buffer is free once the previous block's S is done and its row norms
        // are read (early in that block: this load overlaps its key tiles)
        if (k > 0 && !mbar_wait(qempty, (k - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(qfull, kTileB);
        tma_load_3d(sQ, &tm_q, qfull, 0, rb.qt * 128, rb.bh);
        tma_load_3d(sQ + kBox, &tm_q, qfull, 64, rb.qt * 128, rb.bh);
        *s_qissued = k + 1;
        for (int kt = 0; kt < rb.nkt; ++kt, ++g) {
          const int s = g % kRing;
          const uint32_t ph = ((g / kRing) - 1) & 1;
          if (g >= kRing && !mbar_wait(&sfull[s], ph)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&kfull[s], kTileB);
          tma_load_3d(sK + s * kTileB, &tm_k, &kfull[s], 0, kt * 128, rb.u);
          tma_load_3d(sK + s * kTileB + kBox, &tm_k, &kfull[s], 64, kt * 128, rb.u);
          if (g >= kRing && !mbar_wait(&rkempty[s], ph)) {
            *s_issued = 3 * g + 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&rkfull[s], 128 * 4);
          tma_load_2d(sRK + s * 128, &tm_rk, &rkfull[s], kt * 128, rb.u);
          if (g >= kRing && !mbar_wait(&pvdone[s], ph)) {
            *s_issued = 3 * g + 2;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&vfull[s], kTileB);
          tma_load_3d(sV + s * kTileB, &tm_v, &vfull[s], 0, kt * 128, rb.u);
          tma_load_3d(sV + s * kTileB + kBox, &tm_v, &vfull[s], 64, kt * 128, rb.u);
          *s_issued = 3 * g + 3;
        }
      }
      if (!ok) set_abort_p(s_abort, p.flags);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------------ S issuer
    // S = Q K^T of every tile, as soon as its K stage has landed and its S/P buffer is free
    // (the P V of the tile three back is done); one commit per tile, and one per row block
    // after its last S (the query buffer is then free as far as the tensor cores go).
    if (lane == 0) {
      const uint64_t qdesc = smem_desc_sw128(smem_u32(sQ));
      const uint64_t kdesc = smem_desc_sw128(smem_u32(sK));
      int g = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = block_of(p, k, cta, G);
        if (idx < 0) break;
        const RowBlock rb = row_block(p, idx);
        ok = !*s_abort && mbar_wait(qfull, k & 1);
        for (int kt = 0; ok && kt < rb.nkt; ++kt, ++g) {
          const int sb = g % kRing;
          ok = mbar_wait(&kfull[sb], (g / kRing) & 1) &&
               (g < kRing || mbar_wait(&pvdone[sb], ((g / kRing) - 1) & 1));
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // dims 16kk..16kk+15: 32 bytes into a 128-byte row; dims 64.. start the second box
            const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kBox + (kk & 3) * 32) >> 4);
            tc_mma_bf16(tmem + sb * 128, qdesc + off,
                        kdesc + static_cast<uint64_t>((sb * kTileB) >> 4) + off, kIdescS,
                        kk > 0 ? 1u : 0u);
          }
          tc_commit(&sfull[sb]);
        }
        if (ok) tc_commit(qempty);
      }
      if (!ok) set_abort_p(s_abort, p.flags);
    }
    __syncwarp();
  } else if (warp == kWarpPV) {
    // ------------------------------------------------------------------ P V issuer
    // O += P V of every tile once its P is written and its V stage has landed (a row block's
    // first P V waits until the previous block's O has been read out); one commit per tile,
    // and one per row block after its last (its O is then complete).
    if (lane == 0) {
      int g = 0, blocks = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int idx = block_of(p, k, cta, G);
        if (idx < 0) break;
        const RowBlock rb = row_block(p, idx);
        ok = !*s_abort && (k == 0 || mbar_wait(ofree, (k - 1) & 1));
        for (int t = 0; ok && t < rb.nkt; ++t, ++g) {
          const int pb = g % kRing;
          ok = mbar_wait(&pfull[pb], (g / kRing) & 1) && mbar_wait(&vfull[pb], (g / kRing) & 1);
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            // keys 16kk..16kk+15: in the key group of kEpiCols keys holding them, hi takes
            // the first kEpiCols / 2 columns and lo the next; V rows 16kk.. (2 KB apart)
            const int grp = (16 * kk) / kEpiCols;
            const uint32_t a_hi = tmem + pb * 128 + grp * kEpiCols + ((16 * kk) % kEpiCols) / 2;
            const uint64_t vd = smem_desc_sw128_mn(smem_u32(sV + pb * kTileB + kk * 2048), kBox);
            tc_mma_bf16_tmem_a(tmem + kColO, a_hi, vd, kIdescPV, (t > 0 || kk > 0) ? 1u : 0u);
            if (t < kLoTiles) tc_mma_bf16_tmem_a(tmem + kColO, a_hi + kEpiCols / 2, vd, kIdescPV, 1u);
          }
          tc_commit(&pvdone[pb]);
        }
        if (ok) {
          tc_commit(ofull);
          blocks = k + 1;
        }
      }
      if (!ok) set_abort_p(s_abort, p.flags);
      // every MMA of this thread has completed before the tensor memory is released
      if (blocks > 0) mbar_wait(ofull, (blocks - 1) & 1);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3;          // the tensor-memory lanes this warp may read
    const int cg = (warp - 2) >> 2;        // keys kEpiCols cg .. of each tile
    const int r = quarter * 32 + lane;     // query row
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int g = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int idx = block_of(p, k, cta, G);
      if (idx < 0) break;
      const RowBlock rb = row_block(p, idx);
      const int64_t pos = rb.p0 + r;  // this row's position
      ok = !*s_abort && mbar_wait(qfull, k & 1);
      float a2 = 0.0f;  // alpha^2 / (mean(q^2) + eps)
      if (ok) {
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = 0.0f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          // chunk order rotated by row: 8 neighbouring rows read 8 different bank groups
          const int pc = (c ^ (r & 7)) * 16;
          const uint4 x0 = *reinterpret_cast<const uint4 *>(sQ + r * 128 + pc);
          const uint4 x1 = *reinterpret_cast<const uint4 *>(sQ + kBox + r * 128 + pc);
          sq_acc_bf16x2(x0.x, a[0], a[1]);
          sq_acc_bf16x2(x0.y, a[2], a[3]);
          sq_acc_bf16x2(x0.z, a[4], a[5]);
          sq_acc_bf16x2(x0.w, a[6], a[7]);
          sq_acc_bf16x2(x1.x, a[0], a[1]);
          sq_acc_bf16x2(x1.y, a[2], a[3]);
          sq_acc_bf16x2(x1.z, a[4], a[5]);
          sq_acc_bf16x2(x1.w, a[6], a[7]);
        }
        const float ss = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
        a2 = (p.alpha * p.alpha) / (ss * (1.0f / kHeadDim) + p.eps);
        // the query rows are read: every lane's sum depends on them
        const float used = __shfl_sync(0xffffffffu, ss, 0) + __shfl_sync(0xffffffffu, ss, 31);
        __syncwarp();
        if (lane == 0) mbar_arrive_after(qempty, used);
      }
      float den4[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // four chains of the row's weight sum
      for (int kt = 0; ok && kt < rb.nkt; ++kt, ++g) {
        const int sb = g % kRing;
        ok = mbar_wait(&sfull[sb], (g / kRing) & 1) && mbar_wait(&rkfull[sb], (g / kRing) & 1);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t cols = tmem + lane_base + sb * 128 + cg * kEpiCols;
        uint32_t acc[kEpiCols];
#pragma unroll
        for (int c = 0; c < kEpiCols; c += 32)
          tmem_load_x32(cols + c, *reinterpret_cast<uint32_t(*)[32]>(&acc[c]));
        tmem_wait_ld(acc);
        // squared key norms of these keys, read pair by pair as the weights need them (the
        // same for every lane: broadcast reads); the stage is handed back after the weights
        const float *rkp = sRK + sb * 128 + cg * kEpiCols;
        // keys past this row's position weigh nothing (only tiles that reach past row 0's
        // position need the test): key j0 + c is masked when c > lim
        const int64_t j0 = static_cast<int64_t>(kt) * 128 + cg * kEpiCols;
        const bool masked = j0 + kEpiCols - 1 > rb.p0;
        const int lim = masked ? static_cast<int>(pos - j0 < kEpiCols ? pos - j0 : kEpiCols) : kEpiCols;
        // P over this thread's own S columns (already read): kEpiCols / 2 columns of hi, then
        // (in the first kLoTiles tiles) as many of lo.  One code path per case keeps the
        // registers of each to what it needs.
        auto write_p = [&](auto with_lo, auto with_mask) {
          constexpr bool kLo = decltype(with_lo)::value;
          constexpr bool kMask = decltype(with_mask)::value;
          uint32_t hi[kEpiCols / 2], lo[kLo ? kEpiCols / 2 : 1];
#pragma unroll
          for (int c = 0; c < kEpiCols; c += 2) {
            // w = max(dot, 0)^2 * rk for keys c and c + 1, two lanes per instruction
            float w2[2] = {fmaxf(__uint_as_float(acc[c]), 0.0f), fmaxf(__uint_as_float(acc[c + 1]), 0.0f)};
            const float2 rk2 = *reinterpret_cast<const float2 *>(rkp + c);
            mul_f32x2(w2[0], w2[1], w2[0], w2[1]);
            mul_f32x2(w2[0], w2[1], rk2.x, rk2.y);
            if constexpr (kMask) {
              if (c > lim) w2[0] = 0.0f;
              if (c + 1 > lim) w2[1] = 0.0f;
            }
            const uint32_t hb = pack_bf16x2(w2[0], w2[1]);
            hi[c >> 1] = hb;
            if constexpr (kLo) {
              lo[c >> 1] = pack_bf16x2(w2[0] - bf16lo(hb), w2[1] - bf16hi(hb));
              add_f32x2(den4[c & 3], den4[(c + 1) & 3], w2[0], w2[1]);
            } else {
              // the denominator sums the weights the numerator multiplies
              add_f32x2(den4[c & 3], den4[(c + 1) & 3], bf16lo(hb), bf16hi(hb));
            }
          }
          if constexpr (kEpiCols == 64) {
            tmem_store_x32(cols, *reinterpret_cast<const uint32_t(*)[32]>(hi));
            if constexpr (kLo) tmem_store_x32(cols + 32, *reinterpret_cast<const uint32_t(*)[32]>(lo));
          } else {
            tmem_store_x16(cols, *reinterpret_cast<const uint32_t(*)[16]>(hi));
            if constexpr (kLo) tmem_store_x16(cols + 16, *reinterpret_cast<const uint32_t(*)[16]>(lo));
          }
        };
        // one code path per case (the first tile's lo, the causal mask), so the common one,
        // hi alone and no mask, carries neither
        if (kt < kLoTiles) {
          if (masked)
            write_p(std::true_type{}, std::true_type{});
          else
            write_p(std::true_type{}, std::false_type{});
        } else if (masked) {
          write_p(std::false_type{}, std::true_type{});
        } else {
          write_p(std::false_type{}, std::false_type{});
        }
        tmem_wait_st();
        tc_fence_before_sync();  // P is read by the tensor cores
        // every lane's weight sums depend on all of its key-norm reads
        const float used = __shfl_sync(0xffffffffu, den4[0] + den4[1], 0) +
                           __shfl_sync(0xffffffffu, den4[2] + den4[3], 31);
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&pfull[sb]);
          mbar_arrive_after(&rkempty[sb], used);
        }
      }
      if (ok) ok = mbar_wait(ofull, k & 1) && !*s_abort;
      // The row's output: O from tensor memory; the parts of each row add their weight sums,
      // exchanged through the first O column of each part once every part has read its O.
      uint32_t o[kEpiCols];
      const float mine = (den4[0] + den4[1]) + (den4[2] + den4[3]);
      if (ok) {
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < kEpiCols; c += 32)
          tmem_load_x32(tmem + lane_base + kColO + cg * kEpiCols + c,
                        *reinterpret_cast<uint32_t(*)[32]>(&o[c]));
        tmem_wait_ld(o);
        tmem_store_x1(tmem + lane_base + kColO + cg * kEpiCols, __float_as_uint(mine));
        tmem_wait_st();
        tc_fence_before_sync();
      }
      ok = named_bar_and(1, kEpiWarps * 32, ok);
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t dv[kEpiParts];
#pragma unroll
      for (int part = 0; part < kEpiParts; ++part)
        dv[part] = part == cg ? __float_as_uint(mine) : tmem_load_x1(tmem + lane_base + kColO + part * kEpiCols);
      tmem_wait_ld(dv);
      float dsum = 0.0f;
#pragma unroll
      for (int part = 0; part < kEpiParts; ++part) dsum += __uint_as_float(dv[part]);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(ofree);  // the next block's P V may overwrite O
      // out = a2 O' / (c + a2 den'): one division per row, then a multiply per output
      const float z = p.c + a2 * dsum;
      const float f = z != 0.0f ? a2 / z : 0.0f;
      const int64_t t = static_cast<int64_t>(rb.qt) * 128 + r;
      if (t < p.T) {
        float *dst = p.out + (static_cast<int64_t>(rb.bh) * p.T + t) * kHeadDim + cg * kEpiCols;
        // each store instruction writes one row piece per lane: 32-byte pieces fill whole
        // sectors, with half the instructions of 16-byte ones
        if (p.out32) {
#pragma unroll
          for (int c = 0; c < kEpiCols; c += 8)
            st_global_v8(dst + c, __uint_as_float(o[c]) * f, __uint_as_float(o[c + 1]) * f,
                         __uint_as_float(o[c + 2]) * f, __uint_as_float(o[c + 3]) * f,
                         __uint_as_float(o[c + 4]) * f, __uint_as_float(o[c + 5]) * f,
                         __uint_as_float(o[c + 6]) * f, __uint_as_float(o[c + 7]) * f);
        } else {
#pragma unroll
          for (int c = 0; c < kEpiCols; c += 4) {
            const float4 v = make_float4(__uint_as_float(o[c]) * f, __uint_as_float(o[c + 1]) * f,
                                         __uint_as_float(o[c + 2]) * f, __uint_as_float(o[c + 3]) * f);
            *reinterpret_cast<float4 *>(dst + c) = v;
          }
        }
      }
    }
    if (!ok) set_abort_p(s_abort, p.flags);
  }

  __syncthreads();
  if (threadIdx.x == 0 && *s_abort) {
    // No copy may still be landing in shared memory when the CTA leaves.  Without an abort
    // every copy issued was waited for by the role that used it; after one, wait (bounded)
    // for the last armed phase of every barrier that a copy completes.
    const int qi = *s_qissued;
    if (qi > 0) mbar_wait(qfull, (qi - 1) & 1);
    const int issued = *s_issued;  // 3 per key tile: K, key norms, V
    const int nk = (issued + 2) / 3, nr = (issued + 1) / 3, nv = issued / 3;  // tiles of each
    for (int s = 0; s < kRing; ++s) {
      int uses = nk > s ? (nk - 1 - s) / kRing + 1 : 0;
      if (uses) mbar_wait(&kfull[s], (uses - 1) & 1);
      uses = nr > s ? (nr - 1 - s) / kRing + 1 : 0;
      if (uses) mbar_wait(&rkfull[s], (uses - 1) & 1);
      uses = nv > s ? (nv - 1 - s) / kRing + 1 : 0;
      if (uses) mbar_wait(&vfull[s], (uses - 1) & 1);
    }
  }
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kPTmemCols);
  }
}

// rk2[u][j] = 1 / (mean(k_j^2) + eps), one thread per key.
__global__ void __launch_bounds__(128) prefill_knorm_kernel(const uint8_t *K, float *rk, int64_t n,
                                                            int64_t ncap, int64_t rk_stride,
                                                            float eps) {
  pdl_wait_primary();
  pdl_launch_dependents();
  const int64_t u = blockIdx.y;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= n) return;
  const uint4 *row = reinterpret_cast<const uint4 *>(K + (u * ncap + j) * kHeadDim * 2);
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = 0.0f;
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const uint4 x0 = row[c], x1 = row[c + 1];
    sq_acc_bf16x2(x0.x, a[0], a[1]);
    sq_acc_bf16x2(x0.y, a[2], a[3]);
    sq_acc_bf16x2(x0.z, a[4], a[5]);
    sq_acc_bf16x2(x0.w, a[6], a[7]);
    sq_acc_bf16x2(x1.x, a[0], a[1]);
    sq_acc_bf16x2(x1.y, a[2], a[3]);
    sq_acc_bf16x2(x1.z, a[4], a[5]);
    sq_acc_bf16x2(x1.w, a[6], a[7]);
  }
  const float ss = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
  rk[u * rk_stride + j] = 1.0f / (ss * (1.0f / kHeadDim) + eps);
}

}  // namespace

int64_t prefill_rk_stride(int64_t n) { return (n + 3) & ~static_cast<int64_t>(3); }

size_t prefill_workspace_bytes(int64_t units, int64_t n) {
  return (static_cast<size_t>(units) * static_cast<size_t>(prefill_rk_stride(n)) * 4 + 255) &
         ~static_cast<size_t>(255);
}

cudaError_t launch_prefill(const CUtensorMap &tm_q, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                           const CUtensorMap &tm_rk, const void *k_cache, float *rk, float *out,
                           uint32_t *flags, int B, int Hq, int Hkv, int64_t n, int64_t T,
                           int64_t ncap, float alpha, float c, float eps, int sm_count,
                           cudaStream_t stream) {
  const int64_t units = static_cast<int64_t>(B) * Hkv;
  if (units == 0 || T == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(prefill_knorm_kernel,
                             dim3(static_cast<unsigned>((n + 127) / 128), static_cast<unsigned>(units)),
                             dim3(128), 0, stream, 0u, static_cast<const uint8_t *>(k_cache), rk, n,
                             ncap, prefill_rk_stride(n), eps);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
  if (e != cudaSuccess) return e;
  PrefillParams p;
  p.out = out;
  p.flags = flags;
  p.n = n;
  p.T = T;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.BH = B * Hq;
  p.nqt = static_cast<int32_t>((T + 127) / 128);
  p.items = p.BH * p.nqt;
  p.out32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  p.alpha = alpha;
  p.c = c;
  p.eps = eps;
  // persistent: one CTA per SM (at most one per row block), each taking its row blocks in
  // turn
  const int64_t ctas = p.items < sm_count ? p.items : sm_count;
  return launch_pdl(prefill_kernel, dim3(static_cast<unsigned>(ctas)), dim3(kPThreads),
                    static_cast<size_t>(kPSmem), stream, 0u, tm_q, tm_k, tm_v, tm_rk, p);
}

}  // namespace embla
