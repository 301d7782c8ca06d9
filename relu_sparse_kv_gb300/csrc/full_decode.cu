// Full (ReLU^2) layer decode for one decode token per sequence.
//
// Source: "The Architecture of Embla 1", sections "Sevren Sparse Attention learns
// to be sparse" (weights ReLU(s)^2 of scores between RMS-normalised query and key,
// divided by a constant plus the sum of weights) and "Skipping V" (a value row is
// read only when some query head of the KV group gives its key a weight above zero).
//
// One persistent CTA per SM walks its pieces of the flattened (unit, tile) sequence of
// 128-key tiles, unit = (batch, KV head): the sequence is cut into K pieces per CTA and CTA
// c takes pieces c, c + P, c + 2P, ... (K = 1 while a CTA's share is short), so that units
// with many survivors are shared out.  A stretch is the part of a piece inside one unit: it
// has its own query rows, partial record and histogram flush.  Warp roles:
//   warp 0     TMA producer: 32 KB K tiles (two 64-column boxes, 128-byte swizzle) into
//              a 3-stage ring; the unit's G query rows when a stretch starts.
//   warps 1, 18  tcgen05 issuers taking alternate tiles: D[128 keys x 16] = K . Q^T
//              (raw bf16 operands, fp32 in tensor memory), the eight 16-dim k-steps added
//              into one accumulator of 16 columns; four tiles in flight.
//   warps 14-17  key norms, one thread per key as soon as a tile lands:
//              rk = 1/sqrt(mean(k^2) + eps), handed to the epilogue through a small
//              shared-memory ring; the K stage is free once these and the MMAs are done.
//   warps 2-9  two epilogue warpgroups taking alternate tiles, one thread per key:
//              s_h = dot_h * alpha*rq_h * rk, sigma = max_h s_h; lists the keys with
//              sigma > 0 with their ReLU^2 weights in key order; each group takes that
//              many rows of its own 128-row V ring (in its tile order; every warp of
//              the group tracks the ring itself, so neither group waits for the other),
//              and every surviving key's thread copies its own 256-byte V row there.
//   warp 19    selection scores (when requested): writes each tile's sigma to global
//              memory and counts it into a shared histogram, flushed when a unit's
//              stretch ends.
//   warps 10-13  V accumulators: O^T += V^T W as m16n8k16 bf16 MMAs over 16 survivors at
//              a time (dims split over warps, heads as the N columns, the weights as bf16
//              hi + lo), the denominators in fp32, in tile order; at the end of each
//              stretch of a unit they write a partial record and count the stretch's
//              survivors into the unit's total.
//
// full_combine_kernel, launched after it, sums each unit's records in piece order and writes
// out = num / (c + den): spread over one CTA per (unit, head), so that no SM reads a whole
// unit's records alone, and with no counting-in or fence in the decode kernel.
//
// 8-bit caches (E4M3 codes with one fp32 scale per token and KV head; same roles):
//   - a stage is the 16 KB code tile (one 128-column box, 128-byte swizzle) plus the
//     tile's 512-byte K-scale and V-scale runs; 6 stages.
//   - the key-norm warps pass on the keys' scales and build, once per unit, the query as
//     three E4M3 terms with t1 + t2 / 16 + t3 / 256 = q / 2^e (2^e a power of two per head,
//     so |q / 2^e| < 256), laid out as MMA rows term * G + h; the sum is within 2^-25 of
//     the head's largest |q| of every element, and exact for every element at least 2^-14
//     of it.
//   - the tensor cores take the codes and the terms directly (kind::f8f6f4, K = 32), the
//     k-steps into one accumulator, followed by 128 columns of codes . codes^T whose
//     diagonal is each key's sum of squared codes; two tiles in flight.  The epilogue sums
//     the terms in fp32 and folds 2^e into the query factor, and the key scale into rk:
//     rk = ks / sqrt(ks^2 * mean(code^2) + eps).
//   - 128-byte V rows; the accumulators widen each step's code rows to bf16 (exactly) and
//     weight them by w * vs.
#include "internal.h"
#include "ptx.cuh"

namespace embla {
namespace {

#ifndef EMBLA_K_STAGES
#define EMBLA_K_STAGES 3
#endif
#ifndef EMBLA_K8_STAGES
#define EMBLA_K8_STAGES 6
#endif
#ifndef EMBLA_W_SLOTS
#define EMBLA_W_SLOTS 8
#endif
#ifndef EMBLA_V_RING_ROWS
#define EMBLA_V_RING_ROWS 256
#endif
constexpr int kWSlots = EMBLA_W_SLOTS;             // per-tile survivor lists in flight
constexpr int kRing = EMBLA_V_RING_ROWS;           // V rows in flight
constexpr int kGroups = 2;                         // epilogue warpgroups, alternating tiles
constexpr int kAccBufs = 2 * kGroups;              // tensor-memory accumulators
constexpr int kNormSlots = 8;                      // per-tile key-norm arrays in flight
constexpr int kQBufBytes = 4096;                   // 16 rows x 128 dims of bf16 (MMA N = 16)
constexpr int kQHalfBytes = kQBufBytes / 2;
constexpr int kQ8BufBytes = 4096;                  // up to 32 rows x 128 dims of E4M3
constexpr int kAccStep = 16;                       // survivors per V-accumulation MMA step
constexpr int kAccPitch = 2 * 128 + 16;            // bytes per bf16 row read by ldmatrix
constexpr uint32_t kAccBar = 3;                    // named barrier of the accumulator warps
constexpr int kWarpProducer = 0, kWarpMma = 1, kWarpEpi = 2;
constexpr int kWarpAcc = kWarpEpi + 4 * kGroups;
constexpr int kWarpNorm = kWarpAcc + 4;
constexpr int kWarpMma2 = kWarpNorm + 4;           // second MMA issuer (odd tiles)
constexpr int kWarpHist = kWarpMma2 + 1;           // selection scores and histogram
constexpr int kMmaWarps = 2;
constexpr int kThreads = (kWarpHist + 1) * 32;     // 640
constexpr int kGroupRing = kRing / kGroups;        // each epilogue group's own V ring
static_assert(kGroupRing >= kTileKeys, "a whole tile of survivors must fit a group's V ring");
static_assert((kGroupRing & (kGroupRing - 1)) == 0, "the V ring size is a power of two");
static_assert(kWSlots % kGroups == 0 && kWSlots >= 4 * kGroups,
              "a W slot stays with one group; a group's last three tiles keep their slots");

// What differs between bf16 caches (KV8 false) and 8-bit E4M3 caches with per-token
// scales (KV8 true).
template <int G, bool KV8>
struct Cfg {
  static constexpr int stages = KV8 ? EMBLA_K8_STAGES : EMBLA_K_STAGES;  // K tiles in flight
  // Tile i lands on barrier full[(i % stages) * 2 + (i & 1)]: one barrier per stage and MMA
  // issuer, so the uses of each barrier are consumed in order by one issuer (with an odd
  // stage count a stage's consecutive tiles belong to different issuers, and a parity
  // test by one issuer could be answered by the other's phase).  Barrier uses repeat
  // every full_period tiles.
  static constexpr int full_period = stages % 2 == 0 ? stages : 2 * stages;
  static constexpr int row_bytes = KV8 ? kHeadDim : 2 * kHeadDim;  // one cached K or V row
  // V-ring row pitch: bf16 rows are read by ldmatrix straight from the ring, so they are
  // padded by 16 bytes (eight rows in a row then fall in eight different bank groups);
  // 8-bit rows are first widened to bf16 rows in a small staging area of that pitch.
  static constexpr int ring_pitch = KV8 ? kHeadDim : 2 * kHeadDim + 16;
  static constexpr int tile_bytes = kTileKeys * row_bytes;           // 32 KB / 16 KB
  static constexpr int half_bytes = kTileKeys * 128;                 // one 128-byte-wide box
  static constexpr int scale_bytes = KV8 ? kTileKeys * 4 : 0;        // K (then V) scales
  static constexpr int stage_bytes = tile_bytes + 2 * scale_bytes;
  // scores: 128 keys x mma_n query rows (bf16: G heads; E4M3: 3 terms x G heads)
  static constexpr int mma_n = KV8 ? (3 * G <= 16 ? 16 : 32) : 16;
  static constexpr int kstep_dims = KV8 ? 32 : 16;
  static constexpr int ksteps = kHeadDim / kstep_dims;
  // The k-steps add into one score accumulator.  8-bit: it is followed by 128 columns of
  // codes . codes^T, whose diagonal is each key's sum of squared codes (those key norms come
  // from the tensor cores; bf16 key norms come from the key-norm warps).
  static constexpr int score_cols = mma_n;
  static constexpr int diag_cols = KV8 ? kTileKeys : 0;
  static constexpr int acc_cols = score_cols + diag_cols;            // 16 / 144 / 160
  // Tiles in flight.  Tile i goes to buffer i % acc_bufs, to MMA issuer i % 2 and to
  // epilogue group i % 2; with an even count every buffer has one issuer and one reader,
  // which take its phases in order (with an odd count a fast group could wait for a
  // buffer's next phase before its current one completed, and pass on the stale parity).
  static constexpr int acc_bufs = KV8 ? kGroups : kAccBufs;  // bf16: 4 x 16 columns
  static constexpr int tmem_cols = 512;
  static constexpr uint32_t idesc = KV8 ? idesc_e4m3_f32(128, mma_n) : idesc_bf16_f32(128, 16);
  static constexpr uint32_t idesc_diag = idesc_e4m3_f32(128, kTileKeys);
  static_assert(stage_bytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
  static_assert(tile_bytes == (KV8 ? 1 : 2) * half_bytes, "a tile is one or two boxes");
  static_assert(acc_bufs <= kAccBufs && acc_bufs * acc_cols <= tmem_cols, "tensor memory");
  static_assert(acc_bufs % kGroups == 0 && acc_bufs % kMmaWarps == 0, "one issuer and one reader");
  static_assert(!KV8 || idesc_diag != 0u, "the codes . codes^T instruction");
};

// One tile's survivors in ascending key order: entry e has its V row in row
// (row0 + e) mod kGroupRing of the V ring of the tile's epilogue group.  Also the tile's
// selection scores, for the histogram warp.
template <int G, bool KV8>
struct WSlot {
  int32_t cnt[4];             // survivors per TMEM quarter (32 keys each)
  int32_t row0;               // first V-ring row of this tile
  int32_t m;                  // survivors in the tile
  int32_t pad[2];
  int32_t key[kTileKeys];     // key index within the unit
  float w[kTileKeys][G];      // ReLU^2 weights per head
  float sig[kTileKeys];       // sigma of every key of the tile
  float vs[KV8 ? kTileKeys : 1];  // V scale of each survivor (8-bit caches)
};

template <int G, bool KV8>
struct Smem {
  using C = Cfg<G, KV8>;
  static constexpr int k_off = 0;
  static constexpr int q_off = k_off + C::stages * C::stage_bytes;
  static constexpr int q8_off = q_off + 2 * kQBufBytes;
  static constexpr int ring_off = q8_off + (KV8 ? 2 * kQ8BufBytes : 0);
  // bf16: the ring, then one zero row; 8-bit: the ring, then two staging blocks of
  // kAccStep widened rows and one zero row (the rows an MMA step reads past a tile's list)
  static constexpr int zero_off = ring_off + kRing * C::ring_pitch;
  static constexpr int stage_off = KV8 ? zero_off + kAccPitch : zero_off;
  static constexpr int wslot_off = (KV8 ? stage_off + 2 * kAccStep * kAccPitch : zero_off + kAccPitch);
  static constexpr int hist_off = wslot_off + kWSlots * static_cast<int>(sizeof(WSlot<G, KV8>));
  static constexpr int rk_off = hist_off + kHistBins * 4;
  static constexpr int vs_off = rk_off + kNormSlots * kTileKeys * 4;  // V scales beside rk
  static constexpr int misc_off = vs_off + (KV8 ? kNormSlots * kTileKeys * 4 : 0);
  static constexpr int bar_off = misc_off + 128 + 16 * kMaxPiecesPerCta;
  static constexpr int n_bars = 3 * C::stages + 2 * kAccBufs + 8 + 3 * kWSlots + 2 * kNormSlots;
  static constexpr int total = bar_off + n_bars * 8;
  static constexpr int alloc = total + 1024;  // room to align the base to 1024
  static_assert(alloc <= 227 * 1024, "shared memory per CTA");
  static_assert(misc_off % 16 == 0 && 7 + kWSlots <= 32, "misc words, then the piece table");
};

struct FullParams {
  const uint8_t *v;  // V cache (bf16 rows or E4M3 codes)
  float *sel;        // selection scores or null
  uint32_t *hist;    // selection histogram or null
  float *hsel;       // per-head scores [B, Hq, ncap] or null
  float *rec;        // partial records: one per (piece, unit) stretch, at index piece + unit
  float *out;        // [units][G][D]
  int32_t *n_surv;   // [units]
  float c;           // normaliser constant
  uint32_t *flags;
  int64_t T, TU, n, ncap;
  int32_t P, Q, K, Hq, Hkv, rec_stride;  // CTAs, pieces (K per CTA)
  float alpha, eps;
};

// Power-of-two exponent e with |q| / 2^e < 256 for the head's largest |q| element (the
// E4M3 query terms); kept within [-120, 127] so 2^e and 2^-e are normal floats.
__device__ __forceinline__ int q8_exponent(float maxabs) {
  const int be = static_cast<int>((__float_as_uint(maxabs) >> 23) & 0xFFu);  // biased
  const int e = be - 127 - 7;
  return e < -120 ? -120 : (e > 120 ? 120 : e);
}
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

__device__ __forceinline__ float sumsq8(const uint4 &v) {
  float a = bf16lo(v.x) * bf16lo(v.x);
  float b = bf16hi(v.x) * bf16hi(v.x);
  a = fmaf(bf16lo(v.y), bf16lo(v.y), a);
  b = fmaf(bf16hi(v.y), bf16hi(v.y), b);
  a = fmaf(bf16lo(v.z), bf16lo(v.z), a);
  b = fmaf(bf16hi(v.z), bf16hi(v.z), b);
  a = fmaf(bf16lo(v.w), bf16lo(v.w), a);
  b = fmaf(bf16hi(v.w), bf16hi(v.w), b);
  return a + b;
}

// Largest |x| of the eight bf16 values in v.
__device__ __forceinline__ float maxabs8(const uint4 &v) {
  const float a = fmaxf(fmaxf(fabsf(bf16lo(v.x)), fabsf(bf16hi(v.x))),
                        fmaxf(fabsf(bf16lo(v.y)), fabsf(bf16hi(v.y))));
  const float b = fmaxf(fmaxf(fabsf(bf16lo(v.z)), fabsf(bf16hi(v.z))),
                        fmaxf(fabsf(bf16lo(v.w)), fabsf(bf16hi(v.w))));
  return fmaxf(a, b);
}

// The unit's query rows (bf16, two 64-dim boxes of 128-byte swizzled rows) as three E4M3
// terms per head: x = q / 2^e, t1 = rn(x), t2 = rn(16 (x - t1)), t3 = rn(16 (16 (x - t1) -
// t2)), so q = 2^e (t1 + t2 / 16 + t3 / 256) up to 2^-25 of the head's largest |q| (every
// remainder is at most 8 in magnitude, so no term saturates; the scaling by 16 keeps the
// later terms clear of the E4M3 subnormal range).  Written as rows t * G + h of a
// 128-byte swizzled operand.  Thread t of the 128 takes head
// t / 8 and dims 16 (t % 8) .. 16 (t % 8) + 15; all 32 lanes of a warp must call it.
template <int G>
__device__ __forceinline__ void build_q8_terms(const uint8_t *qsrc, uint8_t *qdst, int t) {
  const int h = t >> 3, c = t & 7;
  float x[16];
  float mx = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) x[k] = 0.0f;
  if (h < G) {
    // dims 16c.. are 16-byte chunks 2c and 2c+1 of the row, in box c / 4
    const uint8_t *qr = qsrc + (c >> 2) * kQHalfBytes + h * 128;
    const uint4 a = *reinterpret_cast<const uint4 *>(qr + ((((2 * c) & 7) ^ (h & 7)) * 16));
    const uint4 b = *reinterpret_cast<const uint4 *>(qr + ((((2 * c + 1) & 7) ^ (h & 7)) * 16));
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      x[2 * k] = bf16lo(w[k]);
      x[2 * k + 1] = bf16hi(w[k]);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) mx = fmaxf(mx, fabsf(x[k]));
  }
  // the head's 8 threads are 8 neighbouring lanes
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (h < G) {
    const float inv = pow2f(-q8_exponent(mx));
#pragma unroll
    for (int k = 0; k < 16; ++k) x[k] *= inv;
#pragma unroll
    for (int term = 0; term < 3; ++term) {
      uint32_t cw[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) cw[g] = f32x4_to_e4m3x4(x[4 * g], x[4 * g + 1], x[4 * g + 2], x[4 * g + 3]);
      const int r = term * G + h;
      *reinterpret_cast<uint4 *>(qdst + r * 128 + ((c ^ (r & 7)) * 16)) =
          make_uint4(cw[0], cw[1], cw[2], cw[3]);
      if (term < 2) {
        // the remainder (exact in fp32, at most 8 in magnitude) times 16 for the next term
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float d0, d1, d2, d3;
          e4m3x4_to_f32(cw[g], d0, d1, d2, d3);
          x[4 * g] = (x[4 * g] - d0) * 16.0f;
          x[4 * g + 1] = (x[4 * g + 1] - d1) * 16.0f;
          x[4 * g + 2] = (x[4 * g + 2] - d2) * 16.0f;
          x[4 * g + 3] = (x[4 * g + 3] - d3) * 16.0f;
        }
      }
    }
  }
}

__device__ __forceinline__ void set_abort(volatile int *abort_flag, uint32_t *flags) {
  *abort_flag = 1;
  atomicOr(flags, kFlagWaitTimeout);
}

// Piece j = 0 .. K-1 of a CTA is piece q = j*P + cta of the Q = K*P, tiles
// [floor(qT/Q), floor((q+1)T/Q)) (split_piece_start): {unit, tile in unit, tiles, q}.
__device__ __forceinline__ int4 piece_entry(const FullParams &p, int j, int cta) {
  const int q = j * p.P + cta;
  int64_t b, e;
  if (((p.T * p.Q) >> 32) == 0) {
    // 32-bit arithmetic (the host limits units * cache_stride to 2^31 rows, so tile numbers
    // fit 32 bits)
    const uint32_t T32 = static_cast<uint32_t>(p.T), Q32 = static_cast<uint32_t>(p.Q);
    b = static_cast<uint32_t>(q) * T32 / Q32;
    e = (static_cast<uint32_t>(q) + 1u) * T32 / Q32;
  } else {
    b = split_piece_start(q, p.T, p.Q);
    e = split_piece_start(q + 1, p.T, p.Q);
  }
  const int TU = static_cast<int>(p.TU);
  const int u = static_cast<int>(static_cast<uint32_t>(b) / static_cast<uint32_t>(TU));
  return make_int4(u, static_cast<int>(b) - u * TU, static_cast<int>(e - b), q);
}

// Advance (tile-in-unit, unit) to the next tile of the flattened sequence.
__device__ __forceinline__ void next_tile(int &tl, int &u, int TU) {
  if (++tl == TU) {
    tl = 0;
    ++u;
  }
}

// PIECES: K > 1 pieces per CTA (without it the walk is compiled for one piece, a CTA's
// contiguous share).
template <int G, bool KV8, bool PIECES>
__global__ void __launch_bounds__(kThreads, 1)
    full_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_ks,
                       const __grid_constant__ CUtensorMap tm_vs, const FullParams p) {
  using L = Smem<G, KV8>;
  using C = Cfg<G, KV8>;
  constexpr int kStages = C::stages;
  constexpr int kFullPeriod = C::full_period;
  constexpr int kRowBytes = C::row_bytes;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // offset arithmetic on the shared array keeps every access in the shared state space
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t *sK = smem + L::k_off;
  uint8_t *sQ = smem + L::q_off;
  uint8_t *sQ8 = smem + L::q8_off;  // E4M3 query terms (8-bit caches)
  uint8_t *sRing = smem + L::ring_off;
  WSlot<G, KV8> *wslots = reinterpret_cast<WSlot<G, KV8> *>(smem + L::wslot_off);
  uint32_t *s_hist = reinterpret_cast<uint32_t *>(smem + L::hist_off);
  float *s_rk = reinterpret_cast<float *>(smem + L::rk_off);
  float *s_vs = reinterpret_cast<float *>(smem + L::vs_off);
  int *misc = reinterpret_cast<int *>(smem + L::misc_off);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(misc);
  volatile int *s_abort = misc + 1;
  volatile int *s_k_issued = misc + 2;
  volatile int *s_q_issued = misc + 3;
  volatile int *s_final_hist = misc + 5;  // unit whose histogram the whole CTA flushes at the end
  volatile int *s_varm = misc + 7;        // [W slot]: V-copy phases armed on its barrier
  int4 *s_piece = reinterpret_cast<int4 *>(misc + 32);  // [j]: the CTA's pieces
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::bar_off);
  uint64_t *full = bars;                 // K tile landed: [stage][tile parity]
  uint64_t *empty = full + 2 * kStages;  // K tile consumed (MMA and key norms)
  uint64_t *accf = empty + kStages;      // accumulator written
  uint64_t *acce = accf + kAccBufs;      // accumulator read
  uint64_t *qfull = acce + kAccBufs;     // query rows landed
  uint64_t *qempty = qfull + 2;          // query rows no longer needed
  uint64_t *wempty = qempty + 2;         // survivor list and its V rows consumed
  uint64_t *vfull = wempty + kWSlots;    // survivor list written and its V rows landed
  uint64_t *sfull = vfull + kWSlots;     // selection scores of a tile written
  uint64_t *rkfull = sfull + kWSlots;    // key norms of a tile written
  uint64_t *rkempty = rkfull + kNormSlots;  // key norms of a tile read
  uint64_t *q8full = rkempty + kNormSlots;  // E4M3 query terms written
  uint64_t *q8empty = q8full + 2;           // E4M3 query terms no longer needed

  // The zeroing kernel lets this kernel launch before the kernels ahead of it have finished:
  // the set-up below touches no global memory, and thread 0 waits for them (through the
  // zeroing kernel) before its first load; every other global access follows that load.
  // The kernel after this one may launch now (it waits for this kernel to finish).
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = static_cast<int>(blockIdx.x);
  const int TU = static_cast<int>(p.TU);
  const int K = PIECES ? p.K : 1;
  // the CTA's pieces, one lane of warp 0 each, before thread 0 starts the loads
  if (warp == kWarpProducer) {
    if (lane < K) s_piece[lane] = piece_entry(p, lane, cta);
    __syncwarp();
  }

  // TMA producer state (thread 0): it issues the first stages during the set-up below and
  // carries on from there as warp 0's role.
  int pr_i = 0, pr_j = -1, pr_ib = 0, pr_ie = 0, pr_u = 0, pr_tl = 0;
  int pr_seg = -1, pr_s = 0, pr_sphase = 0;
  uint64_t pr_policy = 0;
  // Issue K tiles (and each new stretch's query rows) until tile `limit`; with `setup` set it
  // stops before any load that would have to wait for a buffer to be handed back.
  auto produce = [&](int limit, bool setup) {
    for (; pr_i < limit; ++pr_i, next_tile(pr_tl, pr_u, TU)) {
      if (pr_i == pr_ie) {
        // the next piece, if any
        if (pr_j + 1 == K) break;
        const int4 pe = s_piece[++pr_j];
        pr_u = pe.x;
        pr_tl = pe.y;
        pr_ib = pr_i;
        pr_ie = pr_i + pe.z;
      }
      if (*s_abort) break;
      if (pr_i == pr_ib || pr_tl == 0) {
        const int qb = (pr_seg + 1) & 1;
        if (pr_seg + 1 >= 2) {
          if (setup) break;
          if (!mbar_wait(&qempty[qb], (((pr_seg + 1) >> 1) - 1) & 1)) {
            set_abort(s_abort, p.flags);
            break;
          }
        }
        ++pr_seg;
        mbar_arrive_expect_tx(&qfull[qb], 2 * G * 128);
        const int32_t qrow = static_cast<int32_t>((pr_u / p.Hkv) * p.Hq + (pr_u % p.Hkv) * G);
        tma_load_2d(sQ + qb * kQBufBytes, &tm_q, &qfull[qb], 0, qrow);
        tma_load_2d(sQ + qb * kQBufBytes + kQHalfBytes, &tm_q, &qfull[qb], 64, qrow);
        *s_q_issued = pr_seg + 1;
      }
      if (pr_i >= kStages) {
        if (setup) break;
        if (!mbar_wait(&empty[pr_s], pr_sphase ^ 1)) {
          set_abort(s_abort, p.flags);
          break;
        }
      }
      uint64_t *fb = &full[2 * pr_s + (pr_i & 1)];
      mbar_arrive_expect_tx(fb, C::stage_bytes);
      const int32_t row = static_cast<int32_t>(static_cast<int64_t>(pr_u) * p.ncap) + pr_tl * kTileKeys;
      uint8_t *st = sK + pr_s * C::stage_bytes;
      tma_load_2d_hint(st, &tm_k, fb, 0, row, pr_policy);
      if constexpr (KV8) {
        // the tile's K and V scales: 128 floats each from row u of the [units, ncap] arrays
        tma_load_2d_hint(st + C::tile_bytes, &tm_ks, fb, pr_tl * kTileKeys, pr_u, pr_policy);
        tma_load_2d_hint(st + C::tile_bytes + C::scale_bytes, &tm_vs, fb, pr_tl * kTileKeys, pr_u,
                         pr_policy);
      } else {
        tma_load_2d_hint(st + C::half_bytes, &tm_k, fb, 64, row, pr_policy);
      }
      *s_k_issued = pr_i + 1;
      if (++pr_s == kStages) {
        pr_s = 0;
        pr_sphase ^= 1;
      }
    }
  };

  if (threadIdx.x == 0) {
    // The first K stages and query rows go out before anything else is set up: their
    // barriers first, then the copies (the stages are empty, the query buffers free, and
    // nothing below writes where these copies land).
    for (int f = 0; f < 2 * kStages; ++f) mbar_init(&full[f], 1);
    mbar_init(&qfull[0], 1);
    mbar_init(&qfull[1], 1);
    fence_barrier_init();
    *s_abort = 0;
    *s_k_issued = 0;
    *s_q_issued = 0;
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_q);
    if constexpr (KV8) {
      tma_prefetch_desc(&tm_ks);
      tma_prefetch_desc(&tm_vs);
    }
    pr_policy = policy_evict_first();
    pdl_wait_primary();  // the query, and the caches' newest rows, are written
    produce(kStages, true);
  }
  if (warp == kWarpEpi) {
    // the other barriers, by the lanes of another warp side by side (each lane at most one
    // of each kind)
    static_assert(kStages <= 32 && kAccBufs <= 32 && kWSlots <= 32 && kNormSlots <= 32,
                  "one barrier of each kind per lane");
    if (lane < kStages) mbar_init(&empty[lane], 5);  // MMA commit + the four norm warps
    if (lane < kAccBufs) {
      mbar_init(&accf[lane], 1);
      mbar_init(&acce[lane], 4);
    }
    if (lane < 2) {
      // readers of the bf16 query rows: the epilogue warps, and the MMA issuers (bf16
      // caches) or the norm warps building the E4M3 terms (8-bit caches)
      mbar_init(&qempty[lane], 4 * kGroups + (KV8 ? 4 : kMmaWarps));
      mbar_init(&q8full[lane], 4);
      mbar_init(&q8empty[lane], kMmaWarps);
    }
    if (lane < kWSlots) {
      mbar_init(&wempty[lane], p.sel != nullptr ? 5 : 4);  // accumulators (+ histogram warp)
      mbar_init(&vfull[lane], 4);
      mbar_init(&sfull[lane], 4);
    }
    if (lane < kNormSlots) {
      mbar_init(&rkfull[lane], 4);
      mbar_init(&rkempty[lane], 4);
    }
    if (lane == 0) *s_final_hist = -1;
    if (lane < kWSlots) s_varm[lane] = 0;
    fence_barrier_init();
  }
  // Rows G..15 of the query operand feed only MMA columns that are never read; zero
  // them anyway so no stale bits reach the tensor core (rows 0..G-1 are being loaded).
  for (int i = threadIdx.x; i < 2 * 2 * (16 - G) * 8; i += kThreads) {
    const int box = i / ((16 - G) * 8), rem = i - box * ((16 - G) * 8);
    reinterpret_cast<uint4 *>(sQ + box * kQHalfBytes + G * 128)[rem] = make_uint4(0u, 0u, 0u, 0u);
  }
  if constexpr (KV8)
    for (int i = threadIdx.x; i < 2 * kQ8BufBytes / 16; i += kThreads)
      reinterpret_cast<uint4 *>(sQ8)[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int i = threadIdx.x; i < kHistBins; i += kThreads) s_hist[i] = 0u;
  for (int i = threadIdx.x; i < kAccPitch / 16; i += kThreads)
    reinterpret_cast<uint4 *>(smem + L::zero_off)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (warp == kWarpMma) {
    tmem_alloc(s_tmem, C::tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(s_tmem);

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) produce(INT32_MAX, false);
    __syncwarp();
  } else if (warp == kWarpMma || warp == kWarpMma2) {
    // ------------------------------------------------------------------ MMA issuers
    // Two issuing threads take alternate tiles: every tcgen05 instruction and barrier
    // check costs a single thread a long latency, so one thread alone cannot keep up.
    const int mw = warp == kWarpMma ? 0 : 1;
    if (lane == 0) {
      // descriptors are built once; per k-step only their start-address field moves
      // (8-bit caches: the MMA's query operand is the E4M3 terms, which the norm warps
      // write; the bf16 rows are handed back by those warps instead)
      constexpr int qbuf_bytes = KV8 ? kQ8BufBytes : kQBufBytes;
      uint64_t *qf = KV8 ? q8full : qfull;
      uint64_t *qe = KV8 ? q8empty : qempty;
      const uint64_t kdesc0 = smem_desc_sw128(smem_u32(sK));
      const uint64_t qdesc0 = smem_desc_sw128(smem_u32(KV8 ? sQ8 : sQ));
      uint64_t qdesc = qdesc0;
      int seg = -1, qb = 0, issued = 0;
      int s = 0, b = 0, bphase = 0;
      int i = 0;
      for (int pc = 0; pc < K; ++pc) {
        const int4 pe = s_piece[pc];
        int tl = pe.y;
        const int ib = i, ie = i + pe.z;
        for (; i < ie; ++i) {
          if (*s_abort) break;
          if (i == ib || tl == 0) {
            ++seg;
            qb = seg & 1;
            qdesc = qdesc0 + static_cast<uint64_t>((qb * qbuf_bytes) >> 4);
            if (!mbar_wait(&qf[qb], (seg >> 1) & 1)) {
              set_abort(s_abort, p.flags);
              break;
            }
          }
          if ((i & 1) != mw) {
            // not this issuer's tile; it still hands back the query buffer at a stretch's end
            if (i + 1 == ie || tl + 1 == TU) tc_commit(&qe[qb]);
            if (++tl == TU) tl = 0;
            if (++s == kStages) s = 0;
            if (++b == C::acc_bufs) {
              b = 0;
              bphase ^= 1;
            }
            continue;
          }
          if (!mbar_wait(&full[2 * s + (i & 1)], (i / kFullPeriod) & 1) ||
              (i >= C::acc_bufs && !mbar_wait(&acce[b], bphase ^ 1))) {
            set_abort(s_abort, p.flags);
            break;
          }
          tc_fence_after_sync();
          const uint64_t adesc = kdesc0 + static_cast<uint64_t>((s * C::stage_bytes) >> 4);
          const uint32_t dcol = tmem + b * C::acc_cols;
  #pragma unroll
          for (int kk = 0; kk < C::ksteps; ++kk) {
            if constexpr (KV8) {
              // scores over dims 32kk..32kk+31 added into D[key][t*G + h] = code . t_th, and
              // codes . codes^T into the next 128 columns; k-step kk is 32 bytes into the
              // 128-byte rows of codes and of terms
              const uint64_t a = adesc + ((kk * 32) >> 4);
              tc_mma_e4m3(dcol, a, qdesc + ((kk * 32) >> 4), C::idesc, kk > 0 ? 1u : 0u);
              tc_mma_e4m3(dcol + C::score_cols, a, a, C::idesc_diag, kk > 0 ? 1u : 0u);
            } else {
              // partial scores over dims 16kk..16kk+15: D_kk[key][h] = k . q_h; k-step kk is
              // 32 bytes into a 128-byte row, the second half of the dims starts a new box
              tc_mma_bf16(dcol,
                          adesc + (((kk >> 2) * C::half_bytes + (kk & 3) * 32) >> 4),
                          qdesc + (((kk >> 2) * kQHalfBytes + (kk & 3) * 32) >> 4), C::idesc,
                          kk > 0 ? 1u : 0u);
            }
          }
          tc_commit(&accf[b]);
          tc_commit(&empty[s]);
          issued = i + 1;
          if (i + 1 == ie || tl + 1 == TU) tc_commit(&qe[qb]);
          if (++tl == TU) tl = 0;
          if (++s == kStages) s = 0;
          if (++b == C::acc_bufs) {
            b = 0;
            bphase ^= 1;
          }
        }
        if (i < ie) break;  // stopped early
      }
      // this issuer's accumulators must be idle before the tensor memory is released
      if (issued > 0 && !mbar_wait(&accf[(issued - 1) % C::acc_bufs], ((issued - 1) / C::acc_bufs) & 1))
        set_abort(s_abort, p.flags);
    }
    __syncwarp();
  } else if (warp < kWarpAcc) {
    // ------------------------------------------------------------------ epilogue groups
    // Every decision to stop is taken by the whole group (named_bar_and), so no warp is
    // left waiting at a group barrier that the others have abandoned.
    const int group = (warp - kWarpEpi) >> 2;
    const uint32_t gbar = 1u + static_cast<uint32_t>(group);
    const int quarter = warp & 3;     // the TMEM lanes this warp may read
    const int row = quarter * 32 + lane;
    const uint32_t lanemask_lt = (1u << lane) - 1u;
    float aq[G];
#pragma unroll
    for (int h = 0; h < G; ++h) aq[h] = 0.0f;
    // The group's own V ring: rows reserved so far, and the survivor counts of its last
    // three tiles (i - 2, i - 4, i - 6), whose rows may still be in use.  Every warp of the
    // group keeps the same copy (they all see every count), so no warp waits for another.
    uint8_t *gring = sRing + group * kGroupRing * C::ring_pitch;
    int issued = 0, m1 = 0, m2 = 0, m3 = 0;
    int seg = -1;
    int i = 0;
    for (int pc = 0; pc < K; ++pc) {
      const int4 pe = s_piece[pc];
      int u = pe.x, tl = pe.y;
      const int ib = i, ie = i + pe.z;
      for (; i < ie; ++i, next_tile(tl, u, TU)) {
        if (i == ib || tl == 0) {
          // every epilogue warp takes the new stretch's query norms, whichever tiles it owns
          ++seg;
          const int qb = seg & 1;
          const bool ok = !*s_abort && mbar_wait(&qfull[qb], (seg >> 1) & 1);
          if (!named_bar_and(gbar, 128, ok)) {
            set_abort(s_abort, p.flags);
            break;
          }
          {
            // alpha / sqrt(mean(q_h^2) + eps): 32 / G neighbouring lanes per head, each summing
            // 16-byte chunks of the head's row (the swizzle only permutes chunks within a
            // 128-byte row, which a sum does not see), then every lane takes every head's
            // factor from that head's first lane
            constexpr int kLanesPerHead = 32 / G, kChunks = 16 / kLanesPerHead;
            static_assert(32 % G == 0 && kChunks * kLanesPerHead == 16, "chunks per lane");
            const int hq = lane / kLanesPerHead, sub = lane % kLanesPerHead;
            float ss = 0.0f, mx = 0.0f;
  #pragma unroll
            for (int k = 0; k < kChunks; ++k) {
              const int c = sub * kChunks + k;
              const uint4 x = *reinterpret_cast<const uint4 *>(sQ + qb * kQBufBytes + (c >> 3) * kQHalfBytes +
                                                               hq * 128 + (c & 7) * 16);
              ss += sumsq8(x);
              if constexpr (KV8) mx = fmaxf(mx, maxabs8(x));
            }
  #pragma unroll
            for (int o = kLanesPerHead / 2; o > 0; o >>= 1) {
              ss += __shfl_xor_sync(0xffffffffu, ss, o);
              if constexpr (KV8) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            }
            float a = p.alpha * rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
            // the E4M3 terms hold q / 2^e: put the 2^e back here
            if constexpr (KV8) a *= pow2f(q8_exponent(mx));
  #pragma unroll
            for (int h = 0; h < G; ++h) aq[h] = __shfl_sync(0xffffffffu, a, h * kLanesPerHead);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&qempty[qb]);
        }
        if (static_cast<int>(i % kGroups) != group) continue;
        const int b = static_cast<int>(i % C::acc_bufs);
        const int slot = static_cast<int>(i % kWSlots);
        const int ns = static_cast<int>(i % kNormSlots);
        const bool ok = !*s_abort && mbar_wait(&accf[b], (i / C::acc_bufs) & 1) &&
                        mbar_wait(&rkfull[ns], (i / kNormSlots) & 1) &&
                        (i < kWSlots || mbar_wait(&wempty[slot], ((i / kWSlots) - 1) & 1));
        if (!named_bar_and(gbar, 128, ok)) {
          set_abort(s_abort, p.flags);
          break;
        }
        float dot[G];
        tc_fence_after_sync();
        float ssq = 0.0f;  // 8-bit caches: this key's sum of squared codes
        if constexpr (KV8) {
          // columns t*G + h of the score accumulator; then this warp's 32 x 32 block of
          // codes . codes^T, whose diagonal entry for this lane is its key's sum of squares
          const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + b * C::acc_cols;
          uint32_t r[3 * G];
          uint32_t dg[32];
          if constexpr (G == 4) {
            tmem_load_x8(taddr, *reinterpret_cast<uint32_t(*)[8]>(&r[0]));
            tmem_load_x4(taddr + 8, *reinterpret_cast<uint32_t(*)[4]>(&r[8]));
          } else {
            tmem_load_x16(taddr, *reinterpret_cast<uint32_t(*)[16]>(&r[0]));
            tmem_load_x8(taddr + 16, *reinterpret_cast<uint32_t(*)[8]>(&r[16]));
          }
          tmem_load_x32(taddr + C::score_cols + quarter * 32, dg);
          tmem_wait_ld(r);
          tmem_wait_ld(dg);
  #pragma unroll
          for (int h = 0; h < G; ++h)  // t1 + t2 / 16 + t3 / 256 (the scalings are exact)
            dot[h] = (__uint_as_float(r[2 * G + h]) * 0.0625f + __uint_as_float(r[G + h])) * 0.0625f +
                     __uint_as_float(r[h]);
          // dg[lane] by halving: keep the upper half of the candidates where this lane's bit is set
  #pragma unroll
          for (int k = 16; k >= 1; k >>= 1) {
  #pragma unroll
            for (int e = 0; e < k; ++e) dg[e] = (lane & k) ? dg[e + k] : dg[e];
          }
          ssq = __uint_as_float(dg[0]);
        } else {
          const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + b * C::acc_cols;
          uint32_t r[G];
          if constexpr (G == 4)
            tmem_load_x4(taddr, *reinterpret_cast<uint32_t(*)[4]>(&r[0]));
          else
            tmem_load_x8(taddr, *reinterpret_cast<uint32_t(*)[8]>(&r[0]));
          tmem_wait_ld(r);
  #pragma unroll
          for (int h = 0; h < G; ++h) dot[h] = __uint_as_float(r[h]);
        }
        tc_fence_before_sync();
        // bf16: the key norm; 8-bit: the key's scale ks, whose norm follows from the sum of
        // squared codes: ks / sqrt(ks^2 mean(code^2) + eps)
        const float rkv = s_rk[ns * kTileKeys + row];
        const float vsc = KV8 ? s_vs[ns * kTileKeys + row] : 0.0f;
        // every lane's reads are back
        const float rk_used = __shfl_sync(0xffffffffu, KV8 ? rkv + vsc : rkv, 31);
        const float rk = KV8 ? rkv * rsqrtf(rkv * rkv * (ssq * (1.0f / kHeadDim)) + p.eps) : rkv;
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&acce[b]);
          mbar_arrive_after(&rkempty[ns], rk_used);
        }

        const int j = tl * kTileKeys + row;
        const bool valid = j < p.n;
        float sc[G];
        float sigma = -INFINITY;
  #pragma unroll
        for (int h = 0; h < G; ++h) {
          sc[h] = dot[h] * aq[h] * rk;
          sigma = fmaxf(sigma, sc[h]);
        }
        if (p.hsel != nullptr && valid) {
          // every head's own score, for a selection per query head
          float *hs = p.hsel + (static_cast<int64_t>(u / p.Hkv) * p.Hq + (u % p.Hkv) * G) * p.ncap + j;
  #pragma unroll
          for (int h = 0; h < G; ++h) hs[h * p.ncap] = sc[h];
        }
        WSlot<G, KV8> &ws = wslots[slot];
        if (p.sel != nullptr) {
          ws.sig[row] = sigma;
          __syncwarp();
          if (lane == 0) mbar_arrive(&sfull[slot]);
        }
        const bool surv = valid && sigma > 0.0f;
        const uint32_t bal = __ballot_sync(0xffffffffu, surv);
        if (lane == 0) ws.cnt[quarter] = __popc(bal);
        __syncwarp();
        named_bar_sync(gbar, 128);  // the four counts are in
        int off = 0, m = 0;
  #pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = ws.cnt[q];
          m += c;
          off += q < quarter ? c : 0;
        }
        const int e = off + __popc(bal & lanemask_lt);  // this key's place in the tile's list
        if (surv) {
          ws.key[e] = j;
  #pragma unroll
          for (int h = 0; h < G; ++h) ws.w[e][h] = sc[h] > 0.0f ? sc[h] * sc[h] : 0.0f;
          if constexpr (KV8) ws.vs[e] = vsc;
        }
        // m rows of the group's ring, in the group's tile order.  Tiles i - 8 and older
        // were consumed before this tile's slot was taken; wait, oldest first, for the
        // group's later tiles until the rows in use leave room for m.
        bool rok = true;
        if (m1 + m2 + m3 + m > kGroupRing && i >= 6)
          rok = mbar_wait(&wempty[(i - 6) % kWSlots], ((i - 6) / kWSlots) & 1);
        if (rok && m1 + m2 + m > kGroupRing && i >= 4)
          rok = mbar_wait(&wempty[(i - 4) % kWSlots], ((i - 4) / kWSlots) & 1);
        if (rok && m1 + m > kGroupRing && i >= 2)
          rok = mbar_wait(&wempty[(i - 2) % kWSlots], ((i - 2) / kWSlots) & 1);
        const int row0 = issued & (kGroupRing - 1);
        issued += m;
        m3 = m2;
        m2 = m1;
        m1 = m;
        if (!rok) {
          // no barrier follows in this tile: the group stops together at the next one
          set_abort(s_abort, p.flags);
          continue;
        }
        if (lane == 0) {
          if (quarter == 0) {
            ws.row0 = row0;
            ws.m = m;
          }
          mbar_arrive_expect_tx(&vfull[slot], static_cast<uint32_t>(__popc(bal) * kRowBytes));
          if (quarter == 0) s_varm[slot] = s_varm[slot] + 1;
        }
        __syncwarp();
        if (surv)
          bulk_load(gring + ((row0 + e) & (kGroupRing - 1)) * C::ring_pitch,
                    p.v + (static_cast<int64_t>(u) * p.ncap + j) * kRowBytes, kRowBytes, &vfull[slot]);
      }
      if (i < ie) break;  // stopped early
    }
    __syncwarp();
  } else if (warp == kWarpHist) {
    // ------------------------------------------------------------------ selection scores
    // Tile by tile in order: sigma of the keys j < n to global memory, and counted into
    // the histogram of the order key's top 11 bits; at the end of each stretch of a unit
    // the histogram is added to the unit's global one and cleared.
    if (p.sel != nullptr) {
      int i = 0;
      for (int pc = 0; pc < K; ++pc) {
        const int4 pe = s_piece[pc];
        int u = pe.x, tl = pe.y;
        const int ie = i + pe.z;
        for (; i < ie; ++i, next_tile(tl, u, TU)) {
          const int slot = static_cast<int>(i % kWSlots);
          const bool ok = __all_sync(0xffffffffu, !*s_abort && mbar_wait(&sfull[slot], (i / kWSlots) & 1));
          if (!ok) {
            set_abort(s_abort, p.flags);
            break;
          }
          const WSlot<G, KV8> &ws = wslots[slot];
          float sg[4];
  #pragma unroll
          for (int r = 0; r < 4; ++r) sg[r] = ws.sig[lane + 32 * r];
          float used = (sg[0] + sg[1]) + (sg[2] + sg[3]);
          used = __shfl_sync(0xffffffffu, used, 31) + used;  // the whole warp takes part
          __syncwarp();
          if (lane == 0) mbar_arrive_after(&wempty[slot], used);
          float *dst = p.sel + static_cast<int64_t>(u) * p.ncap + tl * kTileKeys;
  #pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int row = lane + 32 * r;
            if (tl * kTileKeys + row < p.n) {
              dst[row] = sg[r];
              atomicAdd(&s_hist[order_key(sg[r]) >> 21], 1u);
            }
          }
          if (i + 1 == ie && pc + 1 == K) {
            // the CTA's last stretch: the whole CTA flushes it once every role is done
            __syncwarp();
            if (lane == 0) *s_final_hist = u;
          } else if (i + 1 == ie || tl + 1 == TU) {
            __syncwarp();
            pdl_wait_primary();  // the global histogram has been zeroed
            for (int bin = lane; bin < kHistBins; bin += 32) {
              const uint32_t cnt = s_hist[bin];
              if (cnt) {
                atomicAdd(&p.hist[static_cast<int64_t>(u) * kHistBins + bin], cnt);
                s_hist[bin] = 0u;
              }
            }
            __syncwarp();
          }
        }
        if (i < ie) break;  // stopped early
      }
    }
    __syncwarp();
  } else if (warp >= kWarpNorm) {
    // ------------------------------------------------------------------ key norms
    // One thread per key of each landed tile: 1 / sqrt(mean(k^2) + eps) (8-bit caches: the
    // key's two scales, passed along; the epilogue finishes the norm from the tensor cores'
    // sum of squared codes).  The stage is released as soon as these four warps and the
    // tile's MMAs are done with it.
    const int row = (warp - kWarpNorm) * 32 + lane;
    int seg = -1;
    int i = 0;
    for (int pc = 0; pc < K; ++pc) {
      const int4 pe = s_piece[pc];
      int u = pe.x, tl = pe.y;
      const int ib = i, ie = i + pe.z;
      (void)ib;  // the stretch starts matter to the 8-bit caches only
      for (; i < ie; ++i, next_tile(tl, u, TU)) {
        if (__any_sync(0xffffffffu, *s_abort)) break;
        if constexpr (KV8) {
          if (i == ib || tl == 0) {
            // the stretch's query as E4M3 terms for the tensor cores
            ++seg;
            const int qb = seg & 1;
            const bool qok = __all_sync(0xffffffffu,
                                        mbar_wait(&qfull[qb], (seg >> 1) & 1) &&
                                            (seg < 2 || mbar_wait(&q8empty[qb], ((seg >> 1) - 1) & 1)));
            if (!qok) {
              set_abort(s_abort, p.flags);
              break;
            }
            build_q8_terms<G>(sQ + qb * kQBufBytes, sQ8 + qb * kQ8BufBytes, row);
            fence_proxy_async_smem();  // the terms are read by the tensor cores
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&q8full[qb]);
              mbar_arrive(&qempty[qb]);
            }
          }
        }
        const int s = static_cast<int>(i % kStages);
        const int ns = static_cast<int>(i % kNormSlots);
        const bool ok = __all_sync(0xffffffffu,
                                   mbar_wait(&full[2 * s + (i & 1)], (i / kFullPeriod) & 1) &&
                                       (i < kNormSlots ||
                                        mbar_wait(&rkempty[ns], ((i / kNormSlots) - 1) & 1)));
        if (!ok) {
          set_abort(s_abort, p.flags);
          break;
        }
        // chunk order rotated by row so 8 neighbouring rows hit 8 different bank groups
        // (the swizzle permutes 16-byte chunks within a row; the order does not matter)
        const uint8_t *st = sK + s * C::stage_bytes;
        const uint8_t *rowp = st + row * 128;
        float rk, vsc = 0.0f, done;
        if constexpr (KV8) {
          // the key's two scales go on with the tile; its sum of squared codes comes from the
          // tensor cores (codes . codes^T)
          const float ks = reinterpret_cast<const float *>(st + C::tile_bytes)[row];
          vsc = reinterpret_cast<const float *>(st + C::tile_bytes + C::scale_bytes)[row];
          const float dep = ks + vsc;  // every lane's value depends on its reads
          done = __shfl_sync(0xffffffffu, dep, 0) + __shfl_sync(0xffffffffu, dep, 31);
          rk = ks;
          (void)rowp;
        } else {
          float a[8];
  #pragma unroll
          for (int c = 0; c < 8; ++c) a[c] = 0.0f;
  #pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int pc = (c ^ (row & 7)) * 16;
            const uint4 x0 = *reinterpret_cast<const uint4 *>(rowp + pc);
            const uint4 x1 = *reinterpret_cast<const uint4 *>(rowp + C::half_bytes + pc);
            sq_acc_bf16x2(x0.x, a[0], a[1]);
            sq_acc_bf16x2(x0.y, a[2], a[3]);
            sq_acc_bf16x2(x0.z, a[4], a[5]);
            sq_acc_bf16x2(x0.w, a[6], a[7]);
            sq_acc_bf16x2(x1.x, a[0], a[1]);
            sq_acc_bf16x2(x1.y, a[2], a[3]);
            sq_acc_bf16x2(x1.z, a[4], a[5]);
            sq_acc_bf16x2(x1.w, a[6], a[7]);
          }
          // every lane's sum depends on all of its reads of the stage
          const float ss = ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
          done = __shfl_sync(0xffffffffu, ss, 0) + __shfl_sync(0xffffffffu, ss, 31);
          rk = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_after(&empty[s], done);
        s_rk[ns * kTileKeys + row] = rk;
        if constexpr (KV8) s_vs[ns * kTileKeys + row] = vsc;
        __syncwarp();
        if (lane == 0) mbar_arrive(&rkfull[ns]);
      }
      if (i < ie) break;  // stopped early
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ V accumulators
    // O^T[d][h] += sum_e V[e][d] w_h[e] on the tensor cores (m16n8k16 bf16 MMAs), kAccStep
    // survivors per step: warp aw owns dims 32aw .. 32aw+31 (two 16-dim M tiles), the N = 8
    // columns are the heads (G = 4 leaves four of them zero).  The A operand is read from
    // the ring by ldmatrix (rows past the tile's list read a zero row); the weights enter
    // as two bf16 parts (hi + lo, about 16 bits), and the denominators sum the fp32
    // weights.  8-bit caches: each step first widens its code rows (exactly) to bf16 rows
    // in a staging block, a quarter of the rows per warp, and the weights carry the V
    // scales.  The four warps take every decision to stop together (bar.red.and), so none
    // is left at a barrier the others have abandoned.
    const int aw = warp - kWarpAcc;
    const int g = lane >> 2, t = lane & 3;
    const int mat = lane >> 3, mr = lane & 7;
    const uint32_t zero_u32 = smem_u32(smem + L::zero_off);
    const uint32_t ring_u32 = smem_u32(sRing);
    uint8_t *stage = smem + L::stage_off;
    float o[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
    float den = 0.0f;  // lane (g, t): head g's weights of rows 2t, 2t+1, 2t+8, 2t+9 of each step
    int seg_surv = 0, step = 0;
    int i = 0;
    for (int pc = 0; pc < K; ++pc) {
      const int4 pe = s_piece[pc];
      int u = pe.x, tl = pe.y;
      const int ie = i + pe.z;
      const int q = pe.w;
      for (; i < ie; ++i, next_tile(tl, u, TU)) {
        const int slot = static_cast<int>(i % kWSlots);
        const bool ok = !*s_abort && mbar_wait(&vfull[slot], (i / kWSlots) & 1);
        if (!named_bar_and(kAccBar, 128, ok)) {
          set_abort(s_abort, p.flags);
          break;
        }
        const WSlot<G, KV8> &ws = wslots[slot];
        const int row0 = ws.row0, m = ws.m;
        const uint32_t gring_u32 = ring_u32 + (i % kGroups) * kGroupRing * C::ring_pitch;
        for (int e0 = 0; e0 < m; e0 += kAccStep, ++step) {
          uint32_t base_u32;  // row 0 of this step's A operand
          if constexpr (KV8) {
            // widen rows e0 + 4aw .. +3 (lane: codes 4 lane .. 4 lane + 3) into the staging block
            uint8_t *sb = stage + (step & 1) * kAccStep * kAccPitch;
  #pragma unroll
            for (int k = 0; k < kAccStep / 4; ++k) {
              const int e = e0 + aw * (kAccStep / 4) + k;
              if (e < m) {
                const uint32_t c4 = *reinterpret_cast<const uint32_t *>(
                    sRing + (i % kGroups) * kGroupRing * C::ring_pitch +
                    ((row0 + e) & (kGroupRing - 1)) * C::ring_pitch + lane * 4);
                float v0, v1, v2, v3;
                e4m3x4_to_f32(c4, v0, v1, v2, v3);
                *reinterpret_cast<uint2 *>(sb + (e - e0) * kAccPitch + lane * 8) =
                    make_uint2(pack_bf16x2(v0, v1), pack_bf16x2(v2, v3));
              }
            }
            named_bar_sync(kAccBar, 128);  // the step's rows are widened
            base_u32 = smem_u32(sb);
          }
          // A: this lane's matrix row r of the step (matrices: rows 0-7 / 8-15 x dims +0 / +8)
          const int r = (mat >> 1) * 8 + mr;
          uint32_t raddr;
          if constexpr (KV8)
            raddr = e0 + r < m ? base_u32 + r * kAccPitch : zero_u32;
          else
            raddr = e0 + r < m ? gring_u32 + ((row0 + e0 + r) & (kGroupRing - 1)) * C::ring_pitch
                               : zero_u32;
          uint32_t a[2][4];
  #pragma unroll
          for (int mt = 0; mt < 2; ++mt)
            ldmatrix_x4_trans(a[mt], raddr + (2 * (2 * aw + mt) + (mat & 1)) * 16);
          // B: head g's weights of rows 2t, 2t+1 (b0) and 2t+8, 2t+9 (b1)
          float w[4], wq[4];
  #pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int e = e0 + 2 * t + (k & 1) + (k >> 1) * 8;
            const bool have = e < m && g < G;
            w[k] = have ? ws.w[e][g < G ? g : 0] : 0.0f;
            wq[k] = w[k];
            if constexpr (KV8) wq[k] = have ? w[k] * ws.vs[e] : 0.0f;
          }
          den += (w[0] + w[1]) + (w[2] + w[3]);
          const uint32_t h0 = pack_bf16x2(wq[0], wq[1]), h1 = pack_bf16x2(wq[2], wq[3]);
          const uint32_t l0 = pack_bf16x2(wq[0] - bf16lo(h0), wq[1] - bf16hi(h0));
          const uint32_t l1 = pack_bf16x2(wq[2] - bf16lo(h1), wq[3] - bf16hi(h1));
  #pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            mma_16816_bf16(o[mt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], h0, h1);
            mma_16816_bf16(o[mt], a[mt][0], a[mt][1], a[mt][2], a[mt][3], l0, l1);
          }
        }
        seg_surv += m;
        // the running sums depend on every ring row and weight this lane read
        float used = den + ((o[0][0] + o[0][1]) + (o[0][2] + o[0][3])) +
                     ((o[1][0] + o[1][1]) + (o[1][2] + o[1][3]));
        used = __shfl_sync(0xffffffffu, used, 31) + used;
        __syncwarp();
        if (lane == 0) mbar_arrive_after(&wempty[slot], used);
        if (i + 1 == ie || tl + 1 == TU) {
          float *r = p.rec + static_cast<int64_t>(q + u) * p.rec_stride;
          // this warp's dims of every head
  #pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const int d = 32 * aw + 16 * mt + g;
            if (2 * t < G) {
              r[(2 * t) * kHeadDim + d] = o[mt][0];
              r[(2 * t) * kHeadDim + d + 8] = o[mt][2];
            }
            if (2 * t + 1 < G) {
              r[(2 * t + 1) * kHeadDim + d] = o[mt][1];
              r[(2 * t + 1) * kHeadDim + d + 8] = o[mt][3];
            }
            o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.0f;
          }
          // every warp sees the same weights: warp 0 writes the denominators
          float dh = den + __shfl_xor_sync(0xffffffffu, den, 1);
          dh += __shfl_xor_sync(0xffffffffu, dh, 2);
          den = 0.0f;
          if (aw == 0 && t == 0 && g < G) r[G * kHeadDim + g] = dh;

          // the stretch's survivors are counted in (integer sums: the same in any order); the
          // records are summed by full_combine_kernel, which follows this kernel
          if (aw == 0 && lane == 0) {
            pdl_wait_primary();  // the survivor counts have been zeroed
            atomicAdd(&p.n_surv[u], seg_surv);
          }
          seg_surv = 0;
        }
      }
      if (i < ie) break;  // stopped early
    }
    __syncwarp();
  }

  __syncthreads();
  // The histogram of the CTA's last stretch, with every thread of the CTA.
  if (*s_final_hist >= 0) {
    pdl_wait_primary();  // the global histogram has been zeroed
    const int64_t hu = *s_final_hist;
    for (int bin = threadIdx.x; bin < kHistBins; bin += kThreads) {
      const uint32_t cnt = s_hist[bin];
      if (cnt) atomicAdd(&p.hist[hu * kHistBins + bin], cnt);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && *s_abort) {
    // No copy may still be landing in shared memory when the CTA leaves.  Without an abort
    // every copy issued was waited for by the role that used it; after one, wait (bounded)
    // for the last armed phase of every barrier that a copy completes.
    const int k_issued = *s_k_issued, q_issued = *s_q_issued;
    for (int f = 0; f < 2 * kStages; ++f) {
      // tiles i < k_issued with i % kStages == f / 2 and i % 2 == f % 2
      int uses = 0;
      for (int i = 0; i < k_issued && i < kFullPeriod; ++i)
        if (i % kStages == f / 2 && (i & 1) == (f & 1))
          uses += (k_issued - 1 - i) / kFullPeriod + 1;
      if (uses) mbar_wait(&full[f], (uses - 1) & 1);
    }
    for (int w = 0; w < kWSlots; ++w) {
      const int uses = s_varm[w];
      if (uses) mbar_wait(&vfull[w], (uses - 1) & 1);
    }
    for (int q = 0; q < 2; ++q) {
      const int uses = q_issued > q ? (q_issued - 1 - q) / 2 + 1 : 0;
      if (uses) mbar_wait(&qfull[q], (uses - 1) & 1);
    }
  }
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::tmem_cols);
  }
}

// Zeroes what the decode accumulates into with atomics: the selection histogram (if any)
// and the survivor counts, once the kernel before it has finished.  It lets the decode
// kernel launch at once, which sets up and then waits for it before its first load.
__global__ void __launch_bounds__(256) full_zero_kernel(uint4 *hist, int64_t hist_vecs,
                                                        int32_t *n_surv, int64_t units) {
  pdl_launch_dependents();  // the decode kernel sets up meanwhile; it waits for this one
  pdl_wait_primary();       // what the earlier kernels read here is no longer needed
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t i = t; i < hist_vecs; i += stride) hist[i] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t i = t; i < units; i += stride) n_surv[i] = 0;
}

// out[u][h][d] = num / (c + den), num and den the sums of unit u's records (its stretches in
// the pieces c0 .. c1 that hold its tiles, records c0 + u .. c1 + u), in a fixed order.  One CTA
// of dc x S threads per dc dims of a (unit, head) (dc = 128, 64 or 32, so that there are
// about as many CTAs as SMs), S = the slices (a power of two, at most 8, from the records per
// unit): thread (s, d) sums records s, s + S, s + 2S, ... of its dim (up to eight loads in
// flight), and the S slices are added in slice order; each slice's first warp sums the
// head's denominators the same way.
constexpr int kCombMaxSlices = 8;
constexpr int kCombLoads = 8;
template <int G>
__global__ void __launch_bounds__(kHeadDim * kCombMaxSlices) full_combine_kernel(const FullParams p,
                                                                                 int dc,
                                                                                 int after_select) {
  __shared__ float s_num[kCombMaxSlices][kHeadDim];
  __shared__ float s_den[kCombMaxSlices];
  const int S = static_cast<int>(blockDim.x) / dc;
  const int per_head = kHeadDim / dc;
  const int64_t u = blockIdx.x / (G * per_head);
  const int h = static_cast<int>(blockIdx.x / per_head % G);
  const int dl = static_cast<int>(threadIdx.x) % dc, sl = static_cast<int>(threadIdx.x) / dc;
  const int d = static_cast<int>(blockIdx.x % per_head) * dc + dl;
  // the unit's first and last piece (split_piece_of_tile, in 32-bit arithmetic when T * Q fits)
  int64_t c0, c1;
  if (((p.T * p.Q) >> 32) == 0) {
    const uint32_t T32 = static_cast<uint32_t>(p.T), Q32 = static_cast<uint32_t>(p.Q);
    const uint32_t t0 = static_cast<uint32_t>(u * p.TU), t1 = t0 + static_cast<uint32_t>(p.TU) - 1u;
    c0 = ((t0 + 1u) * Q32 - 1u) / T32;
    c1 = ((t1 + 1u) * Q32 - 1u) / T32;
  } else {
    c0 = split_piece_of_tile(u * p.TU, p.T, p.Q);
    c1 = split_piece_of_tile(u * p.TU + p.TU - 1, p.T, p.Q);
  }
  const int parts = static_cast<int>(c1 - c0 + 1);
  const float *rr = p.rec + (c0 + u) * p.rec_stride;
  const int col = h * kHeadDim + d;
  // Right after the decode kernel, the CTA is launched while that kernel runs: its first
  // record lines go to L2 (with their address translations) before the wait (a prefetch
  // reads nothing into the SM).  After a selection kernel, the CTA starts only once every
  // selection CTA has passed its own wait for the decode kernel, so every record is
  // written already; it runs beside the selection and waits for it only at the end, so
  // that the kernels after it see the selection finished.  The records are read from L2.
  if (!after_select) {
    if (sl < parts)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(rr + static_cast<int64_t>(sl) * p.rec_stride + col));
    pdl_wait_primary();  // every record is written
  }
  pdl_launch_dependents();
  float num = 0.0f, den = 0.0f;
  for (int k0 = sl; k0 < parts; k0 += S * kCombLoads) {
    float x[kCombLoads], y[kCombLoads];
#pragma unroll
    for (int k = 0; k < kCombLoads; ++k) {
      const int kk = k0 + k * S;
      x[k] = kk < parts ? __ldcg(rr + static_cast<int64_t>(kk) * p.rec_stride + col) : 0.0f;
      y[k] = kk < parts && dl < 32 ? __ldcg(rr + static_cast<int64_t>(kk) * p.rec_stride + G * kHeadDim + h)
                                   : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < kCombLoads; ++k) {
      num += x[k];
      den += y[k];
    }
  }
  s_num[sl][dl] = num;
  if (dl == 0) s_den[sl] = den;
  __syncthreads();
  if (sl == 0) {
    float n = s_num[0][dl], z = s_den[0];
    for (int k = 1; k < S; ++k) {
      n += s_num[k][dl];
      z += s_den[k];
    }
    z += p.c;
    p.out[u * G * kHeadDim + col] = z != 0.0f ? n / z : 0.0f;
  }
  if (after_select) pdl_wait_primary();  // the selection has finished
}

template <int G, bool KV8>
cudaError_t launch_full_decode_t(const CUtensorMap &tm_k, const CUtensorMap &tm_q,
                                 const CUtensorMap &tm_ks, const CUtensorMap &tm_vs,
                                 const FullParams &p, int64_t units, cudaStream_t stream,
                                 const SelectJob *sj) {
  const int smem = Smem<G, KV8>::alloc;
  auto kernel = p.K > 1 ? full_decode_kernel<G, KV8, true> : full_decode_kernel<G, KV8, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t hist_vecs = p.hist ? units * kHistBins / 4 : 0;
  const int64_t work = hist_vecs > units ? hist_vecs : units;
  const int64_t zblocks = (work + 255) / 256;
  e = launch_pdl(full_zero_kernel, dim3(static_cast<unsigned>(zblocks < 1024 ? zblocks : 1024)),
                 dim3(256), 0, stream, 0u, reinterpret_cast<uint4 *>(p.hist), hist_vecs,
                 p.n_surv, units);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kernel, dim3(static_cast<unsigned>(p.P)), dim3(kThreads),
                 static_cast<size_t>(smem), stream, 0u, tm_k, tm_q, tm_ks, tm_vs, p);
  if (e != cudaSuccess) return e;
  if (sj) {
    e = launch_select(p.sel, p.hist, units, p.n, p.ncap, sj->topk, sj->recent, sj->idx,
                      sj->idx_stride, sj->count, sj->workspace, p.flags, sj->sm_count, stream);
    if (e != cudaSuccess) return e;
  }
  // slices: the records of the unit with the most, rounded up to a power of two (at most 8)
  const int64_t most = (p.TU * p.Q + p.T - 1) / p.T + 1;
  int slices = 1;
  while (slices < kCombMaxSlices && slices < most) slices <<= 1;
  // dims per CTA: 128, halved (to 32 at least) while there are fewer CTAs than SMs
  int dc = kHeadDim;
  while (dc > 32 && units * G * (kHeadDim / dc) < p.P) dc >>= 1;
  return launch_pdl(full_combine_kernel<G>, dim3(static_cast<unsigned>(units * G * (kHeadDim / dc))),
                    dim3(dc * slices), 0, stream, 0u, p, dc, sj ? 1 : 0);
}

}  // namespace

FullSplit full_split(int64_t units, int64_t ctx_len, int sm_count, int max_pieces) {
  FullSplit sp;
  sp.units = units;
  sp.tiles_per_unit = (ctx_len + kTileKeys - 1) / kTileKeys;
  sp.tiles = units * sp.tiles_per_unit;
  sp.ctas = static_cast<int32_t>(sp.tiles < sm_count ? sp.tiles : sm_count);
  // K: as many pieces of kMinPieceTiles tiles or more as a CTA's share holds, odd, at most
  // max_pieces; every piece then holds at least one tile (Q <= T)
  int64_t k = sp.ctas > 0 ? sp.tiles / sp.ctas / kMinPieceTiles : 1;
  if (k > max_pieces) k = max_pieces;
  if (k < 1) k = 1;
  if (k % 2 == 0) --k;
  sp.pieces = static_cast<int32_t>(k * sp.ctas);
  return sp;
}

int full_record_floats(int G) {
  const int f = G * kHeadDim + G + 1;
  return (f + 3) & ~3;
}

size_t full_workspace_bytes(const FullSplit &sp, int G) {
  // the records: one slot per (piece, unit) stretch, slots q + u < Q + units
  return (static_cast<size_t>(sp.units + sp.pieces) * full_record_floats(G) * sizeof(float) + 255) &
         ~static_cast<size_t>(255);
}

cudaError_t launch_full_decode(int G, bool kv8, const CUtensorMap &tm_k, const CUtensorMap &tm_q,
                               const CUtensorMap *tm_ks, const CUtensorMap *tm_vs,
                               const void *v_cache, float *sel_scores, float *head_scores,
                               uint32_t *sel_hist, void *workspace,
                               float *out, int32_t *n_surv, float c, uint32_t *flags,
                               const FullSplit &sp, int64_t n,
                               int64_t ncap, int Hq, int Hkv, float alpha, float eps,
                               cudaStream_t stream, const SelectJob *sj) {
  if (sp.tiles == 0) return cudaSuccess;
  if (sj && (!sel_scores || !sel_hist)) return cudaErrorInvalidValue;
  FullParams p;
  p.v = static_cast<const uint8_t *>(v_cache);
  p.sel = sel_scores;
  p.hist = sel_hist;
  p.hsel = head_scores;
  p.rec = static_cast<float *>(workspace);
  p.out = out;
  p.n_surv = n_surv;
  p.c = c;
  p.flags = flags;
  p.T = sp.tiles;
  p.TU = sp.tiles_per_unit;
  p.n = n;
  p.ncap = ncap;
  p.P = sp.ctas;
  p.Q = sp.pieces;
  p.K = sp.pieces / sp.ctas;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.rec_stride = full_record_floats(G);
  p.alpha = alpha;
  p.eps = eps;
  if (kv8) {
    if (!tm_ks || !tm_vs) return cudaErrorInvalidValue;
    if (G == 4) return launch_full_decode_t<4, true>(tm_k, tm_q, *tm_ks, *tm_vs, p, sp.units, stream, sj);
    if (G == 8) return launch_full_decode_t<8, true>(tm_k, tm_q, *tm_ks, *tm_vs, p, sp.units, stream, sj);
    return cudaErrorInvalidValue;
  }
  // the bf16 kernel does not read the scale maps
  if (G == 4) return launch_full_decode_t<4, false>(tm_k, tm_q, tm_k, tm_k, p, sp.units, stream, sj);
  if (G == 8) return launch_full_decode_t<8, false>(tm_k, tm_q, tm_k, tm_k, p, sp.units, stream, sj);
  return cudaErrorInvalidValue;
}

}  // namespace embla
