// Softmax decode over a list of cache rows: the sparse layers (rows chosen by the
// selection) and the sliding-window layers (the newest `window` rows of a ring).
//
// Source: "The Architecture of Embla 1", section "Three kinds of attention":
//   Sparse  — the block's full-layer cache restricted to the selected keys, its own
//             softmax, no position encoding;
//   Sliding window — the newest 128 keys, ordinary softmax, rotary position
//             embedding (the query is rotated here; keys were rotated when written).
//
// Each warp first copies all of its rows (K and V, 256 bytes each) into its own part of
// shared memory with one bulk copy per row, so every row of the warp is in flight at
// once, then folds them in chunks of 8 rows; a row is read by 16 lanes (8 dims each, one
// 16-byte load of K and of V), so a warp's two lane groups take 4 rows each.  The
// group's 4 x G partial dot products are summed by a reduce-scatter over its 16 lanes
// and gathered back, then every lane updates its group's running max m, sum l and its
// 8-dim slice of the unnormalised output, rescaling once per chunk.  Warps merge in
// shared memory (reusing the rows' space) by rescaling with exp(m_w - M).
// A sparse layer spreads each (batch, KV-head) unit over a cluster of up to 8 CTAs that merge
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
constexpr int kMaxCluster = 8;     // CTAs per sparse unit, at most
constexpr int kWarpRows = 20;      // rows a warp stages per pass
constexpr int kStageBytes = kWarps * kWarpRows * 2 * kHeadDim * 2;  // 80 KB: K and V rows
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

// Chunk rows from a warp's staged rows: present[r] says whether the group's row r holds
// a row; sK/sV point at the group's row 0 (rows 256 bytes apart).
__device__ __forceinline__ void load_chunk(Chunk &c, const uint8_t *sK, const uint8_t *sV,
                                           uint32_t present, int sl) {
  c.present = present;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    if ((present >> r) & 1u) {
      c.k[r] = *reinterpret_cast<const uint4 *>(sK + r * kRowBytes + sl * 16);
      c.v[r] = *reinterpret_cast<const uint4 *>(sV + r * kRowBytes + sl * 16);
    } else {
      c.k[r] = make_uint4(0u, 0u, 0u, 0u);
      c.v[r] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// The rows of one warp in shared memory: K rows then V rows, kWarpRows each.
struct WarpStage {
  uint8_t *k, *v;
  __device__ WarpStage(uint8_t *stage, int warp)
      : k(stage + warp * kWarpRows * 2 * kRowBytes), v(k + kWarpRows * kRowBytes) {}
};

// Copy up to kWarpRows rows (row indices from `row_of(i)` for i < nrows, negative =
// absent) of K and V into the warp's stage: the two lane groups take alternate rows, each
// lane one 16-byte piece of the row's K and of its V, all in flight together.  Returns
// the mask of rows present (bit i).
template <class RowOf>
__device__ __forceinline__ uint32_t stage_rows(const WarpStage &ws, const uint8_t *K,
                                               const uint8_t *V, int nrows, RowOf row_of,
                                               int lane) {
  const int64_t mine = lane < nrows ? row_of(lane) : -1;
  const uint32_t present = __ballot_sync(0xffffffffu, mine >= 0);
  const int grp = lane >> 4, sl = lane & 15;
  for (int r2 = 0; r2 < (nrows + 1) / 2; ++r2) {
    const int r = 2 * r2 + grp;
    const int64_t row = __shfl_sync(0xffffffffu, mine, r < 32 ? r : 31);
    if (r < nrows && row >= 0) {
      cp_async16(ws.k + r * kRowBytes + sl * 16, K + row * kRowBytes + sl * 16);
      cp_async16(ws.v + r * kRowBytes + sl * 16, V + row * kRowBytes + sl * 16);
    }
  }
  cp_async_wait_all();
  __syncwarp();
  return present;
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
//
// Tensor-core path.  A warp takes blocks of 16 selected rows.  It copies their K and V
// rows into shared memory (16-byte pieces permuted within each row by row % 8, so that
// the 8 rows an ldmatrix reads fall in different banks), then
//   S  = Q . K^T  as m16n8k16 MMAs: M = query heads (G of 16 used), N = 8 rows, K = dims;
//   P  = exp2(tau2 * S - m) with a running max m and sum l per head (the accumulator of
//        S holds, per lane, head lane/4 and rows 2(lane%4), +1 of each 8-row tile, which
//        is exactly the B operand layout the next product needs);
//   O^T += V^T . P^T  as MMAs with M = dims (8 tiles of 16), N = heads, K = the 16 rows.
// P enters the second product as two bf16 parts (hi + lo); l sums the fp32 values.

// 9 warps x 16 rows = 144 rows: a cluster of 8 covers 1152 (two CTAs to an SM); the wide
// variant, 18 warps and a cluster of 4 (one CTA to an SM), takes over when 8 CTAs per unit
// would put two on some SMs but 4 fit one each
constexpr int kSpWarps = 9;
constexpr int kSpWideWarps = 18;
constexpr int kSpThreads = kSpWarps * 32;
constexpr int kSpBlock = 16;                // rows per warp step
constexpr int kSpStage = 2 * kSpBlock * kRowBytes;  // K and V rows of one step: 8 KB

template <int G, int W = kSpWarps>
struct SpMerge {
  float m[W][G], l[W][G];
  float acc[W][G][kHeadDim];
  float f[W][G];  // exp2(m[w][h] - the CTA's max for head h)
  float cm[G], cl[G];
  float ca[G][kHeadDim];
};

struct SparseParams {
  const uint16_t *q;
  const uint8_t *K, *V;
  const float *ks, *vs;  // per-token scales of 8-bit caches (else null)
  const int32_t *idx, *count;
  float *out;
  uint32_t *flags;
  int64_t n, ncap;
  int idx_stride, rows_per_cta;
  int cl;    // CTAs per unit (the cluster size): 1, 2, 4 or 8
  int wide;  // the 18-warp variant (cluster of 4)
  float tau;
  // cache plane of unit u: u itself, or for a selection per query head (one unit per
  // (sequence, query head)) (u / Hq) * Hkv + (u % Hq) / Gq
  int per_head, Hq, Hkv, Gq;
  __device__ int64_t plane(int64_t u) const {
    return per_head ? (u / Hq) * Hkv + (u % Hq) / Gq : u;
  }
};

// byte offset of 16-byte piece c of staged row r
__device__ __forceinline__ uint32_t sp_piece(int r, int c) {
  return static_cast<uint32_t>(r * kRowBytes + ((c ^ (r & 7)) << 4));
}

// After every warp has written its running max, sum and unnormalised output into mg:
// combine the warps, then the cluster's CTAs (through distributed shared memory), and
// write this CTA's share of the unit's G x 128 outputs.
template <int G, int CL, int W = kSpWarps>
__device__ __forceinline__ void sp_combine(SpMerge<G, W> &mg, int rank, int64_t u, float *out_base) {
  constexpr int kT = W * 32;
  cg::cluster_group cluster = cg::this_cluster();
  __syncthreads();
  // per head (warp h, lane w for the CTA's warp w): the CTA's running max and sum, and each
  // warp's rescaling factor (once, not once per output element); the sum by a fixed
  // shuffle tree
  static_assert(W <= 32 && G <= W, "a lane per warp, a warp per head");
  if (static_cast<int>(threadIdx.x >> 5) < G) {
    const int h = threadIdx.x >> 5, w = threadIdx.x & 31;
    const float mw = w < W ? mg.m[w][h] : -INFINITY;
    float M = mw;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float f = w < W && M != -INFINITY ? exp2f(mw - M) : 0.0f;
    if (w < W) mg.f[w][h] = f;
    float L = w < W ? mg.l[w][h] * f : 0.0f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (w == 0) {
      mg.cm[h] = M;
      mg.cl[h] = L;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * kHeadDim; i += kT) {
    const int h = i / kHeadDim, d = i % kHeadDim;
    // four chains (warps w = c mod 4), added in a fixed order
    float A[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < W; ++w) A[w & 3] = fmaf(mg.acc[w][h][d], mg.f[w][h], A[w & 3]);
    mg.ca[h][d] = (A[0] + A[1]) + (A[2] + A[3]);
  }
  // the cluster's CTAs each finish their share of the outputs from all the CTAs' states
  cluster.sync();
  constexpr int per = G * kHeadDim / CL;  // outputs of this CTA (at most 4 per thread)
  static_assert(per <= 4 * kT, "at most 4 outputs per thread");
  float res[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    res[k] = 0.0f;
    const int li = threadIdx.x + k * kT;
    if (li < per) {
      const int i = rank * per + li;
      const int h = i / kHeadDim, d = i % kHeadDim;
      float cmv[CL];
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < CL; ++c) {
        cmv[c] = cluster.map_shared_rank(&mg, c)->cm[h];
        M = fmaxf(M, cmv[c]);
      }
      float L = 0.0f, A = 0.0f;
      if (M != -INFINITY) {
#pragma unroll
        for (int c = 0; c < CL; ++c) {
          const SpMerge<G, W> *o2 = cluster.map_shared_rank(&mg, c);
          const float f = exp2f(cmv[c] - M);
          L = fmaf(o2->cl[h], f, L);
          A = fmaf(o2->ca[h][d], f, A);
        }
      }
      res[k] = L > 0.0f ? A / L : 0.0f;
    }
  }
  cluster_arrive();  // done reading the other CTAs' shared memory
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int li = threadIdx.x + k * kT;
    if (li < per) out_base[u * G * kHeadDim + rank * per + li] = res[k];
  }
  cluster_wait();  // and they are done reading this one's
}

template <int G, int CL, int W = kSpWarps>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(W * 32, W <= kSpWarps ? 2 : 1)
    sparse_decode_kernel(const SparseParams p) {
  pdl_wait_primary();  // the selection and the query are complete
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];  // staged rows, then the merge state
  SpMerge<G, W> &mg = *reinterpret_cast<SpMerge<G, W> *>(smem);
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t u = blockIdx.x / CL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int32_t *idx = p.idx + u * p.idx_stride;
  const int r0 = rank * p.rows_per_cta;
  // the first block's indices are requested together with the count, not after it (entries
  // past the count are read but not used)
  int32_t jfirst = -1;
  {
    const int b = r0 + warp * kSpBlock + lane;
    if (lane < kSpBlock && b < p.idx_stride && b < r0 + p.rows_per_cta) jfirst = idx[b];
  }
  int cnt = p.count[u];
  cnt = cnt < 0 ? 0 : (cnt > p.idx_stride ? p.idx_stride : cnt);
  const uint8_t *Ku = p.K + p.plane(u) * p.ncap * kRowBytes;
  const uint8_t *Vu = p.V + p.plane(u) * p.ncap * kRowBytes;
  const float tau2 = p.tau * kLog2e;
  uint8_t *sK = smem + warp * kSpStage;
  uint8_t *sV = sK + kSpBlock * kRowBytes;
  const uint32_t sK_u = smem_u32(sK), sV_u = smem_u32(sV);

  // query as the A operand of S = Q . K^T: row g (head g), dims 16ks + 2t, +1 and +8, +9
  uint32_t qa0[8], qa2[8];
  {
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(p.q + (u * G + (g < G ? g : 0)) * kHeadDim);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa0[ks] = g < G ? qrow[8 * ks + t] : 0u;
      qa2[ks] = g < G ? qrow[8 * ks + 4 + t] : 0u;
    }
  }
  float m = -INFINITY, l = 0.0f;  // head g's running max (base 2) and sum
  float o[8][4];                  // O^T tile i: dims 16i + g (+8), heads 2t, 2t + 1
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;

  const int r1 = min(cnt, r0 + p.rows_per_cta);
  for (int b0 = r0 + warp * kSpBlock; b0 < r1; b0 += W * kSpBlock) {
    // stage: lane r < 16 looks up row r (absent past the count, or for an index outside
    // [0, n), which is flagged); then each copy instruction moves two whole rows, lanes
    // 0-15 the 16 pieces of one and lanes 16-31 those of the next; absent rows are zeros
    int64_t j = -1;
    if (lane < kSpBlock && b0 + lane < r1) {
      const int32_t jj = b0 == r0 + warp * kSpBlock ? jfirst : idx[b0 + lane];
      if (jj < 0 || static_cast<int64_t>(jj) >= p.n)
        atomicOr(p.flags, kFlagIndexRange);
      else
        j = jj;
    }
    const uint32_t present = __ballot_sync(0xffffffffu, j >= 0);  // bit r: row r
    const int piece = lane & 15;
#pragma unroll
    for (int k = 0; k < kSpBlock / 2; ++k) {
      const int r = 2 * k + (lane >> 4);
      const int64_t jr = __shfl_sync(0xffffffffu, j, r);
      const uint32_t nbytes = jr >= 0 ? 16u : 0u;
      const int64_t off = (jr >= 0 ? jr : 0) * kRowBytes + piece * 16;
      cp_async16_zfill(sK + sp_piece(r, piece), Ku + off, nbytes);
      cp_async16_zfill(sV + sp_piece(r, piece), Vu + off, nbytes);
    }
    cp_async_wait_all();
    __syncwarp();

    // S = Q . K^T for rows 0-7 (s0) and 8-15 (s1)
    float s0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    {
      const int mat = lane >> 3, mr = lane & 7;
      const int row = (mat >> 1) * 8 + mr;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t bk[4];
        ldmatrix_x4(bk, sK_u + sp_piece(row, 2 * ks + (mat & 1)));
        mma_16816_bf16(s0, qa0[ks], 0u, qa2[ks], 0u, bk[0], bk[1]);
        mma_16816_bf16(s1, qa0[ks], 0u, qa2[ks], 0u, bk[2], bk[3]);
      }
    }
    // online softmax for head g over rows 2t, 2t+1 (s0) and 8+2t, 9+2t (s1)
    float z[4];
    z[0] = (present >> (2 * t)) & 1u ? tau2 * s0[0] : -INFINITY;
    z[1] = (present >> (2 * t + 1)) & 1u ? tau2 * s0[1] : -INFINITY;
    z[2] = (present >> (8 + 2 * t)) & 1u ? tau2 * s1[0] : -INFINITY;
    z[3] = (present >> (9 + 2 * t)) & 1u ? tau2 * s1[1] : -INFINITY;
    float mx = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m, mx);
    float sc = 1.0f, pz[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (mn != -INFINITY) {
      sc = exp2f(m - mn);  // 0 while nothing had been seen
#pragma unroll
      for (int k = 0; k < 4; ++k) pz[k] = exp2f(z[k] - mn);
    }
    float ps = (pz[0] + pz[1]) + (pz[2] + pz[3]);
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    m = mn;
    l = fmaf(l, sc, ps);
    // rescale O^T: this lane holds heads 2t and 2t + 1, whose factors live in lanes 8t, 8t + 4
    const float sc_a = __shfl_sync(0xffffffffu, sc, 8 * t);
    const float sc_b = __shfl_sync(0xffffffffu, sc, 8 * t + 4);
    // P enters the product as two bf16 parts (hi + lo, about 16 bits), so the weights the
    // values are summed with are the ones l sums
    const uint32_t ph0 = pack_bf16x2(pz[0], pz[1]), ph1 = pack_bf16x2(pz[2], pz[3]);
    const uint32_t pl0 = pack_bf16x2(pz[0] - bf16lo(ph0), pz[1] - bf16hi(ph0));
    const uint32_t pl1 = pack_bf16x2(pz[2] - bf16lo(ph1), pz[3] - bf16hi(ph1));
    {
      const int mat = lane >> 3, mr = lane & 7;
      const int row = (mat >> 1) * 8 + mr;  // matrices: rows 0-7 / 8-15 x dims +0 / +8
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t av[4];
        ldmatrix_x4_trans(av, sV_u + sp_piece(row, 2 * i + (mat & 1)));
        o[i][0] *= sc_a;
        o[i][1] *= sc_b;
        o[i][2] *= sc_a;
        o[i][3] *= sc_b;
        // A = V^T tile: a0 rows(dims) g / k rows 0-7, a1 dims g+8 / rows 0-7,
        // a2 dims g / rows 8-15, a3 dims g+8 / rows 8-15
        mma_16816_bf16(o[i], av[0], av[1], av[2], av[3], ph0, ph1);
        mma_16816_bf16(o[i], av[0], av[1], av[2], av[3], pl0, pl1);
      }
    }
    __syncwarp();  // the stage is read before the next block's copies land in it
  }

  // this warp's state into shared memory (reusing the stages: wait for every warp)
  __syncthreads();
  if (t == 0 && g < G) {
    mg.m[warp][g] = m;
    mg.l[warp][g] = l;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (2 * t < G) {
      mg.acc[warp][2 * t][16 * i + g] = o[i][0];
      mg.acc[warp][2 * t][16 * i + g + 8] = o[i][2];
    }
    if (2 * t + 1 < G) {
      mg.acc[warp][2 * t + 1][16 * i + g] = o[i][1];
      mg.acc[warp][2 * t + 1][16 * i + g + 8] = o[i][3];
    }
  }
  sp_combine<G, CL, W>(mg, rank, u, p.out);
}

// 8-bit caches: E4M3 codes (128-byte rows) with one fp32 scale per token.  Per block of 16
// selected rows a warp stages the K and V code rows (16-byte pieces permuted by row % 8)
// and looks up their scales, then
//   S = (Q / 2^e) . codes^T as f16 m16n8k16 MMAs (2^e a power of two per head with
//       |q / 2^e| < 256, so the f16 query is the bf16 query exactly for every element
//       at least 2^-24 of its head's largest; each lane widens its own pairs of codes to
//       f16, exactly);
//   z = tau2 * 2^e * ks_j * S, the same online softmax as above;
//   O += (p_j * vs_j) * codes_j on the CUDA cores in fp32 (lane: dims 4 lane .. +3 of
//       every head), l sums p_j.
constexpr int kSp8Row = kHeadDim;                              // bytes per 8-bit row
constexpr int kSp8Stage = 2 * kSpBlock * kSp8Row + kSpBlock * 8 * 4;  // K, V, weights[16][8]

__device__ __forceinline__ uint32_t sp8_piece(int r, int c) {
  return static_cast<uint32_t>(r * kSp8Row + ((c ^ (r & 7)) << 4));
}

template <int G, int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(kSpThreads, 2)
    sparse_decode_e4m3_kernel(const SparseParams p) {
  pdl_wait_primary();  // the selection and the query are complete
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];  // staged rows, then the merge state
  SpMerge<G> &mg = *reinterpret_cast<SpMerge<G> *>(smem);
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int64_t u = blockIdx.x / CL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  int cnt = p.count[u];
  cnt = cnt < 0 ? 0 : (cnt > p.idx_stride ? p.idx_stride : cnt);
  const int32_t *idx = p.idx + u * p.idx_stride;
  const uint8_t *Ku = p.K + p.plane(u) * p.ncap * kSp8Row;
  const uint8_t *Vu = p.V + p.plane(u) * p.ncap * kSp8Row;
  const float *ksu = p.ks + p.plane(u) * p.ncap;
  const float *vsu = p.vs + p.plane(u) * p.ncap;
  uint8_t *sK = smem + warp * kSp8Stage;
  uint8_t *sV = sK + kSpBlock * kSp8Row;
  float *sW = reinterpret_cast<float *>(sV + kSpBlock * kSp8Row);  // [16 rows][8 heads]

  // query of head g as the f16 A operand of S: dims 16ks + 2t, +1 (qa0) and +8, +9 (qa2),
  // divided by 2^e; the head's 4 lanes together hold all 128 dims
  uint32_t qa0[8], qa2[8];
  float escale;
  {
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(p.q + (u * G + (g < G ? g : 0)) * kHeadDim);
    uint32_t w0[8], w2[8];
    float mx = 0.0f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      w0[ks] = g < G ? qrow[8 * ks + t] : 0u;
      w2[ks] = g < G ? qrow[8 * ks + 4 + t] : 0u;
      mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16lo(w0[ks])), fabsf(bf16hi(w0[ks]))),
                           fmaxf(fabsf(bf16lo(w2[ks])), fabsf(bf16hi(w2[ks])))));
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    int e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xFFu) - 127 - 7;
    e = e < -120 ? -120 : (e > 120 ? 120 : e);
    escale = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa0[ks] = pack_f16x2(bf16lo(w0[ks]) * inv, bf16hi(w0[ks]) * inv);
      qa2[ks] = pack_f16x2(bf16lo(w2[ks]) * inv, bf16hi(w2[ks]) * inv);
    }
  }
  const float zs = p.tau * kLog2e * escale;
  float m = -INFINITY, l = 0.0f;  // head g's running max (base 2) and sum
  float acc[G][4];                // dims 4 lane .. 4 lane + 3 of every head
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.0f;

  const int r0 = rank * p.rows_per_cta;
  const int r1 = min(cnt, r0 + p.rows_per_cta);
  for (int b0 = r0 + warp * kSpBlock; b0 < r1; b0 += kSpWarps * kSpBlock) {
    // lane r < 16 looks up row r and its two scales (absent past the count, or for an
    // index outside [0, n), which is flagged)
    int64_t j = -1;
    float ksr = 0.0f, vsr = 0.0f;
    if (lane < kSpBlock && b0 + lane < r1) {
      const int32_t jj = idx[b0 + lane];
      if (jj < 0 || static_cast<int64_t>(jj) >= p.n) {
        atomicOr(p.flags, kFlagIndexRange);
      } else {
        j = jj;
        ksr = ksu[j];
        vsr = vsu[j];
      }
    }
    const uint32_t present = __ballot_sync(0xffffffffu, j >= 0);  // bit r: row r
    // each copy instruction moves four whole rows: lanes 8k .. 8k + 7 the 8 pieces of one
    const int piece = lane & 7;
#pragma unroll
    for (int k = 0; k < kSpBlock / 4; ++k) {
      const int r = 4 * k + (lane >> 3);
      const int64_t jr = __shfl_sync(0xffffffffu, j, r);
      const uint32_t nbytes = jr >= 0 ? 16u : 0u;
      const int64_t off = (jr >= 0 ? jr : 0) * kSp8Row + piece * 16;
      cp_async16_zfill(sK + sp8_piece(r, piece), Ku + off, nbytes);
      cp_async16_zfill(sV + sp8_piece(r, piece), Vu + off, nbytes);
    }
    cp_async_wait_all();
    __syncwarp();

    // S for rows 0-7 (s0) and 8-15 (s1): B operand = codes of row g (8 + g), dims
    // 16ks + 2t, +1 and 16ks + 2t + 8, +9
    float s0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint8_t *ra = sK + sp8_piece(g, ks) + 2 * t;
      const uint8_t *rb = sK + sp8_piece(8 + g, ks) + 2 * t;
      const uint32_t a0 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t *>(ra));
      const uint32_t a1 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t *>(ra + 8));
      const uint32_t b0 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t *>(rb));
      const uint32_t b1 = e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t *>(rb + 8));
      mma_16816_f16(s0, qa0[ks], 0u, qa2[ks], 0u, a0, a1);
      mma_16816_f16(s1, qa0[ks], 0u, qa2[ks], 0u, b0, b1);
    }
    // online softmax for head g over rows 2t, 2t+1 (s0) and 8+2t, 9+2t (s1)
    const int rr[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
    const float sv[4] = {s0[0], s0[1], s1[0], s1[1]};
    float z[4], vrow[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float kr = __shfl_sync(0xffffffffu, ksr, rr[k]);
      vrow[k] = __shfl_sync(0xffffffffu, vsr, rr[k]);
      z[k] = (present >> rr[k]) & 1u ? zs * kr * sv[k] : -INFINITY;
    }
    float mx = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m, mx);
    float sc = 1.0f, pz[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (mn != -INFINITY) {
      sc = exp2f(m - mn);  // 0 while nothing had been seen
#pragma unroll
      for (int k = 0; k < 4; ++k) pz[k] = exp2f(z[k] - mn);
    }
    float ps = (pz[0] + pz[1]) + (pz[2] + pz[3]);
    ps += __shfl_xor_sync(0xffffffffu, ps, 1);
    ps += __shfl_xor_sync(0xffffffffu, ps, 2);
    m = mn;
    l = fmaf(l, sc, ps);
    // the rows' weights times their V scales, for every lane
    if (g < G) {
#pragma unroll
      for (int k = 0; k < 4; ++k) sW[rr[k] * 8 + g] = pz[k] * vrow[k];
    }
    float sch[G];
#pragma unroll
    for (int h = 0; h < G; ++h) sch[h] = __shfl_sync(0xffffffffu, sc, 4 * h);
    __syncwarp();
#pragma unroll
    for (int h = 0; h < G; ++h) {
      acc[h][0] *= sch[h];
      acc[h][1] *= sch[h];
      acc[h][2] *= sch[h];
      acc[h][3] *= sch[h];
    }
    const int last = 32 - __clz(present);  // rows past the last present one weigh 0
    for (int r = 0; r < last; ++r) {
      float v0, v1, v2, v3;
      e4m3x4_to_f32(*reinterpret_cast<const uint32_t *>(sV + sp8_piece(r, lane >> 2) + (lane & 3) * 4),
                    v0, v1, v2, v3);
      const float4 wa = *reinterpret_cast<const float4 *>(sW + r * 8);
      float wr[8] = {wa.x, wa.y, wa.z, wa.w, 0.0f, 0.0f, 0.0f, 0.0f};
      if constexpr (G == 8) {
        const float4 wb = *reinterpret_cast<const float4 *>(sW + r * 8 + 4);
        wr[4] = wb.x;
        wr[5] = wb.y;
        wr[6] = wb.z;
        wr[7] = wb.w;
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        acc[h][0] = fmaf(wr[h], v0, acc[h][0]);
        acc[h][1] = fmaf(wr[h], v1, acc[h][1]);
        acc[h][2] = fmaf(wr[h], v2, acc[h][2]);
        acc[h][3] = fmaf(wr[h], v3, acc[h][3]);
      }
    }
    __syncwarp();  // the stage is read before the next block's copies land in it
  }

  // this warp's state into shared memory (reusing the stages: wait for every warp)
  __syncthreads();
  if (t == 0 && g < G) {
    mg.m[warp][g] = m;
    mg.l[warp][g] = l;
  }
#pragma unroll
  for (int h = 0; h < G; ++h)
    *reinterpret_cast<float4 *>(&mg.acc[warp][h][4 * lane]) =
        make_float4(acc[h][0], acc[h][1], acc[h][2], acc[h][3]);
  sp_combine<G, CL>(mg, rank, u, p.out);
}

// ----------------------------------------------------------------------------- window

struct WindowParams {
  const uint16_t *q;
  const uint8_t *K, *V;
  float *out;
  int64_t pos;
  int window;
  float tau;
  float cs[kHeadDim / 2], sn[kHeadDim / 2];  // cos, sin of the rotation of pair i at pos
};

template <int G>
__global__ void __launch_bounds__(kThreads, G == 4 ? 2 : 1) window_decode_kernel(const WindowParams p) {
  pdl_wait_primary();  // the query and the ring are complete
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];  // staged rows, then the merge state
  Merge<G> &mg = *reinterpret_cast<Merge<G> *>(smem);
  const int64_t u = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane >> 4, sl = lane & 15;
  DotsF32<G> dots;
  // this lane's dims 8sl..8sl+7 are rotary pairs 4sl..4sl+3; the launch supplies each
  // pair's cos and sin at pos
  {
    const uint16_t *qrow = p.q + u * G * kHeadDim + sl * 8;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = 4 * sl + k;
      const float c = p.cs[i], s = p.sn[i];
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
  // the valid positions, split into contiguous runs per warp
  const int per_warp = (nv + kWarps - 1) / kWarps;
  const int w0 = warp * per_warp;
  const int w1 = min(nv, w0 + per_warp);
  const WarpStage ws(smem, warp);
  for (int b0 = w0; b0 < w1; b0 += kWarpRows) {
    const int nrows = min(kWarpRows, w1 - b0);
    const uint32_t present = stage_rows(
        ws, Ku, Vu, nrows,
        [&](int i) -> int64_t { return (first + b0 + i) % p.window; }, lane);
    for (int c = 0; c < nrows; c += kChunk) {
      const int f = c + grp * 4;
      const uint32_t pm = f < 32 ? (present >> f) & 0xFu : 0u;
      Chunk ch;
      load_chunk(ch, ws.k + f * kRowBytes, ws.v + f * kRowBytes, pm, sl);
      fold_chunk<G>(st, dots, tau2, ch, sl);
    }
    __syncwarp();
  }
  __syncthreads();  // every warp is done with its rows before the merge state reuses them
  merge_warps<G>(mg, st, warp, lane);
  for (int i = threadIdx.x; i < G * kHeadDim; i += kThreads) {
    const int h = i / kHeadDim;
    p.out[u * G * kHeadDim + i] = mg.cl[h] > 0.0f ? mg.ca[h][i % kHeadDim] / mg.cl[h] : 0.0f;
  }
}

// Both kernels stage rows in dynamic shared memory that the merge state reuses.
template <class Params>
cudaError_t launch_staged(void (*kernel)(Params), dim3 grid, const Params &p, cudaStream_t stream) {
  static_assert(sizeof(Merge<8>) <= kStageBytes, "the merge state fits the staging space");
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, grid, dim3(kThreads), kStageBytes, stream, 0u, p);
}

template <bool KV8, int W = kSpWarps>
cudaError_t launch_sparse_t(void (*kernel)(SparseParams), dim3 grid, const SparseParams &p,
                            cudaStream_t stream) {
  constexpr int stage = W * (KV8 ? kSp8Stage : kSpStage);
  constexpr int merge = static_cast<int>(sizeof(SpMerge<8, W>));
  constexpr int bytes = stage > merge ? stage : merge;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kernel, grid, dim3(W * 32), bytes, stream, 0u, p);
}

template <int G>
cudaError_t launch_sparse_g(dim3 grid, const SparseParams &p, cudaStream_t stream) {
  if (p.wide) {
    // the wide variant (bf16 caches, clusters of up to 4)
    if (p.ks != nullptr) return cudaErrorInvalidValue;
    if (p.cl == 4)
      return launch_sparse_t<false, kSpWideWarps>(sparse_decode_kernel<G, 4, kSpWideWarps>, grid, p, stream);
    if (p.cl == 2)
      return launch_sparse_t<false, kSpWideWarps>(sparse_decode_kernel<G, 2, kSpWideWarps>, grid, p, stream);
    return cudaErrorInvalidValue;
  }
  if constexpr (G == 1) {
    switch (p.cl) {
      case 8: return launch_sparse_t<false>(sparse_decode_kernel<1, 8>, grid, p, stream);
      case 4: return launch_sparse_t<false>(sparse_decode_kernel<1, 4>, grid, p, stream);
      case 2: return launch_sparse_t<false>(sparse_decode_kernel<1, 2>, grid, p, stream);
      default: return launch_sparse_t<false>(sparse_decode_kernel<1, 1>, grid, p, stream);
    }
  }
  if (p.ks != nullptr) {
    switch (p.cl) {
      case 8: return launch_sparse_t<true>(sparse_decode_e4m3_kernel<G, 8>, grid, p, stream);
      case 4: return launch_sparse_t<true>(sparse_decode_e4m3_kernel<G, 4>, grid, p, stream);
      case 2: return launch_sparse_t<true>(sparse_decode_e4m3_kernel<G, 2>, grid, p, stream);
      default: return launch_sparse_t<true>(sparse_decode_e4m3_kernel<G, 1>, grid, p, stream);
    }
  }
  switch (p.cl) {
    case 8: return launch_sparse_t<false>(sparse_decode_kernel<G, 8>, grid, p, stream);
    case 4: return launch_sparse_t<false>(sparse_decode_kernel<G, 4>, grid, p, stream);
    case 2: return launch_sparse_t<false>(sparse_decode_kernel<G, 2>, grid, p, stream);
    default: return launch_sparse_t<false>(sparse_decode_kernel<G, 1>, grid, p, stream);
  }
}

}  // namespace

size_t sparse_workspace_bytes(int64_t units, int G, int idx_stride) {
  (void)units;
  (void)G;
  (void)idx_stride;
  return 0;
}

cudaError_t launch_sparse_decode(int G, bool per_head, int Hq, const void *q, const void *k_cache,
                                 const void *v_cache,
                                 const float *k_scales, const float *v_scales, const int32_t *idx, int idx_stride, const int32_t *count,
                                 int64_t units, int Hkv, int64_t n, int64_t ncap, float tau,
                                 float *out, void *workspace, uint32_t *flags, int sm_count,
                                 cudaStream_t stream) {
  (void)Hkv;
  (void)workspace;
  if (units == 0) return cudaSuccess;
  SparseParams p;
  p.q = static_cast<const uint16_t *>(q);
  p.K = static_cast<const uint8_t *>(k_cache);
  p.V = static_cast<const uint8_t *>(v_cache);
  p.ks = k_scales;
  p.vs = v_scales;
  p.idx = idx;
  p.count = count;
  p.out = out;
  p.flags = flags;
  p.n = n;
  p.ncap = ncap;
  p.idx_stride = idx_stride;
  // 8 CTAs per unit, one to an SM if they fit; else wide CTAs (18 warps), 4 or 2 per unit,
  // if they fit one to an SM (bf16 caches); else 8 CTAs, two to an SM, or fewer CTAs so that
  // the launch stays one wave.  (One wide CTA per unit measured no faster than two narrow
  // ones sharing an SM.)
  int cl = kMaxCluster;
  p.wide = 0;
  if (units * kMaxCluster > static_cast<int64_t>(sm_count) && k_scales == nullptr) {
    int w = 4;
    while (w > 2 && units * w > static_cast<int64_t>(sm_count)) w >>= 1;
    if (units * w <= static_cast<int64_t>(sm_count)) {
      cl = w;
      p.wide = 1;
    }
  }
  if (!p.wide)
    while (cl > 1 && units * cl > 2 * static_cast<int64_t>(sm_count)) cl >>= 1;
  p.cl = cl;
  p.rows_per_cta = ((idx_stride + cl - 1) / cl + kSpBlock - 1) / kSpBlock * kSpBlock;
  p.tau = tau;
  p.per_head = per_head ? 1 : 0;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Gq = Hq / Hkv;
  const dim3 grid(static_cast<unsigned>(units * cl));
  if (per_head) {
    // one query head per unit (its own rows); 8-bit caches are not built for this variant
    if (k_scales != nullptr) return cudaErrorInvalidValue;
    return launch_sparse_g<1>(grid, p, stream);
  }
  if (G == 4) return launch_sparse_g<4>(grid, p, stream);
  if (G == 8) return launch_sparse_g<8>(grid, p, stream);
  return cudaErrorInvalidValue;
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
  p.tau = tau;
  // pair i turns by pos * base^(-2i/D): the angle in double, reduced to [-pi, pi] before
  // its cosine and sine, so large positions keep their phase
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < kHeadDim / 2; ++i) {
    const double ang = static_cast<double>(pos) * std::pow(static_cast<double>(rope_base), -2.0 * i / kHeadDim);
    const double red = ang - two_pi * std::nearbyint(ang / two_pi);
    p.cs[i] = static_cast<float>(std::cos(red));
    p.sn[i] = static_cast<float>(std::sin(red));
  }
  const dim3 grid(static_cast<unsigned>(units));
  if (G == 4) return launch_staged(window_decode_kernel<4>, grid, p, stream);
  if (G == 8) return launch_staged(window_decode_kernel<8>, grid, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace embla
