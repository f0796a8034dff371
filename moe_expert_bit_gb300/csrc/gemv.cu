// Weight-streaming kernels for the two projections when expert tiles are
// small (decode): the GEMV-style variant.  The layer is then a pure stream of
// packed 4-bit weights from HBM, so what counts is the work per weight on
// the CUDA cores, not matrix throughput.
//
//   gate/up:  h[s, n] = gelu_tanh(sum_k Wg[e][n][k] x_s[k]) * sum_k Wu[e][n][k] x_s[k]
//   down:     y_acc[t, n] += w_a * sum_i Wd[e][n][i] h[s, i],  a = perm[s], t = a / top_k
// with w = scale * q + bias per 64-group (Layr-Labs/mlx PR #4, "What";
// SharpAI/SwiftLM issue #236, "Still missing" and "Already on main").
//
// Per 64-wide group g of one weight row the dot product splits as
//   sum_k w_k x_k = s_g * D_g + (b_g - 128 s_g) * X_g,
//   D_g = sum_k (128 + q_k) x_k,   X_g = sum_k x_k,
// and 128 + q is exact in bf16: OR-ing a nibble into the bf16 pattern of
// 128.0 produces it, and one lop3 on a shifted packed word produces two of
// them at once (nibbles j and j+4).  D_g is one warp-level bf16 MMA
// (m16n8k16, fp32 accumulate) per 16 k: the MMA is used as the dot-product
// engine so that the CUDA cores only unpack nibbles (under one instruction
// per weight) and fold each group once.  The k order inside an MMA is a
// permutation of the group's k; the activations are staged in shared memory
// in the same permuted order, which leaves the sum unchanged.
//
// A warp owns 16 weight rows (the MMA's M) and up to 4 activation rows per
// pass (half of the MMA's N).  Its rows are loaded whole into shared memory
// with bulk copies, so that DRAM sees long sequential runs, and stay there
// while the passes over the tile's activation rows run.  For gate/up the 16 rows are 8 gate rows and the 8 matching up rows, so
// each lane ends with a gate value and its up value side by side.
#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace moeqmm {

constexpr int kTok = 4;  // activation rows staged per pass (MMA columns 4-7 repeat row 3)

__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t mask, uint32_t bits) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));
  return d;
}

// bf16x2 {128 + q_p (low half), 128 + q_{p+4} (high half)} of one packed word
__device__ __forceinline__ uint32_t pair128(uint32_t word, int p) {
  return lop_and_or(word >> (4 * p), 0x000F000Fu, 0x43004300u);
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1, const float (&c)[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ float bf16f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// In place: each 16-byte block c (activations 8c'..8c'+7 of group g, c' = c % 8) becomes the
// MMA B fragments of lane slot t = c'/2 for m = 2(c'%2) + {0,1}: {x0,x4 | x1,x5} and
// {x2,x6 | x3,x7}; the block's sum goes into the group sum.  Rows >= R are zeroed.
// Run by `nthreads` threads (a multiple of 32, starting at thread 0).
__device__ __forceinline__ void permute_rows(uint8_t *xb, float *xs, int xrb, int G, int R,
                                             int nthreads) {
  for (int i = threadIdx.x; i < kTok * G * 8; i += nthreads) {
    const int j = i / (G * 8), rem = i - j * G * 8, g = rem >> 3;
    uint4 *blk = reinterpret_cast<uint4 *>(xb + (size_t)j * xrb + rem * 16);
    uint4 q = make_uint4(0u, 0u, 0u, 0u);
    if (j < R) q = *blk;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    auto el = [&](int e) -> uint32_t { return (e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu); };
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) part += __uint_as_float(el(e) << 16);
    uint4 o;
    o.x = el(0) | (el(4) << 16);
    o.y = el(1) | (el(5) << 16);
    o.z = el(2) | (el(6) << 16);
    o.w = el(3) | (el(7) << 16);
    *blk = o;
    // the 8 blocks of one (row, group) are 8 consecutive lanes
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    part += __shfl_xor_sync(0xffffffffu, part, 4);
    if ((rem & 7) == 0) xs[j * G + g] = part;
  }
}

// Dot products of a warp's 16 weight rows with the staged activation rows.
//   wrows: the warp's 16 packed weight rows in shared memory (rows 0-7: MMA rows g,
//          rows 8-15: MMA rows g + 8), row stride ws
//   scA / scB: scale rows of MMA rows g and g+8 in shared memory (biases at +bofs)
// acc[0], acc[1]: row g with activation rows 2t, 2t+1; acc[2], acc[3]: row g+8.
// Two groups per iteration, each as two independent MMA chains, keep four chains in flight.
__device__ __forceinline__ void group_mma(const uint8_t *rA, const uint8_t *rB, const uint8_t *xrow,
                                          int g, float (&d0)[4], float (&d1)[4]) {
  const uint2 A = *reinterpret_cast<const uint2 *>(rA + g * 32);
  const uint2 B = *reinterpret_cast<const uint2 *>(rB + g * 32);
  // the four B fragments of the group: two 16-byte loads
  const uint4 f01 = *reinterpret_cast<const uint4 *>(xrow + g * 128);
  const uint4 f23 = *reinterpret_cast<const uint4 *>(xrow + g * 128 + 16);
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t wA = (m >> 1) ? A.y : A.x;
    const uint32_t wB = (m >> 1) ? B.y : B.x;
    const int p0 = 2 * (m & 1);
    const uint32_t a[4] = {pair128(wA, p0), pair128(wB, p0), pair128(wA, p0 + 1),
                           pair128(wB, p0 + 1)};
    const uint32_t b0 = m == 0 ? f01.x : m == 1 ? f01.z : m == 2 ? f23.x : f23.z;
    const uint32_t b1 = m == 0 ? f01.y : m == 1 ? f01.w : m == 2 ? f23.y : f23.w;
    if (m < 2)
      mma_bf16_16816(d0, a, b0, b1, d0);
    else
      mma_bf16_16816(d1, a, b0, b1, d1);
  }
}

__device__ __forceinline__ void group_fold(const uint16_t *scA, const uint16_t *scB, int bofs,
                                           const float *xs0, const float *xs1, int g,
                                           const float (&d0)[4], const float (&d1)[4],
                                           float (&acc)[4]) {
  const float s_a = bf16f(scA[g]), s_b = bf16f(scB[g]);
  const float c_a = fmaf(-128.f, s_a, bf16f(scA[bofs + g]));
  const float c_b = fmaf(-128.f, s_b, bf16f(scB[bofs + g]));
  const float x0 = xs0[g], x1 = xs1[g];
  acc[0] = fmaf(s_a, d0[0] + d1[0], fmaf(c_a, x0, acc[0]));
  acc[1] = fmaf(s_a, d0[1] + d1[1], fmaf(c_a, x1, acc[1]));
  acc[2] = fmaf(s_b, d0[2] + d1[2], fmaf(c_b, x0, acc[2]));
  acc[3] = fmaf(s_b, d0[3] + d1[3], fmaf(c_b, x1, acc[3]));
}

__device__ __forceinline__ void warp_rows_dot(const uint8_t *wrows, int ws, const uint16_t *scA,
                                              const uint16_t *scB, int bofs, const uint8_t *xb,
                                              int xrb, const float *xs, int G, int g_begin,
                                              int g_end, float (&acc)[4]) {
  const int lane = threadIdx.x & 31, gq = lane >> 2, t = lane & 3;
  // B column gq = activation row gq; columns past the staged rows repeat the last one
  const uint8_t *xrow = xb + (size_t)min(gq, kTok - 1) * xrb + t * 32;
  const float *xs0 = xs + min(2 * t, kTok - 1) * G, *xs1 = xs + min(2 * t + 1, kTok - 1) * G;
  const uint8_t *rA = wrows + gq * ws + t * 8, *rB = rA + 8 * ws;
  int g = g_begin;
#pragma unroll 1
  for (; g + 1 < g_end; g += 2) {
    float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
    float q0[4] = {0.f, 0.f, 0.f, 0.f}, q1[4] = {0.f, 0.f, 0.f, 0.f};
    group_mma(rA, rB, xrow, g, p0, p1);
    group_mma(rA, rB, xrow, g + 1, q0, q1);
    group_fold(scA, scB, bofs, xs0, xs1, g, p0, p1, acc);
    group_fold(scA, scB, bofs, xs0, xs1, g + 1, q0, q1, acc);
  }
  if (g < g_end) {
    float p0[4] = {0.f, 0.f, 0.f, 0.f}, p1[4] = {0.f, 0.f, 0.f, 0.f};
    group_mma(rA, rB, xrow, g, p0, p1);
    group_fold(scA, scB, bofs, xs0, xs1, g, p0, p1, acc);
  }
}

// The persistent kernel: one CTA per SM walks a contiguous range of work
// chunks (a chunk = 16 weight rows of one expert tile: 8 gate rows + their 8 up
// rows, or 16 down rows).  A producer warp streams each chunk's packed rows and
// scale/bias rows into a ring of shared-memory buffers with 1-D bulk copies
// (every row is contiguous in global memory); up to 16 compute warps take
// chunks in turn.  When the range moves to the next tile, the compute warps stage that
// tile's activation rows (kTok per pass) in MMA fragment order.
// Compute warps per CTA: 16, in 8 pairs (fewer if the ring holds fewer than 8 chunks).
// The two warps of a pair split a chunk's K range and combine their partial sums in the
// chunk's buffer.  Pair p takes chunks p, p + P, ... and chunk i uses buffer i % nbuf; with
// P <= nbuf the previous use of a buffer always belongs to a chunk that landed before the
// pair's previous chunk, so a parity wait on the buffer's barrier never runs a phase ahead.
constexpr int kMaxComputeWarps = 16;

__device__ __forceinline__ void named_sync_pair(int pair) {
  asm volatile("bar.sync %0, 64;" ::"r"(2 + pair) : "memory");
}

// Chunks per segment: the scale and bias rows of a segment's chunks are staged with a
// few large bulk copies at the segment start (a TMA operation costs about the same
// whatever its size, so many small per-chunk scale copies would dominate).
constexpr int kSegChunks = 8;

struct PLayout {
  int G, ws, xrb, chunk_bytes, nbuf, off_x, off_xs, off_sc, sc_part, off_bar, total;
  __host__ __device__ PLayout(int K, int nbuf_) {
    G = K / 64;
    ws = K / 2;                      // packed weight rows, contiguous as in global memory
    xrb = G * 128 + 16;              // activation row stride (fragment order)
    chunk_bytes = (16 * ws + 127) & ~127;
    nbuf = nbuf_;
    off_x = nbuf * chunk_bytes;
    off_xs = off_x + kTok * xrb;
    off_sc = (off_xs + kTok * G * 4 + 15) & ~15;
    sc_part = kSegChunks * 8 * G;    // u16 elements of one quarter of the scale region
    off_bar = off_sc + 4 * sc_part * 2;
    total = off_bar + (2 * nbuf + 2) * 8;
  }
};

__host__ __device__ inline int persist_nbuf(int K) {
  // as many chunk buffers as fit next to the activation and scale regions, at most 16
  for (int nb = 16; nb > 2; --nb)
    if (PLayout(K, nb).total <= 227 * 1024) return nb;
  return 2;
}

__device__ __forceinline__ void named_sync_compute(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// The CTA counts itself done on the int just past y_acc; the last one converts y_acc to
// bf16 y.  The threadfence before the count orders this CTA's reductions before it, and
// the last CTA reads y_acc from L2 (where the reductions were performed).
__device__ __forceinline__ void last_cta_cast(const float *y_acc, uint16_t *y, int64_t n,
                                              int nthreads, bool named) {
  __shared__ int s_last;
  if (threadIdx.x == 0) {
    __threadfence();
    int *done = const_cast<int *>(reinterpret_cast<const int *>(y_acc + n));
    s_last = (atomicAdd(done, 1) == (int)gridDim.x - 1);
    __threadfence();
  }
  if (named)
    named_sync_compute(nthreads);
  else
    __syncthreads();
  if (!s_last) return;
  for (int64_t i = threadIdx.x; i < n / 4; i += nthreads) {
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(y_acc) + i);
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t *>(&lo);
    o.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(y)[i] = o;
  }
}

template <int MODE>  // 0: gate/up + GeGLU -> h; 1: down + weighted scatter -> y_acc
__global__ void __launch_bounds__((kMaxComputeWarps + 1) * 32, 1)
    gemv_persist_kernel(const uint16_t *__restrict__ act, const uint32_t *__restrict__ Wq,
                        const uint16_t *__restrict__ Sc, const uint16_t *__restrict__ Bi,
                        const int32_t *__restrict__ tiles, const int32_t *__restrict__ tile_count,
                        const int32_t *__restrict__ perm, const float *__restrict__ topk_weights,
                        int32_t *__restrict__ status, int32_t top_k, int32_t H, int32_t I,
                        int32_t nbuf, uint16_t *__restrict__ h, float *__restrict__ y_acc,
                        uint16_t *__restrict__ y_out, int64_t n_cast) {
  using namespace umma;
  extern __shared__ __align__(128) uint8_t gsm[];
  if (load_status(status) != 0) return;
  const int K = MODE == 0 ? H : I;
  const PLayout L(K, nbuf);
  const int G = L.G;
  const int CPT = MODE == 0 ? I / 8 : H / 16;  // chunks per tile
  const int rows_per_expert = MODE == 0 ? 2 * I : H;
  const int n_tiles = *tile_count;
  const int total = n_tiles * CPT;
  const int c0 = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int c1 = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  // DOWN with n_cast > 0: the last CTA to finish converts the n_cast elements of y_acc
  // to bf16 y (its arrival counter is the int just past y_acc, zeroed with it).
  if (c0 >= c1) {
    if (MODE == 1 && n_cast > 0) {
      __syncthreads();
      last_cta_cast(y_acc, y_out, n_cast, blockDim.x, false);
    }
    return;
  }
  uint8_t *xb = gsm + L.off_x;
  float *xs = reinterpret_cast<float *>(gsm + L.off_xs);
  uint64_t *full = reinterpret_cast<uint64_t *>(gsm + L.off_bar);
  uint64_t *empty = full + nbuf;
  uint64_t *xbar = empty + nbuf;  // activations + segment scales
  uint16_t *scs = reinterpret_cast<uint16_t *>(gsm + L.off_sc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwc = (int)(blockDim.x >> 5) - 1;  // compute warps; the last warp produces
  if (threadIdx.x == 0) {
    for (int i = 0; i < nbuf; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(xbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  volatile int never = 0;

  // Work order (shared by producer and consumers): tiles of the range in order; per tile
  // ceil(R / kTok) passes; per pass the range's chunks of that tile.
  if (warp == nwc) {
    // ------------------------------------------------ producer
    // A chunk is its 16 packed weight rows: two bulk copies of 8 consecutive rows (gate
    // rows and their up rows) or one of 16 down rows, issued by lanes 0 and 1.
    uint32_t it = 0;
    bool ok = true;
    for (int tile = c0 / CPT; ok && tile * CPT < c1; ++tile) {
      const int e = tiles[3 * tile], R = tiles[3 * tile + 2];
      const int j0 = max(c0 - tile * CPT, 0), j1 = min(c1 - tile * CPT, CPT);
      for (int r0 = 0; ok && r0 < R; r0 += kTok) {
        for (int j = j0; j < j1; ++j, ++it) {
          const int b = it % nbuf;
          ok = mbar_wait(&empty[b], ((it / nbuf) & 1) ^ 1, &never);
          if (!(ok = __all_sync(0xffffffffu, ok))) break;
          uint8_t *buf = gsm + (size_t)b * L.chunk_bytes;
          const uint32_t rbytes = (uint32_t)K / 2;
          if (lane == 0) mbar_arrive_expect_tx(&full[b], 16 * rbytes);
          __syncwarp();
          const int64_t ra = (int64_t)e * rows_per_expert + (MODE == 0 ? 8 * j : 16 * j);
          if (MODE == 0) {
            if (lane < 2)
              bulk_load(buf + lane * 8 * L.ws, Wq + (ra + lane * I) * (K / 8), 8 * rbytes,
                        &full[b]);
          } else if (lane == 0) {
            bulk_load(buf, Wq + ra * (K / 8), 16 * rbytes, &full[b]);
          }
        }
      }
    }
    if (!ok && lane == 0) raise_status(status, MOE_ERR_TIMEOUT);
    // drain: copies still in flight complete before the CTA exits
    __syncwarp();
    if (lane == 0)
      for (uint32_t i = (it > (uint32_t)nbuf ? it - nbuf : 0); i < it; ++i)
        mbar_wait(&full[i % nbuf], (i / nbuf) & 1, nullptr, 200000000ull);
    return;
  }

  // ------------------------------------------------ compute warps
  const int gq = lane >> 2, t = lane & 3;
  const int npairs = nwc / 2, pair = warp >> 1, half = warp & 1;
  uint32_t it = 0, xphase = 0;
  bool ok = true;
  for (int tile = c0 / CPT; tile * CPT < c1; ++tile) {
    const int e = tiles[3 * tile], row0 = tiles[3 * tile + 1], R = tiles[3 * tile + 2];
    const int j0 = max(c0 - tile * CPT, 0), j1 = min(c1 - tile * CPT, CPT);
    for (int r0 = 0; r0 < R; r0 += kTok) {
      const int Rp = min(kTok, R - r0);
      for (int s0 = j0; s0 < j1; s0 += kSegChunks, xphase ^= 1) {
        const int s1 = min(s0 + kSegChunks, j1), nseg = s1 - s0;
        named_sync_compute(nwc * 32);  // every warp is done with the previous staging
        if (warp == 0) {
          // activations of this pass (one row per lane) and the segment's scale rows
          const uint32_t xbytes = (uint32_t)K * 2;
          const uint32_t rows_q = MODE == 0 ? 8u * nseg : 16u * nseg;  // rows per part
          const uint32_t sbytes = rows_q * G * 2;
          const int nparts = MODE == 0 ? 4 : 2;
          if (lane == 0) mbar_arrive_expect_tx(xbar, Rp * xbytes + nparts * sbytes);
          __syncwarp();
          if (lane < Rp) {
            const int64_t src_row =
                MODE == 0 ? perm[row0 + r0 + lane] / top_k : row0 + r0 + lane;
            bulk_load(xb + (size_t)lane * L.xrb, act + src_row * K, xbytes, xbar);
          } else if (lane >= 8 && lane < 8 + nparts) {
            const int q = lane - 8;  // GEGLU: gate s, up s, gate b, up b; DOWN: s, b
            const int64_t r_first = MODE == 0
                                        ? (int64_t)e * rows_per_expert + 8 * s0 + ((q & 1) ? I : 0)
                                        : (int64_t)e * rows_per_expert + 16 * s0;
            const uint16_t *src = (MODE == 0 ? (q < 2 ? Sc : Bi) : (q == 0 ? Sc : Bi)) + r_first * G;
            bulk_load(scs + (size_t)q * (MODE == 0 ? L.sc_part : 2 * L.sc_part), src, sbytes,
                      xbar);
          }
        }
        ok = mbar_wait(xbar, xphase, &never) && ok;
        permute_rows(xb, xs, L.xrb, G, Rp, nwc * 32);
        named_sync_compute(nwc * 32);
        for (int j = s0; j < s1; ++j, ++it) {
          if ((int)(it % npairs) != pair) continue;
          const int b = it % nbuf;
          ok = mbar_wait(&full[b], (it / nbuf) & 1, &never) && ok;
          ok = __all_sync(0xffffffffu, ok);
          uint8_t *buf = gsm + (size_t)b * L.chunk_bytes;
          const int jl = j - s0;
          const uint16_t *scA, *scB;
          int bofs;
          if (MODE == 0) {  // gate row jl*8 + gq in part 0, its up row in part 1
            scA = scs + (size_t)(jl * 8 + gq) * G;
            scB = scs + L.sc_part + (size_t)(jl * 8 + gq) * G;
            bofs = 2 * L.sc_part;
          } else {          // rows jl*16 + gq and + 8 in part 0 (scales), part 2 (biases)
            scA = scs + (size_t)(jl * 16 + gq) * G;
            scB = scs + (size_t)(jl * 16 + 8 + gq) * G;
            bofs = 2 * L.sc_part;
          }
          float acc[4] = {0.f, 0.f, 0.f, 0.f};
          const int gsplit = (G + 1) / 2;
          if (ok)
            warp_rows_dot(buf, L.ws, scA, scB, bofs, xb, L.xrb, xs, G, half ? gsplit : 0,
                          half ? G : gsplit, acc);
          // combine the two halves of K: the second warp parks its sums in the consumed buffer
          named_sync_pair(pair);
          float4 *park = reinterpret_cast<float4 *>(buf) + lane;
          if (half) *park = make_float4(acc[0], acc[1], acc[2], acc[3]);
          named_sync_pair(pair);
          if (half) continue;
          const float4 o = *park;
          acc[0] += o.x;
          acc[1] += o.y;
          acc[2] += o.z;
          acc[3] += o.w;
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[b]);
          if (!ok) continue;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int jr = 2 * t + c;
            if (jr >= Rp) continue;
            if (MODE == 0) {
              const int n = 8 * j + gq;  // acc[c]: gate, acc[2 + c]: up
              h[(int64_t)(row0 + r0 + jr) * I + n] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(gelu_tanh(acc[c]) * acc[2 + c]));
            } else {
              const int a = perm[row0 + r0 + jr];
              const float w = topk_weights[a];
              float *yrow = y_acc + (int64_t)(a / top_k) * H + 16 * j;
              atomicAdd(yrow + gq, w * acc[c]);
              atomicAdd(yrow + gq + 8, w * acc[2 + c]);
            }
          }
        }
      }
    }
  }
  if (!ok) raise_status(status, MOE_ERR_TIMEOUT);
  if (MODE == 1 && n_cast > 0) {
    named_sync_compute(nwc * 32);  // every reduction of this CTA has been issued
    last_cta_cast(y_acc, y_out, n_cast, nwc * 32, true);
  }
}

// y = bf16(y_acc), four elements per thread step
__global__ void cast_bf16_kernel(const float *__restrict__ y_acc, uint16_t *__restrict__ y,
                                 int64_t n4, const int32_t *__restrict__ status) {
  if (load_status(status) != 0) return;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = reinterpret_cast<const float4 *>(y_acc)[i];
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t *>(&lo);
    o.y = *reinterpret_cast<uint32_t *>(&hi);
    reinterpret_cast<uint2 *>(y)[i] = o;
  }
}

static moe_status set_smem(const void *fn, size_t smem) {
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

static int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

bool gemv_supported(int32_t H, int32_t I) {
  return PLayout(H, 2).total <= 227 * 1024 && PLayout(I, 2).total <= 227 * 1024;
}

template <int MODE>
static moe_status launch_persist(const uint16_t *act, const uint32_t *Wq, const uint16_t *Sc,
                                 const uint16_t *Bi, const moe_tiles_t &t, const float *tw,
                                 int32_t H, int32_t I, uint16_t *h, float *y_acc, uint16_t *y,
                                 int64_t n_cast, cudaStream_t stream, const char *what) {
  const int K = MODE == 0 ? H : I;
  const int nbuf = persist_nbuf(K);
  const size_t smem = PLayout(K, nbuf).total;
  if (set_smem((const void *)gemv_persist_kernel<MODE>, smem) != MOE_OK) return check_launch(what);
  const int64_t max_chunks = (int64_t)t.max_tiles * (MODE == 0 ? I / 8 : H / 16);
  int grid = sm_count();
  if (max_chunks < grid) grid = (int)max_chunks;
  const int nwc = 2 * nbuf < kMaxComputeWarps ? 2 * nbuf : kMaxComputeWarps;
  gemv_persist_kernel<MODE><<<grid, (nwc + 1) * 32, smem, stream>>>(
      act, Wq, Sc, Bi, t.tiles, t.tile_count, t.perm, tw, t.status, t.top_k, H, I, nbuf, h,
      y_acc, y, n_cast);
  return check_launch(what);
}

moe_status launch_geglu_gemv(const uint16_t *x, const uint32_t *Wgu, const uint16_t *Sgu,
                             const uint16_t *Bgu, const moe_tiles_t &t, int32_t H, int32_t I,
                             uint16_t *h, cudaStream_t stream) {
  return launch_persist<0>(x, Wgu, Sgu, Bgu, t, nullptr, H, I, h, nullptr, nullptr, 0, stream,
                           "moe_gather_qmm_geglu (gemv)");
}

moe_status launch_down_gemv(const uint16_t *hin, const uint32_t *Wd, const uint16_t *Sd,
                            const uint16_t *Bd, const moe_tiles_t &t, const float *topk_weights,
                            int32_t H, int32_t I, float *y_acc, uint16_t *y, int64_t n_cast,
                            cudaStream_t stream) {
  return launch_persist<1>(hin, Wd, Sd, Bd, t, topk_weights, H, I, nullptr, y_acc, y, n_cast,
                           stream, "moe_gather_qmm_down_unsort (gemv)");
}

moe_status launch_cast_bf16(const float *y_acc, uint16_t *y, int64_t n, const int32_t *status,
                            cudaStream_t stream) {
  const int64_t n4 = n / 4;  // n = T * H with H % 64 == 0
  int blocks = (int)((n4 + 255) / 256);
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  cast_bf16_kernel<<<blocks, 256, 0, stream>>>(y_acc, y, n4, status);
  return check_launch("moe_gather_qmm_down_unsort (cast)");
}

}  // namespace moeqmm
