// tcgen05 tensor-core grouped GEMM over expert tiles, with the 4-bit affine
// weights dequantised into shared memory (Layr-Labs/mlx PR #4, "What": a
// gathered quantized matmul per sorted expert tile, affine 4-bit group-64
// weights, bf16 activations).  Two modes share the kernel:
//
//   GEGLU: h[s, n] = gelu_tanh(sum_k Wg[e][n][k] x[t_s][k]) * sum_k Wu[e][n][k] x[t_s][k]
//          (SharpAI/SwiftLM issue #236, "Still missing": the GeGLU product fused
//          into one dispatch; here it is the GEMM epilogue)
//   DOWN:  y_acc[t_s, n] += w_s * sum_i Wd[e][n][i] h[s][i]
//          (weightedExpertSum / direct weighted un-sort as the GEMM epilogue)
//
// The weights are the MMA's M side ("swap AB"): one work unit is one expert
// tile (<= 128 token rows, the MMA's N) times 128 weight rows, accumulated
// over K in 64-wide k-blocks, one quantisation group per k-block.
//
// One persistent CTA per SM, 16 warps with fixed roles:
//   warp 0      W producer: TMA of the packed nibbles (4 KB per k-block) and a
//               bulk copy of the unit's bf16 scales and biases
//   warp 1      TMEM owner and MMA issuer (one thread issues tcgen05.mma)
//   warp 2      X producer: TMA of the activation rows of the tile (B operand),
//               gathered row by row through the sort permutation (GEGLU) or
//               contiguous sorted rows of h (DOWN)
//   warps 4-7   epilogue: TMEM -> registers -> GeGLU product -> h, or
//               router-weighted fp32 reductions into y_acc
//   warps 8-15  dequant: nibbles + scale/bias -> bf16 weights in the
//               128-byte-swizzled K-major layout the MMA reads
// Rings of mbarriers connect the roles; every wait is bounded (a timeout
// sets the status word to MOE_ERR_TIMEOUT and the CTA drains and exits).
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace moeqmm {
namespace tc {

using namespace umma;

constexpr int kThreads = 512;
constexpr int kDeqWarp0 = 8;
constexpr int kDeqThreads = 256;
constexpr int kEpiWarp0 = 4;
constexpr int kBM = 128;      // weight rows per unit (MMA M)
constexpr int kMaxN = 128;    // token rows per unit (MMA N upper bound)
constexpr int kNibStages = 8;
constexpr int kAStages = 3;
constexpr int kBStages = 4;
constexpr int kNibBytes = kBM * 32;   // 64 nibbles per row per k-block
constexpr int kABytes = kBM * 128;    // 64 bf16 per row per k-block
constexpr int kBBytes = kMaxN * 128;
constexpr int kAccCols = 128;
constexpr int kTmemCols = 2 * kAccCols;
constexpr int kMaxK = 4096;

enum Mode { GEGLU = 0, DOWN = 1 };

struct Params {
  const int32_t *tiles;
  const int32_t *tile_count;
  const int32_t *perm;
  int32_t *status;
  const uint16_t *scales;  // [E, rows, K/64]
  const uint16_t *biases;
  const float *topk_weights;
  uint16_t *h;     // GEGLU output [A, I]
  float *y_acc;    // DOWN output [T, H]
  int32_t top_k;
  int32_t K;       // reduction length: H (GEGLU) or I (DOWN)
  int32_t N_out;   // I (GEGLU) or H (DOWN)
  int32_t rows_per_expert;  // 2I (GEGLU) or H (DOWN)
  int32_t num_blocks;       // weight-row blocks per tile: I/64 (GEGLU) or ceil(H/128) (DOWN)
};

struct Smem {
  uint64_t nib_full[kNibStages], nib_empty[kNibStages];
  uint64_t a_full[kAStages], a_empty[kAStages];
  uint64_t b_full[kBStages], b_empty[kBStages];
  uint64_t sc_full[2], sc_empty[2];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// byte offsets inside the 1024-aligned dynamic shared memory
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kAStages * kABytes;
constexpr int kOffNib = kOffB + kBStages * kBBytes;
constexpr int kOffSc = kOffNib + kNibStages * kNibBytes;

__host__ __device__ constexpr int sc_buf_bytes(int K) { return kBM * (K / 64) * 2 * 2; }
__host__ __device__ constexpr int smem_total(int K) {
  return kOffSc + 2 * sc_buf_bytes(K) + (int)sizeof(Smem) + 1024;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & mask) | bits
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t mask, uint32_t bits) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));
  return d;
}

// Eight nibbles of one packed word (k = 8w .. 8w+7, lowest nibble first) ->
// four bf16x2 words (k, k+1), w = s*q + b rounded once to bf16.  The pair
// (q_k, q_k+1) is moved into the low nibbles of the two halves with a byte
// permute, OR-ed into the bf16 pattern of 128.0 (giving 128 + q exactly),
// 128 is subtracted exactly, and one bf16x2 fma applies the affine map.
__device__ __forceinline__ void dequant8(uint32_t q, __nv_bfloat162 s2, __nv_bfloat162 b2,
                                         uint32_t (&out)[4]) {
  const uint32_t z = q >> 4;
  const uint32_t k128 = 0x43004300u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t sel = (uint32_t)i | ((uint32_t)i << 4) | ((uint32_t)(4 + i) << 8) |
                         ((uint32_t)(4 + i) << 12);
    uint32_t v = and_or(prmt(q, z, sel), 0x000F000Fu, k128);
    __nv_bfloat162 qv = __hsub2(*reinterpret_cast<__nv_bfloat162 *>(&v),
                                *reinterpret_cast<const __nv_bfloat162 *>(&k128));
    __nv_bfloat162 w = __hfma2(qv, s2, b2);
    out[i] = *reinterpret_cast<uint32_t *>(&w);
  }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void red_add_f32(float *p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_x, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int G = p.K / 64;  // groups per row == k-blocks per unit
  const int scb = sc_buf_bytes(p.K);
  Smem &S = *reinterpret_cast<Smem *>(smem + kOffSc + 2 * scb);
  uint8_t *ringA = smem + kOffA;
  uint8_t *ringB = smem + kOffB;
  uint8_t *ringN = smem + kOffNib;
  uint8_t *ringS = smem + kOffSc;
  volatile int *abort = &S.abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (load_status(p.status) != 0) return;
  const int tile_count = *p.tile_count;
  const int total_units = tile_count * p.num_blocks;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNibStages; ++i) {
      mbar_init(&S.nib_full[i], 1);
      mbar_init(&S.nib_empty[i], kDeqThreads / 32);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&S.a_full[i], kDeqThreads / 32);
      mbar_init(&S.a_empty[i], 1);
    }
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&S.b_full[i], 1);
      mbar_init(&S.b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.sc_full[i], 1);
      mbar_init(&S.sc_empty[i], kDeqThreads / 32);
      mbar_init(&S.acc_full[i], 1);
      mbar_init(&S.acc_empty[i], 4);
    }
    mbar_init(&S.mma_done, 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmap_w);
    prefetch_tensormap(&tmap_x);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = S.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------ W producer
    if (lane == 0) {
      uint32_t it = 0, it_sc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const int tile = u / p.num_blocks, nb = u - tile * p.num_blocks;
        const int e = p.tiles[3 * tile];
        const int sb = it_sc & 1;
        if (!(ok = mbar_wait(&S.sc_empty[sb], ((it_sc >> 1) & 1) ^ 1, abort))) break;
        uint8_t *dst = ringS + sb * scb;
        const int row_bytes = G * 2;
        if (MODE == GEGLU) {
          const int64_t rg = (int64_t)e * p.rows_per_expert + nb * 64;
          const int64_t ru = rg + p.N_out;  // up rows start I rows later
          const uint32_t part = 64 * row_bytes;
          mbar_arrive_expect_tx(&S.sc_full[sb], 4 * part);
          bulk_load(dst, p.scales + rg * G, part, &S.sc_full[sb]);
          bulk_load(dst + part, p.scales + ru * G, part, &S.sc_full[sb]);
          bulk_load(dst + 2 * part, p.biases + rg * G, part, &S.sc_full[sb]);
          bulk_load(dst + 3 * part, p.biases + ru * G, part, &S.sc_full[sb]);
        } else {
          const int n0 = nb * kBM;
          const int rows = min(kBM, p.N_out - n0);
          const int64_t r0 = (int64_t)e * p.rows_per_expert + n0;
          const uint32_t part = rows * row_bytes;
          mbar_arrive_expect_tx(&S.sc_full[sb], 2 * part);
          bulk_load(dst, p.scales + r0 * G, part, &S.sc_full[sb]);
          bulk_load(dst + kBM * row_bytes, p.biases + r0 * G, part, &S.sc_full[sb]);
        }
        ++it_sc;
        for (int kb = 0; kb < G; ++kb, ++it) {
          const int st = it % kNibStages;
          if (!(ok = mbar_wait(&S.nib_empty[st], ((it / kNibStages) & 1) ^ 1, abort))) break;
          mbar_arrive_expect_tx(&S.nib_full[st], kNibBytes);
          uint8_t *nd = ringN + st * kNibBytes;
          if (MODE == GEGLU) {
            const int rg = e * p.rows_per_expert + nb * 64;
            tma_load_2d(nd, &tmap_w, kb * 8, rg, &S.nib_full[st]);
            tma_load_2d(nd + kNibBytes / 2, &tmap_w, kb * 8, rg + p.N_out, &S.nib_full[st]);
          } else {
            tma_load_2d(nd, &tmap_w, kb * 8, e * p.rows_per_expert + nb * kBM, &S.nib_full[st]);
          }
        }
      }
      // drain: wait (bounded) for copies still in flight before the CTA exits
      for (uint32_t i = (it > kNibStages ? it - kNibStages : 0); i < it; ++i)
        mbar_wait(&S.nib_full[i % kNibStages], (i / kNibStages) & 1, nullptr, 200000000ull);
      if (it_sc > 0)
        for (uint32_t i = (it_sc > 2 ? it_sc - 2 : 0); i < it_sc; ++i)
          mbar_wait(&S.sc_full[i & 1], (i >> 1) & 1, nullptr, 200000000ull);
    }
  } else if (warp == 2) {
    // ------------------------------------------------ X producer (B operand rows)
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const int tile = u / p.num_blocks;
      const int row0 = p.tiles[3 * tile + 1], R = p.tiles[3 * tile + 2];
      int src_row[kMaxN / 32];
#pragma unroll
      for (int m = 0; m < kMaxN / 32; ++m) {
        const int j = lane + 32 * m;
        if (MODE == GEGLU)
          src_row[m] = (j < R) ? p.perm[row0 + j] / p.top_k : 0;
        else
          src_row[m] = row0 + 16 * j;  // 16-row boxes of sorted h
      }
      const int nbox = (MODE == GEGLU) ? R : (R + 15) / 16;
      const uint32_t bytes = (MODE == GEGLU) ? R * 128u : nbox * 16u * 128u;
      for (int kb = 0; kb < G; ++kb, ++it) {
        const int st = it % kBStages;
        if (!(ok = mbar_wait(&S.b_empty[st], ((it / kBStages) & 1) ^ 1, abort))) break;
        if (lane == 0) mbar_arrive_expect_tx(&S.b_full[st], bytes);
        __syncwarp();
        uint8_t *bd = ringB + st * kBBytes;
#pragma unroll
        for (int m = 0; m < kMaxN / 32; ++m) {
          const int j = lane + 32 * m;
          if (j < nbox) {
            if (MODE == GEGLU)
              tma_load_2d(bd + j * 128, &tmap_x, kb * 64, src_row[m], &S.b_full[st]);
            else
              tma_load_2d(bd + j * 16 * 128, &tmap_x, kb * 64, src_row[m], &S.b_full[st]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0)
      for (uint32_t i = (it > kBStages ? it - kBStages : 0); i < it; ++i)
        mbar_wait(&S.b_full[i % kBStages], (i / kBStages) & 1, nullptr, 200000000ull);
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t ia = 0, ib = 0, iacc = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const int tile = u / p.num_blocks;
        const int R = p.tiles[3 * tile + 2];
        const uint32_t N = (uint32_t)max(16, (R + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(kBM, N);
        const int buf = iacc & 1;
        if (!(ok = mbar_wait(&S.acc_empty[buf], ((iacc >> 1) & 1) ^ 1, abort))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * kAccCols;
        for (int kb = 0; kb < G; ++kb, ++ia, ++ib) {
          const int sa = ia % kAStages, sbb = ib % kBStages;
          if (!(ok = mbar_wait(&S.a_full[sa], (ia / kAStages) & 1, abort))) break;
          if (!(ok = mbar_wait(&S.b_full[sbb], (ib / kBStages) & 1, abort))) break;
          tc_fence_after();
          const uint32_t a0 = smem_addr(ringA + sa * kABytes);
          const uint32_t b0 = smem_addr(ringB + sbb * kBBytes);
#pragma unroll
          for (int k16 = 0; k16 < 4; ++k16) {
            umma_f16(d_tmem, smem_desc_k128(a0 + 32 * k16), smem_desc_k128(b0 + 32 * k16), idesc,
                     (kb | k16) != 0);
          }
          umma_commit(&S.a_empty[sa]);
          umma_commit(&S.b_empty[sbb]);
        }
        if (!ok) break;
        umma_commit(&S.acc_full[buf]);
        ++iacc;
      }
      // every MMA issued by this thread has completed before TMEM is released
      umma_commit(&S.mma_done);
      mbar_wait(&S.mma_done, 0, nullptr, 200000000ull);
    }
    __syncwarp();
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ------------------------------------------------ epilogue
    const int q = warp - kEpiWarp0;  // TMEM lane quarter of this warp
    uint32_t iacc = 0;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++iacc) {
      const int tile = u / p.num_blocks, nb = u - tile * p.num_blocks;
      const int row0 = p.tiles[3 * tile + 1], R = p.tiles[3 * tile + 2];
      const int buf = iacc & 1;
      if (!mbar_wait(&S.acc_full[buf], (iacc >> 1) & 1, abort)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + buf * kAccCols;
      for (int c0 = 0; c0 < R; c0 += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tbase + c0, v);
        tmem_ld_wait();
        if (MODE == GEGLU) {
          // lanes 0-15 hold gate rows, lanes 16-31 the matching up rows
          const int n = nb * 64 + 16 * q + (lane & 15);
          const int odd = lane >> 4;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float mine = __uint_as_float(v[j]);
            const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
            const float g = odd ? other : mine;
            const float uu = odd ? mine : other;
            if ((j & 1) == odd && c0 + j < R) {
              const float hv = gelu_tanh(g) * uu;
              p.h[(int64_t)(row0 + c0 + j) * p.N_out + n] =
                  __bfloat16_as_ushort(__float2bfloat16_rn(hv));
            }
          }
        } else {
          const int n = nb * kBM + 32 * q + lane;
          const int col = c0 + lane;
          int tok = 0;
          float w = 0.f;
          if (col < R) {
            const int a = p.perm[row0 + col];
            tok = a / p.top_k;
            w = p.topk_weights[a];
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int tj = __shfl_sync(0xffffffffu, tok, j);
            const float wj = __shfl_sync(0xffffffffu, w, j);
            if (c0 + j < R && n < p.N_out)
              red_add_f32(p.y_acc + (int64_t)tj * p.N_out + n, wj * __uint_as_float(v[j]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acc_empty[buf]);
    }
  } else if (warp >= kDeqWarp0) {
    // ------------------------------------------------ dequant
    const int t = threadIdx.x - kDeqWarp0 * 32;
    const int r = t >> 1, half = t & 1;
    int nibrow;
    if (MODE == GEGLU) {
      const int qq = r >> 5, i = r & 31;
      nibrow = (i < 16) ? (16 * qq + i) : (64 + 16 * qq + (i - 16));
    } else {
      nibrow = r;
    }
    const uint32_t a_row_off = (uint32_t)r * 128u;
    const uint32_t sw = (uint32_t)(r & 7);
    uint32_t in = 0, ia = 0, isc = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const int sb = isc & 1;
      if (!(ok = mbar_wait(&S.sc_full[sb], (isc >> 1) & 1, abort))) break;
      const uint16_t *srow = reinterpret_cast<const uint16_t *>(ringS + sb * scb) + nibrow * G;
      const uint16_t *brow = srow + kBM * G;
      for (int kb = 0; kb < G; ++kb, ++in, ++ia) {
        const int sn = in % kNibStages;
        if (!(ok = mbar_wait(&S.nib_full[sn], (in / kNibStages) & 1, abort))) break;
        const uint4 qv =
            *reinterpret_cast<const uint4 *>(ringN + sn * kNibBytes + nibrow * 32 + half * 16);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.nib_empty[sn]);
        const uint16_t s16 = srow[kb], b16 = brow[kb];
        const uint32_t s2u = (uint32_t)s16 | ((uint32_t)s16 << 16);
        const uint32_t b2u = (uint32_t)b16 | ((uint32_t)b16 << 16);
        const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162 *>(&s2u);
        const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162 *>(&b2u);
        uint32_t w0[4], w1[4], w2[4], w3[4];
        dequant8(qv.x, s2, b2, w0);
        dequant8(qv.y, s2, b2, w1);
        dequant8(qv.z, s2, b2, w2);
        dequant8(qv.w, s2, b2, w3);
        const int sa = ia % kAStages;
        if (!(ok = mbar_wait(&S.a_empty[sa], ((ia / kAStages) & 1) ^ 1, abort))) break;
        const uint32_t abase = smem_addr(ringA + sa * kABytes) + a_row_off;
        const uint32_t c = 4u * half;  // first 16-byte chunk of this half row
        st_shared_v4(abase + (((c + 0) ^ sw) << 4), w0[0], w0[1], w0[2], w0[3]);
        st_shared_v4(abase + (((c + 1) ^ sw) << 4), w1[0], w1[1], w1[2], w1[3]);
        st_shared_v4(abase + (((c + 2) ^ sw) << 4), w2[0], w2[1], w2[2], w2[3]);
        st_shared_v4(abase + (((c + 3) ^ sw) << 4), w3[0], w3[1], w3[2], w3[3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.a_full[sa]);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.sc_empty[sb]);
      ++isc;
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && S.abort_flag) raise_status(p.status, MOE_ERR_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

static bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, size_t elem, const void *base,
                        uint64_t dim0, uint64_t dim1, uint32_t box0, uint32_t box1,
                        CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {dim0, dim1};
  const cuuint64_t strides[1] = {dim0 * elem};
  const cuuint32_t box[2] = {box0, box1};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int MODE>
static moe_status launch(const CUtensorMap &mw, const CUtensorMap &mx, const Params &p,
                         int max_units, cudaStream_t stream, const char *what) {
  const int smem = smem_total(p.K);
  static int configured_smem[2] = {0, 0};
  if (configured_smem[MODE] < smem) {
    if (cudaFuncSetAttribute(gemm_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem) != cudaSuccess)
      return check_launch(what);
    configured_smem[MODE] = smem;
  }
  int grid = num_sms();
  if (max_units < grid) grid = max_units;
  if (grid < 1) grid = 1;
  gemm_tc_kernel<MODE><<<grid, kThreads, smem, stream>>>(mw, mx, p);
  return check_launch(what);
}

}  // namespace tc

moe_status tc_supported(int32_t H, int32_t I, int32_t tile_m) {
  if (tile_m > tc::kMaxN) return MOE_ERR_UNSUPPORTED;
  if (H > tc::kMaxK || I > tc::kMaxK) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status launch_geglu_tc(const uint16_t *x, const uint32_t *Wgu, const uint16_t *Sgu,
                           const uint16_t *Bgu, const moe_tiles_t &t, int32_t H, int32_t I,
                           uint16_t *h, cudaStream_t stream) {
  const char *what = "moe_gather_qmm_geglu (tensor cores)";
  CUtensorMap mw, mx;
  if (!tc::make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, Wgu, H / 8,
                       (uint64_t)t.num_experts * 2 * I, 8, 64, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !tc::make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, H, t.num_tokens, 64, 1,
                       CU_TENSOR_MAP_SWIZZLE_128B)) {
    set_error("%s: tensor map encoding failed", what);
    return MOE_ERR_CUDA;
  }
  tc::Params p;
  memset(&p, 0, sizeof p);
  p.tiles = t.tiles;
  p.tile_count = t.tile_count;
  p.perm = t.perm;
  p.status = t.status;
  p.scales = Sgu;
  p.biases = Bgu;
  p.h = h;
  p.top_k = t.top_k;
  p.K = H;
  p.N_out = I;
  p.rows_per_expert = 2 * I;
  p.num_blocks = I / 64;
  return tc::launch<tc::GEGLU>(mw, mx, p, t.max_tiles * p.num_blocks, stream, what);
}

moe_status launch_down_tc(const uint16_t *hin, const uint32_t *Wd, const uint16_t *Sd,
                          const uint16_t *Bd, const moe_tiles_t &t, const float *topk_weights,
                          int32_t H, int32_t I, float *y_acc, cudaStream_t stream) {
  const char *what = "moe_gather_qmm_down_unsort (tensor cores)";
  CUtensorMap mw, mx;
  if (!tc::make_map_2d(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, Wd, I / 8,
                       (uint64_t)t.num_experts * H, 8, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !tc::make_map_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, hin, I, t.num_assignments, 64,
                       16, CU_TENSOR_MAP_SWIZZLE_128B)) {
    set_error("%s: tensor map encoding failed", what);
    return MOE_ERR_CUDA;
  }
  tc::Params p;
  memset(&p, 0, sizeof p);
  p.tiles = t.tiles;
  p.tile_count = t.tile_count;
  p.perm = t.perm;
  p.status = t.status;
  p.scales = Sd;
  p.biases = Bd;
  p.topk_weights = topk_weights;
  p.y_acc = y_acc;
  p.top_k = t.top_k;
  p.K = I;
  p.N_out = H;
  p.rows_per_expert = H;
  p.num_blocks = (H + tc::kBM - 1) / tc::kBM;
  return tc::launch<tc::DOWN>(mw, mx, p, t.max_tiles * p.num_blocks, stream, what);
}

}  // namespace moeqmm
