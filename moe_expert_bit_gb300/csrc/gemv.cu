// CUDA-core weight-streaming kernels for the two projections (the GEMV-style
// variant).  One warp owns one output row of one expert tile and streams
// that row's packed nibbles once, applying each dequantised weight to the
// tile's activation rows (up to kRows at a time, staged in shared memory).
// Suited to decode, where a tile holds one or two rows and the layer is a
// pure weight stream.
//
//   gate/up:  h[s, n] = gelu_tanh(sum_k Wg[e][n][k] x_s[k]) * sum_k Wu[e][n][k] x_s[k]
//   down:     y_acc[t, n] += w_a * sum_i Wd[e][n][i] h[s, i],  a = perm[s], t = a / top_k
// with w = scale * q + bias per 64-group (Layr-Labs/mlx PR #4, "What";
// SharpAI/SwiftLM issue #236, "Still missing" and "Already on main").
#include "common.cuh"
#include "kernels.h"

namespace moeqmm {

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kRows = 4;  // activation rows per pass

// 8 consecutive bf16 (one uint4) -> fp32
__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

// grid: (max_tiles, ceil(I / kGemvWarps)); dynamic smem: kRows * H bf16
__global__ void __launch_bounds__(kGemvThreads)
    geglu_gemv_kernel(const uint16_t *__restrict__ x, const uint32_t *__restrict__ Wgu,
                      const uint16_t *__restrict__ Sgu, const uint16_t *__restrict__ Bgu,
                      const int32_t *__restrict__ tiles, const int32_t *__restrict__ tile_count,
                      const int32_t *__restrict__ perm, const int32_t *__restrict__ status,
                      int32_t top_k, int32_t H, int32_t I, uint16_t *__restrict__ h) {
  extern __shared__ __align__(16) uint16_t xs[];  // [kRows][H]
  if (load_status(status) != 0) return;
  const int tile = blockIdx.x;
  if (tile >= *tile_count) return;
  const int e = tiles[3 * tile], row0 = tiles[3 * tile + 1], rows = tiles[3 * tile + 2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.y * kGemvWarps + warp;
  const int words = H / 8, groups = H / 64;
  const int64_t rg = (int64_t)e * 2 * I + n;  // gate row
  const int64_t ru = rg + I;                  // up row
  for (int r0 = 0; r0 < rows; r0 += kRows) {
    const int R = min(kRows, rows - r0);
    __syncthreads();
    for (int i = threadIdx.x; i < R * words; i += kGemvThreads) {  // 16-byte chunks
      const int r = i / words, c = i - r * words;
      const int t = perm[row0 + r0 + r] / top_k;
      reinterpret_cast<uint4 *>(xs + (size_t)r * H)[c] =
          reinterpret_cast<const uint4 *>(x + (size_t)t * H)[c];
    }
    __syncthreads();
    if (n >= I) continue;
    float ag[kRows], au[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) ag[r] = au[r] = 0.f;
    for (int w = lane; w < words; w += 32) {
      const uint32_t qg = Wgu[rg * words + w], qu = Wgu[ru * words + w];
      const int g = w >> 3;
      const float sg = bf16_bits_to_float(Sgu[rg * groups + g]);
      const float bg = bf16_bits_to_float(Bgu[rg * groups + g]);
      const float su = bf16_bits_to_float(Sgu[ru * groups + g]);
      const float bu = bf16_bits_to_float(Bgu[ru * groups + g]);
      float wg[8], wu[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        wg[j] = fmaf(sg, (float)((qg >> (4 * j)) & 15u), bg);
        wu[j] = fmaf(su, (float)((qu >> (4 * j)) & 15u), bu);
      }
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        if (r < R) {
          float xf[8];
          bf16x8_to_f32(reinterpret_cast<const uint4 *>(xs + (size_t)r * H)[w], xf);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            ag[r] = fmaf(wg[j], xf[j], ag[r]);
            au[r] = fmaf(wu[j], xf[j], au[r]);
          }
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const float g = warp_sum(ag[r]), u = warp_sum(au[r]);
      if (lane == r && r < R) {
        const float hv = gelu_tanh(g) * u;
        h[(int64_t)(row0 + r0 + r) * I + n] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
      }
    }
  }
}

// grid: (max_tiles, ceil(H / kGemvWarps)); dynamic smem: kRows * I bf16
__global__ void __launch_bounds__(kGemvThreads)
    down_gemv_kernel(const uint16_t *__restrict__ hin, const uint32_t *__restrict__ Wd,
                     const uint16_t *__restrict__ Sd, const uint16_t *__restrict__ Bd,
                     const int32_t *__restrict__ tiles, const int32_t *__restrict__ tile_count,
                     const int32_t *__restrict__ perm, const float *__restrict__ topk_weights,
                     const int32_t *__restrict__ status, int32_t top_k, int32_t H, int32_t I,
                     float *__restrict__ y_acc) {
  extern __shared__ __align__(16) uint16_t hs[];  // [kRows][I]
  if (load_status(status) != 0) return;
  const int tile = blockIdx.x;
  if (tile >= *tile_count) return;
  const int e = tiles[3 * tile], row0 = tiles[3 * tile + 1], rows = tiles[3 * tile + 2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.y * kGemvWarps + warp;
  const int words = I / 8, groups = I / 64;
  const int64_t rd = (int64_t)e * H + n;
  for (int r0 = 0; r0 < rows; r0 += kRows) {
    const int R = min(kRows, rows - r0);
    __syncthreads();
    for (int i = threadIdx.x; i < R * words; i += kGemvThreads) {
      const int r = i / words, c = i - r * words;
      reinterpret_cast<uint4 *>(hs + (size_t)r * I)[c] =
          reinterpret_cast<const uint4 *>(hin + (size_t)(row0 + r0 + r) * I)[c];
    }
    __syncthreads();
    if (n >= H) continue;
    float acc[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r) acc[r] = 0.f;
    for (int w = lane; w < words; w += 32) {
      const uint32_t q = Wd[rd * words + w];
      const int g = w >> 3;
      const float s = bf16_bits_to_float(Sd[rd * groups + g]);
      const float b = bf16_bits_to_float(Bd[rd * groups + g]);
      float wv[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) wv[j] = fmaf(s, (float)((q >> (4 * j)) & 15u), b);
#pragma unroll
      for (int r = 0; r < kRows; ++r) {
        if (r < R) {
          float hf[8];
          bf16x8_to_f32(reinterpret_cast<const uint4 *>(hs + (size_t)r * I)[w], hf);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[r] = fmaf(wv[j], hf[j], acc[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const float o = warp_sum(acc[r]);
      if (lane == r && r < R) {
        const int a = perm[row0 + r0 + r];
        const int t = a / top_k;
        atomicAdd(&y_acc[(int64_t)t * H + n], topk_weights[a] * o);
      }
    }
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

moe_status launch_geglu_gemv(const uint16_t *x, const uint32_t *Wgu, const uint16_t *Sgu,
                             const uint16_t *Bgu, const moe_tiles_t &t, int32_t H, int32_t I,
                             uint16_t *h, cudaStream_t stream) {
  const size_t smem = (size_t)kRows * H * sizeof(uint16_t);
  if (smem > 48 * 1024) {
    cudaFuncSetAttribute(geglu_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  }
  dim3 grid(t.max_tiles, (I + kGemvWarps - 1) / kGemvWarps);
  geglu_gemv_kernel<<<grid, kGemvThreads, smem, stream>>>(x, Wgu, Sgu, Bgu, t.tiles, t.tile_count,
                                                          t.perm, t.status, t.top_k, H, I, h);
  return check_launch("moe_gather_qmm_geglu (gemv)");
}

moe_status launch_down_gemv(const uint16_t *hin, const uint32_t *Wd, const uint16_t *Sd,
                            const uint16_t *Bd, const moe_tiles_t &t, const float *topk_weights,
                            int32_t H, int32_t I, float *y_acc, cudaStream_t stream) {
  const size_t smem = (size_t)kRows * I * sizeof(uint16_t);
  if (smem > 48 * 1024) {
    cudaFuncSetAttribute(down_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  }
  dim3 grid(t.max_tiles, (H + kGemvWarps - 1) / kGemvWarps);
  down_gemv_kernel<<<grid, kGemvThreads, smem, stream>>>(hin, Wd, Sd, Bd, t.tiles, t.tile_count,
                                                         t.perm, topk_weights, t.status, t.top_k,
                                                         H, I, y_acc);
  return check_launch("moe_gather_qmm_down_unsort (gemv)");
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
