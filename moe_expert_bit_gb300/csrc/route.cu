// Routing half of the layer: the stable counting sort of the top-k
// assignments by expert (step a1) and the tile-descriptor builder with its
// sortedness self-check (step a2).  Both are single-CTA kernels: the inputs
// are at most a few tens of KB, and one CTA keeps every step on-chip.
//
// Layr-Labs/mlx PR #4, "What": the gathered QMM consumes contiguous sorted
// indices; its descriptor builder runs on one threadgroup (binary search of
// each expert's sorted range, exclusive scan of per-expert tile counts,
// strided emission).  Review finding F2 and the final review wave: an
// adjacent-pair scan proves global order; a violation yields zero tiles.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "common.cuh"

namespace moeqmm {

static thread_local char g_err[512];

void set_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
}

void clear_error() { g_err[0] = 0; }

moe_status check_launch(const char *what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s: %s", what, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

constexpr int kSortThreads = 1024;  // the most threads of a sort block
constexpr int kSortWarps = kSortThreads / 32;
constexpr int kSmemSorted = 2048;   // up to this many sorted ids are also kept on-chip

// Threads of a sort block: one per assignment (rounded to whole warps), at most 1024;
// small calls (decode) then pay for no idle warps at the block barriers.
static int sort_threads(int64_t A) {
  const int64_t t = (A + 31) / 32 * 32;
  return t < 64 ? 64 : t > kSortThreads ? kSortThreads : (int)t;
}

// Stable counting sort, one CTA, two passes over the ids with no block barrier inside a
// pass.  Warp w owns a contiguous range of the flat indices (ranges ascend with w).
//  pass 1: each warp counts its range's ids per expert, 32 at a time: __match_any_sync
//          groups equal experts and the group's lowest lane adds the group size to the
//          warp's counter of that expert (+ range check);
//  scan:   per expert, its total over the warps; an exclusive scan over experts gives each
//          expert's first slot; per expert, the warps' counts are scanned in warp order,
//          giving each (warp, expert) the first slot of its ids;
//  pass 2: each warp walks its range again: an id's slot is its (warp, expert) cursor plus
//          its rank among equal ids of the same 32 (a popcount of the lower lanes), then
//          the group's lowest lane advances the cursor.
// Slots therefore follow ascending flat index within every expert.
struct SortSmem {
  int32_t hist[MOE_MAX_EXPERTS];
  int32_t off[MOE_MAX_EXPERTS + 1];  // first slot of each expert (+ A)
  int32_t warp[kSortWarps][MOE_MAX_EXPERTS];
  int32_t sorted[kSmemSorted];  // copy of sorted_ids when A <= kSmemSorted
  int32_t bad;
};

// Returns false (status raised) if an id is out of range.  Block of 64 .. kSortThreads
// threads, a multiple of 32.
__device__ bool sort_body(SortSmem &sm, const int32_t *__restrict__ ids, int32_t A, int32_t E,
                          int32_t *__restrict__ sorted_ids, int32_t *__restrict__ perm,
                          int32_t *__restrict__ counts, int32_t *__restrict__ status) {
  int32_t(*cnt)[MOE_MAX_EXPERTS] = sm.warp;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x, nw = nthr >> 5;
  // this warp's range, in whole rounds of 32
  const int per = ((A + nw - 1) / nw + 31) & ~31;
  const int w0 = min(A, warp * per), w1 = min(A, w0 + per);
  const uint32_t lt_mask = (1u << lane) - 1u;

  for (int i = tid; i < nw * MOE_MAX_EXPERTS; i += nthr) (&cnt[0][0])[i] = 0;
  if (tid == 0) sm.bad = 0;
  __syncthreads();

  bool bad = false;
  for (int base = w0; base < w1; base += 32) {
    const int a = base + lane;
    int32_t e = a < w1 ? ids[a] : -1;
    if (a < w1 && (e < 0 || e >= E)) {
      bad = true;
      e = -2;  // out of range: not counted
    }
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    if (e >= 0 && (same & lt_mask) == 0) cnt[warp][e] += __popc(same);
  }
  if (bad) sm.bad = 1;
  __syncthreads();
  if (sm.bad) {
    if (tid == 0) raise_status(status, MOE_ERR_RANGE);
    return false;
  }
  for (int ex = tid; ex < E; ex += nthr) {  // per-expert totals
    int32_t t = 0;
    for (int w = 0; w < nw; ++w) t += cnt[w][ex];
    sm.hist[ex] = t;
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan over <= 256 experts, 8 per lane
    int32_t local[8];
    int32_t sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      local[i] = (e < E) ? sm.hist[e] : 0;
      sum += local[i];
    }
    int32_t incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int32_t run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < E) {
        sm.off[e] = run;
        counts[e] = local[i];
      }
      run += local[i];
    }
    if (lane == 31) sm.off[E] = run;
  }
  __syncthreads();
  for (int ex = tid; ex < E; ex += nthr) {  // each (warp, expert): its first slot
    int32_t run = sm.off[ex];
    for (int w = 0; w < nw; ++w) {
      const int32_t c = cnt[w][ex];
      cnt[w][ex] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int base = w0; base < w1; base += 32) {
    const int a = base + lane;
    const bool valid = a < w1;
    const int32_t e = valid ? ids[a] : -1;
    const uint32_t same = __match_any_sync(0xffffffffu, e);
    const int32_t rank = __popc(same & lt_mask);
    if (valid) {
      const int32_t slot = cnt[warp][e] + rank;
      sorted_ids[slot] = e;
      perm[slot] = a;
      if (A <= kSmemSorted) sm.sorted[slot] = e;
    }
    __syncwarp();
    if (valid && rank == 0) cnt[warp][e] += __popc(same);
    __syncwarp();
  }
  return true;
}

__global__ void __launch_bounds__(kSortThreads)
    sort_assignments_kernel(const int32_t *__restrict__ ids, int32_t A, int32_t E,
                            int32_t *__restrict__ sorted_ids, int32_t *__restrict__ perm,
                            int32_t *__restrict__ counts, int32_t *__restrict__ status) {
  __shared__ SortSmem sm;
  griddep_wait();
  griddep_launch();
  if (load_status(status) != 0) return;
  sort_body(sm, ids, A, E, sorted_ids, perm, counts, status);
}

constexpr int kTileThreads = 512;

struct TileSmem {
  int32_t off[MOE_MAX_EXPERTS + 1];
  int32_t tstart[MOE_MAX_EXPERTS + 1];
};

__device__ __forceinline__ int32_t lower_bound_dev(const int32_t *v, int32_t n, int32_t key) {
  int32_t lo = 0, hi = n;
  while (lo < hi) {
    int32_t mid = (lo + hi) >> 1;
    if (v[mid] < key)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

// Offsets, tile counts, exclusive scan and strided descriptor emission, one CTA.
// Block of any multiple of 32 threads (>= 32).  known_off: each expert's first slot when
// the caller already has it (the fused kernel's sort), else found by binary search.
__device__ void build_body(TileSmem &sm, const int32_t *__restrict__ sorted_ids, int32_t A,
                           int32_t E, int32_t BM, int32_t *__restrict__ offsets,
                           int32_t *__restrict__ tiles, int32_t *__restrict__ tile_count,
                           int32_t *__restrict__ status, const int32_t *known_off = nullptr) {
  int32_t *s_off = sm.off, *s_tstart = sm.tstart;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthr = blockDim.x;
  // self-check: every id in range and every adjacent pair in order
  int range_bad = 0, order_bad = 0;
  for (int s = tid; s < A; s += nthr) {
    int32_t v = sorted_ids[s];
    range_bad |= (v < 0 || v >= E);
    if (s + 1 < A) order_bad |= (v > sorted_ids[s + 1]);
  }
  range_bad = __syncthreads_or(range_bad);
  order_bad = __syncthreads_or(order_bad);
  if (range_bad || order_bad) {
    if (tid == 0) {
      *tile_count = 0;
      raise_status(status, range_bad ? MOE_ERR_RANGE : MOE_ERR_UNSORTED);
    }
    return;
  }
  // per-expert sorted range (on a sorted array the binary search and the sort's scan agree)
  for (int e = tid; e <= E; e += nthr)
    s_off[e] = known_off ? known_off[e] : (e == E) ? A : lower_bound_dev(sorted_ids, A, e);
  __syncthreads();
  // tiles per expert, exclusive scan by warp 0 (8 experts per lane)
  if (warp == 0) {
    int32_t local[8];
    int32_t sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int e = lane * 8 + i;
      int32_t c = (e < E) ? (s_off[e + 1] - s_off[e]) : 0;
      local[i] = (c + BM - 1) / BM;
      sum += local[i];
    }
    int32_t incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int32_t v = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += v;
    }
    int32_t run = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int e = lane * 8 + i;
      if (e < E) s_tstart[e] = run;
      run += local[i];
    }
    if (lane == 31) s_tstart[E] = incl;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += nthr) offsets[e] = s_off[e];
  const int32_t total = s_tstart[E];
  // strided emission: tile i belongs to the last expert whose first tile is <= i
  for (int i = tid; i < total; i += nthr) {
    int32_t lo = 0, hi = E;  // largest e in [0, E) with s_tstart[e] <= i
    while (hi - lo > 1) {
      int32_t mid = (lo + hi) >> 1;
      if (s_tstart[mid] <= i)
        lo = mid;
      else
        hi = mid;
    }
    const int32_t e = lo;
    const int32_t r = i - s_tstart[e];
    const int32_t c = s_off[e + 1] - s_off[e];
    tiles[3 * i + 0] = e;
    tiles[3 * i + 1] = s_off[e] + r * BM;
    tiles[3 * i + 2] = min(BM, c - r * BM);
  }
  if (tid == 0) *tile_count = total;
}

__global__ void __launch_bounds__(kTileThreads)
    build_expert_tiles_kernel(const int32_t *__restrict__ sorted_ids, int32_t A, int32_t E,
                              int32_t BM, int32_t *__restrict__ offsets,
                              int32_t *__restrict__ tiles, int32_t *__restrict__ tile_count,
                              int32_t *__restrict__ status) {
  __shared__ TileSmem sm;
  griddep_wait();
  griddep_launch();
  if (load_status(status) != 0) {
    if (threadIdx.x == 0) *tile_count = 0;
    return;
  }
  build_body(sm, sorted_ids, A, E, BM, offsets, tiles, tile_count, status);
}

// Steps a1 and a2 in one launch: the sort, then (after a block barrier, which also
// makes this block's global writes of sorted_ids visible to it) the tile builder.
__global__ void __launch_bounds__(kSortThreads)
    route_kernel(const int32_t *__restrict__ ids, int32_t A, int32_t E, int32_t BM,
                 int32_t *__restrict__ sorted_ids, int32_t *__restrict__ perm,
                 int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                 int32_t *__restrict__ tiles, int32_t *__restrict__ tile_count,
                 int32_t *__restrict__ status) {
  __shared__ SortSmem ssm;
  __shared__ TileSmem tsm;
  griddep_wait();
  griddep_launch();
  if (load_status(status) != 0) {
    if (threadIdx.x == 0) *tile_count = 0;
    return;
  }
  if (!sort_body(ssm, ids, A, E, sorted_ids, perm, counts, status)) {
    if (threadIdx.x == 0) *tile_count = 0;
    return;
  }
  __syncthreads();
  // the builder checks the sort's output: its on-chip copy when there is one
  build_body(tsm, A <= kSmemSorted ? ssm.sorted : sorted_ids, A, E, BM, offsets, tiles,
             tile_count, status, ssm.off);
}

}  // namespace moeqmm

using namespace moeqmm;

extern "C" {

const char *moe_last_error_string(void) { return g_err; }

size_t moe_max_tiles(int32_t A, int32_t E, int32_t BM) {
  if (A < 0 || E < 1 || BM < 1) return 0;
  return static_cast<size_t>(A / BM) + static_cast<size_t>(A < E ? A : E);
}

size_t moe_workspace_bytes(int32_t T, int32_t H) {
  if (T < 1 || H < 1) return 0;
  // the fp32 accumulator, then one int counter per 16 output columns and the fused
  // layer's grid barrier (a 64-bit arrival count, two spare ints), 16-byte padded
  const size_t counters = ((static_cast<size_t>(H) / 16 + 4) * sizeof(int32_t) + 15) / 16 * 16;
  return static_cast<size_t>(T) * static_cast<size_t>(H) * sizeof(float) + counters;
}

size_t moe_unsort_workspace_bytes(int32_t T, int32_t k, int32_t H, int32_t deterministic) {
  if (T < 1 || k < 1 || H < 1) return 0;
  if (!deterministic) return moe_workspace_bytes(T, H);
  // one fp32 row per assignment instead of per token; the same counters after it
  const int64_t A = static_cast<int64_t>(T) * k;
  if (A > INT32_MAX) return 0;
  return moe_workspace_bytes(static_cast<int32_t>(A), H);
}

moe_status moe_sort_assignments(const int32_t *topk_ids, int32_t T, int32_t k, int32_t E,
                                int32_t *sorted_ids, int32_t *perm, int32_t *counts,
                                int32_t *status, cudaStream_t stream) {
  clear_error();
  if (!topk_ids || !sorted_ids || !perm || !counts || !status) {
    set_error("moe_sort_assignments: null pointer");
    return MOE_ERR_INVALID_ARG;
  }
  if (E < 1 || E > MOE_MAX_EXPERTS) {
    set_error("moe_sort_assignments: num_experts %d outside [1, %d]", E, MOE_MAX_EXPERTS);
    return MOE_ERR_UNSUPPORTED;
  }
  if (T < 1 || k < 1 || k > E) {
    set_error("moe_sort_assignments: need T >= 1 and 1 <= k <= E (T=%d k=%d E=%d)", T, k, E);
    return MOE_ERR_INVALID_ARG;
  }
  const int64_t A = static_cast<int64_t>(T) * k;
  if (A > (int64_t(1) << 24)) {
    set_error("moe_sort_assignments: %lld assignments exceed 2^24", (long long)A);
    return MOE_ERR_UNSUPPORTED;
  }
  launch_pdl(sort_assignments_kernel, dim3(1), dim3(sort_threads(A)), 0, stream, topk_ids,
             static_cast<int32_t>(A), E, sorted_ids, perm, counts, status);
  return check_launch("moe_sort_assignments");
}

moe_status moe_build_expert_tiles(const int32_t *sorted_ids, int32_t A, int32_t E, int32_t BM,
                                  int32_t max_tiles, int32_t *offsets, int32_t *tiles,
                                  int32_t *tile_count, int32_t *status, cudaStream_t stream) {
  clear_error();
  if (!sorted_ids || !offsets || !tiles || !tile_count || !status) {
    set_error("moe_build_expert_tiles: null pointer");
    return MOE_ERR_INVALID_ARG;
  }
  if (E < 1 || E > MOE_MAX_EXPERTS) {
    set_error("moe_build_expert_tiles: num_experts %d outside [1, %d]", E, MOE_MAX_EXPERTS);
    return MOE_ERR_UNSUPPORTED;
  }
  if (BM != 16 && BM != 32 && BM != 64 && BM != 128 && BM != 256) {
    set_error("moe_build_expert_tiles: tile_m %d not in {16, 32, 64, 128, 256}", BM);
    return MOE_ERR_UNSUPPORTED;
  }
  if (A < 1 || A > (1 << 24)) {
    set_error("moe_build_expert_tiles: num_assignments %d outside [1, 2^24]", A);
    return MOE_ERR_INVALID_ARG;
  }
  const size_t need = moe_max_tiles(A, E, BM);
  if (max_tiles < 0 || static_cast<size_t>(max_tiles) < need) {
    set_error("moe_build_expert_tiles: max_tiles %d < required %zu", max_tiles, need);
    return MOE_ERR_INVALID_ARG;
  }
  launch_pdl(build_expert_tiles_kernel, dim3(1), dim3(kTileThreads), 0, stream, sorted_ids, A, E,
             BM, offsets, tiles, tile_count, status);
  return check_launch("moe_build_expert_tiles");
}

moe_status moe_sort_and_build_tiles(const int32_t *topk_ids, int32_t T, int32_t k, int32_t E,
                                    int32_t tile_m, int32_t max_tiles, int32_t *sorted_ids,
                                    int32_t *perm, int32_t *counts, int32_t *offsets,
                                    int32_t *tiles, int32_t *tile_count, int32_t *status,
                                    cudaStream_t stream) {
  clear_error();
  if (!topk_ids || !sorted_ids || !perm || !counts || !offsets || !tiles || !tile_count ||
      !status) {
    set_error("moe_sort_and_build_tiles: null pointer");
    return MOE_ERR_INVALID_ARG;
  }
  if (E < 1 || E > MOE_MAX_EXPERTS) {
    set_error("moe_sort_and_build_tiles: num_experts %d outside [1, %d]", E, MOE_MAX_EXPERTS);
    return MOE_ERR_UNSUPPORTED;
  }
  if (T < 1 || k < 1 || k > E) {
    set_error("moe_sort_and_build_tiles: need T >= 1 and 1 <= k <= E (T=%d k=%d E=%d)", T, k, E);
    return MOE_ERR_INVALID_ARG;
  }
  const int64_t A = static_cast<int64_t>(T) * k;
  if (A > (int64_t(1) << 24)) {
    set_error("moe_sort_and_build_tiles: %lld assignments exceed 2^24", (long long)A);
    return MOE_ERR_UNSUPPORTED;
  }
  if (tile_m != 16 && tile_m != 32 && tile_m != 64 && tile_m != 128 && tile_m != 256) {
    set_error("moe_sort_and_build_tiles: tile_m %d not in {16, 32, 64, 128, 256}", tile_m);
    return MOE_ERR_UNSUPPORTED;
  }
  const size_t need = moe_max_tiles(static_cast<int32_t>(A), E, tile_m);
  if (max_tiles < 0 || static_cast<size_t>(max_tiles) < need) {
    set_error("moe_sort_and_build_tiles: max_tiles %d < required %zu", max_tiles, need);
    return MOE_ERR_INVALID_ARG;
  }
  launch_pdl(route_kernel, dim3(1), dim3(sort_threads(A)), 0, stream, topk_ids,
             static_cast<int32_t>(A), E, tile_m, sorted_ids, perm, counts, offsets, tiles,
             tile_count, status);
  return check_launch("moe_sort_and_build_tiles");
}

}  // extern "C"
