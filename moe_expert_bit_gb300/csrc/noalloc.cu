// moe_gather_qmm_down_unsort_noalloc: the down projection + weighted un-sort
// for callers that cannot allocate device memory.
//
// Who needs it: code that runs where a cudaMalloc is not allowed or not
// wanted -- an inference-runtime plugin whose execute step may not allocate,
// a caller with no allocator of its own to hand out a workspace, or a
// latency-critical loop that must never hit the allocator.  This entry point
// takes inputs and the output only; its fp32 y accumulator lives in a
// fixed-size array of device memory declared in this file, which every GPU
// that loads the library holds until the process exits.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moeqmm {

// The shared accumulator: [T, H] fp32 (deterministic: [A, H]), at most
// MOE_NOALLOC_MAX_Y_ELEMENTS floats (16 MiB) with its counters.
static __device__ __align__(256) float g_noalloc_y_acc[MOE_NOALLOC_MAX_Y_ELEMENTS];

constexpr int kMaxDevices = 64;
static std::mutex g_noalloc_mutex;
static float *g_noalloc_ptr[kMaxDevices];  // device address of the array, per device

// The host-side name of the array is not a device address: look the address
// up once per device, with that device current, and cache it.
static moe_status noalloc_scratch(float **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    set_error("moe_gather_qmm_down_unsort_noalloc: no usable current device (%d)", dev);
    return MOE_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_y_acc);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      set_error("moe_gather_qmm_down_unsort_noalloc: cudaGetSymbolAddress failed: %s",
                cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_noalloc_ptr[dev];
  return MOE_OK;
}

}  // namespace moeqmm

using namespace moeqmm;

extern "C" moe_status moe_gather_qmm_down_unsort_noalloc(
    const moe_bf16_t *h, const uint32_t *Wd, const moe_bf16_t *Sd, const moe_bf16_t *Bd,
    const moe_tiles_t *tiles, const float *topk_weights, int32_t H, int32_t I, int32_t variant,
    int32_t deterministic, moe_bf16_t *y, cudaStream_t stream) {
  const char *fn = "moe_gather_qmm_down_unsort_noalloc";
  clear_error();
  if (!tiles) {
    set_error("%s: tiles is null", fn);
    return MOE_ERR_INVALID_ARG;
  }
  if (deterministic != 0 && deterministic != 1) {
    set_error("%s: deterministic must be 0 or 1 (got %d)", fn, deterministic);
    return MOE_ERR_INVALID_ARG;
  }
  if (tiles->num_tokens > 0 && tiles->top_k > 0 && H > 0 &&
      moe_unsort_workspace_bytes(tiles->num_tokens, tiles->top_k, H, deterministic) >
          sizeof(float) * MOE_NOALLOC_MAX_Y_ELEMENTS) {
    set_error("%s: %s*H = %lld exceeds the built-in accumulator of %d fp32 elements; "
              "use moe_gather_qmm_down_unsort with a caller workspace",
              fn, deterministic ? "A" : "T",
              (long long)(deterministic ? tiles->num_assignments : tiles->num_tokens) * H,
              MOE_NOALLOC_MAX_Y_ELEMENTS);
    return MOE_ERR_UNSUPPORTED;
  }
  if (!h || !Wd || !Sd || !Bd || !topk_weights || !y) {
    set_error("%s: null pointer", fn);
    return MOE_ERR_INVALID_ARG;
  }
  float *scratch = nullptr;
  moe_status st = noalloc_scratch(&scratch);
  if (st != MOE_OK) return st;
  // The full validation and launch sequence of the workspace entry point, pointed at
  // the built-in accumulator, which is cleared first (after validation): a call that
  // stopped on a device error cannot leave it dirty for the next one.
  return down_unsort(fn, h, Wd, Sd, Bd, tiles, topk_weights, H, I, variant, scratch,
                     deterministic, y, true, stream);
}
