// Shared device/host helpers of the CUDA library (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_qmm.h"

namespace moeqmm {

// Per-tile gate/up completion counters of the one-launch layer in the down call's
// workspace: two sets of this many (one per call parity), after the grid's arrival count.
constexpr int kFusedTileFlags = 512;

// ---- host-side error reporting (per host thread) ----
void set_error(const char *fmt, ...);
void clear_error();
moe_status check_launch(const char *what);

// ---- device status word ----
// The first error wins; later kernels see a non-zero word and return.
__device__ __forceinline__ void raise_status(int32_t *status, int32_t code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ int32_t load_status(const int32_t *status) {
  return *reinterpret_cast<const volatile int32_t *>(status);
}

// ---- programmatic dependent launch ----
// A kernel launched with launch_pdl may start while the previous kernel on the stream is
// still running: it does its prologue (shared memory, barriers), then griddep_wait()
// before it reads anything an earlier kernel wrote or writes anything an earlier kernel
// reads; griddep_launch() lets the next kernel start its own prologue.  Without the
// launch attribute both are no-ops.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- numerics ----
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float tanh_approx(float v) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}

// geluApproximate: 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))
// (Hendrycks & Gimpel 2016), evaluated in fp32 with the hardware tanh.
__device__ __forceinline__ float gelu_tanh(float z) {
  const float k0 = 0.7978845608028654f;  // sqrt(2/pi)
  const float k1 = 0.044715f;
  float inner = k0 * fmaf(k1 * z, z * z, z);
  return 0.5f * z * (1.0f + tanh_approx(inner));
}

// SiLU, z * sigmoid(z), with sigmoid(z) = (1 + tanh(z / 2)) / 2: the gate activation of the
// SwiGLU product (SharpAI/SwiftLM issue #236, "What #27 set out to do" and "Already on
// main": the silu-mul product), on the same hardware tanh.
__device__ __forceinline__ float silu_f(float z) {
  return 0.5f * z * (1.0f + tanh_approx(0.5f * z));
}

// the gate activation of the gated product: MOE_ACT_GELU_TANH or MOE_ACT_SILU
__device__ __forceinline__ float glu_act(float z, int act) {
  return act == MOE_ACT_SILU ? silu_f(z) : gelu_tanh(z);
}

}  // namespace moeqmm
