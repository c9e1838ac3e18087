// Internal helpers shared by the CUDA translation units of libfa3.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "fa3.h"

#define FA3_API extern "C" __attribute__((visibility("default")))

namespace fa3 {

// Host-side check for the current device; the kernels are built for sm_103a only.
int check_device(int* num_sms);

// Optional caller events recorded around the main kernel of a call (fa3_set_kernel_timing).
void timing_begin(cudaStream_t s);
void timing_end(cudaStream_t s);

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FA3_OK : FA3_ECUDA; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// bf16 bit pattern -> float (exact).
__device__ __forceinline__ float bf16_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Symmetric INT8 code: clamp(round_half_even(x / s), -127, 127), s == 0 -> 0.
// __fdiv_rn is the IEEE float32 division; __float2int_rn rounds half to even.
__device__ __forceinline__ int quant_code(float x, float s) {
  if (s == 0.0f) return 0;
  float r = __fdiv_rn(x, s);
  r = fminf(fmaxf(r, -127.0f), 127.0f);
  return __float2int_rn(r);
}

// Approximate reciprocal (hardware rcp, flush-to-zero); only used to pick codes
// where the decision cannot differ from the IEEE quotient's (see quant_code_fast).
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// Same code as quant_code(x, s), without a division in the common case.  With
// rs = rcp_approx(s), y = x * rs is within 2.2e-4 of the correctly rounded
// quotient whenever |x / s| < 200 (rcp error <= 2^-20, two roundings), so when y
// is farther than 1e-3 from every half-integer its round-half-even is the
// quotient's; beyond 127.01 both clamp to +-127.  Everything else (ties,
// overflow, subnormal scales) takes the IEEE division.
__device__ __forceinline__ int quant_code_fast(float x, float s, float rs) {
  if (s == 0.0f) return 0;
  const float y = x * rs;
  const float a = fabsf(y);
  if (a < 127.0f) {
    if (fabsf(a - floorf(a) - 0.5f) >= 1e-3f) return __float2int_rn(y);
  } else if (a >= 127.01f && a <= 3.0e38f) {
    return y > 0.0f ? 127 : -127;
  }
  return quant_code(x, s);
}

// Programmatic dependent launch.  Every kernel of the library is launched as a
// programmatic dependent of the work before it on the stream (launch_pdl): it
// calls pdl_wait() before its first access to memory another kernel may write,
// and pdl_launch_dependents() once the next kernel may start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void set_dev_err(int32_t* err, int bit) {
  if (err) atomicOr(reinterpret_cast<int*>(err), bit);
}

}  // namespace fa3
