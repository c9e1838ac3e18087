// Internal helpers shared by the CUDA translation units of libfa3.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fa3.h"

#define FA3_API extern "C" __attribute__((visibility("default")))

namespace fa3 {

// Host-side check for the current device; the kernels are built for sm_103a only.
int check_device(int* num_sms);

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

__device__ __forceinline__ void set_dev_err(int32_t* err, int bit) {
  if (err) atomicOr(reinterpret_cast<int*>(err), bit);
}

}  // namespace fa3
