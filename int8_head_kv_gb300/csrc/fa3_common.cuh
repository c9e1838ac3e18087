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
// where the decision cannot differ from the IEEE quotient's (see quant_group8_biased).
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// ---------------------------------------------------------------------------
// Codes of eight bf16 values at once (one 16-byte group), bit-identical to
// quant_code(x, s) for every input.
//
// Fast path, two values per packed f32x2 instruction: t = fma(x, rs, 1.5*2^23)
// rounds x*rs half-to-even into the low mantissa bits of t (exact for |x*rs| <
// 2^22), so the integer clamp of t's bit pattern to [magic-127, magic+127]
// leaves the clamped code in its low byte, and also handles |x*rs| >= 2^22 and
// +-inf (the bit patterns fall outside the range on the correct side).  The code
// is the quotient's whenever d = x*rs - RNE(x*rs) stays within kTieBand of 1/2:
// rcp.approx is within 2^-23.28 relative on sm_103a (measured over every
// mantissa), so x*rs is within 2.5e-4 of x/s for |x/s| <= 128 even at 2^-19,
// and |x/s - RNE(x*rs)| < 1/2 by a margin the float32 rounding of the quotient
// cannot cross.
//
// Rare path, per lane, for values within the band of a half-integer h (or NaN,
// or any value when s is not a normal scale in [2^-100, 2^100]): the decision
// is taken exactly from the sign of a - |h|*s (a = |x|), which one fma computes
// without rounding because a and |h|*s agree to within 2^-10 * s and both are
// multiples of ulp(s)/2.  fl(a/s) rounds to |h| exactly when a/s lies within
// half an ulp of |h| (the ulp below |h| is half as wide at |h| = 1/2), and |h|
// itself, having at most 8 significant bits, is an even float32.
// ---------------------------------------------------------------------------
constexpr float kTieBand = 2.5e-4f;

__device__ __forceinline__ bool exact_scale(float s) {
  return s >= 7.888609052210118e-31f && s <= 1.2676506002282294e30f;   // [2^-100, 2^100]
}

// clamp(RNE(fl(x / s))) for x / s within 5e-4 of a half-integer of magnitude <= 127.5,
// s an exact_scale and x finite.
__device__ __forceinline__ int tie_code(float x, float s, float rs) {
  const float a = fabsf(x);
  const float h = floorf(a * rs) + 0.5f;
  const float t = fmaf(-h, s, a);                                                     // a - h*s, exact
  const float ulp = __uint_as_float((__float_as_uint(h) & 0x7f800000u) - (23u << 23));
  const float up = ulp * 0.5f * s;
  const float dn = h == 0.5f ? 0.5f * up : up;
  float c = t > up ? h + 0.5f : (t < -dn ? h - 0.5f : rintf(h));
  c = fminf(c, 127.0f);
  const int ci = (int)c;
  return x < 0.0f ? -ci : ci;
}

__device__ __forceinline__ unsigned long long f32x2_pack(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_unpack(unsigned long long v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f32x2_fma(unsigned long long a, unsigned long long b,
                                                        unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long f32x2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

constexpr float kCodeMagic = 12582912.0f;                  // 1.5 * 2^23
constexpr int kCodeMagicBits = 0x4B400000;                 // its bit pattern

// v: eight bf16 values (element e in bits 16*(e%2) of word e/2).  q[e] receives the
// bit pattern of the float 1.5*2^23 + code(e): its low byte is the code's, and
// __int_as_float(q[e]) - 1.5*2^23 is the code as an exact float.  rs =
// rcp_approx(s), exact = exact_scale(s).
__device__ __forceinline__ void quant_group8_biased(uint4 v, float s, float rs, bool exact, int (&q)[8]) {
  constexpr int kLo = kCodeMagicBits - 127, kHi = kCodeMagicBits + 127;
  const unsigned long long m2 = f32x2_pack(kCodeMagic, kCodeMagic), rs2 = f32x2_pack(rs, rs);
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  bool rare = !exact;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const unsigned long long x2 = f32x2_pack(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xffff0000u));
    const unsigned long long t2 = f32x2_fma(x2, rs2, m2);                 // magic + RNE(x * rs)
    const unsigned long long d2 = f32x2_fma(x2, rs2, f32x2_sub(m2, t2));  // x * rs - RNE(x * rs)
    float t0, t1, d0, d1;
    f32x2_unpack(t2, t0, t1);
    f32x2_unpack(d2, d0, d1);
    rare = rare || !(fabsf(d0) <= 0.5f - kTieBand) || !(fabsf(d1) <= 0.5f - kTieBand);
    q[2 * k] = min(max((int)__float_as_uint(t0), kLo), kHi);
    q[2 * k + 1] = min(max((int)__float_as_uint(t1), kLo), kHi);
  }
  if (rare) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x = (e & 1) ? __uint_as_float(w[e >> 1] & 0xffff0000u) : __uint_as_float(w[e >> 1] << 16);
      const float t = fmaf(x, rs, kCodeMagic), r = t - kCodeMagic, d = fmaf(x, rs, -r);
      if (!exact || (!(fabsf(d) <= 0.5f - kTieBand) && !(fabsf(r) >= 128.0f)))
        q[e] = kCodeMagicBits + ((exact && fabsf(r) <= 127.0f) ? tie_code(x, s, rs) : quant_code(x, s));
    }
  }
}

// The eight codes as bytes, element e in byte e.
__device__ __forceinline__ uint2 quant_group8(uint4 v, float s, float rs, bool exact) {
  int q[8];
  quant_group8_biased(v, s, rs, exact, q);
  const uint32_t lo = __byte_perm(__byte_perm(q[0], q[1], 0x0040), __byte_perm(q[2], q[3], 0x0040), 0x5410);
  const uint32_t hi = __byte_perm(__byte_perm(q[4], q[5], 0x0040), __byte_perm(q[6], q[7], 0x0040), 0x5410);
  return make_uint2(lo, hi);
}

// Division of 32-bit unsigned integers by a divisor fixed for the launch, as a
// multiply-high and two shifts (Granlund and Montgomery, "Division by Invariant
// Integers using Multiplication", 1994, the unsigned N-bit method with l =
// ceil(log2 d)): exact for every 32-bit dividend.
struct DivU32 {
  uint32_t m, s1, s2;
};
inline DivU32 make_divu32(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  DivU32 f;
  f.m = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
  f.s1 = l < 1 ? l : 1;
  f.s2 = l > 0 ? l - 1 : 0;
  return f;
}
__device__ __forceinline__ uint32_t divu32(uint32_t n, DivU32 f) {
  const uint32_t t1 = __umulhi(f.m, n);
  return (t1 + ((n - t1) >> f.s1)) >> f.s2;
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
