// GQA decode attention over an INT8 KV cache with INT8 queries.
//
// MindIE "Attention Quantization", Overview, and MindIE Turbo "Attention量化":
// q, k and v are quantized to 8 bits per head and the decode-phase attention
// reads them directly; deq_scale restores floating point.  Scales are the
// per-head symmetric ones of msModelSlim "FA3量化" 原理 / 算法流程 step 4.
//
// The path is HBM-bound (about 16 operations per KV byte), so the design keeps
// every KV byte on its way from HBM to the tensor pipe in registers:
//   * grid = (split, kv head g, batch b); 4 warps per CTA, each warp walking
//     16-token steps of the CTA's token range with its own online softmax;
//   * scores  S^T[16 tok x 8 heads] = K[16 x 128] . Q^T  as m16n8k16 f16 MMAs:
//     int8 codes are exact in fp16 and 128-term sums of products < 2^24 are
//     exact in the fp32 accumulator, so the score is the exact integer dot;
//     the contraction order is permuted so that each thread converts 4
//     contiguous K bytes per k-step (Q is permuted the same way);
//   * P^T (fp16) comes from the score fragment by movmatrix.trans;
//   * O^T[128 x 8] += V^T . P^T, the 16 output dims of a thread contiguous so
//     every thread loads 16 contiguous V bytes per token;
//   * split-K partials (unnormalised O, running max m, sum l) are merged by a
//     small combine kernel with log-sum-exp weights.
#include "fa3_common.cuh"

#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>

namespace fa3 {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kHeadsPerTile = 8;

struct GqaArgs {
  const int8_t* q;
  const int8_t* k;
  const int8_t* v;
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  const int32_t* lens;
  __nv_bfloat16* out;
  float* part_o;    // [B][Hkv][splits][8][D]
  float2* part_ml;  // [B][Hkv][splits][8]
  int32_t* err;
  int B, Hq, Hkv, G, T_max, splits, chunk;
  float sm_log2;    // softmax_scale * log2(e)
};

// Four signed int8 codes -> two f16x2 (exact): bias to unsigned, place each
// byte under the f16 exponent of 1024, subtract 1024 + 128.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t x) {
  __half2 h = *reinterpret_cast<__half2*>(&x);
  return __half22float2(h);
}

__device__ __forceinline__ uint4 ldg_stream(const int8_t* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__global__ void __launch_bounds__(kThreads) gqa_decode_kernel(const GqaArgs p) {
  __shared__ float sm_o[kWarps][kHeadsPerTile][kD];
  __shared__ float sm_m[kWarps][kHeadsPerTile];
  __shared__ float sm_l[kWarps][kHeadsPerTile];

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, qd = lane & 3;
  const int G = p.G;

  int n = p.lens[b];
  if (n < 0 || n > p.T_max) {
    if (split == 0 && g == 0 && tid == 0) set_dev_err(p.err, FA3_DEVERR_LENS);
    n = 0;
  }
  const int t_begin = split * p.chunk;
  const int t_end = min(t_begin + p.chunk, n);

  // Q^T fragments of head r of this group, contraction order permuted so that
  // k-step s takes bytes [16qd + 4s, +4) (s < 4) or [64 + 16qd + 4(s-4), +4).
  uint32_t qb[8][2];
  {
    uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
    if (r < G) {
      const int8_t* qrow = p.q + ((int64_t)b * p.Hq + g * G + r) * kD;
      q0 = *reinterpret_cast<const uint4*>(qrow + 16 * qd);
      q1 = *reinterpret_cast<const uint4*>(qrow + 64 + 16 * qd);
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      i8x4_to_f16x4(word(q0, s), qb[s][0], qb[s][1]);
      i8x4_to_f16x4(word(q1, s), qb[s + 4][0], qb[s + 4][1]);
    }
  }
  const int h0 = 2 * qd, h1 = 2 * qd + 1;
  const float ks = p.k_scale[g] * p.sm_log2;
  const float c0s = h0 < G ? p.q_scale[g * G + h0] * ks : 0.f;
  const float c1s = h1 < G ? p.q_scale[g * G + h1] * ks : 0.f;

  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  const int64_t tok_stride = (int64_t)p.Hkv * kD;
  const int8_t* kbase = p.k + ((int64_t)b * p.T_max) * tok_stride + (int64_t)g * kD;
  const int8_t* vbase = p.v + ((int64_t)b * p.T_max) * tok_stride + (int64_t)g * kD;

  auto load_tile = [&](int t0, uint4 (&kr)[4], uint4 (&vr)[4]) {
    const uint4 z = make_uint4(0, 0, 0, 0);
    const int ta = t0 + r, tb = t0 + r + 8;
    kr[0] = ta < t_end ? ldg_stream(kbase + ta * tok_stride + 16 * qd) : z;
    kr[1] = ta < t_end ? ldg_stream(kbase + ta * tok_stride + 64 + 16 * qd) : z;
    kr[2] = tb < t_end ? ldg_stream(kbase + tb * tok_stride + 16 * qd) : z;
    kr[3] = tb < t_end ? ldg_stream(kbase + tb * tok_stride + 64 + 16 * qd) : z;
    const int tv[4] = {t0 + 2 * qd, t0 + 2 * qd + 1, t0 + 2 * qd + 8, t0 + 2 * qd + 9};
#pragma unroll
    for (int i = 0; i < 4; ++i) vr[i] = tv[i] < t_end ? ldg_stream(vbase + tv[i] * tok_stride + 16 * r) : z;
  };

  const int span = t_end - t_begin;
  const int n_tiles = span > 0 ? (span + 15) / 16 : 0;
  uint4 kr[4], vr[4];
  if (warp < n_tiles) load_tile(t_begin + 16 * warp, kr, vr);
  for (int it = warp; it < n_tiles; it += kWarps) {
    const int t0 = t_begin + 16 * it;
    uint4 nkr[4], nvr[4];
    if (it + kWarps < n_tiles) load_tile(t0 + 16 * kWarps, nkr, nvr);

    // ---- scores S^T = K . Q^T (exact integer dot products in fp32)
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      uint32_t a0, a1, a2, a3;
      i8x4_to_f16x4(word(kr[s < 4 ? 0 : 1], s & 3), a0, a2);
      i8x4_to_f16x4(word(kr[s < 4 ? 2 : 3], s & 3), a1, a3);
      mma16816(c, a0, a1, a2, a3, qb[s][0], qb[s][1]);
    }
    const bool va = t0 + r < t_end, vb = t0 + r + 8 < t_end;
    float x0 = va ? c[0] * c0s : -CUDART_INF_F;
    float x1 = va ? c[1] * c1s : -CUDART_INF_F;
    float x2 = vb ? c[2] * c0s : -CUDART_INF_F;
    float x3 = vb ? c[3] * c1s : -CUDART_INF_F;

    // ---- online softmax (log2 domain); rows of a head live in the 8 lanes sharing qd
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int o_ = 4; o_ < 32; o_ <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o_));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o_));
    }
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float ref0 = mn0 == -CUDART_INF_F ? 0.f : mn0;
    const float ref1 = mn1 == -CUDART_INF_F ? 0.f : mn1;
    const float al0 = exp2f(m0 - ref0), al1 = exp2f(m1 - ref1);
    m0 = mn0;
    m1 = mn1;
    const uint32_t X = pack_f16x2(exp2f(x0 - ref0), exp2f(x1 - ref1));   // token r
    const uint32_t Y = pack_f16x2(exp2f(x2 - ref0), exp2f(x3 - ref1));   // token r + 8
    const float2 fx = unpack_f16x2(X), fy = unpack_f16x2(Y);
    l0 = l0 * al0 + (fx.x + fy.x);
    l1 = l1 * al1 + (fx.y + fy.y);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[i][0] *= al0; o[i][1] *= al1; o[i][2] *= al0; o[i][3] *= al1;
    }
    const uint32_t b0 = movmatrix_trans(X), b1 = movmatrix_trans(Y);

    // ---- O^T += V^T . P^T; m-tile i covers dims 16r + 2i (row r) and 16r + 2i + 1 (row r + 8)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
      const uint32_t p01 = __byte_perm(word(vr[0], i >> 1), word(vr[1], i >> 1), sel);
      const uint32_t p23 = __byte_perm(word(vr[2], i >> 1), word(vr[3], i >> 1), sel);
      uint32_t a0, a1, a2, a3;
      i8x4_to_f16x4(p01, a0, a1);
      i8x4_to_f16x4(p23, a2, a3);
      mma16816(o[i], a0, a1, a2, a3, b0, b1);
    }
    if (it + kWarps < n_tiles) {
#pragma unroll
      for (int i = 0; i < 4; ++i) { kr[i] = nkr[i]; vr[i] = nvr[i]; }
    }
  }

  // ---- merge the 4 warps of the CTA
#pragma unroll
  for (int o_ = 4; o_ < 32; o_ <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
    l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
  }
  if (r == 0) {
    sm_m[warp][h0] = m0; sm_m[warp][h1] = m1;
    sm_l[warp][h0] = l0; sm_l[warp][h1] = l1;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    sm_o[warp][h0][16 * r + 2 * i] = o[i][0];
    sm_o[warp][h1][16 * r + 2 * i] = o[i][1];
    sm_o[warp][h0][16 * r + 2 * i + 1] = o[i][2];
    sm_o[warp][h1][16 * r + 2 * i + 1] = o[i][3];
  }
  __syncthreads();
  const int d = tid;  // one output dim per thread
  for (int hh = 0; hh < G; ++hh) {
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][hh]);
    float L = 0.f, O = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float f = exp2f(sm_m[w][hh] - M);
        L += sm_l[w][hh] * f;
        O += sm_o[w][hh][d] * f;
      }
    }
    if (p.splits == 1) {
      const float val = L > 0.f ? p.v_scale[g] * (O / L) : 0.f;
      p.out[((int64_t)b * p.Hq + g * G + hh) * kD + d] = __float2bfloat16_rn(val);
    } else {
      const int64_t slot = (((int64_t)b * p.Hkv + g) * p.splits + split) * kHeadsPerTile + hh;
      p.part_o[slot * kD + d] = O;
      if (d == 0) p.part_ml[slot] = make_float2(M, L);
    }
  }
}

__global__ void __launch_bounds__(kD) gqa_combine_kernel(const GqaArgs p) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  const int g = h / p.G, hh = h - g * p.G;
  const int64_t slot0 = (((int64_t)b * p.Hkv + g) * p.splits) * kHeadsPerTile + hh;
  float M = -CUDART_INF_F;
  for (int s = 0; s < p.splits; ++s) {
    const float2 ml = p.part_ml[slot0 + (int64_t)s * kHeadsPerTile];
    if (ml.y > 0.f) M = fmaxf(M, ml.x);
  }
  float L = 0.f, O = 0.f;
  if (M != -CUDART_INF_F) {
    for (int s = 0; s < p.splits; ++s) {
      const int64_t slot = slot0 + (int64_t)s * kHeadsPerTile;
      const float2 ml = p.part_ml[slot];
      if (ml.y > 0.f) {
        const float f = exp2f(ml.x - M);
        L += ml.y * f;
        O += p.part_o[slot * kD + d] * f;
      }
    }
  }
  const float val = L > 0.f ? p.v_scale[g] * (O / L) : 0.f;
  p.out[((int64_t)b * p.Hq + h) * kD + d] = __float2bfloat16_rn(val);
}

int gqa_blocks_per_sm();

// Split-K plan: the (split, KV head, sequence) grid is sized to a whole number of
// waves of resident CTAs, with chunks of at least 64 tokens.
void gqa_plan(int B, int Hkv, int T_max, int num_sms, int* splits, int* chunk) {
  const int64_t units = (int64_t)B * Hkv;
  const int64_t wave = (int64_t)num_sms * gqa_blocks_per_sm();
  int best_s = 1;
  double best_cost = 1e30;
  const int max_s = (int)std::max<int64_t>(1, (T_max + 63) / 64);
  for (int sp = 1; sp <= max_s && sp <= 64; ++sp) {
    const int64_t ctas = units * sp;
    const int64_t waves = (ctas + wave - 1) / wave;
    const int64_t per = ((int64_t)T_max + sp - 1) / sp;
    // time ~ waves x tokens per CTA, plus a fixed per-CTA cost worth ~32 tokens
    const double cost = (double)waves * (double)(per + 32);
    if (cost < best_cost - 1e-9) { best_cost = cost; best_s = sp; }
  }
  int64_t per = ((int64_t)T_max + best_s - 1) / best_s;
  per = ((per + 15) / 16) * 16;
  *chunk = (int)per;
  *splits = (int)((T_max + per - 1) / per);
}

int gqa_blocks_per_sm() {
  static int cached = 0;
  if (cached <= 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_decode_kernel, kThreads, 0) != cudaSuccess || n <= 0)
      n = 3;
    cached = n;
  }
  return cached;
}

}  // namespace
}  // namespace fa3

using namespace fa3;

FA3_API size_t fa3_gqa_workspace_size(int B, int Hq, int Hkv, int D, int T_max) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D != kD || T_max <= 0) return 0;
  int sms = 0;
  if (check_device(&sms) != FA3_OK) sms = 148;
  int splits, chunk;
  gqa_plan(B, Hkv, T_max, sms, &splits, &chunk);
  if (splits == 1) return 0;
  const size_t slots = (size_t)B * Hkv * splits * kHeadsPerTile;
  return slots * kD * sizeof(float) + slots * sizeof(float2) + 256;
}

FA3_API int fa3_decode_attn_gqa(const int8_t* q, const int8_t* k, const int8_t* v, const float* q_scale,
                                const float* k_scale, const float* v_scale, const int32_t* lens, uint16_t* out,
                                int B, int Hq, int Hkv, int D, int T_max, float softmax_scale, void* workspace,
                                size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (!q || !k || !v || !q_scale || !k_scale || !v_scale || !lens || !out) return FA3_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || T_max <= 0) return FA3_EINVAL;
  if (Hq % Hkv != 0) return FA3_EINVAL;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return FA3_EINVAL;
  const int G = Hq / Hkv;
  if (D != kD || G > kHeadsPerTile || B > 65535 || Hkv > 65535) return FA3_ERANGE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return FA3_ERANGE;
  int sms = 0;
  int st = check_device(&sms);
  if (st != FA3_OK) return st;
  int splits, chunk;
  gqa_plan(B, Hkv, T_max, sms, &splits, &chunk);
  const size_t need = fa3_gqa_workspace_size(B, Hq, Hkv, D, T_max);
  if (need && (!workspace || workspace_bytes < need || !aligned16(workspace))) return FA3_EWORKSPACE;
  GqaArgs a;
  a.q = q; a.k = k; a.v = v; a.q_scale = q_scale; a.k_scale = k_scale; a.v_scale = v_scale; a.lens = lens;
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  const size_t slots = (size_t)B * Hkv * splits * kHeadsPerTile;
  a.part_o = static_cast<float*>(workspace);
  a.part_ml = need ? reinterpret_cast<float2*>(static_cast<char*>(workspace) + slots * kD * sizeof(float)) : nullptr;
  a.err = dev_err;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = G; a.T_max = T_max; a.splits = splits; a.chunk = chunk;
  a.sm_log2 = softmax_scale * 1.4426950408889634f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  timing_begin(s);
  gqa_decode_kernel<<<dim3(splits, Hkv, B), kThreads, 0, s>>>(a);
  timing_end(s);
  if (cudaGetLastError() != cudaSuccess) return FA3_ECUDA;
  if (splits > 1) {
    gqa_combine_kernel<<<dim3(Hq, B), kD, 0, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return FA3_ECUDA;
  }
  return FA3_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of fa3_decode_attn_gqa.
//
// Some callers cannot call cudaMalloc at the point where they run decode
// attention: code inside a custom allocator or memory-pool callback, runtimes
// that pre-plan every device allocation up front, and embedded or safety-
// certified deployments that forbid allocation after start-up.  For them the
// split-K partials live in a fixed array in the library's own device memory.
// Every GPU that loads libfa3.so holds this array (kGqaStaticScratchBytes)
// until the process exits.
namespace fa3 {
namespace {
constexpr size_t kGqaStaticScratchBytes = size_t(8) << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_gqa_static_scratch[kGqaStaticScratchBytes];

// Device address of the array, looked up once per device.  In host code the
// array's name is only a host-side stand-in, never a device address.
void* g_gqa_static_scratch_addr[64] = {nullptr};
}  // namespace
}  // namespace fa3

FA3_API int fa3_decode_attn_gqa_noalloc(const int8_t* q, const int8_t* k, const int8_t* v, const float* q_scale,
                                        const float* k_scale, const float* v_scale, const int32_t* lens,
                                        uint16_t* out, int B, int Hq, int Hkv, int D, int T_max,
                                        float softmax_scale, int32_t* dev_err, void* stream) {
  if (!q || !k || !v || !q_scale || !k_scale || !v_scale || !lens || !out) return FA3_EINVAL;
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || T_max <= 0) return FA3_EINVAL;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FA3_ECUDA;
  const size_t need = fa3_gqa_workspace_size(B, Hq, Hkv, D, T_max);
  if (need > kGqaStaticScratchBytes) return FA3_EWORKSPACE;   // beyond the fixed 8 MiB scratch
  if (g_gqa_static_scratch_addr[dev] == nullptr) {
    // Set-up, once per device, with that device current.
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_gqa_static_scratch) != cudaSuccess || ptr == nullptr) return FA3_ECUDA;
    g_gqa_static_scratch_addr[dev] = ptr;
  }
  // Every slot of the partials is written before it is read, so nothing needs clearing.
  return fa3_decode_attn_gqa(q, k, v, q_scale, k_scale, v_scale, lens, out, B, Hq, Hkv, D, T_max, softmax_scale,
                             g_gqa_static_scratch_addr[dev], kGqaStaticScratchBytes, dev_err, stream);
}
