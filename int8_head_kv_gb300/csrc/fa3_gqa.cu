// GQA decode attention over an INT8 KV cache with INT8 queries.
//
// MindIE "Attention Quantization", Overview, and MindIE Turbo "Attention量化":
// q, k and v are quantized to 8 bits per head and the decode-phase attention
// reads them directly; deq_scale restores floating point.  Scales are the
// per-head symmetric ones of msModelSlim "FA3量化" 原理 / 算法流程 step 4.
//
// The path is HBM-bound (about 16 operations per KV byte):
//   * grid = (split, kv head g, batch b); 4 warps per CTA, each warp walking
//     16-token steps of the CTA's token range with its own online softmax;
//   * each warp streams its steps through a 2-stage cp.async ring in shared
//     memory (K then V rows, 16-byte chunks swizzled so that the fragment loads
//     are free of bank conflicts);
//   * scores  S^T[16 tok x 8 heads] = K[16 x 128] . Q^T  as exact integer
//     m16n8k32 s8 MMAs (s32 accumulate); the contraction order is permuted so
//     that each thread's K and Q words are the bytes it already holds;
//   * P^T (fp16) comes from the score fragment by movmatrix.trans;
//   * O^T[128 x 8] += V^T . P^T as m16n8k16 f16 MMAs; V enters as code + 1152
//     (two byte permutes per four codes, no subtraction), and the bias times the
//     row sum of P is taken off once at the end;
//   * split-K partials (unnormalised O, running max m, sum l) are merged by a
//     small combine kernel with log-sum-exp weights.
#include "fa3_common.cuh"

#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <atomic>

namespace fa3 {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kHeadsPerTile = 8;
#ifndef FA3_GQA_STAGES
#define FA3_GQA_STAGES 2
#endif
// cp.async ring depth per warp: with the one-wave split plan (long chunks), two
// stages and more resident CTAs beat deeper rings (measured 29.8 / 30.3 / 31.2 /
// 32.7 us for 2 / 3 / 4 / 5 stages on the Llama-70B shape).
constexpr int kStages = FA3_GQA_STAGES;
constexpr int kStageBytes = 2 * 16 * kD;        // one 16-token step: K then V rows (4 KB)
constexpr int kSmemBytes = kWarps * kStages * kStageBytes;

struct GqaArgs {
  const int8_t* q;
  const int8_t* k;       // [B][T_max][Hkv][D], or a [pool rows][Hkv][D] page pool
  const int8_t* v;
  const int32_t* block_table;   // [B][max_pages] pool pages, or nullptr for the contiguous layout
  const float* q_scale;   // [Hq], or [Hq][D] per channel
  const float* k_scale;   // [Hkv], or [Hkv][D]
  const float* v_scale;   // [Hkv], or [Hkv][D]
  const float* q_off;     // per channel only: [Hq][D] offsets of q and v (k's cancel in the softmax)
  const float* v_off;
  const int32_t* lens;
  __nv_bfloat16* out;
  float* part_o;    // [B][Hkv][splits][8][D]
  float2* part_ml;  // [B][Hkv][splits][8]
  int32_t* err;
  int B, Hq, Hkv, G, T_max, splits, chunk;
  int page_size, max_pages, num_pages;
  DivU32 div_ps;    // / page_size
  float sm_log2;    // softmax_scale * log2(e)
};

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four signed int8 codes -> two f16x2 holding code + 1152 (exact): the bias to
// unsigned and the f16 exponent of 1024 without the subtraction.  P.V on these
// values is P.V + 1152 * sum(P), and sum(P) is the row sum l that the softmax keeps
// from the same fp16 P values, so the output is v_scale * (O / l - 1152).
constexpr float kVBias = 1152.f;
__device__ __forceinline__ void i8x4_to_f16x4_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
}

// Four signed int8 codes -> two f16x2 holding the codes themselves (exact).
__device__ __forceinline__ void i8x4_to_f16x4_exact(uint32_t w, uint32_t& lo, uint32_t& hi) {
  i8x4_to_f16x4_biased(w, lo, hi);
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));    // - (1024 + 128)
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

// Exact integer m16n8k32 MMA on int8 codes (s32 accumulate).
__device__ __forceinline__ void mma16832_s8(int (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// CHANNEL: per-channel asymmetric q, k, v (MindIE Turbo "Attention量化", 表1 / 表2:
// [heads][D] scales and offsets).  The score of key j is
//   sum_d (q8[d] - qo[d]) qs[d] * (k8_j[d] - ko[d]) ks[d]
//     = sum_d w[d] k8_j[d] - sum_d w[d] ko[d],   w[d] = (q8[d] - qo[d]) qs[d] ks[d],
// and the second term is the same for every key, so the softmax drops it: the
// scores are K codes times the real vector w, taken as fp16 hi + lo parts (w
// scaled per head by a power of two into fp16's range; the factor returns with
// the softmax scale) in two f16 MMAs per 16 dims.  V: out[d] = vs[d] * (O[d] / l - vo[d]).
template <bool PAGED, bool CHANNEL>
__global__ void __launch_bounds__(kThreads) gqa_decode_kernel(const GqaArgs p) {
  pdl_wait();
  pdl_launch_dependents();
  // Per-warp rings of 16-token K/V steps.  A 128-byte row stores its 16-byte
  // chunk c at position c ^ f(row & 7), f(r) = (r & 6) ^ 4 (r & 1): every 8-lane
  // phase of the K and V fragment loads below then touches 8 distinct 16-byte
  // bank groups.  After the token loop the same memory holds the warps' partial O.
  extern __shared__ __align__(128) uint8_t gsm[];
  float (*sm_o)[kHeadsPerTile][kD] = reinterpret_cast<float (*)[kHeadsPerTile][kD]>(gsm);
  __shared__ float sm_m[kWarps][kHeadsPerTile];
  __shared__ float sm_l[kWarps][kHeadsPerTile];
  static_assert(kWarps * kHeadsPerTile * kD * 4 <= kSmemBytes, "partial O fits in the rings");

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

  // Q^T fragments of head r of this group as int8 words, contraction order
  // permuted: thread (r, qd) holds row bytes [16qd, +16) as words 0-3 and
  // [64 + 16qd, +16) as words 4-7; k32-step s takes words 2s and 2s + 1 of Q
  // (B operand) and of its K rows r and r + 8 (A operand) alike.
  uint32_t qw[8];
  {
    uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
    if (r < G) {
      const int8_t* qrow = p.q + ((int64_t)b * p.Hq + g * G + r) * kD;
      q0 = *reinterpret_cast<const uint4*>(qrow + 16 * qd);
      q1 = *reinterpret_cast<const uint4*>(qrow + 64 + 16 * qd);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      qw[j] = word(q0, j);
      qw[4 + j] = word(q1, j);
    }
  }
  const int h0 = 2 * qd, h1 = 2 * qd + 1;
  float c0s, c1s;
  // per channel: the B fragments of w (hi, lo) for the 8 k16 steps; step s takes
  // dims base(s) + 0..3, base(s) = 4s within the first 16-byte chunk of this
  // thread (s < 4), then within its second chunk
  uint32_t wh[8][2], wl[8][2];
  if (!CHANNEL) {
    const float ks = p.k_scale[g] * p.sm_log2;
    c0s = h0 < G ? p.q_scale[g * G + h0] * ks : 0.f;
    c1s = h1 < G ? p.q_scale[g * G + h1] * ks : 0.f;
  } else {
    float wv[32];
    float amax = 0.f;
    const int hq = g * G + r;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int d = (j < 16 ? 16 * qd : 64 + 16 * qd) + (j & 15);
      const int code = (int)(int8_t)((qw[j >> 2] >> (8 * (j & 3))) & 0xffu);
      float wj = 0.f;
      if (r < G)
        wj = ((float)code - p.q_off[(int64_t)hq * kD + d]) * p.q_scale[(int64_t)hq * kD + d] *
             p.k_scale[(int64_t)g * kD + d];
      wv[j] = wj;
      amax = fmaxf(amax, fabsf(wj));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    // power-of-two factor putting the head's largest |w| into [2^13, 2^14)
    int e = 0;
    if (amax > 0.f) (void)frexpf(amax, &e);
    const float down = amax > 0.f ? ldexpf(1.f, 14 - e) : 1.f;
#pragma unroll
    for (int s_ = 0; s_ < 8; ++s_) {
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {
        const int j = 4 * s_ + 2 * hlf;
        const float a = wv[j] * down, b2 = wv[j + 1] * down;
        const __half ah = __float2half_rn(a), bh = __float2half_rn(b2);
        const __half al = __float2half_rn(a - __half2float(ah)), bl = __float2half_rn(b2 - __half2float(bh));
        wh[s_][hlf] = (uint32_t)__half_as_ushort(ah) | ((uint32_t)__half_as_ushort(bh) << 16);
        wl[s_][hlf] = (uint32_t)__half_as_ushort(al) | ((uint32_t)__half_as_ushort(bl) << 16);
      }
    }
    const float up = 1.f / down;                       // exact: a power of two
    const float up0 = __shfl_sync(0xffffffffu, up, 4 * h0);
    const float up1 = __shfl_sync(0xffffffffu, up, 4 * h1);
    c0s = h0 < G ? up0 * p.sm_log2 : 0.f;
    c1s = h1 < G ? up1 * p.sm_log2 : 0.f;
  }

  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  const int64_t tok_stride = (int64_t)p.Hkv * kD;
  const int64_t seq_row0 = PAGED ? 0 : (int64_t)b * p.T_max;             // cache row of the sequence's token 0
  const int8_t* kbase = p.k + seq_row0 * tok_stride + (int64_t)g * kD;
  const int8_t* vbase = p.v + seq_row0 * tok_stride + (int64_t)g * kD;

  const uint32_t ring = (uint32_t)__cvta_generic_to_shared(gsm) + (uint32_t)(warp * kStages * kStageBytes);
  auto swz = [](int row) { return (row & 6) ^ ((row & 1) << 2); };
  // Step it of the CTA's range (16 tokens) -> ring stage: 256 chunks of 16 bytes,
  // 8 per lane; rows past the range are zero-filled (their scores are masked).
  // Paged: chunks start at multiples of 16 tokens and pages hold multiples of 16, so
  // a step's 16 rows lie in one page; a block-table entry outside the pool reads zeros.
  // The entry of a step is loaded one issue ahead (entry_of) and used at the next
  // issue (row_of), so that the load's latency is not spent waiting.
  auto entry_of = [&](int t0) -> int {
    return p.block_table[(int64_t)b * p.max_pages + divu32((uint32_t)t0, p.div_ps)];
  };
  auto row_of = [&](int pg, int t0) -> int64_t {     // pool row of token t0 (-1: entry outside the pool)
    const int off = t0 - (int)divu32((uint32_t)t0, p.div_ps) * p.page_size;
    return (pg >= 0 && pg < p.num_pages) ? (int64_t)pg * p.page_size + off : -1;
  };
  const int span = t_end - t_begin;
  const int n_tiles = span > 0 ? (span + 15) / 16 : 0;
  const int n_my = warp < n_tiles ? (n_tiles - warp + kWarps - 1) / kWarps : 0;   // steps warp, warp+4, ...
  // Steps are issued in order m = 0, 1, ...
  int pg_next = (PAGED && n_my > 0) ? entry_of(t_begin + 16 * warp) : 0;
  auto issue = [&](int m, int stage) {
    const int t0 = t_begin + 16 * (warp + kWarps * m);
    int64_t r0 = t0;                                  // row of token t0 from the bases
    if (PAGED) {
      r0 = row_of(pg_next, t0);
      if (m + 1 < n_my) pg_next = entry_of(t0 + 16 * kWarps);
      if (r0 < 0 && lane == 0) set_dev_err(p.err, FA3_DEVERR_PAGE);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = lane + 32 * k, kv = i >> 7, row = (i >> 3) & 15, col = i & 7;
      const bool ok = t0 + row < t_end && r0 >= 0;
      const int8_t* src = (kv ? vbase : kbase) + (ok ? r0 + row : 0) * tok_stride + col * 16;
      cp_async16(ring + stage * kStageBytes + kv * 2048 + row * 128 + ((col ^ swz(row)) << 4), src, ok ? 16u : 0u);
    }
  };
  auto chunk_addr = [&](uint32_t base, int row, int col) { return base + row * 128 + ((col ^ swz(row)) << 4); };

#pragma unroll
  for (int m = 0; m < kStages - 1; ++m) {
    if (m < n_my) issue(m, m);
    cp_async_commit();
  }
  for (int m = 0; m < n_my; ++m) {
    const int it = warp + kWarps * m;
    const int t0 = t_begin + 16 * it;
    if (m + kStages - 1 < n_my) issue(m + kStages - 1, (m + kStages - 1) % kStages);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const uint32_t kst = ring + (m % kStages) * kStageBytes, vst = kst + 2048;
    uint4 kr[4], vr[4];
    kr[0] = lds128(chunk_addr(kst, r, qd));
    kr[1] = lds128(chunk_addr(kst, r, 4 + qd));
    kr[2] = lds128(chunk_addr(kst, r + 8, qd));
    kr[3] = lds128(chunk_addr(kst, r + 8, 4 + qd));
    vr[0] = lds128(chunk_addr(vst, 2 * qd, r));
    vr[1] = lds128(chunk_addr(vst, 2 * qd + 1, r));
    vr[2] = lds128(chunk_addr(vst, 2 * qd + 8, r));
    vr[3] = lds128(chunk_addr(vst, 2 * qd + 9, r));
    __syncwarp();   // every lane has its fragments: the stage may be refilled
    float cf[4];
    if (!CHANNEL) {
      // ---- scores S^T = K . Q^T: exact integer dot products (int8 MMA, s32)
      int c[4] = {0, 0, 0, 0};
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint4& ka = kr[s < 2 ? 0 : 1];
        const uint4& kb = kr[s < 2 ? 2 : 3];
        const int w0 = (2 * s) & 3, w1 = (2 * s + 1) & 3;
        mma16832_s8(c, word(ka, w0), word(kb, w0), word(ka, w1), word(kb, w1), qw[2 * s], qw[2 * s + 1]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) cf[e] = (float)c[e];
    } else {
      // ---- scores S^T = K . w (fp16 codes x fp16 hi + lo parts, fp32 accumulate)
      cf[0] = cf[1] = cf[2] = cf[3] = 0.f;
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        uint32_t a0, a1, a2, a3;
        i8x4_to_f16x4_exact(word(kr[s >> 2], s & 3), a0, a2);          // row r:     dims base(s) + 0..3
        i8x4_to_f16x4_exact(word(kr[2 + (s >> 2)], s & 3), a1, a3);    // row r + 8
        mma16816(cf, a0, a1, a2, a3, wh[s][0], wh[s][1]);
        mma16816(cf, a0, a1, a2, a3, wl[s][0], wl[s][1]);
      }
    }
    const bool va = t0 + r < t_end, vb = t0 + r + 8 < t_end;
    float x0 = va ? cf[0] * c0s : -CUDART_INF_F;
    float x1 = va ? cf[1] * c1s : -CUDART_INF_F;
    float x2 = vb ? cf[2] * c0s : -CUDART_INF_F;
    float x3 = vb ? cf[3] * c1s : -CUDART_INF_F;

    // ---- online softmax (log2 domain); rows of a head live in the 8 lanes sharing qd
    float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
    for (int o_ = 4; o_ < 32; o_ <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o_));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o_));
    }
    // Lazy reference: m moves only when a head's maximum grows by more than 8 (so P
    // stays below 2^8 in fp16), and only then are O and l rescaled.
    const bool g0 = mx0 > m0 + 8.f, g1 = mx1 > m1 + 8.f;
    if (__any_sync(0xffffffffu, g0 || g1)) {
      const float n0 = g0 ? mx0 : m0, n1 = g1 ? mx1 : m1;
      const float al0 = g0 ? (m0 == -CUDART_INF_F ? 0.f : ex2_approx(m0 - n0)) : 1.f;
      const float al1 = g1 ? (m1 == -CUDART_INF_F ? 0.f : ex2_approx(m1 - n1)) : 1.f;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        o[i][0] *= al0; o[i][1] *= al1; o[i][2] *= al0; o[i][3] *= al1;
      }
      m0 = n0;
      m1 = n1;
    }
    const float ref0 = m0 == -CUDART_INF_F ? 0.f : m0;
    const float ref1 = m1 == -CUDART_INF_F ? 0.f : m1;
    const uint32_t X = pack_f16x2(ex2_approx(x0 - ref0), ex2_approx(x1 - ref1));   // token r
    const uint32_t Y = pack_f16x2(ex2_approx(x2 - ref0), ex2_approx(x3 - ref1));   // token r + 8
    const float2 fx = unpack_f16x2(X), fy = unpack_f16x2(Y);
    l0 += fx.x + fy.x;
    l1 += fx.y + fy.y;
    const uint32_t b0 = movmatrix_trans(X), b1 = movmatrix_trans(Y);

    // ---- O^T += V^T . P^T; m-tile i covers dims 16r + 2i (row r) and 16r + 2i + 1 (row r + 8)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
      const uint32_t p01 = __byte_perm(word(vr[0], i >> 1), word(vr[1], i >> 1), sel);
      const uint32_t p23 = __byte_perm(word(vr[2], i >> 1), word(vr[3], i >> 1), sel);
      uint32_t a0, a1, a2, a3;
      i8x4_to_f16x4_biased(p01, a0, a1);
      i8x4_to_f16x4_biased(p23, a2, a3);
      mma16816(o[i], a0, a1, a2, a3, b0, b1);
    }
  }
  cp_async_wait<0>();

  // ---- merge the 4 warps of the CTA (the rings become the partial-O buffer)
  __syncthreads();
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
      float val = 0.f;
      if (L > 0.f)
        val = CHANNEL ? p.v_scale[(int64_t)g * kD + d] * (O / L - kVBias - p.v_off[(int64_t)g * kD + d])
                      : p.v_scale[g] * (O / L - kVBias);
      p.out[((int64_t)b * p.Hq + g * G + hh) * kD + d] = __float2bfloat16_rn(val);
    } else {
      const int64_t slot = (((int64_t)b * p.Hkv + g) * p.splits + split) * kHeadsPerTile + hh;
      p.part_o[slot * kD + d] = O;
      if (d == 0) p.part_ml[slot] = make_float2(M, L);
    }
  }
}

template <bool CHANNEL>
__global__ void __launch_bounds__(kD) gqa_combine_kernel(const GqaArgs p) {
  pdl_wait();
  pdl_launch_dependents();
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
  float val = 0.f;
  if (L > 0.f)
    val = CHANNEL ? p.v_scale[(int64_t)g * kD + d] * (O / L - kVBias - p.v_off[(int64_t)g * kD + d])
                  : p.v_scale[g] * (O / L - kVBias);
  p.out[((int64_t)b * p.Hq + h) * kD + d] = __float2bfloat16_rn(val);
}

int gqa_blocks_per_sm();

// Split-K plan: as many splits as keep the (split, KV head, sequence) grid within
// one wave of resident CTAs (at least one split, chunks of at least 64 tokens).
// Measured on the Llama-70B shape (128 units, 456 resident CTAs): 3 splits
// (384 CTAs, one wave) 31.5 us, 4 splits (512 CTAs, a second partial wave)
// 37.6 us, 7 splits (896 CTAs, two full waves) 34.5 us: each CTA's prologue and
// merge are worth far more than a few tokens, so a single wave of longer chunks wins.
void gqa_plan(int B, int Hkv, int T_max, int num_sms, int* splits, int* chunk) {
  const int64_t units = (int64_t)B * Hkv;
  const int64_t wave = (int64_t)num_sms * gqa_blocks_per_sm();
  const int64_t max_s = std::max<int64_t>(1, std::min<int64_t>(64, (T_max + 63) / 64));
  const int64_t sp = std::max<int64_t>(1, std::min<int64_t>(max_s, wave / units));
  int64_t per = ((int64_t)T_max + sp - 1) / sp;
  per = ((per + 15) / 16) * 16;
  *chunk = (int)per;
  *splits = (int)((T_max + per - 1) / per);
}

int gqa_blocks_per_sm() {
  static int cached = 0;
  if (cached <= 0) {
    int n = 0;
    if (cudaFuncSetAttribute(gqa_decode_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_decode_kernel<false, false>, kThreads, kSmemBytes) !=
            cudaSuccess ||
        n <= 0)
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

namespace {
// Both layouts: block_table == nullptr is the contiguous [B][T_max] cache; otherwise
// k / v are pools of num_pages pages of page_size rows and T_max = max_pages * page_size.
int gqa_decode(const int8_t* q, const int8_t* k, const int8_t* v, const float* q_scale, const float* k_scale,
               const float* v_scale, const int32_t* lens, const int32_t* block_table, uint16_t* out, int B, int Hq,
               int Hkv, int D, int T_max, int num_pages, int page_size, int max_pages, float softmax_scale,
               void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream,
               const float* q_off = nullptr, const float* v_off = nullptr) {
  const bool channel = q_off != nullptr;
  if (!q || !k || !v || !q_scale || !k_scale || !v_scale || !lens || !out) return FA3_EINVAL;
  if (channel && (!v_off || block_table)) return FA3_EINVAL;
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
  a.q_off = q_off; a.v_off = v_off;
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  const size_t slots = (size_t)B * Hkv * splits * kHeadsPerTile;
  a.part_o = static_cast<float*>(workspace);
  a.part_ml = need ? reinterpret_cast<float2*>(static_cast<char*>(workspace) + slots * kD * sizeof(float)) : nullptr;
  a.err = dev_err;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = G; a.T_max = T_max; a.splits = splits; a.chunk = chunk;
  a.block_table = block_table; a.page_size = page_size; a.max_pages = max_pages; a.num_pages = num_pages;
  a.div_ps = make_divu32((uint32_t)(page_size > 0 ? page_size : 1));
  a.sm_log2 = softmax_scale * 1.4426950408889634f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* kernel = channel ? gqa_decode_kernel<false, true>
                         : block_table ? gqa_decode_kernel<true, false> : gqa_decode_kernel<false, false>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
    return FA3_ECUDA;
  timing_begin(s);
  const cudaError_t le = launch_pdl(kernel, dim3(splits, Hkv, B), dim3(kThreads), kSmemBytes, s, a);
  timing_end(s);
  if (le != cudaSuccess) return FA3_ECUDA;
  if (splits > 1 && launch_pdl(channel ? gqa_combine_kernel<true> : gqa_combine_kernel<false>, dim3(Hq, B),
                              dim3(kD), 0, s, a) != cudaSuccess)
    return FA3_ECUDA;
  return FA3_OK;
}
}  // namespace

FA3_API int fa3_decode_attn_gqa(const int8_t* q, const int8_t* k, const int8_t* v, const float* q_scale,
                                const float* k_scale, const float* v_scale, const int32_t* lens, uint16_t* out,
                                int B, int Hq, int Hkv, int D, int T_max, float softmax_scale, void* workspace,
                                size_t workspace_bytes, int32_t* dev_err, void* stream) {
  return gqa_decode(q, k, v, q_scale, k_scale, v_scale, lens, nullptr, out, B, Hq, Hkv, D, T_max, 0, 0, 0,
                    softmax_scale, workspace, workspace_bytes, dev_err, stream);
}

FA3_API int fa3_decode_attn_gqa_channel(const int8_t* q, const int8_t* k, const int8_t* v, const float* q_scale,
                                        const float* q_offset, const float* k_scale, const float* k_offset,
                                        const float* v_scale, const float* v_offset, const int32_t* lens,
                                        uint16_t* out, int B, int Hq, int Hkv, int D, int T_max, float softmax_scale,
                                        void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream) {
  // k_offset shifts every score of a row by the same amount, which the softmax
  // removes; it is part of the signature (the pages' tensor set) and not read.
  if (!q_offset || !k_offset || !v_offset) return FA3_EINVAL;
  return gqa_decode(q, k, v, q_scale, k_scale, v_scale, lens, nullptr, out, B, Hq, Hkv, D, T_max, 0, 0, 0,
                    softmax_scale, workspace, workspace_bytes, dev_err, stream, q_offset, v_offset);
}

FA3_API int fa3_decode_attn_gqa_paged(const int8_t* q, const int8_t* k, const int8_t* v, const float* q_scale,
                                      const float* k_scale, const float* v_scale, const int32_t* lens,
                                      const int32_t* block_table, uint16_t* out, int B, int Hq, int Hkv, int D,
                                      int num_pages, int page_size, int max_pages, float softmax_scale,
                                      void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (!block_table) return FA3_EINVAL;
  if (num_pages <= 0 || page_size <= 0 || max_pages <= 0) return FA3_EINVAL;
  if (page_size % 16 != 0 || (int64_t)max_pages * page_size >= ((int64_t)1 << 31)) return FA3_ERANGE;
  return gqa_decode(q, k, v, q_scale, k_scale, v_scale, lens, block_table, out, B, Hq, Hkv, D,
                    max_pages * page_size, num_pages, page_size, max_pages, softmax_scale, workspace,
                    workspace_bytes, dev_err, stream);
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
// array's name is only a host-side stand-in, never a device address.  Atomic
// slots: two host threads making their first call at once may both look the
// address up, and both store the same value.
std::atomic<void*> g_gqa_static_scratch_addr[64];
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
  void* scratch = g_gqa_static_scratch_addr[dev].load(std::memory_order_acquire);
  if (scratch == nullptr) {
    // Set-up, once per device, with that device current.
    if (cudaGetSymbolAddress(&scratch, g_gqa_static_scratch) != cudaSuccess || scratch == nullptr) return FA3_ECUDA;
    g_gqa_static_scratch_addr[dev].store(scratch, std::memory_order_release);
  }
  // Every slot of the partials is written before it is read, so nothing needs clearing.
  return fa3_decode_attn_gqa(q, k, v, q_scale, k_scale, v_scale, lens, out, B, Hq, Hkv, D, T_max, softmax_scale,
                             scratch, kGqaStaticScratchBytes, dev_err, stream);
}
