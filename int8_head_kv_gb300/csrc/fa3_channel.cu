// Per-channel Recall-Window calibration.
//
// MindIE Turbo "Attention量化", 表1 / 表2 keeps one scale and offset per (head,
// channel), [head_num, head_dim]; the Recall Window of msModelSlim "FA3量化"
// 原理 / 算法流程 steps 2-3 then runs on each channel's N = B*S values.
//
// Every window [sorted[i], sorted[i + t - 1]], i = 0 .. R - 1 with R = N - t + 1,
// starts among the R smallest values and ends among the R largest, so a channel
// needs only its two tails.  Supported: R <= 32 (the pages' ratio 0.9999 keeps R
// at most 32 up to N = 320,000 values per channel).
//
// One CTA per (head, 32 channels): lane l reads channel d0 + l (one 64-byte row
// segment per warp and row), warp w takes rows w, w + 8, ...; each thread keeps
// its rows' R smallest and R largest order-preserving 16-bit keys (ascending, in
// shared memory), then one thread per channel merges the eight warps' lists,
// compares the R windows' exact widths (fp32 TwoSum pairs; ties keep the
// smallest start) and folds the window into the running range in IEEE
// totalOrder (-0.0 below +0.0).
#include "fa3_common.cuh"

#include <math_constants.h>

namespace fa3 {
namespace {

constexpr int kChR = 32;           // largest supported number of window starts
constexpr int kChWarps = 8;

__device__ __forceinline__ uint32_t ch_key(uint32_t bits) {        // bf16 bits -> order-preserving key
  return (bits & 0x8000u) ? (~bits & 0xffffu) : (bits | 0x8000u);
}
__device__ __forceinline__ float ch_value(uint32_t key) {
  const uint32_t bits = (key & 0x8000u) ? (key ^ 0x8000u) : (~key & 0xffffu);
  return __uint_as_float(bits << 16);
}
__device__ __forceinline__ bool ch_less(float a, float b) {
  return a < b || (a == b && signbit(a) && !signbit(b));
}

struct ChParams {
  const uint16_t* x;
  int64_t B, S;
  int H, D;
  int64_t sb, sh, ss;      // element strides of b, h, s (d is contiguous)
  int R;                   // window starts: N - target_num + 1
  float* min_io;           // [H][D]
  float* max_io;
};

__global__ void __launch_bounds__(32 * kChWarps)
calibrate_channel_kernel(const ChParams p) {
  __shared__ uint16_t small_k[kChWarps][32][kChR];
  __shared__ uint16_t large_k[kChWarps][32][kChR];
  pdl_wait();
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.y, d = blockIdx.x * 32 + lane;
  const bool on = d < p.D;
  const int R = p.R;
  uint16_t* sk = small_k[warp][lane];
  uint16_t* lk = large_k[warp][lane];
  int ns = 0, nl = 0;                      // filled entries
  uint32_t thr_s = 0xffffu, thr_l = 0u;    // the R-th smallest / largest once full
  auto insert = [&](uint32_t key) {
    if (ns < R || key < thr_s) {           // keep the R smallest, ascending
      int j = ns < R ? ns++ : R - 1;
      while (j > 0 && sk[j - 1] > key) { sk[j] = sk[j - 1]; --j; }
      sk[j] = (uint16_t)key;
      if (ns == R) thr_s = sk[R - 1];
    }
    if (nl < R || key > thr_l) {           // keep the R largest, ascending
      int j;
      if (nl < R) {
        j = nl++;
        while (j > 0 && lk[j - 1] > key) { lk[j] = lk[j - 1]; --j; }
      } else {
        j = 0;                             // drop the smallest, shift down
        while (j + 1 < R && lk[j + 1] < key) { lk[j] = lk[j + 1]; ++j; }
      }
      lk[j] = (uint16_t)key;
      if (nl == R) thr_l = lk[0];
    }
  };
  if (on) {
    const uint16_t* xh = p.x + (int64_t)h * p.sh + d;
    for (int64_t b = 0; b < p.B; ++b) {
      const uint16_t* xb = xh + b * p.sb;
      int64_t s = warp;
      for (; s + 3 * kChWarps < p.S; s += 4 * kChWarps) {      // four rows in flight
        uint32_t v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldg(xb + (s + u * kChWarps) * p.ss);
#pragma unroll
        for (int u = 0; u < 4; ++u) insert(ch_key(v[u]));
      }
      for (; s < p.S; s += kChWarps) insert(ch_key(__ldg(xb + s * p.ss)));
    }
  }
  __syncthreads();
  if (warp != 0 || !on) return;
  // Merge the eight warps' lists of this channel (each ascending).
  uint16_t small_m[kChR], large_m[kChR];
  {
    int ps[kChWarps], pl[kChWarps], cnt_s[kChWarps], cnt_l[kChWarps];
#pragma unroll
    for (int w = 0; w < kChWarps; ++w) {
      // rows of warp w: those s with s % 8 == w, in every b
      const int64_t rows = p.B * ((p.S > w) ? (p.S - w + kChWarps - 1) / kChWarps : 0);
      cnt_s[w] = cnt_l[w] = (int)(rows < R ? rows : (int64_t)R);
      ps[w] = 0;
      pl[w] = cnt_l[w] - 1;               // the largest lists are merged from their tops
    }
    for (int k = 0; k < R; ++k) {         // k-th smallest overall
      int best = -1;
      uint32_t bv = 0x10000u;
#pragma unroll
      for (int w = 0; w < kChWarps; ++w)
        if (ps[w] < cnt_s[w] && small_k[w][lane][ps[w]] < bv) { bv = small_k[w][lane][ps[w]]; best = w; }
      small_m[k] = (uint16_t)bv;
      if (best >= 0) ++ps[best];
    }
    for (int k = R - 1; k >= 0; --k) {    // (R-1-k)-th largest overall, stored ascending
      int best = -1;
      int bv = -1;
#pragma unroll
      for (int w = 0; w < kChWarps; ++w)
        if (pl[w] >= 0 && (int)large_k[w][lane][pl[w]] > bv) { bv = large_k[w][lane][pl[w]]; best = w; }
      large_m[k] = (uint16_t)bv;
      if (best >= 0) --pl[best];
    }
  }
  // Window i = [small_m[i], large_m[i]]: exact width as an fp32 TwoSum pair.
  float best_s = CUDART_INF_F, best_e = 0.f;
  int best_i = 0;
  for (int i = 0; i < R; ++i) {
    const float b = ch_value(large_m[i]), y = -ch_value(small_m[i]);
    const float s = __fadd_rn(b, y);
    const float bp = __fsub_rn(s, b);
    const float ap = __fsub_rn(s, bp);
    const float e = __fadd_rn(__fsub_rn(b, ap), __fsub_rn(y, bp));
    if (s < best_s || (s == best_s && e < best_e)) { best_s = s; best_e = e; best_i = i; }
  }
  const float lo = ch_value(small_m[best_i]), hi = ch_value(large_m[best_i]);
  const int64_t o = (int64_t)h * p.D + d;
  if (ch_less(lo, p.min_io[o])) p.min_io[o] = lo;
  if (ch_less(p.max_io[o], hi)) p.max_io[o] = hi;
}

}  // namespace
}  // namespace fa3

using namespace fa3;

FA3_API int fa3_calibrate_perchannel(const uint16_t* x, int64_t B, int H, int64_t S, int D, int64_t stride_b,
                                     int64_t stride_h, int64_t stride_s, double ratio, float* min_io,
                                     float* max_io, void* stream) {
  if (!x || !min_io || !max_io) return FA3_EINVAL;
  if (B <= 0 || H <= 0 || S <= 0 || D <= 0) return FA3_EINVAL;
  if (!(ratio > 0.0 && ratio <= 1.0)) return FA3_EINVAL;
  if (H > 65535) return FA3_ERANGE;
  const int64_t N = B * S;
  // FA3量化 step 2: target_num = int(ratio * N), float64 product, truncation; at least 1.
  int64_t t = (int64_t)(ratio * (double)N);
  if (t < 1) t = 1;
  const int64_t R = N - t + 1;
  if (R > kChR) return FA3_ERANGE;
  int sms = 0;
  const int st = check_device(&sms);
  if (st != FA3_OK) return st;
  ChParams p;
  p.x = x; p.B = B; p.S = S; p.H = H; p.D = D; p.sb = stride_b; p.sh = stride_h; p.ss = stride_s;
  p.R = (int)R; p.min_io = min_io; p.max_io = max_io;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_pdl(calibrate_channel_kernel, dim3((D + 31) / 32, H), dim3(32 * kChWarps), 0, s, p));
}
