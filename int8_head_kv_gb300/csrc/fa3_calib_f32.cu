// Per-head Recall-Window calibration of float32 activations.
//
// msModelSlim "FA3量化" page, 原理 / 算法流程 steps 1-3 (as fa3_calibrate_perhead),
// for float32 input.  A float32 value has a 32-bit order-preserving key, too many
// for one counting table, so the tails are found by a two-level radix select:
//
//   pass 1  per head, a histogram of the keys' high 16 bits (shared-memory
//           counters per chunk, flushed into a per-head table);
//   select  the high-16 bins holding rank R - 1 (the R-th smallest value) and
//           rank N - R (the R-th largest), R = N - target_num + 1 window starts;
//   pass 2  histograms of the low 16 bits of the keys inside those two bins;
//   select  the exact 32-bit keys at those ranks and how many values lie
//           strictly beyond them;
//   pass 3  the values strictly below the lower key and strictly above the upper
//           key (fewer than R each) are appended to two lists;
//   window  per head: the lists are sorted in shared memory, padded with copies
//           of the two threshold values to the R smallest and R largest values,
//           and the R windows [sorted[i], sorted[i + target_num - 1]] are compared
//           by exact width (fp32 TwoSum pairs), ties to the smallest i; the
//           running min/max update uses IEEE totalOrder (-0.0 below +0.0).
//
// Every window starts among the R smallest values and ends among the R largest, so
// the result is exactly that of sorting every value.  Supported: R <= 4096.
// The workspace's tables are left zeroed by every call.
#include "fa3_common.cuh"

#include <math_constants.h>

#include <algorithm>

namespace fa3 {
namespace {

constexpr int kF32Bins = 65536;
constexpr int kF32MaxStarts = 4096;       // largest supported R
constexpr int kF32Chunk = 65535;          // values per pass-1 CTA (16-bit counters cannot overflow)
constexpr int kF32Threads = 512;

struct F32Info {
  uint32_t bin_lo, bin_hi;                // high-16 bins holding ranks R - 1 and N - R
  uint32_t below_lo, above_hi;            // values in bins below bin_lo / above bin_hi
  uint32_t key_lo, key_hi;                // keys at ranks R - 1 and N - R
  uint32_t less_lo, greater_hi;           // values with key < key_lo / key > key_hi
  uint32_t cnt_lo, cnt_hi;                // list fill counters
  uint32_t pad[6];
};

struct F32Params {
  const float* x;
  int64_t B, L, sb, sh, N;
  int H;
  uint32_t R;                             // window starts
  uint32_t t;                             // target_num
  uint32_t* hist_hi;                      // [H][65536]
  uint32_t* hist_lo;                      // [H][2][65536]
  F32Info* info;                          // [H]
  uint32_t* lists;                        // [H][2][kF32MaxStarts]
  float* min_io;
  float* max_io;
  int32_t* err;
};

__device__ __forceinline__ uint32_t f32_key(float v) {
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float f32_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}
__device__ __forceinline__ bool f32_tot_less(float a, float b) {
  return a < b || (a == b && signbit(a) && !signbit(b));
}
// Value n of head h (n = b * L + l).
__device__ __forceinline__ float f32_at(const F32Params& p, int h, int64_t n) {
  const int64_t b = n / p.L, l = n - b * p.L;
  return __ldcs(p.x + b * p.sb + (int64_t)h * p.sh + l);
}

// pass 1: grid (chunks, H); 16-bit counters packed two per shared word.
__global__ void __launch_bounds__(kF32Threads) f32_hist_hi_kernel(const F32Params p) {
  extern __shared__ uint32_t f32_bins[];   // 32768 words
  pdl_wait();
  pdl_launch_dependents();
  const int h = blockIdx.y;
  const int64_t n0 = (int64_t)blockIdx.x * kF32Chunk, n1 = min(n0 + (int64_t)kF32Chunk, p.N);
  for (int i = threadIdx.x; i < kF32Bins / 2; i += kF32Threads) f32_bins[i] = 0u;
  __syncthreads();
  for (int64_t n = n0 + threadIdx.x; n < n1; n += kF32Threads) {
    const uint32_t k = f32_key(f32_at(p, h, n)) >> 16;
    atomicAdd(&f32_bins[k >> 1], 1u << ((k & 1u) << 4));
  }
  __syncthreads();
  uint32_t* table = p.hist_hi + (int64_t)h * kF32Bins;
  for (int i = threadIdx.x; i < kF32Bins / 2; i += kF32Threads) {
    const uint32_t w = f32_bins[i];
    if (w & 0xffffu) atomicAdd(&table[2 * i], w & 0xffffu);
    if (w >> 16) atomicAdd(&table[2 * i + 1], w >> 16);
  }
}

// Block-wide search over 65536 counters: the first bin at which the running count
// from the bottom reaches `rank + 1` (from_top: the last bin at which the running
// count from the top does).  Returns the bin and the count strictly before it.
// Zeroes the counters it read.  kF32Threads threads, 128 bins each.
__device__ void f32_find_rank(uint32_t* table, uint32_t rank, bool from_top, uint32_t& bin_out,
                              uint32_t& before_out) {
  __shared__ uint32_t part[kF32Threads];
  __shared__ uint32_t res[2];
  constexpr int kPer = kF32Bins / kF32Threads;
  const int t = threadIdx.x;
  const int tt = from_top ? kF32Threads - 1 - t : t;      // this thread's block of bins, in search order
  if (t == 0) res[0] = res[1] = 0u;
  uint32_t sum = 0;
  for (int i = 0; i < kPer; ++i) sum += table[tt * kPer + i];
  part[t] = sum;
  __syncthreads();
  // inclusive scan (Hillis-Steele) over the blocks in search order
  for (int o = 1; o < kF32Threads; o <<= 1) {
    const uint32_t v = t >= o ? part[t - o] : 0u;
    __syncthreads();
    part[t] += v;
    __syncthreads();
  }
  const uint32_t incl = part[t], excl = incl - sum;
  if (excl <= rank && rank < incl) {                        // the block holding the rank
    uint32_t run = excl;
    for (int i = 0; i < kPer; ++i) {
      const int bin = from_top ? tt * kPer + (kPer - 1 - i) : tt * kPer + i;
      const uint32_t c = table[bin];
      if (run + c > rank) {
        res[0] = (uint32_t)bin;
        res[1] = run;
        break;
      }
      run += c;
    }
  }
  __syncthreads();
  bin_out = res[0];
  before_out = res[1];
  for (int i = 0; i < kPer; ++i) table[tt * kPer + i] = 0u;
  __syncthreads();
}

// select on the high 16 bits; one CTA per head
__global__ void __launch_bounds__(kF32Threads) f32_select_hi_kernel(const F32Params p) {
  pdl_wait();
  pdl_launch_dependents();
  const int h = blockIdx.x;
  uint32_t* table = p.hist_hi + (int64_t)h * kF32Bins;
  uint32_t b_lo, before_lo, b_hi, before_hi;
  // bottom: rank R - 1 from below; top: rank R - 1 from above (= rank N - R); the
  // first search zeroes the table, so the top search runs on a copy (in the high
  // half of hist_lo, which pass 2 needs zeroed: the search leaves it so)
  uint32_t* copy = p.hist_lo + (int64_t)h * 2 * kF32Bins + kF32Bins;
  for (int i = threadIdx.x; i < kF32Bins; i += kF32Threads) copy[i] = table[i];
  __syncthreads();
  f32_find_rank(table, p.R - 1, false, b_lo, before_lo);
  f32_find_rank(copy, p.R - 1, true, b_hi, before_hi);
  if (threadIdx.x == 0) {
    F32Info& in = p.info[h];
    in.bin_lo = b_lo;
    in.below_lo = before_lo;
    in.bin_hi = b_hi;
    in.above_hi = before_hi;
    in.cnt_lo = in.cnt_hi = 0u;
  }
}

// pass 2: low-16 histograms inside the two selected bins (warp-aggregated: equal
// keys of a warp add once)
__global__ void __launch_bounds__(kF32Threads) f32_hist_lo_kernel(const F32Params p) {
  pdl_wait();
  pdl_launch_dependents();
  const int h = blockIdx.y;
  const uint32_t b_lo = p.info[h].bin_lo, b_hi = p.info[h].bin_hi;
  uint32_t* t_lo = p.hist_lo + (int64_t)h * 2 * kF32Bins;
  uint32_t* t_hi = t_lo + kF32Bins;
  const int64_t stride = (int64_t)gridDim.x * kF32Threads;
  for (int64_t n0 = (int64_t)blockIdx.x * kF32Threads; n0 < p.N; n0 += stride) {
    const int64_t n = n0 + threadIdx.x;
    uint32_t k = 0xffffffffu;
    if (n < p.N) k = f32_key(f32_at(p, h, n));
    // the two bins may be the same one: count into each table separately
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const bool in = n < p.N && (k >> 16) == (which ? b_hi : b_lo);
      const uint32_t tag = in ? (k & 0xffffu) : 0xffffffffu;
      const uint32_t peers = __match_any_sync(0xffffffffu, tag);
      if (in && (__ffs(peers) - 1) == (int)(threadIdx.x & 31))
        atomicAdd(&(which ? t_hi : t_lo)[k & 0xffffu], (uint32_t)__popc(peers));
    }
  }
}

// select on the low 16 bits; one CTA per head
__global__ void __launch_bounds__(kF32Threads) f32_select_lo_kernel(const F32Params p) {
  pdl_wait();
  pdl_launch_dependents();
  const int h = blockIdx.x;
  F32Info& in = p.info[h];
  uint32_t* t_lo = p.hist_lo + (int64_t)h * 2 * kF32Bins;
  uint32_t l_lo, b4_lo, l_hi, b4_hi;
  f32_find_rank(t_lo, p.R - 1 - in.below_lo, false, l_lo, b4_lo);
  f32_find_rank(t_lo + kF32Bins, p.R - 1 - in.above_hi, true, l_hi, b4_hi);
  if (threadIdx.x == 0) {
    in.key_lo = (in.bin_lo << 16) | l_lo;
    in.less_lo = in.below_lo + b4_lo;
    in.key_hi = (in.bin_hi << 16) | l_hi;
    in.greater_hi = in.above_hi + b4_hi;
  }
}

// pass 3: the values strictly beyond the two keys (fewer than R each)
__global__ void __launch_bounds__(kF32Threads) f32_collect_kernel(const F32Params p) {
  pdl_wait();
  pdl_launch_dependents();
  const int h = blockIdx.y;
  F32Info& in = p.info[h];
  const uint32_t k_lo = in.key_lo, k_hi = in.key_hi;
  uint32_t* l_lo = p.lists + (int64_t)h * 2 * kF32MaxStarts;
  uint32_t* l_hi = l_lo + kF32MaxStarts;
  const int64_t stride = (int64_t)gridDim.x * kF32Threads;
  for (int64_t n = (int64_t)blockIdx.x * kF32Threads + threadIdx.x; n < p.N; n += stride) {
    const uint32_t k = f32_key(f32_at(p, h, n));
    if (k < k_lo) {
      const uint32_t i = atomicAdd(&in.cnt_lo, 1u);
      if (i < kF32MaxStarts) l_lo[i] = k;
    } else if (k > k_hi) {
      const uint32_t i = atomicAdd(&in.cnt_hi, 1u);
      if (i < kF32MaxStarts) l_hi[i] = k;
    }
  }
}

// Ascending bitonic sort of n <= kF32MaxStarts keys in shared memory (padded with
// 0xffffffff to the next power of two).
__device__ void f32_sort(uint32_t* a, uint32_t n) {
  uint32_t m = 1;
  while (m < n) m <<= 1;
  for (uint32_t i = n + threadIdx.x; i < m; i += kF32Threads) a[i] = 0xffffffffu;
  __syncthreads();
  for (uint32_t k = 2; k <= m; k <<= 1)
    for (uint32_t j = k >> 1; j > 0; j >>= 1) {
      for (uint32_t i = threadIdx.x; i < m; i += kF32Threads) {
        const uint32_t l = i ^ j;
        if (l > i) {
          const bool up = (i & k) == 0;
          const uint32_t x = a[i], y = a[l];
          if ((x > y) == up) { a[i] = y; a[l] = x; }
        }
      }
      __syncthreads();
    }
}

__global__ void __launch_bounds__(kF32Threads) f32_window_kernel(const F32Params p) {
  __shared__ uint32_t s_lo[kF32MaxStarts];
  __shared__ uint32_t s_hi[kF32MaxStarts];
  __shared__ float red_s[kF32Threads / 32], red_e[kF32Threads / 32];
  __shared__ uint32_t red_i[kF32Threads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int h = blockIdx.x;
  F32Info& in = p.info[h];
  const uint32_t R = p.R, nlo = in.less_lo, nhi = in.greater_hi;
  const uint32_t* l_lo = p.lists + (int64_t)h * 2 * kF32MaxStarts;
  const uint32_t* l_hi = l_lo + kF32MaxStarts;
  // counts agree with the selection, or the head is left as it is
  const bool good = in.cnt_lo == nlo && in.cnt_hi == nhi && nlo < R && nhi < R;
  for (uint32_t i = threadIdx.x; i < nlo && good; i += kF32Threads) s_lo[i] = l_lo[i];
  for (uint32_t i = threadIdx.x; i < nhi && good; i += kF32Threads) s_hi[i] = l_hi[i];
  __syncthreads();
  if (!good) {
    if (threadIdx.x == 0) {
      set_dev_err(p.err, FA3_DEVERR_CALIB);
      in.cnt_lo = in.cnt_hi = 0u;
    }
    return;
  }
  f32_sort(s_lo, nlo);
  f32_sort(s_hi, nhi);
  // small(i) = s_i for i < R: the sorted list, then copies of key_lo;
  // large(i) = s_{N-R+i}: copies of key_hi, then the sorted list
  float best_s = CUDART_INF_F, best_e = 0.f;
  uint32_t best_i = 0xffffffffu;
  for (uint32_t i = threadIdx.x; i < R; i += kF32Threads) {
    const uint32_t ka = i < nlo ? s_lo[i] : in.key_lo;
    const uint32_t kb = i < R - nhi ? in.key_hi : s_hi[i - (R - nhi)];
    const float b = f32_value(kb), y = -f32_value(ka);
    const float s = __fadd_rn(b, y);
    const float bp = __fsub_rn(s, b);
    const float ap = __fsub_rn(s, bp);
    const float e = __fadd_rn(__fsub_rn(b, ap), __fsub_rn(y, bp));
    if (s < best_s || (s == best_s && (e < best_e || (e == best_e && i < best_i)))) {
      best_s = s; best_e = e; best_i = i;
    }
  }
  // block argmin (width pair, then index)
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) {
    const float os = __shfl_xor_sync(0xffffffffu, best_s, o), oe = __shfl_xor_sync(0xffffffffu, best_e, o);
    const uint32_t oi = __shfl_xor_sync(0xffffffffu, best_i, o);
    if (os < best_s || (os == best_s && (oe < best_e || (oe == best_e && oi < best_i)))) {
      best_s = os; best_e = oe; best_i = oi;
    }
  }
  if (lane == 0) { red_s[wid] = best_s; red_e[wid] = best_e; red_i[wid] = best_i; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kF32Threads / 32; ++w)
      if (red_s[w] < red_s[0] || (red_s[w] == red_s[0] && (red_e[w] < red_e[0] ||
                                                          (red_e[w] == red_e[0] && red_i[w] < red_i[0])))) {
        red_s[0] = red_s[w]; red_e[0] = red_e[w]; red_i[0] = red_i[w];
      }
    const uint32_t i = red_i[0];
    const float lo = f32_value(i < nlo ? s_lo[i] : in.key_lo);
    const float hi = f32_value(i < R - nhi ? in.key_hi : s_hi[i - (R - nhi)]);
    if (f32_tot_less(lo, p.min_io[h])) p.min_io[h] = lo;
    if (f32_tot_less(p.max_io[h], hi)) p.max_io[h] = hi;
    in.cnt_lo = in.cnt_hi = 0u;
  }
}

}  // namespace
}  // namespace fa3

using namespace fa3;

FA3_API size_t fa3_calibrate_f32_workspace_size(int H) {
  if (H <= 0) return 0;
  return (size_t)H * (3 * kF32Bins * sizeof(uint32_t) + sizeof(F32Info) + 2 * kF32MaxStarts * sizeof(uint32_t)) + 256;
}

FA3_API int fa3_calibrate_perhead_f32(const float* x, int64_t B, int H, int64_t L, int64_t stride_b,
                                      int64_t stride_h, double ratio, float* min_io, float* max_io,
                                      void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (!x || !min_io || !max_io) return FA3_EINVAL;
  if (B <= 0 || H <= 0 || L <= 0 || stride_b < 0 || stride_h < 0) return FA3_EINVAL;
  if (!(ratio > 0.0 && ratio <= 1.0)) return FA3_EINVAL;
  const int64_t N = B * L;
  if (N <= 0 || N >= ((int64_t)1 << 31) || H > 65535) return FA3_ERANGE;
  // FA3量化 step 2: target_num = int(ratio * N), float64 product, truncation; at least 1.
  int64_t t = (int64_t)(ratio * (double)N);
  if (t < 1) t = 1;
  if (t > N) t = N;
  const int64_t R = N - t + 1;
  if (R > kF32MaxStarts) return FA3_ERANGE;
  if (!workspace || workspace_bytes < fa3_calibrate_f32_workspace_size(H) || !aligned16(workspace))
    return FA3_EWORKSPACE;
  int sms = 0;
  const int st = check_device(&sms);
  if (st != FA3_OK) return st;
  F32Params p;
  p.x = x; p.B = B; p.L = L; p.sb = stride_b; p.sh = stride_h; p.N = N; p.H = H;
  p.R = (uint32_t)R; p.t = (uint32_t)t;
  char* ws = static_cast<char*>(workspace);
  p.hist_hi = reinterpret_cast<uint32_t*>(ws);
  p.hist_lo = p.hist_hi + (size_t)H * kF32Bins;
  p.lists = p.hist_lo + (size_t)H * 2 * kF32Bins;
  p.info = reinterpret_cast<F32Info*>(p.lists + (size_t)H * 2 * kF32MaxStarts);
  p.min_io = min_io; p.max_io = max_io; p.err = dev_err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int smem = kF32Bins * 2;   // 128 KB of 16-bit counters
  if (cudaFuncSetAttribute(f32_hist_hi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return FA3_ECUDA;
  const unsigned chunks = (unsigned)((N + kF32Chunk - 1) / kF32Chunk);
  const unsigned stream_blocks = (unsigned)std::max<int64_t>(1, std::min<int64_t>((N + kF32Threads - 1) / kF32Threads,
                                                                                  (int64_t)sms * 4 / H + 1));
  if (launch_pdl(f32_hist_hi_kernel, dim3(chunks, H), dim3(kF32Threads), smem, s, p) != cudaSuccess ||
      launch_pdl(f32_select_hi_kernel, dim3(H), dim3(kF32Threads), 0, s, p) != cudaSuccess ||
      launch_pdl(f32_hist_lo_kernel, dim3(stream_blocks, H), dim3(kF32Threads), 0, s, p) != cudaSuccess ||
      launch_pdl(f32_select_lo_kernel, dim3(H), dim3(kF32Threads), 0, s, p) != cudaSuccess ||
      launch_pdl(f32_collect_kernel, dim3(stream_blocks, H), dim3(kF32Threads), 0, s, p) != cudaSuccess ||
      launch_pdl(f32_window_kernel, dim3(H), dim3(kF32Threads), 0, s, p) != cudaSuccess)
    return FA3_ECUDA;
  return FA3_OK;
}
