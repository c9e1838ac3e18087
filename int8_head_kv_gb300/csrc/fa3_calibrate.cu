// Per-head Recall-Window calibration.
//
// msModelSlim "FA3量化" page, 原理 / 算法流程:
//   step 1  every head collects its N = B*S*D activation values;
//   step 2  sort them, target_num = int(ratio*N), and keep the narrowest window
//           [sorted[i], sorted[i+target_num-1]] over i = 0 .. N - target_num;
//   step 3  running min/max of the window ends across calibration batches.
//
// GB300 design.  bf16 has only 65536 bit patterns, and a monotone 16-bit key
// maps them onto the total order of their values (-0 before +0).  Counting
// each key (a counting sort) therefore carries the whole sorted sequence, so
// one pass over HBM replaces the sort:
//   kernel 1  persistent CTAs walk (head, 65528-value chunk) pairs: a 65536-bin
//             histogram of 16-bit counters packed two per word in 128 KB of
//             shared memory (a chunk is shorter than 65536, so no counter can
//             overflow), then the non-zero bins are added into the per-head u32
//             table in the workspace and cleared, while the next chunk loads.
//   kernel 2  per head: prefix sums over the 65536 bins; a window can only be
//             narrowest if it starts at the first copy of a value, so each
//             occupied bin v with start position P(v) <= N - target_num is a
//             candidate whose window ends in the bin holding position
//             P(v) + target_num - 1.  Exact widths (fp32 TwoSum pairs), argmin
//             with ties to the smallest start, then the running min/max update.  The kernel
//             zeroes the bins it read, leaving the workspace clean.
// When few windows exist (N - target_num + 1 <= 16384, e.g. ratio 0.9999), every
// window starts among the N - target_num + 1 smallest values and ends among the
// as many largest, so only the two tails of a head need counting: a sampling
// kernel picks per-head tail thresholds, kernel 1 counts only keys beyond them
// (HBM-bound instead of atomic-bound), and kernel 2 places the uncounted middle
// as one block of known size between the tails, checking that each tail holds
// enough values.  A head that fails the check is counted again in full by a
// second launch of kernel 2, which returns at once for every other head; the
// result is the same exact window either way.
#include "fa3_common.cuh"

#include <math_constants.h>

namespace fa3 {
namespace {

constexpr int kBins = 65536;
constexpr int kHistThreads = 1024;
constexpr int kChunk = 65528;                       // values per histogram CTA (multiple of 8, < 65536)
constexpr int kGroupsPerThread = (kChunk / 8 + kHistThreads - 1) / kHistThreads;   // 8
constexpr int kScalarPerThread = (kChunk + kHistThreads - 1) / kHistThreads;       // 64
constexpr int kWinThreads = 1024;
constexpr int kBinsPerThread = kBins / kWinThreads;  // 64
constexpr int kCandCap = 16384;     // window starts the fast search can table (N - t + 1 <= kCandCap)
constexpr int kSampleUnits = 512;   // strided samples per head for the tail thresholds (16-byte groups or values)
constexpr int kSampleThreads = 256;
constexpr int kTailThreads = 256;
constexpr int kTailGroups = 8;      // 16-byte groups per thread of the tail-count kernel

// Per-head state of the tail-only path, in the workspace after the counters.
// key_lo / key_hi: count keys <= key_lo or >= key_hi (key_lo = 0xffff: all keys);
// flag: the tails were too thin, count this head again in full.
struct TailInfo {
  uint32_t key_lo, key_hi, flag, pad;
};

// Order-preserving 16-bit key of a bf16 value: positive values get the top bit
// set, negative values are bit-inverted, so key order == value order and -0.0
// (0x8000) maps just below +0.0 (0x0000).  key_value is the inverse.
__device__ __forceinline__ float key_value(uint32_t key) {
  uint32_t bits = (key & 0x8000u) ? (key ^ 0x8000u) : (~key & 0xffffu);
  return __uint_as_float(bits << 16);
}

// Two order-preserving keys from one 32-bit word holding two bf16 values:
// negative halves are inverted, positive halves get their top bit set.
__device__ __forceinline__ uint32_t bf16x2_keys(uint32_t w) {
  const uint32_t neg = (w >> 15) & 0x00010001u;            // sign bit of each half, at bit 0 / 16
  return w ^ ((neg * 0x7fffu) | 0x80008000u);
}

// Adds one count for the 16-bit key `key` (two 16-bit counters per shared word).
__device__ __forceinline__ void count16(uint32_t* bins, uint32_t key) {
  atomicAdd(&bins[key >> 1], 1u << ((key & 1u) << 4));
}
// Counts `key` only if it lies in a counted tail (key <= lo or key >= hi).
__device__ __forceinline__ void count16_tails(uint32_t* bins, uint32_t key, uint32_t lo, uint32_t hi) {
  if (key <= lo || key >= hi) count16(bins, key);
}

// Packed bf16x2 min / max (IEEE: -0 == +0).
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Counts the 8 values of one 16-byte group (only keys <= lo or >= hi).  The common
// case, no counted key in the whole warp's groups, is ruled out by comparing the
// group's bf16 min and max with the values of the thresholds (strictly, so a tie or
// a signed zero at a threshold always takes the exact per-key path) and one vote.
// When the whole warp holds one and the same 16 bytes made of a single repeated
// value (a constant head), one lane adds 256 at once instead of 256 conflicting
// atomics.
__device__ __forceinline__ void count_group(uint32_t* bins, const uint4 v, bool valid, uint32_t lo, uint32_t hi,
                                            float v_lo, float v_hi) {
  const uint32_t mn = bmin2(bmin2(v.x, v.y), bmin2(v.z, v.w)), mx = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
  const float gmin = fminf(__uint_as_float(mn << 16), __uint_as_float(mn & 0xffff0000u));
  const float gmax = fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xffff0000u));
  const bool maybe = valid && !(gmin > v_lo && gmax < v_hi);
  if (!__any_sync(0xffffffffu, maybe)) return;
  const uint32_t w0 = __shfl_sync(0xffffffffu, v.x, 0);
  const bool uniform = __all_sync(0xffffffffu, valid && v.x == w0 && v.y == w0 && v.z == w0 && v.w == w0 &&
                                                   (w0 >> 16) == (w0 & 0xffffu));
  if (uniform) {
    if ((threadIdx.x & 31) == 0) {
      const uint32_t key = bf16x2_keys(w0) & 0xffffu;
      if (key <= lo || key >= hi) atomicAdd(&bins[key >> 1], 256u << ((key & 1u) << 4));
    }
    return;
  }
  if (!maybe) return;
  const uint32_t k[4] = {bf16x2_keys(v.x), bf16x2_keys(v.y), bf16x2_keys(v.z), bf16x2_keys(v.w)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    count16_tails(bins, k[i] & 0xffffu, lo, hi);
    count16_tails(bins, k[i] >> 16, lo, hi);
  }
}

// Persistent: CTA g walks chunks g, g + gridDim.x, ... of the (head, chunk) list.
// While the histogram of one chunk is flushed (and re-zeroed in the same pass),
// the loads of the next chunk are already in flight.
__global__ void __launch_bounds__(kHistThreads, 1)
hist_kernel(const uint16_t* __restrict__ x, int64_t L, int64_t stride_b, int64_t stride_h, int64_t N,
            int chunks_per_head, int total_chunks, uint32_t* __restrict__ counts, int vec,
            const TailInfo* __restrict__ tails) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ uint4 smem_hist[];
  uint32_t* bins = reinterpret_cast<uint32_t*>(smem_hist);   // 32768 words = 65536 16-bit bins
  const int tid = threadIdx.x;
  for (int i = tid; i < kBins / 8; i += kHistThreads) smem_hist[i] = make_uint4(0, 0, 0, 0);

  auto chunk_span = [&](int ci, int& h, int64_t& n0, int64_t& n1) {
    h = ci / chunks_per_head;
    n0 = (int64_t)(ci - h * chunks_per_head) * kChunk;
    n1 = min(n0 + (int64_t)kChunk, N);
  };
  auto load_chunk = [&](int ci, uint4 (&v)[kGroupsPerThread]) {
    int h; int64_t n0, n1;
    chunk_span(ci, h, n0, n1);
    const uint16_t* xh = x + (int64_t)h * stride_h;
    // position n = b * L + l: one division per chunk, then at most a few row steps
    // (a thread's positions grow by 8 * kHistThreads per load)
    const int64_t b0 = n0 / L;
    int64_t b = b0, l = n0 - b0 * L + 8 * tid;
    while (l >= L) { l -= L; ++b; }
#pragma unroll
    for (int k = 0; k < kGroupsPerThread; ++k) {
      v[k] = make_uint4(0, 0, 0, 0);
      if (b * L + l < n1) v[k] = __ldcs(reinterpret_cast<const uint4*>(xh + b * stride_b + l));
      l += 8 * kHistThreads;
      while (l >= L) { l -= L; ++b; }
    }
  };

  uint4 v[kGroupsPerThread];
  int ci = blockIdx.x;
  if (vec && ci < total_chunks) load_chunk(ci, v);
  __syncthreads();
  while (ci < total_chunks) {
    int h; int64_t n0, n1;
    chunk_span(ci, h, n0, n1);
    uint32_t lo = 0xffffu, hi = 0x10000u;       // count every key ...
    if (tails) { lo = tails[h].key_lo; hi = tails[h].key_hi; }   // ... or only the tails
    // the thresholds as values (-inf / +inf when everything is counted)
    const float v_lo = lo >= 0xffffu ? CUDART_INF_F : key_value(lo);
    const float v_hi = hi > 0xffffu ? -CUDART_INF_F : key_value(hi);
    if (vec) {
#pragma unroll
      for (int k = 0; k < kGroupsPerThread; ++k) {
        const int64_t n = n0 + 8 * (int64_t)(tid + k * kHistThreads);
        count_group(bins, v[k], n < n1, lo, hi, v_lo, v_hi);
      }
    } else {
      const uint16_t* xh = x + (int64_t)h * stride_h;
      for (int k = 0; k < kScalarPerThread; ++k) {
        const int64_t n = n0 + tid + (int64_t)k * kHistThreads;
        if (n < n1) {
          const int64_t b = n / L, l = n - b * L;
          count16_tails(bins, bf16x2_keys(xh[b * stride_b + l]) & 0xffffu, lo, hi);
        }
      }
    }
    __syncthreads();
    const int cn = ci + gridDim.x;
    if (vec && cn < total_chunks) load_chunk(cn, v);
    // flush the non-zero counters into the head's table and clear them (only the
    // counted key ranges can hold any: groups of 8 bins [0, lo] and [hi, 0xffff])
    uint32_t* ch = counts + (int64_t)h * kBins;
    const int g_lo = lo >= 0xffffu ? kBins / 8 : (int)(lo >> 3) + 1, g_hi = hi > 0xffffu ? kBins / 8 : (int)(hi >> 3);
    for (int i0 = tid; i0 < kBins / 8; i0 += kHistThreads) {
      const int i = i0 < g_lo ? i0 : (g_hi > g_lo ? g_hi + (i0 - g_lo) : kBins / 8);
      if (i >= kBins / 8) break;
      const uint4 q = smem_hist[i];
      if ((q.x | q.y | q.z | q.w) == 0u) continue;
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t c0 = w[j] & 0xffffu, c1 = w[j] >> 16;
        if (c0) atomicAdd(&ch[8 * i + 2 * j], c0);
        if (c1) atomicAdd(&ch[8 * i + 2 * j + 1], c1);
      }
      smem_hist[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    ci = cn;
  }
}

// Tail-only counting for 16-byte aligned rows: grid (ranges of a row, rows b * H + h);
// each thread loads kTailGroups groups of 8 values at once, rules most of them out
// with the packed min / max test of count_group, and adds the keys of the rest
// straight into the head's u32 table (they are rare: a few 1e-4 of the values).
__global__ void __launch_bounds__(kTailThreads)
tail_count_kernel(const uint16_t* __restrict__ x, int64_t L, int64_t stride_b, int64_t stride_h, int H,
                  uint32_t* __restrict__ counts, const TailInfo* __restrict__ tails) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.y, h = row % H, b = row / H;
  const uint4* src = reinterpret_cast<const uint4*>(x + (int64_t)b * stride_b + (int64_t)h * stride_h);
  const int64_t groups = L / 8;
  const int64_t g0 = (int64_t)blockIdx.x * (kTailThreads * kTailGroups) + threadIdx.x;
  const uint32_t lo = tails[h].key_lo, hi = tails[h].key_hi;
  const float v_lo = lo >= 0xffffu ? CUDART_INF_F : key_value(lo);
  const float v_hi = hi > 0xffffu ? -CUDART_INF_F : key_value(hi);
  uint32_t* ch = counts + (int64_t)h * kBins;
  uint4 v[kTailGroups];
#pragma unroll
  for (int k = 0; k < kTailGroups; ++k) {
    const int64_t g = g0 + (int64_t)k * kTailThreads;
    v[k] = g < groups ? __ldcs(src + g) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int k = 0; k < kTailGroups; ++k) {
    const bool valid = g0 + (int64_t)k * kTailThreads < groups;
    const uint32_t mn = bmin2(bmin2(v[k].x, v[k].y), bmin2(v[k].z, v[k].w));
    const uint32_t mx = bmax2(bmax2(v[k].x, v[k].y), bmax2(v[k].z, v[k].w));
    const float gmin = fminf(__uint_as_float(mn << 16), __uint_as_float(mn & 0xffff0000u));
    const float gmax = fmaxf(__uint_as_float(mx << 16), __uint_as_float(mx & 0xffff0000u));
    if (valid && !(gmin > v_lo && gmax < v_hi)) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t k2 = bf16x2_keys(w[i]);
        const uint32_t a = k2 & 0xffffu, c = k2 >> 16;
        if (a <= lo || a >= hi) atomicAdd(&ch[a], 1u);
        if (c <= lo || c >= hi) atomicAdd(&ch[c], 1u);
      }
    }
  }
}

// Warp-wide: the bin of a 256-bin histogram holding its r-th smallest element
// (from_top: r-th largest) and that element's 1-based rank inside the bin.  Lane l
// owns 8 consecutive bins; r must not exceed the histogram's total.
__device__ __forceinline__ void select_bin(const uint32_t* hist, uint32_t r, bool from_top, uint32_t& bin,
                                           uint32_t& rank) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8], sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int i = 8 * lane + j;
    c[j] = hist[from_top ? 255 - i : i];
    sum += c[j];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t m = __ballot_sync(0xffffffffu, incl >= r);
  const int owner = m ? __ffs(m) - 1 : 31;
  uint32_t b = 0, rk = 1, acc = incl - sum;
  if (lane == owner) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (acc + c[j] >= r) { const int i = 8 * lane + j; b = (uint32_t)(from_top ? 255 - i : i); rk = r - acc; break; }
      acc += c[j];
    }
  }
  bin = __shfl_sync(0xffffffffu, b, owner);
  rank = __shfl_sync(0xffffffffu, rk, owner);
}

// Tail thresholds of head h from kSampleUnits strided samples (16-byte groups when
// vec, single values otherwise).  With S sampled keys and p = (N - t + 1) / N, the
// sample's r-th smallest key, r = 3 S p + 4, lies above the N - t + 1 smallest
// values of the head unless the sample over-represents the low tail badly (the
// window kernel checks and falls back); key_lo is that key, key_hi the r-th
// largest.  The order statistics come from a two-level radix select on the key
// bytes.  Overlapping tails count everything.
__global__ void __launch_bounds__(kSampleThreads)
tail_kernel(const uint16_t* __restrict__ x, int64_t L, int64_t stride_b, int64_t stride_h, int64_t N,
            unsigned long long span, int vec, TailInfo* __restrict__ tails) {
  pdl_wait();
  pdl_launch_dependents();
  constexpr int kUnits = kSampleUnits / kSampleThreads;    // 16 samples per thread
  constexpr int kWarps = kSampleThreads / 32;
  __shared__ uint32_t whist[kWarps][256];        // per-warp high-byte histograms
  __shared__ uint32_t hist[3][256];              // high byte; low byte in the low bin; low byte in the high bin
  __shared__ uint32_t sel[4];                    // b_lo, b_hi, residual rank in b_lo, in b_hi
  const int h = blockIdx.x, tid = threadIdx.x, warp = tid >> 5;
  for (int i = tid; i < kWarps * 256; i += kSampleThreads) (&whist[0][0])[i] = 0u;
  for (int i = tid; i < 3 * 256; i += kSampleThreads) (&hist[0][0])[i] = 0u;
  const uint16_t* xh = x + (int64_t)h * stride_h;
  const int64_t units = vec ? N / 8 : N;
  const int per = vec ? 8 : 1;
  // all loads first (independent), keys kept in registers for both passes
  uint4 q[kUnits];
  bool ok[kUnits];
#pragma unroll
  for (int j = 0; j < kUnits; ++j) {
    const int g = tid + j * kSampleThreads;
    const int64_t u = (int64_t)((unsigned long long)g * (unsigned long long)units / kSampleUnits);
    ok[j] = u < units;
    q[j] = make_uint4(0u, 0u, 0u, 0u);
    if (ok[j]) {
      const int64_t n = u * per, b = n / L, l = n - b * L;
      if (vec) q[j] = *reinterpret_cast<const uint4*>(xh + b * stride_b + l);
      else q[j].x = xh[b * stride_b + l];
    }
  }
  __syncthreads();
  // fn(key, valid) is called by every lane the same number of times (warp-uniform)
  auto for_keys = [&](auto&& fn) {
#pragma unroll
    for (int j = 0; j < kUnits; ++j) {
      if (vec) {
        const uint32_t w[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t k2 = bf16x2_keys(w[i]);
          fn(k2 & 0xffffu, ok[j]);
          fn(k2 >> 16, ok[j]);
        }
      } else {
        fn(bf16x2_keys(q[j].x) & 0xffffu, ok[j]);
      }
    }
  };
  // high-byte histogram, one atomic per distinct bin and warp step (the sample
  // concentrates in a few bins, so per-lane atomics would mostly collide)
  const int lane = tid & 31;
  for_keys([&](uint32_t key, bool valid) {
    const uint32_t bin = valid ? (key >> 8) : 256u;
    const uint32_t m = __match_any_sync(0xffffffffu, bin);
    if (valid && lane == __ffs(m) - 1) atomicAdd(&whist[warp][bin], (uint32_t)__popc(m));
  });
  __syncthreads();
  for (int i = tid; i < 256; i += kSampleThreads) {
    uint32_t c = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) c += whist[w][i];
    hist[0][i] = c;
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t total = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) total += hist[0][8 * lane + j];
    total = __reduce_add_sync(0xffffffffu, total);
    const double want = 3.0 * (double)total * (double)span / (double)N + 4.0;
    const uint32_t r = want >= (double)total ? total : (uint32_t)want;
    uint32_t b_lo = 256u, b_hi = 0u, r_lo = 1u, r_hi = 1u;
    if (r > 0 && r < total) {
      select_bin(hist[0], r, false, b_lo, r_lo);
      select_bin(hist[0], r, true, b_hi, r_hi);
    }                                            // else too few samples: count everything
    if (lane == 0) { sel[0] = b_lo; sel[1] = b_hi; sel[2] = r_lo; sel[3] = r_hi; }
  }
  __syncthreads();
  const uint32_t s0 = sel[0], s1 = sel[1];
  for_keys([&](uint32_t key, bool valid) {
    if (valid && (key >> 8) == s0) atomicAdd(&hist[1][key & 0xffu], 1u);
    if (valid && (key >> 8) == s1) atomicAdd(&hist[2][key & 0xffu], 1u);
  });
  __syncthreads();
  if (warp == 0) {
    TailInfo ti{0xffffu, 0x10000u, 0u, 0u};
    if (s0 < 256u) {
      uint32_t k_lo, k_hi, rk;
      select_bin(hist[1], sel[2], false, k_lo, rk);
      select_bin(hist[2], sel[3], true, k_hi, rk);
      const uint32_t lo = (s0 << 8) | k_lo, hi = (s1 << 8) | k_hi;
      if (lo + 1u < hi) { ti.key_lo = lo; ti.key_hi = hi; }
    }
    if (lane == 0) tails[h] = ti;
  }
}

// A window: its exact width hi - lo as the unevaluated fp32 sum ws + we (the
// rounded difference and its rounding error, Knuth's TwoSum: exact for the finite
// fp32 differences of two bf16 values), and its keys.  fp32 throughout: this
// GPU's fp64 rate is a small fraction of its fp32 rate.
struct Cand {
  float ws, we;
  uint32_t lo_key;
  uint32_t hi_key;
};

__device__ __forceinline__ Cand make_cand(uint32_t lo_key, uint32_t hi_key) {
  const float b = key_value(hi_key), y = -key_value(lo_key);
  const float s = __fadd_rn(b, y);
  const float bp = __fsub_rn(s, b);
  const float ap = __fsub_rn(s, bp);
  const float e = __fadd_rn(__fsub_rn(b, ap), __fsub_rn(y, bp));
  return Cand{s, e, lo_key, hi_key};
}

// Orders windows by exact width, then by start key: rounding is monotonic, so a
// smaller rounded difference means a smaller exact one, and equal rounded
// differences are ordered by their errors.
__device__ __forceinline__ bool cand_less(const Cand& a, const Cand& b) {
  return a.ws < b.ws || (a.ws == b.ws && (a.we < b.we || (a.we == b.we && a.lo_key < b.lo_key)));
}

__device__ __forceinline__ bool tot_less(float a, float b) {
  return a < b || (a == b && signbit(a) && !signbit(b));
}

__global__ void __launch_bounds__(kWinThreads, 1)
window_kernel(uint32_t* __restrict__ counts, unsigned long long N, unsigned long long t,
              float* __restrict__ min_io, float* __restrict__ max_io, TailInfo* __restrict__ tails, int mode,
              const uint16_t* __restrict__ x, int64_t L, int64_t stride_b, int64_t stride_h, int vec) {
  pdl_wait();
  pdl_launch_dependents();
  // mode 0: tail counts (few windows); mode 1: the heads flagged by mode 0 are
  // counted here in full and searched again, other heads return at once;
  // mode 2: full counts from the histogram kernel, no tail state.
  __shared__ unsigned long long base_s[kWinThreads + 1];
  __shared__ unsigned long long warp_tot[kWinThreads / 32];
  __shared__ Cand warp_best[kWinThreads / 32];
  __shared__ unsigned long long count_lo_s;
  const int h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* ch = counts + (int64_t)h * kBins;
  if (mode == 1 && tails[h].flag == 0u) return;
  if (mode == 1) {
    // Full count of this head (rare): global atomics, one per distinct key and warp step.
    const uint16_t* xh = x + (int64_t)h * stride_h;
    const int64_t units = vec ? (int64_t)N / 8 : (int64_t)N;
    const int nk = vec ? 8 : 1;
    for (int64_t u0 = 0; u0 < units; u0 += kWinThreads) {
      const int64_t u = u0 + tid;
      const bool valid = u < units;
      uint32_t keys[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) keys[i] = 0x10000u;
      if (valid) {
        const int64_t n = u * nk, b = n / L, l = n - b * L;
        if (vec) {
          const uint4 q = *reinterpret_cast<const uint4*>(xh + b * stride_b + l);
          const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t k2 = bf16x2_keys(w[i]);
            keys[2 * i] = k2 & 0xffffu;
            keys[2 * i + 1] = k2 >> 16;
          }
        } else {
          keys[0] = bf16x2_keys(xh[b * stride_b + l]) & 0xffffu;
        }
      }
      for (int i = 0; i < nk; ++i) {
        const uint32_t m = __match_any_sync(0xffffffffu, keys[i]);
        if (keys[i] < 0x10000u && lane == __ffs(m) - 1) atomicAdd(&ch[keys[i]], (uint32_t)__popc(m));
      }
    }
    __syncthreads();
  }
  const uint32_t key_lo = mode == 0 ? tails[h].key_lo : 0xffffu;   // read before thread 0 clears it
  const uint32_t key_hi = mode == 0 ? tails[h].key_hi : 0u;
  // in mode 0 the bins strictly between the tails were never counted: skip reading them
  const uint32_t my_first = (uint32_t)tid * kBinsPerThread, my_last = my_first + kBinsPerThread - 1;
  const bool skip = mode == 0 && key_lo < 0xffffu && my_first > key_lo && my_last < key_hi;

  // 64 consecutive bins per thread (re-read later from L2 rather than held in registers).
  const uint4* src = reinterpret_cast<const uint4*>(ch + tid * kBinsPerThread);
  unsigned long long sum = 0;
  uint32_t any = 0;
#pragma unroll 4
  for (int i = 0; i < kBinsPerThread / 4 && !skip; ++i) {
    const uint4 q = src[i];
    sum += (unsigned long long)q.x + q.y + q.z + q.w;
    any |= q.x | q.y | q.z | q.w;
  }

  // Block-wide exclusive scan of the per-thread sums.
  unsigned long long incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    unsigned long long wv = warp_tot[lane];
    unsigned long long wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - wv;                      // exclusive prefix of warp totals
  }
  __syncthreads();
  unsigned long long base = warp_tot[warp] + incl - sum;
  base_s[tid] = base;
  if (tid == kWinThreads - 1) base_s[kWinThreads] = base + sum;
  __syncthreads();
  bool search = true;
  if (mode == 0) {
    // Only keys <= key_lo and >= key_hi were counted: the N - total uncounted values
    // sit between them, so one virtual bin key_lo + 1 of that size gives every
    // counted bin its true position.  The windows are exact if each tail holds at
    // least N - t + 1 values; otherwise flag the head for the full pass.
    const unsigned long long total = base_s[kWinThreads];
    const unsigned long long span = N - t + 1;
    if (key_lo < 0xffffu) {
      const uint32_t vb = key_lo + 1u;
      const int owner = (int)(vb / kBinsPerThread);
      const unsigned long long M = N - total;
      if (tid == owner) {
        unsigned long long below = base;
        for (uint32_t i = (uint32_t)owner * kBinsPerThread; i < vb; ++i) below += ch[i];
        count_lo_s = below;
        if (M != 0) {
          ch[vb] += (uint32_t)M;            // read back by this thread only
          sum += M;
          any = 1u;
        }
      }
      if (tid > owner) base += M;
      __syncthreads();
      const unsigned long long count_lo = count_lo_s, count_hi = total - count_lo;
      search = count_lo >= span && count_hi >= span;
    }
    if (tid == 0) {
      tails[h].key_lo = 0u;
      tails[h].key_hi = 0u;
      if (!search) tails[h].flag = 1u;
    }
  } else if (mode == 1 && tid == 0) {
    tails[h].flag = 0u;
  }

  Cand best{__int_as_float(0x7f800000), 0.f, 0xffffffffu, 0xffffffffu};
  unsigned long long P = base;
  if (!search) {
    // thin tails: the full pass decides this head
  } else if (N - t + 1 <= (unsigned long long)kCandCap) {
    // Few window starts (ratio near 1).  Table the first position of every value
    // that can start a window, start_tab[position] = its bin, and the bin of every
    // position a window can end at, end_tab[position - (t - 1)]; then window i runs
    // from start_tab[i] to end_tab[i], and all of them are checked in parallel.
    extern __shared__ uint32_t tab[];
    const uint32_t span = (uint32_t)(N - t + 1);
    uint32_t* start_tab = tab;
    uint32_t* end_tab = tab + span;
    for (uint32_t i = tid; i < span; i += kWinThreads) start_tab[i] = 0xffffffffu;
    __syncthreads();
    unsigned long long pos = base;
    if (any != 0 && base < span) {
      for (int q = 0; q < kBinsPerThread / 4; ++q) {
        const uint4 c4 = src[q];
        const uint32_t c[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (c[j] != 0 && pos < span) start_tab[pos] = (uint32_t)(tid * kBinsPerThread + 4 * q + j);
          pos += c[j];
        }
        if (pos >= span) break;
      }
    }
    // end positions live in [t - 1, N); this thread's bins cover [base, base + sum)
    pos = base;
    if (any != 0 && base + sum > t - 1) {
      for (int q = 0; q < kBinsPerThread / 4; ++q) {
        const uint4 c4 = src[q];
        const uint32_t c[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const unsigned long long lo_e = pos > t - 1 ? pos : t - 1, hi_e = pos + c[j];
          const uint32_t bin = (uint32_t)(tid * kBinsPerThread + 4 * q + j);
          for (unsigned long long e = lo_e; e < hi_e; ++e) end_tab[e - (t - 1)] = bin;
          pos = hi_e;
        }
      }
    }
    __syncthreads();
    for (uint32_t i = tid; i < span; i += kWinThreads) {
      const uint32_t v = start_tab[i];
      if (v != 0xffffffffu) {
        const Cand cd = make_cand(v, end_tab[i]);
        if (cand_less(cd, best)) best = cd;
      }
    }
  } else if (any != 0 && base + t <= N) {
    // Candidate windows starting in this thread's bins.
    for (int i = 0; i < kBinsPerThread; ++i) {
      const uint32_t cnt = ch[tid * kBinsPerThread + i];
      if (cnt != 0 && P + t <= N) {
        const unsigned long long e = P + t - 1;     // position of the window's last value
        int lo_s = 0, hi_s = kWinThreads - 1;       // largest segment s with base_s[s] <= e
        while (lo_s < hi_s) {
          const int mid = (lo_s + hi_s + 1) >> 1;
          if (base_s[mid] <= e) lo_s = mid; else hi_s = mid - 1;
        }
        unsigned long long pos = base_s[lo_s];
        uint32_t end_bin = lo_s * kBinsPerThread + kBinsPerThread - 1;
        for (int j = 0; j < kBinsPerThread; ++j) {
          pos += ch[lo_s * kBinsPerThread + j];
          if (e < pos) { end_bin = lo_s * kBinsPerThread + j; break; }
        }
        const Cand cand = make_cand(tid * kBinsPerThread + i, end_bin);
        if (cand_less(cand, best)) best = cand;
      }
      P += cnt;
    }
  }

  // Block argmin (width, then start key).
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Cand other;
    other.ws = __shfl_xor_sync(0xffffffffu, best.ws, o);
    other.we = __shfl_xor_sync(0xffffffffu, best.we, o);
    other.lo_key = __shfl_xor_sync(0xffffffffu, best.lo_key, o);
    other.hi_key = __shfl_xor_sync(0xffffffffu, best.hi_key, o);
    if (cand_less(other, best)) best = other;
  }
  if (lane == 0) warp_best[warp] = best;
  __syncthreads();                                  // also: every read of ch[] is done
  if (warp == 0) {
    best = warp_best[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Cand other;
      other.ws = __shfl_xor_sync(0xffffffffu, best.ws, o);
      other.we = __shfl_xor_sync(0xffffffffu, best.we, o);
      other.lo_key = __shfl_xor_sync(0xffffffffu, best.lo_key, o);
      other.hi_key = __shfl_xor_sync(0xffffffffu, best.hi_key, o);
      if (cand_less(other, best)) best = other;
    }
    if (lane == 0 && best.lo_key != 0xffffffffu) {
      const float lo = key_value(best.lo_key), hi = key_value(best.hi_key);
      if (tot_less(lo, min_io[h])) min_io[h] = lo;
      if (tot_less(max_io[h], hi)) max_io[h] = hi;
    }
  }
  // Leave the workspace zero-filled for the next call (only occupied bins are written).
  if (any != 0) {
    uint4* dst = reinterpret_cast<uint4*>(ch + tid * kBinsPerThread);
    for (int i = 0; i < kBinsPerThread / 4; ++i) {
      const uint4 q = dst[i];
      if (q.x | q.y | q.z | q.w) dst[i] = make_uint4(0, 0, 0, 0);
    }
  }
}

}  // namespace
}  // namespace fa3

using namespace fa3;

FA3_API size_t fa3_calibrate_workspace_size(int H) {
  return H > 0 ? (size_t)H * kBins * sizeof(uint32_t) + (size_t)H * sizeof(TailInfo) : 0;
}

FA3_API int fa3_calibrate_perhead(const uint16_t* x, int64_t B, int H, int64_t L, int64_t stride_b,
                                  int64_t stride_h, double ratio, float* min_io, float* max_io,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (!x || !min_io || !max_io) return FA3_EINVAL;
  if (B <= 0 || H <= 0 || L <= 0 || stride_b < 0 || stride_h < 0) return FA3_EINVAL;
  if (!(ratio > 0.0 && ratio <= 1.0)) return FA3_EINVAL;
  const int64_t N = B * L;
  if (N <= 0 || N >= (int64_t)1 << 32 || L > ((int64_t)1 << 40) / B) return FA3_ERANGE;
  if (H > 65535) return FA3_ERANGE;
  if (!workspace || workspace_bytes < fa3_calibrate_workspace_size(H) || !aligned16(workspace))
    return FA3_EWORKSPACE;
  int st = check_device(nullptr);
  if (st != FA3_OK) return st;
  // FA3量化 step 2: target_num = int(ratio * N), float64 product, truncation; at least 1.
  int64_t t = (int64_t)(ratio * (double)N);
  if (t < 1) t = 1;
  if (t > N) t = N;
  const int vec = (L % 8 == 0) && aligned16(x) && (stride_b % 8 == 0) && (stride_h % 8 == 0);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int smem = kBins * 2;   // 128 KB of 16-bit bins
  if (cudaFuncSetAttribute(hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return FA3_ECUDA;
  const int chunks_per_head = (int)((N + kChunk - 1) / kChunk);
  const int64_t total_chunks = (int64_t)chunks_per_head * H;
  if (total_chunks > (int64_t)1 << 30) return FA3_ERANGE;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0) != cudaSuccess || sms <= 0) sms = 148;
  {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  }
  const unsigned grid = (unsigned)(total_chunks < sms ? total_chunks : sms);
  uint32_t* counts = static_cast<uint32_t*>(workspace);
  TailInfo* tails = reinterpret_cast<TailInfo*>(counts + (size_t)H * kBins);
  const unsigned long long span = (unsigned long long)(N - t + 1);
  const bool fast = span <= (unsigned long long)kCandCap;
  const int wsmem = fast ? (int)(2 * span * sizeof(uint32_t)) : 0;   // start and end tables
  if (wsmem > 48 * 1024 &&
      cudaFuncSetAttribute(window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, wsmem) != cudaSuccess)
    return FA3_ECUDA;
  if (fast) {
    // tails only, then a full pass over the heads whose tails turned out too thin
    if (launch_pdl(tail_kernel, dim3(H), dim3(kSampleThreads), 0, s, x, L, stride_b, stride_h, N, span, vec, tails) !=
        cudaSuccess)
      return FA3_ECUDA;
    timing_begin(s);
    const int64_t per_cta = (int64_t)kTailThreads * kTailGroups;
    const int64_t xb = (L / 8 + per_cta - 1) / per_cta, rows = B * (int64_t)H;
    if (vec && xb <= 0x7fffffff && rows <= 65535) {
      if (launch_pdl(tail_count_kernel, dim3((unsigned)xb, (unsigned)rows), dim3(kTailThreads), 0, s, x, L,
                     stride_b, stride_h, H, counts, static_cast<const TailInfo*>(tails)) != cudaSuccess)
        return FA3_ECUDA;
    } else {
      if (launch_pdl(hist_kernel, dim3(grid), dim3(kHistThreads), smem, s, x, L, stride_b, stride_h, N,
                     chunks_per_head, (int)total_chunks, counts, vec, static_cast<const TailInfo*>(tails)) != cudaSuccess)
        return FA3_ECUDA;
    }
    timing_end(s);
    for (int mode = 0; mode < 2; ++mode)
      if (launch_pdl(window_kernel, dim3(H), dim3(kWinThreads), wsmem, s, counts, (unsigned long long)N,
                     (unsigned long long)t, min_io, max_io, tails, mode, x, L, stride_b, stride_h, vec) != cudaSuccess)
        return FA3_ECUDA;
  } else {
    timing_begin(s);
    if (launch_pdl(hist_kernel, dim3(grid), dim3(kHistThreads), smem, s, x, L, stride_b, stride_h, N,
                   chunks_per_head, (int)total_chunks, counts, vec, static_cast<const TailInfo*>(nullptr)) != cudaSuccess)
      return FA3_ECUDA;
    timing_end(s);
    if (launch_pdl(window_kernel, dim3(H), dim3(kWinThreads), wsmem, s, counts, (unsigned long long)N,
                   (unsigned long long)t, min_io, max_io, tails, 2, x, L, stride_b, stride_h, vec) != cudaSuccess)
      return FA3_ECUDA;
  }
  return cuda_status(cudaGetLastError());
}
