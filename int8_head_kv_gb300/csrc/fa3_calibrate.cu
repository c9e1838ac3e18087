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
//             P(v) + target_num - 1.  Width in float64, argmin with ties to the
//             smallest start, then the running min/max update.  The kernel
//             zeroes the bins it read, leaving the workspace clean.
#include "fa3_common.cuh"

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

// Counts the 8 values of one 16-byte group.  When the whole warp holds one and the
// same 16 bytes made of a single repeated value (a constant head), one lane adds
// 256 at once instead of 256 conflicting atomics.
__device__ __forceinline__ void count_group(uint32_t* bins, const uint4 v, bool valid) {
  const uint32_t w0 = __shfl_sync(0xffffffffu, v.x, 0);
  const bool uniform = __all_sync(0xffffffffu, valid && v.x == w0 && v.y == w0 && v.z == w0 && v.w == w0 &&
                                                   (w0 >> 16) == (w0 & 0xffffu));
  if (uniform) {
    if ((threadIdx.x & 31) == 0) {
      const uint32_t key = bf16x2_keys(w0) & 0xffffu;
      atomicAdd(&bins[key >> 1], 256u << ((key & 1u) << 4));
    }
    return;
  }
  if (!valid) return;
  const uint32_t k[4] = {bf16x2_keys(v.x), bf16x2_keys(v.y), bf16x2_keys(v.z), bf16x2_keys(v.w)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    count16(bins, k[i] & 0xffffu);
    count16(bins, k[i] >> 16);
  }
}

// Persistent: CTA g walks chunks g, g + gridDim.x, ... of the (head, chunk) list.
// While the histogram of one chunk is flushed (and re-zeroed in the same pass),
// the loads of the next chunk are already in flight.
__global__ void __launch_bounds__(kHistThreads, 1)
hist_kernel(const uint16_t* __restrict__ x, int64_t L, int64_t stride_b, int64_t stride_h, int64_t N,
            int chunks_per_head, int total_chunks, uint32_t* __restrict__ counts, int vec) {
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
#pragma unroll
    for (int k = 0; k < kGroupsPerThread; ++k) {
      v[k] = make_uint4(0, 0, 0, 0);
      const int64_t n = n0 + 8 * (int64_t)(tid + k * kHistThreads);
      if (n < n1) {
        const int64_t b = n / L, l = n - b * L;
        v[k] = __ldcs(reinterpret_cast<const uint4*>(xh + b * stride_b + l));
      }
    }
  };

  uint4 v[kGroupsPerThread];
  int ci = blockIdx.x;
  if (vec && ci < total_chunks) load_chunk(ci, v);
  __syncthreads();
  for (; ci < total_chunks; ci += gridDim.x) {
    int h; int64_t n0, n1;
    chunk_span(ci, h, n0, n1);
    if (vec) {
#pragma unroll
      for (int k = 0; k < kGroupsPerThread; ++k) {
        const int64_t n = n0 + 8 * (int64_t)(tid + k * kHistThreads);
        count_group(bins, v[k], n < n1);
      }
    } else {
      const uint16_t* xh = x + (int64_t)h * stride_h;
      for (int k = 0; k < kScalarPerThread; ++k) {
        const int64_t n = n0 + tid + (int64_t)k * kHistThreads;
        if (n < n1) {
          const int64_t b = n / L, l = n - b * L;
          count16(bins, bf16x2_keys(xh[b * stride_b + l]) & 0xffffu);
        }
      }
    }
    __syncthreads();
    if (vec && ci + (int)gridDim.x < total_chunks) load_chunk(ci + gridDim.x, v);
    // flush the non-zero counters into the head's table and clear them
    uint32_t* ch = counts + (int64_t)h * kBins;
    for (int i = tid; i < kBins / 8; i += kHistThreads) {
      const uint4 q = smem_hist[i];
      if ((q.x | q.y | q.z | q.w) == 0u) continue;
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t lo = w[j] & 0xffffu, hi = w[j] >> 16;
        if (lo) atomicAdd(&ch[8 * i + 2 * j], lo);
        if (hi) atomicAdd(&ch[8 * i + 2 * j + 1], hi);
      }
      smem_hist[i] = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
  }
}

struct Cand {
  double width;
  uint32_t lo_key;
  uint32_t hi_key;
};

__device__ __forceinline__ bool cand_less(const Cand& a, const Cand& b) {
  return a.width < b.width || (a.width == b.width && a.lo_key < b.lo_key);
}

__device__ __forceinline__ bool tot_less(float a, float b) {
  return a < b || (a == b && signbit(a) && !signbit(b));
}

__global__ void __launch_bounds__(kWinThreads, 1)
window_kernel(uint32_t* __restrict__ counts, unsigned long long N, unsigned long long t,
              float* __restrict__ min_io, float* __restrict__ max_io) {
  __shared__ unsigned long long base_s[kWinThreads + 1];
  __shared__ unsigned long long warp_tot[kWinThreads / 32];
  __shared__ Cand warp_best[kWinThreads / 32];
  const int h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* ch = counts + (int64_t)h * kBins;

  // 64 consecutive bins per thread (re-read later from L2 rather than held in registers).
  const uint4* src = reinterpret_cast<const uint4*>(ch + tid * kBinsPerThread);
  unsigned long long sum = 0;
  uint32_t any = 0;
#pragma unroll 4
  for (int i = 0; i < kBinsPerThread / 4; ++i) {
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
  const unsigned long long base = warp_tot[warp] + incl - sum;
  base_s[tid] = base;
  if (tid == kWinThreads - 1) base_s[kWinThreads] = base + sum;
  __syncthreads();

  Cand best{__longlong_as_double(0x7ff0000000000000LL), 0xffffffffu, 0xffffffffu};
  unsigned long long P = base;
  if (N - t + 1 <= (unsigned long long)kCandCap) {
    // Few window starts (ratio near 1): table the first position of every value that
    // can start a window, cand[position] = its bin; then each bin w looks up the
    // starts whose window ends inside w: start position = end position - (t - 1).
    extern __shared__ uint32_t cand[];
    const uint32_t span = (uint32_t)(N - t + 1);
    for (uint32_t i = tid; i < span; i += kWinThreads) cand[i] = 0xffffffffu;
    __syncthreads();
    unsigned long long pos = base;
    if (any != 0 && base < span) {
      for (int q = 0; q < kBinsPerThread / 4; ++q) {
        const uint4 c4 = src[q];
        const uint32_t c[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (c[j] != 0 && pos < span) cand[pos] = (uint32_t)(tid * kBinsPerThread + 4 * q + j);
          pos += c[j];
        }
        if (pos >= span) break;
      }
    }
    __syncthreads();
    // end positions live in [t - 1, N); this thread's bins cover [base, base + sum)
    pos = base;
    if (any != 0 && base + sum > t - 1) {
      for (int q = 0; q < kBinsPerThread / 4; ++q) {
        const uint4 c4 = src[q];
        const uint32_t c[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const unsigned long long lo_e = pos > t - 1 ? pos : t - 1, hi_e = pos + c[j];
          for (unsigned long long e = lo_e; e < hi_e; ++e) {
            const uint32_t v = cand[e - (t - 1)];
            if (v != 0xffffffffu) {
              const uint32_t end_bin = (uint32_t)(tid * kBinsPerThread + 4 * q + j);
              const double w = (double)key_value(end_bin) - (double)key_value(v);
              const Cand cd{w, v, end_bin};
              if (cand_less(cd, best)) best = cd;
            }
          }
          pos = hi_e;
        }
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
        const uint32_t start_bin = tid * kBinsPerThread + i;
        const double w = (double)key_value(end_bin) - (double)key_value(start_bin);
        const Cand cand{w, start_bin, end_bin};
        if (cand_less(cand, best)) best = cand;
      }
      P += cnt;
    }
  }

  // Block argmin (width, then start key).
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Cand other;
    other.width = __shfl_xor_sync(0xffffffffu, best.width, o);
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
      other.width = __shfl_xor_sync(0xffffffffu, best.width, o);
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
  return H > 0 ? (size_t)H * kBins * sizeof(uint32_t) : 0;
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
  timing_begin(s);
  hist_kernel<<<grid, kHistThreads, smem, s>>>(x, L, stride_b, stride_h, N, chunks_per_head, (int)total_chunks,
                                                counts, vec);
  timing_end(s);
  if (cudaGetLastError() != cudaSuccess) return FA3_ECUDA;
  const bool fast = (uint64_t)(N - t + 1) <= (uint64_t)kCandCap;
  const int wsmem = fast ? (int)((N - t + 1) * sizeof(uint32_t)) : 0;
  if (wsmem > 48 * 1024 &&
      cudaFuncSetAttribute(window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, wsmem) != cudaSuccess)
    return FA3_ECUDA;
  window_kernel<<<H, kWinThreads, wsmem, s>>>(counts, (unsigned long long)N, (unsigned long long)t, min_io, max_io);
  return cuda_status(cudaGetLastError());
}
