// Per-head Recall-Window calibration.
//
// msModelSlim "FA3量化" page, 原理 / 算法流程:
//   step 1  every head collects its N = B*S*D activation values;
//   step 2  sort them, target_num = int(ratio*N), and keep the narrowest window
//           [sorted[i], sorted[i+target_num-1]] over i = 0 .. N - target_num;
//   step 3  running min/max of the window ends across calibration batches.
//
// GB300 design.  bf16 has only 65536 bit patterns, and a monotone 16-bit key
// maps them onto the total order of their values (-0 before +0), so counting
// keys (a counting sort) carries the whole sorted sequence and one pass over HBM
// replaces the sort.  Two paths, both exact:
//
// Tail-list path (few windows: N - target_num + 1 small, e.g. the pages' ratio
// 0.9999).  Every window then starts among the N - t + 1 smallest values and
// ends among as many largest, so only the two tails of a head matter.
//   tail_pick_kernel  per head: tail thresholds from a fixed sample of the head
//             (16 runs of 2 KB), the r-th smallest of the sampling threads' minima
//             and the r-th largest of their maxima.
//   tail_stream_kernel  one persistent CTA per SM takes every G-th 64 KB piece of
//             the input; each warp streams its 4 KB slice of every piece with bulk
//             copies through its own 3-slot ring, rules out most values with packed
//             bf16 min/max tests, and stages the keys beyond its head's thresholds
//             (tagged with their piece) until the CTA moves them into two per-head
//             lists.
//   window_kernel  per head: counts the listed keys into a shared-memory
//             histogram, prefix sums give each listed key its rank, and the
//             windows i = 0 .. N - t pair the i-th smallest listed key with the
//             matching one of the largest.  A head whose tails turn out too thin
//             (fewer than N - t + 1 values in a list), whose lists overflow, or
//             whose sample was degenerate is counted in full by the same CTA and
//             searched like the histogram path's heads.
// Histogram path (many windows, or input rows not 16-byte aligned):
//   hist_kernel  persistent CTAs walk (head, 65528-value chunk) pairs: a 65536-bin
//             histogram of 16-bit counters packed two per word in 128 KB of
//             shared memory (a chunk is shorter than 65536, so no counter can
//             overflow), flushed into the per-head u32 table in the workspace.
//   window_kernel  per head: prefix sums over the 65536 bins; a window can only
//             be narrowest if it starts at the first copy of a value, so each
//             occupied bin v with start position P(v) <= N - t is a candidate
//             whose window ends in the bin holding position P(v) + t - 1.
// Widths are exact (fp32 TwoSum pairs), the argmin takes ties to the smallest
// start, and the running min/max update follows.  Every call leaves the
// workspace zero-filled again for the next one.
#include "fa3_common.cuh"
#include "fa3_tc.cuh"

#include <math_constants.h>

namespace fa3 {
namespace {

constexpr int kBins = 65536;
// histogram path
constexpr int kHistThreads = 1024;
constexpr int kChunk = 65528;                       // values per histogram CTA (multiple of 8, < 65536)
constexpr int kGroupsPerThread = (kChunk / 8 + kHistThreads - 1) / kHistThreads;   // 8
constexpr int kScalarPerThread = (kChunk + kHistThreads - 1) / kHistThreads;       // 64
// window search
constexpr int kWinThreads = 1024;
constexpr int kBinsPerThread = kBins / kWinThreads;  // 64
constexpr int kCandCap = 16384;     // window starts the table search handles (N - t + 1 <= kCandCap)
// tail-list path
constexpr int kStreamThreads = 512;
constexpr int kStreamWarps = kStreamThreads / 32;
constexpr int kStageBytes = 65536;  // one piece of a row
constexpr int kStages = 3;          // ring depth (per warp: each warp streams its own slices)
constexpr int kSliceBytes = kStageBytes / kStreamWarps;              // a warp's 4 KB share of a piece
constexpr int kGroupsPerStage = kStageBytes / 16 / kStreamThreads;   // 8 groups of 8 values per lane
constexpr int kListCap = 16384;     // tail keys per list and head in the workspace
constexpr int kSampleGroups = 2048; // strided 16-byte groups per head for the tail thresholds
constexpr int kMaxRank = 64;        // largest sample rank the tail thresholds are drawn at
// ring, then the staged keys (kStagedCap words)
constexpr size_t kStreamSmem = (size_t)kStages * kStageBytes + 8192 * sizeof(uint32_t);
static_assert(kGroupsPerStage == 8, "the per-thread min / max tree below takes eight groups");

// Per-head state of the tail-list path, in the workspace after the counters:
// n_lo / n_hi: keys appended to the low / high list (may exceed kListCap: then
// the lists are incomplete); flag: the head's sample was degenerate, or a bounded
// wait gave up (the head is then counted in full); keys: the tail thresholds
// tail_pick_kernel drew.  The window kernel reads and
// re-zeroes it.
struct TailInfo {
  uint32_t n_lo, n_hi, flag, keys;   // keys: the thresholds, key_lo | key_hi << 16
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

// Counts the 8 values of one 16-byte group.  When the whole warp holds one and
// the same 16 bytes made of a single repeated value (a constant head), one lane
// adds 256 at once instead of 256 conflicting atomics.
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
    const int cn = ci + gridDim.x;
    if (vec && cn < total_chunks) load_chunk(cn, v);
    // flush the non-zero counters into the head's table and clear them
    uint32_t* ch = counts + (int64_t)h * kBins;
    for (int i = tid; i < kBins / 8; i += kHistThreads) {
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

// Shared state of tail_stream_kernel beside its dynamic buffers.
struct StreamShared {
  uint64_t full[kStreamWarps][kStages];  // a warp's ring slot filled (bulk copy bytes landed)
  uint32_t tag_cnt[128];           // flush: staged keys per tag, then the next free position per tag
  uint32_t tag_base[128];          // flush: the list position reserved for each tag
  uint32_t n_staged;               // keys staged since the last flush (may pass the capacity)
  uint32_t abort;                  // a bounded wait gave up: stop using the ring
};

// Tail thresholds, one CTA per head (tail_pick_kernel).  The sample: kSampleGroups
// 16-byte groups of the head in 16 runs of 128 consecutive groups (run r starts at
// group r * (N / 8) / 16, wrapping past the end), so that each run reads whole
// DRAM pages.  Thread t reads eight groups of run t / 16.  (A small CTA: it can
// share an SM with the stream kernel's CTA, whose ring loads start meanwhile.)
constexpr int kPickThreads = 256;
constexpr int kPickWarps = kPickThreads / 32;
constexpr int kSampleRuns = 16;
constexpr int kRunThreads = kPickThreads / kSampleRuns;        // 16 threads per run
constexpr int kSampleUnits = kSampleGroups / kPickThreads;     // 8 groups per thread
static_assert(kSampleGroups == kSampleRuns * kRunThreads * kSampleUnits, "sample layout");

// key_lo = the r-th smallest of the threads' sample minima (64 keys each), key_hi
// = the r-th largest of their maxima (searches over the 16-bit keys, a hex digit
// per step, counted with ballots).  r threads hold a sampled key at or below
// key_lo, so at least r of the S sampled keys are; for r well below the thread
// count it sits near the sample's r-th smallest key.  With p = (N - t + 1) / N and
// r = 3 S p + 4, the low list (keys <= key_lo) then holds the N - t + 1 smallest
// values of the head unless the sample over-represents the low tail badly (the
// window kernel checks and falls back); likewise the high list.  Thresholds that
// meet mark the head degenerate (flag 1: counted in full).
__global__ void __launch_bounds__(kPickThreads, 1)
tail_pick_kernel(const uint16_t* __restrict__ x, int64_t L, int64_t stride_b, int64_t stride_h,
                 unsigned long long N, uint32_t r, TailInfo* __restrict__ tails) {
  __shared__ uint32_t part[2][kPickWarps][32];
  pdl_wait();
  pdl_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, h = blockIdx.x;
  const uint16_t* xh = x + (int64_t)h * stride_h;
  const unsigned long long units = N / 8;
  // this thread's groups: run0 + (tid % 16) + 16 j; one division for the first, then
  // steps of 128 values along the row (and on to the next row, or back to the first)
  const unsigned long long u0 =
      ((unsigned long long)(tid / kRunThreads) * units / kSampleRuns + (tid % kRunThreads)) % units;
  int64_t b = (int64_t)(u0 * 8) / L, l = (int64_t)(u0 * 8) - b * L;
  const int64_t rows = (int64_t)(N / (unsigned long long)L);
  uint4 q[kSampleUnits];
#pragma unroll
  for (int j = 0; j < kSampleUnits; ++j) {
    q[j] = *reinterpret_cast<const uint4*>(xh + b * stride_b + l);
    l += 8 * kRunThreads;
    while (l >= L) {
      l -= L;
      if (++b == rows) b = 0;
    }
  }
  uint32_t mn = 0xffffu, mx = 0u;
#pragma unroll
  for (int j = 0; j < kSampleUnits; ++j) {
    const uint32_t w[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t k2 = bf16x2_keys(w[i]), a = k2 & 0xffffu, c = k2 >> 16;
      mn = min(mn, min(a, c));
      mx = max(mx, max(a, c));
    }
  }
  // radix-16 searches, one hex digit of both keys per step: lane i of each warp
  // counts the threads whose minimum is at most (prefix, digit i, then all ones),
  // lane 16 + i those whose maximum is at least (prefix, digit i + 1, then zeros)
  uint32_t a_lo = 0u, a_hi = 0u;
#pragma unroll 1
  for (int st = 0; st < 4; ++st) {
    const int shift = 12 - 4 * st;
    const uint32_t ones = (1u << shift) - 1u;
    uint32_t mine = 0u;
#pragma unroll
    for (int i = 0; i < 15; ++i) {
      const uint32_t bl = __ballot_sync(0xffffffffu, mn <= (a_lo | ((uint32_t)i << shift) | ones));
      const uint32_t bh = __ballot_sync(0xffffffffu, mx >= (a_hi | ((uint32_t)(i + 1) << shift)));
      if (lane == i) mine = (uint32_t)__popc(bl);
      if (lane == 16 + i) mine = (uint32_t)__popc(bh);
    }
    part[st & 1][warp][lane] = mine;
    __syncthreads();
    uint32_t tot = 0u;
#pragma unroll
    for (int w = 0; w < kPickWarps; ++w) tot += part[st & 1][w][lane];
    const uint32_t okl = __ballot_sync(0xffffffffu, lane < 15 && tot >= r);
    const uint32_t okh = __ballot_sync(0xffffffffu, lane >= 16 && lane < 31 && tot >= r);
    a_lo |= (okl ? (uint32_t)(__ffs(okl) - 1) : 15u) << shift;          // smallest digit reaching r
    a_hi |= (okh ? (uint32_t)(31 - __clz(okh) - 15) : 0u) << shift;     // largest digit reaching r
  }
  if (tid == 0) {
    tails[h].keys = a_lo | (a_hi << 16);
    if (!(a_lo + 1u < a_hi)) tails[h].flag = 1u;
  }
}

// Staged tail keys of a CTA: one list of key | tag << 16, the tag naming the
// CTA's item (its position k in the CTA's sequence, modulo kTagItems) and the side
// (low list 0, high list 1): tag = 2 (k mod kTagItems) + side.
constexpr int kTagItems = 64;                 // items staged between two flushes
constexpr int kTags = 2 * kTagItems;
constexpr int kStagedCap = 8192;              // staged keys per CTA between two flushes

// Stages one tail key (one lane; the keys are rare).  Keys past kStagedCap go
// straight to the head's list, one reservation each.
__device__ __forceinline__ void stage_key(uint32_t* staged, uint32_t* n_staged, uint32_t tag, uint32_t key,
                                          TailInfo* ti, uint16_t* list, int side) {
  const uint32_t pos = atomicAdd(n_staged, 1u);
  if (pos < (uint32_t)kStagedCap) {
    staged[pos] = key | (tag << 16);
  } else {
    const uint32_t p = atomicAdd(side ? &ti->n_hi : &ti->n_lo, 1u);
    if (p < (uint32_t)kListCap) list[side * kListCap + p] = (uint16_t)key;
  }
}

// Packed bf16 compares, 0xffff per true half (IEEE: -0 == +0).
__device__ __forceinline__ uint32_t ble2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("set.le.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bge2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Tail-list pass (16-byte aligned rows).  The input is cut into items of up to
// kStageBytes of one row, numbered head-major (head, batch row, piece); CTA g of G
// takes items g, g + G, g + 2 G, ... (spread over all heads and addresses, so the
// CTAs finish together).  Warp w handles the 4 KB slice w of every item: its lane
// 0 streams the slices with bulk copies into the warp's own kStages-slot ring (one
// mbarrier per slot), so the warps run independently; tail keys are staged with a
// tag naming their item and side, and every kTagItems items the CTA meets once to
// move them into the heads' lists.  A bounded wait that gives up flags every head
// of the CTA for the full count, so the result stays exact.
struct ItemMap {                    // item i -> (head h, batch row b, piece c)
  DivU32 per_head, pieces;
  uint32_t n_pieces, n_per_head;
};
__device__ __forceinline__ void item_coords(uint32_t i, const ItemMap& m, uint32_t& h, uint32_t& b, uint32_t& c) {
  h = divu32(i, m.per_head);
  const uint32_t r = i - h * m.n_per_head;
  b = divu32(r, m.pieces);
  c = r - b * m.n_pieces;
}

// Moves the CTA's staged keys into the heads' lists (block-wide): counts per tag,
// one reservation per tag in its head's list, then every key to its place.  Tag t
// belongs to the CTA's item k0 + t / 2.
__device__ void flush_staged(const uint32_t* staged, StreamShared& sh, int k0, uint32_t g, uint32_t G,
                             const ItemMap& m, TailInfo* __restrict__ tails, uint16_t* __restrict__ lists) {
  const int tid = threadIdx.x;
  __syncthreads();
  const uint32_t n = min(sh.n_staged, (uint32_t)kStagedCap);
  for (uint32_t e = tid; e < n; e += kStreamThreads) atomicAdd(&sh.tag_cnt[staged[e] >> 16], 1u);
  __syncthreads();
  if (tid < kTags) {
    const uint32_t c = sh.tag_cnt[tid];
    if (c != 0u) {
      uint32_t h, b, pc;
      item_coords(g + (uint32_t)(k0 + tid / 2) * G, m, h, b, pc);
      sh.tag_base[tid] = atomicAdd((tid & 1) ? &tails[h].n_hi : &tails[h].n_lo, c);
    }
    sh.tag_cnt[tid] = 0u;
  }
  __syncthreads();
  for (uint32_t e = tid; e < n; e += kStreamThreads) {
    const uint32_t v = staged[e], t = v >> 16;
    const uint32_t pos = sh.tag_base[t] + atomicAdd(&sh.tag_cnt[t], 1u);
    if (pos < (uint32_t)kListCap) {
      uint32_t h, b, pc;
      item_coords(g + (uint32_t)(k0 + (int)t / 2) * G, m, h, b, pc);
      lists[((size_t)h * 2 + (t & 1)) * kListCap + pos] = (uint16_t)(v & 0xffffu);
    }
  }
  __syncthreads();
  if (tid < kTags) sh.tag_cnt[tid] = 0u;
  if (tid == 0) sh.n_staged = 0u;
  __syncthreads();
}

__global__ void __launch_bounds__(kStreamThreads, 1)
tail_stream_kernel(const uint16_t* __restrict__ x, int64_t stride_b, int64_t stride_h, uint32_t total_items,
                   ItemMap m, uint32_t last_bytes, TailInfo* __restrict__ tails, uint16_t* __restrict__ lists) {
  extern __shared__ __align__(128) uint8_t sm_stream[];
  uint32_t* staged = reinterpret_cast<uint32_t*>(sm_stream + kStages * kStageBytes);   // [kStagedCap]
  __shared__ StreamShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t* ring = sm_stream + warp * kStages * kSliceBytes;                           // this warp's slots
  const uint32_t g = blockIdx.x, G = gridDim.x;
  const int n_items = (int)((total_items - g + G - 1) / G);
  if (tid < kTags) sh.tag_cnt[tid] = 0u;
  if (tid == 0) {
    sh.n_staged = 0u;
    sh.abort = 0u;
  }
  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&sh.full[warp][s]), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();                                      // the warp's barriers are initialised

  // this warp's slice of item k of the CTA (bytes, source)
  auto slice = [&](int k, const uint8_t*& src) {
    uint32_t h, b, c;
    item_coords(g + (uint32_t)k * G, m, h, b, c);
    const int32_t r = (int32_t)(c == m.n_pieces - 1 ? last_bytes : (uint32_t)kStageBytes) - warp * kSliceBytes;
    src = reinterpret_cast<const uint8_t*>(x + (int64_t)b * stride_b + (int64_t)h * stride_h) +
          (size_t)c * kStageBytes + (size_t)warp * kSliceBytes;
    return (uint32_t)(r <= 0 ? 0 : (r < kSliceBytes ? r : kSliceBytes));
  };
  int q_next = 0;
  auto produce = [&]() {                             // lane 0: this warp's slice of item q_next
    const int slot = q_next % kStages;
    const uint8_t* src;
    const uint32_t bytes = slice(q_next, src);
    const uint32_t bar = smem_u32(&sh.full[warp][slot]);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the warp's reads of the slot came first
    mbar_expect_tx(bar, bytes);                      // (a zero-byte slice completes the phase at once)
    if (bytes) bulk_g2s(smem_u32(ring + slot * kSliceBytes), src, bytes, bar);
    ++q_next;
  };
  // The ring's first loads go out while tail_pick_kernel (the grid this one
  // depends on) runs: the input is complete by then, because that grid lets this
  // one start only after its own wait for the work before it.  The workspace is
  // touched only after the wait below.
  if (lane == 0)
    for (int s = 0; s < kStages && s < n_items; ++s) produce();
  pdl_wait();
  pdl_launch_dependents();
  __syncthreads();                                   // the staging counters are initialised

  // thresholds of item k's head, loaded one item ahead
  auto head_info = [&](int k, uint32_t& h) {
    uint32_t b, c;
    item_coords(g + (uint32_t)k * G, m, h, b, c);
    return *reinterpret_cast<const uint4*>(&tails[h]);
  };
  uint32_t h_next = 0;
  uint4 ti_next = n_items > 0 ? head_info(0, h_next) : make_uint4(0u, 0u, 1u, 0u);
  int k0 = 0;                                        // first item of the current tag window
  for (int j = 0; j < n_items; ++j) {
    const uint32_t h = h_next;
    const uint4 ti = ti_next;
    if (j + 1 < n_items) ti_next = head_info(j + 1, h_next);
    if (j - k0 == kTagItems) {                       // the tags wrap: move the staged keys out
      flush_staged(staged, sh, k0, g, G, m, tails, lists);
      k0 = j;
    }
    const uint32_t key_lo = ti.w & 0xffffu, key_hi = ti.w >> 16;
    const bool skip = ti.z != 0u;                    // degenerate head: counted in full
    const uint32_t vlo2 = (__float_as_uint(key_value(key_lo)) >> 16) * 0x10001u;
    const uint32_t vhi2 = (__float_as_uint(key_value(key_hi)) >> 16) * 0x10001u;
    // a bf16 pair strictly between the thresholds: stands in for bytes past a short slice
    const uint32_t mid2 = (__float_as_uint(key_value(key_lo + 1u)) >> 16) * 0x10001u;
    const uint32_t tag = 2u * (uint32_t)(j - k0);
    uint16_t* list = lists + (size_t)h * 2 * kListCap;
    const int slot = j % kStages;
    const bool ok = warp_all(wait_bar(smem_u32(&sh.full[warp][slot]), (uint32_t)((j / kStages) & 1), &sh.abort, nullptr));
    uint32_t hh, hb, hc;
    item_coords(g + (uint32_t)j * G, m, hh, hb, hc);
    const int32_t rb = (int32_t)(hc == m.n_pieces - 1 ? last_bytes : (uint32_t)kStageBytes) - warp * kSliceBytes;
    const uint32_t bytes = (uint32_t)(rb <= 0 ? 0 : (rb < kSliceBytes ? rb : kSliceBytes));
    const uint8_t* slot_base = ring + slot * kSliceBytes;
    if (ok && !skip && bytes != 0u) {
      const uint8_t* st = slot_base + 16 * lane;
      // bf16 min / max of each of the lane's groups; the groups past a short slice
      // read as values strictly between the thresholds
      uint32_t gmn[kGroupsPerStage], gmx[kGroupsPerStage];
      if (bytes == (uint32_t)kSliceBytes) {
#pragma unroll
        for (int k = 0; k < kGroupsPerStage; ++k) {
          const uint4 v = *reinterpret_cast<const uint4*>(st + 16 * 32 * k);
          gmn[k] = bmin2(bmin2(v.x, v.y), bmin2(v.z, v.w));
          gmx[k] = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
        }
      } else {
#pragma unroll
        for (int k = 0; k < kGroupsPerStage; ++k) {
          gmn[k] = gmx[k] = mid2;
          if (16u * (uint32_t)(lane + 32 * k) < bytes) {
            const uint4 v = *reinterpret_cast<const uint4*>(st + 16 * 32 * k);
            gmn[k] = bmin2(bmin2(v.x, v.y), bmin2(v.z, v.w));
            gmx[k] = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
          }
        }
      }
      const uint32_t tmn = bmin2(bmin2(bmin2(gmn[0], gmn[1]), bmin2(gmn[2], gmn[3])),
                                 bmin2(bmin2(gmn[4], gmn[5]), bmin2(gmn[6], gmn[7])));
      const uint32_t tmx = bmax2(bmax2(bmax2(gmx[0], gmx[1]), bmax2(gmx[2], gmx[3])),
                                 bmax2(bmax2(gmx[4], gmx[5]), bmax2(gmx[6], gmx[7])));
      // packed IEEE compares: a value at or beyond a threshold's value may be a tail key
      const bool flagged = (ble2(tmn, vlo2) | bge2(tmx, vhi2)) != 0u;
      // rare: the warp's flagged lanes, four at a time, hand their eight groups each
      // to the 32 lanes, which locate the candidates and run the exact key test
      uint32_t pending = __ballot_sync(0xffffffffu, flagged);
      while (pending != 0u) {
        int src = 32;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int l = pending ? __ffs(pending) - 1 : 32;
          if (pending) pending &= pending - 1u;
          if ((lane >> 3) == r) src = l;
        }
        const int k = lane & 7;
        if (src < 32 && 16u * (uint32_t)(src + 32 * k) < bytes) {
          const uint4 gr = *reinterpret_cast<const uint4*>(slot_base + 16 * (src + 32 * k));
          const uint32_t w[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if ((ble2(w[i], vlo2) | bge2(w[i], vhi2)) == 0u) continue;
            const uint32_t k2 = bf16x2_keys(w[i]);
#pragma unroll
            for (int half = 0; half < 2; ++half) {            // the exact test, on keys
              const uint32_t key = half ? k2 >> 16 : k2 & 0xffffu;
              if (key <= key_lo) stage_key(staged, &sh.n_staged, tag, key, tails + h, list, 0);
              else if (key >= key_hi) stage_key(staged, &sh.n_staged, tag + 1u, key, tails + h, list, 1);
            }
          }
        }
      }
    }
    __syncwarp();                                    // the warp is done with the slot: refill it
    if (lane == 0 && q_next < n_items && !*reinterpret_cast<volatile uint32_t*>(&sh.abort)) produce();
  }
  if (lane == 0 && *reinterpret_cast<volatile uint32_t*>(&sh.abort)) {
    // gave up: the heads of the CTA's items are counted in full; the warp's copies
    // still in flight (its last slots filled) get one more bounded wait before exit
    for (int k = 0; k < n_items; ++k) {
      uint32_t h, b, c;
      item_coords(g + (uint32_t)k * G, m, h, b, c);
      tails[h].flag = 1u;
    }
    uint32_t no_abort = 0u;
    for (int jj = q_next > kStages ? q_next - kStages : 0; jj < q_next; ++jj)
      wait_bar(smem_u32(&sh.full[warp][jj % kStages]), (uint32_t)((jj / kStages) & 1), &no_abort, nullptr);
  }
  flush_staged(staged, sh, k0, g, G, m, tails, lists);
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
// differences are ordered by their errors.  Two windows equal in both have the
// same ends, so the order among them does not matter.
__device__ __forceinline__ bool cand_less(const Cand& a, const Cand& b) {
  return a.ws < b.ws || (a.ws == b.ws && (a.we < b.we || (a.we == b.we && a.lo_key < b.lo_key)));
}

__device__ __forceinline__ bool tot_less(float a, float b) {
  return a < b || (a == b && signbit(a) && !signbit(b));
}

__device__ __forceinline__ Cand warp_min_cand(Cand best) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Cand other;
    other.ws = __shfl_xor_sync(0xffffffffu, best.ws, o);
    other.we = __shfl_xor_sync(0xffffffffu, best.we, o);
    other.lo_key = __shfl_xor_sync(0xffffffffu, best.lo_key, o);
    other.hi_key = __shfl_xor_sync(0xffffffffu, best.hi_key, o);
    if (cand_less(other, best)) best = other;
  }
  return best;
}

// Block-wide exclusive prefix of one value per thread (kWinThreads threads).
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* warp_tot, T& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const T wv = warp_tot[lane];
    T wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - wv;                      // exclusive prefix of warp totals
    if (lane == 31) warp_tot[32] = wi;
  }
  __syncthreads();
  total = warp_tot[32];
  return warp_tot[warp] + incl - v;
}

// Narrowest window of a head from its two tail lists (n_lo and n_hi keys, each at
// least span = N - t + 1): the listed keys, sorted, are the n_lo smallest and the
// n_hi largest values of the head, so window i (i < span) starts at listed rank i
// and ends at listed rank n - span + i (n = n_lo + n_hi).  A counting sort in
// shared memory gives the ranks: 16-bit counters of the 65536 keys (thread t owns
// keys [64 t, 64 t + 64), its 32 words padded by 4 so that 16-byte reads of eight
// threads hit distinct banks), turned in place into exclusive prefix sums, then
// every listed key takes its rank with one atomic increment of its key's slot.
constexpr int kPadWords = 36;       // words per thread's 64 counters, padded
__device__ __forceinline__ uint32_t padded_word(uint32_t key) { return (key >> 1) + 4u * (key >> 6); }

__device__ Cand search_lists(const uint16_t* __restrict__ list, uint32_t n_lo, uint32_t n_hi, uint32_t span,
                             uint8_t* dyn, uint32_t* warp_tot) {
  const int tid = threadIdx.x;
  uint32_t* bins = reinterpret_cast<uint32_t*>(dyn);
  uint16_t* start_tab = reinterpret_cast<uint16_t*>(dyn + kWinThreads * kPadWords * 4);
  uint16_t* end_tab = start_tab + span;
  for (int i = tid; i < kWinThreads * kPadWords / 4; i += kWinThreads)
    reinterpret_cast<uint4*>(bins)[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  auto bump = [&](uint32_t key) {       // returns the slot's value before the increment
    const uint32_t sh = (key & 1u) << 4;
    return (atomicAdd(&bins[padded_word(key)], 1u << sh) >> sh) & 0xffffu;
  };
  for (uint32_t i = tid; i < n_lo; i += kWinThreads) bump(list[i]);
  for (uint32_t i = tid; i < n_hi; i += kWinThreads) bump(list[kListCap + i]);
  __syncthreads();
  uint4* own = reinterpret_cast<uint4*>(bins + tid * kPadWords);
  uint32_t sum = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint4 q = own[w];
    sum += (q.x & 0xffffu) + (q.x >> 16) + (q.y & 0xffffu) + (q.y >> 16) + (q.z & 0xffffu) + (q.z >> 16) +
           (q.w & 0xffffu) + (q.w >> 16);
  }
  uint32_t n;
  uint32_t run = block_exclusive_scan<uint32_t>(sum, warp_tot, n);
  // counters -> exclusive prefix sums (ranks of each key's first copy); n < 65536
  auto pre = [&](uint32_t w) {
    const uint32_t lo = run;
    run += w & 0xffffu;
    const uint32_t hi = run;
    run += w >> 16;
    return lo | (hi << 16);
  };
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint4 q = own[w];
    uint4 r;
    r.x = pre(q.x);
    r.y = pre(q.y);
    r.z = pre(q.z);
    r.w = pre(q.w);
    own[w] = r;
  }
  __syncthreads();
  const uint32_t e0 = n - span;                      // rank of the first window's end
  auto place = [&](uint32_t key) {
    const uint32_t rank = bump(key);
    if (rank < span) start_tab[rank] = (uint16_t)key;
    if (rank >= e0) end_tab[rank - e0] = (uint16_t)key;
  };
  for (uint32_t i = tid; i < n_lo; i += kWinThreads) place(list[i]);
  for (uint32_t i = tid; i < n_hi; i += kWinThreads) place(list[kListCap + i]);
  __syncthreads();
  Cand best{__int_as_float(0x7f800000), 0.f, 0xffffffffu, 0xffffffffu};
  for (uint32_t i = tid; i < span; i += kWinThreads) {
    const Cand cd = make_cand(start_tab[i], end_tab[i]);
    if (cand_less(cd, best)) best = cd;
  }
  return best;
}

// Full count of head h into its u32 table (global atomics, one per distinct key
// and warp step): the rare fallback of the tail-list path.
__device__ void count_head_full(uint32_t* __restrict__ ch, const uint16_t* __restrict__ xh, unsigned long long N,
                                int64_t L, int64_t stride_b) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t units = (int64_t)N / 8;
  for (int64_t u0 = 0; u0 < units; u0 += kWinThreads) {
    const int64_t u = u0 + tid;
    uint32_t keys[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) keys[i] = 0x10000u;
    if (u < units) {
      const int64_t n = u * 8, b = n / L, l = n - b * L;
      const uint4 q = *reinterpret_cast<const uint4*>(xh + b * stride_b + l);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t k2 = bf16x2_keys(w[i]);
        keys[2 * i] = k2 & 0xffffu;
        keys[2 * i + 1] = k2 >> 16;
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t m = __match_any_sync(0xffffffffu, keys[i]);
      if (keys[i] < 0x10000u && lane == __ffs(m) - 1) atomicAdd(&ch[keys[i]], (uint32_t)__popc(m));
    }
  }
  __syncthreads();
}

// Narrowest window of a head from its full u32 key table ch (N values, windows of
// t); zeroes the table's occupied words on the way out.
__device__ Cand search_counts(uint32_t* __restrict__ ch, unsigned long long N, unsigned long long t, uint8_t* dyn,
                              unsigned long long* base_s, unsigned long long* warp_tot) {
  const int tid = threadIdx.x;
  // 64 consecutive bins per thread (re-read later from L2 rather than held in registers)
  const uint4* src = reinterpret_cast<const uint4*>(ch + tid * kBinsPerThread);
  unsigned long long sum = 0;
  uint32_t any = 0;
#pragma unroll 4
  for (int i = 0; i < kBinsPerThread / 4; ++i) {
    const uint4 q = src[i];
    sum += (unsigned long long)q.x + q.y + q.z + q.w;
    any |= q.x | q.y | q.z | q.w;
  }
  unsigned long long total;
  const unsigned long long base = block_exclusive_scan<unsigned long long>(sum, warp_tot, total);
  base_s[tid] = base;
  if (tid == kWinThreads - 1) base_s[kWinThreads] = base + sum;
  __syncthreads();

  Cand best{__int_as_float(0x7f800000), 0.f, 0xffffffffu, 0xffffffffu};
  unsigned long long P = base;
  if (N - t + 1 <= (unsigned long long)kCandCap) {
    // Few window starts.  Table the first position of every value that can start
    // a window, start_tab[position] = its bin, and the bin of every position a
    // window can end at, end_tab[position - (t - 1)]; then window i runs from
    // start_tab[i] to end_tab[i], and all of them are checked in parallel.
    const uint32_t span = (uint32_t)(N - t + 1);
    uint32_t* start_tab = reinterpret_cast<uint32_t*>(dyn);
    uint32_t* end_tab = start_tab + span;
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
  __syncthreads();                                  // every read of ch[] is done
  // Leave the table zero-filled for the next call (only occupied words are written).
  if (any != 0) {
    uint4* dst = reinterpret_cast<uint4*>(ch + tid * kBinsPerThread);
    for (int i = 0; i < kBinsPerThread / 4; ++i) {
      const uint4 q = dst[i];
      if (q.x | q.y | q.z | q.w) dst[i] = make_uint4(0, 0, 0, 0);
    }
  }
  return best;
}

// One CTA per head.  lists != nullptr: the tail-list path (a head that cannot be
// decided from its lists is counted in full here); otherwise the u32 table holds
// the head's full counts from hist_kernel.
__global__ void __launch_bounds__(kWinThreads, 1)
window_kernel(uint32_t* __restrict__ counts, unsigned long long N, unsigned long long t,
              float* __restrict__ min_io, float* __restrict__ max_io, TailInfo* __restrict__ tails,
              uint16_t* __restrict__ lists, const uint16_t* __restrict__ x, int64_t L, int64_t stride_b,
              int64_t stride_h) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ unsigned long long base_s[kWinThreads + 1];
  __shared__ unsigned long long warp_tot[33];
  __shared__ uint32_t warp_tot32[33];
  __shared__ Cand warp_best[kWinThreads / 32];
  const int h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* ch = counts + (int64_t)h * kBins;
  const unsigned long long span = N - t + 1;
  Cand best;
  bool full = lists == nullptr;
  if (lists != nullptr) {
    const TailInfo ti = tails[h];
    __syncthreads();
    if (tid == 0) tails[h] = TailInfo{0u, 0u, 0u, 0u};
    const bool decided = ti.flag == 0u && ti.n_lo >= span && ti.n_hi >= span && ti.n_lo <= (uint32_t)kListCap &&
                         ti.n_hi <= (uint32_t)kListCap;
    uint16_t* list = lists + (int64_t)h * 2 * kListCap;
    if (decided) {
      best = search_lists(list, ti.n_lo, ti.n_hi, (uint32_t)span, dyn, warp_tot32);
    } else {
      count_head_full(ch, x + (int64_t)h * stride_h, N, L, stride_b);
      full = true;
    }
    // Zero the list entries the pass wrote (whole 16-byte groups), so the workspace
    // is all zero again, whatever head count the next call lays it out for.
    __syncthreads();
#pragma unroll
    for (int side = 0; side < 2; ++side) {
      const uint32_t n = min(side ? ti.n_hi : ti.n_lo, (uint32_t)kListCap);
      uint4* dst = reinterpret_cast<uint4*>(list + side * kListCap);
      for (uint32_t i = tid; i < (n + 7) / 8; i += kWinThreads) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (full) best = search_counts(ch, N, t, dyn, base_s, warp_tot);

  // Block argmin (width, then start key).
  best = warp_min_cand(best);
  if (lane == 0) warp_best[warp] = best;
  __syncthreads();
  if (warp == 0) {
    best = warp_min_cand(warp_best[lane]);
    if (lane == 0 && best.lo_key != 0xffffffffu) {
      const float lo = key_value(best.lo_key), hi = key_value(best.hi_key);
      if (tot_less(lo, min_io[h])) min_io[h] = lo;
      if (tot_less(max_io[h], hi)) max_io[h] = hi;
    }
  }
}

}  // namespace
}  // namespace fa3

using namespace fa3;

namespace {
size_t counts_bytes(int H) { return (size_t)H * kBins * sizeof(uint32_t); }
size_t tails_bytes(int H) { return (size_t)H * sizeof(TailInfo); }
}  // namespace

FA3_API size_t fa3_calibrate_workspace_size(int H) {
  return H > 0 ? counts_bytes(H) + tails_bytes(H) + (size_t)H * 2 * kListCap * sizeof(uint16_t) : 0;
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
  int sms = 0;
  int st = check_device(&sms);
  if (st != FA3_OK) return st;
  if (sms <= 0) sms = 148;
  // FA3量化 step 2: target_num = int(ratio * N), float64 product, truncation; at least 1.
  int64_t t = (int64_t)(ratio * (double)N);
  if (t < 1) t = 1;
  if (t > N) t = N;
  const int vec = (L % 8 == 0) && aligned16(x) && (stride_b % 8 == 0) && (stride_h % 8 == 0);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* counts = static_cast<uint32_t*>(workspace);
  TailInfo* tails = reinterpret_cast<TailInfo*>(static_cast<uint8_t*>(workspace) + counts_bytes(H));
  uint16_t* lists = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + counts_bytes(H) + tails_bytes(H));
  const unsigned long long span = (unsigned long long)(N - t + 1);
  // Tail lists when both can be expected well inside their capacity: with S
  // sampled keys, r = int(3 S (N - t + 1) / N + 4) sampled keys lie in each tail,
  // which then holds about N r / S values; r must stay well below the thread
  // count for the thresholds to track the sample's order statistics.
  constexpr double kS = 8.0 * kSampleGroups;
  const double r_want = 3.0 * kS * (double)span / (double)N + 4.0;
  const uint32_t rank = r_want >= kS ? (uint32_t)kS : (uint32_t)r_want;
  const bool use_lists = vec && rank <= (uint32_t)kMaxRank && (double)N * rank / kS <= 0.5 * kListCap;
  const int64_t pieces = (2 * L + kStageBytes - 1) / kStageBytes;
  const int64_t total_items = pieces * B * H;
  if (use_lists && total_items < ((int64_t)1 << 31)) {
    const unsigned grid = (unsigned)(total_items < sms ? total_items : sms);
    ItemMap m;
    m.n_pieces = (uint32_t)pieces;
    m.n_per_head = (uint32_t)(pieces * B);
    m.pieces = make_divu32(m.n_pieces);
    m.per_head = make_divu32(m.n_per_head);
    const uint32_t last_bytes = (uint32_t)(2 * L - (pieces - 1) * kStageBytes);
    if (cudaFuncSetAttribute(tail_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStreamSmem) !=
        cudaSuccess)
      return FA3_ECUDA;
    // padded counters and tables of the list search; the same bytes hold the u32
    // tables of a head that falls back to its full count (8 * span fits)
    const int wsmem = (int)(kWinThreads * kPadWords * 4 + 4 * span);
    if (cudaFuncSetAttribute(window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, wsmem) != cudaSuccess)
      return FA3_ECUDA;
    // the pick kernel's CTAs share SMs with the stream kernel's, whose ring needs
    // nearly all of the shared memory: ask for the same carve-out
    if (cudaFuncSetAttribute(tail_pick_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
      return FA3_ECUDA;
    if (launch_pdl(tail_pick_kernel, dim3(H), dim3(kPickThreads), 0, s, x, L, stride_b, stride_h,
                   (unsigned long long)N, rank, tails) != cudaSuccess)
      return FA3_ECUDA;
    timing_begin(s);
    if (launch_pdl(tail_stream_kernel, dim3(grid), dim3(kStreamThreads), kStreamSmem, s, x, stride_b, stride_h,
                   (uint32_t)total_items, m, last_bytes, tails, lists) != cudaSuccess)
      return FA3_ECUDA;
    timing_end(s);
    if (launch_pdl(window_kernel, dim3(H), dim3(kWinThreads), wsmem, s, counts, (unsigned long long)N,
                   (unsigned long long)t, min_io, max_io, tails, lists, x, L, stride_b,
                   stride_h) != cudaSuccess)
      return FA3_ECUDA;
  } else {
    const int smem = kBins * 2;   // 128 KB of 16-bit bins
    if (cudaFuncSetAttribute(hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return FA3_ECUDA;
    const int chunks_per_head = (int)((N + kChunk - 1) / kChunk);
    const int64_t total_chunks = (int64_t)chunks_per_head * H;
    if (total_chunks > (int64_t)1 << 30) return FA3_ERANGE;
    const unsigned grid = (unsigned)(total_chunks < sms ? total_chunks : sms);
    const int wsmem = span <= (unsigned long long)kCandCap ? (int)(8 * span) : 0;   // start and end tables
    if (wsmem > 48 * 1024 &&
        cudaFuncSetAttribute(window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, wsmem) != cudaSuccess)
      return FA3_ECUDA;
    timing_begin(s);
    if (launch_pdl(hist_kernel, dim3(grid), dim3(kHistThreads), smem, s, x, L, stride_b, stride_h, N,
                   chunks_per_head, (int)total_chunks, counts, vec) != cudaSuccess)
      return FA3_ECUDA;
    timing_end(s);
    if (launch_pdl(window_kernel, dim3(H), dim3(kWinThreads), wsmem, s, counts, (unsigned long long)N,
                   (unsigned long long)t, min_io, max_io, tails, static_cast<uint16_t*>(nullptr), x, L,
                   stride_b, stride_h) != cudaSuccess)
      return FA3_ECUDA;
  }
  return cuda_status(cudaGetLastError());
}
