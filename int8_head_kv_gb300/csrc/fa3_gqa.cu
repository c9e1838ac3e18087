// GQA decode attention over an INT8 KV cache with INT8 queries.
//
// MindIE "Attention Quantization", Overview, and MindIE Turbo "Attention量化":
// q, k and v are quantized to 8 bits per head and the decode-phase attention
// reads them directly; deq_scale restores floating point.  Scales are the
// per-head symmetric ones of msModelSlim "FA3量化" 原理 / 算法流程 step 4.
//
// The path is HBM-bound (about 16 operations per KV byte):
//   * grid = (split, kv head g, batch b); per CTA one producer warp and 4 consumer
//     warps; the CTA's token range is cut into 64-token tiles and consumer warp w
//     takes 16-token step w of every tile, with its own online softmax;
//   * the producer's lane 0 streams the tiles through a 3-stage ring in shared
//     memory with TMA tensor copies (one 64-row box of K and one of V per tile, or
//     page-sized boxes of a paged pool), 128-byte swizzled so that the fragment
//     loads are free of bank conflicts; full / empty mbarriers pace the ring and
//     every wait on them is bounded;
//   * scores  S^T[16 tok x 8 heads] = K[16 x 128] . Q^T  as m16n8k16 f16 MMAs on
//     the codes themselves (exact: integers below 2^21 in fp32); the contraction
//     order is permuted so that each thread's K and Q words are the bytes it
//     already holds;
//   * P^T (fp16) comes from the score fragment by movmatrix.trans;
//   * O^T[128 x 8] += V^T . P^T as m16n8k16 f16 MMAs; V enters as code + 1152
//     (two byte permutes per four codes, no subtraction), and the bias times the
//     row sum of P is taken off once at the end;
//   * split-K partials (unnormalised O, running max m, sum l) are merged by a
//     small combine kernel with log-sum-exp weights.
#include "fa3_common.cuh"
#include "fa3_tc.cuh"

#include <cuda_bf16.h>
#include <math_constants.h>

#include <algorithm>
#include <atomic>

namespace fa3 {
namespace {

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;            // the consumer warps
constexpr int kThreadsAll = kThreads + 32;        // + one producer warp
constexpr int kHeadsPerTile = 8;
// A ring stage is one 64-token tile (warp w takes its 16-token step w): K rows then
// V rows of this KV head, loaded by TMA with the 128-byte swizzle.  Three stages:
// two tiles in flight while one is read.
constexpr int kTileTok = 16 * kWarps;
constexpr int kTileBytes = kTileTok * kD;         // 8 KB of K, as much of V
constexpr int kBoxBytes = 16 * kD;                // one warp's 16 rows
constexpr int kStages = 3;
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kMergeBytes = kWarps * kHeadsPerTile * kD * 4;   // the warps' partial O of a unit
constexpr int kQBytes = kHeadsPerTile * kD;       // a unit's query rows, with its first tile's stage
// ring (aligned to 1024 bytes) + the merge buffer + the query slots + room for the alignment
constexpr int kSmemBytes = kStages * kStageBytes + kMergeBytes + kStages * kQBytes + 1024;
constexpr int kMinTilesPerCta = 3;   // (with the switch cost below, keeps every run non-empty)
constexpr int kMergeBatch = 8;   // partials whose loads a merge issues together

// Work split: the sequences' tokens are cut into n_t = ceil(T_max / 64) tiles
// each, and the W = B * n_t tile rows, taken sequence after sequence, are dealt
// to R groups of Hkv CTAs in runs (run_begin below: S equal runs inside each
// sequence, or runs of equal cost across sequences); CTA c = k * Hkv + g takes
// KV head g of run k.  The Hkv CTAs of a group read the same 1 KB cache rows
// side by side (each its 128-byte head slice), as the DRAM pages and the
// 256-byte L2 fetches like.  The (sequence b, KV head g) pairs are the units
// u = b * Hkv + g; a unit that lies in one run is finished there, the CTAs that
// share a unit each leave a partial (unnormalised O, running max, sum) and the
// last of them to arrive merges the partials into the output.
struct GqaArgs {
  CUtensorMap tm_k;      // K / V as (Hkv * D bytes, rows): boxes of 128 bytes x box_rows rows, 128-byte swizzle
  CUtensorMap tm_v;
  const int8_t* q;
  const int32_t* block_table;   // [B][max_pages] pool pages, or nullptr for the contiguous layout
  const float* q_scale;   // [Hq], or [Hq][D] per channel
  const float* k_scale;   // [Hkv], or [Hkv][D]
  const float* v_scale;   // [Hkv], or [Hkv][D]
  const float* q_off;     // per channel only: [Hq][D] offsets of q and v (k's cancel in the softmax)
  const float* v_off;
  const int32_t* lens;
  __nv_bfloat16* out;
  int32_t* arrivals;  // [B * Hkv] CTAs of a shared unit that have left their partial (0 between calls)
  float2* part_ml;    // [2 C][8]: slot 2c + 0 for CTA c's first unit, 2c + 1 for its last
  float* part_o;      // [2 C][8][D]
  int32_t* err;
  int W;              // tile rows in all, B * n_t (below 2^31)
  int n_t;            // tile rows per sequence
  int R;              // run groups (gridDim.x = R * Hkv)
  int S;              // > 0: every sequence cut into S equal runs (R = B * S); 0: runs of equal cost
  int B, Hq, Hkv, G, T_max;
  int page_size, max_pages, num_pages;
  int box_rows;     // rows of a TMA box: 64, or the largest of 32 / 16 that divides the page size
  DivU32 div_ps;    // / page_size
  float sm_log2;    // softmax_scale * log2(e)
};

// Runs of equal cost, in quarter tiles: a tile costs 4 and a switch from one
// sequence to the next inside a run kSwitchCost4 (the 4-warp merge and the new
// unit's first tile, measured at about 1.5 tiles), so a run that crosses a
// sequence boundary takes fewer tiles.  In cost coordinates sequence b spans
// [b P, b P + 4 n_t) followed by a gap of kSwitchCost4, P = 4 n_t + kSwitchCost4,
// B P - kSwitchCost4 in all; run k starts at cost floor(k total / R), mapped back
// to the first tile row at or after it.  Sequences under 4 tiles take no switch
// cost.  With R <= W / 3 every run holds at least one tile (checked exhaustively
// for n_t < 70, B < 40, R < 200).
constexpr int kSwitchCost4 = 6;
__host__ __device__ __forceinline__ int switch_cost4(int n_t) { return n_t >= 4 ? kSwitchCost4 : 0; }
__host__ __device__ __forceinline__ int run_begin(int k, int n_t, int B, int R, int S) {
  if (S > 0) return (k / S) * n_t + ((k % S) * n_t) / S;   // runs inside one sequence each
  const int sw = switch_cost4(n_t);
  const int64_t P = 4 * (int64_t)n_t + sw, total = B * P - sw;
  const int64_t c4 = (int64_t)k * total / R;
  const int64_t b = c4 / P, off4 = c4 - b * P;
  const int64_t off = off4 >= 4 * (int64_t)n_t ? n_t : (off4 + 3) / 4;
  return (int)(b * n_t + off);
}
// The run that holds tile row w: the largest k with floor(k total / R) at or
// below the cost where row w starts, in closed form (checked against run_begin
// for every row of the sizes above).
__device__ __forceinline__ int run_owner(int w, int n_t, int B, int R, int S) {
  if (S > 0) {
    const int b = w / n_t, x = w - b * n_t;
    return b * S + ((x + 1) * S - 1) / n_t;
  }
  const int sw = switch_cost4(n_t);
  const int64_t P = 4 * (int64_t)n_t + sw, total = B * P - sw;
  const int64_t cp = (int64_t)(w / n_t) * P + 4 * (int64_t)(w % n_t);
  return (int)min((int64_t)R - 1, ((cp + 1) * R - 1) / total);
}

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

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t x) {
  __half2 h = *reinterpret_cast<__half2*>(&x);
  return __half22float2(h);
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Output of head g*G + hh of sequence b from the merged O and l of a dim d.
template <bool CHANNEL>
__device__ __forceinline__ void store_out(const GqaArgs& p, int b, int g, int hh, int d, float O, float L) {
  float val = 0.f;
  if (L > 0.f)
    val = CHANNEL ? p.v_scale[(int64_t)g * kD + d] * (O / L - kVBias - p.v_off[(int64_t)g * kD + d])
                  : p.v_scale[g] * (O / L - kVBias);
  p.out[((int64_t)b * p.Hq + g * p.G + hh) * kD + d] = __float2bfloat16_rn(val);
}

// The 4 consumer warps alone (the producer warp may have left).
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

__device__ __forceinline__ int atomic_add_release(int32_t* a, int v) {
  int old;
  asm volatile("atom.add.release.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}

// Partial slot of unit (b, g) in the run of group rg: 2 c + 0 if the unit is the
// run's first, 2 c + 1 if its last (c = rg * Hkv + g).  Of the groups sharing a
// unit only the first (owner0) can have started before it: its slot is
// 2 c + first_off, first_off = 1 if it did.
__device__ __forceinline__ int64_t partial_slot(const GqaArgs& p, int rg, int g, int owner0, int first_off) {
  return 2 * ((int64_t)rg * p.Hkv + g) + (rg == owner0 ? first_off : 0);
}

// Merge of the partials of unit (b, g) left by run groups owner0..owner1, by the
// 4 consumer warps: thread (e, lane) takes head 2 (lane & 3) + (e & 1) and dims
// 16 (lane >> 2) + (e >> 1) + 2 i, i = 0..7, one online pass over the
// contributors, 8 at a time (a partial with l = 0 has O = 0).  The slots read go
// back to zeros, and so does the unit's arrival counter.
template <bool CHANNEL>
__device__ void merge_partials(const GqaArgs& p, int b, int g, int base, int owner0, int owner1, int R) {
  const int tid = threadIdx.x, em = tid >> 5, lane = tid & 31;
  const int hm = 2 * (lane & 3) + (em & 1), dm = 16 * (lane >> 2) + (em >> 1);
  const int first_off = run_begin(owner0, p.n_t, p.B, R, p.S) < base ? 1 : 0;
  float Mx = -CUDART_INF_F, Lx = 0.f, Ox[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) Ox[i] = 0.f;
  for (int cq = owner0; cq <= owner1; cq += kMergeBatch) {
    int64_t sl[kMergeBatch];
    float2 ml[kMergeBatch];
    float ov[kMergeBatch][8];
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      sl[k] = partial_slot(p, min(cq + k, owner1), g, owner0, first_off);
      ml[k] = __ldcg(&p.part_ml[sl[k] * kHeadsPerTile + hm]);
#pragma unroll
      for (int i = 0; i < 8; ++i) ov[k][i] = __ldcg(&p.part_o[sl[k] * 1024 + (4 * i + em) * 32 + lane]);
    }
#pragma unroll
    for (int k = 0; k < kMergeBatch; ++k) {
      if (cq + k <= owner1 && ml[k].y > 0.f) {
        const float nm = fmaxf(Mx, ml[k].x);
        const float fa = Mx == -CUDART_INF_F ? 0.f : ex2_approx(Mx - nm), fb = ex2_approx(ml[k].x - nm);
        Lx = Lx * fa + ml[k].y * fb;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          Ox[i] = Ox[i] * fa + ov[k][i] * fb;
          p.part_o[sl[k] * 1024 + (4 * i + em) * 32 + lane] = 0.f;
        }
        Mx = nm;
      }
    }
  }
  if (hm < p.G) {
#pragma unroll
    for (int i = 0; i < 8; ++i) store_out<CHANNEL>(p, b, g, hm, dm + 2 * i, Ox[i], Lx);
  }
  consumer_sync();   // every thread has read the (m, l) pairs
  const int n_ml = (owner1 - owner0 + 1) * kHeadsPerTile;
  for (int i = tid; i < n_ml; i += kThreads)
    p.part_ml[partial_slot(p, owner0 + i / kHeadsPerTile, g, owner0, first_off) * kHeadsPerTile + i % kHeadsPerTile] =
        make_float2(0.f, 0.f);
  if (tid == 0) p.arrivals[(int64_t)b * p.Hkv + g] = 0;
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
__global__ void __launch_bounds__(kThreadsAll, 3) gqa_decode_kernel(const __grid_constant__ GqaArgs p) {
  const int c = blockIdx.x;
  const int R = p.R, rg = c / p.Hkv, g = c - rg * p.Hkv;   // run group, KV head
  const int n_t = p.n_t;
  const int w_lo = run_begin(rg, n_t, p.B, R, p.S), w_hi = run_begin(rg + 1, n_t, p.B, R, p.S);
  const int b_first = w_lo / n_t, b_last = (w_hi - 1) / n_t;
  if (!PAGED && threadIdx.x == kThreads) {
    // The run's first tiles into L2 before the wait for the work ahead on the
    // stream: L2 is coherent, so this reads nothing stale, and these fetches run
    // while the kernel before (often the previous call) finishes its merges.
    for (int i = 0; i < kStages && w_lo + i < w_hi; ++i) {
      const int w = w_lo + i, b = w / n_t, row = b * p.T_max + (w - b * n_t) * kTileTok;
      tma_prefetch_2d(&p.tm_k, g * kD, row);
      tma_prefetch_2d(&p.tm_v, g * kD, row);
    }
  }
  pdl_wait();
  pdl_launch_dependents();
  // Ring of 64-token tiles filled by TMA with the 128-byte swizzle: a 128-byte row
  // keeps its 16-byte chunk c at position c ^ (row & 7), so the V fragment loads
  // below touch 8 distinct bank groups per 8-lane phase (the K loads two-way).
  // Behind the ring, the buffer where the 4 warps merge a unit.
  extern __shared__ __align__(1024) uint8_t gsm_raw[];
  const uint32_t raw_s = smem_u32(gsm_raw), ring_s = (raw_s + 1023u) & ~1023u;
  // sm_o[warp][4 i + e][lane] = that lane's o[i][e]: every store and every read of
  // the merge touches 32 consecutive words
  float (*sm_o)[32][32] = reinterpret_cast<float (*)[32][32]>(gsm_raw + (ring_s - raw_s) + kStages * kStageBytes);
  const uint32_t q_s = ring_s + kStages * kStageBytes + kMergeBytes;   // query slot of stage s at + s * kQBytes
  __shared__ int sm_n[kStages];   // length of the unit whose first tile the stage holds
  __shared__ uint64_t bar_full[kStages], bar_empty[kStages];
  __shared__ uint64_t bar_part, bar_agent;   // first unit's partial stored / its arrival counted
  __shared__ int sm_agent_last;
  __shared__ uint32_t ring_abort;
  __shared__ int sm_last;
  __shared__ float sm_m[kWarps][kHeadsPerTile];
  __shared__ float sm_l[kWarps][kHeadsPerTile];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, qd = lane & 3;
  const int G = p.G;
  const int lens_first = p.lens[b_first];   // in flight while the barriers are set up
  // the run's first and last units, and the run groups that share each
  const bool two = b_last != b_first;
  // A run of several units counts its arrival at a shared first unit as soon as
  // the partial is stored, through an agent lane of the producer warp: then the
  // others sharing that unit, which finish it at the ends of their runs, merge it.
  const bool agent_first =
      two && run_owner(b_first * n_t, n_t, p.B, R, p.S) != run_owner(b_first * n_t + n_t - 1, n_t, p.B, R, p.S);
  const int qbytes = G * kD;

  if (warp == kWarps && lane == 0) {
    ring_abort = 0u;
    for (int st = 0; st < kStages; ++st) {
      mbar_init(smem_u32(&bar_full[st]), 1);
      mbar_init(smem_u32(&bar_empty[st]), kWarps);
    }
    mbar_init(smem_u32(&bar_part), kWarps);
    mbar_init(smem_u32(&bar_agent), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kWarps) {
    // The producer warp (its lane 0) walks the run unit by unit and fills stage
    // j % 3 with tile j of the run once every consumer warp has released the tile
    // that used the stage before.  A tile that starts below the sequence's length
    // is loaded: one 64-row box of K and one of V (contiguous layout), or the boxes
    // of its rows that start below the length (paged: a tile starts at a multiple
    // of 64 tokens and a box's rows divide both 64 and the page size, so a box lies
    // in one page; a block-table entry outside the pool loads the rows past the
    // pool's end, zeros).  A tile past the length is only signalled, no data.  The
    // contiguous layout loads the run's first 3 tiles before the length has arrived
    // (reading rows that may go unused is harmless there).
    if (lane == 1 && agent_first) {
      // The agent: once the 4 warps have stored the first unit's partial (their
      // arrivals release it at CTA scope), one release add at GPU scope publishes it.
      int last = 0;
      const int f_own0 = run_owner(b_first * n_t, n_t, p.B, R, p.S);
      const int f_own1 = run_owner(b_first * n_t + n_t - 1, n_t, p.B, R, p.S);
      if (wait_bar(smem_u32(&bar_part), 0u, &ring_abort, p.err)) {
        const int before = atomic_add_release(&p.arrivals[(int64_t)b_first * p.Hkv + g], 1);
        last = before == f_own1 - f_own0;
        if (last) asm volatile("fence.acq_rel.gpu;" ::: "memory");   // the others' partials
      }
      sm_agent_last = last;
      mbar_arrive(smem_u32(&bar_agent));
      return;
    }
    if (lane != 0) return;
    int produced = 0;
    bool stop = false;
    if (!PAGED) {   // the descriptors, ahead of the first copies
      asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_k) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(&p.tm_v) : "memory");
    }
    int lens_next = lens_first;
    const int box = PAGED ? p.box_rows : kTileTok;
    for (int b = b_first; b <= b_last && !stop; ++b) {
      const int base = b * n_t;
      const int ta = max(w_lo, base) - base, tb = min(w_hi, base + n_t) - base;
      const int lens_b = lens_next;
      lens_next = b < b_last ? p.lens[b + 1] : 0;   // one unit ahead
      int n = -1;   // not needed yet
      for (int t = ta; t < tb; ++t) {
        const int j = produced;
        const int slot = j % kStages;
        if (j >= kStages &&
            !wait_bar(smem_u32(&bar_empty[slot]), (uint32_t)((j / kStages - 1) & 1), &ring_abort, p.err)) {
          stop = true;
          break;
        }
        const int t0 = t * kTileTok;
        const bool first = t == ta;   // the unit's query rows and length go with it
        const bool early = !PAGED && j < kStages;
        if (!early && n < 0) {
          n = lens_b;
          if (n < 0 || n > p.T_max) {
            if (g == 0 && ta == 0) set_dev_err(p.err, FA3_DEVERR_LENS);
            n = 0;
          }
        }
        const uint32_t bar = smem_u32(&bar_full[slot]);
        const uint32_t dst = ring_s + (uint32_t)(slot * kStageBytes);
        const bool load = early || t0 < n;
        const int nb = !load ? 0 : PAGED ? min(kTileTok / box, (n - t0 + box - 1) / box) : 1;
        const uint32_t tile_tx = (uint32_t)(nb * 2 * box * kD);
        // the consumers' reads of the stage (generic proxy) come before this tile's
        // copies (async proxy)
        if (load || first) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (first) mbar_expect_only(bar, tile_tx + (uint32_t)qbytes);
        else if (load) mbar_expect_tx(bar, tile_tx);
        if (first) bulk_g2s(q_s + slot * kQBytes, p.q + ((int64_t)b * p.Hq + g * G) * kD, (uint32_t)qbytes, bar);
        if (load) {
          if (!PAGED) {
            tma_2d(dst, &p.tm_k, g * kD, b * p.T_max + t0, bar);
            tma_2d(dst + kTileBytes, &p.tm_v, g * kD, b * p.T_max + t0, bar);
          } else {
            for (int i = 0; i < nb; ++i) {
              const int ts = t0 + box * i;
              const uint32_t pi = divu32((uint32_t)ts, p.div_ps);
              const int pg = p.block_table[(int64_t)b * p.max_pages + pi];
              int row = p.num_pages * p.page_size;
              if (pg >= 0 && pg < p.num_pages) row = pg * p.page_size + (ts - (int)pi * p.page_size);
              else set_dev_err(p.err, FA3_DEVERR_PAGE);
              tma_2d(dst + i * box * kD, &p.tm_k, g * kD, row, bar);
              tma_2d(dst + kTileBytes + i * box * kD, &p.tm_v, g * kD, row, bar);
            }
          }
        }
        if (first) {
          if (n < 0) {   // (an early tile: the length has arrived meanwhile)
            n = lens_b;
            if (n < 0 || n > p.T_max) {
              if (g == 0 && ta == 0) set_dev_err(p.err, FA3_DEVERR_LENS);
              n = 0;
            }
          }
          sm_n[slot] = n;
          mbar_arrive(bar);
        } else if (!load) {
          mbar_arrive(bar);
        }
        produced = j + 1;
      }
    }
    if (*reinterpret_cast<volatile uint32_t*>(&ring_abort)) {
      // a wait gave up (the output is flagged invalid): the tiles still in flight
      // get one more bounded wait before the CTA may exit
      uint32_t no_abort = 0u;
      for (int jj = produced > kStages ? produced - kStages : 0; jj < produced; ++jj)
        wait_bar(smem_u32(&bar_full[jj % kStages]), (uint32_t)((jj / kStages) & 1), &no_abort, nullptr);
    }
    return;
  }

  auto chunk_addr = [&](uint32_t base, int row, int col) { return base + row * 128 + ((col ^ (row & 7)) << 4); };
  const int h0 = 2 * qd, h1 = 2 * qd + 1;
  float c0s_h = 0.f, c1s_h = 0.f;   // per-head score factors (per-tensor scales: the same for every unit)
  if (!CHANNEL) {
    const float ks = p.k_scale[g] * p.sm_log2;
    c0s_h = h0 < G ? p.q_scale[g * G + h0] * ks : 0.f;
    c1s_h = h1 < G ? p.q_scale[g * G + h1] * ks : 0.f;
  }
  int j = 0;   // ring position, in step with the producer
  for (int b = b_first; b <= b_last; ++b) {
    const int base = b * n_t;
    const int ta = max(w_lo, base) - base, tb = min(w_hi, base + n_t) - base;
    // The unit's query rows and length come with its first tile: fetched here by
    // loads of their own, under the full stream of tiles, they waited behind the
    // SM's copies in flight (3 us and more at a unit switch).
    const int slot0 = j % kStages;
    const bool ok0 =
        warp_all(wait_bar(smem_u32(&bar_full[slot0]), (uint32_t)((j / kStages) & 1), &ring_abort, p.err));
    const int n = ok0 ? sm_n[slot0] : 0;
    // Q^T fragments of head r of this group as int8 words, contraction order
    // permuted: thread (r, qd) holds row bytes [16qd, +16) as words 0-3 and
    // [64 + 16qd, +16) as words 4-7; k16 step s takes word s of Q (B operand)
    // and of its K rows r and r + 8 (A operand) alike.
    uint32_t qw[8];
    {
      uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0;
      if (ok0 && r < G) {
        const uint32_t qrow = q_s + slot0 * kQBytes + r * kD;
        q0 = lds128(qrow + 16 * qd);
        q1 = lds128(qrow + 64 + 16 * qd);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        qw[i] = word(q0, i);
        qw[4 + i] = word(q1, i);
      }
    }
    float c0s = c0s_h, c1s = c1s_h;
    // Q^T as fp16 codes, the B fragments of the 8 k16 steps: step s takes word s
    // (dims base(s) + 0..3, base(s) defined below), bytes 0-1 as b0 and 2-3 as b1
    uint32_t qh[8][2];
    if (!CHANNEL) {
#pragma unroll
      for (int s_ = 0; s_ < 8; ++s_) i8x4_to_f16x4_exact(qw[s_], qh[s_][0], qh[s_][1]);
    }
    // per channel: the B fragments of w (hi, lo) for the 8 k16 steps; step s takes
    // dims base(s) + 0..3, base(s) = 4s within the first 16-byte chunk of this
    // thread (s < 4), then within its second chunk
    uint32_t wh[8][2], wl[8][2];
    if (CHANNEL) {
      float wv[32];
      float amax = 0.f;
      const int hq = g * G + r;
#pragma unroll
      for (int jd = 0; jd < 32; ++jd) {
        const int d = (jd < 16 ? 16 * qd : 64 + 16 * qd) + (jd & 15);
        const int code = (int)(int8_t)((qw[jd >> 2] >> (8 * (jd & 3))) & 0xffu);
        float wj = 0.f;
        if (r < G)
          wj = ((float)code - p.q_off[(int64_t)hq * kD + d]) * p.q_scale[(int64_t)hq * kD + d] *
               p.k_scale[(int64_t)g * kD + d];
        wv[jd] = wj;
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
          const int jd = 4 * s_ + 2 * hlf;
          const float a = wv[jd] * down, b2 = wv[jd + 1] * down;
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

    for (int t = ta; t < tb; ++t, ++j) {
      const int slot = j % kStages;
      const int t0 = t * kTileTok + 16 * warp;     // this warp's 16-token step
      const bool ok =
          warp_all(wait_bar(smem_u32(&bar_full[slot]), (uint32_t)((j / kStages) & 1), &ring_abort, p.err));
      const bool mine = ok && t0 < n;
      const uint32_t kst = ring_s + (uint32_t)(slot * kStageBytes + warp * kBoxBytes), vst = kst + kTileBytes;
      uint4 kr[4], vr[4];
      if (mine) {
        kr[0] = lds128(chunk_addr(kst, r, qd));
        kr[1] = lds128(chunk_addr(kst, r, 4 + qd));
        kr[2] = lds128(chunk_addr(kst, r + 8, qd));
        kr[3] = lds128(chunk_addr(kst, r + 8, 4 + qd));
        vr[0] = lds128(chunk_addr(vst, 2 * qd, r));
        vr[1] = lds128(chunk_addr(vst, 2 * qd + 1, r));
        vr[2] = lds128(chunk_addr(vst, 2 * qd + 8, r));
        vr[3] = lds128(chunk_addr(vst, 2 * qd + 9, r));
      }
      __syncwarp();   // every lane has its fragments: the stage may be refilled
      if (lane == 0) mbar_arrive(smem_u32(&bar_empty[slot]));
      if (!mine) continue;
      float cf[4];
      if (!CHANNEL) {
        // ---- scores S^T = K . Q^T: exact integer dot products on fp16 codes (fp32
        // accumulate; every partial sum is an integer below 2^21, so no rounding).
        // The int8 MMA path of this part runs at a quarter of the f16 one and bounded
        // the whole kernel; two accumulators halve the dependent MMA chain.
        float ca[4] = {0.f, 0.f, 0.f, 0.f}, cb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s = 0; s < 8; ++s) {
          uint32_t a0, a1, a2, a3;
          i8x4_to_f16x4_exact(word(kr[s >> 2], s & 3), a0, a2);          // row r:     dims base(s) + 0..3
          i8x4_to_f16x4_exact(word(kr[2 + (s >> 2)], s & 3), a1, a3);    // row r + 8
          mma16816((s & 1) ? cb : ca, a0, a1, a2, a3, qh[s][0], qh[s][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) cf[e] = ca[e] + cb[e];
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
      const bool va = t0 + r < n, vb = t0 + r + 8 < n;
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

    // ---- merge the 4 warps over this unit's tiles.  Merge thread (e, lane) takes
    // o[i][e] of that lane in every warp, i = 0..7: head hm and dims dm + 2i.
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
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) sm_o[warp][4 * i + e][lane] = o[i][e];
    consumer_sync();
    const int em = warp, hm = 2 * (lane & 3) + (em & 1), dm = 16 * (lane >> 2) + (em >> 1);
    const int owner0 = run_owner(base, n_t, p.B, R, p.S), owner1 = run_owner(base + n_t - 1, n_t, p.B, R, p.S);   // run groups
    const int64_t slot = 2 * c + (b == b_first ? 0 : 1);
    float Om[8], Lm = 0.f;
    float Mm = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) Mm = fmaxf(Mm, sm_m[w][hm]);
    {
      float f[kWarps];
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        f[w] = Mm == -CUDART_INF_F ? 0.f : ex2_approx(sm_m[w][hm] - Mm);
        Lm += sm_l[w][hm] * f[w];
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) acc += sm_o[w][4 * i + em][lane] * f[w];
        Om[i] = acc;
      }
    }
    if (owner0 == owner1) {
      if (hm < G) {
#pragma unroll
        for (int i = 0; i < 8; ++i) store_out<CHANNEL>(p, b, g, hm, dm + 2 * i, Om[i], Lm);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) p.part_o[slot * 1024 + (4 * i + em) * 32 + lane] = Om[i];
      if (lane < 4 && em < 2) p.part_ml[slot * kHeadsPerTile + hm] = make_float2(Mm, Lm);
      if (agent_first && b == b_first) {
        __syncwarp();   // the warp's stores, then its arrival
        if (lane == 0) mbar_arrive(smem_u32(&bar_part));
      }
    }
    consumer_sync();   // the merge buffer is free for the next unit
  }

  const int f_own0 = run_owner(b_first * n_t, n_t, p.B, R, p.S), f_own1 = run_owner(b_first * n_t + n_t - 1, n_t, p.B, R, p.S);
  const int l_own0 = run_owner(b_last * n_t, n_t, p.B, R, p.S), l_own1 = run_owner(b_last * n_t + n_t - 1, n_t, p.B, R, p.S);
  // ---- arrival at the shared units not counted by the agent (the run's last,
  // or a one-unit run's only unit), after the run: the barrier then one thread's
  // release add publishes the partial.  (A release by a consumer thread mid-run
  // waited for the partial's stores under the full memory stream and held the
  // next unit's tiles up for 3-4 us.)
  if (tid == 0) {
    int last = 0;
    if (!agent_first && f_own0 != f_own1 &&
        atomic_add_release(&p.arrivals[(int64_t)b_first * p.Hkv + g], 1) == f_own1 - f_own0)
      last |= 1;
    if (two && l_own0 != l_own1 &&
        atomic_add_release(&p.arrivals[(int64_t)b_last * p.Hkv + g], 1) == l_own1 - l_own0)
      last |= 2;
    if (agent_first && wait_bar(smem_u32(&bar_agent), 0u, &ring_abort, p.err) && sm_agent_last) last |= 1;
    if (last) asm volatile("fence.acq_rel.gpu;" ::: "memory");   // the others' partials
    sm_last = last;
  }
  consumer_sync();
  // ---- merges of the units whose partial arrived last from here, in one online
  // pass over the contributors
  const int last = sm_last;
  if (last & 1) {
    merge_partials<CHANNEL>(p, b_first, g, b_first * n_t, f_own0, f_own1, R);
    consumer_sync();
  }
  if (last & 2) {
    merge_partials<CHANNEL>(p, b_last, g, b_last * n_t, l_own0, l_own1, R);
    consumer_sync();
  }
}

int gqa_blocks_per_sm();

// Work plan: at most one resident wave of CTAs (fewer when there are under 3
// tile rows per run group), and no combine kernel: the last CTA to finish a
// shared unit merges it.
struct GqaPlan {
  int64_t W;      // tile rows in all (a launch needs W < 2^31)
  int n_t;        // tile rows per sequence
  int R;          // run groups of Hkv CTAs
  int S;          // > 0: S equal runs per sequence; 0: runs of equal cost across sequences
  int64_t C;      // CTAs, R * Hkv
  bool shared;    // some unit is split between runs (partials and arrival counters needed)
};

GqaPlan gqa_plan(int B, int Hkv, int T_max, int num_sms) {
  GqaPlan pl;
  pl.n_t = (T_max + kTileTok - 1) / kTileTok;
  pl.W = (int64_t)B * pl.n_t;
  const int64_t wave = (int64_t)num_sms * gqa_blocks_per_sm();
  const int64_t groups = std::max<int64_t>(1, std::min<int64_t>(wave / Hkv, pl.W / kMinTilesPerCta));
  // S equal runs per sequence when those fill at least 80% of the wave: no run
  // then switches sequences (a switch costs a merge and a first-tile wait), which
  // measured faster than runs of equal cost across sequences (Llama-70B shape,
  // 4096 tokens: B 16 30.6 against 32.5 us, B 8 19.1 against 20.5 us), and slower
  // once the equal runs left much of the wave idle (B 32: 256 CTAs, 63.3 against
  // 52.3 us).
  const int64_t S = std::min<int64_t>(groups / B, pl.n_t / kMinTilesPerCta);
  pl.S = S >= 1 && 5 * B * S >= 4 * groups ? (int)S : 0;
  pl.R = pl.S > 0 ? B * pl.S : (int)groups;
  pl.C = (int64_t)pl.R * Hkv;
  pl.shared = false;
  if (pl.W < ((int64_t)1 << 31)) {
    for (int c = 1; c < pl.R && !pl.shared; ++c) pl.shared = run_begin(c, pl.n_t, B, pl.R, pl.S) % pl.n_t != 0;
  }
  return pl;
}

// Workspace: arrival counters [U] (int32), then the partials' (m, l) [2C][8] and O [2C][8][D].
struct GqaWorkspace {
  size_t counters, ml, o, total;
};

GqaWorkspace gqa_workspace_layout(int B, int Hkv, const GqaPlan& pl) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  GqaWorkspace w;
  const size_t slots = 2 * (size_t)pl.C * kHeadsPerTile;
  w.counters = 0;
  w.ml = up((size_t)B * Hkv * sizeof(int32_t));
  w.o = w.ml + up(slots * sizeof(float2));
  w.total = pl.shared ? w.o + slots * kD * sizeof(float) : 0;
  return w;
}

// Shared memory attributes of a kernel variant: its dynamic size, and the whole
// carveout for shared memory (3 CTAs of 67 KB need it; left to the driver, the
// carveout held 2, and a third of the wave ran after the rest).
cudaError_t set_smem_attrs(void (*kernel)(GqaArgs)) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  return e;
}

int gqa_blocks_per_sm() {
  static int cached = 0;
  if (cached <= 0) {
    int n = 0;
    if (set_smem_attrs(gqa_decode_kernel<false, false>) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gqa_decode_kernel<false, false>, kThreadsAll, kSmemBytes) !=
            cudaSuccess ||
        n <= 0)
      n = 3;
    cached = n;
  }
  return cached;
}

// The attributes are set once per (kernel variant, device).
std::atomic<uint64_t> g_smem_attr_set[3];

int ensure_smem_attr(void (*kernel)(GqaArgs), int variant) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA3_ECUDA;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (bit && (g_smem_attr_set[variant].load(std::memory_order_acquire) & bit)) return FA3_OK;
  if (set_smem_attrs(kernel) != cudaSuccess) return FA3_ECUDA;
  if (bit) g_smem_attr_set[variant].fetch_or(bit, std::memory_order_acq_rel);
  return FA3_OK;
}

}  // namespace
}  // namespace fa3

using namespace fa3;

FA3_API size_t fa3_gqa_workspace_size(int B, int Hq, int Hkv, int D, int T_max) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D != kD || T_max <= 0) return 0;
  int sms = 0;
  if (check_device(&sms) != FA3_OK) sms = 148;
  const GqaPlan pl = gqa_plan(B, Hkv, T_max, sms);
  return gqa_workspace_layout(B, Hkv, pl).total;
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
  const GqaPlan pl = gqa_plan(B, Hkv, T_max, sms);
  if (pl.W >= ((int64_t)1 << 31)) return FA3_ERANGE;   // tile indices are 32-bit
  const GqaWorkspace wl = gqa_workspace_layout(B, Hkv, pl);
  if (wl.total && (!workspace || workspace_bytes < wl.total || !aligned16(workspace))) return FA3_EWORKSPACE;
  GqaArgs a;
  a.q = q; a.q_scale = q_scale; a.k_scale = k_scale; a.v_scale = v_scale; a.lens = lens;
  a.q_off = q_off; a.v_off = v_off;
  a.out = reinterpret_cast<__nv_bfloat16*>(out);
  char* ws = static_cast<char*>(workspace);
  a.arrivals = wl.total ? reinterpret_cast<int32_t*>(ws + wl.counters) : nullptr;
  a.part_ml = wl.total ? reinterpret_cast<float2*>(ws + wl.ml) : nullptr;
  a.part_o = wl.total ? reinterpret_cast<float*>(ws + wl.o) : nullptr;
  a.err = dev_err;
  a.W = (int)pl.W; a.n_t = pl.n_t; a.R = pl.R; a.S = pl.S;
  a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.G = G; a.T_max = T_max;
  a.block_table = block_table; a.page_size = page_size; a.max_pages = max_pages; a.num_pages = num_pages;
  a.div_ps = make_divu32((uint32_t)(page_size > 0 ? page_size : 1));
  a.sm_log2 = softmax_scale * 1.4426950408889634f;
  // K and V as 2D byte tensors (Hkv * D, rows): rows of every sequence one after
  // another, or the pool's rows; TMA coordinates are 32-bit.
  const int64_t rows = block_table ? (int64_t)num_pages * page_size : (int64_t)B * T_max;
  if (rows >= ((int64_t)1 << 31) - kTileTok) return FA3_ERANGE;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return FA3_ECUDA;
  {
    const cuuint64_t dims[2] = {(cuuint64_t)Hkv * kD, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)Hkv * kD};
    a.box_rows = !block_table ? kTileTok : page_size % 64 == 0 ? 64 : page_size % 32 == 0 ? 32 : 16;
    const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)a.box_rows};
    const cuuint32_t es[2] = {1u, 1u};
    for (int t = 0; t < 2; ++t)
      if (encode(t ? &a.tm_v : &a.tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(t ? v : k), dims,
                 strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return FA3_ECUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int variant = channel ? 2 : block_table ? 1 : 0;
  auto* kernel = channel ? gqa_decode_kernel<false, true>
                         : block_table ? gqa_decode_kernel<true, false> : gqa_decode_kernel<false, false>;
  st = ensure_smem_attr(kernel, variant);
  if (st != FA3_OK) return st;
  timing_begin(s);
  const cudaError_t le = launch_pdl(kernel, dim3((unsigned)pl.C), dim3(kThreadsAll), kSmemBytes, s, a);
  timing_end(s);
  return le == cudaSuccess ? FA3_OK : FA3_ECUDA;
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
// workspace (arrival counters and partials) is a fixed array in the library's
// own device memory, zero-filled when the module loads.
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
  // The array starts zero-filled with the module and every call leaves it so.
  return fa3_decode_attn_gqa(q, k, v, q_scale, k_scale, v_scale, lens, out, B, Hq, Hkv, D, T_max, softmax_scale,
                             scratch, kGqaStaticScratchBytes, dev_err, stream);
}
