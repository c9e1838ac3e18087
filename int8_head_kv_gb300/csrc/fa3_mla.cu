// Absorbed-MLA decode attention over an INT8 latent cache (tcgen05 + TMA, sm_103a).
//
// MindIE "FA3 quantization", Overview: for MLA only the non-RoPE part of K (the
// latent c_kv, shared by K-nope and V) is quantized to 8 bits per head; the
// RoPE part of K stays in floating point; the decode-phase attention operator
// reads the INT8 cache.  Scales are the symmetric per-head ones of msModelSlim
// "FA3量化" 原理 / 算法流程 step 4; the latent query is quantized with its static
// per-head scale so that the latent score is an integer contraction.
//
//   s[h, j] = (sum_c q8[h, c] ckv[j, c]) * q_scale[h] * kv_scale + q_rope[h] . k_rope[j]
//   out[h]  = kv_scale * sum_j softmax(s * softmax_scale)_j * ckv[j, :]
//
// GB300 design (tcgen05 has no int8 MMA kind on sm_103a):
//   * int8 codes are exact in fp16 and a 256-term sum of their products stays
//     below 2^24, so kind::f16 MMAs with fp32 accumulation give the exact
//     integer latent score;
//   * the fp32 accumulator of 128 heads x 512 latent is all of one SM's TMEM, so
//     a 2-CTA cluster splits the latent in halves: CTA r owns latent columns
//     [r*Dl/2, (r+1)*Dl/2), loads only that half of each 64-token tile into
//     registers one tile ahead (with an L2 bulk prefetch four tiles ahead),
//     converts it to fp16 core matrices in one of four shared-memory buffers
//     (one buffer is the K-major B operand of Q.C^T and the MN-major B operand
//     of P.C) and keeps its O half in TMEM;
//   * the quantized latent query lives in TMEM as the A operand of Q.C^T; the
//     RoPE term is split over the pair (each CTA contracts half of the RoPE
//     dims from a TMA-loaded bf16 key tile); each CTA scales its exact latent
//     partial, adds its RoPE share and sends the fp32 partial score to the peer
//     by st.async into its shared memory; own + peer is the same fp32 sum in
//     both CTAs, so both run the same online softmax on identical scores (lazy
//     rescale when the max grows by more than 8 in log2 units);
//   * warp roles: 8 softmax warps (two per TMEM lane quarter: lane = head, each
//     warp takes half of a tile's tokens), 1 MMA issuer, 3 int8->fp16
//     converter warps (the first converter thread also issues the RoPE TMA);
//   * split-K: the tiles of all sequences are dealt out evenly to the clusters
//     that fit on the GPU; a cluster's piece of a sequence is a segment; for a
//     split sequence each softmax warp leaves its block of O (unnormalised, with
//     the rows' m and l) in the workspace, and mla_combine_kernel merges all
//     segments' blocks with log-sum-exp weights into the output rows;
//   * the query pre-pass, this kernel and the combine kernel are programmatic
//     dependent launches: each waits (griddepcontrol) for the previous grid
//     before it reads what that grid wrote.
// Every wait is bounded; on time-out the kernel sets FA3_DEVERR_TIMEOUT, drains
// its own copies and MMAs, frees its TMEM and returns.
#include "fa3_common.cuh"
#include "fa3_tc.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <math_constants.h>

namespace fa3 {
namespace {

constexpr int kTok = 64;          // tokens per tile
constexpr int kThreads = 384;     // 12 warps: at most 3 per SM sub-partition, so up to 168 registers each
constexpr int kSmWarps = 8;       // softmax: two warps per TMEM lane quarter, one per half of the tile's tokens
constexpr int kMmaWarp = 8;
constexpr int kConvWarp0 = 9;     // converters (3 warps); the first thread also issues the RoPE key TMA
constexpr int kConvThreads = 96;
constexpr int kRows = 128;        // heads (TMEM lanes)
constexpr int NR = 2;             // RoPE key tile stages (TMA)
constexpr int NC = 4;             // fp16 latent tile buffers (Q.C^T runs two tiles ahead of P.C)

// Shared memory map (bytes from a 1024-byte aligned base).
constexpr uint32_t QR_BYTES = 16384;                             // prepared RoPE query image of a sequence
constexpr uint32_t OFF_QR = 0;                                   // this CTA's RoPE query share (<= 8 KB)
constexpr uint32_t QR_CTA_BYTES = 8192;
constexpr uint32_t OFF_C16 = OFF_QR + QR_CTA_BYTES;              // NC x fp16 latent tile half (<= 32 KB)
constexpr uint32_t C16_BYTES = 32768;
constexpr uint32_t OFF_ROPE = OFF_C16 + NC * C16_BYTES;          // NR x this CTA's share of a bf16 RoPE key tile
constexpr uint32_t ROPE_BYTES = 4096;
constexpr uint32_t OFF_P = OFF_ROPE + NR * ROPE_BYTES;           // fp16 P, 128 x 64 (16 KB)
// Partial-score exchange, double-buffered: slot s of X receives the peer's fp32
// partial scores of every other tile, written by the peer's st.async.  Each
// softmax warp owns a 4 KB region of a slot: [chunk 0..7][lane][16 bytes], 32
// values per lane.
constexpr int kXChunks = 8;
constexpr uint32_t kXWarpBytes = kXChunks * 32 * 16;
constexpr uint32_t kXSlotBytes = kSmWarps * kXWarpBytes;         // 32 KB
constexpr uint32_t OFF_X = OFF_P + 16384;
constexpr uint32_t OFF_BAR = OFF_X + 2 * kXSlotBytes;
constexpr uint32_t OFF_MX = OFF_BAR + 1024;                      // float [2][128]: per-half row maxima / sums
constexpr uint32_t SMEM_BYTES = OFF_MX + 1024 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");

// TMEM columns.
constexpr uint32_t TM_O = 0;      // fp32 O half: Dl/2 columns
constexpr uint32_t TM_QA = 256;   // fp16 latent query half as the A operand: Dl/4 columns
constexpr uint32_t TM_S = 384;    // latent partial scores, 64 columns
constexpr uint32_t TM_R = 448;    // RoPE scores, 64 columns

// Barrier slots (8 bytes each) at OFF_BAR.
enum {
  B_ROPE_FULL = 0, B_ROPE_EMPTY = B_ROPE_FULL + NR,
  B_C16_FULL = B_ROPE_EMPTY + NR, B_C16_EMPTY = B_C16_FULL + NC,
  B_S_FULL = B_C16_EMPTY + NC, B_S_EMPTY, B_P_FULL, B_PV_DONE, B_Q_READY, B_QR_FULL, B_QK_DONE,
  B_DRAIN,
  B_XF,                          // [slot][warp]: that warp's region of X slot landed (3 KB of tx)
  B_XE = B_XF + 2 * kSmWarps,    // [slot][warp]: the peer's warp has read its region of that X slot
  B_PAIR_W = B_XE + 2 * kSmWarps, B_PAIR_R = B_PAIR_W + 4, NBAR = B_PAIR_R + 4
};
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * NBAR;   // u32 TMEM base address
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;         // u32 abort flag
constexpr uint32_t OFF_SCHED = OFF_TMEM_SLOT + 8;         // 4 x int64: b_first, pre_first, x0, x1
static_assert(OFF_SCHED + 32 <= OFF_BAR + 1024, "barrier area");

struct MlaParams {
  CUtensorMap tm_rope;   // bf16 viewed as (8, T_max, Dr/8, B), or (8, pool rows, Dr/8, 1) when paged
  const uint16_t* q;
  const int8_t* ckv;     // [B][T_max][Dl], or the [pool rows][Dl] page pool
  const uint16_t* krope; // the same rows of Dr bf16 (L2 prefetch; the tiles themselves come through tm_rope)
  const int32_t* block_table;   // [B][max_pages] pool pages, or nullptr for the contiguous layout
  int page_size, max_pages, num_pages;
  const float* q_scale;
  const float* kv_scale;
  const int32_t* lens;
  float* out;
  float* part_o;         // [slot][2][warp][O columns / 4][32][4]: unnormalised O block of each softmax warp
  float2* part_ml;       // [slot][2][warp][32]: (m, l) of each head row of that block
  uint16_t* q_lat;       // [B][2][128][Dl/2] fp16 latent query codes (prepared per call)
  uint8_t* q_rope;       // [B][QR_BYTES] bf16 RoPE query in core-matrix layout (prepared per call)
  int* seg_lo;           // [B]: first cluster of a split sequence, -1 if one cluster (or none) holds it
  int* seg_hi;           // [B]: last cluster of a split sequence
  int64_t* total_tiles;  // tiles of all sequences (written by the query pre-pass)
  int32_t* err;
  int B, H, Dl, Dr, T_max;
  int DH;                // Dl / 2
  int num_clusters;
  float sm_log2;         // softmax_scale * log2(e)
};

// Paged pool: tile tt of sequence b lies in the page that the block table names
// (page_size is a multiple of 64, so a tile never spans two pages).  The entry is
// loaded by page_ref and used only by page_row, one tile later, so that the load's
// latency is not spent waiting.
struct PageRef {
  int pg;    // block-table entry as loaded
  int off;   // row of the tile's first token inside that page
};
__device__ __forceinline__ PageRef page_ref(const MlaParams& p, int b, int tt) {
  const int t0 = tt * kTok;
  return PageRef{p.block_table[(int64_t)b * p.max_pages + t0 / p.page_size], t0 % p.page_size};
}
// Pool row of the tile's first token, or -1 when the entry is outside the pool.
__device__ __forceinline__ int64_t page_row(const MlaParams& p, PageRef r) {
  return (r.pg < 0 || r.pg >= p.num_pages) ? -1 : (int64_t)r.pg * p.page_size + r.off;
}

__device__ __forceinline__ int seq_tiles(const MlaParams& p, int b) {
  const int len = p.lens[b];
  if (len < 0 || len > p.T_max) return 0;
  return (len + kTok - 1) / kTok;
}

// Walks this cluster's segments (b, first tile, end tile) in order.
struct SegWalk {
  int64_t x0, x1, pre;
  int b;
  __device__ bool next(const MlaParams& p, int& sb, int& lo, int& hi, int& tb) {
    while (b < p.B && pre < x1) {
      const int t = seq_tiles(p, b);
      const int64_t l = max(x0, pre) - pre, h = min(x1, pre + t) - pre;
      const int cur = b;
      pre += t;
      ++b;
      if (h > l) {
        sb = cur; lo = (int)l; hi = (int)h; tb = t;
        return true;
      }
    }
    return false;
  }
};

// Walks this cluster's tiles one by one (sequence, tile index).
struct TileWalk {
  SegWalk w;
  int b = 0, tt = 0, hi = 0;
  bool valid = false;
  __device__ bool next(const MlaParams& p) {
    if (valid && tt + 1 < hi) { ++tt; return true; }
    int lo, tb;
    valid = w.next(p, b, lo, hi, tb);
    tt = lo;
    return valid;
  }
};

template <int DH, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1)
mla_decode_kernel(const __grid_constant__ MlaParams p) {
  constexpr int CONV_TOTAL = kTok * (DH / 16);      // 16-byte int8 chunks of a tile (this CTA's latent half)
  constexpr int CONV_UNITS = (CONV_TOTAL + kConvThreads - 1) / kConvThreads;   // per converter thread

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int cluster = blockIdx.x >> 1;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_ABORT);
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * (uint32_t)i; };
  // The RoPE term is split over the pair: CTA r contracts 16-wide chunks [rk0, rk1).
  const int rope_k = p.Dr / 16;
  const int rk0 = rank == 0 ? 0 : (rope_k + 1) / 2, rk1 = rank == 0 ? (rope_k + 1) / 2 : rope_k;
  const bool has_rope = rk1 > rk0;

  // ---- set-up: barriers, TMEM, schedule
  if (tid == 0) {
    for (int i = 0; i < NR; ++i) {
      mbar_init(bar(B_ROPE_FULL + i), 1);
      mbar_init(bar(B_ROPE_EMPTY + i), 1);
    }
    for (int i = 0; i < NC; ++i) {
      mbar_init(bar(B_C16_FULL + i), kConvThreads);
      mbar_init(bar(B_C16_EMPTY + i), 1);
    }
    mbar_init(bar(B_S_FULL), 1);            // latent and RoPE partial scores of a tile
    mbar_init(bar(B_S_EMPTY), kSmWarps);     // both read
    mbar_init(bar(B_P_FULL), kSmWarps);
    mbar_init(bar(B_PV_DONE), 1);
    mbar_init(bar(B_Q_READY), kSmWarps);
    mbar_init(bar(B_QR_FULL), 1);
    mbar_init(bar(B_QK_DONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    for (int i = 0; i < 2 * kSmWarps; ++i) {
      mbar_init(bar(B_XF + i), 1);
      mbar_init(bar(B_XE + i), 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(B_PAIR_W + i), 2);    // both warps of a lane quarter wrote their value
      mbar_init(bar(B_PAIR_R + i), 2);    // both warps of a lane quarter read the other's value
    }
    *abort_flag = 0u;
    // first use of every X region: expect the peer's 3 KB
    for (int i = 0; i < 2 * kSmWarps; ++i) mbar_expect_tx(bar(B_XF + i), kXWarpBytes);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(sbase + OFF_TMEM_SLOT), "r"(512) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp == 0) {
    // Even split of all tiles over the clusters; find this cluster's first sequence.
    int64_t total = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      int t = (b0 + lane < p.B) ? seq_tiles(p, b0 + lane) : 0;
      if (rank == 0 && cluster == 0 && b0 + lane < p.B) {
        const int len = p.lens[b0 + lane];
        if (len < 0 || len > p.T_max) set_dev_err(p.err, FA3_DEVERR_LENS);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      total += t;
    }
    const int64_t x0 = total * cluster / p.num_clusters;
    const int64_t x1 = total * (cluster + 1) / p.num_clusters;
    int64_t pre = 0;
    int bfirst = p.B;
    int64_t pfirst = total;
    for (int b0 = 0; b0 < p.B && bfirst == p.B; b0 += 32) {
      const int t = (b0 + lane < p.B) ? seq_tiles(p, b0 + lane) : 0;
      int incl = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      // first sequence whose tile range ends after x0
      const bool hit = (b0 + lane < p.B) && (pre + incl > x0);
      const uint32_t m = __ballot_sync(0xffffffffu, hit);
      if (m) {
        const int L = __ffs(m) - 1;
        bfirst = b0 + L;
        pfirst = pre + __shfl_sync(0xffffffffu, incl - t, L);
      }
      pre += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      int64_t* sched = reinterpret_cast<int64_t*>(smem + OFF_SCHED);
      sched[0] = bfirst; sched[1] = pfirst; sched[2] = x0; sched[3] = x1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();   // peer barriers are initialised before any remote arrive or copy

  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);
  const int64_t* sched = reinterpret_cast<const int64_t*>(smem + OFF_SCHED);
  // The prepared queries come from the pre-pass kernel, launched just before as
  // this kernel's programmatic prerequisite; the set-up above overlapped its tail.
  pdl_wait();
  pdl_launch_dependents();
  SegWalk walk0{sched[2], sched[3], sched[1], (int)sched[0]};
  // RoPE key TMA box: 2 * ((Dr/16 + 1) / 2) 8-wide chunks from chunk 2 * rk0 (a box
  // reaching past Dr is zero-filled and its bytes still count).
  const uint32_t rope_tx = (uint32_t)(kTok * 16 * 2 * ((rope_k + 1) / 2));

  if (warp >= kConvWarp0) {
    // ------------------------------------------------------ int8 -> fp16 converters
    // Unit u = (token u % 64, 16-byte chunk u / 64) of a tile; consecutive threads
    // take consecutive tokens.  Each thread loads its units of the next tile into
    // registers while the current one waits for its buffer.  Writes land as
    // K-major core matrices (8 tokens x 16 bytes): consecutive threads write
    // consecutive 16-byte rows, without bank conflicts.
    // The first converter thread also streams the RoPE key tiles in with TMA.
    const int ct = tid - kConvWarp0 * 32;
    const bool rope_issuer = (ct == 0) && has_rope;
    uint32_t it = 0;
    if constexpr (PAGED) {
      TileWalk tw{walk0};
      uint4 v[CONV_UNITS];
      // row0: the tile's first pool row (page_row of the entry loaded one tile earlier).
      auto load = [&](int tt, int64_t row0) {
        const int rows = row0 < 0 ? 0 : kTok;
        if (row0 < 0 && ct == 0) set_dev_err(p.err, FA3_DEVERR_PAGE);
#pragma unroll
        for (int i = 0; i < CONV_UNITS; ++i) {
          const int u = ct + kConvThreads * i, n = u % kTok, cc = u / kTok;
          v[i] = make_uint4(0u, 0u, 0u, 0u);
          if (u < CONV_TOTAL && n < rows)
            v[i] = __ldg(reinterpret_cast<const uint4*>(p.ckv + (row0 + n) * p.Dl + rank * DH) + cc);
        }
      };
      // The register loads run one tile ahead, which is shorter than the HBM latency:
      // the first converter thread of CTA 0 also prefetches into L2 the latent rows
      // (both halves) and RoPE key rows of the tile kPrefetch tiles ahead.
      constexpr int kPrefetch = 4;
      const bool pf_issuer = ct == 0 && rank == 0;
      TileWalk pfw{walk0};
      bool pf_more = pf_issuer && pfw.next(p);
      PageRef pf_ref = pf_more ? page_ref(p, pfw.b, pfw.tt) : PageRef{0, 0};
      // Prefetches pfw's tile, steps pfw, and loads the next tile's entry (used on the next call).
      auto prefetch = [&]() {
        const int64_t pf_row = page_row(p, pf_ref);
        if (pf_row >= 0) {
          prefetch_l2(p.ckv + pf_row * p.Dl, (uint32_t)(kTok * p.Dl));
          if (p.Dr > 0) prefetch_l2(p.krope + pf_row * p.Dr, (uint32_t)(kTok * p.Dr * 2));
        }
        pf_more = pfw.next(p);
        if (pf_more) pf_ref = page_ref(p, pfw.b, pfw.tt);
      };
      for (int i = 0; i < kPrefetch && pf_more; ++i) prefetch();
      // aw walks one tile ahead of tw, and its row is looked up while tw's tile
      // converts, so that the block-table load is off the path of the tile loads.
      TileWalk aw{walk0};
      bool more = tw.next(p);
      bool a_more = aw.next(p) && aw.next(p);
      int64_t cur_row = more ? page_row(p, page_ref(p, tw.b, tw.tt)) : 0;
      PageRef ahead = a_more ? page_ref(p, aw.b, aw.tt) : PageRef{0, 0};
      if (more) load(tw.tt, cur_row);
      bool ok = true;
      for (; ok && more; ++it) {
        if (pf_more) prefetch();
        if (rope_issuer) {
          const uint32_t st = it % NR;
          ok = wait_bar(bar(B_ROPE_EMPTY + st), ((it / NR) & 1u) ^ 1u, abort_flag, p.err);
          if (ok) {
            mbar_expect_tx(bar(B_ROPE_FULL + st), rope_tx);
            // Pool row of the tile (a bad page reads rows past the pool: zeros).
            const int y = cur_row < 0 ? p.num_pages * p.page_size : (int)cur_row;
            tma_4d(sbase + OFF_ROPE + st * ROPE_BYTES, &p.tm_rope, 0, y, 2 * rk0, 0, bar(B_ROPE_FULL + st));
          }
        }
        const uint32_t cs = it % NC;
        ok = ok && wait_bar(bar(B_C16_EMPTY + cs), ((it / NC) & 1u) ^ 1u, abort_flag, p.err);
        if (!ok) break;
        uint8_t* c16 = smem + OFF_C16 + cs * C16_BYTES;
#pragma unroll
        for (int i = 0; i < CONV_UNITS; ++i) {
          const int u = ct + kConvThreads * i, n = u % kTok, cc = u / kTok;
          if (u < CONV_TOTAL) {
            uint4 o0, o1;
            i8x4_to_f16x4(v[i].x, o0.x, o0.y);
            i8x4_to_f16x4(v[i].y, o0.z, o0.w);
            i8x4_to_f16x4(v[i].z, o1.x, o1.y);
            i8x4_to_f16x4(v[i].w, o1.z, o1.w);
            *reinterpret_cast<uint4*>(c16 + (2 * cc) * 1024 + n * 16) = o0;
            *reinterpret_cast<uint4*>(c16 + (2 * cc + 1) * 1024 + n * 16) = o1;
          }
        }
        fence_proxy_async();
        mbar_arrive(bar(B_C16_FULL + cs));
        more = tw.next(p);
        if (more) {
          cur_row = page_row(p, ahead);
          load(tw.tt, cur_row);
        }
        a_more = a_more && aw.next(p);
        if (a_more) ahead = page_ref(p, aw.b, aw.tt);
      }
    } else {
      TileWalk tw{walk0};
      uint4 v[CONV_UNITS];
      auto load = [&](int b, int tt) {
#pragma unroll
        for (int i = 0; i < CONV_UNITS; ++i) {
          const int u = ct + kConvThreads * i, n = u % kTok, cc = u / kTok;
          const int row = tt * kTok + n;
          v[i] = make_uint4(0u, 0u, 0u, 0u);
          if (u < CONV_TOTAL && row < p.T_max)
            v[i] = __ldg(reinterpret_cast<const uint4*>(p.ckv + ((int64_t)b * p.T_max + row) * p.Dl + rank * DH) + cc);
        }
      };
      // The register loads run one tile ahead, which is shorter than the HBM latency:
      // the first converter thread of CTA 0 also prefetches into L2 the latent rows
      // (both halves) and RoPE key rows of the tile kPrefetch tiles ahead.
      constexpr int kPrefetch = 4;
      const bool pf_issuer = ct == 0 && rank == 0;
      TileWalk pfw{walk0};
      auto prefetch = [&]() {
        const int rows = min(kTok, p.T_max - pfw.tt * kTok);
        const int64_t row0 = (int64_t)pfw.b * p.T_max + (int64_t)pfw.tt * kTok;
        prefetch_l2(p.ckv + row0 * p.Dl, (uint32_t)(rows * p.Dl));
        if (p.Dr > 0) prefetch_l2(p.krope + row0 * p.Dr, (uint32_t)(rows * p.Dr * 2));
      };
      bool pf_more = pf_issuer && pfw.next(p);
      for (int i = 0; i < kPrefetch && pf_more; ++i) {
        prefetch();
        pf_more = pfw.next(p);
      }
      bool more = tw.next(p);
      if (more) load(tw.b, tw.tt);
      bool ok = true;
      for (; ok && more; ++it) {
        if (pf_more) {
          prefetch();
          pf_more = pfw.next(p);
        }
        if (rope_issuer) {
          const uint32_t st = it % NR;
          ok = wait_bar(bar(B_ROPE_EMPTY + st), ((it / NR) & 1u) ^ 1u, abort_flag, p.err);
          if (ok) {
            mbar_expect_tx(bar(B_ROPE_FULL + st), rope_tx);
            tma_4d(sbase + OFF_ROPE + st * ROPE_BYTES, &p.tm_rope, 0, tw.tt * kTok, 2 * rk0, tw.b,
                   bar(B_ROPE_FULL + st));
          }
        }
        const uint32_t cs = it % NC;
        ok = ok && wait_bar(bar(B_C16_EMPTY + cs), ((it / NC) & 1u) ^ 1u, abort_flag, p.err);
        if (!ok) break;
        uint8_t* c16 = smem + OFF_C16 + cs * C16_BYTES;
#pragma unroll
        for (int i = 0; i < CONV_UNITS; ++i) {
          const int u = ct + kConvThreads * i, n = u % kTok, cc = u / kTok;
          if (u < CONV_TOTAL) {
            uint4 o0, o1;
            i8x4_to_f16x4(v[i].x, o0.x, o0.y);
            i8x4_to_f16x4(v[i].y, o0.z, o0.w);
            i8x4_to_f16x4(v[i].z, o1.x, o1.y);
            i8x4_to_f16x4(v[i].w, o1.z, o1.w);
            *reinterpret_cast<uint4*>(c16 + (2 * cc) * 1024 + n * 16) = o0;
            *reinterpret_cast<uint4*>(c16 + (2 * cc + 1) * 1024 + n * 16) = o1;
          }
        }
        fence_proxy_async();
        mbar_arrive(bar(B_C16_FULL + cs));
        more = tw.next(p);
        if (more) load(tw.b, tw.tt);
      }
    }
    // Drain: every issued RoPE copy must land before the CTA may exit.
    if (rope_issuer)
      for (uint32_t k = (it >= NR ? it - NR : 0); k < it; ++k)
        wait_bar(bar(B_ROPE_FULL + k % NR), (k / NR) & 1u, abort_flag, p.err);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_f16(128, kTok, false, false);
      const uint32_t id_rope = idesc_f16(128, kTok, true, false);
      const uint32_t id_pv = idesc_f16(128, DH, false, true);
      const uint32_t qr_bytes = (uint32_t)(rk1 - rk0) * 4096u;
      SegWalk w = walk0;
      int b, lo, hi, tb;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      // P.C of tile j; completion frees P and the C buffer.
      auto issue_pv = [&](uint32_t j, bool first) -> bool {
        if (!wait_bar(bar(B_P_FULL), j & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t cs = j % NC;
        const uint32_t pbase = sbase + OFF_P;
#pragma unroll
        for (int kk = 0; kk < kTok / 16; ++kk) {
          const uint64_t a = sdesc(pbase + kk * 4096, 2048, 128);
          // MN-major, no swizzle: LBO strides the K (token) core groups, SBO the N (latent) ones.
          const uint64_t bd = sdesc(sbase + OFF_C16 + cs * C16_BYTES + kk * 256, 128, 1024);
          mma_f16(tmem + TM_O, a, bd, id_pv, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(bar(B_PV_DONE));
        mma_commit(bar(B_C16_EMPTY + cs));
        return true;
      };
      // Q.C^T of tile j into S (latent partial scores) and this CTA's share of the
      // RoPE term into R; the last tile of a segment also releases both query operands.
      auto issue_qk = [&](uint32_t j, bool last) -> bool {
        const uint32_t cs = j % NC, st = j % NR;
        if (!(wait_bar(bar(B_C16_FULL + cs), (j / NC) & 1u, abort_flag, p.err) &&
              wait_bar(bar(B_S_EMPTY), (j & 1u) ^ 1u, abort_flag, p.err)))
          return false;
        if (has_rope && !wait_bar(bar(B_ROPE_FULL + st), (j / NR) & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint64_t bd = sdesc(sbase + OFF_C16 + cs * C16_BYTES + kk * 2048, 1024, 128);
          mma_f16_ts(tmem + TM_S, tmem + TM_QA + kk * 8, bd, id_qk, kk > 0 ? 1u : 0u);
        }
        for (int kk = rk0; kk < rk1; ++kk) {
          const uint64_t a = sdesc(sbase + OFF_QR + (kk - rk0) * 4096, 2048, 128);
          const uint64_t bd = sdesc(sbase + OFF_ROPE + st * ROPE_BYTES + (kk - rk0) * 2048, 1024, 128);
          mma_f16(tmem + TM_R, a, bd, id_rope, kk > rk0 ? 1u : 0u);
        }
        mma_commit(bar(B_S_FULL));
        mma_commit(bar(B_ROPE_EMPTY + st));
        if (last) mma_commit(bar(B_QK_DONE));
        return true;
      };
      while (ok && w.next(p, b, lo, hi, tb)) {
        // The RoPE query image of this sequence replaces the previous one once the
        // previous segment's scores are done with it.
        if (seg > 0) ok = wait_bar(bar(B_QK_DONE), (seg - 1) & 1u, abort_flag, p.err);
        if (!ok) break;
        if (qr_bytes) {
          mbar_expect_tx(bar(B_QR_FULL), qr_bytes);
          bulk_g2s(sbase + OFF_QR, p.q_rope + (size_t)b * QR_BYTES + rk0 * 4096, qr_bytes, bar(B_QR_FULL));
          ok = wait_bar(bar(B_QR_FULL), seg & 1u, abort_flag, p.err);
        }
        ok = ok && wait_bar(bar(B_Q_READY), seg & 1u, abort_flag, p.err);   // latent query in TMEM
        ++seg;
        // Order on the tensor pipe: Q.C^T runs two tiles ahead of P.C, so that the
        // softmax finds the next tile's partial scores ready while it works on the
        // current one.
        const uint32_t n = (uint32_t)(hi - lo), base = it;
        ok = ok && issue_qk(base, n == 1) && (n < 2 || issue_qk(base + 1, n == 2));
        for (uint32_t k = 0; k < n && ok; ++k) {
          if (k + 2 < n) ok = issue_qk(base + k + 2, k + 3 == n);
          if (ok) ok = issue_pv(base + k, k == 0);
        }
        it = base + n;
      }
      // Drain every MMA this thread issued before the CTA may release TMEM.
      mma_commit(bar(B_DRAIN));
      wait_bar(bar(B_DRAIN), 0, abort_flag, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    // Warp w handles heads 32*(w%4) .. +31 (its TMEM lane quarter) and the tile's
    // tokens 32*(w/4) .. +31; the two warps of a quarter agree on the row maximum
    // through shared memory and each keeps its own part of the row sum.
    const int qd = warp & 3, hf = warp >> 2;
    const int h = qd * 32 + lane;                          // head == TMEM lane
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    float* mx_own = reinterpret_cast<float*>(smem + OFF_MX) + hf * kRows + h;
    const float* mx_oth = reinterpret_cast<const float*>(smem + OFF_MX) + (hf ^ 1) * kRows + h;
    const float kvs = p.kv_scale[0];
    const float c_rope = p.sm_log2;
    const float c_lat = (h < p.H ? p.q_scale[h] : 0.f) * kvs * p.sm_log2;
    const uint32_t region = (uint32_t)warp * kXWarpBytes + (uint32_t)lane * 16;   // + slot, + chunk * 512
    const uint32_t peer_x = mapa(sbase + OFF_X, peer);
    const uint32_t peer_xf = mapa(bar(B_XF), peer);
    // Column ranges of O (fp32 words) and of the fp16 query (32-bit words) this warp handles.
    constexpr int O_PER = DH >= 64 ? DH / 2 : DH;
    constexpr int QW = DH / 2, QW_PER = QW >= 16 ? QW / 2 : QW;
    const int o_lo = hf * O_PER, o_hi = min(DH, o_lo + O_PER);
    const int q_lo = hf * QW_PER, q_hi = min(QW, q_lo + QW_PER);
    uint32_t n_pair = 0;
    // One arrival per softmax warp (the warp-collective waits and __syncwarp order
    // every lane's work before it).
    auto warp_arrive = [&](int which) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(which));
    };
    const uint32_t peer_xe = mapa(bar(B_XE), peer);
    // This CTA's partial score of tile j for this warp's 32 tokens, in log2 units:
    //   (latent partial) * q_scale * kv_scale * c + (RoPE share) * c.
    // It stays in registers (own) and goes, as fp32, into the peer's X slot by
    // st.async; both CTAs then add the same two values, so their scores agree bit
    // for bit.
    float own[32];
    auto send_partial = [&](uint32_t j) -> bool {
      const uint32_t s = j & 1u, xe = s * kSmWarps + (uint32_t)warp;
      // XE: the peer's warp has read tile j-2 from this slot.
      if (!warp_all(wait_bar(bar(B_S_FULL), j & 1u, abort_flag, p.err)) ||
          !warp_all(wait_bar(bar(B_XE + xe), ((j >> 1) & 1u) ^ 1u, abort_flag, p.err, true)))
        return false;
      tc_fence_after();
      const uint32_t dst = peer_x + s * kXSlotBytes + region;
      const uint32_t rbar = peer_xf + 8u * xe;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t v[16], r[16];
        FA3_TMEM_LD16(tmem + lane_base + TM_S + hf * 32 + hh * 16, v);
        if (has_rope) FA3_TMEM_LD16(tmem + lane_base + TM_R + hf * 32 + hh * 16, r);
        tmem_wait_ld();
        float* o = own + 16 * hh;
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          float r0 = 0.f, r1 = 0.f;
          if (has_rope) mul2(r0, r1, __uint_as_float(r[i]), __uint_as_float(r[i + 1]), c_rope, c_rope);
          fma2(o[i], o[i + 1], __uint_as_float(v[i]), __uint_as_float(v[i + 1]), c_lat, c_lat, r0, r1);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
          asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
                       ::"r"(dst + (4 * hh + c) * 512), "r"(__float_as_uint(o[4 * c])),
                         "r"(__float_as_uint(o[4 * c + 1])), "r"(__float_as_uint(o[4 * c + 2])),
                         "r"(__float_as_uint(o[4 * c + 3])), "r"(rbar) : "memory");
      }
      tc_fence_before();
      warp_arrive(B_S_EMPTY);
      return true;
    };
    // Swaps one float per head with the other warp of this lane quarter, in two
    // halves so that other work can run between them.
    auto pair_put = [&](float mine) -> bool {
      if (n_pair > 0 && !warp_all(wait_bar(bar(B_PAIR_R + qd), (n_pair - 1) & 1u, abort_flag, p.err)))
        return false;                                       // the other warp still reads the previous value
      *mx_own = mine;
      warp_arrive(B_PAIR_W + qd);
      return true;
    };
    auto pair_get = [&](float& other) -> bool {
      if (!warp_all(wait_bar(bar(B_PAIR_W + qd), n_pair & 1u, abort_flag, p.err))) return false;
      other = *mx_oth;
      warp_arrive(B_PAIR_R + qd);
      ++n_pair;
      return true;
    };
    SegWalk w = walk0;
    int b, lo, hi, tb;
    uint32_t it = 0;
    bool ok = true;
    while (ok && w.next(p, b, lo, hi, tb)) {
      // ---- latent query of this sequence into TMEM (the previous segment's last
      //      Q.C^T has completed: this thread consumed its scores)
      {
        const uint4* src = reinterpret_cast<const uint4*>(p.q_lat + (((size_t)b * 2 + rank) * kRows + h) * DH);
#pragma unroll 1
        for (int c0 = q_lo; c0 < q_hi; c0 += 8) {
          const uint4 v0 = src[c0 / 4], v1 = src[c0 / 4 + 1];
          asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                       ::"r"(tmem + lane_base + TM_QA + c0), "r"(v0.x), "r"(v0.y), "r"(v0.z), "r"(v0.w), "r"(v1.x),
                         "r"(v1.y), "r"(v1.z), "r"(v1.w));
        }
        tmem_wait_st();
      }
      tc_fence_before();
      warp_arrive(B_Q_READY);

      const int len = p.lens[b];
      float m_ref = -CUDART_INF_F, l = 0.f;
      ok = send_partial(it);
      for (int tt = lo; tt < hi && ok; ++tt, ++it) {
        const uint32_t s = it & 1u, use = (it >> 1) & 1u, xs = s * kSmWarps + (uint32_t)warp;
        const int nvalid = min(kTok, len - tt * kTok) - hf * 32;   // valid tokens in this warp's half
        ok = warp_all(wait_bar(bar(B_XF + xs), use, abort_flag, p.err, true));
        if (!ok) break;
        // ---- scores: own + peer partial (the same two values in both CTAs)
        float part[32];
        {
          const uint32_t xo_ = OFF_X + s * kXSlotBytes + region;
#pragma unroll
          for (int c = 0; c < kXChunks; ++c) {
            const float4 xo = *reinterpret_cast<const float4*>(smem + xo_ + c * 512);
            add2(part[4 * c], part[4 * c + 1], own[4 * c], own[4 * c + 1], xo.x, xo.y);
            add2(part[4 * c + 2], part[4 * c + 3], own[4 * c + 2], own[4 * c + 3], xo.z, xo.w);
          }
        }
        // This warp's X region is consumed: expect the peer's tile after next and
        // tell the peer's warp that the region is free.
        __syncwarp();
        if (lane == 0) {
          mbar_expect_tx(bar(B_XF + xs), kXWarpBytes);
          mbar_arrive_remote(peer_xe + 8u * xs);
        }
        // The next tile's partial goes out now: its copy has the rest of this tile to land.
        if (tt + 1 < hi) {
          ok = send_partial(it + 1);
          if (!ok) break;
        }
        if (nvalid < 32) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) part[jj] = jj < nvalid ? part[jj] : -CUDART_INF_F;
        }
        // tile maximum of this half as a tree (short dependency chains), then across the pair
        float mx[11];
#pragma unroll
        for (int q = 0; q < 10; ++q) mx[q] = max3(part[3 * q], part[3 * q + 1], part[3 * q + 2]);
        mx[10] = fmaxf(part[30], part[31]);
        const float mh = fmaxf(max3(max3(mx[0], mx[1], mx[2]), max3(mx[3], mx[4], mx[5]), max3(mx[6], mx[7], mx[8])),
                               fmaxf(mx[9], mx[10]));
        float mo;
        ok = pair_put(mh) && pair_get(mo);
        if (!ok) break;
        const float mt = fmaxf(mh, mo);

        // ---- online softmax with a lazily moved reference maximum (both warps of
        //      the pair take the same decisions from the same tile maximum)
        float alpha = 1.f;
        bool rescale = false;
        if (mt > m_ref + 8.f) {
          alpha = (m_ref == -CUDART_INF_F) ? 0.f : ex2_approx(m_ref - mt);
          rescale = tt > lo;
          m_ref = mt;
        }
        uint32_t pk[16];
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float d0, d1;
          add2(d0, d1, part[2 * j], part[2 * j + 1], -m_ref, -m_ref);
          const float e0 = ex2_approx(d0), e1 = ex2_approx(d1);
          pk[j] = pack_f16x2(e0, e1);
          add2(ps[2 * (j & 1)], ps[2 * (j & 1) + 1], ps[2 * (j & 1)], ps[2 * (j & 1) + 1], e0, e1);
        }
        l = l * alpha + ((ps[0] + ps[1]) + (ps[2] + ps[3]));
        // P is single-buffered and O must hold P.C of the previous tile.
        if (tt > lo) {
          ok = warp_all(wait_bar(bar(B_PV_DONE), (it - 1) & 1u, abort_flag, p.err));
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int kc = 0; kc < 4; ++kc)
          *reinterpret_cast<uint4*>(smem + OFF_P + (4 * hf + kc) * 2048 + (h >> 3) * 128 + (h & 7) * 16) =
              make_uint4(pk[4 * kc], pk[4 * kc + 1], pk[4 * kc + 2], pk[4 * kc + 3]);
        // The rescale is decided per head (lane) but tcgen05.ld/st are warp-wide:
        // the whole warp takes part, lanes that keep their reference scale by 1.
        // O must already hold P.C of the previous tile.
        if (__any_sync(0xffffffffu, rescale)) {
          if (!rescale) alpha = 1.f;
#pragma unroll 1
          for (int c0 = o_lo; c0 < o_hi; c0 += 32) {
            uint32_t v[32];
            FA3_TMEM_LD32(tmem + lane_base + TM_O + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
            FA3_TMEM_ST32(tmem + lane_base + TM_O + c0, v);
          }
          tmem_wait_st();
        }
        fence_proxy_async();
        tc_fence_before();
        warp_arrive(B_P_FULL);
      }
      if (!ok) break;
      // ---- segment done: the row sum over both halves, then wait for the last
      //      P.C and write the output (or a partial)
      float lo_sum;
      ok = pair_put(l) && pair_get(lo_sum);
      if (!ok) break;
      const float l_row = l + lo_sum;
      ok = warp_all(wait_bar(bar(B_PV_DONE), (it - 1) & 1u, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      const bool full = (lo == 0 && hi == tb);
      const float inv = (full && l_row > 0.f) ? kvs / l_row : 0.f;
      // A split sequence leaves this warp's block of O (its 32 head rows x its O
      // columns, unnormalised, lane-interleaved float4 columns) and the rows' (m, l)
      // in the workspace slot of (sequence + cluster) for mla_combine_kernel.
      const int64_t blk = ((int64_t)(b + cluster) * 2 + rank) * kSmWarps + warp;
      float* blk_o = p.part_o + blk * (32 * O_PER);
#pragma unroll 1
      for (int c0 = o_lo; c0 < o_hi; c0 += 32) {
        uint32_t v[32];
        FA3_TMEM_LD32(tmem + lane_base + TM_O + c0, v);
        tmem_wait_ld();
        if (full) {
          if (h < p.H) {
            float* dst = p.out + ((int64_t)b * p.H + h) * p.Dl + rank * DH + c0;
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + j) =
                  make_float4(__uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv,
                              __uint_as_float(v[j + 2]) * inv, __uint_as_float(v[j + 3]) * inv);
          }
        } else {
          const int j0 = (c0 - o_lo) / 4;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(blk_o + ((j0 + q) * 32 + lane) * 4) =
                make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
      }
      if (!full && o_lo < o_hi) p.part_ml[blk * 32 + lane] = make_float2(m_ref, l_row);
      tc_fence_before();
    }
  }

  // ---- teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();     // the peer no longer writes into this CTA's shared memory
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

// Quantizes every latent query once per call (per-head static scale, exact
// codes stored as fp16, row-major per (sequence, latent half, head) for the
// TMEM A operand) and lays out the RoPE query of each sequence as the
// shared-memory image of K-major core matrices (8 heads x 8 values).
// One thread per 8 values of one (sequence, head); heads >= H are zero.  Also
// writes the zero output rows of sequences without tiles and lists the clusters
// of every split sequence for mla_combine_kernel.
__global__ void __launch_bounds__(256, 6) mla_prepare_q_kernel(const MlaParams p) {
  pdl_wait();
  pdl_launch_dependents();   // the decode kernel may start its set-up
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 32) {
    // Clusters of each sequence under the decode kernel's even split of all tiles
    // (cluster c covers tile positions [total*c/C, total*(c+1)/C)).
    const int lane = threadIdx.x;
    const int C = p.num_clusters;
    int64_t total = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      int t = b0 + lane < p.B ? seq_tiles(p, b0 + lane) : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      total += t;
    }
    if (lane == 0) *p.total_tiles = total;
    // the cluster whose range holds tile position x: the largest c with total*c/C <= x
    auto owner = [&](int64_t x) -> int { return (int)min((int64_t)(C - 1), ((x + 1) * C - 1) / total); };
    int64_t pre = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int bb = b0 + lane;
      const int t = bb < p.B ? seq_tiles(p, bb) : 0;
      int incl = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (bb < p.B) {
        const int64_t start = pre + incl - t;
        int c0 = -1, c1 = -1;
        if (t > 0) {
          c0 = owner(start);
          c1 = owner(start + t - 1);
          if (c0 == c1) c0 = c1 = -1;
        }
        p.seg_lo[bb] = c0;
        p.seg_hi[bb] = c1;
      }
      pre += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  // Block row y = sequence; one 16-byte item per thread: the latent items first
  // (head = idx / chunks, chunks = Dl / 8 a power of two), then the RoPE items.
  const int b = blockIdx.y;
  const int lat_shift = __ffs(p.Dl / 8) - 1;
  const int n_lat = kRows << lat_shift, chunks_rope = p.Dr / 8;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const uint16_t* qb = p.q + (int64_t)b * p.H * (p.Dl + p.Dr);
  if (idx < n_lat) {
    const int h = idx >> lat_shift, c = idx & ((1 << lat_shift) - 1);
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (h < p.H) {
      const uint4 v = *reinterpret_cast<const uint4*>(qb + (int64_t)h * (p.Dl + p.Dr) + 8 * c);
      const float qs = p.q_scale[h];
      if (seq_tiles(p, b) == 0) {      // no tiles (length 0 or invalid): a zero output row
        float4* orow = reinterpret_cast<float4*>(p.out + ((int64_t)b * p.H + h) * p.Dl + 8 * c);
        orow[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        orow[1] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      int q8[8];
      quant_group8_biased(v, qs, rcp_approx(qs), exact_scale(qs), q8);
      uint32_t r4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        r4[e] = pack_f16x2(__int_as_float(q8[2 * e]) - kCodeMagic, __int_as_float(q8[2 * e + 1]) - kCodeMagic);
      o = make_uint4(r4[0], r4[1], r4[2], r4[3]);
    }
    const int hc = 1 << (lat_shift - 1);              // chunks per latent half
    const int r = c >> (lat_shift - 1), k = c & (hc - 1);
    *reinterpret_cast<uint4*>(p.q_lat + (((int64_t)b * 2 + r) * kRows + h) * p.DH + 8 * k) = o;
  } else if (idx < n_lat + kRows * chunks_rope) {
    const int j = idx - n_lat, h = j / chunks_rope, k = j - h * chunks_rope;
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (h < p.H) o = *reinterpret_cast<const uint4*>(qb + (int64_t)h * (p.Dl + p.Dr) + p.Dl + 8 * k);
    *reinterpret_cast<uint4*>(p.q_rope + (int64_t)b * QR_BYTES + k * 2048 + (h >> 3) * 128 + (h & 7) * 16) = o;
  }
}

// Merges the segments of every split sequence with log-sum-exp weights.  One
// block per (sequence, latent half, softmax-warp block of 32 heads x O columns):
// the (m, l) pairs of all segments in one round of loads, the per-head weights,
// then every column as the weighted sum of the segments' blocks (two segments'
// loads in flight per thread, four blocks resident per SM: one wave for the
// usual sizes), transposed through shared memory into coalesced output rows.  Launched as the decode kernel's programmatic dependent: it waits
// for that grid before reading the partials.
template <int DH>
__global__ void __launch_bounds__(256, 4) mla_combine_kernel(const MlaParams p) {
  constexpr int O_PER = DH >= 64 ? DH / 2 : DH;
  constexpr int NQ = O_PER / 4;                        // float4 columns of a block row
  constexpr int PER = (32 * NQ + 255) / 256;           // float4 positions per thread
  constexpr int KB = 2;                                // segments per round of loads
  extern __shared__ float csm[];
  float* tile = csm;                                   // [32][O_PER + 4]
  float* wts = tile + 32 * (O_PER + 4);                // [segments][32]
  float2* mls = reinterpret_cast<float2*>(wts + 32 * p.num_clusters);   // [segments][32]
  pdl_wait();
  const int b = blockIdx.x, rank = blockIdx.y / kSmWarps, wp = blockIdx.y % kSmWarps;
  const int hf = wp >> 2, qd = wp & 3;
  const int c_first = p.seg_lo[b], c_last = p.seg_hi[b];
  const int64_t total = *p.total_tiles;
  if (c_first < 0 || hf * O_PER >= DH) return;
  const int tid = threadIdx.x, lane = tid & 31;
  const int C = p.num_clusters;
  auto covers = [&](int c) -> bool { return total >= C || total * c / C < total * (c + 1) / C; };
  auto blk = [&](int c) -> int64_t { return ((int64_t)(b + c) * 2 + rank) * kSmWarps + wp; };
  const int n = c_last - c_first + 1;
  for (int k = tid >> 5; k < n; k += 8)
    mls[k * 32 + lane] = covers(c_first + k) ? __ldcg(p.part_ml + blk(c_first + k) * 32 + lane)
                                             : make_float2(-CUDART_INF_F, 0.f);
  __syncthreads();
  if (tid < 32) {
    float M = -CUDART_INF_F;
    for (int k = 0; k < n; ++k) M = fmaxf(M, mls[k * 32 + lane].x);
    float L = 0.f;
    for (int k = 0; k < n; ++k) {
      const float2 ml = mls[k * 32 + lane];
      const float w = ml.y > 0.f ? exp2f(ml.x - M) : 0.f;
      wts[k * 32 + lane] = w;
      L += ml.y * w;
    }
    const float f = L > 0.f ? p.kv_scale[0] / L : 0.f;
    for (int k = 0; k < n; ++k) wts[k * 32 + lane] *= f;
  }
  __syncthreads();
  float4 acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < n; k0 += KB) {
    float4 v[KB][PER];
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      const int k = k0 + u;
      const bool use = k < n && wts[min(k, n - 1) * 32 + lane] != 0.f;
      const float4* src = reinterpret_cast<const float4*>(p.part_o + blk(c_first + min(k, n - 1)) * (32 * O_PER));
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int pos = tid + 256 * i;
        v[u][i] = (use && pos < 32 * NQ) ? __ldcg(src + pos) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < KB; ++u) {
      const float w = k0 + u < n ? wts[(k0 + u) * 32 + lane] : 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        acc[i].x = fmaf(v[u][i].x, w, acc[i].x); acc[i].y = fmaf(v[u][i].y, w, acc[i].y);
        acc[i].z = fmaf(v[u][i].z, w, acc[i].z); acc[i].w = fmaf(v[u][i].w, w, acc[i].w);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int pos = tid + 256 * i;
    if (pos < 32 * NQ) *reinterpret_cast<float4*>(tile + lane * (O_PER + 4) + 4 * (pos >> 5)) = acc[i];
  }
  __syncthreads();
  for (int i = tid; i < 32 * NQ; i += 256) {
    const int r = i / NQ, q = i - r * NQ, hh = qd * 32 + r;
    if (hh < p.H)
      *reinterpret_cast<float4*>(p.out + ((int64_t)b * p.H + hh) * p.Dl + rank * DH + hf * O_PER + 4 * q) =
          *reinterpret_cast<const float4*>(tile + r * (O_PER + 4) + 4 * q);
  }
}

// Number of 2-CTA clusters that can be resident at once (cached per device).
int max_clusters() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(mla_decode_kernel<256, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2; attr.val.clusterDim.y = 1; attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  // Every width instantiation has the same block size and shared memory, hence the same residency.
  if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel<256, false>, &cfg) != cudaSuccess || n <= 0) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

bool mla_shape_ok(int H, int Dl, int Dr) {
  const bool dl_ok = Dl == 64 || Dl == 128 || Dl == 256 || Dl == 512;
  return H >= 1 && H <= kRows && dl_ok && Dr >= 0 && Dr <= 64 && Dr % 16 == 0;
}


// Decode kernel (timed by the optional caller events) and its combine kernel.
template <int DH>
cudaError_t launch_mla(cudaLaunchConfig_t cfg, cudaLaunchConfig_t ccfg, const MlaParams& prm) {
  auto* kernel = prm.block_table ? mla_decode_kernel<DH, true> : mla_decode_kernel<DH, false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  e = cudaLaunchKernelEx(&cfg, kernel, prm);
  timing_end(cfg.stream);
  if (e != cudaSuccess) return e;
  constexpr int O_PER = DH >= 64 ? DH / 2 : DH;
  ccfg.dynamicSmemBytes = (size_t)32 * (O_PER + 4) * sizeof(float) + (size_t)prm.num_clusters * 32 * 3 * sizeof(float);
  if (ccfg.dynamicSmemBytes > 48 * 1024) {
    e = cudaFuncSetAttribute(mla_combine_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)ccfg.dynamicSmemBytes);
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&ccfg, mla_combine_kernel<DH>, prm);
}

}  // namespace
}  // namespace fa3

using namespace fa3;

namespace {
// Workspace: per partial slot (sequence + cluster) and latent half, one block per
// softmax warp (32 head rows x that warp's O columns) and its (m, l) pairs; then the
// prepared queries, the total tile count and the clusters of each split sequence.
size_t mla_ws_parts(int B, int Dl, int C, size_t* off_ml, size_t* off_qlat, size_t* off_qrope, size_t* off_seg) {
  const size_t slots = (size_t)B + (size_t)C;
  const int DH = Dl / 2, o_cols = DH >= 64 ? DH / 2 : DH;
  size_t off = slots * 2 * kSmWarps * 32 * (size_t)o_cols * sizeof(float);
  *off_ml = off;
  off += slots * 2 * kSmWarps * 32 * sizeof(float2);
  off = (off + 255) & ~size_t(255);
  *off_qlat = off;
  off += (size_t)B * kRows * (size_t)Dl * sizeof(uint16_t);
  off = (off + 255) & ~size_t(255);
  *off_qrope = off;
  off += (size_t)B * QR_BYTES;
  off = (off + 255) & ~size_t(255);
  *off_seg = off;
  off += sizeof(int64_t) + (size_t)B * 2 * sizeof(int);
  return off + 256;
}
}  // namespace

FA3_API size_t fa3_mla_workspace_size(int B, int H, int Dl, int T_max) {
  if (B <= 0 || H <= 0 || Dl <= 0 || T_max <= 0) return 0;
  int C = 0;
  if (check_device(nullptr) == FA3_OK) C = max_clusters();
  if (C <= 0) C = 128;
  size_t a, b2, c, d;
  return mla_ws_parts(B, Dl, C, &a, &b2, &c, &d);
}

namespace {
// Both layouts: block_table == nullptr is the contiguous [B][T_max] cache; otherwise
// ckv / krope are pools of num_pages pages of page_size rows and T_max = max_pages * page_size.
int mla_decode(const uint16_t* q, const int8_t* ckv, const uint16_t* krope, const float* q_scale,
               const float* kv_scale, const int32_t* lens, const int32_t* block_table, float* out, int B, int H,
               int Dl, int Dr, int T_max, int num_pages, int page_size, int max_pages, float softmax_scale,
               void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (!q || !ckv || !q_scale || !kv_scale || !lens || !out) return FA3_EINVAL;
  if (Dr > 0 && !krope) return FA3_EINVAL;
  if (B <= 0 || H <= 0 || Dl <= 0 || Dr < 0 || T_max <= 0) return FA3_EINVAL;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return FA3_EINVAL;
  if (!mla_shape_ok(H, Dl, Dr) || B > 65535 || T_max > (1 << 30) / 2) return FA3_ERANGE;
  if (!aligned16(q) || !aligned16(ckv) || (Dr > 0 && !aligned16(krope)) || !aligned16(out)) return FA3_ERANGE;
  int st = check_device(nullptr);
  if (st != FA3_OK) return st;
  const int C = max_clusters();
  if (C <= 0) return FA3_ECUDA;
  size_t off_ml, off_qlat, off_qrope, off_seg;
  const size_t need = mla_ws_parts(B, Dl, C, &off_ml, &off_qlat, &off_qrope, &off_seg);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FA3_EWORKSPACE;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return FA3_ECUDA;

  MlaParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.DH = Dl / 2;
  if (Dr > 0) {
    // (8 values, token, 8-wide chunk, sequence): one box lands as K-major core matrices.
    // A paged pool is one "sequence" of num_pages * page_size rows.
    const cuuint64_t rows = block_table ? (cuuint64_t)num_pages * page_size : (cuuint64_t)T_max;
    const cuuint64_t dims[4] = {8, rows, (cuuint64_t)(Dr / 8), block_table ? 1u : (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)Dr * 2, 16, (cuuint64_t)Dr * 2 * rows};
    // one CTA's share: 2 * ((Dr/16 + 1) / 2) chunks (the decode kernel's RoPE split over the pair)
    const cuuint32_t box[4] = {8, (cuuint32_t)kTok, (cuuint32_t)(2 * ((Dr / 16 + 1) / 2)), 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    if (encode(&prm.tm_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(krope), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FA3_ECUDA;
  }
  char* ws = static_cast<char*>(workspace);
  prm.q = q; prm.ckv = ckv; prm.krope = krope; prm.q_scale = q_scale; prm.kv_scale = kv_scale; prm.lens = lens; prm.out = out;
  prm.part_o = reinterpret_cast<float*>(ws);
  prm.part_ml = reinterpret_cast<float2*>(ws + off_ml);
  prm.q_lat = reinterpret_cast<uint16_t*>(ws + off_qlat);
  prm.q_rope = reinterpret_cast<uint8_t*>(ws + off_qrope);
  prm.total_tiles = reinterpret_cast<int64_t*>(ws + off_seg);
  prm.seg_lo = reinterpret_cast<int*>(ws + off_seg + sizeof(int64_t));
  prm.seg_hi = prm.seg_lo + B;
  prm.err = dev_err;
  prm.B = B; prm.H = H; prm.Dl = Dl; prm.Dr = Dr; prm.T_max = T_max;
  prm.block_table = block_table; prm.num_pages = num_pages; prm.page_size = page_size; prm.max_pages = max_pages;
  prm.num_clusters = C;
  prm.sm_log2 = softmax_scale * 1.4426950408889634f;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    const int per_seq = kRows * ((Dl + Dr) / 8);
    if (launch_pdl(mla_prepare_q_kernel, dim3((unsigned)((per_seq + 255) / 256), (unsigned)B), dim3(256), 0, s,
                   prm) != cudaSuccess)
      return FA3_ECUDA;
  }
  // The decode kernel and the combine kernel are programmatic dependents of the
  // kernel before them: their launch and set-up overlap its tail.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2; attr[0].val.clusterDim.y = 1; attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaLaunchConfig_t ccfg = {};
  ccfg.gridDim = dim3(B, 2 * kSmWarps, 1);
  ccfg.blockDim = dim3(256, 1, 1);
  ccfg.stream = s;
  ccfg.attrs = &attr[1];
  ccfg.numAttrs = 1;
  cudaError_t le = cudaErrorInvalidValue;
  timing_begin(s);
  switch (prm.DH) {
    case 32: le = launch_mla<32>(cfg, ccfg, prm); break;
    case 64: le = launch_mla<64>(cfg, ccfg, prm); break;
    case 128: le = launch_mla<128>(cfg, ccfg, prm); break;
    case 256: le = launch_mla<256>(cfg, ccfg, prm); break;
  }
  if (le != cudaSuccess) return FA3_ECUDA;
  return cuda_status(cudaGetLastError());
}
}  // namespace

FA3_API int fa3_decode_attn_mla(const uint16_t* q, const int8_t* ckv, const uint16_t* krope, const float* q_scale,
                                const float* kv_scale, const int32_t* lens, float* out, int B, int H, int Dl,
                                int Dr, int T_max, float softmax_scale, void* workspace, size_t workspace_bytes,
                                int32_t* dev_err, void* stream) {
  return mla_decode(q, ckv, krope, q_scale, kv_scale, lens, nullptr, out, B, H, Dl, Dr, T_max, 0, 0, 0,
                    softmax_scale, workspace, workspace_bytes, dev_err, stream);
}

FA3_API int fa3_decode_attn_mla_paged(const uint16_t* q, const int8_t* ckv, const uint16_t* krope,
                                      const float* q_scale, const float* kv_scale, const int32_t* lens,
                                      const int32_t* block_table, float* out, int B, int H, int Dl, int Dr,
                                      int num_pages, int page_size, int max_pages, float softmax_scale,
                                      void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (!block_table) return FA3_EINVAL;
  if (num_pages <= 0 || page_size <= 0 || max_pages <= 0) return FA3_EINVAL;
  if (page_size % kTok != 0 || (int64_t)num_pages * page_size >= ((int64_t)1 << 31) ||
      (int64_t)max_pages * page_size > (1 << 30) / 2)
    return FA3_ERANGE;
  return mla_decode(q, ckv, krope, q_scale, kv_scale, lens, block_table, out, B, H, Dl, Dr, max_pages * page_size,
                    num_pages, page_size, max_pages, softmax_scale, workspace, workspace_bytes, dev_err, stream);
}
