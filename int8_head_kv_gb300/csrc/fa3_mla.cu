// Absorbed-MLA decode attention over an INT8 latent cache (tcgen05 + TMA, sm_103a).
//
// MindIE "FA3 quantization", Overview: for MLA only the non-RoPE part of K (the
// latent c_kv, shared by K-nope and V) is quantized to 8 bits per head; the
// RoPE part of K stays in floating point; the decode-phase attention operator
// reads the INT8 cache.  Scales are the symmetric per-head ones of msModelSlim
// "FA3量化" 原理 / 算法流程 step 4; the latent query is quantized with its static
// per-head scale so that the score contraction is an integer one.
//
//   s[h, j] = (sum_c q8[h, c] ckv[j, c]) * q_scale[h] * kv_scale + q_rope[h] . k_rope[j]
//   out[h]  = kv_scale * sum_j softmax(s * softmax_scale)_j * ckv[j, :]
//
// GB300 design (tcgen05 has no int8 MMA kind on sm_103a):
//   * int8 codes are exact in fp16, and every partial sum of products of two
//     codes over <= 256 terms stays below 2^24, so a kind::f16 MMA with fp32
//     accumulation returns the exact integer latent score;
//   * the fp32 output accumulator of 128 heads x 512 latent is 256 KB -- all of
//     one SM's TMEM -- so a 2-CTA cluster splits the latent in halves: CTA r
//     owns latent columns [r*Dl/2, (r+1)*Dl/2) (and half of the RoPE dims),
//     TMA-loads only that half of each 64-token tile, converts it to fp16 in
//     shared memory, and computes a partial score over its half;
//   * the two CTAs swap their fp32 partial scores through distributed shared
//     memory and both run the same online softmax (fp32 addition commutes, so
//     both see bit-identical scores, maxima and P);
//   * P (fp16) . C_r accumulates the CTA's half of O in TMEM; the same fp16
//     tile serves as the K-major B operand of Q.C^T and the MN-major B operand
//     of P.C;
//   * warp roles: 4 softmax warps (one TMEM lane = one head each), 1 TMA
//     producer, 1 MMA issuer, 4 int8->fp16 converter warps;
//   * split-K: the tiles of all sequences are dealt out evenly to the clusters
//     that fit on the GPU; a cluster's piece of a sequence is a segment; split
//     sequences are merged by a small log-sum-exp combine kernel.
// Every wait is bounded; on time-out the kernel sets FA3_DEVERR_TIMEOUT, drains
// its own copies and MMAs, frees its TMEM and returns.
#include "fa3_common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <math_constants.h>

namespace fa3 {
namespace {

constexpr int kTok = 64;          // tokens per tile
constexpr int kThreads = 320;     // 10 warps
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kConvWarp0 = 6;
constexpr int kConvThreads = 128;
constexpr int kRows = 128;        // heads (TMEM lanes)

// Shared memory map (bytes from a 1024-byte aligned base).
constexpr uint32_t OFF_Q = 0;             // fp16 latent query half, K-major core matrices (<= 64 KB)
constexpr uint32_t OFF_QR = 65536;        // bf16 RoPE query half (<= 8 KB)
// The query of every (sequence, latent half) is prepared once per call by
// mla_prepare_q_kernel as an exact image of [OFF_Q, OFF_QR + 8 KB) and fetched
// per segment with one bulk copy.
constexpr uint32_t QIMG_BYTES = 65536 + 8192;
constexpr uint32_t OFF_C16 = 73728;       // 2 x fp16 latent tile (<= 32 KB each)
constexpr uint32_t C16_BYTES = 32768;
constexpr uint32_t OFF_STG = 139264;      // 2 x int8 TMA staging tile (<= 16 KB each)
constexpr uint32_t STG_BYTES = 16384;
constexpr uint32_t OFF_ROPE = 172032;     // 2 x bf16 RoPE key tile (<= 4 KB each)
constexpr uint32_t ROPE_BYTES = 4096;
constexpr uint32_t OFF_P = 180224;        // fp16 P, 128 x 64 (16 KB)
constexpr uint32_t OFF_X = 196608;        // fp32 partial scores from the peer, 128 x 64 (32 KB)
constexpr uint32_t OFF_BAR = 229376;
constexpr uint32_t kXBytes = 128 * 64 * 4;   // one tile of fp32 partial scores, all heads
constexpr uint32_t SMEM_BYTES = OFF_BAR + 256 + 1024;

// TMEM columns.
constexpr uint32_t TM_O = 0;      // fp32 O half: Dl/2 columns
constexpr uint32_t TM_S = 256;    // 2 x 64 latent-score buffers
constexpr uint32_t TM_R = 384;    // 2 x 64 RoPE-score buffers

// Barrier slots (8 bytes each) at OFF_BAR.
enum {
  B_TILE_FULL = 0, B_STG_EMPTY = 2, B_ROPE_EMPTY = 4, B_C16_FULL = 6, B_C16_EMPTY = 8,
  B_S_FULL = 10, B_S_EMPTY = 12, B_P_FULL = 14, B_PV_DONE = 15, B_Q_FULL = 16,
  B_XF = 17, B_XE = 18, B_DRAIN = 19, B_QK_DONE = 20, NBAR = 21
};
constexpr uint32_t OFF_TMEM_SLOT = OFF_BAR + 8 * NBAR;   // u32 TMEM base address
constexpr uint32_t OFF_ABORT = OFF_TMEM_SLOT + 4;         // u32 abort flag
constexpr uint32_t OFF_SCHED = OFF_TMEM_SLOT + 8;         // 4 x int64: b_first, pre_first, x0, x1

constexpr uint64_t kWaitNs = 1000000000ull;   // 1 s: normal waits last microseconds

struct MlaParams {
  CUtensorMap tm_ckv;    // int8 [B][T_max][Dl], box {min(Dl/2,128), 64, 1}
  CUtensorMap tm_rope;   // bf16 viewed as (8, T_max, Dr/8, B), box {8, 64, Dr/16, 1}
  const uint16_t* q;
  const float* q_scale;
  const float* kv_scale;
  const int32_t* lens;
  float* out;
  float* part_o;         // [slot][2][128][Dl/2]
  float2* part_ml;       // [slot][128]
  const uint8_t* q_img;  // [B][2][QIMG_BYTES] query images (fp16 latent codes, bf16 RoPE)
  int32_t* err;
  int B, H, Dl, Dr, T_max;
  int DH;                // Dl / 2
  int box_w;             // bytes per TMA box row of the latent (<= 128)
  int n_box;             // boxes per latent half
  int rope_chunks;       // 8-wide RoPE chunks per CTA (Dr / 16)
  int KR;                // RoPE contraction per CTA padded to a multiple of 16 (0 if Dr == 0)
  int num_clusters;
  float sm_log2;         // softmax_scale * log2(e)
};

// ----------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t a, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t a) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(a) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t a, uint32_t tx) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(tx) : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(a), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_cluster(uint32_t a, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      "selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok) : "r"(a), "r"(parity) : "memory");
  return ok != 0;
}
// Asynchronous remote store; its bytes complete_tx on the destination CTA's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t raddr, float a, float b, float c, float d, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
               ::"r"(raddr), "f"(a), "f"(b), "f"(c), "f"(d), "r"(rbar) : "memory");
}
// Bulk asynchronous copy global -> this CTA's shared memory, completing on an mbarrier.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ uint32_t mapa(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(bar) : "memory");
}
__device__ __forceinline__ void tma_4d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2, int c3,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar) : "memory");
}

// Shared-memory matrix descriptor, no swizzle: core matrices of 8 rows x 16 bytes.
// K-major operand: lbo = byte stride between core matrices along K, sbo = along M/N.
// MN-major operand: lbo = along K, sbo = along M/N as well (8-element MN groups).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::f16 with fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool ab_bf16, bool b_mn_major) {
  return (1u << 4) | ((ab_bf16 ? 1u : 0u) << 7) | ((ab_bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

#define FA3_TMEM_LD32(taddr, v)                                                                                   \
  asm volatile(                                                                                                   \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18," \
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                              \
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),          \
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),    \
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),  \
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])   \
      : "r"(taddr))

#define FA3_TMEM_ST32(taddr, v)                                                                                   \
  asm volatile(                                                                                                   \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17," \
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"                                             \
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),      \
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),           \
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),         \
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]))

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t x) {
  __half2 h = *reinterpret_cast<__half2*>(&x);
  return __half22float2(h);
}
// Four signed int8 codes -> two f16x2 (exact).
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  lo = __byte_perm(u, 0x64646464u, 0x4140);
  hi = __byte_perm(u, 0x64646464u, 0x4342);
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(lo) : "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %0, %1;" : "+r"(hi) : "r"(0x64806480u));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: gives up after kWaitNs nanoseconds of wall-clock time, or as
// soon as another role of this CTA has given up.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                         int32_t* err, bool cluster_scope = false) {
  if (cluster_scope ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (cluster_scope ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > kWaitNs) break;
  }
  *abort_flag = 1u;
  set_dev_err(err, FA3_DEVERR_TIMEOUT);
  return false;
}

// Softmax warps run tcgen05.ld/st (warp-collective): keep their control flow warp-uniform.
__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

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

template <int DH>
__global__ void __launch_bounds__(kThreads, 1)
mla_decode_kernel(const __grid_constant__ MlaParams p) {
  // Compile-time geometry of this CTA's latent half.
  constexpr int BOX_W = DH < 128 ? DH : 128;        // bytes per TMA box row (<= the 128-byte swizzle span)
  constexpr int N_BOX = DH / BOX_W;
  constexpr int CPB = BOX_W / 16;                   // 16-byte chunks per box row
  constexpr uint32_t SWZ_MASK = BOX_W == 128 ? 7u : BOX_W == 64 ? 3u : 1u;
  constexpr int LAT_CHUNKS = DH / 8;                // 8-wide fp16 chunks of the latent half
  constexpr int CONV_UNITS = kTok * (DH / 16) / kConvThreads;   // 16-byte int8 chunks per converter thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t peer = rank ^ 1u;
  const int cluster = blockIdx.x >> 1;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFF_ABORT);
  auto bar = [&](int i) { return sbase + OFF_BAR + 8u * (uint32_t)i; };

  // ---- set-up: barriers, TMEM, zero padding, schedule
  if (tid == 0) {
    mbar_init(bar(B_TILE_FULL), 1); mbar_init(bar(B_TILE_FULL + 1), 1);
    mbar_init(bar(B_STG_EMPTY), kConvThreads); mbar_init(bar(B_STG_EMPTY + 1), kConvThreads);
    mbar_init(bar(B_ROPE_EMPTY), 1); mbar_init(bar(B_ROPE_EMPTY + 1), 1);
    mbar_init(bar(B_C16_FULL), kConvThreads); mbar_init(bar(B_C16_FULL + 1), kConvThreads);
    mbar_init(bar(B_C16_EMPTY), 1); mbar_init(bar(B_C16_EMPTY + 1), 1);
    mbar_init(bar(B_S_FULL), 1); mbar_init(bar(B_S_FULL + 1), 1);
    mbar_init(bar(B_S_EMPTY), kRows); mbar_init(bar(B_S_EMPTY + 1), kRows);
    mbar_init(bar(B_P_FULL), kRows);
    mbar_init(bar(B_PV_DONE), 1);
    mbar_init(bar(B_Q_FULL), 1);
    mbar_init(bar(B_QK_DONE), 1);
    mbar_init(bar(B_XF), 1);          // armed with the expected bytes, filled by the peer's st.async
    mbar_init(bar(B_XE), kRows);
    mbar_init(bar(B_DRAIN), 1);
    *abort_flag = 0u;
    mbar_expect_tx(bar(B_XF), kXBytes);   // phase 0 of the partial-score exchange
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(sbase + OFF_TMEM_SLOT), "r"(512) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (warp >= kConvWarp0 && p.KR > 0) {
    // RoPE key chunks beyond this CTA's share stay zero (contraction padding).
    for (int s = 0; s < 2; ++s)
      for (uint32_t off = (uint32_t)p.rope_chunks * 1024u + (uint32_t)(tid - kConvWarp0 * 32) * 16u;
           off < (uint32_t)(p.KR / 8) * 1024u; off += kConvThreads * 16u)
        *reinterpret_cast<uint4*>(smem + OFF_ROPE + s * ROPE_BYTES + off) = make_uint4(0, 0, 0, 0);
  }
  if (warp == 0) {
    // Even split of all tiles over the clusters; find this cluster's first sequence.
    int64_t total = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      int t = (b0 + lane < p.B) ? seq_tiles(p, b0 + lane) : 0;
      if (lane == 0 && rank == 0 && cluster == 0) {
        for (int bb = b0; bb < min(b0 + 32, p.B); ++bb) {
          const int len = p.lens[bb];
          if (len < 0 || len > p.T_max) set_dev_err(p.err, FA3_DEVERR_LENS);
        }
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
  cluster_sync();   // peer barriers are initialised before any remote arrive

  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM_SLOT);
  const int64_t* sched = reinterpret_cast<const int64_t*>(smem + OFF_SCHED);
  SegWalk walk0{sched[2], sched[3], sched[1], (int)sched[0]};
  const uint32_t tile_tx = (uint32_t)(kTok * DH) + (uint32_t)(kTok * 16 * p.rope_chunks);

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      SegWalk w = walk0;
      int b, lo, hi, tb;
      uint32_t it = 0;
      bool ok = true;
      while (ok && w.next(p, b, lo, hi, tb)) {
        for (int tt = lo; tt < hi && ok; ++tt, ++it) {
          const uint32_t s = it & 1u, ph = (it >> 1) & 1u;
          ok = wait_bar(bar(B_STG_EMPTY + s), ph ^ 1u, abort_flag, p.err) &&
               wait_bar(bar(B_ROPE_EMPTY + s), ph ^ 1u, abort_flag, p.err);
          if (!ok) break;
          mbar_expect_tx(bar(B_TILE_FULL + s), tile_tx);
#pragma unroll
          for (int j = 0; j < N_BOX; ++j)
            tma_3d(sbase + OFF_STG + s * STG_BYTES + (uint32_t)(j * kTok * BOX_W), &p.tm_ckv,
                   (int)rank * DH + j * BOX_W, tt * kTok, b, bar(B_TILE_FULL + s));
          if (p.rope_chunks > 0)
            tma_4d(sbase + OFF_ROPE + s * ROPE_BYTES, &p.tm_rope, 0, tt * kTok, (int)rank * p.rope_chunks, b,
                   bar(B_TILE_FULL + s));
        }
      }
      // Drain: every issued copy must land before the CTA may exit.
      for (uint32_t k = (it >= 2 ? it - 2 : 0); k < it; ++k)
        wait_bar(bar(B_TILE_FULL + (k & 1u)), (k >> 1) & 1u, abort_flag, p.err);
    }
  } else if (warp >= kConvWarp0) {
    // ------------------------------------------------------ int8 -> fp16 converters
    const int ct = tid - kConvWarp0 * 32;
    SegWalk w = walk0;
    int b, lo, hi, tb;
    uint32_t it = 0;
    bool ok = true;
    while (ok && w.next(p, b, lo, hi, tb)) {
      for (int tt = lo; tt < hi && ok; ++tt, ++it) {
        const uint32_t s = it & 1u, ph = (it >> 1) & 1u;
        ok = wait_bar(bar(B_TILE_FULL + s), ph, abort_flag, p.err) &&
             wait_bar(bar(B_C16_EMPTY + s), ph ^ 1u, abort_flag, p.err);
        if (!ok) break;
        const uint8_t* stg = smem + OFF_STG + s * STG_BYTES;
        uint8_t* c16 = smem + OFF_C16 + s * C16_BYTES;
        // Unit u = (token n, 16-byte latent chunk cc); consecutive threads take
        // consecutive tokens, so both the swizzled reads and the core-matrix
        // writes are conflict-free.  All loads are issued before any convert.
        uint4 v[CONV_UNITS];
#pragma unroll
        for (int i = 0; i < CONV_UNITS; ++i) {
          const int u = ct + kConvThreads * i;
          const int n = u % kTok, cc = u / kTok;
          const int j = cc / CPB, c = cc % CPB;
          // TMA swizzle: the 16-byte chunk index is XORed with bits 7.. of the row address.
          const uint32_t row_addr = (uint32_t)(n * BOX_W);
          const uint32_t phys = ((uint32_t)c ^ ((row_addr >> 7) & SWZ_MASK)) * 16u;
          v[i] = *reinterpret_cast<const uint4*>(stg + j * kTok * BOX_W + row_addr + phys);
        }
#pragma unroll
        for (int i = 0; i < CONV_UNITS; ++i) {
          const int u = ct + kConvThreads * i;
          const int n = u % kTok, cc = u / kTok;
          uint4 o0, o1;
          i8x4_to_f16x4(v[i].x, o0.x, o0.y);
          i8x4_to_f16x4(v[i].y, o0.z, o0.w);
          i8x4_to_f16x4(v[i].z, o1.x, o1.y);
          i8x4_to_f16x4(v[i].w, o1.z, o1.w);
          const int kc = 2 * cc;             // 8-wide latent chunk of the first 8 values
          *reinterpret_cast<uint4*>(c16 + kc * 1024 + n * 16) = o0;
          *reinterpret_cast<uint4*>(c16 + (kc + 1) * 1024 + n * 16) = o1;
        }
        fence_proxy_async();
        mbar_arrive(bar(B_C16_FULL + s));
        mbar_arrive(bar(B_STG_EMPTY + s));
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_f16(128, kTok, false, false);
      const uint32_t id_rope = idesc_f16(128, kTok, true, false);
      const uint32_t id_pv = idesc_f16(128, DH, false, true);
      SegWalk w = walk0;
      int b, lo, hi, tb;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      auto issue_pv = [&](uint32_t j, bool first) -> bool {
        if (!wait_bar(bar(B_P_FULL), j & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t cs = j & 1u;
#pragma unroll
        for (int kk = 0; kk < kTok / 16; ++kk) {
          const uint64_t a = sdesc(sbase + OFF_P + kk * 4096, 2048, 128);
          // MN-major, no swizzle: LBO strides the K (token) core groups, SBO the N (latent) ones.
          const uint64_t bd = sdesc(sbase + OFF_C16 + cs * C16_BYTES + kk * 256, 128, 1024);
          mma_f16(tmem + TM_O, a, bd, id_pv, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(bar(B_PV_DONE));
        mma_commit(bar(B_C16_EMPTY + cs));
        return true;
      };
      while (ok && w.next(p, b, lo, hi, tb)) {
        // This segment's query: wait until the previous segment's Q.C^T is done
        // with the old one, then bulk-copy the prepared image.
        if (seg > 0) ok = wait_bar(bar(B_QK_DONE), (seg - 1) & 1u, abort_flag, p.err);
        if (!ok) break;
        {
          const uint8_t* img = p.q_img + ((size_t)b * 2 + rank) * QIMG_BYTES;
          const uint32_t lat_bytes = (uint32_t)(DH / 8) * 2048u, rope_bytes = (uint32_t)(p.KR / 8) * 2048u;
          mbar_expect_tx(bar(B_Q_FULL), lat_bytes + rope_bytes);
          bulk_g2s(sbase + OFF_Q, img, lat_bytes, bar(B_Q_FULL));
          if (rope_bytes) bulk_g2s(sbase + OFF_QR, img + 65536, rope_bytes, bar(B_Q_FULL));
        }
        ok = wait_bar(bar(B_Q_FULL), seg & 1u, abort_flag, p.err);
        ++seg;
        for (int tt = lo; tt < hi && ok; ++tt, ++it) {
          const uint32_t s = it & 1u, ph = (it >> 1) & 1u;
          ok = wait_bar(bar(B_TILE_FULL + s), ph, abort_flag, p.err) &&
               wait_bar(bar(B_C16_FULL + s), ph, abort_flag, p.err) &&
               wait_bar(bar(B_S_EMPTY + s), ph ^ 1u, abort_flag, p.err);
          if (!ok) break;
          tc_fence_after();
          for (int kk = 0; kk < DH / 16; ++kk) {
            const uint64_t a = sdesc(sbase + OFF_Q + kk * 4096, 2048, 128);
            const uint64_t bd = sdesc(sbase + OFF_C16 + s * C16_BYTES + kk * 2048, 1024, 128);
            mma_f16(tmem + TM_S + s * 64, a, bd, id_qk, kk > 0 ? 1u : 0u);
          }
          for (int kk = 0; kk < p.KR / 16; ++kk) {
            const uint64_t a = sdesc(sbase + OFF_QR + kk * 4096, 2048, 128);
            const uint64_t bd = sdesc(sbase + OFF_ROPE + s * ROPE_BYTES + kk * 2048, 1024, 128);
            mma_f16(tmem + TM_R + s * 64, a, bd, id_rope, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_S_FULL + s));
          mma_commit(bar(B_ROPE_EMPTY + s));
          if (tt == hi - 1) mma_commit(bar(B_QK_DONE));   // the query may be replaced
          // P.C of the previous tile of this segment overlaps the softmax of this one.
          if (tt > lo) ok = issue_pv(it - 1, tt - 1 == lo);
          if (ok && tt == hi - 1) ok = issue_pv(it, tt == lo);
        }
      }
      // Drain every MMA this thread issued before the CTA may release TMEM.
      mma_commit(bar(B_DRAIN));
      wait_bar(bar(B_DRAIN), 0, abort_flag, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int h = tid;                                   // head == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float kvs = p.kv_scale[0];
    const float c_rope = p.sm_log2;
    const uint32_t peer_x = mapa(sbase + OFF_X, peer);
    const uint32_t peer_xf = mapa(bar(B_XF), peer);
    const uint32_t peer_xe = mapa(bar(B_XE), peer);
    SegWalk w = walk0;
    int b, lo, hi, tb;
    uint32_t it = 0;
    bool ok = true;
    while (ok && w.next(p, b, lo, hi, tb)) {
      const float qs = h < p.H ? p.q_scale[h] : 0.f;
      const float c_lat = qs * kvs * p.sm_log2;
      const int len = p.lens[b];
      float m_ref = -CUDART_INF_F, l = 0.f;
      for (int tt = lo; tt < hi && ok; ++tt, ++it) {
        const uint32_t s = it & 1u, ph = (it >> 1) & 1u;
        const int nvalid = min(kTok, len - tt * kTok);
        ok = warp_all(wait_bar(bar(B_S_FULL + s), ph, abort_flag, p.err));
        if (!ok) break;
        tc_fence_after();
        float part[64];
        {
          uint32_t v[32], r[32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            FA3_TMEM_LD32(tmem + lane_base + TM_S + s * 64 + half * 32, v);
            if (p.KR > 0) {
              FA3_TMEM_LD32(tmem + lane_base + TM_R + s * 64 + half * 32, r);
            }
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float rr = p.KR > 0 ? __uint_as_float(r[j]) : 0.f;
              part[half * 32 + j] = fmaf(__uint_as_float(v[j]), c_lat, rr * c_rope);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(bar(B_S_EMPTY + s));

        // ---- swap partial scores with the peer CTA
        ok = warp_all(wait_bar(bar(B_XE), (it & 1u) ^ 1u, abort_flag, p.err, true));
        if (!ok) break;
#pragma unroll
        for (int j4 = 0; j4 < 16; ++j4)
          st_async_v4(peer_x + (uint32_t)((j4 * kRows + h) * 16), part[4 * j4], part[4 * j4 + 1], part[4 * j4 + 2],
                      part[4 * j4 + 3], peer_xf);
        ok = warp_all(wait_bar(bar(B_XF), it & 1u, abort_flag, p.err, true));
        if (!ok) break;
        float mt = -CUDART_INF_F;
#pragma unroll
        for (int j4 = 0; j4 < 16; ++j4) {
          const float4 o = *reinterpret_cast<const float4*>(smem + OFF_X + (j4 * kRows + h) * 16);
          const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * j4 + e;
            const float sc = part[j] + ov[e];
            part[j] = j < nvalid ? sc : -CUDART_INF_F;
            mt = fmaxf(mt, part[j]);
          }
        }
        // Re-arm for the next tile before telling the peer that its buffer is free.
        if (h == 0) mbar_expect_tx(bar(B_XF), kXBytes);
        mbar_arrive_remote(peer_xe);

        // ---- online softmax with a lazily moved reference maximum
        float alpha = 1.f;
        bool rescale = false;
        if (mt > m_ref + 8.f) {
          alpha = (m_ref == -CUDART_INF_F) ? 0.f : exp2f(m_ref - mt);
          rescale = tt > lo;
          m_ref = mt;
        }
        uint32_t pk[32];
        float psum = 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          pk[j] = pack_f16x2(exp2f(part[2 * j] - m_ref), exp2f(part[2 * j + 1] - m_ref));
          const float2 f = unpack_f16x2(pk[j]);
          psum += f.x + f.y;
        }
        l = l * alpha + psum;
        if (tt > lo) {
          // P is single-buffered and O must hold P.C of the previous tile.
          ok = warp_all(wait_bar(bar(B_PV_DONE), (it - 1) & 1u, abort_flag, p.err));
          if (!ok) break;
          tc_fence_after();
          // The rescale is decided per head (lane) but tcgen05.ld/st are warp-wide:
          // the whole warp takes part, lanes that keep their reference scale by 1.
          if (__any_sync(0xffffffffu, rescale)) {
            if (!rescale) alpha = 1.f;
            for (int c0 = 0; c0 < DH; c0 += 32) {
              uint32_t v[32];
              FA3_TMEM_LD32(tmem + lane_base + TM_O + c0, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
              FA3_TMEM_ST32(tmem + lane_base + TM_O + c0, v);
            }
            tmem_wait_st();
          }
        }
#pragma unroll
        for (int kc = 0; kc < 8; ++kc)
          *reinterpret_cast<uint4*>(smem + OFF_P + kc * 2048 + (h >> 3) * 128 + (h & 7) * 16) =
              make_uint4(pk[4 * kc], pk[4 * kc + 1], pk[4 * kc + 2], pk[4 * kc + 3]);
        fence_proxy_async();
        tc_fence_before();
        mbar_arrive(bar(B_P_FULL));
      }
      if (!ok) break;
      // ---- segment done: wait for the last P.C, then write the output (or a partial)
      ok = warp_all(wait_bar(bar(B_PV_DONE), (it - 1) & 1u, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      const bool full = (lo == 0 && hi == tb);
      const float inv = (full && l > 0.f) ? kvs / l : 0.f;
      const int slot = b + cluster;
#pragma unroll 1
      for (int c0 = 0; c0 < DH; c0 += 32) {
        uint32_t v[32];
        FA3_TMEM_LD32(tmem + lane_base + TM_O + c0, v);
        tmem_wait_ld();
        if (h < p.H) {
          float* dst = full ? p.out + ((int64_t)b * p.H + h) * p.Dl + rank * DH + c0
                            : p.part_o + (((int64_t)slot * 2 + rank) * kRows + h) * DH + c0;
          const float f = full ? inv : 1.f;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + j) =
                make_float4(__uint_as_float(v[j]) * f, __uint_as_float(v[j + 1]) * f,
                            __uint_as_float(v[j + 2]) * f, __uint_as_float(v[j + 3]) * f);
        }
      }
      if (!full && rank == 0 && h < p.H) p.part_ml[(int64_t)slot * kRows + h] = make_float2(m_ref, l);
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
// codes as fp16) and lays it out, with the RoPE query, as the shared-memory
// image the decode kernel copies: K-major core matrices of 8 heads x 8 values.
// One thread per 8 values of one (sequence, head).
__global__ void __launch_bounds__(256) mla_prepare_q_kernel(const MlaParams p) {
  const int chunks_lat = p.Dl / 8, chunks_rope = p.Dr / 8;
  const int per_row = chunks_lat + chunks_rope;
  const int64_t n = (int64_t)p.B * kRows * per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % per_row);
    const int64_t bh = i / per_row;
    const int h = (int)(bh % kRows), b = (int)(bh / kRows);
    uint4 o = make_uint4(0, 0, 0, 0);
    int r, k;
    uint32_t region;
    if (c < chunks_lat) {
      r = c / (p.DH / 8);
      k = c % (p.DH / 8);
      region = 0;
      if (h < p.H) {
        const uint4 v = *reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.H + h) * (p.Dl + p.Dr) + 8 * c);
        const float qs = p.q_scale[h], rqs = rcp_approx(qs);
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        uint32_t r4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          r4[e] = pack_f16x2((float)quant_code_fast(bf16_to_float(wv[e] & 0xffffu), qs, rqs),
                             (float)quant_code_fast(bf16_to_float(wv[e] >> 16), qs, rqs));
        o = make_uint4(r4[0], r4[1], r4[2], r4[3]);
      }
    } else {
      const int cr = c - chunks_lat;
      r = cr / p.rope_chunks;
      k = cr % p.rope_chunks;
      region = 65536;
      if (h < p.H) o = *reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.H + h) * (p.Dl + p.Dr) + 8 * c);
    }
    uint8_t* img = const_cast<uint8_t*>(p.q_img) + ((size_t)b * 2 + r) * QIMG_BYTES + region;
    *reinterpret_cast<uint4*>(img + k * 2048 + (h >> 3) * 128 + (h & 7) * 16) = o;
    // RoPE contraction padding (KR > Dr/2): the extra 8-wide chunk is zero.
    if (c >= chunks_lat && k == p.rope_chunks - 1 && p.KR / 8 > p.rope_chunks)
      *reinterpret_cast<uint4*>(img + (k + 1) * 2048 + (h >> 3) * 128 + (h & 7) * 16) = make_uint4(0, 0, 0, 0);
  }
}

// Merges the split segments of each sequence; writes zero rows for empty sequences.
__global__ void mla_combine_kernel(const MlaParams p, int64_t total_tiles_unused) {
  const int h = blockIdx.x, b = blockIdx.y;
  __shared__ int64_t s_info[3];
  if (threadIdx.x == 0) {
    int64_t total = 0, pre = 0;
    for (int bb = 0; bb < p.B; ++bb) {
      const int t = seq_tiles(p, bb);
      if (bb < b) pre += t;
      total += t;
    }
    s_info[0] = total; s_info[1] = pre; s_info[2] = seq_tiles(p, b);
  }
  __syncthreads();
  const int64_t total = s_info[0], pre = s_info[1], tb = s_info[2];
  const int C = p.num_clusters;
  if (h >= p.H) return;
  float* dst = p.out + ((int64_t)b * p.H + h) * p.Dl;
  if (tb == 0) {
    for (int c = threadIdx.x; c < p.Dl; c += blockDim.x) dst[c] = 0.f;
    return;
  }
  // owner cluster of tile position x: the largest c with floor(total*c/C) <= x
  auto owner = [&](int64_t x) {
    int lo = 0, hi = C - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (total * mid / C <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  const int c0 = owner(pre), c1 = owner(pre + tb - 1);
  if (c0 == c1) return;   // one cluster held the whole sequence and wrote it already
  // Clusters between the two owners hold a segment of this sequence unless their
  // range is empty (fewer tiles than clusters); empty ones wrote nothing.
  auto holds = [&](int c) { return total * c / C < total * (c + 1) / C; };
  float M = -CUDART_INF_F;
  for (int c = c0; c <= c1; ++c)
    if (holds(c)) M = fmaxf(M, p.part_ml[(int64_t)(b + c) * kRows + h].x);
  float L = 0.f;
  for (int c = c0; c <= c1; ++c) {
    if (!holds(c)) continue;
    const float2 ml = p.part_ml[(int64_t)(b + c) * kRows + h];
    L += ml.y * exp2f(ml.x - M);
  }
  const float kvs = p.kv_scale[0];
  for (int d = threadIdx.x; d < p.Dl; d += blockDim.x) {
    const int r = d / p.DH, dd = d - r * p.DH;
    float O = 0.f;
    for (int c = c0; c <= c1; ++c) {
      if (!holds(c)) continue;
      const int64_t slot = b + c;
      O += p.part_o[((slot * 2 + r) * kRows + h) * p.DH + dd] * exp2f(p.part_ml[slot * kRows + h].x - M);
    }
    dst[d] = L > 0.f ? kvs * (O / L) : 0.f;
  }
}

template <int DH>
cudaError_t launch_mla(cudaLaunchConfig_t cfg, const MlaParams& prm) {
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<DH>, prm);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// Number of 2-CTA clusters that can be resident at once (cached per device).
int max_clusters() {
  static int cached[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(mla_decode_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
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
  if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel<256>, &cfg) != cudaSuccess || n <= 0) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

bool mla_shape_ok(int H, int Dl, int Dr) {
  const bool dl_ok = Dl == 64 || Dl == 128 || Dl == 256 || Dl == 512;
  return H >= 1 && H <= kRows && dl_ok && Dr >= 0 && Dr <= 64 && Dr % 16 == 0;
}

}  // namespace
}  // namespace fa3

using namespace fa3;

FA3_API size_t fa3_mla_workspace_size(int B, int H, int Dl, int T_max) {
  if (B <= 0 || H <= 0 || Dl <= 0 || T_max <= 0) return 0;
  int C = 0;
  if (check_device(nullptr) == FA3_OK) C = max_clusters();
  if (C <= 0) C = 128;
  const size_t slots = (size_t)B + (size_t)C;
  return slots * 2 * kRows * (size_t)(Dl / 2) * sizeof(float) + slots * kRows * sizeof(float2) + 256 +
         (size_t)B * 2 * QIMG_BYTES;
}

FA3_API int fa3_decode_attn_mla(const uint16_t* q, const int8_t* ckv, const uint16_t* krope, const float* q_scale,
                                const float* kv_scale, const int32_t* lens, float* out, int B, int H, int Dl,
                                int Dr, int T_max, float softmax_scale, void* workspace, size_t workspace_bytes,
                                int32_t* dev_err, void* stream) {
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
  const size_t need = fa3_mla_workspace_size(B, H, Dl, T_max);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return FA3_EWORKSPACE;
  PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
  if (!encode) return FA3_ECUDA;

  MlaParams prm;
  memset(&prm, 0, sizeof(prm));
  prm.DH = Dl / 2;
  prm.box_w = prm.DH < 128 ? prm.DH : 128;
  prm.n_box = prm.DH / prm.box_w;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)Dl, (cuuint64_t)T_max, (cuuint64_t)B};
    const cuuint64_t strides[2] = {(cuuint64_t)Dl, (cuuint64_t)Dl * T_max};
    const cuuint32_t box[3] = {(cuuint32_t)prm.box_w, (cuuint32_t)kTok, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUtensorMapSwizzle sw = prm.box_w == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : prm.box_w == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                    : CU_TENSOR_MAP_SWIZZLE_32B;
    if (encode(&prm.tm_ckv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<int8_t*>(ckv), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FA3_ECUDA;
  }
  if (Dr > 0) {
    prm.rope_chunks = Dr / 16;
    prm.KR = ((Dr / 2 + 15) / 16) * 16;
    const cuuint64_t dims[4] = {8, (cuuint64_t)T_max, (cuuint64_t)(Dr / 8), (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)Dr * 2, 16, (cuuint64_t)Dr * 2 * T_max};
    const cuuint32_t box[4] = {8, (cuuint32_t)kTok, (cuuint32_t)prm.rope_chunks, 1};
    const cuuint32_t es[4] = {1, 1, 1, 1};
    if (encode(&prm.tm_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<uint16_t*>(krope), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return FA3_ECUDA;
  }
  prm.q = q; prm.q_scale = q_scale; prm.kv_scale = kv_scale; prm.lens = lens; prm.out = out;
  const size_t slots = (size_t)B + (size_t)C;
  prm.part_o = static_cast<float*>(workspace);
  prm.part_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) + slots * 2 * kRows * prm.DH * sizeof(float));
  {
    size_t off = slots * 2 * kRows * prm.DH * sizeof(float) + slots * kRows * sizeof(float2);
    off = (off + 255) & ~size_t(255);
    prm.q_img = static_cast<const uint8_t*>(workspace) + off;
  }
  prm.err = dev_err;
  prm.B = B; prm.H = H; prm.Dl = Dl; prm.Dr = Dr; prm.T_max = T_max;
  prm.num_clusters = C;
  prm.sm_log2 = softmax_scale * 1.4426950408889634f;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  {
    const int64_t n = (int64_t)B * kRows * ((Dl + Dr) / 8);
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    mla_prepare_q_kernel<<<(unsigned)blocks, 256, 0, s>>>(prm);
    if (cudaGetLastError() != cudaSuccess) return FA3_ECUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * C, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2; attr.val.clusterDim.y = 1; attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  cudaError_t le = cudaErrorInvalidValue;
  switch (prm.DH) {
    case 32: le = launch_mla<32>(cfg, prm); break;
    case 64: le = launch_mla<64>(cfg, prm); break;
    case 128: le = launch_mla<128>(cfg, prm); break;
    case 256: le = launch_mla<256>(cfg, prm); break;
  }
  if (le != cudaSuccess) return FA3_ECUDA;
  mla_combine_kernel<<<dim3(kRows, B), 256, 0, s>>>(prm, 0);
  return cuda_status(cudaGetLastError());
}
