// Prefill-phase GQA attention with INT8 q, k and v (tcgen05, sm_103a).
//
// MindIE "Attention Quantization", Overview, and MindIE Turbo "Attention量化":
// q, k and v are quantized to 8 bits with per-head scales (msModelSlim "FA3量化"
// 原理 / 算法流程 step 4) and the attention operator consumes the codes; at long
// sequence lengths these activations dominate memory (msModelSlim "FA3量化",
// 简介).  The prefill phase attends the q_len new rows of a sequence, the last
// q_len tokens of its kv_len-token context, causally:
//
//   s[i, h, t] = (q8[i, h] . k8[t, g]) * q_scale[h] * k_scale[g] * softmax_scale,
//                t <= pos(i) = kv_len - q_len + i,   g = h / (Hq / Hkv)
//   out[i, h]  = bf16( v_scale[g] * sum_t softmax(s[i, h, :])_t * v8[t, g] )
//
// The contraction is dense (2 * 2 * D FLOP per (row, key) pair), so the kernel
// is built around the tensor pipe:
//   * one CTA per (block of 2 x 128 rows, KV head g, sequence b): two query tiles
//     A and B of 128 rows, each P = 128 / G query positions x the G query heads of
//     the group, so that every converted K/V tile feeds 256 rows (row r of a tile
//     = TMEM lane r: position r / G, head r % G);
//   * int8 codes are exact in fp16 and a 128-term sum of their products stays
//     below 2^24, so kind::f16 MMAs with fp32 accumulation give the exact integer
//     score (sm_103a has no integer tcgen05 kind);
//   * warp 0 issues the MMAs; warps 1-3 load 128-token int8 K and V tiles into
//     registers one tile ahead and write them as fp16 core matrices into one of
//     two shared-memory stages (K-major for Q.K^T, MN-major for P.V); warps 4-7
//     (tile A) and 8-11 (tile B) own one row each for the online softmax;
//   * TMEM: O_A, O_B, S_A, S_B, 128 columns each; while one tile's softmax runs
//     the tensor pipe works on the other tile's S or P.V;
//   * the softmax writes P (fp16, unnormalised, relative to a lazily moved row
//     maximum) over its own S in TMEM, the A operand of P.V; it sums the same
//     fp16 weights for the row's normaliser (so the output is a weighted mean of
//     V whatever the rounding of P), and rescales O in TMEM only when a row's
//     maximum grows by more than 8 (log2 units);
//   * blocks run longest first (the last positions see the most keys).
// Every wait is bounded; on time-out the kernel sets FA3_DEVERR_TIMEOUT, drains
// its MMAs, frees its TMEM and returns.
#include "fa3_common.cuh"
#include "fa3_tc.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

namespace fa3 {
namespace {

constexpr int kD = 128;            // head dim
constexpr int kKeys = 128;         // keys per tile
constexpr int kRowsP = 128;        // rows (TMEM lanes) per query tile
constexpr int kThreadsP = 384;     // warp 0: MMA, warps 1-3: converters, 4-7: softmax A, 8-11: softmax B
constexpr int kConvP = 96;
constexpr uint32_t TMP_O = 0, TMP_S = 256;                 // O_x [128x, +128), S_x [256 + 128x, +128)
constexpr uint32_t KV_TILE = kKeys * kD * 2;               // 32 KB of fp16
constexpr uint32_t Q_TILE = kRowsP * kD * 2;               // 32 KB of fp16
constexpr uint32_t OFFP_Q = 0;                             // 2 x fp16 query rows, K-major
constexpr uint32_t OFFP_K = OFFP_Q + 2 * Q_TILE;           // 2 stages
constexpr uint32_t OFFP_V = OFFP_K + 2 * KV_TILE;          // 2 stages
constexpr uint32_t OFFP_BAR = OFFP_V + 2 * KV_TILE;
enum {
  PB_K_FULL = 0, PB_K_EMPTY = 2, PB_V_FULL = 4, PB_V_EMPTY = 6,
  PB_S_FULL = 8,                   // [2]: tile x's scores of the current key tile
  PB_P_FULL = 10,                  // [2]: tile x's P written over its S
  PB_PV_DONE = 12,                 // [2]: P_x.V done (O_x holds it; S_x free)
  PB_Q_READY = 14, PB_DRAIN, PB_N
};
constexpr uint32_t OFFP_TSLOT = OFFP_BAR + 8 * PB_N;
constexpr uint32_t OFFP_ABORT = OFFP_TSLOT + 4;
constexpr uint32_t SMEM_PREFILL = OFFP_BAR + 256 + 1024;   // + alignment slack
static_assert(OFFP_ABORT + 4 <= OFFP_BAR + 256, "barrier area");
static_assert(SMEM_PREFILL <= 232448, "shared memory");

struct PrefillParams {
  const int8_t* q;         // [B][S][Hq][128]
  const int8_t* k;         // [B][T][Hkv][128]
  const int8_t* v;
  const float* q_scale;    // [Hq]
  const float* k_scale;    // [Hkv]
  const float* v_scale;
  const int32_t* q_lens;   // [B]
  const int32_t* kv_lens;  // [B]
  uint16_t* out;           // bf16 [B][S][Hq][128]
  int32_t* err;
  int B, S, T, Hq, Hkv, G, P;
  float sm_log2;           // softmax_scale * log2(e)
};

__global__ void __launch_bounds__(kThreadsP, 1) gqa_prefill_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rb = (int)gridDim.x - 1 - (int)blockIdx.x;      // longest blocks first
  const int g = blockIdx.y, b = blockIdx.z;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + OFFP_ABORT);
  auto bar = [&](int i) { return sbase + OFFP_BAR + 8u * (uint32_t)i; };
  pdl_wait();
  pdl_launch_dependents();

  const int nq = p.q_lens[b], nkv = p.kv_lens[b];
  if (nq < 0 || nq > p.S || nkv < nq || nkv > p.T) {
    if (rb == 0 && g == 0 && tid == 0) set_dev_err(p.err, FA3_DEVERR_LENS);
    return;
  }
  const int i0 = rb * 2 * p.P;                             // first position of tile A; tile B follows
  if (i0 >= nq) return;                                    // no row of this block is a new row
  const int prefix = nkv - nq;
  const int n_keys = prefix + min(nq, i0 + 2 * p.P);       // keys up to the block's last position
  const int nt = (n_keys + kKeys - 1) / kKeys;

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(PB_K_FULL + s), kConvP);
      mbar_init(bar(PB_K_EMPTY + s), 1);
      mbar_init(bar(PB_V_FULL + s), kConvP);
      mbar_init(bar(PB_V_EMPTY + s), 1);
      mbar_init(bar(PB_S_FULL + s), 1);
      mbar_init(bar(PB_P_FULL + s), 4);
      mbar_init(bar(PB_PV_DONE + s), 1);
    }
    mbar_init(bar(PB_Q_READY), 8);
    mbar_init(bar(PB_DRAIN), 1);
    *abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(sbase + OFFP_TSLOT), "r"(512) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFFP_TSLOT);

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_qk = idesc_f16(kRowsP, kKeys, false, false);
      const uint32_t id_pv = idesc_f16(kRowsP, kD, false, true);
      bool ok = wait_bar(bar(PB_Q_READY), 0, abort_flag, p.err);
      // S_x = Q_x . K_j^T: Q_x the K-major A operand in shared memory (8-row core
      // groups 128 B apart, 8-wide d groups 2048 B apart), K the K-major B operand.
      // S_x holds the P of key tile j - 1 until P_x.V(j - 1) is done.
      auto issue_qk = [&](int j, int x) -> bool {
        const int s = j & 1;
        if (!wait_bar(bar(PB_K_FULL + s), (uint32_t)(j >> 1) & 1u, abort_flag, p.err)) return false;
        if (j > 0 && !wait_bar(bar(PB_PV_DONE + x), (uint32_t)(j - 1) & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t a = sdesc(sbase + OFFP_Q + x * Q_TILE + kk * 4096, 2048, 128);
          const uint64_t bd = sdesc(sbase + OFFP_K + s * KV_TILE + kk * 4096, 2048, 128);
          mma_f16(tmem + TMP_S + x * 128, a, bd, id_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(PB_S_FULL + x));
        if (x == 1) mma_commit(bar(PB_K_EMPTY + s));         // both tiles are done with K_j
        return true;
      };
      // O_x += P_x . V_j: P_x (fp16, written over S_x: column k holds keys 2k, 2k + 1)
      // is the A operand in TMEM, V the MN-major B operand (token groups 128 B apart,
      // d groups 2048 B apart).
      auto issue_pv = [&](int j, int x) -> bool {
        const int s = j & 1;
        if (!wait_bar(bar(PB_P_FULL + x), (uint32_t)j & 1u, abort_flag, p.err)) return false;
        if (x == 0 && !wait_bar(bar(PB_V_FULL + s), (uint32_t)(j >> 1) & 1u, abort_flag, p.err)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk) {
          const uint64_t bd = sdesc(sbase + OFFP_V + s * KV_TILE + kk * 256, 128, 2048);
          mma_f16_ts(tmem + TMP_O + x * 128, tmem + TMP_S + x * 128 + kk * 8, bd, id_pv,
                     (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(PB_PV_DONE + x));
        if (x == 1) mma_commit(bar(PB_V_EMPTY + s));          // both tiles are done with V_j
        return true;
      };
      ok = ok && issue_qk(0, 0) && issue_qk(0, 1);
      for (int j = 0; j < nt && ok; ++j) {
        ok = issue_pv(j, 0) && issue_pv(j, 1);
        if (ok && j + 1 < nt) ok = issue_qk(j + 1, 0) && issue_qk(j + 1, 1);
      }
      // Drain: every MMA issued has completed before TMEM is freed.
      mma_commit(bar(PB_DRAIN));
      wait_bar(bar(PB_DRAIN), 0, abort_flag, p.err);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------ int8 -> fp16 converters
    // A tile is 2 x 128 rows x 8 chunks of 16 bytes (K, then V).  Each group of 32
    // consecutive units is 16 tokens x 2 chunks, lane l taking token l % 16 and
    // chunk l / 16: a warp loads 16 full 32-byte sectors and its fp16 stores hit
    // every bank once per 128 bytes.  fp16 element (token n, d) lands at
    // (d / 8) * 2048 + n * 16 + (d % 8) * 2.  K(j) may be written once both
    // Q.K^T of tile j - 2 are done, V(j) once both P.V of tile j - 2 are.
    constexpr int kUnits = 2 * kKeys * (kD / 16);                 // 2048
    constexpr int kPer = (kUnits + kConvP - 1) / kConvP;           // 22
    const int ct = tid - 32;
    const int64_t row_stride = (int64_t)p.Hkv * kD;
    const int8_t* kb = p.k + (int64_t)b * p.T * row_stride + (int64_t)g * kD;
    const int8_t* vb = p.v + (int64_t)b * p.T * row_stride + (int64_t)g * kD;
    auto unit = [&](int i, int& kv, int& n, int& cc) {
      const int u = ct + kConvP * i;
      const int grp = u >> 5, l = u & 31;                          // grp < 64 for u < kUnits
      kv = grp >> 5;
      n = (grp & 7) * 16 + (l & 15);
      cc = ((grp >> 3) & 3) * 2 + (l >> 4);
      return u < kUnits;
    };
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1;
      const uint32_t par = ((uint32_t)(j >> 1) & 1u) ^ 1u;
      uint4 w[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        int kv, n, cc;
        const bool in = unit(i, kv, n, cc);
        const int t = j * kKeys + n;
        w[i] = make_uint4(0u, 0u, 0u, 0u);
        if (in && t < n_keys) w[i] = __ldg(reinterpret_cast<const uint4*>((kv ? vb : kb) + t * row_stride) + cc);
      }
      bool ok = true;
#pragma unroll
      for (int half = 0; half < 2 && ok; ++half) {
        if (!wait_bar(bar((half ? PB_V_EMPTY : PB_K_EMPTY) + s), par, abort_flag, p.err)) { ok = false; break; }
        uint8_t* dst = smem + (half ? OFFP_V : OFFP_K) + s * KV_TILE;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
          int kv, n, cc;
          if (unit(i, kv, n, cc) && kv == half) {
            uint4 o0, o1;
            i8x4_to_f16x4(w[i].x, o0.x, o0.y);
            i8x4_to_f16x4(w[i].y, o0.z, o0.w);
            i8x4_to_f16x4(w[i].z, o1.x, o1.y);
            i8x4_to_f16x4(w[i].w, o1.z, o1.w);
            *reinterpret_cast<uint4*>(dst + (2 * cc) * 2048 + n * 16) = o0;
            *reinterpret_cast<uint4*>(dst + (2 * cc + 1) * 2048 + n * 16) = o1;
          }
        }
        fence_proxy_async();
        mbar_arrive(bar((half ? PB_V_FULL : PB_K_FULL) + s));
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int x = (warp - 4) >> 2;                          // query tile: 0 = A, 1 = B
    const int r = ((warp - 4) & 3) * 32 + lane;             // row == TMEM lane
    const uint32_t lane_base = (uint32_t)(((warp - 4) & 3) * 32) << 16;
    const int i = i0 + x * p.P + r / p.G, h = g * p.G + r % p.G;
    const bool active = i < nq;
    const int pos = active ? prefix + i : -1;               // last key this row sees
    // an inactive row masks every key (its scale stays finite so that -inf * c is -inf)
    const float c = active ? p.q_scale[h] * p.k_scale[g] * p.sm_log2 : 1.f;
    const int pos_min = prefix + i0 + x * p.P;              // the tile's first position
    const bool ragged = i0 + (x + 1) * p.P > nq;            // the tile has inactive rows
    const uint32_t o_col = tmem + lane_base + TMP_O + x * 128;
    const uint32_t scol = tmem + lane_base + TMP_S + x * 128;
    auto warp_arrive = [&](int which) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(which));
    };
    // The row's query codes as fp16 into tile x's K-major A operand (chunk of 8 d at
    // (d / 8) * 2048 + row * 16).
    {
      const int8_t* qrow = p.q + (((int64_t)b * p.S + (active ? i : 0)) * p.Hq + h) * kD;
      uint8_t* qdst = smem + OFFP_Q + x * Q_TILE + r * 16;
#pragma unroll
      for (int c16 = 0; c16 < 8; ++c16) {
        uint4 xq = make_uint4(0u, 0u, 0u, 0u);
        if (active) xq = *reinterpret_cast<const uint4*>(qrow + 16 * c16);
        uint4 o0, o1;
        i8x4_to_f16x4(xq.x, o0.x, o0.y);
        i8x4_to_f16x4(xq.y, o0.z, o0.w);
        i8x4_to_f16x4(xq.z, o1.x, o1.y);
        i8x4_to_f16x4(xq.w, o1.z, o1.w);
        *reinterpret_cast<uint4*>(qdst + (2 * c16) * 2048) = o0;
        *reinterpret_cast<uint4*>(qdst + (2 * c16 + 1) * 2048) = o1;
      }
      fence_proxy_async();
      warp_arrive(PB_Q_READY);
    }
    float m_run = -CUDART_INF_F, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nt && ok; ++j) {
      if (!warp_all(wait_bar(bar(PB_S_FULL + x), (uint32_t)j & 1u, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int t0 = j * kKeys;
      // keys of this tile beyond some row's position (the diagonal) or inactive rows
      const bool masked = ragged || t0 + kKeys - 1 > pos_min;
      // pass 1: the tile's row maximum of the raw integer scores, then scaled (c > 0)
      float mx = -CUDART_INF_F;
#pragma unroll 1
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t v[32];
        FA3_TMEM_LD32(scol + c4 * 32, v);
        tmem_wait_ld();
        if (masked) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            mx = fmaxf(mx, t0 + c4 * 32 + e <= pos ? __uint_as_float(v[e]) : -CUDART_INF_F);
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) mx = max3(mx, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
        }
      }
      mx *= c;
      const float m_new = fmaxf(m_run, mx);
      // Lazy rescale: the reference maximum moves only when the row maximum grew by
      // more than 8; then O (holding P.V up to key tile j - 1) is scaled in place.
      const bool grow = m_new != -CUDART_INF_F && (m_run == -CUDART_INF_F || m_new > m_run + 8.f);
      if (__any_sync(0xffffffffu, grow && m_run != -CUDART_INF_F)) {
        if (!warp_all(wait_bar(bar(PB_PV_DONE + x), (uint32_t)(j - 1) & 1u, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = (grow && m_run != -CUDART_INF_F) ? ex2_approx(m_run - m_new) : 1.f;
#pragma unroll 1
        for (int c4 = 0; c4 < 4; ++c4) {
          uint32_t v[32];
          FA3_TMEM_LD32(o_col + c4 * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * f);
          FA3_TMEM_ST32(o_col + c4 * 32, v);
        }
      }
      if (grow) {
        l_run = m_run == -CUDART_INF_F ? 0.f : l_run * ex2_approx(m_run - m_new);
        m_run = m_new;
      }
      const float mc = m_run == -CUDART_INF_F ? 0.f : m_run;
      // pass 2: P = exp2(s c - m) as fp16 pairs over the S columns already read
      // (keys 32 c4 .. 32 c4 + 31 go to columns 16 c4 .. 16 c4 + 15); the row sum
      // takes the same fp16 weights, so the output is a weighted mean of V.
#pragma unroll 1
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t v[32];
        FA3_TMEM_LD32(scol + c4 * 32, v);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int t = t0 + c4 * 32 + e;
          float p0 = ex2_approx(fmaf(__uint_as_float(v[e]), c, -mc));
          float p1 = ex2_approx(fmaf(__uint_as_float(v[e + 1]), c, -mc));
          if (masked) {
            p0 = t <= pos ? p0 : 0.f;
            p1 = t + 1 <= pos ? p1 : 0.f;
          }
          pk[e / 2] = pack_f16x2(p0, p1);
          const float2 pr = __half22float2(*reinterpret_cast<const __half2*>(&pk[e / 2]));
          l_run += pr.x + pr.y;
        }
        FA3_TMEM_ST16(scol + c4 * 16, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(PB_P_FULL + x);
    }
    // epilogue: out = v_scale * O / l
    if (ok && warp_all(wait_bar(bar(PB_PV_DONE + x), (uint32_t)(nt - 1) & 1u, abort_flag, p.err))) {
      tc_fence_after();
      const float inv = (active && l_run > 0.f) ? p.v_scale[g] / l_run : 0.f;
      uint16_t* orow = p.out + (((int64_t)b * p.S + (active ? i : 0)) * p.Hq + h) * kD;
#pragma unroll 1
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t v[32];
        FA3_TMEM_LD32(o_col + c4 * 32, v);
        tmem_wait_ld();
        if (active) {
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const __nv_bfloat162 bb =
                __floats2bfloat162_rn(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
            w[e / 2] = *reinterpret_cast<const uint32_t*>(&bb);
          }
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            *reinterpret_cast<uint4*>(orow + c4 * 32 + q4 * 8) =
                make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
  }
}

}  // namespace
}  // namespace fa3

using namespace fa3;

FA3_API int fa3_prefill_attn_gqa(const int8_t* q, const int8_t* k, const int8_t* v, const float* q_scale,
                                 const float* k_scale, const float* v_scale, const int32_t* q_lens,
                                 const int32_t* kv_lens, uint16_t* out, int B, int S, int T, int Hq, int Hkv, int D,
                                 float softmax_scale, int32_t* dev_err, void* stream) {
  if (!q || !k || !v || !q_scale || !k_scale || !v_scale || !q_lens || !kv_lens || !out) return FA3_EINVAL;
  if (B <= 0 || S <= 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return FA3_EINVAL;
  if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return FA3_EINVAL;
  const int G = Hq / Hkv;
  if (D != kD || kRowsP % G != 0 || B > 65535 || Hkv > 65535) return FA3_ERANGE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return FA3_ERANGE;
  int sms = 0;
  const int st = check_device(&sms);
  if (st != FA3_OK) return st;
  PrefillParams prm;
  prm.q = q; prm.k = k; prm.v = v; prm.q_scale = q_scale; prm.k_scale = k_scale; prm.v_scale = v_scale;
  prm.q_lens = q_lens; prm.kv_lens = kv_lens; prm.out = out; prm.err = dev_err;
  prm.B = B; prm.S = S; prm.T = T; prm.Hq = Hq; prm.Hkv = Hkv; prm.G = G; prm.P = kRowsP / G;
  prm.sm_log2 = softmax_scale * 1.4426950408889634f;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaFuncSetAttribute(gqa_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_PREFILL) !=
      cudaSuccess)
    return FA3_ECUDA;
  const dim3 grid((unsigned)((S + 2 * prm.P - 1) / (2 * prm.P)), (unsigned)Hkv, (unsigned)B);
  timing_begin(s);
  const cudaError_t le = launch_pdl(gqa_prefill_kernel, grid, dim3(kThreadsP), SMEM_PREFILL, s, prm);
  timing_end(s);
  return le == cudaSuccess ? FA3_OK : FA3_ECUDA;
}
