// Per-head quantization parameters and quantize-on-append.
//
// msModelSlim "FA3量化" page, 原理 / 算法流程 step 4: scale[h] = max(|min|,|max|)/127.
// MindIE "FA3 quantization" / "Attention Quantization", Overview: input_scale turns
// the attention activations into INT8 codes that the decode kernels read.
#include "fa3_common.cuh"

#include <cuda_bf16.h>

#include <algorithm>

namespace fa3 {

namespace {
cudaEvent_t g_timing_start = nullptr, g_timing_stop = nullptr;
}  // namespace

void timing_begin(cudaStream_t s) {
  if (g_timing_start && g_timing_stop) cudaEventRecord(g_timing_start, s);
}
void timing_end(cudaStream_t s) {
  if (g_timing_start && g_timing_stop) cudaEventRecord(g_timing_stop, s);
}

int check_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA3_ECUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FA3_ECUDA;
  if (major != 10 || minor != 3) return FA3_EDEVICE;
  if (num_sms) *num_sms = sms;
  return FA3_OK;
}

// One thread per head.
__global__ void qparams_kernel(const float* __restrict__ mn, const float* __restrict__ mx,
                               float* __restrict__ scale, int H) {
  pdl_wait();
  pdl_launch_dependents();
  int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h < H) scale[h] = __fdiv_rn(fmaxf(fabsf(mn[h]), fabsf(mx[h])), 127.0f);
}

// Step 3 over R ranges at once: min_io[h] = min(min_io[h], mins[r][h]) and max
// likewise for every r, in IEEE totalOrder (-0.0 below +0.0), so the result does
// not depend on how the calibration batches were split or ordered.
__device__ __forceinline__ bool range_less(float a, float b) {
  return a < b || (a == b && signbit(a) && !signbit(b));
}
__global__ void range_merge_kernel(const float* __restrict__ mins, const float* __restrict__ maxs, int R, int H,
                                   float* __restrict__ min_io, float* __restrict__ max_io) {
  pdl_wait();
  pdl_launch_dependents();
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= H) return;
  float lo = min_io[h], hi = max_io[h];
  for (int r = 0; r < R; ++r) {
    const float a = mins[(int64_t)r * H + h], b = maxs[(int64_t)r * H + h];
    if (range_less(a, lo)) lo = a;
    if (range_less(hi, b)) hi = b;
  }
  min_io[h] = lo;
  max_io[h] = hi;
}

// Paged cache: position x of sequence b is row block_table[b][x / page_size] *
// page_size + x % page_size of the pool.
struct PageMap {
  const int32_t* block_table;   // [B][max_pages]
  int max_pages, num_pages, page_size;
  DivU32 div_ps;                // / page_size
  DivU32 div_row;               // / (H * D / 8): 16-byte groups per token row
  DivU32 div_rope;              // / (Dr / 8)
};

// Vector path.  The T_new new rows of sequence b are contiguous in the source and,
// from cache row pos[b] on, contiguous in the cache as well, so the append of one
// sequence is a stream conversion: 16-byte source group i (8 bf16 values of head
// (i / (D/8)) mod H) becomes 8-byte cache group i, and the RoPE rows are a 16-byte
// copy.  blockIdx.y walks the sequences, so pos[b] is one uniform load per block.
// With G = 2 a thread converts two neighbouring groups and stores them as one
// 16-byte word (the host picks G = 2 when every such word is 16-byte aligned; then
// the groups of a token row are even in number and a pair never spans two rows).
// PAGED: the cache is a page pool; each group's token row is looked up in the
// block table (a pair shares one lookup).
template <int G, bool PAGED>
__global__ void __launch_bounds__(256) quantize_append_vec_kernel(
    const uint4* __restrict__ kv, const float* __restrict__ scale, int8_t* __restrict__ cache,
    const int32_t* __restrict__ pos, int B, int T_new, int H, int D, int T_max,
    const uint4* __restrict__ rope_src, uint16_t* __restrict__ rope_cache, int Dr, int32_t* err,
    DivU32 div_g, DivU32 div_h, PageMap pm) {
  pdl_wait();
  pdl_launch_dependents();
  const uint32_t gpr = (uint32_t)(D / 8);
  const uint32_t nl = (uint32_t)T_new * (uint32_t)H * gpr;                // latent groups per sequence
  const uint32_t nr = rope_cache ? (uint32_t)T_new * (uint32_t)(Dr / 8) : 0u;
  const uint32_t tid = blockIdx.x * blockDim.x + threadIdx.x, nthreads = gridDim.x * blockDim.x;
  const float s_one = scale[0];                                             // the only scale when H == 1
  const float rs_one = rcp_approx(s_one);
  const bool ex_one = exact_scale(s_one);
  for (int b = blockIdx.y; b < B; b += gridDim.y) {
    const int p = pos[b];
    if (p < 0 || p > T_max - T_new) {
      if (blockIdx.x == 0 && threadIdx.x == 0) set_dev_err(err, FA3_DEVERR_POS);
      continue;
    }
    const int64_t row0 = (int64_t)b * T_max + p;                         // first cache row written
    const uint4* src = kv + (uint64_t)b * nl;
    uint2* dst = reinterpret_cast<uint2*>(cache + (PAGED ? 0 : row0 * H * D));
    // Pool row of position x of this sequence, or -1 for an entry outside the pool.
    auto page_row = [&](uint32_t x) -> int64_t {
      const uint32_t pi = divu32(x, pm.div_ps);
      const int pg = pm.block_table[(int64_t)b * pm.max_pages + pi];
      if (pg < 0 || pg >= pm.num_pages) {
        set_dev_err(err, FA3_DEVERR_PAGE);
        return -1;
      }
      return (int64_t)pg * pm.page_size + (x - pi * (uint32_t)pm.page_size);
    };
    for (uint32_t i = tid * G; i < nl; i += nthreads * G) {
      int64_t di = i;                                                       // uint2 index of group i in dst
      if (PAGED) {
        const uint32_t R = (uint32_t)H * gpr;
        const uint32_t t = divu32(i, pm.div_row);
        const int64_t row = page_row((uint32_t)p + t);
        if (row < 0) continue;
        di = row * R + (i - t * R);
      }
      uint4 v[G];
#pragma unroll
      for (int u = 0; u < G; ++u)
        if (u == 0 || i + u < nl) v[u] = src[i + u];
      float s = s_one, rs = rs_one, s1 = s_one, rs1 = rs_one;
      bool ex = ex_one, ex1 = ex_one;
      if (H > 1) {
        const uint32_t r = divu32(i, div_g);                                // (token, head) row of group i
        const uint32_t h = r - divu32(r, div_h) * (uint32_t)H;
        s = scale[h];
        rs = rcp_approx(s);
        ex = exact_scale(s);
        s1 = s, rs1 = rs, ex1 = ex;
        if (G == 2 && i - r * gpr + 1 == gpr) {                             // group i + 1 starts the next head
          s1 = scale[h + 1 == (uint32_t)H ? 0 : h + 1];
          rs1 = rcp_approx(s1);
          ex1 = exact_scale(s1);
        }
      }
      const uint2 c0 = quant_group8(v[0], s, rs, ex);
      if (G == 2 && i + 1 < nl) {
        const uint2 c1 = quant_group8(v[G - 1], s1, rs1, ex1);
        *reinterpret_cast<uint4*>(dst + di) = make_uint4(c0.x, c0.y, c1.x, c1.y);
      } else {
        dst[di] = c0;
      }
    }
    const uint4* rsrc = rope_src + (uint64_t)b * nr;
    uint4* rdst = reinterpret_cast<uint4*>(rope_cache + (PAGED ? 0 : row0 * Dr));
    for (uint32_t i = tid; i < nr; i += nthreads) {
      int64_t di = i;
      if (PAGED) {
        const uint32_t gr = (uint32_t)(Dr / 8);
        const uint32_t t = divu32(i, pm.div_rope);
        const int64_t row = page_row((uint32_t)p + t);
        if (row < 0) continue;
        di = row * gr + (i - t * gr);
      }
      rdst[di] = rsrc[i];
    }
  }
}

// Scalar path for rows that are not 16-byte aligned.
__global__ void __launch_bounds__(256) quantize_append_scalar_kernel(
    const uint16_t* __restrict__ kv, const float* __restrict__ scale, int8_t* __restrict__ cache,
    const int32_t* __restrict__ pos, int B, int T_new, int H, int D, int T_max,
    const uint16_t* __restrict__ rope_src, uint16_t* __restrict__ rope_cache, int Dr, int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t n = (int64_t)B * T_new * H * D;
  const int64_t n_rope = rope_cache ? (int64_t)B * T_new * Dr : 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n + n_rope; i += stride) {
    if (i < n) {
      int d = (int)(i % D);
      int64_t row = i / D;
      int h = (int)(row % H);
      int64_t bt = row / H;
      int t = (int)(bt % T_new);
      int b = (int)(bt / T_new);
      int p = pos[b];
      if (p < 0 || p > T_max - T_new) {
        if (t == 0 && h == 0 && d == 0) set_dev_err(err, FA3_DEVERR_POS);
        continue;
      }
      int c = quant_code(bf16_to_float(kv[i]), scale[h]);
      cache[((((int64_t)b * T_max + p + t) * H + h) * D) + d] = (int8_t)c;
    } else {
      int64_t ri = i - n;
      int d = (int)(ri % Dr);
      int64_t row = ri / Dr;
      int t = (int)(row % T_new);
      int b = (int)(row / T_new);
      int p = pos[b];
      if (p < 0 || p > T_max - T_new) continue;
      rope_cache[(((int64_t)b * T_max + p + t) * Dr) + d] = rope_src[ri];
    }
  }
}

}  // namespace fa3

using namespace fa3;

FA3_API const char* fa3_status_string(int status) {
  switch (status) {
    case FA3_OK: return "FA3_OK";
    case FA3_EINVAL: return "FA3_EINVAL: null pointer, non-positive size or bad option";
    case FA3_ERANGE: return "FA3_ERANGE: size or alignment not supported by the kernels";
    case FA3_ECUDA: return "FA3_ECUDA: CUDA runtime error while enqueuing";
    case FA3_EWORKSPACE: return "FA3_EWORKSPACE: workspace missing or too small";
    case FA3_EDEVICE: return "FA3_EDEVICE: current device is not sm_103 (GB300 class)";
    default: return "FA3: unknown status";
  }
}

FA3_API int fa3_version(void) { return 100; }

FA3_API int fa3_set_kernel_timing(void* start_event, void* stop_event) {
  if ((start_event == nullptr) != (stop_event == nullptr)) return FA3_EINVAL;
  g_timing_start = static_cast<cudaEvent_t>(start_event);
  g_timing_stop = static_cast<cudaEvent_t>(stop_event);
  return FA3_OK;
}

FA3_API int fa3_qparams(const float* min_v, const float* max_v, float* scale, int H, void* stream) {
  if (!min_v || !max_v || !scale || H <= 0) return FA3_EINVAL;
  int st = check_device(nullptr);
  if (st != FA3_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_pdl(qparams_kernel, dim3((H + 127) / 128), dim3(128), 0, s, min_v, max_v, scale, H));
}

FA3_API int fa3_range_merge(const float* mins, const float* maxs, int R, int H, float* min_io, float* max_io,
                            void* stream) {
  if (!mins || !maxs || !min_io || !max_io) return FA3_EINVAL;
  if (R <= 0 || H <= 0) return FA3_EINVAL;
  int sms = 0;
  const int st = check_device(&sms);
  if (st != FA3_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_pdl(range_merge_kernel, dim3((H + 127) / 128), dim3(128), 0, s, mins, maxs, R, H,
                                min_io, max_io));
}

namespace {
// Both layouts: pm == nullptr is the contiguous [B][T_max] cache; otherwise the
// cache (and the RoPE cache) are page pools addressed through *pm.
int quantize_append(const uint16_t* kv, const float* scale, int8_t* cache, const int32_t* pos, int B, int T_new,
                    int H, int D, int T_max, const uint16_t* rope_src, uint16_t* rope_cache, int Dr,
                    int32_t* dev_err, void* stream, const PageMap* pm) {
  if (!kv || !scale || !cache || !pos) return FA3_EINVAL;
  if (B <= 0 || T_new <= 0 || H <= 0 || D <= 0 || T_max <= 0) return FA3_EINVAL;
  if (T_new > T_max) return FA3_EINVAL;
  if ((rope_src == nullptr) != (rope_cache == nullptr)) return FA3_EINVAL;
  if (rope_cache && Dr <= 0) return FA3_EINVAL;
  if (!rope_cache) Dr = 0;
  int sms = 0;
  int st = check_device(&sms);
  if (st != FA3_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t per_seq_groups = (int64_t)T_new * ((int64_t)H * (D / 8) + Dr / 8);
  const bool vec = (D % 8 == 0) && aligned16(kv) && (((uintptr_t)cache & 7u) == 0) &&
                   (!rope_cache || ((Dr % 8 == 0) && aligned16(rope_src) && aligned16(rope_cache))) &&
                   per_seq_groups < ((int64_t)1 << 31);
  if (pm && !vec) return FA3_ERANGE;                   // the paged path has the vector kernel only
  const bool pairs = vec && aligned16(cache) && ((int64_t)H * D) % 16 == 0;   // 16-byte stores of two groups
  using VecKernel = decltype(&quantize_append_vec_kernel<1, false>);
  const VecKernel vk = pm ? (pairs ? quantize_append_vec_kernel<2, true> : quantize_append_vec_kernel<1, true>)
                          : (pairs ? quantize_append_vec_kernel<2, false> : quantize_append_vec_kernel<1, false>);
  // Grid-stride loops; blocks for a few waves of the SMs.
  static int resident[5] = {0, 0, 0, 0, 0};            // scalar, then the four vector kernels
  const int kind = vec ? 1 + (pairs ? 1 : 0) + (pm ? 2 : 0) : 0;
  if (resident[kind] == 0) {
    int r = 0;
    const cudaError_t oe = vec ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, vk, 256, 0)
                               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&r, quantize_append_scalar_kernel, 256, 0);
    if (oe != cudaSuccess) return cuda_status(oe);
    resident[kind] = r > 0 ? r : 1;
  }
  const int64_t cap = (int64_t)sms * resident[kind];
  cudaError_t e;
  if (vec) {
    const int G = pairs ? 2 : 1;
    const int64_t gy = std::min<int64_t>(B, 65535);
    const int64_t items = std::max<int64_t>((int64_t)T_new * H * (D / 8) / G, (int64_t)T_new * (Dr / 8));
    const int64_t gx = std::max<int64_t>(1, std::min<int64_t>((items + 255) / 256, 4 * ((cap + gy - 1) / gy)));
    const DivU32 dg = make_divu32((uint32_t)(D / 8)), dh = make_divu32((uint32_t)H);
    PageMap map = {};
    if (pm) map = *pm;
    e = launch_pdl(vk, dim3((unsigned)gx, (unsigned)gy), dim3(256), 0, s, reinterpret_cast<const uint4*>(kv), scale,
                   cache, pos, B, T_new, H, D, T_max, reinterpret_cast<const uint4*>(rope_src), rope_cache, Dr,
                   dev_err, dg, dh, map);
  } else {
    const int64_t work = (int64_t)B * T_new * (H * (int64_t)D + Dr);
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, cap));
    e = launch_pdl(quantize_append_scalar_kernel, dim3((unsigned)blocks), dim3(256), 0, s, kv, scale, cache, pos, B,
                   T_new, H, D, T_max, rope_src, rope_cache, Dr, dev_err);
  }
  return cuda_status(e);
}
}  // namespace

FA3_API int fa3_quantize_append(const uint16_t* kv, const float* scale, int8_t* cache, const int32_t* pos,
                                int B, int T_new, int H, int D, int T_max, const uint16_t* rope_src,
                                uint16_t* rope_cache, int Dr, int32_t* dev_err, void* stream) {
  return quantize_append(kv, scale, cache, pos, B, T_new, H, D, T_max, rope_src, rope_cache, Dr, dev_err, stream,
                         nullptr);
}

FA3_API int fa3_quantize_append_paged(const uint16_t* kv, const float* scale, int8_t* cache,
                                      const int32_t* block_table, const int32_t* pos, int B, int T_new, int H, int D,
                                      int num_pages, int page_size, int max_pages, const uint16_t* rope_src,
                                      uint16_t* rope_cache, int Dr, int32_t* dev_err, void* stream) {
  if (!block_table) return FA3_EINVAL;
  if (num_pages <= 0 || page_size <= 0 || max_pages <= 0) return FA3_EINVAL;
  if ((int64_t)max_pages * page_size >= ((int64_t)1 << 31)) return FA3_ERANGE;
  PageMap pm = {};
  pm.block_table = block_table;
  pm.max_pages = max_pages;
  pm.num_pages = num_pages;
  pm.page_size = page_size;
  pm.div_ps = make_divu32((uint32_t)page_size);
  pm.div_row = make_divu32((uint32_t)std::max(1, H * (D / 8)));
  pm.div_rope = make_divu32((uint32_t)std::max(1, Dr / 8));
  return quantize_append(kv, scale, cache, pos, B, T_new, H, D, max_pages * page_size, rope_src, rope_cache, Dr,
                         dev_err, stream, &pm);
}

// ---------------------------------------------------------------------------
// Per-channel parameters -- MindIE Turbo "Attention量化", 表1 / 表2: q/k/v_scale
// and q/k/v_offset of shape [head_num, head_dim].
//
// Symmetric: scale = max(|min|, |max|) / 127 (msModelSlim FA3量化 step 4 per
// channel), offset 0.  Asymmetric: the range widened to contain 0,
// [lo, hi] = [min(min, 0), max(max, 0)], maps onto the codes -128 .. 127:
//   scale = (hi - lo) / 255,  offset = round_half_even(-lo / scale) - 128
// (float32 IEEE subtraction and divisions; scale 0 gives offset 0).  Codes:
//   symmetric  q = clamp(round_half_even(x / scale), -127, 127)
//   asymmetric q = clamp(round_half_even(x / scale) + offset, -128, 127)
// ---------------------------------------------------------------------------
namespace fa3 {
namespace {

__global__ void qparams_channel_kernel(const float* __restrict__ mn, const float* __restrict__ mx, int n,
                                       int asym, float* __restrict__ scale, float* __restrict__ offset) {
  pdl_wait();
  pdl_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  if (!asym) {
    scale[i] = __fdiv_rn(fmaxf(fabsf(mn[i]), fabsf(mx[i])), 127.0f);
    offset[i] = 0.f;
    return;
  }
  const float lo = fminf(mn[i], 0.f), hi = fmaxf(mx[i], 0.f);
  const float s = __fdiv_rn(__fsub_rn(hi, lo), 255.0f);
  scale[i] = s;
  offset[i] = s == 0.f ? 0.f : rintf(__fdiv_rn(-lo, s)) - 128.f;
}

__device__ __forceinline__ int channel_code(float x, float s, float o, bool asym) {
  float r = s == 0.f ? 0.f : __fdiv_rn(x, s);
  if (!asym) return __float2int_rn(fminf(fmaxf(r, -127.f), 127.f));
  r = fminf(fmaxf(r, -1e9f), 1e9f);
  return max(-128, min(127, __float2int_rn(r) + (int)o));
}

// One thread per 8 consecutive values (16 bytes of bf16) of the new rows; the
// channel parameters of those 8 values are read as two float4 pairs.
__global__ void quantize_append_channel_kernel(const uint16_t* __restrict__ kv, const float* __restrict__ scale,
                                               const float* __restrict__ offset, int asym,
                                               int8_t* __restrict__ cache, const int32_t* __restrict__ pos,
                                               int B, int T_new, int HD, int T_max, int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t groups_row = HD / 8, groups_seq = (int64_t)T_new * groups_row;
  const int64_t total = (int64_t)B * groups_seq;
  for (int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gi < total;
       gi += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(gi / groups_seq);
    const int64_t rem = gi - (int64_t)b * groups_seq;
    const int t = (int)(rem / groups_row);
    const int c8 = (int)(rem - (int64_t)t * groups_row) * 8;     // first of the 8 values in the row
    const int p0 = pos[b];
    if (p0 < 0 || p0 + T_new > T_max) {
      if (rem == 0) set_dev_err(err, FA3_DEVERR_POS);
      continue;
    }
    const uint4 v = *reinterpret_cast<const uint4*>(kv + gi * 8);
    const float4 s0 = *reinterpret_cast<const float4*>(scale + c8);
    const float4 s1 = *reinterpret_cast<const float4*>(scale + c8 + 4);
    float4 o0 = make_float4(0.f, 0.f, 0.f, 0.f), o1 = o0;
    if (asym) {
      o0 = *reinterpret_cast<const float4*>(offset + c8);
      o1 = *reinterpret_cast<const float4*>(offset + c8 + 4);
    }
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const float oo[8] = {o0.x, o0.y, o0.z, o0.w, o1.x, o1.y, o1.z, o1.w};
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x = bf16_to_float((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
      const int q = channel_code(x, ss[e], oo[e], asym != 0);
      packed[e >> 2] |= ((uint32_t)(q & 0xFF)) << (8 * (e & 3));
    }
    int8_t* dst = cache + (((int64_t)b * T_max + p0 + t) * HD + c8);
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  }
}

}  // namespace
}  // namespace fa3

using namespace fa3;

FA3_API int fa3_qparams_channel(const float* min_v, const float* max_v, int n, int asymmetric, float* scale,
                                float* offset, void* stream) {
  if (!min_v || !max_v || !scale || !offset || n <= 0) return FA3_EINVAL;
  int sms = 0;
  const int st = check_device(&sms);
  if (st != FA3_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_pdl(qparams_channel_kernel, dim3((n + 127) / 128), dim3(128), 0, s, min_v, max_v, n,
                                asymmetric ? 1 : 0, scale, offset));
}

FA3_API int fa3_quantize_append_channel(const uint16_t* kv, const float* scale, const float* offset,
                                        int asymmetric, int8_t* cache, const int32_t* pos, int B, int T_new, int H,
                                        int D, int T_max, int32_t* dev_err, void* stream) {
  if (!kv || !scale || !cache || !pos || (asymmetric && !offset)) return FA3_EINVAL;
  if (B <= 0 || T_new <= 0 || H <= 0 || D <= 0 || T_max <= 0 || T_new > T_max) return FA3_EINVAL;
  if (D % 8 != 0 || !aligned16(kv) || !aligned16(scale) || (asymmetric && !aligned16(offset)) ||
      (reinterpret_cast<uintptr_t>(cache) & 7u) != 0)
    return FA3_ERANGE;
  if ((int64_t)H * D >= ((int64_t)1 << 31)) return FA3_ERANGE;
  int sms = 0;
  const int st = check_device(&sms);
  if (st != FA3_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t total = (int64_t)B * T_new * H * D / 8;
  const int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)sms * 8);
  return cuda_status(launch_pdl(quantize_append_channel_kernel, dim3(blocks), dim3(256), 0, s, kv, scale, offset,
                                asymmetric ? 1 : 0, cache, pos, B, T_new, H * D, T_max, dev_err));
}
