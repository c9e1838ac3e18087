// Per-head quantization parameters and quantize-on-append.
//
// msModelSlim "FA3量化" page, 原理 / 算法流程 step 4: scale[h] = max(|min|,|max|)/127.
// MindIE "FA3 quantization" / "Attention Quantization", Overview: input_scale turns
// the attention activations into INT8 codes that the decode kernels read.
#include "fa3_common.cuh"

#include <cuda_bf16.h>

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

// Vector path: each thread converts 8 consecutive values of one row (16 B in, 8 B out).
// Rows are (b, t, h) triples; groups of 8 values never straddle a row because D % 8 == 0.
__global__ void __launch_bounds__(256) quantize_append_vec_kernel(
    const uint4* __restrict__ kv, const float* __restrict__ scale, int8_t* __restrict__ cache,
    const int32_t* __restrict__ pos, int B, int T_new, int H, int D, int T_max,
    const uint4* __restrict__ rope_src, uint16_t* __restrict__ rope_cache, int Dr, int32_t* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t groups_per_row = D / 8;
  const int64_t n_groups = (int64_t)B * T_new * H * groups_per_row;
  const int64_t rope_groups_per_row = Dr / 8;
  const int64_t n_rope = rope_cache ? (int64_t)B * T_new * rope_groups_per_row : 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t gi = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; gi < n_groups + n_rope; gi += stride) {
    if (gi < n_groups) {
      int64_t row = gi / groups_per_row;            // (b * T_new + t) * H + h
      int g = (int)(gi - row * groups_per_row);
      int h = (int)(row % H);
      int64_t bt = row / H;
      int t = (int)(bt % T_new);
      int b = (int)(bt / T_new);
      int p = pos[b];
      if (p < 0 || p > T_max - T_new) {
        if (t == 0 && h == 0 && g == 0) set_dev_err(err, FA3_DEVERR_POS);
        continue;
      }
      uint4 v = kv[gi];
      const float s = scale[h];
      const float rs = rcp_approx(s);
      uint32_t w[4] = {v.x, v.y, v.z, v.w};
      uint32_t packed[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        uint32_t acc = 0;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          uint32_t word = w[2 * i + j];
          const int c0 = quant_code_fast(bf16_to_float(word & 0xffffu), s, rs);
          const int c1 = quant_code_fast(bf16_to_float(word >> 16), s, rs);
          acc |= ((uint32_t)(c0 & 0xff) | ((uint32_t)(c1 & 0xff) << 8)) << (16 * j);
        }
        packed[i] = acc;
      }
      int64_t dst = ((((int64_t)b * T_max + p + t) * H + h) * D) + (int64_t)g * 8;
      *reinterpret_cast<uint2*>(cache + dst) = make_uint2(packed[0], packed[1]);
    } else {
      int64_t ri = gi - n_groups;
      int64_t row = ri / rope_groups_per_row;         // b * T_new + t
      int g = (int)(ri - row * rope_groups_per_row);
      int t = (int)(row % T_new);
      int b = (int)(row / T_new);
      int p = pos[b];
      if (p < 0 || p > T_max - T_new) continue;
      int64_t dst = (((int64_t)b * T_max + p + t) * Dr) + (int64_t)g * 8;
      *reinterpret_cast<uint4*>(rope_cache + dst) = rope_src[ri];
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

FA3_API int fa3_quantize_append(const uint16_t* kv, const float* scale, int8_t* cache, const int32_t* pos,
                                int B, int T_new, int H, int D, int T_max, const uint16_t* rope_src,
                                uint16_t* rope_cache, int Dr, int32_t* dev_err, void* stream) {
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
  const bool vec = (D % 8 == 0) && aligned16(kv) && (((uintptr_t)cache & 7u) == 0) &&
                   (!rope_cache || ((Dr % 8 == 0) && aligned16(rope_src) && aligned16(rope_cache)));
  const int64_t work = (int64_t)B * T_new * (H * (int64_t)D + Dr) / (vec ? 8 : 1);
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaError_t e;
  if (vec) {
    e = launch_pdl(quantize_append_vec_kernel, dim3((unsigned)blocks), dim3(256), 0, s,
                   reinterpret_cast<const uint4*>(kv), scale, cache, pos, B, T_new, H, D, T_max,
                   reinterpret_cast<const uint4*>(rope_src), rope_cache, Dr, dev_err);
  } else {
    e = launch_pdl(quantize_append_scalar_kernel, dim3((unsigned)blocks), dim3(256), 0, s, kv, scale, cache, pos, B,
                   T_new, H, D, T_max, rope_src, rope_cache, Dr, dev_err);
  }
  return cuda_status(e);
}
