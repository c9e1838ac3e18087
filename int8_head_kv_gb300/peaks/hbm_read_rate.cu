// HBM read-only bandwidth: every thread streams 16-byte loads (evict-first) over a
// buffer much larger than L2 and folds them into one word, so nothing is written
// but one word per thread.  Reports GB/s (best of several timed passes, CUDA events).
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
__global__ void __launch_bounds__(512) rd(const uint4* __restrict__ p, size_t n16, uint32_t* sink) {
  uint32_t acc = 0;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    const uint4 a = __ldcs(p + i), b = __ldcs(p + i + stride), c = __ldcs(p + i + 2 * stride),
                d = __ldcs(p + i + 3 * stride);
    acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^ d.z ^ d.w;
  }
  for (; i < n16; i += stride) { const uint4 a = __ldcs(p + i); acc ^= a.x ^ a.y ^ a.z ^ a.w; }
  if (acc == 0x12345678u) sink[threadIdx.x] = acc;     // keeps the loads alive; practically never stores
}
int main() {
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const size_t bytes = (size_t)4 << 30;                 // 4 GiB
  uint4* p; uint32_t* sink;
  if (cudaMalloc(&p, bytes) != cudaSuccess || cudaMalloc(&sink, 4096) != cudaSuccess) { printf("alloc failed\n"); return 1; }
  cudaMemset(p, 1, bytes);
  cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
  float best = 1e30f;
  for (int rep = 0; rep < 8; ++rep) {
    cudaEventRecord(e0);
    rd<<<sms * 4, 512>>>(p, bytes / 16, sink);
    cudaEventRecord(e1);
    cudaEventSynchronize(e1);
    float ms = 0; cudaEventElapsedTime(&ms, e0, e1);
    if (rep > 0 && ms < best) best = ms;
  }
  printf("{\"probe\": \"hbm_read\", \"bytes\": %zu, \"best_ms\": %.4f, \"GB/s\": %.1f, \"status\": \"%s\"}\n", bytes, best,
         bytes / (best * 1e-3) / 1e9, cudaGetErrorString(cudaGetLastError()));
  return 0;
}
