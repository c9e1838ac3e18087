// Sustained tcgen05.mma rate (a peak probe for the rooflines): every CTA (one per SM) issues ITERS back-to-back
// M=128, K=16 kind::f16 MMAs of width N into one accumulator, A and B from shared
// memory (or A from TMEM), then commits and waits (bounded).  Reports cycles per MMA.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
__host__ __device__ constexpr uint32_t idesc(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
template <int N, bool ATMEM>
__global__ void __launch_bounds__(128, 1) k(long long* out, int iters, int* err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t mbar;
  __shared__ uint32_t tslot;
  const uint32_t sb = (uint32_t)__cvta_generic_to_shared(sm);
  for (int i = threadIdx.x; i < 98304 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(sm)[i] = 0x3c003c00u;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"((uint32_t)__cvta_generic_to_shared(&mbar)));
    asm volatile("fence.mbarrier_init.release.cluster;");
  }
  if (threadIdx.x < 32) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"((uint32_t)__cvta_generic_to_shared(&tslot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("fence.proxy.async.shared::cta;");
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tm = tslot;
  if (threadIdx.x == 0) {
    const uint32_t id = idesc(128, N);
    const uint32_t mb = (uint32_t)__cvta_generic_to_shared(&mbar);
    // B: N rows x K=16, K-major (8-row groups 128 B apart, the two 8-wide K groups N*16 B apart)
    const uint64_t b0 = sdesc(sb, N * 16, 128);
    // A: 128 rows x 16, K-major in shared memory at +64 KB (K groups 2048 B apart)
    const uint64_t a0 = sdesc(sb + 65536, 2048, 128);
    const uint32_t acol = 256;     // A in TMEM: columns 256 .. 263
    long long t0 = clock64();
#pragma unroll 8
    for (int i = 0; i < iters; ++i) {
      const uint64_t bd = b0 + (uint64_t)((i & 3) * 2);      // walk a little through B (stays inside)
      if (ATMEM)
        asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
                     ::"r"(tm), "r"(tm + acol), "l"(bd), "r"(id), "r"((uint32_t)(i > 0)));
      else
        asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                     ::"r"(tm), "l"(a0), "l"(bd), "r"(id), "r"((uint32_t)(i > 0)));
    }
    long long t1 = clock64();
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mb));
    uint32_t ok = 0;
    for (int spin = 0; spin < 20000000 && !ok; ++spin)
      asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n" : "=r"(ok) : "r"(mb), "r"(0));
    long long t2 = clock64();
    if (!ok) atomicOr(err, 1);
    out[blockIdx.x * 2] = t1 - t0;
    out[blockIdx.x * 2 + 1] = t2 - t0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (threadIdx.x < 32) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tm));
}
template <int N, bool AT>
void run(int sms, long long* d, int* err, int iters) {
  cudaFuncSetAttribute(k<N, AT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 98304);
  k<N, AT><<<sms, 128, 98304>>>(d, iters, err);
  cudaError_t e = cudaDeviceSynchronize();
  static long long h[2 * 1024];
  cudaMemcpy(h, d, sizeof(long long) * 2 * sms, cudaMemcpyDeviceToHost);
  double iss = 0, tot = 0;
  for (int i = 0; i < sms; ++i) { iss += h[2 * i]; tot += h[2 * i + 1]; }
  iss /= sms; tot /= sms;
  const double ideal = 128.0 * N * 16 * 2 / 8192.0;
  printf("N=%3d A=%s (%s): issue %.1f, complete %.1f cycles per MMA; ideal %.1f -> %.0f%% of the pipe\n", N,
         AT ? "tmem" : "smem", cudaGetErrorString(e), iss / iters, tot / iters, ideal, 100.0 * ideal / (tot / iters));
}
int main() {
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  long long* d; int* err; cudaMalloc(&d, 2 * 1024 * sizeof(long long)); cudaMalloc(&err, 4); cudaMemset(err, 0, 4);
  const int iters = 2048;
  run<64, false>(sms, d, err, iters); run<64, true>(sms, d, err, iters);
  run<128, false>(sms, d, err, iters); run<128, true>(sms, d, err, iters);
  run<256, false>(sms, d, err, iters); run<256, true>(sms, d, err, iters);
  int herr; cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost); printf("err %d sms %d\n", herr, sms);
  return 0;
}
