// Sustained DSMEM exchange rate: every 2-CTA cluster swaps ROUNDS rounds of 32 KB
// per direction through double-buffered slots (the pattern of a pairwise
// partial-score exchange), 256 threads per CTA each sending 8 x 16 B by st.async.
// All waits bounded.  Reports bytes per clock per direction per SM.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
__device__ __forceinline__ uint32_t su(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ bool try_wait(uint32_t a, uint32_t ph) {
  uint32_t ok;
  asm volatile("{.reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; selp.u32 %0,1,0,p;}"
               : "=r"(ok) : "r"(a), "r"(ph) : "memory");
  return ok;
}
__device__ __forceinline__ void csync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ bool wait(uint32_t a, uint32_t ph, int* err) {
  for (uint32_t k = 0; k < (1u << 22); ++k) if (try_wait(a, ph)) return true;
  atomicOr(err, 1);
  return false;
}
constexpr int kT = 256, kSlot = 32768;
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kT, 1) probe(int rounds, long long* out, int* err) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t* slot = sm;                                   // 2 x 32 KB receive slots
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + 2 * kSlot);
  uint64_t* fre = full + 2;
  uint32_t rank; asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const uint32_t peer = rank ^ 1;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(su(full + s)) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(su(fre + s)) : "memory");
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads(); csync();
  uint32_t rslot, rfull, rfree;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rslot) : "r"(su(slot)), "r"(peer));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rfull) : "r"(su(full)), "r"(peer));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rfree) : "r"(su(fre)), "r"(peer));
  // arm both receive slots
  if (tid == 0)
    for (int s = 0; s < 2; ++s)
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(su(full + s)), "r"(kSlot) : "memory");
  __syncthreads(); csync();
  long long t0 = clock64();
  bool ok = true;
  for (int r = 0; r < rounds && ok; ++r) {
    const int s = r & 1;
    if (r >= 2) ok = wait(su(fre + s), ((r >> 1) - 1) & 1, err);      // the peer consumed round r - 2
    if (!ok) break;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t off = (uint32_t)(j * kT + tid) * 16;
      asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1,%2,%3,%4}, [%5];"
                   :: "r"(rslot + s * kSlot + off), "r"(r), "r"(tid), "r"(j), "r"(rank), "r"(rfull + 8 * s) : "memory");
    }
    ok = wait(su(full + s), (r >> 1) & 1, err);                         // the peer's round r landed here
    if (!ok) break;
    __syncthreads();                                                    // everyone read it
    if (tid == 0) {
      if (r + 2 < rounds)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(su(full + s)), "r"(kSlot) : "memory");
      asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" :: "r"(rfree + 8 * s) : "memory");
    }
  }
  long long t1 = clock64();
  if (tid == 0) out[blockIdx.x] = t1 - t0;
  // drain: wait for the last two rounds' frees so no remote arrive is in flight at exit
  if (ok && tid == 0)
    for (int r = (rounds >= 2 ? rounds - 2 : 0); r < rounds; ++r) wait(su(fre + (r & 1)), (r >> 1) & 1, err);
  __syncthreads(); csync();
}
int main() {
  int sms = 0; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  const int blocks = sms & ~1, rounds = 200;
  long long* d; int* err; cudaMalloc(&d, 1024 * sizeof(long long)); cudaMalloc(&err, 4); cudaMemset(err, 0, 4);
  cudaFuncSetAttribute(probe, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * kSlot + 64);
  for (int rep = 0; rep < 2; ++rep) {
    probe<<<blocks, kT, 2 * kSlot + 64>>>(rounds, d, err);
    cudaError_t e = cudaDeviceSynchronize();
    static long long h[1024]; cudaMemcpy(h, d, sizeof(long long) * blocks, cudaMemcpyDeviceToHost);
    double avg = 0; for (int i = 0; i < blocks; ++i) avg += h[i]; avg /= blocks;
    int herr; cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
    printf("%s err %d: %d CTAs, %.0f cycles per 32 KB round -> %.1f B/clk per direction per SM\n",
           cudaGetErrorString(e), herr, blocks, avg / rounds, 32768.0 * rounds / avg);
  }
  return 0;
}
