// Store-burst probe: the local (single-GPU) analog of the X-Stage remote-store
// microbenchmarks (Pith review: "What would settle it" — a zero-gap periodic
// burst run and an isolated-burst sweep; Figure 3 caption: remote-store
// microbenchmark characterisation), used to calibrate the Burst-Gap parameters
// T_iss^0, R and Q for stores into local HBM.
//
// K producer CTAs (128 threads each) issue n_bursts bursts of burst_bytes each,
// separated by a producer-side gap of gap_ns during which they issue no stores.
// Every burst writes fresh memory. Per burst, thread 0 records the
// %globaltimer when the CTA starts issuing and when the last thread has issued
// its last store (sender-visible issue span).
//   mode 0: posted st.global.v4 from all 128 threads (16 B each, coalesced);
//   mode 1: one TMA bulk copy shared -> global per 16 KiB; the span ends when
//           the copies have read their shared-memory source (the point at which
//           the issuer may reuse it), i.e. when the stores are accepted.
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace xs {
namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeSmem = 16384;   // TMA source buffer (mode 1)

__device__ __forceinline__ void spin_until(uint64_t t_end) {
  while (globaltimer_ns() < t_end) {
  }
}

__global__ void __launch_bounds__(kProbeThreads) burst_probe_kernel(
    uint8_t *dst, long long burst_bytes, int n_bursts, long long gap_ns, int mode,
    unsigned long long *times) {
  __shared__ __align__(128) uint8_t src[kProbeSmem];
  __shared__ uint64_t t_start;
  for (int i = threadIdx.x; i < kProbeSmem / 16; i += kProbeThreads)
    reinterpret_cast<uint4 *>(src)[i] = make_uint4(i, blockIdx.x, 0x5a5a5a5au, 0u);
  fence_proxy_async_smem();
  __syncthreads();
  uint8_t *base = dst + static_cast<long long>(blockIdx.x) * n_bursts * burst_bytes;
  const uint4 val = make_uint4(threadIdx.x, blockIdx.x, 1u, 2u);
  for (int b = 0; b < n_bursts; ++b) {
    uint8_t *out = base + static_cast<long long>(b) * burst_bytes;
    __syncthreads();
    if (threadIdx.x == 0) t_start = globaltimer_ns();
    __syncthreads();
    if (mode == 0) {
      uint4 *o = reinterpret_cast<uint4 *>(out);
      const long long n = burst_bytes / 16;
      for (long long i = threadIdx.x; i < n; i += kProbeThreads) {
        asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(o + i), "r"(val.x),
                     "r"(val.y), "r"(val.z), "r"(val.w)
                     : "memory");
      }
    } else if (threadIdx.x == 0) {
      for (long long off = 0; off < burst_bytes; off += kProbeSmem) {
        const long long n = burst_bytes - off < kProbeSmem ? burst_bytes - off : kProbeSmem;
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(out + off),
                     "r"(smem_u32(src)), "r"(static_cast<uint32_t>(n))
                     : "memory");
      }
      bulk_commit();
      bulk_wait_read_all();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      const uint64_t t_end = globaltimer_ns();
      const long long idx = (static_cast<long long>(blockIdx.x) * n_bursts + b) * 2;
      times[idx] = t_start;
      times[idx + 1] = t_end;
      if (gap_ns > 0) spin_until(t_end + static_cast<uint64_t>(gap_ns));   // bounded by gap_ns
    }
  }
  if (mode == 1 && threadIdx.x == 0) bulk_wait_all();
}

}  // namespace

cudaError_t launch_burst_probe(void *dst, int K, long long burst_bytes, int n_bursts,
                               long long gap_ns, int mode, unsigned long long *times,
                               cudaStream_t s) {
  burst_probe_kernel<<<K, kProbeThreads, 0, s>>>(static_cast<uint8_t *>(dst), burst_bytes,
                                                 n_bursts, gap_ns, mode, times);
  return cudaGetLastError();
}

}  // namespace xs
