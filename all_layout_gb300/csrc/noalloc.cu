// Serial attention-then-layout for callers that cannot allocate device memory.
//
// xs_attn_serial needs an intermediate o buffer [B][H][N][d] between the
// attention kernel and the layout kernel, which its caller must allocate. Some
// callers cannot: code embedded in a host framework that owns every byte of
// device memory through its own allocator or a fixed memory plan and forbids
// side allocations, or latency-critical loops where a cudaMalloc/cudaFree pair
// would synchronise the device. For them, xs_attn_serial_noalloc keeps the
// intermediate in a fixed-size array compiled into this library.
//
// The array is a file-scope __device__ object: every GPU that loads the library
// holds its XS_NOALLOC_SCRATCH_BYTES until the process exits. Host code cannot
// use the array's name as a device address, so on the first call on each device
// (with that device current) the entry point asks the runtime for the array's
// device address and caches it; later calls on that device reuse it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/xs.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[XS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_scratch on the current device (set up once per device).
xs_status scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return XS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return XS_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return XS_OK;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) xs_status xs_attn_serial_noalloc(
    const void *q, const void *k, const void *v, void *const *out_shards, int B, int N, int H,
    int d, int P, void *stream) {
  if (B < 0 || N < 0 || H < 0 || d < 0) return XS_ERR_INVALID;
  const unsigned long long need = static_cast<unsigned long long>(B) * H * N * d * 2ull;
  if (need > XS_NOALLOC_SCRATCH_BYTES) return XS_ERR_INVALID;
  void *scratch = nullptr;
  const xs_status st = scratch_address(&scratch);
  if (st != XS_OK) return st;
  return xs_attn_serial(q, k, v, scratch, out_shards, B, N, H, d, P, stream);
}
