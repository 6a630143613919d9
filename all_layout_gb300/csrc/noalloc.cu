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
// use the array's name as a device address (on the host it names a stand-in),
// so every call asks the runtime for the array's device address on the current
// device. That lookup allocates nothing; after the first call on a device it
// only reads the loaded module's symbol table, and because it is repeated per
// call, a device reset that reloads the module (and may move the array) never
// leaves a stale address behind. The first call on a device may load the
// library's device code, so it should come before any stream capture.
#include <cuda_runtime.h>

#include "../../include/xs.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[XS_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device.
xs_status scratch_address(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return XS_ERR_CUDA;
  *out = p;
  return XS_OK;
}

// True when B*H*N*d bf16 values fit the array. Each factor is checked against
// what is left of the budget before multiplying, so no product can wrap.
bool fits(int B, int N, int H, int d) {
  unsigned long long left = XS_NOALLOC_SCRATCH_BYTES / 2;   // bf16 elements
  const int f[4] = {B, H, N, d};
  for (int i = 0; i < 4; ++i) {
    if (f[i] == 0) return true;                             // empty problem
    const unsigned long long x = static_cast<unsigned long long>(f[i]);
    if (x > left) return false;
    left /= x;
  }
  return true;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) xs_status xs_attn_serial_noalloc(
    const void *q, const void *k, const void *v, void *const *out_shards, int B, int N, int H,
    int d, int P, void *stream) {
  if (B < 0 || N < 0 || H < 0 || d < 0) return XS_ERR_INVALID;
  if (!fits(B, N, H, d)) return XS_ERR_INVALID;
  void *scratch = nullptr;
  const xs_status st = scratch_address(&scratch);
  if (st != XS_OK) return st;
  return xs_attn_serial(q, k, v, scratch, out_shards, B, N, H, d, P, stream);
}
