// The post-attention All-to-All layout as a standalone copy kernel (the
// separate A2A step of serial execution; X-Stage abstract and Figure 5 (e)):
//   o [B][H][N][d]  ->  shard p [B][N/P][H][d],  p = n / (N/P), i = n % (N/P).
// HBM-bound: every byte is read once and written once. Each row of d bf16
// (128, 256 or 512 contiguous bytes on both sides) is moved by d/8 lanes with one
// 16-byte vector each, so a warp touches whole 128-byte lines on both sides.
#include <cstdint>

#include "internal.h"

namespace xs {
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// A warp moves tiles of kTileRowsW consecutive rows of one (b, h): one 64-bit
// division per tile finds b, h and the first row n0, so the per-row index work
// is one 32-bit division for the shard; all of a tile's loads are in flight
// before its stores.
constexpr int kTileRowsW = 32;

template <int D>
__global__ void __launch_bounds__(256) scatter_kernel(const uint4 *__restrict__ o,
                                                      const __grid_constant__ ShardPtrs sh, int N,
                                                      int H, int R, long long rows_total) {
  constexpr int VPR = D / 8;               // 16-byte vectors per row
  constexpr int RPW = 32 / VPR;            // rows per warp step
  constexpr int STEPS = kTileRowsW / RPW;  // warp steps per tile
  const int lane = threadIdx.x & 31;
  const int sub = lane / VPR, c = lane % VPR;
  const long long warp_id = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long tiles = rows_total / kTileRowsW;   // N is a multiple of 128
  for (long long tile = warp_id; tile < tiles; tile += n_warps) {
    const long long row0 = tile * kTileRowsW;        // row = (b*H + h)*N + n
    const long long bh = row0 / N;
    const int n0 = static_cast<int>(row0 - bh * N);
    const int b = static_cast<int>(bh / H), h = static_cast<int>(bh - static_cast<long long>(b) * H);
    const uint4 *src = o + (row0 + sub) * VPR + c;
    uint4 v[STEPS];
#pragma unroll
    for (int k = 0; k < STEPS; ++k) v[k] = ld_stream(src + k * RPW * VPR);
#pragma unroll
    for (int k = 0; k < STEPS; ++k) {
      const int n = n0 + k * RPW + sub;
      const int p = n / R, i = n - p * R;
      uint4 *dst = reinterpret_cast<uint4 *>(sh.p[p]) +
                   ((static_cast<long long>(b) * R + i) * H + h) * VPR + c;
      st_stream(dst, v[k]);
    }
  }
}

}  // namespace

cudaError_t launch_scatter(const void *o, const ShardPtrs &sh, int B, int N, int H, int d,
                           int rows_per_shard, int grid, cudaStream_t s) {
  const long long rows = static_cast<long long>(B) * H * N;
  if (d == 256)
    scatter_kernel<256><<<grid, 256, 0, s>>>(static_cast<const uint4 *>(o), sh, N, H,
                                             rows_per_shard, rows);
  else if (d == 128)
    scatter_kernel<128><<<grid, 256, 0, s>>>(static_cast<const uint4 *>(o), sh, N, H,
                                             rows_per_shard, rows);
  else
    scatter_kernel<64><<<grid, 256, 0, s>>>(static_cast<const uint4 *>(o), sh, N, H,
                                            rows_per_shard, rows);
  return cudaGetLastError();
}

}  // namespace xs
