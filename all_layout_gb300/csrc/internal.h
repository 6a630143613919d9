// Internal interface between the C-ABI entry points (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace xs {

constexpr int kMaxShards = 8;
constexpr int kTileRows = 128;   // query rows per output tile and keys per KV tile
constexpr int kSlabRows = 16;    // rows per store slab (one burst unit)

// Device status codes written by the kernels (same numbers as xs_status).
constexpr int kDevTimeout = 5;

// Everything the attention kernel needs; passed as a __grid_constant__ parameter.
struct AttnParams {
  CUtensorMap tm_q, tm_k, tm_v;      // 3-D {d, N, B*H}, box {64, 128, 1}, 128B swizzle
  CUtensorMap tm_out[kMaxShards];    // 2-D destinations, box {64, 16}, 128B swizzle
  int B, N, H, P;
  int rows_per_shard;                // N / P
  int shard_mode;                    // 0: o [B][H][N][d] (tm_out[0]); 1: P shards
  int store_tile;                    // slabs issued per KV iteration: 1, 2, 4, 8
  int shared_staging;                // 1 (store_tile 8): both groups share one staging tile
  int kv_stages;                     // K/V ring depth, attn_kv_stages(d, shared_staging)
  int n_qtiles;                      // N / 128
  int n_pairs;                       // ceil(n_qtiles / 2): a work unit is a pair of Q tiles
  int n_units;                       // B * H * n_pairs
  int n_kv;                          // N / 128
  float scale_log2;                  // log2(e) / sqrt(d)
  unsigned long long wait_limit_ns;  // bound on every on-chip wait
};

struct ShardPtrs {
  void *p[kMaxShards];
};

int attn_smem_bytes(int d);
int attn_kv_stages(int d, bool shared_staging);
cudaError_t launch_attn(const AttnParams &p, int d, int grid, cudaStream_t s);
cudaError_t launch_scatter(const void *o, const ShardPtrs &sh, int B, int N, int H, int d,
                           int rows_per_shard, int grid, cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s);
cudaError_t read_and_clear_status(cudaStream_t s, int *out);

}  // namespace xs
