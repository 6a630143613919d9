// Internal interface between the C-ABI entry points (api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace xs {

constexpr int kMaxShards = 8;
constexpr int kTileRows = 128;   // query rows per output tile and keys per KV tile
constexpr int kSlabRows = 16;    // rows per store slab (one burst unit)

// Device status codes written by the kernels (same numbers as xs_status).
constexpr int kMaxSplit = 8;   // pieces per split unit at most
constexpr int kDevTimeout = 5;
constexpr int kDevBadPlan = 6;   // a unit cut into more pieces than a merge takes

// Everything the attention kernel needs; passed as a __grid_constant__ parameter.
struct AttnParams {
  // Inputs. in_mode 0: q/k/v [B][H][N][d], one 3-D map each {d, N, B*H}, box {64, 128, 1}.
  // in_mode 1: P sequence shards [B][N/P][H_total][d] per tensor, 3-D maps
  // {d, H_total, B*N/P}, box {64, 1, 128}. All with 128-byte swizzle.
  CUtensorMap tm_q[kMaxShards], tm_k[kMaxShards], tm_v[kMaxShards];
  CUtensorMap tm_out[kMaxShards];    // 2-D destinations, box {64, 16}, 128B swizzle
  int B, N, H, P;                    // H: heads this call computes
  int in_mode;                       // 0: head-partition inputs; 1: sequence-shard inputs
  int in_rows;                       // rows per input sequence shard (in_mode 1)
  int h0, H_total;                   // global index of local head 0; heads per destination row
  int rows_per_shard;                // N / P
  int shard_mode;                    // 0: o [B][H][N][d] (tm_out[0]); 1: P shards
  int store_tile;                    // slabs issued per KV iteration: 1, 2, 4, 8
  int shared_staging;                // 1 (store_tile 8): both groups share one staging tile
  int kv_stages;                     // K/V ring depth, attn_kv_stages(d, shared_staging)
  int n_qtiles;                      // N / 128
  int n_pairs;                       // ceil(n_qtiles / 2): a work unit is a pair of Q tiles
  int n_units;                       // B * H * n_pairs
  int n_kv;                          // N / 128
  // Work list of a CTA (G = gridDim.x). sk = 0: whole units u = blockIdx.x + i*G.
  // sk = 1: first sk_waves whole units the same way (u < sk_waves*G), then
  // (stream-K) the sk_total = (n_units - sk_waves*G)*n_kv remaining (unit, KV
  // tile) iterations, unit-major, cut into G contiguous ranges, CTA c taking
  // [c*sk_total/G, (c+1)*sk_total/G); a unit cut by a range boundary is
  // finished in pieces whose partial results meet in the workspace.
  int sk, sk_waves;
  long long sk_total;
  float *ws_part;   // sk: partials [G][2 slots][2 tiles][d+2][128] fp32
  int *ws_count;    // sk: finished pieces per (first CTA of a cut unit, tile, warp)
  float scale_log2;                  // log2(e) / sqrt(d)
  int coupled;                       // 1: the issuer waits for its stores to complete
  unsigned long long *spans;         // optional: per output tile, store-issue start/end (ns)
  unsigned long long wait_limit_ns;  // bound on every on-chip wait
};

struct ShardPtrs {
  void *p[kMaxShards];
};

int attn_smem_bytes(int d);
int attn_kv_stages(int d, bool shared_staging);
cudaError_t launch_attn(const AttnParams &p, int d, int grid, cudaStream_t s);
// The single-tile kernel with double-buffered scores (d = 256): keys per KV
// step, CTAs per SM, launch.
int wide_keys_per_step(int d);
int wide_ctas_per_sm(int d);
cudaError_t launch_attn_wide(const AttnParams &p, int d, int grid, cudaStream_t s);
cudaError_t launch_scatter(const void *o, const ShardPtrs &sh, int B, int N, int H, int d,
                           int rows_per_shard, int grid, cudaStream_t s);
cudaError_t launch_burst_probe(void *dst, int K, long long burst_bytes, int n_bursts,
                               long long gap_ns, int mode, unsigned long long *times,
                               cudaStream_t s);
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s);
cudaError_t launch_exp2_selftest(const float *x, float *out_poly, float *out_mufu, int n,
                                 cudaStream_t s);
cudaError_t read_and_clear_status(cudaStream_t s, int *out);

}  // namespace xs
