// C-ABI entry points of libxs (declared in include/xs.h): argument validation,
// TMA tensor-map encoding and kernel launches. Host code only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/xs.h"
#include "internal.h"

#define XS_API extern "C" __attribute__((visibility("default")))

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;
std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  static std::mutex mu;
  static int cached[64] = {0};
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return -1;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cached[dev] = n;
  }
  return cached[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Caller-owned workspace for the stream-K schedule, one per device (xs_set_workspace).
struct Workspace {
  void *ptr;
  unsigned long long bytes;
};
std::mutex g_ws_mu;
Workspace g_ws[64] = {};

Workspace current_workspace() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Workspace{nullptr, 0};
  std::lock_guard<std::mutex> lock(g_ws_mu);
  return g_ws[dev];
}

// Schedule of one launch: whole units strided over `grid` persistent CTAs, or
// whole units for all but the last full wave followed by a balanced (stream-K)
// split of the rest into equal contiguous ranges of (unit, KV tile)
// iterations. The strided waves keep the CTAs on neighbouring units (the same
// heads' K/V in L2); the stream-K region is at most two waves wide, so its
// ranges stay within a few neighbouring heads too.
struct Plan {
  int sk, sk_waves, grid;
  unsigned long long bytes;   // workspace the plan needs (0 for whole units)
};

// Cost model in KV-tile iterations of one CTA: each item adds a fill/drain and
// epilogue cost, each cut unit a partial write or merge.
constexpr long kItemCost = 2;
constexpr long kPieceCost = 3;
constexpr long kMinPerCta = 4;

unsigned long long sk_bytes(int grid, int d) {
  return XS_WORKSPACE_HEADER_BYTES +
         static_cast<unsigned long long>(grid) * 2 * 2 * (d + 2) * xs::kTileRows * 4;
}

// The stream-K plan when a workspace of `ws_bytes` holds it and the model says
// it is shorter than whole units; every unit is cut into at most kMaxSplit pieces.
Plan plan_launch(int units, int sms, int n_kv, int d, unsigned long long ws_bytes) {
  const int grid0 = units < sms ? units : sms;
  const Plan whole{0, 0, grid0, 0};
  if (n_kv < 2 || (units % grid0 == 0 && units >= sms)) return whole;
  const int waves = units >= sms ? units / sms - 1 : 0;
  const long long T = static_cast<long long>(units - waves * sms) * n_kv;
  long long per = (T + sms - 1) / sms, grid = sms;
  if (waves == 0) {
    if (per < kMinPerCta) per = kMinPerCta;
    grid = (T + per - 1) / per;
    // A unit overlaps at most ceil((n_kv - 1) / shortest range) + 1 ranges.
    while ((n_kv - 1 + T / grid - 1) / (T / grid) + 1 > xs::kMaxSplit) {
      ++per;
      grid = (T + per - 1) / per;
    }
  }
  const long items = static_cast<long>((per + n_kv - 1) / n_kv) + 1;
  const long cost_sk = waves * (n_kv + kItemCost) + static_cast<long>(per) + items * kItemCost +
                       2 * kPieceCost;
  const long cost_whole = static_cast<long>((units + grid0 - 1) / grid0) * (n_kv + kItemCost);
  const unsigned long long need = sk_bytes(static_cast<int>(grid), d);
  if (cost_sk >= cost_whole || need > ws_bytes ||
      static_cast<unsigned long long>(grid) * 2 * 4 * sizeof(int) > XS_WORKSPACE_HEADER_BYTES)
    return whole;
  return Plan{1, waves, static_cast<int>(grid), need};
}

// Validation shared by every entry point, in the order the header states.
xs_status validate(const void *const *ptrs, int nptrs, void *const *shards, int B, int N, int H,
                   int d, int P, int store_tile) {
  for (int i = 0; i < nptrs; ++i)
    if (!ptrs[i]) return XS_ERR_INVALID;
  if (B < 0 || N < 0 || H < 0) return XS_ERR_INVALID;
  if (shards) {
    if (P < 1 || P > xs::kMaxShards) return XS_ERR_INVALID;
    for (int p = 0; p < P; ++p)
      if (!shards[p]) return XS_ERR_INVALID;
    if (N % P != 0) return XS_ERR_INVALID;
  }
  if (store_tile != 1 && store_tile != 2 && store_tile != 4 && store_tile != 8)
    return XS_ERR_INVALID;
  if (d != 64 && d != 128 && d != 256) return XS_ERR_UNSUPPORTED;
  // d = 256 stores each finished tile at once (no room to stage a deferred one).
  if (d == 256 && store_tile != 8) return XS_ERR_UNSUPPORTED;
  if (N % xs::kTileRows != 0) return XS_ERR_UNSUPPORTED;
  // Row coordinates of the tensor maps (b*H + h)*N + n are 32-bit.
  if (static_cast<long long>(B) * H * N > 0x7fffffffLL) return XS_ERR_UNSUPPORTED;
  for (int i = 0; i < nptrs; ++i)
    if (!aligned16(ptrs[i])) return XS_ERR_ALIGN;
  if (shards)
    for (int p = 0; p < P; ++p)
      if (!aligned16(shards[p])) return XS_ERR_ALIGN;
  return XS_OK;
}

// Tensor maps already encoded, keyed by everything the encoder reads (base
// address, rank, sizes, strides, box; the element type, swizzle and fill are the
// same for every map here). A map is a self-contained descriptor with no device
// state, so an entry stays valid whatever happens to the memory behind it; a
// repeated call on the same buffers then costs a lookup instead of 3 + P driver
// encodes. Least recently used entries are replaced.
struct MapKey {
  const void *base;
  int rank;
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
};
struct MapEntry {
  MapKey key;
  unsigned long long stamp;   // 0: empty
  CUtensorMap map;
};
constexpr int kMapCache = 96;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache] = {};
unsigned long long g_map_clock = 0;

bool encode(CUtensorMap *m, void *base, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides_bytes, const cuuint32_t *box) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));   // padding included, so keys compare bytewise
  key.base = base;
  key.rank = rank;
  for (int i = 0; i < rank; ++i) {
    key.dims[i] = dims[i];
    key.box[i] = box[i];
    if (i + 1 < rank) key.strides[i] = strides_bytes[i];
  }
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (MapEntry &e : g_maps)
      if (e.stamp && std::memcmp(&e.key, &key, sizeof(key)) == 0) {
        e.stamp = ++g_map_clock;
        *m = e.map;
        return true;
      }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), base, dims,
         strides_bytes, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapEntry *victim = &g_maps[0];
  for (MapEntry &e : g_maps)
    if (e.stamp < victim->stamp) victim = &e;
  victim->key = key;
  victim->map = *m;
  victim->stamp = ++g_map_clock;
  return true;
}

// q/k/v: 3-D {d, N, B*H}, box {64, box_rows, 1} (128 rows, or the keys of one KV
// step of the single-tile kernel for K and V).
bool encode_qkv(CUtensorMap *m, const void *base, int B, int N, int H, int d,
                int box_rows = xs::kTileRows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(B) * H};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  return encode(m, const_cast<void *>(base), 3, dims, strides, box);
}

// A sequence shard [B][rows][H_total][d] as 3-D {d, H_total, B*rows}, box {64, 1,
// box_rows}: one box is box_rows consecutive rows of one head.
bool encode_seq_shard(CUtensorMap *m, const void *base, int B, int rows, int H_total, int d,
                      int box_rows = xs::kTileRows) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H_total),
                              static_cast<cuuint64_t>(B) * rows};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(H_total) * d * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  return encode(m, const_cast<void *>(base), 3, dims, strides, box);
}

// Which kernel a launch takes: the single-tile kernel with double-buffered
// scores at d = 256 (two tiles do not fit Tensor Memory), the two-tile kernel
// otherwise.
bool single_tile(int d) { return d == 256; }

// Destination rows: 2-D {cols, rows}, row pitch cols*2 bytes, box {64, 16}.
bool encode_rows(CUtensorMap *m, void *base, unsigned long long cols, unsigned long long rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(xs::kSlabRows)};
  return encode(m, base, 2, dims, strides, box);
}

// Where the attention inputs come from: head-partition tensors (one pointer each),
// or P sequence shards per tensor with the computed heads [h0, h0 + H) of H_total.
struct Inputs {
  int seq_shards;
  const void *const *q, *const *k, *const *v;
  int h0, H_total;
};

xs_status launch_attention(const Inputs &in, void *o, void *const *shards, int B, int N, int H,
                           int d, int P, int store_tile, cudaStream_t stream, int coupled = 0,
                           unsigned long long *spans = nullptr) {
  xs::AttnParams prm;
  std::memset(&prm, 0, sizeof(prm));
  const int R = N / P;
  const bool wide = single_tile(d);
  const int kv_rows = wide ? xs::wide_keys_per_step(d) : xs::kTileRows;   // keys per KV step
  if (!in.seq_shards) {
    if (!encode_qkv(&prm.tm_q[0], in.q[0], B, N, H, d) ||
        !encode_qkv(&prm.tm_k[0], in.k[0], B, N, H, d, kv_rows) ||
        !encode_qkv(&prm.tm_v[0], in.v[0], B, N, H, d, kv_rows))
      return XS_ERR_CUDA;
    prm.in_mode = 0;
    prm.in_rows = N;
  } else {
    for (int p = 0; p < P; ++p)
      if (!encode_seq_shard(&prm.tm_q[p], in.q[p], B, R, in.H_total, d) ||
          !encode_seq_shard(&prm.tm_k[p], in.k[p], B, R, in.H_total, d, kv_rows) ||
          !encode_seq_shard(&prm.tm_v[p], in.v[p], B, R, in.H_total, d, kv_rows))
        return XS_ERR_CUDA;
    prm.in_mode = 1;
    prm.in_rows = R;
  }
  prm.h0 = in.h0;
  prm.H_total = in.H_total;
  if (shards) {
    for (int p = 0; p < P; ++p)
      if (!encode_rows(&prm.tm_out[p], shards[p], static_cast<unsigned long long>(in.H_total) * d,
                       static_cast<unsigned long long>(B) * R))
        return XS_ERR_CUDA;
    prm.shard_mode = 1;
    prm.rows_per_shard = R;
    prm.P = P;
  } else {
    if (!encode_rows(&prm.tm_out[0], o, static_cast<unsigned long long>(d),
                     static_cast<unsigned long long>(B) * H * N))
      return XS_ERR_CUDA;
    prm.shard_mode = 0;
    prm.rows_per_shard = N;
    prm.P = 1;
  }
  prm.B = B;
  prm.N = N;
  prm.H = H;
  prm.store_tile = store_tile;
  prm.coupled = coupled;
  prm.spans = spans;
  prm.shared_staging = store_tile == 8 ? 1 : 0;
  prm.kv_stages = wide ? 0 : xs::attn_kv_stages(d, store_tile == 8);
  prm.n_qtiles = N / xs::kTileRows;
  // Two-tile kernel: a unit is a pair of query tiles; single-tile kernel: one tile.
  prm.n_pairs = wide ? prm.n_qtiles : (prm.n_qtiles + 1) / 2;
  prm.n_units = B * H * prm.n_pairs;
  prm.n_kv = N / kv_rows;
  prm.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
  prm.wait_limit_ns = g_wait_limit_ns.load();
  const int sms = sm_count();
  if (sms <= 0) return XS_ERR_CUDA;
  const Workspace ws = current_workspace();
  // Persistent CTAs: one per SM, or the single-tile kernel's CTAs per SM.
  const int slots = sms * (wide ? xs::wide_ctas_per_sm(d) : 1);
  const Plan pl = plan_launch(prm.n_units, slots, prm.n_kv, d, ws.ptr ? ws.bytes : 0);
  const int grid = pl.grid;
  prm.sk = pl.sk;
  prm.sk_waves = pl.sk_waves;
  prm.sk_total = static_cast<long long>(prm.n_units - pl.sk_waves * grid) * prm.n_kv;
  if (pl.sk) {
    prm.ws_count = static_cast<int *>(ws.ptr);
    prm.ws_part = reinterpret_cast<float *>(static_cast<char *>(ws.ptr) + XS_WORKSPACE_HEADER_BYTES);
  }
  const cudaError_t e = wide ? xs::launch_attn_wide(prm, d, grid, stream)
                            : xs::launch_attn(prm, d, grid, stream);
  return e == cudaSuccess ? XS_OK : XS_ERR_CUDA;
}

xs_status launch_layout(const void *o, void *const *shards, int B, int N, int H, int d, int P,
                        cudaStream_t stream) {
  xs::ShardPtrs sh;
  for (int p = 0; p < xs::kMaxShards; ++p) sh.p[p] = p < P ? shards[p] : nullptr;
  const int sms = sm_count();
  if (sms <= 0) return XS_ERR_CUDA;
  // One warp per 32-row tile, 8 warps per block, at most 8 blocks per SM.
  const long long tiles = static_cast<long long>(B) * H * N / 32;
  long long grid = (tiles + 7) / 8;
  if (grid > static_cast<long long>(sms) * 8) grid = static_cast<long long>(sms) * 8;
  if (grid < 1) grid = 1;
  return xs::launch_scatter(o, sh, B, N, H, d, N / P, static_cast<int>(grid), stream) == cudaSuccess
             ? XS_OK
             : XS_ERR_CUDA;
}

bool empty(int B, int N, int H) { return B == 0 || N == 0 || H == 0; }

}  // namespace

XS_API xs_status xs_attn_fused(const void *q, const void *k, const void *v,
                               void *const *out_shards, int B, int N, int H, int d, int P,
                               int store_tile, void *stream) {
  if (!out_shards) return XS_ERR_INVALID;
  const void *ptrs[3] = {q, k, v};
  xs_status st = validate(ptrs, 3, out_shards, B, N, H, d, P, store_tile);
  if (st != XS_OK || empty(B, N, H)) return st;
  const Inputs in{0, &ptrs[0], &ptrs[1], &ptrs[2], 0, H};
  return launch_attention(in, nullptr, out_shards, B, N, H, d, P, store_tile,
                          static_cast<cudaStream_t>(stream));
}

XS_API xs_status xs_attn_fused_ex(const void *q, const void *k, const void *v,
                                  void *const *out_shards, int B, int N, int H, int d, int P,
                                  int store_tile, int flags, unsigned long long *spans,
                                  void *stream) {
  if (!out_shards) return XS_ERR_INVALID;
  const void *ptrs[3] = {q, k, v};
  xs_status st = validate(ptrs, 3, out_shards, B, N, H, d, P, store_tile);
  if (st != XS_OK) return st;
  if ((flags & ~XS_FLAG_COMPLETION_COUPLED) != 0) return XS_ERR_INVALID;
  const int coupled = (flags & XS_FLAG_COMPLETION_COUPLED) ? 1 : 0;
  if (coupled && store_tile != 8) return XS_ERR_INVALID;
  if (spans && (reinterpret_cast<uintptr_t>(spans) & 7u) != 0) return XS_ERR_ALIGN;
  if (empty(B, N, H)) return XS_OK;
  const Inputs in{0, &ptrs[0], &ptrs[1], &ptrs[2], 0, H};
  return launch_attention(in, nullptr, out_shards, B, N, H, d, P, store_tile,
                          static_cast<cudaStream_t>(stream), coupled, spans);
}

XS_API xs_status xs_attn(const void *q, const void *k, const void *v, void *o, int B, int N, int H,
                         int d, void *stream) {
  const void *ptrs[4] = {q, k, v, o};
  xs_status st = validate(ptrs, 4, nullptr, B, N, H, d, 1, 8);
  if (st != XS_OK || empty(B, N, H)) return st;
  const Inputs in{0, &ptrs[0], &ptrs[1], &ptrs[2], 0, H};
  return launch_attention(in, o, nullptr, B, N, H, d, 1, 8,
                          static_cast<cudaStream_t>(stream));
}

XS_API xs_status xs_scatter(const void *o, void *const *out_shards, int B, int N, int H, int d,
                            int P, void *stream) {
  if (!out_shards) return XS_ERR_INVALID;
  const void *ptrs[1] = {o};
  xs_status st = validate(ptrs, 1, out_shards, B, N, H, d, P, 8);
  if (st != XS_OK || empty(B, N, H)) return st;
  return launch_layout(o, out_shards, B, N, H, d, P, static_cast<cudaStream_t>(stream));
}

XS_API xs_status xs_attn_serial(const void *q, const void *k, const void *v, void *o_scratch,
                                void *const *out_shards, int B, int N, int H, int d, int P,
                                void *stream) {
  if (!out_shards) return XS_ERR_INVALID;
  const void *ptrs[4] = {q, k, v, o_scratch};
  xs_status st = validate(ptrs, 4, out_shards, B, N, H, d, P, 8);
  if (st != XS_OK || empty(B, N, H)) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Inputs in{0, &ptrs[0], &ptrs[1], &ptrs[2], 0, H};
  st = launch_attention(in, o_scratch, nullptr, B, N, H, d, 1, 8, s);
  if (st != XS_OK) return st;
  return launch_layout(o_scratch, out_shards, B, N, H, d, P, s);
}

XS_API xs_status xs_attn_ulysses(const void *const *q_shards, const void *const *k_shards,
                                 const void *const *v_shards, void *const *out_shards, int B,
                                 int N, int H_total, int h0, int H, int d, int P, int store_tile,
                                 void *stream) {
  if (!q_shards || !k_shards || !v_shards || !out_shards) return XS_ERR_INVALID;
  if (P < 1 || P > xs::kMaxShards) return XS_ERR_INVALID;
  for (int p = 0; p < P; ++p)
    if (!q_shards[p] || !k_shards[p] || !v_shards[p]) return XS_ERR_INVALID;
  if (H_total < 1 || h0 < 0 || H < 0 || h0 + H > H_total) return XS_ERR_INVALID;
  xs_status st = validate(nullptr, 0, out_shards, B, N, H, d, P, store_tile);
  if (st != XS_OK) return st;
  if ((N / P) % xs::kTileRows != 0) return XS_ERR_UNSUPPORTED;
  for (int p = 0; p < P; ++p)
    if (!aligned16(q_shards[p]) || !aligned16(k_shards[p]) || !aligned16(v_shards[p]))
      return XS_ERR_ALIGN;
  if (empty(B, N, H)) return XS_OK;
  const Inputs in{1, q_shards, k_shards, v_shards, h0, H_total};
  return launch_attention(in, nullptr, out_shards, B, N, H, d, P, store_tile,
                          static_cast<cudaStream_t>(stream));
}

XS_API xs_status xs_store_burst_probe(void *dst, unsigned long long dst_bytes, int K,
                                      unsigned long long burst_bytes, int n_bursts,
                                      unsigned long long gap_ns, int mode,
                                      unsigned long long *times, void *stream) {
  if (!dst || !times || K < 1 || K > 1024 || n_bursts < 1 || (mode != 0 && mode != 1) ||
      burst_bytes < 2048 || burst_bytes % 2048 != 0 || gap_ns > 1000000000ull)
    return XS_ERR_INVALID;
  if (dst_bytes / burst_bytes / static_cast<unsigned long long>(n_bursts) <
      static_cast<unsigned long long>(K))
    return XS_ERR_INVALID;
  if (!aligned16(dst) || (reinterpret_cast<uintptr_t>(times) & 7u) != 0) return XS_ERR_ALIGN;
  return xs::launch_burst_probe(dst, K, static_cast<long long>(burst_bytes), n_bursts,
                                static_cast<long long>(gap_ns), mode, times,
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? XS_OK
             : XS_ERR_CUDA;
}

XS_API const char *xs_status_string(xs_status s) {
  switch (s) {
    case XS_OK: return "ok";
    case XS_ERR_INVALID: return "invalid argument";
    case XS_ERR_UNSUPPORTED:
      return "unsupported shape (d must be 64, 128 or 256, N a multiple of 128; d = 256 needs "
             "store_tile 8)";
    case XS_ERR_ALIGN: return "pointer not 16-byte aligned";
    case XS_ERR_CUDA: return "CUDA error";
    case XS_ERR_TIMEOUT: return "on-chip wait timed out";
  }
  return "unknown status";
}

XS_API xs_status xs_last_device_status(void *stream) {
  int v = 0;
  if (xs::read_and_clear_status(static_cast<cudaStream_t>(stream), &v) != cudaSuccess)
    return XS_ERR_CUDA;
  return v == xs::kDevTimeout ? XS_ERR_TIMEOUT : (v == 0 ? XS_OK : XS_ERR_CUDA);
}

XS_API unsigned long long xs_set_wait_limit_ns(unsigned long long limit_ns) {
  return g_wait_limit_ns.exchange(limit_ns ? limit_ns : kDefaultWaitLimitNs);
}

XS_API xs_status xs_selftest_bounded_wait(void *stream) {
  return xs::launch_wait_selftest(g_wait_limit_ns.load(), static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? XS_OK
             : XS_ERR_CUDA;
}

XS_API xs_status xs_selftest_exp2(const float *x, float *out_poly, float *out_mufu, int n,
                                  void *stream) {
  if (!x || !out_poly || !out_mufu || n < 0) return XS_ERR_INVALID;
  if (n == 0) return XS_OK;
  return xs::launch_exp2_selftest(x, out_poly, out_mufu, n, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? XS_OK
             : XS_ERR_CUDA;
}

XS_API xs_status xs_set_workspace(void *ws, unsigned long long bytes, void *stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return XS_ERR_CUDA;
  if (ws) {
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return XS_ERR_ALIGN;
    if (bytes < XS_WORKSPACE_HEADER_BYTES) return XS_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, XS_WORKSPACE_HEADER_BYTES, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return XS_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_ws_mu);
  g_ws[dev] = ws ? Workspace{ws, bytes} : Workspace{nullptr, 0};
  return XS_OK;
}

XS_API xs_status xs_workspace_bytes(int B, int N, int H, int d, unsigned long long *bytes,
                                    int *cut) {
  if (!bytes || B < 0 || N < 0 || H < 0) return XS_ERR_INVALID;
  if (d != 64 && d != 128 && d != 256) return XS_ERR_UNSUPPORTED;
  if (N % xs::kTileRows != 0) return XS_ERR_UNSUPPORTED;
  *bytes = 0;
  if (cut) *cut = 0;
  if (empty(B, N, H)) return XS_OK;
  const int sms = sm_count();
  if (sms <= 0) return XS_ERR_CUDA;
  const int n_qtiles = N / xs::kTileRows;
  const bool wide = single_tile(d);
  const int kv_rows = wide ? xs::wide_keys_per_step(d) : xs::kTileRows;
  const int units = B * H * (wide ? n_qtiles : (n_qtiles + 1) / 2);
  const Plan pl = plan_launch(units, sms * (wide ? xs::wide_ctas_per_sm(d) : 1), N / kv_rows, d,
                              ~0ull);
  *bytes = pl.bytes;
  if (cut) *cut = pl.sk;
  return XS_OK;
}

XS_API int xs_abi_version(void) { return 1; }
