// Non-causal attention fused with the post-attention Ulysses All-to-All layout,
// for sm_103a (tcgen05 tensor cores, Tensor Memory, TMA).
//
// Method: "X-Stage: An Overlooked Pipeline Stage for Communication-Computation
// Overlap in DiT Inference". Abstract: tile-granular fusion of the post-attention
// All-to-All with FlashAttention, where the owner of an output tile issues the
// tile's stores itself and resumes computation, without a dedicated
// communication warp or SM. Figure 6: FlashAttention Q-loop and output tiling.
// Figure 7 / Figure 1: the stores of one tile drain while the next mainloop
// computes. Pith review, "If this is right": a Q-loop longer than the recovery
// gap absorbs the drain.
//
// Work unit: one (batch, head) and a PAIR of 128-row query tiles (a single tile
// for the last unit of a head with an odd tile count: group 1 sits that unit
// out). A persistent CTA walks units head-major, so a head's K/V stay hot in L2
// across CTAs. With a
// caller workspace the last waves may instead be cut into equal ranges of
// (unit, KV tile) iterations (stream-K); a unit cut by a range boundary runs as
// pieces whose partial results are merged on the GPU (get_item, finish_piece).
//
// Roles (320 threads at d = 128, 352 at d = 64; one CTA per SM):
//   warps 0-3  softmax warp group 0: owns query tile 0 of the unit (S0, P0, O0)
//   warps 4-7  softmax warp group 1: owns query tile 1 (S1, P1, O1)
//   warp 8     MMA issuer + Tensor Memory allocation (d = 64: the QK^T issuer)
//   warp 9     TMA loader
//   warp 10    d = 64 only: the PV issuer
// The issuer and loader warps run their control flow as whole warps (values stay
// warp-uniform) and one elected lane issues each group of tcgen05 or TMA
// operations.
// Each softmax warp group also rescales its O rows, finalises them, stages the
// bf16 tile in shared memory and issues the tile's stores to the destination
// shards as TMA bulk stores: with store_tile = 8 each warp stages and stores its
// own 32 rows as two 16-row slabs through a private one-slab buffer; with
// store_tile < 8, store_tile 16-row slabs go out after each KV iteration of the
// group's next unit. No warp exists only to store.
//
// Tensor Memory (512 columns x 128 lanes, row r of a tile = lane r):
//   S0 [0,128)  S1 [128,256)  O0 [256,256+d)  O1 [256+d,256+2d)
//   d = 128: P_t (bf16, two per column) overwrites the first 64 columns of S_t.
//   d = 64:  P0 [384,448)  P1 [448,512), so S_t is free once it is read (EARLY_QK).
// Shared memory (d = 128): Q0 Q1 | five 32 KiB regions: 4 K/V slots + 1 staging
// tile cut into eight 4 KiB one-slab buffers, one per softmax warp (store_tile =
// 8), or 3 K/V slots + 1 staging tile per group (store_tile < 8) | barriers. Every
// tile is stored as 64-column halves of its rows x 128 bytes, 128-byte swizzle.
//
// MMA order per KV step j at d = 128 (t = 0, 1): O_t += P_t(j-1) V(j-1);
// S_t = Q_t K(j)^T. tcgen05 operations issued by one thread execute in order, so
// S_t(j) cannot overwrite P_t(j-1) before the PV MMA that reads it; and the
// commit that signals S_t(j) also covers PV_t(j-1), so the softmax group may
// rescale O_t as soon as it sees S_t(j).
// At d = 64 (EARLY_QK) S_t(j+1) = Q_t K(j+1)^T is issued as soon as the group
// has read S_t(j) into registers, by its own warp, and O_t += P_t(j) V(j) by
// another once P_t(j) is written; the group waits for PV_t(j-1) (pv_done) before
// it overwrites P_t or rescales O_t (qk_issuer, pv_issuer).
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"


namespace xs {

__device__ int g_status;

namespace {

constexpr int BM = kTileRows;            // query rows per tile
constexpr int BN = kTileRows;            // keys per KV tile
constexpr int NSLAB = BM / kSlabRows;    // 8 slabs per output tile
constexpr int kMmaWarp = 8;    // the MMA issuer (with EARLY_QK: the QK^T issuer)
constexpr int kLoadWarp = 9;
constexpr int kPvWarp = 10;    // EARLY_QK only: the PV issuer
constexpr int kHalfBytes = BM * 128;     // one 64-column half of a 128-row tile
constexpr uint32_t kWaitSleepNs = 100000;   // longest suspension per try in a blocked wait
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

// Exponentials computed by the polynomial (exp2_poly_x2) instead of MUFU ex2:
// the pairs i of each 32-column chunk with (i * N) % 16 < N, i.e. N of every 16
// pairs spread evenly. Measured at N = 16384 with a single MMA issuer (TFLOP/s
// for N = 0, 1, 2, 3, 4, 6): d = 64 H = 48: 1105, 1105, 1085, 1003, 865, 861;
// d = 128 H = 24: 1764, 1779, 1632 for N = 0, 1, 2. The exponential phase is
// issue-bound, not MUFU-bound: an arithmetic-only test of it (two warps per SM
// sub-partition, packed row sums) takes 39% and 60% more cycles per row with 2
// and 4 of 16 pairs on the polynomial, which costs ten instructions per pair
// against two MUFU issues. So no pair takes it.
template <int D>
struct PolyPairs {
  static constexpr int N = 0;
  static __device__ __forceinline__ constexpr bool take(int i) { return N > 0 && (i * N) % 16 < N; }
};

template <int D, bool SHARED>
struct Cfg {
  static constexpr int NH = D / 64;
  static constexpr int TILE = BM * D * 2;
  // After the two Q tiles come NREG tile-sized regions shared by the K/V ring and
  // the output staging: with store_tile = 8 the two warp groups take turns on one
  // staging tile (NREG-1 ring slots); with deferred bursts each group keeps its
  // own staging tile (NREG-2 ring slots).
  static constexpr int NREG = (D == 128) ? 5 : 11;
  static constexpr int MAX_STAGES = NREG - 1;
  static constexpr int KV_STAGES = SHARED ? NREG - 1 : NREG - 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + 2 * TILE;
  static constexpr int OFF_BAR = OFF_KV + NREG * TILE;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;   // + slack to align the base to 1024
  static constexpr uint32_t COL_S0 = 0, COL_S1 = 128;
  static constexpr uint32_t COL_O0 = 256, COL_O1 = 256 + D;
  // d = 64 leaves 128 Tensor Memory columns free, so P gets its own columns
  // (bf16 pairs, 64 per tile) instead of overwriting S. S is then free once the
  // softmax has read it, and the next QK^T of a tile is issued at that point,
  // overlapping the tile's exponentials (EARLY_QK). At d = 128 S and O fill all
  // 512 columns and P overwrites the S it came from.
  static constexpr bool EARLY_QK = (D == 64);
  static constexpr int THREADS = EARLY_QK ? 352 : 320;   // 8 softmax warps, issuer(s), loader
  static constexpr uint32_t COL_P0 = EARLY_QK ? 256 + 2 * D : COL_S0;
  static constexpr uint32_t COL_P1 = EARLY_QK ? 256 + 2 * D + 64 : COL_S1;
  static_assert(!EARLY_QK || COL_P1 + 64 <= 512, "P columns past the Tensor Memory allocation");
};

// Store bookkeeping of one warp group, kept in shared memory and touched only by
// the group's elected thread (keeps registers free for the softmax).
struct StoreState {
  int bh, q0, next;   // pending tile and the next slab to issue (NSLAB: nothing pending)
  int pad;
  uint64_t t0;        // when the tile's first slab was issued (span recording)
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[10], kv_empty[10];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t s_free[2], pv_done[2];   // EARLY_QK only: S read by the softmax; PV(j) complete
  uint64_t wg_sync[2];
  uint64_t drain;
  StoreState store[2];  // per warp group
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block too large");

__device__ __forceinline__ void record_timeout(volatile int *abort_flag) {
  *abort_flag = 1;
  atomicExch(&g_status, kDevTimeout);
}

// Bounded wait on a barrier phase, slow path. Gives up when another role has
// aborted or when `limit` ns pass, in which case it records a timeout.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity,
                                             volatile int *abort_flag, uint64_t limit) {
  // The MMA issuer polls (it must react to a finished P at once); every other
  // role sleeps between polls so its waiting costs no issue slots.
  const bool sleepy = (threadIdx.x / 32) != kMmaWarp && (threadIdx.x / 32) != kPvWarp;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (sleepy ? mbar_try_wait_sleep(bar, parity, kWaitSleepNs) : mbar_try_wait(bar, parity))
      return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit) {
        record_timeout(abort_flag);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                           uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_phase_slow(bar, parity, abort_flag, limit);
}

// The same bounded wait with no out-of-line call, for a wait made while most
// registers are live (a call there would force them to be spilled around it).
__device__ __forceinline__ bool wait_phase_inline(uint32_t bar, uint32_t parity,
                                                  volatile int *abort_flag, uint64_t limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > limit) {
        record_timeout(abort_flag);
        return false;
      }
    }
  }
}

// Wait used while tearing down after an abort: ignores the abort flag, still bounded.
__device__ __noinline__ bool drain_phase(uint32_t bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit) return false;
  }
  return true;
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ------------------------------------------------------------------ TMA loader
// Where the 64-column half `hf` of rows [row0, row0 + 128) of local head-unit bh
// lives. Head-partition inputs: one map, (x, row, b*H + h). Sequence-shard
// inputs (the pre-attention All-to-All folded into the load, Figure 5 (a)-(c)):
// the shard holding row0, (x, h0 + h, b*rows + row0 - shard*rows); 128-row tiles
// never straddle two shards because rows per shard is a multiple of 128.
struct TileSrc {
  const CUtensorMap *m;
  int x, y, z;
};
__device__ __forceinline__ TileSrc tile_src(const AttnParams &p, const CUtensorMap *maps, int hf,
                                            int row0, int bh) {
  if (p.in_mode == 0) return TileSrc{&maps[0], hf * 64, row0, bh};
  const int b = bh / p.H, h = bh - b * p.H;
  const int sh = row0 / p.in_rows;
  return TileSrc{&maps[sh], hf * 64, p.h0 + h, b * p.in_rows + (row0 - sh * p.in_rows)};
}
__device__ __forceinline__ void load_tile(const AttnParams &p, const CUtensorMap *maps,
                                          uint32_t dst, uint32_t bar, int hf, int row0, int bh) {
  const TileSrc t = tile_src(p, maps, hf, row0, bh);
  tma_load_3d(dst, t.m, bar, t.x, t.y, t.z);
}
__device__ __forceinline__ void prefetch_tile(const AttnParams &p, const CUtensorMap *maps, int hf,
                                              int row0, int bh) {
  const TileSrc t = tile_src(p, maps, hf, row0, bh);
  tma_prefetch_l2_3d(t.m, t.x, t.y, t.z);
}

// One entry of a CTA's work list: a unit (b*H + h, pair of query tiles) and the
// KV tiles [kv0, kv1) to process; piece != 0 marks a piece of a cut unit.
struct Item {
  int unit, kv0, kv1, piece;
};

// Query tiles of a unit: 2, or 1 for the last pair of a head with an odd tile
// count (its second tile would lie past the sequence; nothing computes it).
__device__ __forceinline__ int unit_tiles(const AttnParams &p, int unit) {
  return 2 * (unit % p.n_pairs) + 1 < p.n_qtiles ? 2 : 1;
}

// First iteration of CTA c's stream-K range.
__device__ __forceinline__ long long sk_start(const AttnParams &p, int c) {
  return static_cast<long long>(c) * p.sk_total / static_cast<long long>(gridDim.x);
}

// The k-th item of this CTA's work list; false past its end.
__device__ __forceinline__ bool get_item(const AttnParams &p, int k, Item &it) {
  if (!p.sk || k < p.sk_waves) {
    const int u = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
    it = Item{u, 0, p.n_kv, 0};
    return u < p.n_units;
  }
  k -= p.sk_waves;
  const long long s0 = sk_start(p, blockIdx.x), e0 = sk_start(p, blockIdx.x + 1);
  const long long pos = k == 0 ? s0 : (s0 / p.n_kv + k) * p.n_kv;
  if (pos >= e0) return false;
  const int v = static_cast<int>(pos / p.n_kv);   // unit within the stream-K region
  const int kv0 = static_cast<int>(pos - static_cast<long long>(v) * p.n_kv);
  const long long left = e0 - pos;
  const int kv1 = left < p.n_kv - kv0 ? kv0 + static_cast<int>(left) : p.n_kv;
  it = Item{p.sk_waves * static_cast<int>(gridDim.x) + v, kv0, kv1,
            (kv0 > 0 || kv1 < p.n_kv) ? 1 : 0};
  return true;
}

template <int D, bool SHARED>
__device__ void load_role(const AttnParams &p, uint8_t *smem, Bars *bars, volatile int *abort_flag) {
  using C = Cfg<D, SHARED>;
  const uint64_t lim = p.wait_limit_ns;
  constexpr uint32_t stages = C::KV_STAGES;
  uint32_t it = 0;          // K/V slot uses so far (K and V each take one)
  uint32_t q_armed = 0;     // q_full phases armed so far
  uint32_t lu = 0;          // units processed by this CTA
  const uint32_t q_full = smem_u32(&bars->q_full), q_empty = smem_u32(&bars->q_empty);
  auto wait = [&](uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, lim));
  };
  Item item;
  for (; get_item(p, static_cast<int>(lu), item); ++lu) {
    const int bh = item.unit / p.n_pairs, pair = item.unit % p.n_pairs;
    const int q0a = pair * 2 * BM;
    const int nt = unit_tiles(p, item.unit);
    if (lu > 0 && !wait(q_empty, (lu - 1) & 1)) goto drain;
    if (elect_one()) {
      mbar_arrive_expect_tx(q_full, nt * C::TILE);
      for (int hf = 0; hf < C::NH; ++hf) {
        load_tile(p, p.tm_q, smem_u32(smem + C::OFF_Q + hf * kHalfBytes), q_full, hf, q0a, bh);
        if (nt == 2)
          load_tile(p, p.tm_q, smem_u32(smem + C::OFF_Q + C::TILE + hf * kHalfBytes), q_full, hf,
                    q0a + BM, bh);
      }
    }
    __syncwarp();
    ++q_armed;
    if (elect_one()) {
      // Warm L2 with the next item's query tiles. K/V tiles are not warmed: the
      // CTAs of one head read them within a few microseconds of each other, so
      // they mostly hit in L2, and the extra prefetch requests measured slower.
      Item nx;
      if (get_item(p, static_cast<int>(lu) + 1, nx)) {
        const int bhn = nx.unit / p.n_pairs, pn = nx.unit % p.n_pairs;
        for (int hf = 0; hf < C::NH; ++hf) {
          prefetch_tile(p, p.tm_q, hf, pn * 2 * BM, bhn);
          if (2 * pn + 1 < p.n_qtiles) prefetch_tile(p, p.tm_q, hf, pn * 2 * BM + BM, bhn);
        }
      }
    }
    __syncwarp();
    for (int j = item.kv0; j < item.kv1; ++j) {
      for (int kind = 0; kind < 2; ++kind, ++it) {
        const uint32_t slot = it % stages, ph = (it / stages) & 1;
        if (!wait(smem_u32(&bars->kv_empty[slot]), ph ^ 1)) goto drain;
        const uint32_t full = smem_u32(&bars->kv_full[slot]);
        const CUtensorMap *maps = kind == 0 ? p.tm_k : p.tm_v;
        if (elect_one()) {
          mbar_arrive_expect_tx(full, C::TILE);
          for (int hf = 0; hf < C::NH; ++hf)
            load_tile(p, maps, smem_u32(smem + C::OFF_KV + slot * C::TILE + hf * kHalfBytes), full,
                      hf, j * BN, bh);
        }
        __syncwarp();
      }
    }
  }
drain:
  // Every load this thread issued must land before the CTA releases its smem:
  // wait for the most recently armed phase of each barrier it armed.
  for (uint32_t s = 0; s < stages && s < it; ++s) {
    const uint32_t last = s + ((it - 1 - s) / stages) * stages;  // last use of slot s
    drain_phase(smem_u32(&bars->kv_full[s]), (last / stages) & 1, lim);
  }
  if (q_armed > 0) drain_phase(q_full, (q_armed - 1) & 1, lim);
}

// ------------------------------------------------------------------ MMA issuer
// Descriptors are built once per tile buffer; the k-th MMA of a tile only adds a
// constant to the start-address field (the low 14 bits hold address >> 4 and
// shared addresses stay below 256 KiB, so the add never carries out of it).
// This keeps the issuing lane's work per MMA to a couple of instructions.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t dcol, uint64_t qdesc, uint64_t kdesc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk / 4) * kHalfBytes + (kk % 4) * 32) >> 4);
    tc_mma_ss(dcol, qdesc + off, kdesc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t dcol, uint32_t pcol, uint64_t vdesc,
                                         uint32_t accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, 1);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    // V is the MN-major B operand: 16 key rows per MMA (2 KiB of the swizzled
    // tile); the next 64 columns of d sit one half (kHalfBytes, the LBO) further.
    tc_mma_ts(dcol, pcol + kk * 8, vdesc + static_cast<uint64_t>((kk * 2048) >> 4), idesc,
              (kk > 0 || accumulate) ? 1u : 0u);
  }
}

// Run by the whole MMA warp: the control flow and every descriptor stay
// warp-uniform, and one elected lane issues each group of tcgen05 operations
// (the same lane every time, as commits track the issuing thread's MMAs). Kept
// uniform, the per-MMA descriptor arithmetic stays off the issue path, so the
// issuer keeps the tensor pipe fed.
template <int D, bool SHARED>
__device__ void mma_role(const AttnParams &p, uint8_t *smem, Bars *bars, uint32_t tmem_in,
                         volatile int *abort_flag) {
  using C = Cfg<D, SHARED>;
  const uint64_t lim = p.wait_limit_ns;
  constexpr uint32_t stages = C::KV_STAGES;
  const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_in, 0);
  uint32_t it = 0, lu = 0;
  uint32_t pc[2] = {0, 0};
  const uint32_t q_full = smem_u32(&bars->q_full), q_empty = smem_u32(&bars->q_empty);
  auto kv_full = [&](uint32_t s) { return smem_u32(&bars->kv_full[s]); };
  auto kv_empty = [&](uint32_t s) { return smem_u32(&bars->kv_empty[s]); };
  auto wait = [&](uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, lim));
  };
  uint64_t qdesc[2];
#pragma unroll
  for (int t = 0; t < 2; ++t)
    qdesc[t] = smem_desc_sw128(smem_u32(smem + C::OFF_Q + t * C::TILE), 16, 1024);
  // Slot s of the K/V ring starts s * TILE bytes after slot 0: add (s * TILE) >> 4.
  const uint64_t kdesc0 = smem_desc_sw128(smem_u32(smem + C::OFF_KV), 16, 1024);
  const uint64_t vdesc0 = smem_desc_sw128(smem_u32(smem + C::OFF_KV), kHalfBytes, 1024);
  auto kdesc = [&](uint32_t s) { return kdesc0 + static_cast<uint64_t>(s * (C::TILE >> 4)); };
  auto vdesc = [&](uint32_t s) { return vdesc0 + static_cast<uint64_t>(s * (C::TILE >> 4)); };
  const uint32_t col_s[2] = {tmem + C::COL_S0, tmem + C::COL_S1};
  const uint32_t col_o[2] = {tmem + C::COL_O0, tmem + C::COL_O1};
  Item item;
  for (; get_item(p, static_cast<int>(lu), item); ++lu) {
    const int nk = item.kv1 - item.kv0;
    const int nt = unit_tiles(p, item.unit);   // the last tile's MMAs release K/V and Q
    if (!wait(q_full, lu & 1)) goto drain;
    {
      const uint32_t sk = it % stages;
      if (!wait(kv_full(sk), (it / stages) & 1)) goto drain;
      tc_fence_after();
      if (elect_one()) {
        for (int t = 0; t < nt; ++t) {
          issue_qk<D>(col_s[t], qdesc[t], kdesc(sk));
          tc_commit(smem_u32(&bars->s_full[t]));
        }
        tc_commit(kv_empty(sk));
        if (nk == 1) tc_commit(q_empty);
      }
      __syncwarp();
      ++it;
    }
    for (int j = 1; j < nk; ++j) {
      const uint32_t sv = it % stages, sk = (it + 1) % stages;
      if (!wait(kv_full(sv), (it / stages) & 1)) goto drain;
      for (int t = 0; t < nt; ++t) {
        if (!wait(smem_u32(&bars->p_full[t]), pc[t] & 1)) goto drain;
        ++pc[t];
        tc_fence_after();
        if (elect_one()) {
          issue_pv<D>(col_o[t], col_s[t], vdesc(sv), j > 1 ? 1u : 0u);
          if (t == nt - 1) tc_commit(kv_empty(sv));   // V(j-1) is free once the last PV is done
        }
        __syncwarp();
        // K(j) is waited for only after PV0 is issued, which never depends on it.
        if (t == 0) {
          if (!wait(kv_full(sk), ((it + 1) / stages) & 1)) goto drain;
          tc_fence_after();
        }
        if (elect_one()) {
          issue_qk<D>(col_s[t], qdesc[t], kdesc(sk));
          tc_commit(smem_u32(&bars->s_full[t]));
          if (t == nt - 1) {
            tc_commit(kv_empty(sk));
            if (j == nk - 1) tc_commit(q_empty);
          }
        }
        __syncwarp();
      }
      it += 2;
    }
    {
      const uint32_t sv = it % stages;
      if (!wait(kv_full(sv), (it / stages) & 1)) goto drain;
      for (int t = 0; t < nt; ++t) {
        if (!wait(smem_u32(&bars->p_full[t]), pc[t] & 1)) goto drain;
        ++pc[t];
        tc_fence_after();
        if (elect_one()) {
          issue_pv<D>(col_o[t], col_s[t], vdesc(sv), nk > 1 ? 1u : 0u);
          tc_commit(smem_u32(&bars->o_full[t]));
          if (t == nt - 1) tc_commit(kv_empty(sv));
          if (nt == 1) tc_commit(smem_u32(&bars->o_full[1]));   // group 1 sits this unit out
        }
        __syncwarp();
      }
      ++it;
    }
  }
drain:
  // All MMAs this warp issued must finish before Tensor Memory is released.
  if (elect_one()) tc_commit(smem_u32(&bars->drain));
  __syncwarp();
  drain_phase(smem_u32(&bars->drain), 0, lim);
}

// Issuers of the EARLY_QK schedule (d = 64). QK^T(j+1) of tile t goes into S_t
// as soon as the softmax has read S(j) (s_free), so the next scores are computed
// while the softmax works on the current ones; PV(j) of tile t reads P_t once
// P(j) is written (p_full) and completes pv_done, which the softmax waits for
// before it overwrites P_t or rescales O_t. QK^T and PV touch disjoint Tensor
// Memory columns and have no order between them, so each has its own warp: an
// issuing thread is held for about the run time of the MMAs it issues, and a
// satisfied barrier wait costs ~150 cycles, so one thread doing both leaves the
// tensor pipe idle during its waits; with two, one waits while the other's
// MMAs run. A commit tracks only its own thread's MMAs, so each barrier below
// is completed by the warp that issues the MMAs it stands for. The K/V ring
// keeps the order K0 V0 K1 V1 ...: the QK warp consumes the even uses, the PV
// warp the odd ones, each releasing its slot once both tiles' MMAs are done.
template <int D, bool SHARED>
__device__ void qk_issuer(const AttnParams &p, uint8_t *smem, Bars *bars, uint32_t tmem_in,
                          volatile int *abort_flag) {
  using C = Cfg<D, SHARED>;
  static_assert(C::EARLY_QK, "EARLY_QK schedule only");
  const uint64_t lim = p.wait_limit_ns;
  constexpr uint32_t stages = C::KV_STAGES;
  const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_in, 0);
  uint32_t base = 0, lu = 0;       // ring use of the unit's K0; items processed
  uint32_t fc[2] = {0, 0};         // s_free phases waited for, per tile
  bool used[2] = {false, false};   // S_t written before (its last scores must be read first)
  const uint32_t q_full = smem_u32(&bars->q_full), q_empty = smem_u32(&bars->q_empty);
  auto wait = [&](uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, lim));
  };
  uint64_t qdesc[2];
#pragma unroll
  for (int t = 0; t < 2; ++t)
    qdesc[t] = smem_desc_sw128(smem_u32(smem + C::OFF_Q + t * C::TILE), 16, 1024);
  const uint64_t kdesc0 = smem_desc_sw128(smem_u32(smem + C::OFF_KV), 16, 1024);
  auto kdesc = [&](uint32_t s) { return kdesc0 + static_cast<uint64_t>(s * (C::TILE >> 4)); };
  const uint32_t col_s[2] = {tmem + C::COL_S0, tmem + C::COL_S1};
  Item item;
  for (; get_item(p, static_cast<int>(lu), item); ++lu) {
    const int nk = item.kv1 - item.kv0;
    const int nt = unit_tiles(p, item.unit);
    if (!wait(q_full, lu & 1)) goto drain;
    for (int j = 0; j < nk; ++j) {
      const uint32_t use = base + 2 * j, sk = use % stages;
      if (!wait(smem_u32(&bars->kv_full[sk]), (use / stages) & 1)) goto drain;
      for (int t = 0; t < nt; ++t) {
        if (used[t]) {
          if (!wait(smem_u32(&bars->s_free[t]), fc[t] & 1)) goto drain;
          ++fc[t];
        }
        used[t] = true;
        tc_fence_after();
        if (elect_one()) {
          issue_qk<D>(col_s[t], qdesc[t], kdesc(sk));
          tc_commit(smem_u32(&bars->s_full[t]));
          if (t == nt - 1) {
            tc_commit(smem_u32(&bars->kv_empty[sk]));
            if (j == nk - 1) tc_commit(q_empty);
          }
        }
        __syncwarp();
      }
    }
    base += 2 * nk;
  }
drain:
  // All MMAs this warp issued must finish before Tensor Memory is released.
  if (elect_one()) tc_commit(smem_u32(&bars->drain));
  __syncwarp();
  drain_phase(smem_u32(&bars->drain), 0, lim);
}

template <int D, bool SHARED>
__device__ void pv_issuer(const AttnParams &p, uint8_t *smem, Bars *bars, uint32_t tmem_in,
                          volatile int *abort_flag) {
  using C = Cfg<D, SHARED>;
  static_assert(C::EARLY_QK, "EARLY_QK schedule only");
  const uint64_t lim = p.wait_limit_ns;
  constexpr uint32_t stages = C::KV_STAGES;
  const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_in, 0);
  uint32_t base = 0, lu = 0;
  uint32_t pc[2] = {0, 0};
  auto wait = [&](uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, lim));
  };
  const uint64_t vdesc0 = smem_desc_sw128(smem_u32(smem + C::OFF_KV), kHalfBytes, 1024);
  auto vdesc = [&](uint32_t s) { return vdesc0 + static_cast<uint64_t>(s * (C::TILE >> 4)); };
  const uint32_t col_o[2] = {tmem + C::COL_O0, tmem + C::COL_O1};
  const uint32_t col_p[2] = {tmem + C::COL_P0, tmem + C::COL_P1};
  Item item;
  for (; get_item(p, static_cast<int>(lu), item); ++lu) {
    const int nk = item.kv1 - item.kv0;
    const int nt = unit_tiles(p, item.unit);
    for (int j = 0; j < nk; ++j) {
      const bool last = j == nk - 1;
      const uint32_t use = base + 2 * j + 1, sv = use % stages;
      if (!wait(smem_u32(&bars->kv_full[sv]), (use / stages) & 1)) goto drain;
      for (int t = 0; t < nt; ++t) {
        if (!wait(smem_u32(&bars->p_full[t]), pc[t] & 1)) goto drain;
        ++pc[t];
        tc_fence_after();
        if (elect_one()) {
          issue_pv<D>(col_o[t], col_p[t], vdesc(sv), j > 0 ? 1u : 0u);
          tc_commit(smem_u32(last ? &bars->o_full[t] : &bars->pv_done[t]));
          if (t == nt - 1) tc_commit(smem_u32(&bars->kv_empty[sv]));
          if (last && nt == 1) tc_commit(smem_u32(&bars->o_full[1]));   // group 1 sits this unit out
        }
        __syncwarp();
      }
    }
    base += 2 * nk;
  }
drain:
  if (elect_one()) tc_commit(smem_u32(&bars->drain));
  __syncwarp();
  drain_phase(smem_u32(&bars->drain), 0, lim);
}

// ------------------------------------------------------------------ softmax / epilogue
// Records an output tile's store-issue span when the caller asked for spans.
__device__ __forceinline__ void record_span(const AttnParams &p, int bh, int q0, uint64_t t0,
                                            uint64_t t1) {
  if (p.spans) {
    const long long tile = static_cast<long long>(bh) * p.n_qtiles + q0 / BM;
    p.spans[2 * tile] = t0;
    p.spans[2 * tile + 1] = t1;
  }
}

// One of the warps that store a tile's rows: the span runs from the earliest
// first issue to the latest release over all of them (they may sit in different
// CTAs when the tile was cut into pieces). The entries start at zero and timer
// values are positive, so the first warp's start replaces the zero and every
// later one keeps the minimum.
__device__ __forceinline__ void record_span_part(const AttnParams &p, int bh, int qtile,
                                                 uint64_t t0, uint64_t t1) {
  const long long tile = static_cast<long long>(bh) * p.n_qtiles + qtile;
  unsigned long long *s = p.spans + 2 * tile;
  const unsigned long long seen = atomicCAS(s, 0ull, static_cast<unsigned long long>(t0));
  if (seen != 0ull && t0 < seen) atomicMin(s, static_cast<unsigned long long>(t0));
  atomicMax(s + 1, static_cast<unsigned long long>(t1));
}

// One 16-row slab of a staged tile (rows q0 + 16s ... of head unit bh) to its
// destination: TMA bulk stores of the slab's 64-column halves.
template <int D>
__device__ __forceinline__ void issue_slab(const AttnParams &p, const uint8_t *stg, int bh, int q0,
                                           int s) {
  constexpr int NH = D / 64;
  const int n0 = q0 + s * kSlabRows;
  const CUtensorMap *m;
  int x0, y;
  if (p.shard_mode == 0) {
    m = &p.tm_out[0];
    x0 = 0;
    y = bh * p.N + n0;
  } else {
    const int b = bh / p.H, h = bh - b * p.H;
    const int sh = n0 / p.rows_per_shard;   // a 16-row slab never straddles two shards
    const int i0 = n0 - sh * p.rows_per_shard;
    m = &p.tm_out[sh];
    x0 = (p.h0 + h) * D;
    y = b * p.rows_per_shard + i0;
  }
#pragma unroll
  for (int hf = 0; hf < NH; ++hf)
    tma_store_2d(m, smem_u32(stg + (s * NH + hf) * (kSlabRows * 128)), x0 + hf * 64, y);
}

// Slab s of a tile (rows q0 + 16s ...) from a one-slab shared buffer.
template <int D>
__device__ __forceinline__ void issue_slab_from(const AttnParams &p, const uint8_t *src, int bh,
                                                int q0, int s) {
  constexpr int NH = D / 64;
  const int n0 = q0 + s * kSlabRows;
  const CUtensorMap *m;
  int x0, y;
  if (p.shard_mode == 0) {
    m = &p.tm_out[0];
    x0 = 0;
    y = bh * p.N + n0;
  } else {
    const int b = bh / p.H, h = bh - b * p.H;
    const int sh = n0 / p.rows_per_shard;
    const int i0 = n0 - sh * p.rows_per_shard;
    m = &p.tm_out[sh];
    x0 = (p.h0 + h) * D;
    y = b * p.rows_per_shard + i0;
  }
#pragma unroll
  for (int hf = 0; hf < NH; ++hf)
    tma_store_2d(m, smem_u32(src + hf * (kSlabRows * 128)), x0 + hf * 64, y);
}

// Issues up to `count` pending slabs of the group's staged tile (deferred bursts).
template <int D>
__device__ __forceinline__ void issue_slabs(const AttnParams &p, const uint8_t *stg,
                                            StoreState &ss, int count) {
  int issued = 0;
  if (ss.next == 0 && count > 0 && p.spans) ss.t0 = globaltimer_ns();
  while (ss.next < NSLAB && issued < count) {
    issue_slab<D>(p, stg, ss.bh, ss.q0, ss.next);
    ++ss.next;
    ++issued;
  }
  if (issued) {
    bulk_commit();
    if (ss.next == NSLAB) record_span(p, ss.bh, ss.q0, ss.t0, globaltimer_ns());
  }
}

// Writes 32 output columns (chunk c) of one row, scaled by inv_l and rounded to
// bf16, into the 128B-swizzled staging tile (slab-major, 64-column halves).
template <int D>
__device__ __forceinline__ void stage_chunk(uint8_t *stg, int row, int c, const uint32_t (&o)[32],
                                            float inv_l) {
  constexpr int NH = D / 64;
  const int slab = row / kSlabRows, r16 = row % kSlabRows;
  const int hf = (32 * c) / 64;
  uint8_t *box = stg + (slab * NH + hf) * (kSlabRows * 128) + r16 * 128;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int chunk = ((32 * c) % 64) / 8 + k;   // 16-byte chunk within the 128-byte row
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv_l, __uint_as_float(o[8 * k + 1]) * inv_l);
    v.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv_l, __uint_as_float(o[8 * k + 3]) * inv_l);
    v.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv_l, __uint_as_float(o[8 * k + 5]) * inv_l);
    v.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv_l, __uint_as_float(o[8 * k + 7]) * inv_l);
    *reinterpret_cast<uint4 *>(box + ((chunk ^ (r16 & 7)) * 16)) = v;
  }
}

// A warp stores the 32 staged rows it owns (slabs 2*wq and 2*wq + 1) and waits
// until the stores have read the staging tile (or, completion-coupled, until
// they are complete). Lane 0 only.
template <int D>
__device__ __forceinline__ void store_own_rows(const AttnParams &p, const uint8_t *stg, int bh,
                                               int qtile, int wq) {
  const uint64_t t0 = p.spans ? globaltimer_ns() : 0;
  issue_slab<D>(p, stg, bh, qtile * BM, 2 * wq);
  issue_slab<D>(p, stg, bh, qtile * BM, 2 * wq + 1);
  bulk_commit();
  if (p.coupled) {
    // Counterfactual: the issuer is released only when its stores are complete.
    bulk_wait_all();
  } else {
    bulk_wait_read_all();
  }
  if (p.spans) record_span_part(p, bh, qtile, t0, globaltimer_ns());
}

// Partial result of one (piece, query tile) in the workspace, fp32: output
// columns as float4 groups, [warp][col/4][lane][4] so that one warp instruction
// moves 512 contiguous bytes, then the running maxima [128] and row sums [128].
template <int D>
__device__ __forceinline__ float4 *part_o(float *blk, int wq, int lane, int c4) {
  return reinterpret_cast<float4 *>(blk) + (wq * (D / 4) + c4) * 32 + lane;
}

// End of one piece of a split unit, per warp (its 32 rows of query tile t).
// A piece that is not the last of its unit leaves its partial result
// (unnormalised O, running maximum m in the log2 domain, row sum l) in the
// workspace; the warp that completes the last piece of these rows merges all
// pieces by the same rescaling identity that the online softmax applies
// between KV tiles, leaving the merged unnormalised O in its Tensor Memory
// columns and the merged row sum in l, to be staged like a whole unit's.
// Returns true for that warp.
template <int D>
__device__ __forceinline__ bool finish_piece(const AttnParams &p, const Item &item, int t, int wq,
                                             int lane, int row, uint32_t tO, float m, float &l) {
  constexpr int BLK = (D + 2) * 128;   // floats of one (piece, tile) partial
  // The unit's pieces run on the consecutive CTAs whose ranges overlap it.
  const long long u0 =
      static_cast<long long>(item.unit - p.sk_waves * static_cast<int>(gridDim.x)) * p.n_kv;
  auto owner = [&](long long pos) {
    int c = static_cast<int>(pos * gridDim.x / p.sk_total);
    while (c + 1 < static_cast<int>(gridDim.x) && sk_start(p, c + 1) <= pos) ++c;
    while (c > 0 && sk_start(p, c) > pos) --c;
    return c;
  };
  const int c_first = owner(u0);
  const int S = owner(u0 + p.n_kv - 1) - c_first + 1;
  const int s_own = static_cast<int>(blockIdx.x) - c_first;
  // Piece s of the unit lives in CTA c_first + s's slot 1 (the unit starts in
  // the range of c_first, so it is that CTA's last item) or slot 0 (the first
  // item of every later CTA).
  auto part = [&](int k) {
    return p.ws_part + ((static_cast<size_t>(c_first + k) * 2 + (k == 0 ? 1 : 0)) * 2 + t) * BLK;
  };
  int *cnt = p.ws_count + (c_first * 2 + t) * 4 + wq;
  if (S > kMaxSplit) {   // the host plans at most kMaxSplit pieces per unit
    if (lane == 0) atomicExch(&g_status, kDevBadPlan);
    return false;
  }
  // Every other piece already counted (each counts after its partial is written
  // and fenced): this one is last and needs to write nothing. Only piece 0 (the
  // last item of its CTA's range, usually the last to finish) looks; the later
  // pieces run first in their CTAs' ranges.
  int last = 0;
  if (lane == 0 && s_own == 0) {
    int seen;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(seen) : "l"(cnt) : "memory");
    last = seen == S - 1;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) {
    float *own = part(s_own);
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(tO + 32 * c, o);
      tmem_wait_ld_regs(o);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        __stcg(part_o<D>(own, wq, lane, 8 * c + i),
               make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                           __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3])));
    }
    __stcg(own + D * 128 + row, m);
    __stcg(own + D * 128 + 128 + row, l);
    __threadfence();
    __syncwarp();
    if (lane == 0) last = atomicAdd(cnt, 1) == S - 1;
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return false;
    __threadfence();
  }
  if (lane == 0) *cnt = 0;   // every piece has arrived: ready for the next launch
  // Weights of the pieces relative to the common maximum. Every sum runs over
  // the pieces in order 0..S-1, so the result does not depend on which piece
  // finished last.
  float mk[kMaxSplit], fk[kMaxSplit];
  float mx = m;
#pragma unroll
  for (int k = 0; k < kMaxSplit; ++k) {
    mk[k] = -INFINITY;
    if (k < S) mk[k] = k == s_own ? m : __ldcg(part(k) + D * 128 + row);
    mx = fmaxf(mx, mk[k]);
  }
  float lsum = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxSplit; ++k) {
    fk[k] = 0.f;
    if (k < S) {
      fk[k] = ex2_approx(mk[k] - mx);
      lsum = fmaf(fk[k], k == s_own ? l : __ldcg(part(k) + D * 128 + 128 + row), lsum);
    }
  }
  // 32 columns of piece k: from Tensor Memory for this piece, else from the workspace.
  auto fetch = [&](int k, int c, float4 (&x)[8]) {
    if (k == s_own) {
      uint32_t o[32];
      tmem_ld32(tO + 32 * c, o);
      tmem_wait_ld_regs(o);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        x[i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                           __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
    } else if (k < S) {
      float *src = part(k);
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __ldcg(part_o<D>(src, wq, lane, 8 * c + i));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    // Two pieces' 32 columns in flight at a time.
#pragma unroll
    for (int k = 0; k < kMaxSplit; k += 2) {
      if (k >= S) break;
      float4 a[8], b[8];
      fetch(k, c, a);
      fetch(k + 1, c, b);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc[4 * i + 0] = fmaf(fk[k], a[i].x, acc[4 * i + 0]);
        acc[4 * i + 1] = fmaf(fk[k], a[i].y, acc[4 * i + 1]);
        acc[4 * i + 2] = fmaf(fk[k], a[i].z, acc[4 * i + 2]);
        acc[4 * i + 3] = fmaf(fk[k], a[i].w, acc[4 * i + 3]);
        acc[4 * i + 0] = fmaf(fk[k + 1], b[i].x, acc[4 * i + 0]);
        acc[4 * i + 1] = fmaf(fk[k + 1], b[i].y, acc[4 * i + 1]);
        acc[4 * i + 2] = fmaf(fk[k + 1], b[i].z, acc[4 * i + 2]);
        acc[4 * i + 3] = fmaf(fk[k + 1], b[i].w, acc[4 * i + 3]);
      }
    }
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(acc[i]);
    tmem_st32(tO + 32 * c, r);
  }
  tmem_wait_st();
  l = lsum;
  return true;
}

// Running maxima over 64 raw scores (two 32-register chunks) in 8 independent
// chains of 3-input max; `first` starts the chains.
__device__ __forceinline__ void row_max_part(const uint32_t (&a)[32], const uint32_t (&b)[32],
                                             float (&mp)[8], bool first) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float x = __uint_as_float(a[i]), y = __uint_as_float(a[i + 8]);
    mp[i] = first ? fmaxf(x, y) : max3(mp[i], x, y);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i)
    mp[i] = max3(mp[i], __uint_as_float(a[i + 16]), __uint_as_float(a[i + 24]));
#pragma unroll
  for (int i = 0; i < 8; ++i)
    mp[i] = max3(mp[i], __uint_as_float(b[i]), __uint_as_float(b[i + 8]));
#pragma unroll
  for (int i = 0; i < 8; ++i)
    mp[i] = max3(mp[i], __uint_as_float(b[i + 16]), __uint_as_float(b[i + 24]));
}

template <int D, bool SHARED>
__device__ void softmax_role(const AttnParams &p, uint8_t *smem, Bars *bars, uint32_t tmem,
                             volatile int *abort_flag) {
  using C = Cfg<D, SHARED>;
  const uint64_t lim = p.wait_limit_ns;
  const int t = threadIdx.x / 128;          // warp group = query tile of the unit
  const int wq = (threadIdx.x / 32) & 3;    // warp within the group = TMEM lane quarter
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;           // tile row owned by this thread
  const bool elected = (threadIdx.x & 127) == 0;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tmem + lane_base + (t == 0 ? C::COL_S0 : C::COL_S1);
  const uint32_t tO = tmem + lane_base + (t == 0 ? C::COL_O0 : C::COL_O1);
  const uint32_t tP = tmem + lane_base + (t == 0 ? C::COL_P0 : C::COL_P1);
  const uint32_t s_full = smem_u32(&bars->s_full[t]), p_full = smem_u32(&bars->p_full[t]);
  const uint32_t s_free = smem_u32(&bars->s_free[t]), pv_done = smem_u32(&bars->pv_done[t]);
  const uint32_t o_full = smem_u32(&bars->o_full[t]), wg_sync = smem_u32(&bars->wg_sync[t]);
  uint8_t *stg = smem + C::OFF_KV + (SHARED ? C::NREG - 1 : C::NREG - 2 + t) * C::TILE;
  const float scale = p.scale_log2;
  uint32_t sc = 0, wgc = 0, lu = 0, pvc = 0;
  StoreState &ss = bars->store[t];
  if (elected) ss = StoreState{0, 0, NSLAB, 0, 0};

  Item item;
  for (; get_item(p, static_cast<int>(lu), item); ++lu) {
    const int bh = item.unit / p.n_pairs, pair = item.unit % p.n_pairs;
    const int qtile = 2 * pair + t;
    // A unit with one query tile leaves group 1 nothing to compute: the issuer
    // runs no MMA for it and only completes the group's o_full phase (so the
    // phases stay one per item), which the group consumes and moves on.
    if (t >= unit_tiles(p, item.unit)) {
      if (!__all_sync(0xffffffffu, wait_phase(o_full, lu & 1, abort_flag, lim))) goto teardown;
      continue;
    }
    const int nk = item.kv1 - item.kv0;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < nk; ++j) {
      bool ok = wait_phase(s_full, sc & 1, abort_flag, lim);
      ++sc;
      if (!__all_sync(0xffffffffu, ok)) goto teardown;
      tc_fence_after();
      // S row in two halves: the max over the first half overlaps the load of
      // the second.
      uint32_t s[4][32];
      tmem_ld32(tS, s[0]);
      tmem_ld32(tS + 32, s[1]);
      tmem_wait_ld_regs(s[0]);
      tmem_wait_ld_regs(s[1]);
      tmem_ld32(tS + 64, s[2]);
      tmem_ld32(tS + 96, s[3]);
      float mp[8];
      row_max_part(s[0], s[1], mp, true);
      tmem_wait_ld_regs(s[2]);
      tmem_wait_ld_regs(s[3]);
      if constexpr (C::EARLY_QK) {
        // S is in registers: the issuer may compute the next scores into it.
        tc_fence_before();
        mbar_arrive(s_free);
      }
      row_max_part(s[2], s[3], mp, false);
      const float mx = max3(max3(mp[0], mp[1], mp[2]), max3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
      const float m_new = fmaxf(m, mx * scale);
      // Conditional rescale: keep the running max unless it grew by more than
      // 2^kRescaleThreshold, so O is rescaled only on the rare large jumps.
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0) {
        m = m_new;
      } else {
        const bool need = m_new > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          rescale = true;
          if (need) {
            alpha = ex2_approx(m - m_new);
            m = m_new;
          }
        }
      }
      // p = 2^(s*scale - m): the argument on packed pairs, the row sum as four
      // scalar chains at d = 128 (there packing the two MUFU results for a packed
      // add costs more registers than it saves) and as packed pairs at d = 64, P
      // as bf16 pairs (over the S columns already read at d = 128).
      const float neg_m = -m;
      const uint64_t scale2 = f2_pack(scale, scale), negm2 = f2_pack(neg_m, neg_m);
      float lsum[4] = {0.f, 0.f, 0.f, 0.f};
      // With EARLY_QK (d = 64) the softmax is what bounds the kernel, and its
      // exponential phase is issue-bound: the row sum runs as two packed fp32x2
      // chains, one add per pair of columns instead of two (+7% measured at
      // N = 16384; the scalar chains are kept at d = 128, where they cost no time).
      constexpr bool PACKED_SUM = C::EARLY_QK;
      uint64_t l2[2] = {0ull, 0ull};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t x2 = f2_fma(
              f2_pack(__uint_as_float(s[c][2 * i]), __uint_as_float(s[c][2 * i + 1])), scale2, negm2);
          float p0, p1;
          if (PolyPairs<D>::take(i)) {
            f2_unpack(exp2_poly_x2(x2), p0, p1);
          } else {
            float x0, x1;
            f2_unpack(x2, x0, x1);
            p0 = ex2_approx(x0);
            p1 = ex2_approx(x1);
          }
          if constexpr (PACKED_SUM) {
            l2[i & 1] = f2_add(l2[i & 1], f2_pack(p0, p1));
          } else {
            lsum[i & 3] += p0 + p1;
          }
          pk[i] = pack_bf16x2(p0, p1);
        }
        if constexpr (C::EARLY_QK) {
          // P_t and O_t are read by PV(j-1) until pv_done completes: wait before
          // the first store (holding more chunks of P back measured slower).
          if (c == 0 && j > 0) {
            ok = wait_phase_inline(pv_done, pvc & 1, abort_flag, lim);
            ++pvc;
            if (!__all_sync(0xffffffffu, ok)) goto teardown;
            tc_fence_after();
          }
        }
        tmem_st16((C::EARLY_QK ? tP : tS) + 16 * c, pk);
      }
      if constexpr (PACKED_SUM) {
        const uint64_t ls2 = f2_add(l2[0], l2[1]);
        float a0, a1;
        f2_unpack(ls2, a0, a1);
        l = fmaf(l, alpha, a0 + a1);
      } else {
        l = fmaf(l, alpha, (lsum[0] + lsum[1]) + (lsum[2] + lsum[3]));
      }
      if (rescale) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_wait_ld_regs(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tO + 32 * c, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full);
      // Burst shaping: the previous tile's stores ride on this KV iteration.
      if (elected && ss.next < NSLAB) issue_slabs<D>(p, stg, ss, p.store_tile);

    }
    {
      // Epilogue: O_t is final once the last PV MMA completes.
      bool ok = wait_phase(o_full, lu & 1, abort_flag, lim);
      if (!__all_sync(0xffffffffu, ok)) goto teardown;
      tc_fence_after();
      // `mine`: this warp stages and stores its 32 rows of the tile now (always
      // for a whole unit; for a piece only in the warp that completes the rows,
      // after merging).
      bool mine = true;
      if (item.piece) mine = finish_piece<D>(p, item, t, wq, lane, row, tO, m, l);
      if constexpr (SHARED) {
        // store_tile 8: each warp stages and stores its 32 rows as two 16-row
        // slabs through a private one-slab buffer (its eighth of the staging
        // tile), so neither group waits for the other's stores, and only the
        // second slab's buffer read is still pending when the warp moves on.
        uint8_t *slab_buf = stg + (threadIdx.x / 32) * (kSlabRows * D * 2);
        if (mine) {
          const float inv_l = 1.f / l;
          const uint64_t t0 = p.spans ? globaltimer_ns() : 0;
          for (int hs = 0; hs < 2; ++hs) {
            if (lane == 0) bulk_wait_read_all();   // earlier stores have read the buffer
            __syncwarp();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + 32 * c, o);
              tmem_wait_ld_regs(o);
              if ((lane >> 4) == hs) stage_chunk<D>(slab_buf, lane & 15, c, o, inv_l);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              issue_slab_from<D>(p, slab_buf, bh, qtile * BM, 2 * wq + hs);
              bulk_commit();
            }
          }
          if (lane == 0) {
            // Counterfactual: the issuer is released only when its stores are complete.
            if (p.coupled) bulk_wait_all();
            if (p.spans) record_span_part(p, bh, qtile, t0, globaltimer_ns());
          }
        }
        tc_fence_before();
        __syncwarp();
      } else {
        // store_tile < 8: each group keeps its own staging tile; its slabs go
        // out over the next unit's KV iterations (issue_slabs above).
        if (elected) {
          issue_slabs<D>(p, stg, ss, NSLAB);   // leftovers of the previous tile
          bulk_wait_read_all();                // staging buffer may be overwritten now
        }
        mbar_arrive(wg_sync);
        ok = wait_phase(wg_sync, wgc & 1, abort_flag, lim);
        ++wgc;
        if (!__all_sync(0xffffffffu, ok)) goto teardown;
        if (mine) {
          const float inv_l = 1.f / l;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld_regs(o);
            stage_chunk<D>(stg, row, c, o, inv_l);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        // A piece's rows, and the rows of a CTA's last item (no next unit's KV
        // iterations to ride on), are stored at once by their owner warps.
        Item nx;
        const bool at_once = item.piece || !get_item(p, static_cast<int>(lu) + 1, nx);
        if (at_once && mine && lane == 0) store_own_rows<D>(p, stg, bh, qtile, wq);
        __syncwarp();
        mbar_arrive(wg_sync);
        ok = wait_phase(wg_sync, wgc & 1, abort_flag, lim);
        ++wgc;
        if (!__all_sync(0xffffffffu, ok)) goto teardown;
        if (elected && !at_once) ss = StoreState{bh, qtile * BM, 0, 0, 0};
      }
    }
  }
  if (elected) issue_slabs<D>(p, stg, ss, NSLAB);
teardown:
  if (lane == 0) bulk_wait_all();   // every thread that issued bulk stores
}

template <int D, bool SHARED>
__global__ void __launch_bounds__((Cfg<D, SHARED>::THREADS), 1)
    attn_kernel(const __grid_constant__ AttnParams p) {
  using C = Cfg<D, SHARED>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  Bars *bars = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
  volatile int *abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q_empty), 1);
    for (int s = 0; s < C::MAX_STAGES; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 1);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bars->s_full[t]), 1);
      mbar_init(smem_u32(&bars->p_full[t]), 128);
      mbar_init(smem_u32(&bars->o_full[t]), 1);
      mbar_init(smem_u32(&bars->s_free[t]), 128);
      mbar_init(smem_u32(&bars->pv_done[t]), 1);
      mbar_init(smem_u32(&bars->wg_sync[t]), 128);
    }
    mbar_init(smem_u32(&bars->drain), C::EARLY_QK ? 2 : 1);   // one commit per issuing warp
    bars->abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&p.tm_q[0]);
    tma_prefetch_desc(&p.tm_k[0]);
    tma_prefetch_desc(&p.tm_v[0]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == kLoadWarp) {
    load_role<D, SHARED>(p, smem, bars, abort_flag);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if constexpr (C::EARLY_QK)
      qk_issuer<D, SHARED>(p, smem, bars, tmem, abort_flag);
    else
      mma_role<D, SHARED>(p, smem, bars, tmem, abort_flag);
    __syncwarp();
  } else if (warp == kPvWarp) {
    if constexpr (C::EARLY_QK) pv_issuer<D, SHARED>(p, smem, bars, tmem, abort_flag);
    __syncwarp();
  } else {
    softmax_role<D, SHARED>(p, smem, bars, tmem, abort_flag);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

#include "attn_wide.cuh"

__global__ void wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nothing ever arrives on `bar`: the wait must run out and record a timeout.
    wait_phase(smem_u32(&bar), 0, &abort_flag, limit_ns);
  }
  __syncthreads();
}

// Element i: out_poly[i] = the kernel's polynomial 2^x[i], out_mufu[i] = ex2.approx.ftz(x[i]).
__global__ void exp2_selftest_kernel(const float *x, float *out_poly, float *out_mufu, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float a = x[i], b = i + 1 < n ? x[i + 1] : 0.f;
  float p0, p1;
  f2_unpack(exp2_poly_x2(f2_pack(a, b)), p0, p1);
  out_poly[i] = p0;
  out_mufu[i] = ex2_approx(a);
  if (i + 1 < n) {
    out_poly[i + 1] = p1;
    out_mufu[i + 1] = ex2_approx(b);
  }
}

}  // namespace

cudaError_t launch_exp2_selftest(const float *x, float *out_poly, float *out_mufu, int n,
                                 cudaStream_t s) {
  const int pairs = (n + 1) / 2;
  exp2_selftest_kernel<<<(pairs + 255) / 256, 256, 0, s>>>(x, out_poly, out_mufu, n);
  return cudaGetLastError();
}

int attn_smem_bytes(int d) {
  if (d == 256) return wide::Cfg256::SMEM;
  return d == 128 ? Cfg<128, false>::SMEM : Cfg<64, false>::SMEM;
}

int wide_keys_per_step(int) { return wide::Cfg256::BNW; }
int wide_ctas_per_sm(int) { return wide::Cfg256::CTAS; }

template <class C>
static cudaError_t launch_wide(const AttnParams &p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(wide::attn_wide_kernel<C>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  wide::attn_wide_kernel<C><<<grid, wide::kThreadsW, C::SMEM, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn_wide(const AttnParams &p, int d, int grid, cudaStream_t s) {
  if (d == 256) return launch_wide<wide::Cfg256>(p, grid, s);
  return cudaErrorInvalidValue;
}

int attn_kv_stages(int d, bool shared_staging) {
  if (d == 128) return shared_staging ? Cfg<128, true>::KV_STAGES : Cfg<128, false>::KV_STAGES;
  return shared_staging ? Cfg<64, true>::KV_STAGES : Cfg<64, false>::KV_STAGES;
}

template <int D, bool SHARED>
static cudaError_t launch_one(const AttnParams &p, int grid, cudaStream_t s) {
  constexpr int smem = Cfg<D, SHARED>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, SHARED>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  attn_kernel<D, SHARED><<<grid, Cfg<D, SHARED>::THREADS, smem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn(const AttnParams &p, int d, int grid, cudaStream_t s) {
  const bool shared = p.shared_staging != 0;
  if (d == 128) return shared ? launch_one<128, true>(p, grid, s) : launch_one<128, false>(p, grid, s);
  return shared ? launch_one<64, true>(p, grid, s) : launch_one<64, false>(p, grid, s);
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t read_and_clear_status(cudaStream_t s, int *out) {
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status, &zero, sizeof(int));
    if (e != cudaSuccess) return e;
  }
  *out = v;
  return cudaSuccess;
}

}  // namespace xs
