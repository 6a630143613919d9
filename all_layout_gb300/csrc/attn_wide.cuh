// Head dimension 256: the same fused attention + shard store, one 128-row query
// tile per CTA with S double-buffered in Tensor Memory.
//
// Included by attn.cu inside its anonymous namespace (it uses that file's
// waits, loads, staging and slab stores).
//
// At d = 256 a tile needs S (128 columns) and O (256 columns) of Tensor Memory,
// so two tiles do not fit 512 columns as they do at d <= 128. Instead each CTA
// owns one query tile per unit and keeps two S buffers: the tensor pipe
// computes S(j+1) = Q K(j+1)^T while the softmax works on S(j), then O += P(j)
// V(j). Per KV step the tensor work is 2048 cycles (QK 1024, PV 1024) against
// about 1450 for one row's softmax chain, so the pipe need not wait for it.
//
// Roles (192 threads; one CTA per SM at d = 256):
//   warps 0-3  softmax, O rescale and epilogue (row r of the tile = TMEM lane r)
//   warp 4     Tensor Memory allocation and the MMA issuer
//   warp 5     TMA loader
// Tensor Memory (d = 256, 128-key steps): S0 [0,128)  S1 [128,256)  O [256,512);
// P(j) (bf16 pairs) overwrites the first half of S(j & 1).
// Shared memory: Q (64-column halves) | K/V ring of 64-column halves: K tiles in
// KDEP groups of NH slots, then V tiles in VDEP groups, each half released as
// soon as the MMAs reading it are done | four one-slab staging buffers, one per
// softmax warp | barriers.
//
// The kernel is written over its configuration (WCfg below). A d = 64
// configuration with 64-key steps (S0, S1 and O in 256 columns, two CTAs per
// SM, each with its own issuer) was parity-green but 2-3% slower than the
// two-tile kernel at d = 64 (N = 16384: 1088 against 1110 TFLOP/s; 32768: 1102
// against 1131), so only the d = 256 configuration is built.
//
// MMA order: QK(0); then per step j: QK(j+1) into S((j+1) & 1), PV(j). One
// thread's tcgen05 operations execute in order, so QK(j+2) cannot overwrite
// P(j) before PV(j) has read it.
namespace wide {

constexpr int kThreadsW = 192;
constexpr int kMmaWarpW = 4;
constexpr int kLoadWarpW = 5;

// D: head dimension; BNW: keys per KV step; KDEP, VDEP: K and V tiles in flight;
// PVN: columns of O per PV MMA; CTAS: CTAs per SM.
template <int D_, int BNW_, int KDEP_, int VDEP_, int PVN_, int CTAS_>
struct WCfg {
  static constexpr int D = D_, BNW = BNW_, KDEP = KDEP_, VDEP = VDEP_, CTAS = CTAS_;
  static constexpr int NH = D / 64;                  // 64-column halves of a row
  static constexpr int PV_N = PVN_;
  static constexpr int PV_HALVES = PV_N / 64;        // V halves one PV MMA reads
  static constexpr int HALF_Q = BM * 128;            // one half of the 128-row Q tile
  static constexpr int HALF_KV = BNW * 128;          // one half of a BNW-key K or V tile
  static constexpr int NKS = KDEP * NH, NVS = VDEP * NH, NSLOT = NKS + NVS;
  static constexpr int SLAB_BUF = kSlabRows * D * 2; // 16 rows x D columns bf16
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + NH * HALF_Q; // K slots, then V slots
  static constexpr int OFF_STG = OFF_KV + NSLOT * HALF_KV;
  static constexpr int OFF_BAR = OFF_STG + 4 * SLAB_BUF;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t COL_S = 0, COL_O = 2 * BNW;
  static constexpr uint32_t TMEM_COLS = 2 * BNW + D <= 256 ? 256 : 512;
  static_assert(2 * BNW + D <= 512 && BNW % 32 == 0 && D % PV_N == 0, "layout");
  static_assert(SMEM * CTAS <= 232448, "shared memory per SM");
  // Slot of half hf of the K (V) tile of global step gs, and the parity of that
  // slot's use by it.
  static __device__ __forceinline__ int kslot(uint32_t gs, int hf) { return (gs % KDEP) * NH + hf; }
  static __device__ __forceinline__ int vslot(uint32_t gs, int hf) {
    return NKS + (gs % VDEP) * NH + hf;
  }
  static __device__ __forceinline__ uint32_t kpar(uint32_t gs) { return (gs / KDEP) & 1; }
  static __device__ __forceinline__ uint32_t vpar(uint32_t gs) { return (gs / VDEP) & 1; }
};

// Head dimension 256: 128-key steps, one K and one V tile in flight (eight
// 16 KiB halves), 128-column PV MMAs (64: 1451, 128: 1633, 256: 1539 TFLOP/s
// at N = 16384), one CTA per SM.
using Cfg256 = WCfg<256, 128, 1, 1, 128, 1>;

template <int NSLOT>
struct WBars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[NSLOT], kv_empty[NSLOT];
  uint64_t s_full[2];   // S buffer b holds the scores of the step
  uint64_t p_full;      // 128 arrivals: P of the step is in Tensor Memory (O rescaled)
  uint64_t pv_done;     // one phase per PV: O holds the sum through that step
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(WBars<8>) <= 256, "barrier block too large");

// The k-th item of this CTA's work list (get_item: whole units strided over the
// persistent CTAs, or with a workspace, stream-K pieces of the last waves). A
// unit is one query tile: unit = (b*H + h) * n_qtiles + tile.
__device__ __forceinline__ bool wide_item(const AttnParams &p, int k, Item &it, int &bh, int &q0) {
  if (!get_item(p, k, it)) return false;
  bh = it.unit / p.n_qtiles;
  q0 = (it.unit - bh * p.n_qtiles) * BM;
  return true;
}

// Loads are issued in the order the tensor pipe frees their slots: the issue
// order QK(0), QK(1), PV(0), QK(2), PV(1), ... frees K(j) slots (QK(j) done)
// one phase before V(j-1) slots (PV(j-1) done), so the loader fills K one step
// ahead of V: K(0), K(1), V(0), K(2), V(1), ... Loading K(j+1) behind V(j) would
// leave QK(j+1) waiting a whole load latency every step.
template <class C>
__device__ void load_role_w(const AttnParams &p, uint8_t *smem, WBars<C::NSLOT> *bars,
                            volatile int *abort_flag) {
  constexpr int NH = C::NH;
  const uint64_t lim = p.wait_limit_ns;
  const uint32_t q_full = smem_u32(&bars->q_full), q_empty = smem_u32(&bars->q_empty);
  auto wait = [&](uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, wait_phase(bar, parity, abort_flag, lim));
  };
  uint32_t lu = 0, q_armed = 0;
  uint32_t k_loads = 0, v_loads = 0;   // K and V tiles loaded (global steps)
  uint32_t armed[C::NSLOT] = {};        // loads issued into each slot
  // The halves of K (kind 0) or V (kind 1) of key tile j, global step gs.
  auto load_kv = [&](int kind, int j, int bh, uint32_t gs) -> bool {
    for (int hf = 0; hf < NH; ++hf) {
      const int s = kind == 0 ? C::kslot(gs, hf) : C::vslot(gs, hf);
      const uint32_t par = kind == 0 ? C::kpar(gs) : C::vpar(gs);
      if (!wait(smem_u32(&bars->kv_empty[s]), par ^ 1)) return false;
      const uint32_t full = smem_u32(&bars->kv_full[s]);
      if (elect_one()) {
        mbar_arrive_expect_tx(full, C::HALF_KV);
        load_tile(p, kind == 0 ? p.tm_k : p.tm_v, smem_u32(smem + C::OFF_KV + s * C::HALF_KV),
                  full, hf, j * C::BNW, bh);
      }
      __syncwarp();
      ++armed[s];
    }
    return true;
  };
  Item item;
  int bh, q0;
  for (; wide_item(p, static_cast<int>(lu), item, bh, q0); ++lu) {
    if (lu > 0 && !wait(q_empty, (lu - 1) & 1)) goto drain;
    if (elect_one()) {
      mbar_arrive_expect_tx(q_full, NH * C::HALF_Q);
      for (int hf = 0; hf < NH; ++hf)
        load_tile(p, p.tm_q, smem_u32(smem + C::OFF_Q + hf * C::HALF_Q), q_full, hf, q0, bh);
    }
    __syncwarp();
    ++q_armed;
    if (!load_kv(0, item.kv0, bh, k_loads)) goto drain;
    ++k_loads;
    for (int j = item.kv0; j < item.kv1; ++j) {
      if (j + 1 < item.kv1) {
        if (!load_kv(0, j + 1, bh, k_loads)) goto drain;
        ++k_loads;
      }
      if (!load_kv(1, j, bh, v_loads)) goto drain;
      ++v_loads;
    }
  }
drain:
  // Every load issued must land before the CTA releases its shared memory:
  // wait for the last phase armed on each slot.
  for (int s = 0; s < C::NSLOT; ++s)
    if (armed[s]) drain_phase(smem_u32(&bars->kv_full[s]), (armed[s] - 1) & 1, lim);
  if (q_armed > 0) drain_phase(q_full, (q_armed - 1) & 1, lim);
}

// S(b) = Q K^T for global step gs, one 64-column half of d at a time; each
// K half is released when its four MMAs are done.
template <class C>
__device__ __forceinline__ bool issue_qk_w(WBars<C::NSLOT> *bars, uint32_t s_col, uint64_t qdesc,
                                           uint64_t kdesc0, uint32_t gs, volatile int *abort_flag,
                                           uint64_t lim) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, C::BNW, 0);
  for (int hf = 0; hf < C::NH; ++hf) {
    const int ks = C::kslot(gs, hf);
    if (!__all_sync(0xffffffffu,
                    wait_phase(smem_u32(&bars->kv_full[ks]), C::kpar(gs), abort_flag, lim)))
      return false;
    tc_fence_after();
    if (elect_one()) {
      const uint64_t kd = kdesc0 + static_cast<uint64_t>((ks * C::HALF_KV) >> 4);
      const uint64_t qd = qdesc + static_cast<uint64_t>((hf * C::HALF_Q) >> 4);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t off = static_cast<uint64_t>((kk * 32) >> 4);
        tc_mma_ss(s_col, qd + off, kd + off, idesc, (hf > 0 || kk > 0) ? 1u : 0u);
      }
      tc_commit(smem_u32(&bars->kv_empty[ks]));
    }
    __syncwarp();
  }
  if (elect_one()) tc_commit(smem_u32(&bars->s_full[gs & 1]));
  __syncwarp();
  return true;
}

// O (+)= P(gs) V(gs): per group of PV_N columns of O, one MMA per 16 keys (V as
// the MN-major B operand, its 64-column halves HALF_KV apart in consecutive
// slots); the group's V halves are released when its MMAs are done. A 128 x 64
// x 16 MMA took about 50 cycles against 32 of tensor work (the per-instruction
// cost dominates), so d = 256 uses 128-column MMAs.
template <class C>
__device__ __forceinline__ bool issue_pv_w(WBars<C::NSLOT> *bars, uint32_t o_col, uint32_t p_col,
                                           uint64_t vdesc0, uint32_t gs, bool first,
                                           volatile int *abort_flag, uint64_t lim) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, C::PV_N, 1);
  for (int grp = 0; grp < C::NH / C::PV_HALVES; ++grp) {
    for (int h = 0; h < C::PV_HALVES; ++h)
      if (!__all_sync(0xffffffffu,
                      wait_phase(smem_u32(&bars->kv_full[C::vslot(gs, grp * C::PV_HALVES + h)]),
                                 C::vpar(gs), abort_flag, lim)))
        return false;
    tc_fence_after();
    if (elect_one()) {
      const int vs = C::vslot(gs, grp * C::PV_HALVES);
      const uint64_t vd = vdesc0 + static_cast<uint64_t>((vs * C::HALF_KV) >> 4);
#pragma unroll
      for (int ks = 0; ks < C::BNW / 16; ++ks)
        tc_mma_ts(o_col + grp * C::PV_N, p_col + ks * 8,
                  vd + static_cast<uint64_t>((ks * 2048) >> 4), idesc, (!first || ks > 0) ? 1u : 0u);
      for (int h = 0; h < C::PV_HALVES; ++h)
        tc_commit(smem_u32(&bars->kv_empty[vs + h]));
    }
    __syncwarp();
  }
  if (elect_one()) tc_commit(smem_u32(&bars->pv_done));
  __syncwarp();
  return true;
}

template <class C>
__device__ void mma_role_w(const AttnParams &p, uint8_t *smem, WBars<C::NSLOT> *bars,
                           uint32_t tmem_in, volatile int *abort_flag) {
  const uint64_t lim = p.wait_limit_ns;
  const uint32_t tmem = __shfl_sync(0xffffffffu, tmem_in, 0);
  const uint32_t q_full = smem_u32(&bars->q_full), q_empty = smem_u32(&bars->q_empty);
  // Descriptors of the first Q half and of slot 0; a slot's start is added per MMA.
  const uint64_t qdesc = smem_desc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
  const uint64_t kdesc0 = smem_desc_sw128(smem_u32(smem + C::OFF_KV), 16, 1024);
  const uint64_t vdesc0 = smem_desc_sw128(smem_u32(smem + C::OFF_KV), C::HALF_KV, 1024);
  uint32_t lu = 0, g = 0;   // items and KV steps (global) issued
  Item item;
  int bh, q0;
  for (; wide_item(p, static_cast<int>(lu), item, bh, q0); ++lu) {
    const int nk = item.kv1 - item.kv0;
    if (!__all_sync(0xffffffffu, wait_phase(q_full, lu & 1, abort_flag, lim))) goto drain;
    if (!issue_qk_w<C>(bars, tmem + C::COL_S + (g & 1) * C::BNW, qdesc, kdesc0, g, abort_flag,
                       lim))
      goto drain;
    for (int j = 0; j < nk; ++j) {
      const uint32_t gs = g + j;
      if (j + 1 < nk) {
        if (!issue_qk_w<C>(bars, tmem + C::COL_S + ((gs + 1) & 1) * C::BNW, qdesc, kdesc0, gs + 1,
                           abort_flag, lim))
          goto drain;
      } else {
        if (elect_one()) tc_commit(q_empty);   // the unit's last QK has been issued
        __syncwarp();
      }
      if (!__all_sync(0xffffffffu, wait_phase(smem_u32(&bars->p_full), gs & 1, abort_flag, lim)))
        goto drain;
      tc_fence_after();
      if (!issue_pv_w<C>(bars, tmem + C::COL_O, tmem + C::COL_S + (gs & 1) * C::BNW, vdesc0, gs,
                         j == 0, abort_flag, lim))
        goto drain;
    }
    g += nk;
  }
drain:
  if (elect_one()) tc_commit(smem_u32(&bars->drain));
  __syncwarp();
  drain_phase(smem_u32(&bars->drain), 0, lim);
}

template <class C>
__device__ void softmax_role_w(const AttnParams &p, uint8_t *smem, WBars<C::NSLOT> *bars,
                               uint32_t tmem, volatile int *abort_flag) {
  constexpr int D = C::D;
  constexpr int NC = C::BNW / 32;            // 32-column chunks of an S row
  const uint64_t lim = p.wait_limit_ns;
  const int wq = threadIdx.x / 32;           // TMEM lane quarter
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tO = tmem + lane_base + C::COL_O;
  const uint32_t p_full = smem_u32(&bars->p_full), pv_done = smem_u32(&bars->pv_done);
  uint8_t *slab_buf = smem + C::OFF_STG + wq * C::SLAB_BUF;
  const float scale = p.scale_log2;
  uint32_t lu = 0, g = 0;
  Item item;
  int bh, q0;
  for (; wide_item(p, static_cast<int>(lu), item, bh, q0); ++lu) {
    const int nk = item.kv1 - item.kv0;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < nk; ++j) {
      const uint32_t gs = g + j;
      const uint32_t tS = tmem + lane_base + C::COL_S + (gs & 1) * C::BNW;
      if (!__all_sync(0xffffffffu, wait_phase(smem_u32(&bars->s_full[gs & 1]), (gs >> 1) & 1,
                                               abort_flag, lim)))
        goto teardown;
      tc_fence_after();
      uint32_t s[NC][32];
      float mp[8];
      tmem_ld32(tS, s[0]);
      tmem_ld32(tS + 32, s[1]);
      tmem_wait_ld_regs(s[0]);
      tmem_wait_ld_regs(s[1]);
      if constexpr (NC == 4) {
        tmem_ld32(tS + 64, s[2]);
        tmem_ld32(tS + 96, s[3]);
      }
      row_max_part(s[0], s[1], mp, true);
      if constexpr (NC == 4) {
        tmem_wait_ld_regs(s[2]);
        tmem_wait_ld_regs(s[3]);
        row_max_part(s[2], s[3], mp, false);
      }
      const float mx = max3(max3(mp[0], mp[1], mp[2]), max3(mp[3], mp[4], mp[5]), fmaxf(mp[6], mp[7]));
      const float m_new = fmaxf(m, mx * scale);
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
      const float neg_m = -m;
      const uint64_t scale2 = f2_pack(scale, scale), negm2 = f2_pack(neg_m, neg_m);
      // The row sum as one packed fp32x2 accumulator: one add per pair of
      // exponentials instead of two (measured +1.4% at N = 16384, +2.6% at 4096;
      // the two-tile kernel spills with it and keeps scalar sums).
      uint64_t lsum2 = f2_pack(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint64_t x2 = f2_fma(
              f2_pack(__uint_as_float(s[c][2 * i]), __uint_as_float(s[c][2 * i + 1])), scale2, negm2);
          float x0, x1;
          f2_unpack(x2, x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          lsum2 = f2_add(lsum2, f2_pack(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tS + 16 * c, pk);
      }
      float la, lb;
      f2_unpack(lsum2, la, lb);
      l = fmaf(l, alpha, la + lb);
      if (j > 0) {
        // Every step observes PV(gs - 1), the phase of pv_done before the one
        // this step's arrival enables. The wait is exact: S(gs) arrived after
        // PV(gs - 2) completed (the commit covers every earlier MMA) and PV(gs)
        // waits for this arrival, so the barrier is in phase gs - 1 or just
        // past it. PV(gs - 1) runs on the tensor pipe while this softmax works,
        // so it has normally completed by now. O holds the sum through step
        // j - 1 afterwards and may be rescaled.
        if (!__all_sync(0xffffffffu, wait_phase(pv_done, (gs - 1) & 1, abort_flag, lim)))
          goto teardown;
        if (rescale) {
          tc_fence_after();
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
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    {
      // Epilogue: O is final once the unit's last PV is done. The previous
      // phase was observed at the last step (or by the previous epilogue when
      // the unit has one step), so this wait is exact too.
      if (!__all_sync(0xffffffffu, wait_phase(pv_done, (g + nk - 1) & 1, abort_flag, lim)))
        goto teardown;
      tc_fence_after();
      // A piece of a cut unit: the warp that completes its rows merges the
      // pieces and stores them; the others leave their partial result.
      const int row = wq * 32 + lane;
      const bool mine = !item.piece || finish_piece<D>(p, item, 0, wq, lane, row, tO, m, l);
      const float inv_l = 1.f / l;
      const int qtile = q0 / BM;
      const uint64_t t0 = p.spans ? globaltimer_ns() : 0;
      for (int hs = 0; hs < 2 && mine; ++hs) {
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
          issue_slab_from<D>(p, slab_buf, bh, q0, 2 * wq + hs);
          bulk_commit();
        }
      }
      if (lane == 0 && mine) {
        if (p.coupled) bulk_wait_all();   // counterfactual: released once the stores complete
        if (p.spans) record_span_part(p, bh, qtile, t0, globaltimer_ns());
      }
      // The next unit's first PV overwrites O only after this warp's next
      // arrival on p_full, which follows these reads.
      tc_fence_before();
      __syncwarp();
    }
    g += nk;
  }
teardown:
  if (lane == 0) bulk_wait_all();
}

template <class C>
__global__ void __launch_bounds__(kThreadsW, C::CTAS) attn_wide_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  WBars<C::NSLOT> *bars = reinterpret_cast<WBars<C::NSLOT> *>(smem + C::OFF_BAR);
  volatile int *abort_flag = &bars->abort;
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q_empty), 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), 1);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars->s_full[0]), 1);
    mbar_init(smem_u32(&bars->s_full[1]), 1);
    mbar_init(smem_u32(&bars->p_full), 128);
    mbar_init(smem_u32(&bars->pv_done), 1);
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == kMmaWarpW) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == kLoadWarpW && lane == 0) {
    tma_prefetch_desc(&p.tm_q[0]);
    tma_prefetch_desc(&p.tm_k[0]);
    tma_prefetch_desc(&p.tm_v[0]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  if (warp == kLoadWarpW) {
    load_role_w<C>(p, smem, bars, abort_flag);
    __syncwarp();
  } else if (warp == kMmaWarpW) {
    mma_role_w<C>(p, smem, bars, tmem, abort_flag);
    __syncwarp();
  } else {
    softmax_role_w<C>(p, smem, bars, tmem, abort_flag);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarpW) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace wide
