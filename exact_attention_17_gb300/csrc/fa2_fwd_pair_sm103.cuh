// FlashAttention-2 forward on a CTA pair: the two-SM form of the
// fifth-generation tensor core (tcgen05 cta_group::2), head dimension 128.
//
// It computes exactly what fa2_fwd_tc_kernel computes -- per query row,
// O_i = sum_j softmax_j(scale * q_i . k_j) v_j and LSE_i, over all keys or
// the keys j <= i -- with the same FlashAttention-2 steps (Q blocks outside,
// K/V blocks streamed inside, online softmax with lazy normalisation, the
// causal block skip and tail masks; see fa2_fwd_sm103.cuh for the pages'
// sections).  What changes is how the work maps onto the GPU:
//
//  * a cluster of two CTAs (rank 0, the leader, and rank 1, its peer) owns
//    512 query rows; each CTA holds two 128-row query sub-tiles, and "pair
//    sub-tile" s (rows [512u + 256s, +256)) is the leader's sub-tile s (its
//    first 128 rows) together with the peer's sub-tile s (the next 128);
//  * one thread of the leader issues every MMA for both SMs.  S = Q K^T and
//    O += P V run as M = 256 MMAs: each SM computes its own CTA's 128 rows
//    into its own TMEM from A operands in its own shared memory (Q) or TMEM
//    (P), while the B operand (K for S, V for P V) is split along N between
//    the two CTAs: each CTA loads and keeps only half of every K and V tile
//    (64 keys x 128 columns of K, 128 keys x 64 columns of V).  Per SM this
//    halves the K/V copies and the shared-memory reads of the B operands,
//    and halves the MMA instructions one thread must issue per unit of work;
//  * commits arrive on both CTAs' barriers at once (multicast); the peer's
//    copies complete on the peer's own barriers and a forwarding thread of
//    the peer (its otherwise idle MMA warp) arrives on the leader's barrier
//    of the same slot once they have, so the leader's issuer sees a slot
//    full only when both halves have landed; each softmax warp arrives on
//    the leader's p_ready barrier once its P is in TMEM;
//  * each CTA releases its own ring slots from its own softmax thread, as
//    in the one-CTA kernel, and stores its own rows of O and LSE;
//  * both CTAs allocate the pair's TMEM together, and free it together
//    after a cluster-wide barrier, so neither CTA exits while the other may
//    still signal it.
// The protocol is restated and model-checked in tests/test_pair_protocol.py.
#pragma once

#include "fa2_fwd_sm103.cuh"
#include "ptx_pair.cuh"

namespace fa2dev {

struct PairConfig {
  static constexpr int D = 128;
  static constexpr int kRowsPerPair = 512;                 // 2 CTAs x 2 sub-tiles x 128 rows
  static constexpr uint32_t kQBytes = 128 * D * 2;         // one 128-row Q sub-tile (32 KB)
  static constexpr uint32_t kHalfBytes = 64 * D * 2;       // half a K or V tile (16 KB)
  static constexpr uint32_t kKChunkBytes = 64 * 128;       // 64 key rows x 64 columns of K (8 KB)
  static constexpr uint32_t kQChunkBytes = 128 * 128;      // 128 rows x 64 columns of Q (16 KB)
  static constexpr int kStages = 8;                        // ring of K/V halves (K and V alternate)
  static constexpr uint32_t kColsO0 = 256;
  static constexpr uint32_t kColsO1 = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kSmemData = 2 * kQBytes + kStages * kHalfBytes;
  static constexpr uint32_t kSmemBytes = kSmemData + 1024 /*align*/ + 1024 /*barriers*/;
  static constexpr int kThreads = 384;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  // the epilogue stages a sub-tile's second fp32 round (128 rows x 64 columns,
  // 32 KB) in two consecutive ring slots
  static_assert(2 * kHalfBytes == 128 * 64 * 4, "epilogue staging in the ring");
};

// Work item of pair `pair_id`: query block u (512 rows), b*H + h and key range.
struct PairItem {
  int u, bh, split;
};

template <bool CAUSAL>
__device__ __forceinline__ PairItem decode_pair(int pair_id, const FwdParams& p, bool fast) {
  const int U = p.q_blocks;
  const int items = p.BH * p.num_splits;
  const int per_group = p.item_group * U;
  const int group = fast ? fast_div(pair_id, p.div_per_group) : pair_id / per_group;
  const int in_group = pair_id - group * per_group;
  const int g0 = group * p.item_group;
  const int g_items = min(p.item_group, items - g0);
  const int u_rank = (fast && g_items == p.item_group) ? fast_div(in_group, p.div_group) : in_group / g_items;
  const int item = g0 + (in_group - u_rank * g_items);
  PairItem it;
  it.bh = fast ? fast_div(item, p.div_splits) : item / p.num_splits;
  it.split = item - it.bh * p.num_splits;
  it.u = CAUSAL ? U - 1 - u_rank : u_rank;
  return it;
}

// K/V tiles pair sub-tile s of query block u visits in [t_begin, t_end).
template <bool CAUSAL>
__device__ __forceinline__ int pair_tiles_for(int u, int s, int Nq, int t_begin, int t_end) {
  const int first = u * PairConfig::kRowsPerPair + s * 256;
  if (first >= Nq) return 0;
  int stop = t_end;
  if (CAUSAL) {
    const int last = min(first + 255, Nq - 1);
    stop = min(stop, last / kKeysPerTile + 1);
  }
  return max(0, stop - t_begin);
}

__device__ __forceinline__ void raise_abort_pair(volatile int* abort, int* status, uint32_t peer_rank) {
  *abort = 1;
  st_cluster_u32(mapa_shared(smem_addr(const_cast<int*>(abort)), peer_rank), 1u);
  atomicOr(status, kDevErrTimeout);
}

// tm_k: K with 64-row boxes; tm_v: V (and tm_q: Q) with 128-row boxes; all
// 64 columns wide, 128-byte swizzle.  Launched as clusters of two CTAs.
template <bool CAUSAL, bool F16>
__global__ void __launch_bounds__(PairConfig::kThreads, 1)
    fa2_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  using Cfg = PairConfig;
  using Shape = FwdShape<2>;
  constexpr int D = Cfg::D;
  constexpr int kWarpProducer = 8;
  constexpr int kWarpMma = 9;
  constexpr int STAGES = Cfg::kStages;
  constexpr uint32_t QB = Cfg::kQBytes;
  constexpr uint32_t HB = Cfg::kHalfBytes;
  constexpr uint16_t kBoth = 0x3;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;              // 2 sub-tiles
  uint8_t* sKV = smem + 2 * QB;    // STAGES halves
  auto* bars = reinterpret_cast<FwdBarriers<STAGES>*>(smem + Cfg::kSmemData);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;

  const PairItem it = decode_pair<CAUSAL>(static_cast<int>(blockIdx.x >> 1), p, true);
  const int u = it.u, bh = it.bh, split = it.split;
  const int all_tiles = (p.Nk + kKeysPerTile - 1) / kKeysPerTile;
  const int t_begin = split * p.tiles_per_split;
  const int t_end = min(all_tiles, t_begin + p.tiles_per_split);
  const int n0 = pair_tiles_for<CAUSAL>(u, 0, p.Nq, t_begin, t_end);
  const int n1 = pair_tiles_for<CAUSAL>(u, 1, p.Nq, t_begin, t_end);
  const int nmax = max(n0, n1);
  // this CTA's first row of sub-tile s: u*512 + s*256 + rank*128
  const int cta_row0 = u * Cfg::kRowsPerPair + static_cast<int>(rank) * kRowsPerSub;

  const uint32_t qbytes = (n0 > 0 ? QB : 0u) + (n1 > 0 ? QB : 0u);
  const int primed = min(STAGES, 2 * nmax);

  // One K or V half of load g (K_j for g = 2j, V_j for g = 2j + 1) into ring slot `slot`.
  auto load_half = [&](int g, int slot) {
    uint64_t* bar = &bars->kv_full[slot];
    bar_arrive_expect_tx(bar, HB);
    const int key0 = (t_begin + g / 2) * kKeysPerTile;
    uint8_t* dst = sKV + slot * HB;
    if ((g & 1) == 0) {
      // keys [key0 + 64 rank, +64), all 128 columns (two 64-column chunks)
      tma_load_3d(dst, &tm_k, bar, 0, key0 + static_cast<int>(rank) * 64, bh);
      tma_load_3d(dst + Cfg::kKChunkBytes, &tm_k, bar, 64, key0 + static_cast<int>(rank) * 64, bh);
    } else {
      // all 128 keys, columns [64 rank, +64)
      tma_load_3d(dst, &tm_v, bar, static_cast<int>(rank) * 64, key0, bh);
    }
  };

  if (warp == kWarpProducer && lane == 0) {
    // The leader's full barriers take two arrivals: its own (with the bytes
    // of its half) and the peer's forwarded one.
    bar_init(&bars->q_full, leader ? 2 : 1);
    for (int s = 0; s < STAGES; ++s) {
      bar_init(&bars->kv_full[s], leader ? 2 : 1);
      bar_init(&bars->kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      bar_init(&bars->s_full[i], 1);
      bar_init(&bars->p_ready[i], 8);   // the 4 softmax warps of each CTA
      bar_init(&bars->o_done[i], 1);
      bar_init(&bars->staged[i], kRowsPerSub);
      bar_init(&bars->stage_free[i], 1);
    }
    bar_init(&bars->mma_drain, 1);
    bars->abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
    // this CTA's own copies complete on its own barriers: they may start
    // before the cluster-wide synchronisation
    if (qbytes) {
      bar_arrive_expect_tx(&bars->q_full, qbytes);
      for (int s = 0; s < 2; ++s) {
        if ((s == 0 ? n0 : n1) == 0) continue;
        for (int c = 0; c < 2; ++c)
          tma_load_3d(sQ + s * QB + c * Cfg::kQChunkBytes, &tm_q, &bars->q_full, c * 64, cta_row0 + s * 256, bh);
      }
    }
    for (int g = 0; g < primed; ++g) load_half(g, g);
    // the CTA one wave later reads a Q block nobody has touched yet
    const unsigned later = blockIdx.x + p.wave;
    if (later < gridDim.x) {
      const PairItem it2 = decode_pair<CAUSAL>(static_cast<int>(later >> 1), p, false);
      const int row2 = it2.u * Cfg::kRowsPerPair + static_cast<int>(rank) * kRowsPerSub;
      for (int s = 0; s < 2; ++s)
        if (row2 + s * 256 < p.Nq)
          for (int c = 0; c < 2; ++c) tma_prefetch_l2_3d(&tm_q, c * 64, row2 + s * 256, it2.bh);
    }
  }
  if (warp == kWarpMma) {
    // one warp of each CTA of the pair allocates the pair's TMEM together
    tmem_alloc_pair(&bars->tmem_base, Cfg::kTmemCols);
    tmem_relinquish_pair();
    tc_fence_before_sync();
  }
  // Both CTAs' barriers are initialised before any thread signals the other CTA.
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= kWarpProducer) {
    regs_decrease<Shape::kProducer>();
    if (warp == kWarpProducer) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      if (lane == 0) {
        int issued = primed;
        bool ok = true;
        for (int g = primed; g < 2 * nmax && ok; ++g) {
          const int slot = g % STAGES;
          const int lap = g / STAGES;
          if (!wait_bar(&bars->kv_empty[slot], (lap - 1) & 1, abort, p.timeout_ns)) {
            raise_abort_pair(abort, p.status, rank ^ 1u);
            ok = false;
            break;
          }
          load_half(g, slot);
          ++issued;
        }
        // Every copy this CTA started must have landed before it exits; only
        // the last STAGES can still be in flight.  (The leader's barriers
        // also count the peer's forwarded arrivals.)
        volatile int never = 0;
        if (qbytes) wait_bar_cl(&bars->q_full, 0, &never, p.timeout_ns);
        for (int k = max(0, issued - STAGES); k < issued; ++k)
          wait_bar_cl(&bars->kv_full[k % STAGES], (k / STAGES) & 1, &never, p.timeout_ns);
      }
    } else if (warp == kWarpMma && !leader) {
      // ------------------------------------------------------------ forwarder (peer)
      // Once one of this CTA's copies has landed, arrive on the leader's
      // barrier of the same slot.
      if (lane == 0 && nmax > 0) {
        bool ok = wait_bar(&bars->q_full, 0, abort, p.timeout_ns);
        if (ok) bar_arrive_cluster(mapa_shared(smem_addr(&bars->q_full), 0));
        for (int g = 0; g < 2 * nmax && ok; ++g) {
          const int slot = g % STAGES;
          if (!wait_bar(&bars->kv_full[slot], (g / STAGES) & 1, abort, p.timeout_ns)) {
            ok = false;
            break;
          }
          bar_arrive_cluster(mapa_shared(smem_addr(&bars->kv_full[slot]), 0));
        }
        if (!ok) raise_abort_pair(abort, p.status, 0u);
        // The leader's last commit (the drain) must have reached this CTA
        // before the pair's teardown.
        volatile int never = 0;
        wait_bar(&bars->mma_drain, 0, &never, p.timeout_ns);
      }
    } else if (warp == kWarpMma) {
      // ------------------------------------------------------------ MMA issuer (leader)
      if (lane == 0 && nmax > 0) {
        constexpr uint32_t kIdescS = idesc_f32acc(256, kKeysPerTile, false, false, F16);
        constexpr uint32_t kIdescO = idesc_f32acc(256, D, false, true, F16);
        const uint32_t sQaddr = smem_addr(sQ);
        const uint32_t sKVaddr = smem_addr(sKV);

        // S_sub = Q_sub K^T into S buffer `sub`: K-major A (128 rows per CTA,
        // 16 KB per 64-column chunk) and B (64 keys per CTA, 8 KB per chunk);
        // K = 128 in steps of 16 (32 bytes inside a swizzle atom, then the
        // next chunk).
        auto issue_s = [&](int sub, int slot) {
          uint64_t da = sdesc_sw128(sQaddr + sub * QB, 16, 1024);
          uint64_t db = sdesc_sw128(sKVaddr + slot * HB, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            mma_ss_pair(tmem + sub * 128, da, db, kIdescS, kk > 0 ? 1u : 0u);
            da += ((kk & 3) == 3 ? Cfg::kQChunkBytes - 3 * 32 : 32) >> 4;
            db += ((kk & 3) == 3 ? Cfg::kKChunkBytes - 3 * 32 : 32) >> 4;
            asm volatile("" : "+l"(da), "+l"(db));
          }
        };
        // O_sub (+)= P_sub V: P from TMEM, V MN-major (64 columns per CTA, one swizzle atom wide).
        auto issue_pv = [&](int sub, int slot, bool acc) {
          uint64_t dv = sdesc_sw128(sKVaddr + slot * HB, HB, 1024);
          const uint32_t o = tmem + (sub == 0 ? Cfg::kColsO0 : Cfg::kColsO1);
          const uint32_t a = tmem + sub * 128;
#pragma unroll
          for (int kk = 0; kk < kKeysPerTile / 16; ++kk) {
            mma_ts_pair(o, a + kk * 8, dv, kIdescO, (acc || kk > 0) ? 1u : 0u);
            dv += (16 * 128) >> 4;   // next 16 keys of V
            asm volatile("" : "+l"(dv));
          }
        };

        bool ok = wait_bar_cl(&bars->q_full, 0, abort, p.timeout_ns) &&
                  wait_bar_cl(&bars->kv_full[0], 0, abort, p.timeout_ns);
        if (ok) {
          tc_fence_after_sync();
          if (n0 > 0) { issue_s(0, 0); mma_commit_pair(&bars->s_full[0], kBoth); }
          if (n1 > 0) { issue_s(1, 0); mma_commit_pair(&bars->s_full[1], kBoth); }
        }
        for (int j = 0; j < nmax && ok; ++j) {
          const int iv = 2 * j + 1, ik = 2 * j + 2;
          const int slot_v = iv % STAGES, slot_k = ik % STAGES;
          const bool next = j + 1 < nmax;
          // V_j, P_0(j) and K_(j+1) in one wait (a phase not needed is
          // replaced by a repeat of V_j's)
          uint64_t* bv = &bars->kv_full[slot_v];
          const uint32_t pv = (iv / STAGES) & 1;
          uint64_t* bp = j < n0 ? &bars->p_ready[0] : bv;
          const uint32_t pp = j < n0 ? (j & 1) : pv;
          uint64_t* bk = next ? &bars->kv_full[slot_k] : bv;
          const uint32_t pk = next ? (ik / STAGES) & 1 : pv;
          if (!wait_bar3_cl(bv, pv, bp, pp, bk, pk, abort, p.timeout_ns)) { ok = false; break; }
          tc_fence_after_sync();
          if (j < n0) {
            issue_pv(0, slot_v, j > 0);
            if (j + 1 == n0) mma_commit_pair(&bars->o_done[0], kBoth);
          }
          if (next && j + 1 < n0) { issue_s(0, slot_k); mma_commit_pair(&bars->s_full[0], kBoth); }
          if (j < n1) {
            if (!wait_bar_cl(&bars->p_ready[1], j & 1, abort, p.timeout_ns)) { ok = false; break; }
            tc_fence_after_sync();
            issue_pv(1, slot_v, j > 0);
            if (j + 1 == n1) mma_commit_pair(&bars->o_done[1], kBoth);
          }
          if (next && j + 1 < n1) { issue_s(1, slot_k); mma_commit_pair(&bars->s_full[1], kBoth); }
        }
        if (!ok) raise_abort_pair(abort, p.status, 1u);
        // Every MMA must be complete before TMEM is released; the drain
        // commit also tells the peer that no MMA is left.
        mma_commit_pair(&bars->mma_drain, kBoth);
        volatile int never = 0;
        wait_bar(&bars->mma_drain, 0, &never, p.timeout_ns);
      }
    }
  } else {
    regs_increase<Shape::kSoftmax>();
    // ------------------------------------------------------------ softmax (both CTAs)
    const int sub = warp >> 2;
    const int n_tiles = sub == 0 ? n0 : n1;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;                       // TMEM lane = row of the sub-tile
    const int sub_row0 = cta_row0 + sub * 256;
    const int qi = sub_row0 + row;                        // query index within (b, h)
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_bits + sub * 128;
    const uint32_t tO = tmem + lane_bits + (sub == 0 ? Cfg::kColsO0 : Cfg::kColsO1);
    const float sl2 = p.scale_log2;

    // One thread of the sub-tile that visits every key tile releases this
    // CTA's ring slots.
    const bool releaser = (threadIdx.x & (kRowsPerSub - 1)) == 0 && n_tiles == nmax && (sub == 1 || n1 == 0);
    float m = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      if (!__all_sync(0xffffffffu, wait_bar(&bars->s_full[sub], j & 1, abort, p.timeout_ns))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (releaser) {
        // S_sub(j) complete: K_j and V_(j-1) have no reader left on either SM
        if (j > 0) bar_arrive(&bars->kv_empty[(2 * j - 1) % STAGES]);
        bar_arrive(&bars->kv_empty[(2 * j) % STAGES]);
      }
      uint32_t s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(s[c]);

      const int key0 = (t_begin + j) * kKeysPerTile;
      const bool tail = key0 + kKeysPerTile > p.Nk;
      const bool diag = CAUSAL && key0 + kKeysPerTile - 1 > sub_row0;
      if (tail || diag) {
        const int lim = CAUSAL ? min(p.Nk, qi + 1) : p.Nk;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (key0 + c * 32 + e >= lim) s[c][e] = __float_as_uint(-INFINITY);
      }

#define FA2_S(f) __uint_as_float(s[(f) >> 5][(f) & 31])
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = FA2_S(k);
#pragma unroll
      for (int f = 8; f < 120; f += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = fmax3(mx8[k], FA2_S(f + k), FA2_S(f + 8 + k));
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(mx8[k], FA2_S(120 + k));
#undef FA2_S
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                             fmaxf(mx8[6], mx8[7]));
      const float m_cand = fmaxf(m, mx * sl2);
      const bool move = (j == 0) || (m_cand > m + kRescaleLog2);
      const float m_new = move ? m_cand : m;
      const float alpha = !move ? 1.f : (m == -INFINITY ? 0.f : ex2_approx(m - m_new));
      const float off = m_new == -INFINITY ? 0.f : m_new;

      const float2 c2 = make_float2(sl2, sl2);
      const float2 o2 = make_float2(-off, -off);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 t = __ffma2_rn(make_float2(__uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1])), c2, o2);
          const float2 pe = make_float2(ex2_approx(t.x), ex2_approx(t.y));
          acc[(e >> 1) & 3] = __fadd2_rn(acc[(e >> 1) & 3], pe);
          pk[c >> 1][(c & 1) * 16 + (e >> 1)] = pack_x2<F16>(pe.x, pe.y);
        }
        if (c == 1) tmem_st32(tS, pk[0]);
      }
      const float2 a01 = __fadd2_rn(acc[0], acc[1]);
      const float2 a23 = __fadd2_rn(acc[2], acc[3]);
      const float2 a = __fadd2_rn(a01, a23);
      const float rs = a.x + a.y;
      l = l * alpha + rs;
      m = m_new;
      tmem_st32(tS + 32, pk[1]);

      // correction of the running output (the wait for S(j) above already
      // follows P(j-1) V, which was issued before S(j))
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(tO + c * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      // (the leader's barrier address is formed here: kept live across the
      // loop it would cost the warpgroup a spill)
      if (lane == 0) bar_arrive_cluster(mapa_shared(smem_addr(&bars->p_ready[sub]), 0));
    }

    const bool store = qi < p.Nq;
    const size_t row_id = (static_cast<size_t>(p.num_splits > 1 ? split : 0) * p.BH + bh) * p.Nq + qi;
    float* orow = (p.num_splits > 1 ? p.O_part : p.O) + row_id * D;
    float* lse_out = (p.num_splits > 1 ? p.LSE_part : p.LSE) + row_id;
    const bool half_out = p.o_half != 0 && p.num_splits == 1;
    if (n_tiles == 0 && store && p.num_splits > 1) {
      for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      *lse_out = -INFINITY;
    }
    if (n_tiles > 0 && ok) {
      if (store) *lse_out = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (!__all_sync(0xffffffffu, wait_bar(&bars->o_done[sub], 0, abort, p.timeout_ns))) {
        ok = false;
      } else {
        tc_fence_after_sync();
        // As in the one-CTA kernel: O / l staged as 128-byte-swizzled boxes
        // and stored with TMA.  The first fp32 round goes to the sub-tile's
        // Q buffer; the second, for the sub-tile(s) whose last P V is the
        // pair's last MMA, to ring slots 2 sub and 2 sub + 1 once the drain
        // commit has arrived (no copy or MMA touches the ring then).
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const bool use_ring = n_tiles == nmax;
        const int zrow = (p.num_splits > 1 ? split * p.BH : 0) + bh;
        const bool first_thread = (threadIdx.x & (kRowsPerSub - 1)) == 0;
        // the peer's 128 rows of a pair sub-tile can all lie past Nq while
        // the leader's do not: such a CTA stages but stores nothing
        const bool any_row = sub_row0 < p.Nq;
        const int parts = half_out ? 1 : 2;
        for (int r = 0; r < parts && ok; ++r) {
          if (r > 0) {
            uint64_t* free_bar = use_ring ? &bars->mma_drain : &bars->stage_free[sub];
            if (!__all_sync(0xffffffffu, wait_bar(free_bar, 0, abort, p.timeout_ns))) {
              ok = false;
              break;
            }
            if (use_ring) tc_fence_after_sync();
          }
          uint8_t* stage = (r > 0 && use_ring) ? sKV + 2 * sub * HB : sQ + sub * QB;
          const uint32_t stage_row = smem_addr(stage) + row * 128;
#pragma unroll
          for (int b = 0; b < D / 64; ++b) {
            const uint32_t box = stage_row + b * 16384;
            if (!half_out) {
              uint32_t o[32];
              tmem_ld32(tO + r * (D / 2) + 32 * b, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                st_shared_v4(box + ((q ^ (row & 7)) << 4), __float_as_uint(__uint_as_float(o[4 * q]) * inv_l),
                             __float_as_uint(__uint_as_float(o[4 * q + 1]) * inv_l),
                             __float_as_uint(__uint_as_float(o[4 * q + 2]) * inv_l),
                             __float_as_uint(__uint_as_float(o[4 * q + 3]) * inv_l));
            } else {
              uint32_t o[2][32];
              tmem_ld32(tO + 64 * b, o[0]);
              tmem_ld32(tO + 64 * b + 32, o[1]);
              tmem_ld_wait(o[0]);
              tmem_ld_wait(o[1]);
              uint32_t h[32];
#pragma unroll
              for (int e = 0; e < 32; ++e)
                h[e] = pack_x2<F16>(__uint_as_float(o[e >> 4][(2 * e) & 31]) * inv_l,
                                    __uint_as_float(o[e >> 4][(2 * e + 1) & 31]) * inv_l);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                st_shared_v4(box + ((q ^ (row & 7)) << 4), h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
            }
          }
          fence_proxy_async_shared();
          bar_arrive(&bars->staged[sub]);
          if (first_thread) {
            if (!wait_bar(&bars->staged[sub], r & 1, abort, p.timeout_ns)) {
              ok = false;
            } else {
              if (any_row) {
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                  tma_store_3d(&tm_o, stage + b * 16384, half_out ? 64 * b : r * (D / 2) + 32 * b, sub_row0, zrow);
              }
              bulk_commit();
              if (r + 1 < parts && !use_ring) {
                bulk_wait_read();
                bar_arrive(&bars->stage_free[sub]);
              }
            }
          }
          ok = __all_sync(0xffffffffu, ok);
        }
        if (first_thread) bulk_wait_read();
      }
    }
    if (!ok) raise_abort_pair(abort, p.status, rank ^ 1u);
  }

  // ------------------------------------------------------------ teardown
  // Neither CTA exits, and the pair's TMEM is not freed, before both CTAs
  // are done with it and with signalling each other.
  tc_fence_before_sync();
  cluster_sync();
  if (warp == kWarpMma) {
    __syncwarp();   // the dealloc is warp-aligned; the cluster barrier is not
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, Cfg::kTmemCols);
  }
}

}  // namespace fa2dev
