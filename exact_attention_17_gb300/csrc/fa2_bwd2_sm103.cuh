// Backward pass with two query tiles in flight (sm_103a), head dimension 128.
//
// It computes what fa2_bwd_tc_kernel computes -- the chain rule of the
// attention definition for an upstream gradient dO (see fa2_bwd_sm103.cuh
// for the formulas and the pages' sections) -- with the same pre-pass
// (D_i, LSE_i log2(e), dQ zeroed).  What changes is the tiling:
//
//  * one CTA owns a block of 128 keys (K_j, V_j stay in shared memory) and
//    streams query tiles of 64 rows (Q_i, dO_i through a TMA ring);
//  * TMEM holds S^T and dP^T for two tiles (buffer t % 2, 64 columns each)
//    beside the dV and dK accumulators (128 columns each): 512 columns;
//  * the two elementwise warpgroups take the tiles in turn: warpgroup g owns
//    the tiles t with t % 2 == g (buffer g, its own barriers and its own dS
//    tile in shared memory), so one warpgroup's phases -- each bound by
//    fixed latencies (barrier waits, TMEM round trips) more than by its
//    arithmetic -- overlap the other's, and the tensor core computes the
//    scores of one tile while the other tile's dV, dK and dQ MMAs wait for
//    their operands;
//  * dQ is computed transposed, dQ^T(t) = K^T dS^T(t) (M = 128 head columns,
//    N = 64 queries, K = 128 keys), into tile t's S^T buffer once dV(t) has
//    read P^T(t) from it; the owning warpgroup reads it out (TMEM lane =
//    head column), stages it in tile t's ring slot as [query][column] boxes
//    and adds it into dQ with TMA bulk reductions;
//  * per tile one thread issues: dV(t) after P^T(t) is written, then
//    dP^T(t+1) and S^T(t+1) once Q/dO(t+1) have landed and dQ^T(t-1) has
//    been read out of buffer (t+1) % 2, then dK(t) and dQ^T(t) after dS^T(t).
// The protocol is model-checked in tests/test_backward2_protocol.py.
#pragma once

#include "fa2_bwd_sm103.cuh"

namespace fa2dev {

// 32 lanes x 16 consecutive 32-bit TMEM columns from this thread's 16 registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

struct Bwd2Config {
  static constexpr int D = 128;
  static constexpr int kQRows = 64;                          // query rows per tile
  static constexpr uint32_t kKVBytes = 128 * D * 2;          // K or V block (32 KB)
  static constexpr uint32_t kQBytes = kQRows * D * 2;        // Q or dO tile (16 KB)
  static constexpr uint32_t kKVChunk = 128 * 128;            // 64 columns of the 128-row block
  static constexpr uint32_t kQChunk = kQRows * 128;          // 64 columns of a 64-row tile
  static constexpr int kStages = 4;                          // Q/dO ring slots
  static constexpr uint32_t kDsBytes = 128 * kQRows * 2;     // a dS tile [128 keys][64 queries]
  static constexpr uint32_t kSmemData = 2 * kKVBytes + kStages * 2 * kQBytes + 2 * kDsBytes;
  static constexpr uint32_t kSmemBytes = kSmemData + 1024 /*align*/ + 1024 /*barriers*/;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static constexpr uint32_t kColS = 0;      // S^T buffer b at [64 b, 64 b + 64): P^T, then dQ^T
  static constexpr uint32_t kColDP = 128;   // dP^T buffer b at [128 + 64 b, +64): dS^T
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 384;
  // a tile's dQ staging (64 queries x 128 columns fp32) fills its ring slot:
  // queries 0-31 the Q half, 32-63 the dO half
  static_assert(32 * D * 4 == kQBytes, "dQ staging in the ring slot");
};

// Index g: the warpgroup (and TMEM buffer, and dS tile) of tiles t % 2 == g.
template <int STAGES>
struct alignas(8) Bwd2Barriers {
  uint64_t kv_full;
  uint64_t q_full[STAGES];
  uint64_t q_empty[STAGES];   // the owning warpgroup: the tile's dQ staging was read
  uint64_t dq_staged[2];      // the warpgroup's 128 threads wrote their dQ columns
  uint64_t s_full[2];         // S^T(t) and dP^T(t) complete
  uint64_t p_ready[2];
  uint64_t ds_ready[2];
  uint64_t dq_full[2];
  uint64_t dq_free[2];
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort;
};

// tm_q, tm_do: 64-row boxes; tm_k, tm_v: 128-row boxes (64 columns, 128-byte
// swizzle); tm_dq: fp32 dQ with 32 x 32 boxes (128-byte swizzle).
template <bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa2_bwd2_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using Cfg = Bwd2Config;
  constexpr int D = Cfg::D;
  constexpr int STAGES = Cfg::kStages;
  constexpr int QR = Cfg::kQRows;
  constexpr uint32_t KVB = Cfg::kKVBytes;
  constexpr uint32_t QB = Cfg::kQBytes;
  constexpr int kWarpProducer = 8;
  constexpr int kWarpMma = 9;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + KVB;
  uint8_t* sQ = smem + 2 * KVB;            // STAGES tiles
  uint8_t* sdO = sQ + STAGES * QB;         // STAGES tiles
  uint8_t* sdS = sdO + STAGES * QB;        // 2 tiles [128 keys][64 queries], MN-major B of dQ^T
  auto* bars = reinterpret_cast<Bwd2Barriers<STAGES>*>(smem + Cfg::kSmemData);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: (key block jb, b*H + h), grouped and ordered as in the
  // one-tile kernel.
  const int U = p.key_blocks;
  const int per_group = p.item_group * U;
  const int group = blockIdx.x / per_group;
  const int in_group = blockIdx.x - group * per_group;
  const int g0 = group * p.item_group;
  const int g_items = min(p.item_group, p.BH - g0);
  const int jb = in_group / g_items;
  const int bh = g0 + (in_group - jb * g_items);
  const int q_tiles = (p.Nq + QR - 1) / QR;
  const int i0 = CAUSAL ? jb * (128 / QR) : 0;   // first query tile with a query >= the first key
  const int n_tiles = max(0, q_tiles - i0);
  const int key0 = jb * 128;

  if (threadIdx.x == 0) {
    bar_init(&bars->kv_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      bar_init(&bars->q_full[s], 1);
      bar_init(&bars->q_empty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      bar_init(&bars->dq_staged[g], 128);
      bar_init(&bars->s_full[g], 1);
      bar_init(&bars->p_ready[g], 128);
      bar_init(&bars->ds_ready[g], 128);
      bar_init(&bars->dq_full[g], 1);
      bar_init(&bars->dq_free[g], 128);
    }
    bar_init(&bars->mma_drain, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp >= kWarpProducer) {
    regs_decrease<kBwdAuxRegs>();
    if (warp == kWarpProducer) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0 && n_tiles > 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
        bar_arrive_expect_tx(&bars->kv_full, 2 * KVB);
        for (int c = 0; c < 2; ++c) {
          tma_load_3d(sK + c * Cfg::kKVChunk, &tm_k, &bars->kv_full, c * 64, key0, bh);
          tma_load_3d(sV + c * Cfg::kKVChunk, &tm_v, &bars->kv_full, c * 64, key0, bh);
        }
        bool ok = true;
        for (int t = 0; t < n_tiles && ok; ++t) {
          const int slot = t % STAGES;
          const int lap = t / STAGES;
          if (lap > 0 && !wait_bar(&bars->q_empty[slot], (lap - 1) & 1, abort, p.timeout_ns)) {
            raise_abort(abort, p.status);
            ok = false;
            break;
          }
          bar_arrive_expect_tx(&bars->q_full[slot], 2 * QB);
          const int row = (i0 + t) * QR;
          for (int c = 0; c < 2; ++c) {
            tma_load_3d(sQ + slot * QB + c * Cfg::kQChunk, &tm_q, &bars->q_full[slot], c * 64, row, bh);
            tma_load_3d(sdO + slot * QB + c * Cfg::kQChunk, &tm_do, &bars->q_full[slot], c * 64, row, bh);
          }
        }
        volatile int never = 0;
        wait_bar(&bars->kv_full, 0, &never, p.timeout_ns);
        for (int t = max(0, n_tiles - STAGES); t < n_tiles; ++t)
          wait_bar(&bars->q_full[t % STAGES], (t / STAGES) & 1, &never, p.timeout_ns);
      }
    } else if (warp == kWarpMma) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0 && n_tiles > 0) {
        constexpr uint32_t kIdSP = idesc_f32acc(128, QR, false, false, F16);   // S^T, dP^T: N = 64 queries
        constexpr uint32_t kIdAcc = idesc_f32acc(128, D, false, true, F16);    // dV, dK
        constexpr uint32_t kIdDq = idesc_f32acc(128, QR, true, true, F16);     // dQ^T: M = D, N = 64
        const uint32_t aK = smem_addr(sK), aV = smem_addr(sV);
        const uint32_t aQ = smem_addr(sQ), adO = smem_addr(sdO), adS = smem_addr(sdS);
        // D[128 keys x 64 queries] = A B^T: A the K-major key block (16 KB
        // per 64-column chunk), B a K-major 64-row tile (8 KB per chunk).
        auto issue_scores = [&](uint32_t dcol, uint32_t a0, uint32_t b0) {
          uint64_t da = sdesc_sw128(a0, 16, 1024), db = sdesc_sw128(b0, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            mma_ss(tmem + dcol, da, db, kIdSP, kk > 0 ? 1u : 0u);
            da += ((kk & 3) == 3 ? Cfg::kKVChunk - 3 * 32 : 32) >> 4;
            db += ((kk & 3) == 3 ? Cfg::kQChunk - 3 * 32 : 32) >> 4;
            asm volatile("" : "+l"(da), "+l"(db));
          }
        };
        // D[128 keys x D] (+)= A[tmem: 128 keys x 64 queries, packed two per
        // column] B, B an MN-major 64-row tile.
        auto issue_acc = [&](uint32_t dcol, uint32_t acol, uint32_t b0, bool acc) {
          uint64_t db = sdesc_sw128(b0, Cfg::kQChunk, 1024);
#pragma unroll
          for (int kk = 0; kk < QR / 16; ++kk) {
            const uint32_t a = tmem + acol + 8 * kk;
            mma_ts(tmem + dcol, a, db, kIdAcc, (acc || kk > 0) ? 1u : 0u);
            db += 2048 >> 4;   // next 16 queries
            asm volatile("" : "+l"(db));
          }
        };
        auto issue_sp = [&](int t) {
          const int slot = t % STAGES, b = t & 1;
          issue_scores(Cfg::kColDP + 64 * b, aV, adO + slot * QB);   // dP^T = V dO^T
          issue_scores(Cfg::kColS + 64 * b, aK, aQ + slot * QB);     // S^T = K Q^T
          mma_commit(&bars->s_full[b]);
        };

        bool ok = wait_bar(&bars->kv_full, 0, abort, p.timeout_ns) &&
                  wait_bar(&bars->q_full[0], 0, abort, p.timeout_ns);
        if (ok) {
          tc_fence_after_sync();
          issue_sp(0);
        }
        for (int t = 0; t < n_tiles && ok; ++t) {
          const int slot = t % STAGES, b = t & 1;
          const uint32_t kp = (t >> 1) & 1;   // phase of tile t on its warpgroup's barriers
          if (!wait_bar(&bars->p_ready[b], kp, abort, p.timeout_ns)) { ok = false; break; }
          tc_fence_after_sync();
          issue_acc(Cfg::kColDV, Cfg::kColS + 64 * b, adO + slot * QB, t > 0);     // dV += P^T dO
          if (t + 1 < n_tiles) {
            const int s1 = (t + 1) % STAGES;
            if (!wait_bar(&bars->q_full[s1], ((t + 1) / STAGES) & 1, abort, p.timeout_ns)) { ok = false; break; }
            // buffer (t+1) % 2 holds dQ^T(t-1) until its warpgroup has read it out
            if (t >= 1 && !wait_bar(&bars->dq_free[b ^ 1], ((t - 1) >> 1) & 1, abort, p.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_sp(t + 1);
          }
          if (!wait_bar(&bars->ds_ready[b], kp, abort, p.timeout_ns)) { ok = false; break; }
          tc_fence_after_sync();
          issue_acc(Cfg::kColDK, Cfg::kColDP + 64 * b, aQ + slot * QB, t > 0);     // dK += dS^T Q
          {                                                                          // dQ^T = K^T dS^T
            uint64_t dA = sdesc_sw128(aK, Cfg::kKVChunk, 1024);
            uint64_t dB = sdesc_sw128(adS + b * Cfg::kDsBytes, Cfg::kKVChunk, 1024);
#pragma unroll
            for (int kk = 0; kk < 128 / 16; ++kk) {
              mma_ss(tmem + Cfg::kColS + 64 * b, dA, dB, kIdDq, kk > 0 ? 1u : 0u);
              dA += 2048 >> 4;   // next 16 keys
              dB += 2048 >> 4;
              asm volatile("" : "+l"(dA), "+l"(dB));
            }
          }
          mma_commit(&bars->dq_full[b]);
        }
        if (!ok) raise_abort(abort, p.status);
        mma_commit(&bars->mma_drain);
        volatile int never = 0;
        wait_bar(&bars->mma_drain, 0, &never, p.timeout_ns);
      }
    }
  } else {
    regs_increase<kBwdWorkRegs>();
    // ------------------------------------------------------------ elementwise warps
    const int g = warp >> 2;                  // this warpgroup's tiles: t % 2 == g (TMEM buffer g)
    const int wq = warp & 3;
    const int row = wq * 32 + lane;           // TMEM lane: key row (S^T, dP^T, dK, dV) or head column (dQ^T)
    const int key = key0 + row;
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_bits + Cfg::kColS + 64 * g;
    const uint32_t tDP = tmem + lane_bits + Cfg::kColDP + 64 * g;
    const float sl2 = p.scale_log2;
    const float* L2h = p.L2 + static_cast<size_t>(bh) * p.Nq_pad;
    const float* Drh = p.Dr + static_cast<size_t>(bh) * p.Nq_pad;
    const uint32_t ds_row = smem_addr(sdS + g * Cfg::kDsBytes) + row * 128;
    const bool leader = (threadIdx.x & 127) == 0;
    bool ok = true;

    for (int t = g; t < n_tiles && ok; t += 2) {
      const uint32_t kp = (t >> 1) & 1;       // phase of this tile on the warpgroup's barriers
      const int slot = t % STAGES;
      const int qbase = (i0 + t) * QR;
      // this tile's LSE log2(e), fetched while S^T is computed
      float4 l4v[16];
#pragma unroll
      for (int e4 = 0; e4 < 16; ++e4) l4v[e4] = __ldg(reinterpret_cast<const float4*>(L2h + qbase) + e4);
      if (!__all_sync(0xffffffffu, wait_bar(&bars->s_full[g], kp, abort, p.timeout_ns))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      // P^T = exp2(s * scale log2e - LSE log2e) on kept (key, query) pairs
      float P[64];
      uint32_t pk[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t s[32];
        tmem_ld32(tS + 32 * h, s);
        tmem_ld_wait(s);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l = l4v[8 * h + e4];
          const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int e = 4 * e4 + u;
            const int q = qbase + 32 * h + e;
            const bool keep = q < p.Nq && key < p.Nk && (!CAUSAL || key <= q);
            P[32 * h + e] = keep ? ex2_approx(fmaf(__uint_as_float(s[e]), sl2, -lv[u])) : 0.f;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) pk[e] = pack_x2<F16>(P[2 * e], P[2 * e + 1]);
      tmem_st32(tS, pk);
      float4 d4v[16];
#pragma unroll
      for (int e4 = 0; e4 < 16; ++e4) d4v[e4] = __ldg(reinterpret_cast<const float4*>(Drh + qbase) + e4);
      tmem_st_wait();
      tc_fence_before_sync();
      bar_arrive(&bars->p_ready[g]);
      // this warpgroup's previous tile's dQ reductions have had a whole P
      // phase to read their staging: hand that ring slot back to the producer
      if (leader && t >= 2) {
        bulk_wait_read();
        bar_arrive(&bars->q_empty[(t - 2) % STAGES]);
      }

      // dS^T = P^T (dP^T - D): to TMEM (A of dK) and to this warpgroup's dS
      // tile (B of dQ^T; dQ^T of its previous tile has read it: this
      // warpgroup waited for that dq_full)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t gv[32];
        tmem_ld32(tDP + 32 * h, gv);
        tmem_ld_wait(gv);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 dv = d4v[8 * h + e4];
          const float dd[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            const int e = 4 * e4 + u;
            const float a = P[32 * h + e] * (__uint_as_float(gv[e]) - dd[u]);
            const float c = P[32 * h + e + 1] * (__uint_as_float(gv[e + 1]) - dd[u + 1]);
            pk[16 * h + e / 2] = pack_x2<F16>(a, c);
          }
        }
        // this key row's 32 queries of half h as four swizzled 16-byte units
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int unit = 4 * h + v;
          st_shared_v4(ds_row + ((unit ^ (row & 7)) << 4), pk[16 * h + 4 * v], pk[16 * h + 4 * v + 1],
                       pk[16 * h + 4 * v + 2], pk[16 * h + 4 * v + 3]);
        }
      }
      tmem_st32(tDP, pk);
      tmem_st_wait();
      fence_proxy_async_shared();
      tc_fence_before_sync();
      bar_arrive(&bars->ds_ready[g]);

      // dQ^T(t): read it out (this thread's head column `row`, 64 queries),
      // free the buffer, stage it in tile t's ring slot (queries 0-31 in
      // the Q half, 32-63 in the dO half, each as four 128-byte-swizzled
      // boxes of 32 queries x 32 columns) and add it into dQ with TMA
      // reductions.  Every MMA of the tile has completed: no MMA reads the
      // slot any more.
      if (!__all_sync(0xffffffffu, wait_bar(&bars->dq_full[g], kp, abort, p.timeout_ns))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t v[2][32];
      tmem_ld32(tS, v[0]);
      tmem_ld32(tS + 32, v[1]);
      tmem_ld_wait(v[0]);
      tmem_ld_wait(v[1]);
      tc_fence_before_sync();
      bar_arrive(&bars->dq_free[g]);
#pragma unroll
      for (int qh = 0; qh < 2; ++qh) {
        const uint32_t box = smem_addr((qh == 0 ? sQ : sdO) + slot * QB) + wq * 4096 + ((lane & 3) << 2);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const uint32_t addr = box + e * 128 + (((lane >> 2) ^ (e & 7)) << 4);
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr),
                       "r"(__float_as_uint(__uint_as_float(v[qh][e]) * p.scale))
                       : "memory");
        }
      }
      fence_proxy_async_shared();
      bar_arrive(&bars->dq_staged[g]);
      if (leader) {
        if (!wait_bar(&bars->dq_staged[g], kp, abort, p.timeout_ns)) {
          ok = false;
        } else {
#pragma unroll
          for (int qh = 0; qh < 2; ++qh) {
            uint8_t* stage = (qh == 0 ? sQ : sdO) + slot * QB;
#pragma unroll
            for (int c = 0; c < 4; ++c) tma_reduce_add_3d(&tm_dq, stage + c * 4096, 32 * c, qbase + 32 * qh, bh);
          }
          bulk_commit();
        }
      }
      ok = __all_sync(0xffffffffu, ok);
    }
    // the last reductions must have read their staging before the CTA exits
    if (leader) bulk_wait_read();
    // dK and dV are final once every MMA has completed; the warpgroup that
    // does not own the last tile gets here before that tile's MMAs are done
    if (ok && n_tiles > 0) {
      if (!__all_sync(0xffffffffu, wait_bar(&bars->mma_drain, 0, abort, p.timeout_ns)))
        ok = false;
      else
        tc_fence_after_sync();
    }

    // dK = scale dS^T Q and dV = P^T dO for this CTA's keys (zero when no
    // query sees them), as in the one-tile kernel.
    if (ok) {
      float* dk = p.dK + (static_cast<size_t>(bh) * p.Nk + key) * D;
      float* dv = p.dV + (static_cast<size_t>(bh) * p.Nk + key) * D;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = (D / 2) * g + 32 * c;
        uint32_t a[32], bb[32];
        if (n_tiles > 0) {
          tmem_ld32(tmem + lane_bits + Cfg::kColDK + col, a);
          tmem_ld_wait(a);
          tmem_ld32(tmem + lane_bits + Cfg::kColDV + col, bb);
          tmem_ld_wait(bb);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = bb[e] = 0u;
        }
        if (key >= p.Nk) continue;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          *reinterpret_cast<float4*>(dk + col + e) =
              make_float4(__uint_as_float(a[e]) * p.scale, __uint_as_float(a[e + 1]) * p.scale,
                          __uint_as_float(a[e + 2]) * p.scale, __uint_as_float(a[e + 3]) * p.scale);
          *reinterpret_cast<float4*>(dv + col + e) =
              make_float4(__uint_as_float(bb[e]), __uint_as_float(bb[e + 1]), __uint_as_float(bb[e + 2]),
                          __uint_as_float(bb[e + 3]));
        }
      }
    }
    if (!ok) raise_abort(abort, p.status);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace fa2dev
