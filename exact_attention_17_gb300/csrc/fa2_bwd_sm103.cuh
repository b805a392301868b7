// FlashAttention-2 backward pass on the fifth-generation tensor cores (sm_103a).
//
// The pages describe the backward pass only in words: it keeps the per-row
// logsumexp of the forward pass and recomputes the scores block by block
// instead of storing the attention matrix ("FlashAttention 怎么做?online
// softmax 怎么更新?", FlashAttention-2 question; "Triton内核实战", closing
// section).  What it computes is the chain rule of the definition
//   s_ij = scale q_i.k_j,  p_ij = exp(s_ij - LSE_i),  o_i = sum_j p_ij v_j
// for an upstream gradient dO:
//   dV_j = sum_i p_ij dO_i                     dp_ij = dO_i . v_j
//   D_i  = sum_j p_ij dp_ij = dO_i . o_i       ds_ij = p_ij (dp_ij - D_i)
//   dQ_i = scale sum_j ds_ij k_j               dK_j  = scale sum_i ds_ij q_i
// (D_i = dO_i . o_i because o_i = sum_j p_ij v_j.)
//
// GB300 mapping (not from the pages):
//  * a pre-pass (one warp per query row) computes D_i from dO and O, stores
//    LSE_i * log2(e) beside it, and zeroes the dQ accumulator;
//  * the main kernel owns one block of 128 keys per CTA (K_j, V_j stay in
//    shared memory) and streams the query tiles that see those keys (Q_i,
//    dO_i through a TMA ring); per tile, one thread issues five tcgen05 MMAs:
//      S^T  = K_j Q_i^T   (TMEM)          dP^T = V_j dO_i^T   (TMEM)
//      dV  += P^T dO_i    (P^T from TMEM)  dK  += dS^T Q_i    (dS^T from TMEM)
//      dQ_i = dS K_j      (dS from shared memory, MN-major; TMEM over S^T)
//    and eight warps (two warpgroups, each owning half of a key row's query
//    columns -- the backward needs no row reductions) turn S^T into P^T and
//    dP^T into dS^T, then stage the dQ_i partial in shared memory and add it
//    into global memory with TMA bulk reductions;
//  * dK and dV stay in TMEM for the whole CTA and are stored once;
//  * every mbarrier wait is bounded as in the forward kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "fa2_fwd_sm103.cuh"
#include "ptx.cuh"

namespace fa2dev {

struct BwdParams {
  float* dQ;            // [BH, Nq, D] fp32, zeroed by the pre-pass, accumulated here
  float* dK;            // [BH, Nk, D] fp32
  float* dV;            // [BH, Nk, D] fp32
  const float* L2;      // [BH, Nq_pad]: LSE_i * log2(e)
  const float* Dr;      // [BH, Nq_pad]: D_i
  int Nq;
  int Nk;
  int Nq_pad;           // Nq rounded up to 128
  int BH;
  int key_blocks;       // ceil(Nk / 128)
  int item_group;       // heads per scheduling group (see the forward kernel)
  float scale;
  float scale_log2;     // scale * log2(e)
  int* status;
  unsigned long long timeout_ns;
};

constexpr int kBwdThreads = 384;   // 8 elementwise warps, producer, MMA, 2 idle
constexpr int kBwdLaunchRegs = 168;
constexpr int kBwdWorkRegs = 216;
constexpr int kBwdAuxRegs = 72;
static_assert(256 * kBwdWorkRegs + 128 * kBwdAuxRegs <= kBwdLaunchRegs * kBwdThreads,
              "register rebalancing exceeds the launch allocation");

template <int D>
struct BwdConfig {
  static constexpr int kChunks = D / 64;
  static constexpr uint32_t kTileBytes = 128 * D * 2;          // one K, V, Q or dO tile
  static constexpr int kStages = D == 128 ? 2 : 4;              // Q_i/dO_i ring slots
  static constexpr uint32_t kDsBytes = 128 * 128 * 2;           // dS^T staging tile
  static constexpr uint32_t kSmemData = 2 * kTileBytes + kStages * 2 * kTileBytes + kDsBytes;
  static constexpr uint32_t kSmemBytes = kSmemData + 1024 /*align*/ + 1024 /*barriers*/;
  static constexpr uint32_t kColS = 0;           // S^T, then P^T; dQ_i partial after PV
  static constexpr uint32_t kColDP = 128;        // dP^T, then dS^T
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
};

template <int STAGES>
struct alignas(8) BwdBarriers {
  uint64_t kv_full;
  uint64_t q_full[STAGES];
  uint64_t q_empty[STAGES];   // one arrival per warpgroup once its dQ staging was read
  uint64_t dq_staged[2];      // per warpgroup: its 128 threads wrote their dQ rows
  uint64_t s_full;
  uint64_t p_ready;
  uint64_t ds_ready;
  uint64_t dq_full;
  uint64_t dq_free;
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort;
};

// Pre-pass: one warp per query row.  D_i = dO_i . O_i, L2_i = LSE_i log2(e),
// and the row of dQ set to zero.  Entries past Nq in each head's padded
// arrays are set to zero.
template <int D, bool F16>
__global__ void __launch_bounds__(256) fa2_bwd_pre_kernel(const float* __restrict__ O,
                                                          const uint16_t* __restrict__ dO,
                                                          const float* __restrict__ LSE,
                                                          float* __restrict__ dQ,
                                                          float* __restrict__ L2,
                                                          float* __restrict__ Dr, long long rows,
                                                          int Nq, int Nq_pad) {
  constexpr int E = D / 32;  // elements per lane
  const long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const float* o = O + r * D + lane * E;
  const uint16_t* g = dO + r * D + lane * E;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const uint32_t bits = g[e];
    const float gv = F16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(bits)))
                         : __uint_as_float(bits << 16);
    acc = fmaf(gv, o[e], acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  float* dq = dQ + r * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2) *reinterpret_cast<float2*>(dq + e) = make_float2(0.f, 0.f);
  const long long bh = r / Nq;
  const long long q = r - bh * Nq;
  if (lane == 0) {
    Dr[bh * Nq_pad + q] = acc;
    L2[bh * Nq_pad + q] = LSE[r] * 1.4426950408889634f;
  }
  // the last row of a head also clears the padding up to Nq_pad (read, then masked)
  if (q == Nq - 1) {
    for (long long pq = Nq + lane; pq < Nq_pad; pq += 32) {
      Dr[bh * Nq_pad + pq] = 0.f;
      L2[bh * Nq_pad + pq] = 0.f;
    }
  }
}

template <int D, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa2_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using Cfg = BwdConfig<D>;
  constexpr int STAGES = Cfg::kStages;
  constexpr uint32_t TILE = Cfg::kTileBytes;
  constexpr int NCH = Cfg::kChunks;
  constexpr uint32_t kChunkBytes = 128 * 128;  // one 64-column chunk of a 128-row tile
  constexpr int kWarpProducer = 8;
  constexpr int kWarpMma = 9;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sK = smem;
  uint8_t* sV = smem + TILE;
  uint8_t* sQ = smem + 2 * TILE;                 // STAGES tiles
  uint8_t* sdO = sQ + STAGES * TILE;             // STAGES tiles
  uint8_t* sdS = sdO + STAGES * TILE;            // [128 keys][128 queries], MN-major A of dQ
  auto* bars = reinterpret_cast<BwdBarriers<STAGES>*>(smem + Cfg::kSmemData);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: (key block jb, b*H + h), grouped like the forward kernel;
  // under the causal mask the first key blocks see the most query tiles and
  // run first.
  const int U = p.key_blocks;
  const int per_group = p.item_group * U;
  const int group = blockIdx.x / per_group;
  const int in_group = blockIdx.x - group * per_group;
  const int g0 = group * p.item_group;
  const int g_items = min(p.item_group, p.BH - g0);
  const int jb = in_group / g_items;
  const int bh = g0 + (in_group - jb * g_items);
  const int q_tiles = (p.Nq + 127) / 128;
  const int i0 = CAUSAL ? jb : 0;               // first query tile with a query >= the first key
  const int n_tiles = max(0, q_tiles - i0);
  const int key0 = jb * 128;

  if (threadIdx.x == 0) {
    bar_init(&bars->kv_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      bar_init(&bars->q_full[s], 1);
      bar_init(&bars->q_empty[s], 2);
    }
    bar_init(&bars->dq_staged[0], 128);
    bar_init(&bars->dq_staged[1], 128);
    bar_init(&bars->s_full, 1);
    bar_init(&bars->p_ready, 256);
    bar_init(&bars->ds_ready, 256);
    bar_init(&bars->dq_full, 1);
    bar_init(&bars->dq_free, 256);
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
        bar_arrive_expect_tx(&bars->kv_full, 2 * TILE);
        for (int c = 0; c < NCH; ++c) {
          tma_load_3d(sK + c * kChunkBytes, &tm_k, &bars->kv_full, c * 64, key0, bh);
          tma_load_3d(sV + c * kChunkBytes, &tm_v, &bars->kv_full, c * 64, key0, bh);
        }
        bool ok = true;
        for (int t = 0; t < n_tiles && ok; ++t) {
          const int slot = t % STAGES;
          const int lap = t / STAGES;   // laps of the ring completed
          if (lap > 0 && !wait_bar(&bars->q_empty[slot], (lap - 1) & 1, abort, p.timeout_ns)) {
            raise_abort(abort, p.status);
            ok = false;
            break;
          }
          bar_arrive_expect_tx(&bars->q_full[slot], 2 * TILE);
          const int row = (i0 + t) * 128;
          for (int c = 0; c < NCH; ++c) {
            tma_load_3d(sQ + slot * TILE + c * kChunkBytes, &tm_q, &bars->q_full[slot], c * 64, row, bh);
            tma_load_3d(sdO + slot * TILE + c * kChunkBytes, &tm_do, &bars->q_full[slot], c * 64, row, bh);
          }
        }
        // every copy this CTA started must land before it exits
        volatile int never = 0;
        wait_bar(&bars->kv_full, 0, &never, p.timeout_ns);
        for (int t = max(0, n_tiles - STAGES); t < n_tiles; ++t)
          wait_bar(&bars->q_full[t % STAGES], (t / STAGES) & 1, &never, p.timeout_ns);
      }
    } else if (warp == kWarpMma) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0 && n_tiles > 0) {
        constexpr uint32_t kIdSq = idesc_f32acc(128, 128, false, false, F16);   // S^T, dP^T
        constexpr uint32_t kIdAcc = idesc_f32acc(128, D, false, true, F16);     // dV, dK
        constexpr uint32_t kIdDq = idesc_f32acc(128, D, true, true, F16);       // dQ
        const uint32_t aK = smem_addr(sK), aV = smem_addr(sV);
        const uint32_t aQ = smem_addr(sQ), adO = smem_addr(sdO), adS = smem_addr(sdS);
        // Descriptors are formed once per operand tile and stepped by the
        // K-step offset (start-address field; shared addresses stay below
        // 256 KB, so it cannot carry), one step at a time.
        // D[128 x 128] = A B^T with A, B K-major 128 x D tiles
        auto issue_kmajor = [&](uint32_t dcol, uint32_t a0, uint32_t b0) {
          uint64_t da = sdesc_sw128(a0, 16, 1024), db = sdesc_sw128(b0, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            mma_ss(tmem + dcol, da, db, kIdSq, kk > 0 ? 1u : 0u);
            const uint32_t step = ((kk & 3) == 3 ? kChunkBytes - 3 * 32 : 32) >> 4;
            da += step;
            db += step;
            asm volatile("" : "+l"(da), "+l"(db));
          }
        };
        // D[128 x D] (+)= A[tmem, 128 x 128] B, B an MN-major 128 x D tile; the
        // A columns of warpgroup w's queries start at acol + 64 w.
        auto issue_ts = [&](uint32_t dcol, uint32_t acol, uint32_t b0, bool acc) {
          uint64_t dbv = sdesc_sw128(b0, kChunkBytes, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t a = tmem + acol + 64 * (kk >> 2) + 8 * (kk & 3);
            mma_ts(tmem + dcol, a, dbv, kIdAcc, (acc || kk > 0) ? 1u : 0u);
            dbv += 2048 >> 4;
            asm volatile("" : "+l"(dbv));
          }
        };
        bool ok = wait_bar(&bars->kv_full, 0, abort, p.timeout_ns);
        for (int t = 0; t < n_tiles && ok; ++t) {
          const int slot = t % STAGES;
          const uint32_t q0 = aQ + slot * TILE, do0 = adO + slot * TILE;
          if (!wait_bar(&bars->q_full[slot], (t / STAGES) & 1, abort, p.timeout_ns)) { ok = false; break; }
          tc_fence_after_sync();
          issue_kmajor(Cfg::kColDP, aV, do0);                       // dP^T = V dO^T
          if (t > 0 && !wait_bar(&bars->dq_free, (t - 1) & 1, abort, p.timeout_ns)) { ok = false; break; }
          tc_fence_after_sync();
          issue_kmajor(Cfg::kColS, aK, q0);                         // S^T = K Q^T
          mma_commit(&bars->s_full);
          if (!wait_bar(&bars->p_ready, t & 1, abort, p.timeout_ns)) { ok = false; break; }
          tc_fence_after_sync();
          issue_ts(Cfg::kColDV, Cfg::kColS, do0, t > 0);            // dV += P^T dO
          if (!wait_bar(&bars->ds_ready, t & 1, abort, p.timeout_ns)) { ok = false; break; }
          tc_fence_after_sync();
          issue_ts(Cfg::kColDK, Cfg::kColDP, q0, t > 0);            // dK += dS^T Q
          {                                                          // dQ_i = dS K
            uint64_t dA = sdesc_sw128(adS, kChunkBytes, 1024), dB = sdesc_sw128(aK, kChunkBytes, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              mma_ss(tmem + Cfg::kColS, dA, dB, kIdDq, kk > 0 ? 1u : 0u);
              dA += 2048 >> 4;
              dB += 2048 >> 4;
              asm volatile("" : "+l"(dA), "+l"(dB));
            }
          }
          mma_commit(&bars->dq_full);
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
    const int wg = warp >> 2;                 // query columns [64 wg, 64 wg + 64) of a tile
    const int wq = warp & 3;
    const int row = wq * 32 + lane;           // TMEM lane: key row (S^T, dP^T, dK, dV) or query row (dQ)
    const int key = key0 + row;
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    const float* L2h = p.L2 + static_cast<size_t>(bh) * p.Nq_pad;
    const float* Drh = p.Dr + static_cast<size_t>(bh) * p.Nq_pad;
    const uint32_t ds_base = smem_addr(sdS) + wg * kChunkBytes + row * 128;
    bool ok = true;
    const bool leader = (threadIdx.x & 127) == 0;
    for (int t = 0; t < n_tiles; ++t) {
      const int slot = t % STAGES;
      const int qbase = (i0 + t) * 128;
      const int qcol0 = qbase + 64 * wg;      // first query of this warpgroup's columns
      // this tile's LSE log2(e) for the warpgroup's columns, fetched while S^T is computed
      float4 l4v[16];
#pragma unroll
      for (int e4 = 0; e4 < 16; ++e4) l4v[e4] = __ldg(reinterpret_cast<const float4*>(L2h + qcol0) + e4);
      if (!__all_sync(0xffffffffu, wait_bar(&bars->s_full, t & 1, abort, p.timeout_ns))) {
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
        tmem_ld32(tmem + lane_bits + Cfg::kColS + 64 * wg + 32 * h, s);
        tmem_ld_wait(s);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l = l4v[8 * h + e4];
          const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int e = 4 * e4 + u;
            const int q = qcol0 + 32 * h + e;
            const bool keep = q < p.Nq && key < p.Nk && (!CAUSAL || key <= q);
            P[32 * h + e] = keep ? ex2_approx(fmaf(__uint_as_float(s[e]), sl2, -lv[u])) : 0.f;
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 32; ++e) pk[e] = pack_x2<F16>(P[2 * e], P[2 * e + 1]);
      tmem_st32(tmem + lane_bits + Cfg::kColS + 64 * wg, pk);
      // D for the same columns, fetched while the P^T store completes
      float4 d4v[16];
#pragma unroll
      for (int e4 = 0; e4 < 16; ++e4) d4v[e4] = __ldg(reinterpret_cast<const float4*>(Drh + qcol0) + e4);
      tmem_st_wait();
      tc_fence_before_sync();
      bar_arrive(&bars->p_ready);
      // the previous tile's dQ reductions have had a whole P phase to read
      // their staging: release that ring slot to the producer now
      if (leader && t > 0) {
        bulk_wait_read();
        bar_arrive(&bars->q_empty[(t - 1) % STAGES]);
      }

      // dS^T = P^T (dP^T - D): to TMEM (A of dK) and to shared memory (A of dQ)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t g[32];
        tmem_ld32(tmem + lane_bits + Cfg::kColDP + 64 * wg + 32 * h, g);
        tmem_ld_wait(g);
#pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 dv = d4v[8 * h + e4];
          const float dd[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            const int e = 4 * e4 + u;
            const float a = P[32 * h + e] * (__uint_as_float(g[e]) - dd[u]);
            const float b = P[32 * h + e + 1] * (__uint_as_float(g[e + 1]) - dd[u + 1]);
            pk[16 * h + e / 2] = pack_x2<F16>(a, b);
          }
        }
        // this key row's 64 queries as 8 swizzled 16-byte units of chunk wg
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const int unit = 4 * h + v;
          st_shared_v4(ds_base + ((unit ^ (row & 7)) << 4), pk[16 * h + 4 * v], pk[16 * h + 4 * v + 1],
                       pk[16 * h + 4 * v + 2], pk[16 * h + 4 * v + 3]);
        }
      }
      tmem_st32(tmem + lane_bits + Cfg::kColDP + 64 * wg, pk);
      tmem_st_wait();
      fence_proxy_async_shared();
      tc_fence_before_sync();
      bar_arrive(&bars->ds_ready);

      // dQ_i partial (TMEM lanes are query rows now).  Its columns go back to
      // the issuer as soon as they are in registers; the scaled rows are then
      // staged in this tile's Q/dO ring slot (no MMA reads it any more) as
      // 128-byte-swizzled boxes of 32 columns, and one thread per warpgroup
      // adds them into dQ with TMA reductions before releasing the slot.
      if (!__all_sync(0xffffffffu, wait_bar(&bars->dq_full, t & 1, abort, p.timeout_ns))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t v[D / 64][32];
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tmem_ld32(tmem + lane_bits + Cfg::kColS + (D / 2) * wg + 32 * c, v[c]);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) tmem_ld_wait(v[c]);
      tc_fence_before_sync();
      bar_arrive(&bars->dq_free);
      uint8_t* stage = wg == 0 ? sQ + slot * TILE : sdO + slot * TILE;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const uint32_t box = smem_addr(stage) + c * 16384 + row * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(box + ((u ^ (row & 7)) << 4), __float_as_uint(__uint_as_float(v[c][4 * u]) * p.scale),
                       __float_as_uint(__uint_as_float(v[c][4 * u + 1]) * p.scale),
                       __float_as_uint(__uint_as_float(v[c][4 * u + 2]) * p.scale),
                       __float_as_uint(__uint_as_float(v[c][4 * u + 3]) * p.scale));
      }
      fence_proxy_async_shared();
      bar_arrive(&bars->dq_staged[wg]);
      if (leader) {
        if (!wait_bar(&bars->dq_staged[wg], t & 1, abort, p.timeout_ns)) {
          ok = false;
        } else {
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_reduce_add_3d(&tm_dq, stage + c * 16384, (D / 2) * wg + 32 * c, qbase, bh);
          bulk_commit();
        }
      }
      // keep `ok` uniform across the warp: the TMEM accesses after the loop are warp-collective
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
    }
    // The last tile's reductions must have read their staged dQ before the
    // CTA exits; their global updates complete with the grid.
    if (leader) bulk_wait_read();

    // dK = scale dS^T Q and dV = P^T dO for this CTA's keys (zero when no query
    // sees them).  `ok` and n_tiles are uniform across a warp; the TMEM loads
    // are warp-collective, so every lane runs them and only the stores are
    // limited to keys < Nk.
    if (ok) {
      float* dk = p.dK + (static_cast<size_t>(bh) * p.Nk + key) * D;
      float* dv = p.dV + (static_cast<size_t>(bh) * p.Nk + key) * D;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = (D / 2) * wg + 32 * c;
        uint32_t a[32], b[32];
        if (n_tiles > 0) {
          tmem_ld32(tmem + lane_bits + Cfg::kColDK + col, a);
          tmem_ld_wait(a);
          tmem_ld32(tmem + lane_bits + Cfg::kColDV + col, b);
          tmem_ld_wait(b);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) a[e] = b[e] = 0u;
        }
        if (key >= p.Nk) continue;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          *reinterpret_cast<float4*>(dk + col + e) =
              make_float4(__uint_as_float(a[e]) * p.scale, __uint_as_float(a[e + 1]) * p.scale,
                          __uint_as_float(a[e + 2]) * p.scale, __uint_as_float(a[e + 3]) * p.scale);
          *reinterpret_cast<float4*>(dv + col + e) =
              make_float4(__uint_as_float(b[e]), __uint_as_float(b[e + 1]), __uint_as_float(b[e + 2]),
                          __uint_as_float(b[e + 3]));
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
