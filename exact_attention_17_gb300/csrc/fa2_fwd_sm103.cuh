// FlashAttention-2 forward on the fifth-generation tensor cores (sm_103a).
//
// What it computes (per (b, h), per query row i):
//   O_i = sum_j softmax_j(scale * q_i . k_j) v_j,   LSE_i = log sum_j exp(scale * q_i . k_j)
// over the kept keys j (all keys, or j <= i with the top-left causal mask).
//
// How, following the FlashAttention-2 method of the pages:
//  * loop order and grid -- "FlashAttention-2 算法架构升级" section 二 and
//    "Flash Attention 全解析(上)" section 3.2.1: the Q block is the outer loop and
//    owns one CTA; K/V blocks stream through the inner loop; CTAs are
//    independent (no atomics, no inter-CTA communication);
//  * online softmax -- "FlashAttention 怎么做?online softmax 怎么更新?",
//    section 推导/关键公式: m' = max(m, rowmax S), P = exp(S - m'),
//    l' = exp(m - m') l + rowsum P, O' = exp(m - m') O + P V;
//  * lazy normalisation and the per-row logsumexp -- the same page's
//    FlashAttention-2 question and "Flash Attention 全解析(上)" section 3.2.3:
//    O is divided by l once after the K/V loop, L = m + log l is stored;
//  * causal block skipping -- "FlashAttention 怎么做?", FlashAttention-2
//    question: K/V blocks entirely above the diagonal are never visited;
//  * tail masking -- "Triton内核实战" kernel section (masked loads for ragged N).
//
// GB300 mapping (not from the pages):
//  * one CTA = two 128-row Q sub-tiles (256 query rows) sharing one K/V
//    stream (or one sub-tile, with two CTAs per SM); warps 0-3 (and 4-7) are
//    the softmax warpgroups of the sub-tiles (thread t owns query row t =
//    TMEM lane t, so row max and row sum need no cross-thread reduction --
//    the "sliced-Q" split of "Flash Attention 全解析(上)" section 3.2.2 taken to
//    one row per thread); the next warp issues TMA loads, the one after it
//    issues the tcgen05 MMAs and owns TMEM;
//  * S = Q K^T runs as tcgen05.mma (bf16 x bf16 -> f32) from shared memory into
//    TMEM; P is written back to TMEM as bf16 over S's columns and O += P V
//    takes P straight from TMEM (A operand) and V from shared memory (MN-major);
//  * TMEM columns: S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D);
//  * the two sub-tiles ping-pong: while one warpgroup runs its softmax the
//    tensor core works on the other sub-tile's MMAs;
//  * scores are scaled by scale*log2(e) inside one FMA and exponentiated with
//    ex2; m is kept in that log2 domain and LSE converted to natural log once;
//  * the running max used as the exponent offset is only moved when the row
//    max grows by more than RESCALE_LOG2 (2^8): P then stays <= 256 and the
//    correction factor exp(m - m') is applied to O and l together, so the
//    result is the same softmax; O in TMEM is only rescaled when some row of a
//    warp moved its offset;
//  * every mbarrier wait is bounded; on expiry the CTA records a device error
//    bit, unwinds, drains its copies and MMAs and frees TMEM.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"

namespace fa2dev {

// Error bits OR-ed into the library's device status word.
constexpr int kDevErrTimeout = 1;

// Division by a divisor that is fixed for a launch, as one widening multiply
// and a shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994): for 0 <= n < 2^31 and d >= 1, with l = ceil(log2 d),
// m = ceil(2^(31+l) / d) < 2^32 and s = 31 + l, floor(n / d) = (n m) >> s.
// A division by a run-time divisor costs about two hundred cycles, and the
// work-item decode at CTA start had a chain of three.
struct FastDiv {
  uint32_t m;
  int s;
};

__host__ __device__ __forceinline__ int fast_div(int n, const FastDiv& f) {
  return static_cast<int>((static_cast<unsigned long long>(static_cast<uint32_t>(n)) * f.m) >> f.s);
}

struct FwdParams {
  float* O;        // [BH, Nq, D] fp32 (num_splits == 1)
  float* LSE;      // [BH, Nq]    fp32 (num_splits == 1)
  int Nq;
  int Nk;
  int BH;
  int q_blocks;    // ceil(Nq / rows per CTA)
  float scale_log2;  // scale * log2(e)
  int* status;     // device status word
  int wave;        // CTAs that run at once (the L2 prefetch looks one wave ahead)
  unsigned long long timeout_ns;
  // Split of the keys into ranges processed by separate CTAs ("FlashDecoding",
  // "Flash Attention 全解析(上)" section 4): range s covers key tiles
  // [s * tiles_per_split, (s + 1) * tiles_per_split).  With num_splits > 1
  // each CTA writes its range's normalised output and logsumexp to
  // O_part [num_splits, BH, Nq, D] and LSE_part [num_splits, BH, Nq]; a row
  // with no kept key in the range gets O = 0 and LSE = -inf.
  int num_splits;
  int tiles_per_split;
  float* O_part;
  float* LSE_part;
  // O in the input element type (16 bits) instead of fp32 (num_splits == 1).
  int o_half;
  // Work items (b*H + h, key range) are scheduled in groups of item_group:
  // within a group CTAs run query block by query block across the group's
  // items, heaviest causal blocks first.
  int item_group;
  FastDiv div_per_group;  // by item_group * q_blocks
  FastDiv div_group;      // by item_group
  FastDiv div_splits;     // by num_splits
};

constexpr int kRowsPerSub = 128;   // tcgen05 M
constexpr int kKeysPerTile = 128;  // K/V block (N of S, K of P V)
// A CTA holds SUBS query sub-tiles of 128 rows: SUBS = 2 (one CTA per SM,
// the two sub-tiles ping-pong on the tensor core) or SUBS = 1 (two CTAs per
// SM, each with its own MMA-issuing thread).  Threads: 128 per sub-tile
// (softmax) plus one warpgroup for the producer and MMA warps.
template <int SUBS>
struct FwdShape {
  static constexpr int kThreads = SUBS * 128 + 128;
  static constexpr int kCtasPerSm = SUBS == 2 ? 1 : 2;
  // Register budgets after the start-up rebalancing.  At launch every thread
  // has kLaunch registers (65536 / (threads * CTAs per SM), rounded down to a
  // multiple of 8); the softmax warpgroups then take kSoftmax and the
  // producer warpgroup gives back down to kProducer.
  static constexpr int kLaunch = SUBS == 2 ? 168 : 128;
  static constexpr int kSoftmax = SUBS == 2 ? 216 : 208;
  static constexpr int kProducer = SUBS == 2 ? 64 : 48;
  static_assert(SUBS * 128 * kSoftmax + 128 * kProducer <= kLaunch * kThreads,
                "register rebalancing exceeds the launch allocation");
  static_assert(kLaunch * kThreads * kCtasPerSm <= 65536, "launch registers exceed the SM");
};
// The exponent offset of a row moves only when its scores exceed it by more
// than this (log2 units), so every P stays <= 2^kRescaleLog2.
constexpr float kRescaleLog2 = 8.0f;
constexpr float kRescaleBound = 256.0f;   // 2^kRescaleLog2

template <int D, int SUBS>
struct FwdConfig {
  static_assert(D == 64 || D == 128 || D == 256, "head dimension");
  // D = 256: a Q sub-tile or a K/V tile is 64 KB, so one sub-tile per CTA,
  // one CTA per SM and a two-slot ring (192 KB of shared memory).
  static_assert(D < 256 || SUBS == 1, "head dimension 256 takes one sub-tile per CTA");
  static constexpr int kChunks = D / 64;                    // 128-byte swizzle atoms per row
  static constexpr uint32_t kTileBytes = kKeysPerTile * D * 2;  // one K or V tile, one Q sub-tile
  // K/V ring slots (K and V alternate); with two CTAs per SM each gets half
  // of the shared memory.
  static constexpr int kStages = D == 256 ? 2 : SUBS == 2 ? (D == 128 ? 4 : 8) : (D == 128 ? 2 : 5);
  // S buffers in TMEM.  With one CTA per SM (D = 256) the 512 columns hold
  // two S buffers and O: S for the next key tile is computed into the other
  // buffer while the softmax of the current one runs.  Otherwise one per
  // sub-tile, and S of the next tile overwrites P once P V is issued.
  static constexpr bool kDoubleS = D == 256;
  // K/V ring slots released by a softmax thread instead of MMA commits:
  // the completion of S_r(j) (r: the sub-tile that visits every key tile)
  // implies that every MMA reading K_j and V_(j-1) has completed, and a
  // commit costs the issuing thread time that idles the tensor pipe.  With a
  // two-slot ring the V slot must be released as soon as P V completes, and
  // the double-buffered issue order (S(j+1) before P(j) V) does not give the
  // implication, so those keep the commits.
  static constexpr bool kSoftmaxRelease = !kDoubleS && kStages >= 4;
  // O of a sub-tile announced complete only after its last P V: in the
  // single-buffered issue order S(j+1) follows P(j) V, so the softmax's wait
  // for S(j+1) already orders its rescale of O after P(j) V.
  static constexpr bool kOutDoneLast = !kDoubleS;
  // With a ring of four or more slots the issuing thread waits on named
  // (hardware) barriers instead of polling mbarriers: an mbarrier check costs
  // it about 100 cycles while the tensor pipe keeps shared memory busy, and
  // the pipe idles meanwhile.  A watcher warp waits for the K/V copies and
  // joins the first of them (the two-slot ring and the double-buffered order
  // keep their mbarriers).
  static constexpr bool kNamedP = !kDoubleS && kStages >= 4;
  // TMEM columns: S buffers (128 fp32 columns each), then O of each sub-tile (D).
  static constexpr uint32_t kColsO0 = (kDoubleS ? 2 : SUBS) * 128;
  static constexpr uint32_t kColsO1 = kColsO0 + D;
  static constexpr uint32_t kTmemCols = (SUBS == 2 || D == 256) ? 512 : 256;
  static_assert(kColsO0 + SUBS * D <= kTmemCols, "TMEM columns");
  static constexpr uint32_t kSmemData = (SUBS + kStages) * kTileBytes;
  static constexpr uint32_t kSmemBytes = kSmemData + 1024 /*align*/ + 1024 /*barriers*/;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Named barriers of the forward kernels (0 is __syncthreads).  kBarP0: P_0(j)
// written (4 softmax warps) and V_j, K_(j+1) landed (the watcher warp), for
// the issuing warp; kBarP1: P_1(j) written (4 softmax warps), for the issuing
// warp.  Every participant waits at every phase, in order, also after an
// abort, so that no wait on them is left without its arrivals: a named
// barrier has no phase number, so an arrival that ran a phase ahead would
// be counted in the open one.  (The softmax warps lose nothing by waiting:
// their next S cannot be ready before the issuing warp has passed.)
constexpr int kBarP0 = 1;
constexpr int kBarP1 = 2;
constexpr int kBarP0Count = kRowsPerSub + 64;   // softmax warpgroup 0, issuing warp, watcher warp
constexpr int kBarP0Idle = 64;                  // issuing and watcher warps (sub-tile 0 done)
constexpr int kBarP1Count = kRowsPerSub + 32;   // softmax warpgroup 1, issuing warp

// Ties 32 registers written by a tcgen05.ld to a preceding tcgen05.wait::ld
// (asm volatile statements keep their order): no instruction is emitted.
__device__ __forceinline__ void regs_after_wait(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                 "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
                 "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// MMAs from descriptors given as 32-bit halves: only the low word (its
// 14-bit start-address field) steps from one K step to the next, so one
// 32-bit add per step instead of a 64-bit one.
__device__ __forceinline__ void mma_ss_halves(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo,
                                              uint32_t b_hi, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %2};\n\tmov.b64 db, {%3, %4};\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_halves(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <int STAGES>
struct alignas(8) FwdBarriers {
  uint64_t q_full;
  uint64_t kv_full[STAGES];
  uint64_t kv_empty[STAGES];
  uint64_t s_full[2];
  uint64_t p_ready[2];
  uint64_t o_done[2];
  uint64_t staged[2];      // epilogue: a sub-tile's 128 threads wrote O into its Q buffer
  uint64_t stage_free[2];  // epilogue: the TMA stores have read that buffer
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void raise_abort(volatile int* abort, int* status) {
  *abort = 1;
  atomicOr(status, kDevErrTimeout);
}

// Number of K/V tiles query sub-tile `sub` of pair `u` visits within the key
// tile range [t_begin, t_end) (0 = no rows, or every key masked).
template <bool CAUSAL, int SUBS>
__device__ __forceinline__ int kv_tiles_for(int u, int sub, int Nq, int t_begin, int t_end) {
  const int first = (u * SUBS + sub) * kRowsPerSub;
  if (first >= Nq) return 0;
  int stop = t_end;
  if (CAUSAL) {
    const int last = min(first + kRowsPerSub - 1, Nq - 1);
    stop = min(stop, last / kKeysPerTile + 1);
  }
  return max(0, stop - t_begin);
}

// F16: Q, K, V (and P) are fp16 instead of bf16.  SUBS: query sub-tiles per CTA.
template <int D, bool CAUSAL, bool F16, int SUBS>
__global__ void __launch_bounds__(FwdShape<SUBS>::kThreads, FwdShape<SUBS>::kCtasPerSm)
    fa2_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  using Cfg = FwdConfig<D, SUBS>;
  using Shape = FwdShape<SUBS>;
  constexpr int kWarpProducer = 4 * SUBS;      // TMA warp
  constexpr int kWarpMma = 4 * SUBS + 1;       // MMA warp, owns the TMEM allocation
  constexpr int STAGES = Cfg::kStages;
  constexpr uint32_t TILE = Cfg::kTileBytes;
  constexpr int NCH = Cfg::kChunks;
  constexpr uint32_t kChunkBytes = kRowsPerSub * 128;  // one 64-column chunk of a 128-row tile

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                  // SUBS sub-tiles
  uint8_t* sKV = smem + SUBS * TILE;   // STAGES tiles
  auto* bars = reinterpret_cast<FwdBarriers<STAGES>*>(smem + Cfg::kSmemData);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: (query block u, key range, b*H + h).  Blocks are numbered
  // group by group, a group being item_group consecutive (b*H + h, range)
  // items chosen so that their K/V tiles fit in L2 together: concurrently
  // running CTAs then share K/V through L2.  Within a group the numbering
  // runs over the items for one query block before moving to the next, and
  // under the causal mask the heaviest (last) query blocks come first, so the
  // short CTAs fill the tail of the grid.
  const int U = p.q_blocks;
  const int items = p.BH * p.num_splits;
  const int per_group = p.item_group * U;
  const int group = fast_div(static_cast<int>(blockIdx.x), p.div_per_group);
  const int in_group = blockIdx.x - group * per_group;
  const int g0 = group * p.item_group;
  const int g_items = min(p.item_group, items - g0);
  // only the last group can be short
  const int u_rank = g_items == p.item_group ? fast_div(in_group, p.div_group) : in_group / g_items;
  const int item = g0 + (in_group - u_rank * g_items);
  const int bh = fast_div(item, p.div_splits);
  const int split = item - bh * p.num_splits;
  const int u = CAUSAL ? U - 1 - u_rank : u_rank;
  const int all_tiles = (p.Nk + kKeysPerTile - 1) / kKeysPerTile;
  const int t_begin = split * p.tiles_per_split;
  const int t_end = min(all_tiles, t_begin + p.tiles_per_split);
  const int n0 = kv_tiles_for<CAUSAL, SUBS>(u, 0, p.Nq, t_begin, t_end);
  const int n1 = SUBS == 2 ? kv_tiles_for<CAUSAL, SUBS>(u, 1, p.Nq, t_begin, t_end) : 0;
  const int nmax = max(n0, n1);
  const int q_row0 = u * SUBS * kRowsPerSub;

  // The producer thread sets up the barriers and starts the first loads (Q
  // and the first ring slots) before the CTA-wide synchronisation, so that
  // their latency overlaps the TMEM allocation and the synchronisation.
  const uint32_t qbytes = (n0 > 0 ? TILE : 0u) + (n1 > 0 ? TILE : 0u);
  const int primed = min(STAGES, 2 * nmax);   // K/V loads issued before the synchronisation
  if (warp == kWarpProducer && lane == 0) {
    bar_init(&bars->q_full, 1);
    for (int s = 0; s < STAGES; ++s) {
      bar_init(&bars->kv_full[s], 1);
      bar_init(&bars->kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      bar_init(&bars->s_full[i], 1);
      bar_init(&bars->p_ready[i], kRowsPerSub);
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
    if (qbytes) {
      bar_arrive_expect_tx(&bars->q_full, qbytes);
      for (int s = 0; s < SUBS; ++s) {
        if ((s == 0 ? n0 : n1) == 0) continue;
        for (int c = 0; c < NCH; ++c)
          tma_load_3d(sQ + s * TILE + c * kChunkBytes, &tm_q, &bars->q_full, c * 64,
                      q_row0 + s * kRowsPerSub, bh);
      }
    }
    for (int g = 0; g < primed; ++g) {
      bar_arrive_expect_tx(&bars->kv_full[g], TILE);
      const CUtensorMap* map = (g & 1) == 0 ? &tm_k : &tm_v;
      for (int c = 0; c < NCH; ++c)
        tma_load_3d(sKV + g * TILE + c * kChunkBytes, map, &bars->kv_full[g], c * 64,
                    (t_begin + g / 2) * kKeysPerTile, bh);
    }
    // The CTA one wave later (probably the next to run on some SM) reads a Q
    // block nobody has touched yet: start bringing it into L2 now.
    const unsigned later = blockIdx.x + p.wave;
    if (later < gridDim.x) {
      const int item2 = static_cast<int>(later);
      const int group2 = item2 / per_group;
      const int in_group2 = item2 - group2 * per_group;
      const int gi2 = min(p.item_group, items - group2 * p.item_group);
      const int u_rank2 = in_group2 / gi2;
      const int pair2 = group2 * p.item_group + (in_group2 - u_rank2 * gi2);
      const int u2 = CAUSAL ? U - 1 - u_rank2 : u_rank2;
      const int row2 = u2 * SUBS * kRowsPerSub;
      for (int s = 0; s < SUBS; ++s)
        if (row2 + s * kRowsPerSub < p.Nq)
          for (int c = 0; c < NCH; ++c)
            tma_prefetch_l2_3d(&tm_q, c * 64, row2 + s * kRowsPerSub, pair2 / p.num_splits);
    }
  }
  if (warp == kWarpMma) {
    tmem_alloc(&bars->tmem_base, Cfg::kTmemCols);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  // Each role branch starts with its register budget change, so that the
  // compiler can allocate each branch for its own budget.
  if (warp >= kWarpProducer) {
    regs_decrease<Shape::kProducer>();
    if (warp == kWarpProducer) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        // Q and the first `primed` K/V loads were issued before the synchronisation
        int issued = primed;
        bool ok = true;
        for (int j = primed / 2; j < nmax && ok; ++j) {
          for (int kind = (primed & 1) && j == primed / 2 ? 1 : 0; kind < 2; ++kind) {
            const int slot = issued % STAGES;
            const int lap = issued / STAGES;   // laps of the ring completed
            if (lap > 0 && !wait_bar(&bars->kv_empty[slot], (lap - 1) & 1, abort, p.timeout_ns)) {
              raise_abort(abort, p.status);
              ok = false;
              break;
            }
            bar_arrive_expect_tx(&bars->kv_full[slot], TILE);
            const CUtensorMap* map = kind == 0 ? &tm_k : &tm_v;
            for (int c = 0; c < NCH; ++c)
              tma_load_3d(sKV + slot * TILE + c * kChunkBytes, map, &bars->kv_full[slot], c * 64,
                          (t_begin + j) * kKeysPerTile, bh);
            ++issued;
          }
        }
        // Before the CTA may exit, every copy it started must have landed.
        // Only the last STAGES copies can still be in flight.
        volatile int never = 0;
        if (qbytes) wait_bar(&bars->q_full, 0, &never, p.timeout_ns);
        for (int k = max(0, issued - STAGES); k < issued; ++k)
          wait_bar(&bars->kv_full[k % STAGES], (k / STAGES) & 1, &never, p.timeout_ns);
      }
    } else if (warp == kWarpMma + 1 && Cfg::kNamedP) {
      // ------------------------------------------------------------ K/V watcher
      // Tile j's first named-barrier phase also stands for V_j and K_(j+1)
      // having landed.  After an abort the waits are skipped, not the phases.
      bool ok = true;
      for (int j = 0; j < nmax; ++j) {
        if (lane == 0 && ok) {
          const int iv = 2 * j + 1, ik = 2 * j + 2;
          ok = wait_bar(&bars->kv_full[iv % STAGES], (iv / STAGES) & 1, abort, p.timeout_ns);
          if (ok && j + 1 < nmax)
            ok = wait_bar(&bars->kv_full[ik % STAGES], (ik / STAGES) & 1, abort, p.timeout_ns);
          if (!ok) raise_abort(abort, p.status);
        }
        __syncwarp();
        named_sync(kBarP0, j < n0 ? kBarP0Count : kBarP0Idle);
      }
    } else if (warp == kWarpMma && Cfg::kNamedP) {
      // ------------------------------------------------------------ MMA issuer (named barriers)
      // The whole warp takes part in the named barriers; lane 0 issues every
      // MMA and every commit.  After an abort the MMAs still go out (on
      // whatever the buffers hold: the outputs are not written then), so that
      // every phase of the named barriers is passed.
      constexpr uint32_t kIdescS = idesc_f32acc(kRowsPerSub, kKeysPerTile, false, false, F16);
      constexpr uint32_t kIdescO = idesc_f32acc(kRowsPerSub, D, false, true, F16);
      const uint32_t sQaddr = smem_addr(sQ);
      const uint32_t sKVaddr = smem_addr(sKV);
      auto issue_s = [&](int sub, int slot) {
        const uint64_t da = sdesc_sw128(sQaddr + sub * TILE, 16, 1024);
        const uint64_t db = sdesc_sw128(sKVaddr + slot * TILE, 16, 1024);
        uint32_t a_lo = static_cast<uint32_t>(da), b_lo = static_cast<uint32_t>(db);
        const uint32_t a_hi = static_cast<uint32_t>(da >> 32), b_hi = static_cast<uint32_t>(db >> 32);
  #pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          mma_ss_halves(tmem + sub * 128, a_lo, a_hi, b_lo, b_hi, kIdescS, kk > 0 ? 1u : 0u);
          const uint32_t step = ((kk & 3) == 3 ? kChunkBytes - 3 * 32 : 32) >> 4;
          a_lo += step;
          b_lo += step;
          asm volatile("" : "+r"(a_lo), "+r"(b_lo));
        }
      };
      auto issue_pv = [&](int sub, int slot, bool acc) {
        const uint64_t dv = sdesc_sw128(sKVaddr + slot * TILE, kChunkBytes, 1024);
        uint32_t v_lo = static_cast<uint32_t>(dv);
        const uint32_t v_hi = static_cast<uint32_t>(dv >> 32);
        const uint32_t o = tmem + (sub == 0 ? Cfg::kColsO0 : Cfg::kColsO1);
        const uint32_t a = tmem + sub * 128;
  #pragma unroll
        for (int kk = 0; kk < kKeysPerTile / 16; ++kk) {
          mma_ts_halves(o, a + kk * 8, v_lo, v_hi, kIdescO, (acc || kk > 0) ? 1u : 0u);
          v_lo += (16 * 128) >> 4;
          asm volatile("" : "+r"(v_lo));
        }
      };
      if (lane == 0 && nmax > 0) {
        const bool ok = wait_bar(&bars->q_full, 0, abort, p.timeout_ns) &&
                        wait_bar(&bars->kv_full[0], 0, abort, p.timeout_ns);
        if (!ok) raise_abort(abort, p.status);
        tc_fence_after_sync();
        if (n0 > 0) { issue_s(0, 0); mma_commit(&bars->s_full[0]); }
        if (n1 > 0) { issue_s(1, 0); mma_commit(&bars->s_full[1]); }
      }
      __syncwarp();
      for (int j = 0; j < nmax; ++j) {
        const int slot_v = (2 * j + 1) % STAGES, slot_k = (2 * j + 2) % STAGES;
        const bool next = j + 1 < nmax;
        named_sync(kBarP0, j < n0 ? kBarP0Count : kBarP0Idle);   // P_0(j); V_j, K_(j+1) landed
        if (lane == 0) {
          tc_fence_after_sync();
          if (j < n0) {
            issue_pv(0, slot_v, j > 0);
            if (j + 1 == n0) mma_commit(&bars->o_done[0]);
          }
          if (next && j + 1 < n0) { issue_s(0, slot_k); mma_commit(&bars->s_full[0]); }
        }
        __syncwarp();
        if (j < n1) {
          named_sync(kBarP1, kBarP1Count);                      // P_1(j)
          if (lane == 0) {
            tc_fence_after_sync();
            issue_pv(1, slot_v, j > 0);
            if (j + 1 == n1) mma_commit(&bars->o_done[1]);
            if (next && j + 1 < n1) { issue_s(1, slot_k); mma_commit(&bars->s_full[1]); }
          }
          __syncwarp();
        }
      }
      if (lane == 0 && nmax > 0) {
        // Every MMA must be complete before TMEM is released.
        mma_commit(&bars->mma_drain);
        volatile int never = 0;
        wait_bar(&bars->mma_drain, 0, &never, p.timeout_ns);
      }
      __syncwarp();
    } else if (warp == kWarpMma) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0 && nmax > 0) {
        constexpr uint32_t kIdescS = idesc_f32acc(kRowsPerSub, kKeysPerTile, false, false, F16);
        constexpr uint32_t kIdescO = idesc_f32acc(kRowsPerSub, D, false, true, F16);
        const uint32_t sQaddr = smem_addr(sQ);
        const uint32_t sKVaddr = smem_addr(sKV);

        // Descriptors are formed once per operand tile and advanced by adding
        // the K-step offset to the start-address field: shared addresses are
        // below 256 KB and multiples of 16, so the 14-bit field cannot carry.
        // Fewer instructions per MMA matter here: any pause of this thread
        // idles the tensor pipe.
        // S_sub = Q_sub K^T into S buffer `buf` (by default the sub-tile's
        // own): K-major A and B, K = D in steps of 16.
        auto issue_s = [&](int sub, int slot, int buf) {
          const uint64_t da = sdesc_sw128(sQaddr + sub * TILE, 16, 1024);
          const uint64_t db = sdesc_sw128(sKVaddr + slot * TILE, 16, 1024);
          uint32_t a_lo = static_cast<uint32_t>(da), b_lo = static_cast<uint32_t>(db);
          const uint32_t a_hi = static_cast<uint32_t>(da >> 32), b_hi = static_cast<uint32_t>(db >> 32);
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            mma_ss_halves(tmem + buf * 128, a_lo, a_hi, b_lo, b_hi, kIdescS, kk > 0 ? 1u : 0u);
            // next K step: 32 bytes within a 128-byte swizzle atom, else the next 64-column chunk
            const uint32_t step = ((kk & 3) == 3 ? kChunkBytes - 3 * 32 : 32) >> 4;
            a_lo += step;
            b_lo += step;
            asm volatile("" : "+r"(a_lo), "+r"(b_lo));   // one step at a time: keeps two registers live
          }
        };
        // O_sub (+)= P_sub V : P from TMEM S buffer `buf` (bf16, 2 per column), V MN-major.
        auto issue_pv = [&](int sub, int slot, bool acc, int buf) {
          const uint64_t dv = sdesc_sw128(sKVaddr + slot * TILE, kChunkBytes, 1024);
          uint32_t v_lo = static_cast<uint32_t>(dv);
          const uint32_t v_hi = static_cast<uint32_t>(dv >> 32);
          const uint32_t o = tmem + (sub == 0 ? Cfg::kColsO0 : Cfg::kColsO1);
          const uint32_t a = tmem + buf * 128;
  #pragma unroll
          for (int kk = 0; kk < kKeysPerTile / 16; ++kk) {
            mma_ts_halves(o, a + kk * 8, v_lo, v_hi, kIdescO, (acc || kk > 0) ? 1u : 0u);
            v_lo += (16 * 128) >> 4;   // next 16 keys of V
            asm volatile("" : "+r"(v_lo));
          }
        };

        bool ok = wait_bar(&bars->q_full, 0, abort, p.timeout_ns);
        // prologue: S for K tile 0
        if (ok) ok = wait_bar(&bars->kv_full[0], 0, abort, p.timeout_ns);
        if (ok) {
          tc_fence_after_sync();
          if (n0 > 0) { issue_s(0, 0, 0); mma_commit(&bars->s_full[0]); }
          if (n1 > 0) { issue_s(1, 0, 1); mma_commit(&bars->s_full[1]); }
          if (!Cfg::kSoftmaxRelease) mma_commit(&bars->kv_empty[0]);
        }
        if constexpr (Cfg::kDoubleS) {
          // One sub-tile, S double-buffered: S(j+1) goes to the tensor pipe as
          // soon as K(j+1) has landed, ahead of P(j) V, so that the softmax of
          // tile j overlaps it.  S(j+2) overwrites P(j) only after P(j) V,
          // which was issued before it.
          for (int j = 0; j < n0 && ok; ++j) {
            const int iv = 2 * j + 1, ik = 2 * j + 2;
            const int slot_v = iv % STAGES, slot_k = ik % STAGES;
            if (j + 1 < n0) {
              if (!wait_bar(&bars->kv_full[slot_k], (ik / STAGES) & 1, abort, p.timeout_ns)) { ok = false; break; }
              tc_fence_after_sync();
              issue_s(0, slot_k, (j + 1) & 1);
              mma_commit(&bars->s_full[(j + 1) & 1]);
              mma_commit(&bars->kv_empty[slot_k]);
            }
            uint64_t* bv = &bars->kv_full[slot_v];
            const uint32_t pv = (iv / STAGES) & 1;
            // P(j) is announced on p_ready[j % 2]: a softmax that has already
            // finished tile j + 1 cannot complete a second phase of the
            // barrier waited on here.
            if (!wait_bar3(bv, pv, &bars->p_ready[j & 1], (j >> 1) & 1, bv, pv, abort, p.timeout_ns)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            issue_pv(0, slot_v, j > 0, j & 1);
            mma_commit(&bars->o_done[0]);
            mma_commit(&bars->kv_empty[slot_v]);
          }
        }
        for (int j = 0; j < nmax && ok && !Cfg::kDoubleS; ++j) {
          const int iv = 2 * j + 1, ik = 2 * j + 2;
          const int slot_v = iv % STAGES, slot_k = ik % STAGES;
          const bool next = j + 1 < nmax;
          // V_j, P_0(j) and K_(j+1) in one wait (a phase not needed is
          // replaced by a repeat of V_j's): every pause of this thread idles
          // the tensor pipe, and the three checks overlap.  With a two-slot
          // ring K_(j+1) has only just been requested, so it is waited for
          // after PV_0(j) instead.
          constexpr bool kEarlyK = STAGES >= 4;
          uint64_t* bv = &bars->kv_full[slot_v];
          const uint32_t pv = (iv / STAGES) & 1;
          uint64_t* bp = j < n0 ? &bars->p_ready[0] : bv;
          const uint32_t pp = j < n0 ? (j & 1) : pv;
          uint64_t* bk = kEarlyK && next ? &bars->kv_full[slot_k] : bv;
          const uint32_t pk = kEarlyK && next ? (ik / STAGES) & 1 : pv;
          if (!wait_bar3(bv, pv, bp, pp, bk, pk, abort, p.timeout_ns)) { ok = false; break; }
          tc_fence_after_sync();
          if (j < n0) {
            issue_pv(0, slot_v, j > 0, 0);
            if (!Cfg::kOutDoneLast || j + 1 == n0) mma_commit(&bars->o_done[0]);
          }
          if (!kEarlyK && next) {
            if (!wait_bar(&bars->kv_full[slot_k], (ik / STAGES) & 1, abort, p.timeout_ns)) { ok = false; break; }
            tc_fence_after_sync();
          }
          if (next && j + 1 < n0) { issue_s(0, slot_k, 0); mma_commit(&bars->s_full[0]); }
          if (j < n1) {
            if (!wait_bar(&bars->p_ready[1], j & 1, abort, p.timeout_ns)) { ok = false; break; }
            tc_fence_after_sync();
            issue_pv(1, slot_v, j > 0, 1);
            if (!Cfg::kOutDoneLast || j + 1 == n1) mma_commit(&bars->o_done[1]);
          }
          if (!Cfg::kSoftmaxRelease) mma_commit(&bars->kv_empty[slot_v]);
          if (next) {
            if (j + 1 < n1) { issue_s(1, slot_k, 1); mma_commit(&bars->s_full[1]); }
            if (!Cfg::kSoftmaxRelease) mma_commit(&bars->kv_empty[slot_k]);
          }
        }
        if (!ok) raise_abort(abort, p.status);
        // Every MMA must be complete before TMEM is released.
        mma_commit(&bars->mma_drain);
        volatile int never = 0;
        wait_bar(&bars->mma_drain, 0, &never, p.timeout_ns);
      }
    }
  } else {
    regs_increase<Shape::kSoftmax>();
    // ------------------------------------------------------------ softmax
    const int sub = warp >> 2;
    const int n_tiles = sub == 0 ? n0 : n1;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;                       // TMEM lane = row of the sub-tile
    const int sub_row0 = q_row0 + sub * kRowsPerSub;
    const int qi = sub_row0 + row;                        // query index within (b, h)
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS0 = tmem + lane_bits + sub * 128;
    const uint32_t tO = tmem + lane_bits + (sub == 0 ? Cfg::kColsO0 : Cfg::kColsO1);
    const float sl2 = p.scale_log2;

    // One thread of the sub-tile that visits every key tile of the range
    // (the second, unless it has no rows) releases the K/V ring slots.
    const bool releaser = (threadIdx.x & (kRowsPerSub - 1)) == 0 && n_tiles == nmax &&
                          (sub == SUBS - 1 || n1 == 0);
    float m = -INFINITY;  // running max (log2 domain) used as the exponent offset
    float l = 0.f;        // running sum of 2^(t - m)
    bool ok = true;
    int announced = 0;    // tiles whose P was announced to the issuing warp
    for (int j = 0; j < n_tiles; ++j) {
      // all lanes must agree before the warp-collective TMEM accesses
      // S of this tile: the sub-tile's buffer, or buffer j % 2 when double-buffered
      uint64_t* sbar = &bars->s_full[Cfg::kDoubleS ? (j & 1) : sub];
      const uint32_t s_phase = Cfg::kDoubleS ? (j >> 1) & 1 : j & 1;
      const uint32_t tS = Cfg::kDoubleS ? tS0 + (j & 1) * 128 : tS0;
      if (!__all_sync(0xffffffffu, wait_bar(sbar, s_phase, abort, p.timeout_ns))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (Cfg::kSoftmaxRelease && releaser) {
        // S_sub(j) complete: K_j and V_(j-1) have no reader left
        if (j > 0) bar_arrive(&bars->kv_empty[(2 * j - 1) % STAGES]);
        bar_arrive(&bars->kv_empty[(2 * j) % STAGES]);
      }
      // S of this tile, with the masks for keys past the end and keys after
      // the query under the causal mask
      uint32_t s[4][32];
      const int key0 = (t_begin + j) * kKeysPerTile;
      const bool tail = key0 + kKeysPerTile > p.Nk;
      const bool diag = CAUSAL && key0 + kKeysPerTile - 1 > sub_row0;
      auto load_s = [&]() {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
        // one wait covers the four loads; the others' registers are only
        // tied to it, so that nothing reads them before it
        tmem_ld_wait(s[0]);
#pragma unroll
        for (int c = 1; c < 4; ++c) regs_after_wait(s[c]);
        if (tail || diag) {
          const int lim = CAUSAL ? min(p.Nk, qi + 1) : p.Nk;  // keys [0, lim) are kept
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (key0 + c * 32 + e >= lim) s[c][e] = __float_as_uint(-INFINITY);
        }
      };

      // Offset decision: the row max (eight independent 3-input max chains
      // over the 128 scores, then a small tree); the offset moves to it when
      // it exceeds the current one by more than kRescaleLog2.
      float m_new = m;
      float alpha = 1.f;   // correction factor 2^(m - m'): 0 on the first tile, 1 when the offset stays
      auto decide = [&]() {
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
        m_new = move ? m_cand : m;
        alpha = !move ? 1.f : (m == -INFINITY ? 0.f : ex2_approx(m - m_new));
      };

      // P = 2^(s * scale*log2e - offset), packed pairwise; row sum in four packed accumulators
      uint32_t pk[2][32];
      float rs;
      auto exps = [&]() {
        const float off = m_new == -INFINITY ? 0.f : m_new;
        const float2 c2 = make_float2(sl2, sl2);
        const float2 o2 = make_float2(-off, -off);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 t = __ffma2_rn(make_float2(__uint_as_float(s[c][e]), __uint_as_float(s[c][e + 1])), c2, o2);
            const float2 pe = make_float2(ex2_approx(t.x), ex2_approx(t.y));
            acc[(e >> 1) & 3] = __fadd2_rn(acc[(e >> 1) & 3], pe);
            pk[c >> 1][(c & 1) * 16 + (e >> 1)] = pack_x2<F16>(pe.x, pe.y);
          }
        }
        const float2 a01 = __fadd2_rn(acc[0], acc[1]);
        const float2 a23 = __fadd2_rn(acc[2], acc[3]);
        const float2 a = __fadd2_rn(a01, a23);
        rs = a.x + a.y;
      };

      // Once the offset is finite, the exponentials go first with the
      // offset as it stands: the offset can only have to move when some
      // term exceeds 2^kRescaleLog2, and then the row sum does too.  Only
      // then (rarely, once the first tiles have set the offset) is the row
      // max taken, from S read again (P is not yet stored over it), and the
      // exponentials redone with the offset it decides.  Rows that do not
      // move redo the same arithmetic, so every row's offset and P are
      // those of taking the max first, but for a max within rounding of the
      // bound.
      load_s();
      const bool max_first = __any_sync(0xffffffffu, m == -INFINITY);
      bool decided = max_first;   // (otherwise alpha is 1 on every lane)
      if (max_first) decide();
      exps();
      if (!max_first && __any_sync(0xffffffffu, rs > kRescaleBound)) {
        load_s();
        decide();
        exps();
        decided = true;
      }
      tmem_st32(tS, pk[0]);
      tmem_st32(tS + 32, pk[1]);
      l = l * alpha + rs;
      m = m_new;

      // correction of the running output when some row of this warp moved its offset
      // (single-buffered order: the wait for S(j) above already follows P(j-1) V)
      const bool rescale = decided && j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
      // Double-buffered order, O announced after every P V: the wait for
      // P(j-1) V is taken before a rescale, and at the last tile in any case.
      // When S(j) has completed, P(j-2) V has too (it was issued first), so
      // o_done is at most one phase behind the one waited for here; after
      // the last tile's wait it is at most one behind the epilogue's.  (A
      // parity wait cannot tell a phase from the one two before it: without
      // the last tile's wait the epilogue could read O before P(n-2) V and
      // P(n-1) V have completed.)
      if (!Cfg::kOutDoneLast && j > 0 && (rescale || j == n_tiles - 1) &&
          !__all_sync(0xffffffffu, wait_bar(&bars->o_done[sub], (j - 1) & 1, abort, p.timeout_ns))) {
        ok = false;
      }
      if (rescale && ok) {
        {
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
      }
      tmem_st_wait();
      tc_fence_before_sync();
      if constexpr (Cfg::kNamedP) {
        __syncwarp();
        named_sync(sub == 0 ? kBarP0 : kBarP1, sub == 0 ? kBarP0Count : kBarP1Count);
      } else {
        bar_arrive(&bars->p_ready[Cfg::kDoubleS ? (j & 1) : sub]);
      }
      announced = j + 1;
      if (!ok) break;
    }
    if constexpr (Cfg::kNamedP) {
      // after an abort: the remaining phases, in step with the issuing warp
      __syncwarp();
      for (int j = announced; j < n_tiles; ++j)
        named_sync(sub == 0 ? kBarP0 : kBarP1, sub == 0 ? kBarP0Count : kBarP1Count);
    }

    // Outputs of this row: the final ones, or this key range's partial ones.
    const bool store = qi < p.Nq;
    const size_t row_id = (static_cast<size_t>(p.num_splits > 1 ? split : 0) * p.BH + bh) * p.Nq + qi;
    float* orow = (p.num_splits > 1 ? p.O_part : p.O) + row_id * D;
    float* lse_out = (p.num_splits > 1 ? p.LSE_part : p.LSE) + row_id;
    const bool half_out = p.o_half != 0 && p.num_splits == 1;
    if (n_tiles == 0 && store && p.num_splits > 1) {
      // no kept key in this range: contributes nothing to the merge
      for (int c = 0; c < D; c += 4) *reinterpret_cast<float4*>(orow + c) = make_float4(0.f, 0.f, 0.f, 0.f);
      *lse_out = -INFINITY;
    }
    if (n_tiles > 0 && ok) {
      // l == 0 only for a row whose every key in this range is masked
      if (store) *lse_out = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (!__all_sync(0xffffffffu,
                      wait_bar(&bars->o_done[sub], Cfg::kOutDoneLast ? 0u : (n_tiles - 1) & 1, abort,
                               p.timeout_ns))) {
        ok = false;
      } else {
        tc_fence_after_sync();
        // O / l is written into shared memory as 128-byte-swizzled boxes,
        // which one thread stores with TMA; rows past Nq fall outside the map
        // and are dropped.  fp32 O is staged in two column halves of D/2
        // (boxes of 32 columns), O in the input type all at once (boxes of 64
        // columns).  The first half goes to this sub-tile's Q buffer (every S
        // MMA that read it has completed).  The second half of the sub-tile(s)
        // whose last P V is the CTA's last MMA goes to K/V ring slot `sub`,
        // free once every MMA has completed (no load is in flight by then),
        // so that both halves are staged without waiting for the first
        // stores; otherwise it reuses the Q buffer once those have read it.
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const bool use_ring = n_tiles == nmax;
        const int zrow = (p.num_splits > 1 ? split * p.BH : 0) + bh;
        const bool leader = (threadIdx.x & (kRowsPerSub - 1)) == 0;
        const int parts = half_out ? 1 : 2;   // column halves staged one after the other
        for (int r = 0; r < parts && ok; ++r) {
          if (r > 0) {
            uint64_t* free_bar = use_ring ? &bars->mma_drain : &bars->stage_free[sub];
            if (!__all_sync(0xffffffffu, wait_bar(free_bar, 0, abort, p.timeout_ns))) {
              ok = false;
              break;
            }
            if (use_ring) tc_fence_after_sync();
          }
          uint8_t* stage = (r > 0 && use_ring ? sKV : sQ) + sub * TILE;
          const uint32_t stage_row = smem_addr(stage) + row * 128;
#pragma unroll
          for (int b = 0; b < D / 64; ++b) {
            const uint32_t box = stage_row + b * 16384;
            if (!half_out) {
              uint32_t o[32];
              tmem_ld32(tO + r * (D / 2) + 32 * b, o);
              tmem_ld_wait(o);
#pragma unroll
              for (int u = 0; u < 8; ++u)
                st_shared_v4(box + ((u ^ (row & 7)) << 4), __float_as_uint(__uint_as_float(o[4 * u]) * inv_l),
                             __float_as_uint(__uint_as_float(o[4 * u + 1]) * inv_l),
                             __float_as_uint(__uint_as_float(o[4 * u + 2]) * inv_l),
                             __float_as_uint(__uint_as_float(o[4 * u + 3]) * inv_l));
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
              for (int u = 0; u < 8; ++u)
                st_shared_v4(box + ((u ^ (row & 7)) << 4), h[4 * u], h[4 * u + 1], h[4 * u + 2], h[4 * u + 3]);
            }
          }
          fence_proxy_async_shared();
          bar_arrive(&bars->staged[sub]);
          if (leader) {
            if (!wait_bar(&bars->staged[sub], r & 1, abort, p.timeout_ns)) {
              ok = false;
            } else {
#pragma unroll
              for (int b = 0; b < D / 64; ++b)
                tma_store_3d(&tm_o, stage + b * 16384, half_out ? 64 * b : r * (D / 2) + 32 * b, sub_row0, zrow);
              bulk_commit();
              if (r + 1 < parts && !use_ring) {
                bulk_wait_read();
                bar_arrive(&bars->stage_free[sub]);
              }
            }
          }
          ok = __all_sync(0xffffffffu, ok);
        }
        // The stores must have read the staged O before the CTA exits (its
        // shared memory goes away); their global writes complete with the grid.
        if (leader) bulk_wait_read();
      }
    }
    if (!ok) raise_abort(abort, p.status);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace fa2dev
