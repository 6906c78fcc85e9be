// FlashAttention-2 forward on sm_103a: TMA-fed tiles, tcgen05 MMAs with TMEM
// accumulators and an online softmax.  Work unit = (pair of 128-row query
// tiles, head [, key split or sequence]); CTAs are persistent and take units
// from the hardware scheduler (cluster launch control).
//
// Method: "Revolutionizing Web-Based AI: How a Plain JavaScript Prototype
// Paved the Way for High-Performance WebGPU Flash Attention 2", section
// "Translating to WGSL and Optimizing Passes" (forward-pass bullet): one work
// unit per (batch, head, query tile) walks K and V in blocks, keeps the
// online-softmax state (running max m, running sum l) in registers and never
// materialises the N x N score matrix; section "Memory Bandwidth Optimization"
// (softmax reduction computed incrementally).  The per-row log-sum-exp is
// saved for the backward pass (same article, backward-pass bullet).
//
// GB300 design.  Two query tiles (A: rows q0..q0+127, B: q0+128..q0+255)
// share every K/V tile, so the tensor core alternates between them while the
// other tile's softmax runs:
//   warps 0-3  softmax of tile A   (thread t owns row t = TMEM lane t)
//   warps 4-7  softmax of tile B
//   warp  8    TMA producer: Q_A, Q_B per unit, K / V tiles through one 3-slot ring
//   warp  9    MMA issuer for tile A (one thread) + TMEM owner
//   warp 10    MMA issuer for tile B (one thread)
// One issuer per tile, so that waiting on one tile's MMA never delays the
// other tile's; ring slots are released once both issuers are done with them.
// TMEM columns: S_A [0,128), S_B [128,256), O_A and O_B after them (all 512).
// P_X goes from the softmax registers to shared memory (128 x 128 16-bit
// weights per tile, the K-major A operand of O_X += P_X V_j), so S_X(j+1)
// can be computed into S_X as soon as the softmax has read S_X(j) into
// registers, while the exponentials of tile j still run: the chain
// S -> softmax -> P V -> S of one tile no longer serialises the tensor core.
// The shared memory that takes (2 x 32 KB) comes from the K/V staging: K and
// V share three 32 KB slots, filled in the order the MMAs use them (K_0, K_1,
// V_0, K_2, V_1, ...).  P V runs on fp16 operands, with V read from an fp16
// copy that fa2_v_to_f16_kernel writes before the forward kernel runs: fp16
// keeps three more significant bits than bf16, and with bf16 weights their
// rounding alone moves O by up to about 0.2 % on rows dominated by a few
// keys.  A K/V head holding a finite value beyond the fp16 range is copied
// scaled by a power of two, which the epilogue multiplies back.  The split-KV
// form (decoding), whose time is the single read of the cache, runs P V in
// bf16 on V itself.  A barrier wait costs well over a hundred cycles even
// when its phase has completed, so waits that are usually already satisfied
// are tested early without blocking and only waited on when the test failed.
// The reference value m that the exponentials subtract is raised only when a
// tile's row max exceeds it by more than a slack (15 or 8 log2 units), so the
// weights stay below 2^slack and O is rescaled in TMEM (for the whole
// warp) only on those rare tiles.  The softmax arithmetic runs on
// packed fp32 pairs (f32x2 FMA/ADD/MUL) and 3-input max to halve its
// instruction count.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "tiles.cuh"

namespace fa2 {

__device__ int g_fwd_status;

namespace {

constexpr int kFwdThreads = 352;
// Readers of each scheduler response: the producer, the two MMA issuers and
// the eight softmax warps.
constexpr int kSchedReaders = 11;
constexpr uint32_t kTmemCols = 512;
// A row's reference max is raised only when a tile's max exceeds it by more
// than the slack (log2 units): weights 2^(s - m) then stay below 2^slack,
// inside fp16 (65504 > 2^15) and fp32 range, and the result is the same
// softmax up to rounding.  fp16 weights keep their 11 significant bits at
// any magnitude, so their slack is the widest fp16 allows (fewer O rescales
// on sharply peaked rows: +1.5 % on the large-logit stress workload, same
// error); bf16 weights (split-KV form) keep 8, beyond which a row's weight
// drifts into weights whose bf16 rounding the normaliser does not see.
constexpr float kRescaleSlackF16 = 15.f, kRescaleSlackBf16 = 8.f;

enum FwdBar {
  kBarQFull = 0,        // +tile (A, B)
  kBarQEmpty = 2,       // +tile: the tile's issuer is done with its Q tile of a unit
  kBarKVFull = 4,       // +ring slot (3)
  kBarKVEmpty = 7,      // +ring slot, one arrival per issuer
  kBarSFull = 10,       // +tile
  kBarSRead = 12,       // +tile, 4 warp arrivals: S_x is in registers, the next S may overwrite it
  kBarPFull = 14,       // +tile, 4 warp arrivals: P_x is in shared memory
  kBarPVDone = 16,      // +tile
  kBarDrain = 18,       // +tile
  kBarSchedFull = 20,   // +slot (2): scheduler response landed (16 transaction bytes)
  kBarSchedEmpty = 22,  // +slot: every role has read the response (kSchedReaders arrivals)
  kNumFwdBars = 24,
};

// K and V tiles share one ring of three slots, loaded in the order the MMAs
// use them: K_0, then (K_j, V_{j-1}) for j = 1 .. n-1, then V_{n-1}.  Ring
// position of a unit's K_j / V_j (n K/V tiles in the unit).
__device__ __forceinline__ int ring_pos_k(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int ring_pos_v(int j, int n) { return j + 1 < n ? 2 * j + 2 : 2 * n - 1; }
constexpr int kRingSlots = 3;

template <int D>
struct FwdCfg {
  using T = HeadDim<D>;
  static constexpr int kCols = D < 32 ? 32 : D;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128;
  static constexpr uint32_t kColO0 = 256, kColO1 = 256 + kCols;
  static constexpr int kQ = 0;  // Q_A, Q_B
  static constexpr int kKV = kQ + 2 * T::kTileBytes;  // K/V ring
  // P_A, P_B: 128 x 128 16-bit weights each, K-major (Square layout), the A
  // operand of O += P V.  A softmax warp's 32 rows of P_x also stage its O
  // rows for the TMA stores (32 rows x 64 columns = 4 KB per half, D >= 64).
  static constexpr int kP = kKV + kRingSlots * T::kTileBytes;
  static constexpr int kPBytes = kTileRows * kTileRows * 2;
  static constexpr bool kTmaOut = D >= 64;
  static constexpr int kBars = kP + 2 * kPBytes;
  static constexpr int kSched = (kBars + kNumFwdBars * 8 + 15) / 16 * 16;  // 2 x 16-byte responses
  static constexpr int kTmemSlot = kSched + 32;
  static constexpr int kUsed = kTmemSlot + 16;
  // +1024 so the base can be rounded up to a 1024-byte boundary; at least
  // 116 KB so that a single CTA (and its 512 TMEM columns) occupies an SM.
  static constexpr int kBytes = (kUsed + 1024) > 116 * 1024 ? (kUsed + 1024) : 116 * 1024;
};

// kSquare: the plain prefill case (M = Nq = Nk, one split), where a row's
// query index is the row itself and the causal offset is 0.  kGeneral:
// row-head form with Nq != Nk and key splits.  kVarlen: packed
// variable-length batch (per-sequence lengths from cu_q / cu_k).
enum FwdMode : int { kSquare = 0, kGeneral = 1, kVarlen = 2 };

// One work unit: a pair of 128-row query tiles of one row-head, for one key
// split (or one sequence of a variable-length batch).
struct FwdUnit {
  bool valid;                // false: nothing to do (varlen: past the sequence, or bad offsets)
  int rh, rh_kv, q0, split;  // row-head, its K/V head, first row of the pair, key split
  int M, Nk, off;            // rows, keys, causal offset (query i sees key j iff j <= i + off)
  int q_base, k_base;        // first TMA row of the unit's queries / keys (varlen offsets)
  int jb;                    // first K/V tile of the split
  int cnt[2], imin[2];       // K/V tiles each row tile visits; smallest query index of the tile
};

// Unit u, in the order CTAs take them: key split or sequence slowest, then
// groups of heads_per_group row-heads (a group's K/V rows stay in L2 while it
// runs), then pairs heaviest first (causal work grows with the pair index),
// then row-heads.  Row r of row-head rh is query r % Nq; the row-head reads
// K/V head rh / kvdiv.
template <bool CAUSAL, int MODE>
__device__ __forceinline__ FwdUnit fwd_unit(const FwdProblem& p, int u, int num_row_tiles, int num_pairs,
                                            int* status) {
  FwdUnit w;
  const int per_split = num_pairs * p.RH;
  const int outer = u / per_split;
  const int local = u % per_split;
  const int per_group = p.heads_per_group * num_pairs;
  const int hg0 = local / per_group * p.heads_per_group;
  const int hg = min(p.heads_per_group, p.RH - hg0);
  const int pair = num_pairs - 1 - (local % per_group) / hg;
  w.valid = true;
  w.rh = hg0 + (local % per_group) % hg;
  w.rh_kv = w.rh / p.kvdiv;
  w.q0 = pair * 2 * kTileRows;
  w.split = MODE == kVarlen ? 0 : outer;
  w.M = p.M;
  w.Nk = p.Nk;
  w.off = MODE == kGeneral ? p.Nk - p.Nq : 0;
  w.q_base = 0;
  w.k_base = 0;
  if constexpr (MODE == kVarlen) {
    const int sq = p.cu_q[outer], eq = p.cu_q[outer + 1], sk = p.cu_k[outer], ek = p.cu_k[outer + 1];
    if (!(0 <= sq && sq <= eq && eq <= p.total_q && eq - sq <= p.M && 0 <= sk && sk <= ek && ek <= p.total_k &&
          ek - sk <= p.Nk)) {
      if (threadIdx.x == 0) atomicCAS(status, kDevOk, kDevBadSeqlens);
      w.valid = false;
    }
    w.M = eq - sq;
    w.Nk = ek - sk;
    w.off = w.Nk - w.M;
    w.q_base = sq;
    w.k_base = sk;
    if (w.q0 >= w.M) w.valid = false;  // the pair lies past this sequence's queries
  }
  const int num_kv_tiles = (w.Nk + kTileRows - 1) / kTileRows;
  w.jb = w.split * p.tiles_per_split;
  const int je = min(num_kv_tiles, w.jb + p.tiles_per_split);
  if constexpr (MODE == kSquare) {
    // Square problem: tile A sees tiles 0..2*pair (causal), tile B one more.
    w.cnt[0] = CAUSAL ? 2 * pair + 1 : num_kv_tiles;
    w.cnt[1] = 2 * pair + 1 >= num_row_tiles ? 0 : (CAUSAL ? 2 * pair + 2 : num_kv_tiles);
    w.imin[0] = w.q0;
    w.imin[1] = w.q0 + kTileRows;
  } else {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int rx0 = w.q0 + x * kTileRows;
      w.cnt[x] = 0;
      w.imin[x] = 0;
      if (w.valid && rx0 < w.M) {
        const int rlast = min(rx0 + kTileRows - 1, w.M - 1);
        const bool one_head = MODE == kVarlen || rx0 / p.Nq == rlast / p.Nq;
        const int i_max = MODE == kVarlen ? rlast : (one_head ? rlast % p.Nq : p.Nq - 1);
        w.imin[x] = MODE == kVarlen ? rx0 : (one_head ? rx0 % p.Nq : 0);
        // causal: the last key any row of the tile sees is i_max + off (< 0: none)
        const int kv_end = !CAUSAL ? num_kv_tiles
                                   : (i_max + w.off < 0 ? 0 : min(num_kv_tiles, (i_max + w.off) / kTileRows + 1));
        w.cnt[x] = max(0, min(je, kv_end) - w.jb);
      }
    }
  }
  return w;
}

// The unit after a CTA's n-th unit: wait for the n-th scheduler response
// (slot n & 1), decode it (-1: no unit left) and, if `release`, mark the slot
// read.  Every reader calls this once per unit, in unit order.
__device__ __forceinline__ int next_unit(uint64_t* bars, const uint8_t* sched, int n, bool release, int* status,
                                         bool& ok) {
  const int slot = n & 1;
  if (!(ok = mbar_wait(&bars[kBarSchedFull + slot], (n >> 1) & 1, status))) return -1;
  int u = clc_cancelled_block_x(sched + 16 * slot);
  if (u >= static_cast<int>(gridDim.x)) {  // never expected: refuse rather than index past the grid
    atomicCAS(status, kDevOk, kDevBadSchedule);
    u = -1;
  }
  if (release) mbar_arrive(&bars[kBarSchedEmpty + slot]);
  return u;
}

// Persistent with the hardware's dynamic order: the grid has one CTA per
// unit, but a running CTA takes over the next not-yet-started CTA's unit
// (cluster launch control) instead of exiting, for as long as there is one.
// Units still start in blockIdx order (heaviest first), and all barrier
// phases run on across a CTA's units, so the producer loads the next unit's
// Q / K / V and the issuers start its first S while the softmax warps are
// still writing the previous unit's O.  The producer requests the next unit
// once it has issued every load of the current one.
template <int D, bool CAUSAL, int MODE>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa2_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const FwdProblem p, float scale_log2) {
  // P V on fp16 operands (tm_v is then the fp16 copy of V), except in the
  // split-KV form.
  constexpr bool kF16 = MODE != kGeneral;
  using T = HeadDim<D>;
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kTmemSlot);
  uint8_t* sched = smem + C::kSched;
  int* status = &g_fwd_status;

  const int warp = warp_id();
  const int lane = lane_id();
  const int num_row_tiles = (p.M + kTileRows - 1) / kTileRows;
  const int num_pairs = (num_row_tiles + 1) / 2;

  if (threadIdx.x == 8 * 32) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kBarQFull + s], 1);
      mbar_init(&bars[kBarQEmpty + s], 1);
      mbar_init(&bars[kBarSchedFull + s], 1);
      mbar_init(&bars[kBarSchedEmpty + s], kSchedReaders);
      mbar_init(&bars[kBarSFull + s], 1);
      mbar_init(&bars[kBarSRead + s], 4);
      mbar_init(&bars[kBarPFull + s], 4);
      mbar_init(&bars[kBarPVDone + s], 1);
      mbar_init(&bars[kBarDrain + s], 1);
    }
    for (int s = 0; s < kRingSlots; ++s) {
      mbar_init(&bars[kBarKVFull + s], 1);
      mbar_init(&bars[kBarKVEmpty + s], 2);
    }
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int g = 0;             // ring loads so far (slot g % 3, use g / 3)
      int qn0 = 0, qn1 = 0;  // Q_A / Q_B tiles loaded so far
      int last_use[kRingSlots] = {-1, -1, -1};  // last use armed per slot
      bool ok = true;
      int pending = -1;  // scheduler request issued but not yet read here
#pragma unroll 1
      for (int n = 0, u = static_cast<int>(blockIdx.x); ok && u >= 0; ++n) {
        do {
        const FwdUnit w = fwd_unit<CAUSAL, MODE>(p, u, num_row_tiles, num_pairs, status);
        const int n_kv = max(w.cnt[0], w.cnt[1]);
        if (!w.valid || n_kv == 0) break;
        // Q_x smem is free once issuer x's last S of its previous unit is
        // done.  Order: Q_A, K_0, Q_B, then the rest of the ring, so tile A
        // can start the unit while tile B still finishes the last one.
        auto load_q = [&](int x) -> bool {
          int& qn = x ? qn1 : qn0;
          if (qn >= 1 && !mbar_wait(&bars[kBarQEmpty + x], (qn - 1) & 1, status)) return false;
          mbar_arrive_expect_tx(&bars[kBarQFull + x], T::kTileBytes);
          for (int b = 0; b < T::kNumBoxes; ++b)
            tma_load_3d(smem + C::kQ + x * T::kTileBytes + b * T::kBoxBytes, &tm_q, &bars[kBarQFull + x],
                        b * T::kBoxCols, w.q_base + w.q0 + x * kTileRows, w.rh);
          ++qn;
          return true;
        };
        // K_j (v = false) or V_j into the next ring slot, once both issuers
        // have released the slot's previous tile.
        auto load_kv = [&](bool v, int j) -> bool {
          const int slot = g % kRingSlots, use = g / kRingSlots;
          if (use >= 1 && !mbar_wait(&bars[kBarKVEmpty + slot], (use - 1) & 1, status)) return false;
          mbar_arrive_expect_tx(&bars[kBarKVFull + slot], T::kTileBytes);
          for (int b = 0; b < T::kNumBoxes; ++b)
            tma_load_3d(smem + C::kKV + slot * T::kTileBytes + b * T::kBoxBytes, v ? &tm_v : &tm_k,
                        &bars[kBarKVFull + slot], b * T::kBoxCols, w.k_base + (w.jb + j) * kTileRows, w.rh_kv);
          last_use[slot] = use;
          ++g;
          return true;
        };
        if (w.cnt[0] > 0 && !(ok = load_q(0))) break;
        if (!(ok = load_kv(false, 0))) break;
        if (w.cnt[1] > 0 && !(ok = load_q(1))) break;
#pragma unroll 1
        for (int j = 1; j < n_kv; ++j)
          if (!(ok = load_kv(false, j) && load_kv(true, j - 1))) break;
        if (!ok) break;
        if (!(ok = load_kv(true, n_kv - 1))) break;
        } while (false);
        if (!ok) break;
        // Every load of this unit is issued (about a K/V tile ahead of the
        // MMAs): ask for the next unit now, late enough that CTAs which
        // finish first take the remaining units.  Slot n & 1 is free once
        // every reader has taken request n - 2's answer.
        if (n >= 2 && !(ok = mbar_wait(&bars[kBarSchedEmpty + (n & 1)], ((n >> 1) - 1) & 1, status))) break;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[kBarSchedFull + (n & 1)], 16);
        clc_try_cancel(sched + 16 * (n & 1), &bars[kBarSchedFull + (n & 1)]);
        pending = n;
        u = next_unit(bars, sched, n, true, status, ok);
        pending = -1;
      }
      // A scheduler response still on its way must land before the CTA exits.
      if (pending >= 0) mbar_wait(&bars[kBarSchedFull + (pending & 1)], (pending >> 1) & 1, status);
      // Never leave the CTA with a TMA write still landing in shared memory:
      // wait for the last completion of every full barrier that was armed.
      if (qn0 >= 1) mbar_wait(&bars[kBarQFull + 0], (qn0 - 1) & 1, status);
      if (qn1 >= 1) mbar_wait(&bars[kBarQFull + 1], (qn1 - 1) & 1, status);
      for (int s = 0; s < kRingSlots; ++s)
        if (last_use[s] >= 0) mbar_wait(&bars[kBarKVFull + s], last_use[s] & 1, status);
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuer of tile x
    if (lane == 0) {
      const int x = warp - 9;
      constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false, false);  // Q (K-major) x K (K-major)
      // P (K-major) x V (MN-major)
      constexpr uint32_t kIdescO = kF16 ? make_idesc_f16(128, D, false, true) : make_idesc_bf16(128, D, false, true);
      const uint32_t sQ0 = smem_u32(smem + C::kQ), sKV0 = smem_u32(smem + C::kKV);
      const uint32_t sP = smem_u32(smem + C::kP) + x * C::kPBytes;
      const uint32_t tSx = tmem + (x ? C::kColS1 : C::kColS0);
      const uint32_t tOx = tmem + (x ? C::kColO1 : C::kColO0);
      auto full = [&](int pos) {  // wait for the ring tile at global position pos
        return mbar_wait(&bars[kBarKVFull + pos % kRingSlots], (pos / kRingSlots) & 1, status);
      };
      // S_x = Q_x K^T, K in ring position pos.
      auto issue_s = [&](int pos) {
        uint32_t sQ = sQ0, sKV = sKV0;
        opaque(sQ);
        opaque(sKV);
        const uint32_t qb = sQ + x * T::kTileBytes, kb = sKV + (pos % kRingSlots) * T::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tSx, T::kmajor_desc(qb, kk), T::kmajor_desc(kb, kk), kIdescS, kk > 0 ? 1u : 0u);
        mma_commit(&bars[kBarSFull + x]);
        mma_commit(&bars[kBarKVEmpty + pos % kRingSlots]);
      };
      // O_x (+)= P_x V, V in ring position pos.
      auto issue_pv = [&](int pos, bool first) {
        uint32_t sKV = sKV0;
        opaque(sKV);
        const uint32_t vb = sKV + (pos % kRingSlots) * T::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileRows / 16; ++kk)
          mma_bf16_ss(tOx, Square::kmajor_desc(sP, kk), T::mnmajor_desc(vb, kk), kIdescO,
                      (!first || kk > 0) ? 1u : 0u);
        mma_commit(&bars[kBarPVDone + x]);
        mma_commit(&bars[kBarKVEmpty + pos % kRingSlots]);
      };
      int g = 0;   // ring position of the current unit's first tile (same count as the producer's)
      int k = 0;   // S_x / P_x / PV_x issued so far (phase k & 1)
      int qn = 0;  // units whose Q_x tile was loaded so far
      bool ok = true;
#pragma unroll 1
      for (int n = 0, u = static_cast<int>(blockIdx.x); ok && u >= 0; ++n) {
        do {
        const FwdUnit w = fwd_unit<CAUSAL, MODE>(p, u, num_row_tiles, num_pairs, status);
        const int n_kv = max(w.cnt[0], w.cnt[1]);
        if (!w.valid || n_kv == 0) break;
        const int nx = x ? w.cnt[1] : w.cnt[0];  // (selects keep the struct in registers)
        // Order: S(0); then per tile j: S(j+1) as soon as the softmax has
        // read S(j) into registers, then PV(j) once P(j) is in shared memory.
        // S(k) overwrites S_x: it waits for the softmax to have read S(k-1).
        if (nx > 0) {
          if (!(ok = mbar_wait(&bars[kBarQFull + x], qn & 1, status))) break;
          ++qn;
          if (!(ok = (k == 0 || mbar_wait(&bars[kBarSRead + x], (k - 1) & 1, status)) && full(g))) break;
          tc_fence_after();
          issue_s(g);
          if (nx == 1) mma_commit(&bars[kBarQEmpty + x]);  // last use of Q_x in this unit
        }
#pragma unroll 1
        for (int j = 0; j < nx; ++j) {
          if (j + 1 < nx) {
            const int pk = g + ring_pos_k(j + 1);
            if (!(ok = mbar_wait2(&bars[kBarSRead + x], k & 1, &bars[kBarKVFull + pk % kRingSlots], (pk / kRingSlots) & 1, status))) break;
            tc_fence_after();
            issue_s(pk);
            if (j + 2 == nx) mma_commit(&bars[kBarQEmpty + x]);
          }
          const int pv = g + ring_pos_v(j, n_kv);
          if (!(ok = mbar_wait2(&bars[kBarKVFull + pv % kRingSlots], (pv / kRingSlots) & 1, &bars[kBarPFull + x], k & 1, status))) break;
          tc_fence_after();
          issue_pv(pv, j == 0);
          ++k;
        }
        if (!ok) break;
        // K/V tiles this query tile does not visit (those from K_nx on, all
        // at ring positions after every tile it used except V_{nx-1}):
        // release them in ring order, each after taking its full phase (so
        // that this issuer's next wait on the slot is never two phases ahead
        // of the loads; the load also implies that the slot's previous use
        // has been released) and after the slot's previous phase is seen
        // complete.
#pragma unroll 1
        for (int pos = g + (nx == 0 ? 0 : ring_pos_k(nx)); pos < g + 2 * n_kv; ++pos) {
          bool mine;  // is pos a tile this issuer used?
          const int rel = pos - g;
          if (rel == 0) mine = nx > 0;
          else if (rel == 2 * n_kv - 1) mine = nx == n_kv;  // V_{n-1}
          else if (rel & 1) mine = (rel + 1) / 2 < nx;      // K_{(rel+1)/2}
          else mine = (rel - 2) / 2 < nx;                   // V_{(rel-2)/2}
          if (mine) continue;
          const int slot = pos % kRingSlots, use = pos / kRingSlots;
          if (!(ok = full(pos))) break;
          if (use >= 1 && !(ok = mbar_wait(&bars[kBarKVEmpty + slot], (use - 1) & 1, status))) break;
          mbar_arrive(&bars[kBarKVEmpty + slot]);
        }
        g += 2 * n_kv;
        } while (false);
        if (!ok) break;
        u = next_unit(bars, sched, n, true, status, ok);
      }
      // Wait for every MMA this thread issued before TMEM can be released.
      mma_commit(&bars[kBarDrain + x]);
      mbar_wait(&bars[kBarDrain + x], 0, status);
    }
  } else {
    // ------------------------------------------------------------ softmax (tile x)
    const int x = warp >> 2;
    const int r = threadIdx.x & 127;  // row within the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (x ? C::kColS1 : C::kColS0);
    const uint32_t tO = tmem + lane_base + (x ? C::kColO1 : C::kColO0);
    const uint32_t sP = smem_u32(smem + C::kP) + x * C::kPBytes;
    const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
    int k = 0;  // S_x tiles consumed so far
    // Softmax warps w (tile A) and w + 4 (tile B) share an SMSP and its
    // MUFU.  With P in TMEM (an earlier design) they took turns at the
    // exponentials, passing a token per SMSP, and that was 4-11 % faster
    // than letting the loops overlap; with P in shared memory the turns only
    // made one tile wait for the other, and the forward is 1-3 % faster
    // without them.
    bool ok = true;
#pragma unroll 1
    for (int n = 0, u = static_cast<int>(blockIdx.x); ok && u >= 0; ++n) {
      do {
      const FwdUnit w = fwd_unit<CAUSAL, MODE>(p, u, num_row_tiles, num_pairs, status);
      if (!w.valid) break;
      const int nx = x ? w.cnt[1] : w.cnt[0];  // (selects keep the struct in registers)
      const int q_row = w.q0 + x * kTileRows + r;              // row in the row-head
      const int qi = MODE == kGeneral ? q_row % p.Nq : q_row;  // its query index
      const int imin_x = x ? w.imin[1] : w.imin[0];
      const int off = w.off, Nk = w.Nk;
      // V scale of the unit's K/V head (read now, used by the epilogue)
      const float v_scale = (kF16 && p.v_scale != nullptr) ? __ldg(p.v_scale + w.rh_kv) : 1.f;
      float m = -INFINITY;  // reference max, log2 units (scores * scale * log2 e); row max - m <= slack
      float l = 0.f;        // running sum of 2^(x - m) (fp32 weights: the LSE)
      float lo = 0.f;       // the same with each tile's largest weight as 16-bit (normalises O)
#pragma unroll 1
      for (int j = 0; j < nx; ++j, ++k) {
        if (!(ok = mbar_wait(&bars[kBarSFull + x], k & 1, status))) break;
        tc_fence_after();
        float s[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<float(*)[32]>(s + 32 * c));
        tmem_wait_ld();
        // S_x is in registers: the issuer may compute the next S into it.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarSRead + x]);

        const int kv0 = (w.jb + j) * kTileRows;
        if ((CAUSAL && (MODE != kSquare ? kv0 + kTileRows - 1 > imin_x + off : j == nx - 1)) || kv0 + kTileRows > Nk) {
          int lim = Nk - kv0;                                  // keys >= Nk do not exist
          if (CAUSAL) lim = min(lim, qi + off - kv0 + 1);      // key j visible iff j <= query + off
#pragma unroll
          for (int e = 0; e < 128; ++e)
            if (e >= lim) s[e] = -INFINITY;
        }
        // Row max: 8 independent chains of 3-input max.
        float mx8[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          // chain c covers columns c, c + 8, ..., c + 120
          float v = fmax3(s[c], s[c + 8], s[c + 16]);
#pragma unroll
          for (int i = 24; i <= 104; i += 16) v = fmax3(v, s[c + i], s[c + i + 8]);
          mx8[c] = fmaxf(v, s[c + 120]);
        }
        const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
        // Raise m to this tile's max only when that exceeds it by more than
        // the slack (always on the first tile that sees a key).
        const float mt = mx * scale_log2;
        const bool grow = mt > m + (kF16 ? kRescaleSlackF16 : kRescaleSlackBf16);
        const float m_new = grow ? mt : m;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // (no key seen yet)
        const float alpha = ex2_approx(m - m_use);
        // The tile's largest weight (computed exactly as the loop below does)
        // and its 16-bit rounding error.  With the reference max lagging the
        // row max, that weight is not a power of two, and the PV MMA sees it
        // rounded; normalising O by a sum that carries the same rounding
        // keeps O the weighted mean of V that the MMA computed.
        const float pmax = ex2_approx(fmaf(mx, scale_log2, -m_use));
        const float dpmax = (kF16 ? f16lo_to_f32(pack_f16x2(pmax, 0.f)) : unpack_bf16x2(pack_bf16x2(pmax, 0.f)).x) - pmax;
        // P_x is free once PV(k-1), which reads it, has completed (that also
        // makes O_x stable for the rescale below); at a unit's first tile,
        // once this warp's O stores of the previous unit have read their
        // staging rows (this warp's rows of P_x).
        bool pv_seen = k == 0 || mbar_test_wait(&bars[kBarPVDone + x], (k - 1) & 1);
        if (C::kTmaOut && j == 0) {
          if (lane == 0) bulk_wait_group_read0();
          __syncwarp();
        }

        // P = 2^(s * scale_log2 - m) on packed pairs; 4 independent pair sums.
        const uint64_t negm2 = f2_pack(-m_use, -m_use);
        // P goes to shared memory (row r of P_x) 32 columns at a time.
        uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int e = 32 * c + 2 * i;
            const float2 xx = f2_unpack(ffma2(f2_pack(s[e], s[e + 1]), scale2, negm2));
            const float p0 = ex2_approx(xx.x), p1 = ex2_approx(xx.y);
            acc[i & 3] = fadd2(acc[i & 3], f2_pack(p0, p1));
            pk[i] = kF16 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
          }
          if (c == 0 && !pv_seen && !(ok = mbar_wait(&bars[kBarPVDone + x], (k - 1) & 1, status))) break;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            store_square_chunk(sP, r, 4 * c + q, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
        if (!ok) break;
        const float2 a01 = f2_unpack(fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3])));
        const float rs = a01.x + a01.y;

        if (j >= 1 && __any_sync(0xffffffffu, grow)) {
          const uint64_t alpha2 = f2_pack(alpha, alpha);
          if constexpr (D >= 32) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              float o[32];
              tmem_ld32(tO + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                const float2 rr = f2_unpack(fmul2(f2_pack(o[e], o[e + 1]), alpha2));
                o[e] = rr.x;
                o[e + 1] = rr.y;
              }
              tmem_st32(tO + c * 32, o);
            }
          } else {
            float o[16];
            tmem_ld16(tO, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= alpha;
            tmem_st16(tO, o);
          }
          tmem_wait_st();
        }
        // P_x (shared memory, generic proxy) is read by the MMA (async proxy).
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarPFull + x]);
        l = l * alpha + rs;
        lo = lo * alpha + (rs + dpmax);
        m = m_new;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      // One split: O / l in bf16 and LSE.  Several splits: this split's O / l
      // and LSE in fp32 for the combine kernel.  A row that sees no key gets
      // O = 0, LSE = -inf.
      const bool valid = q_row < w.M;
      const bool partial = MODE == kGeneral && p.splits > 1;
      const int vrow = valid ? q_row : 0;
      // o_row: row of o (or o_part) in units of D elements; lse_idx: index into lse.
      size_t o_row, lse_idx;
      if constexpr (MODE == kVarlen) {
        o_row = static_cast<size_t>(w.q_base + vrow) * p.RH + w.rh;
        lse_idx = static_cast<size_t>(w.rh) * p.total_q + w.q_base + vrow;
      } else {
        o_row = (partial ? static_cast<size_t>(w.split) * p.RH + w.rh : static_cast<size_t>(w.rh)) * p.M + vrow;
        lse_idx = o_row;
      }
      if (nx == 0) {
        if (!valid) break;
        if (partial) {
          float4* dst = reinterpret_cast<float4*>(p.o_part + o_row * D);
#pragma unroll
          for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          p.lse_part[o_row] = -INFINITY;
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + o_row * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
          p.lse[lse_idx] = -INFINITY;
        }
        break;
      }
      // The warp reads O (all lanes: tcgen05.ld is warp-wide) only after its
      // unit's last PV_x has completed; the next unit's first PV_x (which
      // overwrites O_x) waits for this warp's next P_x, so the read-out cannot
      // race it.
      if (!(ok = mbar_wait(&bars[kBarPVDone + x], (k - 1) & 1, status))) break;
      tc_fence_after();
      const float inv_l = lo > 0.f ? v_scale / lo : 0.f;
      // bf16 output leaves through shared memory and TMA stores, so the warp
      // does not wait for its rows to reach L2 (TMA drops the rows past M).
      // In a packed batch only a warp whose 32 rows all lie in the sequence
      // does so; the others store directly (their rows past the sequence
      // belong to the next one).
      const int row_w0 = w.q0 + x * kTileRows + (warp & 3) * 32;  // this warp's first row
      const bool tma_out = C::kTmaOut && !partial && (MODE != kVarlen || row_w0 + 32 <= w.M);
      if (tma_out) {
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          // this warp's 32 rows of P_x in 64-column box h (the last PV has read them)
          const uint32_t slice = sP + h * Square::kBoxBytes + (warp & 3) * 4096;
          float o[64];
          tmem_ld32(tO + 64 * h, *reinterpret_cast<float(*)[32]>(o));
          tmem_ld32(tO + 64 * h + 32, *reinterpret_cast<float(*)[32]>(o + 32));
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_shared_v4(slice + sw128_offset(lane, c), pack_bf16x2(o[8 * c + 0] * inv_l, o[8 * c + 1] * inv_l),
                         pack_bf16x2(o[8 * c + 2] * inv_l, o[8 * c + 3] * inv_l),
                         pack_bf16x2(o[8 * c + 4] * inv_l, o[8 * c + 5] * inv_l),
                         pack_bf16x2(o[8 * c + 6] * inv_l, o[8 * c + 7] * inv_l));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row_w0 < w.M) {
            tma_store_3d(&tm_o, slice, 64 * h, w.q_base + row_w0, w.rh);
            bulk_commit_group();
          }
        }
      }
      constexpr int kC = D >= 32 ? 32 : 16;
#pragma unroll
      for (int c = 0; c < D / kC && !tma_out; ++c) {
        float o[kC];
        if constexpr (kC == 32)
          tmem_ld32(tO + c * 32, o);
        else
          tmem_ld16(tO, o);
        tmem_wait_ld();
        if (valid) {
          if (partial) {
            float4* dst = reinterpret_cast<float4*>(p.o_part + o_row * D + c * kC);
#pragma unroll
            for (int q = 0; q < kC / 4; ++q)
              dst[q] = make_float4(o[4 * q] * inv_l, o[4 * q + 1] * inv_l, o[4 * q + 2] * inv_l, o[4 * q + 3] * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + o_row * D + c * kC);
#pragma unroll
            for (int q = 0; q < kC / 8; ++q)
              dst[q] = make_uint4(pack_bf16x2(o[8 * q + 0] * inv_l, o[8 * q + 1] * inv_l),
                                  pack_bf16x2(o[8 * q + 2] * inv_l, o[8 * q + 3] * inv_l),
                                  pack_bf16x2(o[8 * q + 4] * inv_l, o[8 * q + 5] * inv_l),
                                  pack_bf16x2(o[8 * q + 6] * inv_l, o[8 * q + 7] * inv_l));
          }
        }
      }
      // LSE in natural log of the scaled scores: ln 2 * (m + log2 l).
      if (valid) {
        const float lse_row = (m + log2f(l)) * 0.69314718055994531f;
        if (partial)
          p.lse_part[o_row] = lse_row;
        else
          p.lse[lse_idx] = lse_row;
      }
      } while (false);
      if (!ok) break;
      u = next_unit(bars, sched, n, false, status, ok);
      __syncwarp();
      if (lane == 0 && ok) mbar_arrive(&bars[kBarSchedEmpty + (n & 1)]);
    }
    // Every O store has read its slice and landed before the CTA exits.
    if (lane == 0) bulk_wait_group0();
    tc_fence_before();
  }

  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool CAUSAL>
int launch_fwd_t(const TmapSet& tm, FwdProblem p, float scale, cudaStream_t stream) {
  using C = FwdCfg<D>;
  const bool varlen = p.cu_q != nullptr;
  // The square form runs P V in fp16 and needs the fp16 copy of V: a square
  // problem without one (split-KV with one split and Nq = Nk) takes the
  // general form.  Packed batches come with the copy, or (no keys) never
  // read V.
  const bool general = p.v_scale == nullptr || p.splits > 1 || p.M != p.Nq || p.Nq != p.Nk;
  // Every row-head re-reads the K and V rows of its split.
  const int kv_rows = min(p.Nk, p.tiles_per_split * kTileRows);
  p.heads_per_group = heads_per_l2_group(static_cast<size_t>(kv_rows) * D * 4 / p.kvdiv, p.RH);
  auto kern = varlen    ? fa2_fwd_kernel<D, CAUSAL, kVarlen>
              : general ? fa2_fwd_kernel<D, CAUSAL, kGeneral>
                        : fa2_fwd_kernel<D, CAUSAL, kSquare>;
  if (int rc = ensure_max_smem(reinterpret_cast<const void*>(kern), C::kBytes)) return rc;
  const int num_row_tiles = (p.M + kTileRows - 1) / kTileRows;
  const int num_pairs = (num_row_tiles + 1) / 2;
  // One CTA per unit; running CTAs take over the units of CTAs that have
  // not started (cluster launch control), so at most one CTA per SM ever runs.
  const long long units = static_cast<long long>(num_pairs) * p.RH * (varlen ? p.batches : p.splits);
  const dim3 grid(static_cast<unsigned>(units > 0 ? units : 1));
  const float scale_log2 = scale * 1.44269504088896341f;
  // Square and packed problems read the fp16 copy of V.
  return launch_pdl(kern, grid, dim3(kFwdThreads), C::kBytes, stream, tm.q, tm.k, (general && !varlen) ? tm.v : tm.v16,
                    tm.o, p, scale_log2);
}

// V in fp16 for the P V MMA: one pass over V (16-byte loads and stores,
// grid-stride), exact for every bf16 value of magnitude below 2^16 (below
// 2^-14 fp16 keeps fewer significant bits: an absolute error under 2^-25;
// infinities and NaN carry over).  A finite value beyond the fp16 range
// (|v| > 65504) flags its K/V head for fa2_v_scale_kernel.
__global__ void __launch_bounds__(256) fa2_v_to_f16_kernel(const uint4* __restrict__ v, uint4* __restrict__ v16,
                                                           unsigned long long* __restrict__ flags,
                                                           unsigned long long call, long long n8, long long inner,
                                                           int heads) {
  griddep_wait();
  griddep_launch_dependents();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    const uint4 a = __ldg(v + i);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t h[4];
    bool big = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
      big |= (fabsf(lo) > 65504.f && fabsf(lo) < INFINITY) || (fabsf(hi) > 65504.f && fabsf(hi) < INFINITY);
      h[e] = pack_f16x2(lo, hi);
    }
    v16[i] = make_uint4(h[0], h[1], h[2], h[3]);
    if (big) flags[(i * 8 / inner) % heads] = call;
  }
}

// One CTA per K/V head: v_scale[h] = 1, or for a head flagged by
// fa2_v_to_f16_kernel the smallest power of two 2^k with
// max |v| / 2^k <= 2^15 (finite values), after rewriting that head's copy as
// fp16(v / 2^k) (exact scaling by a power of two).
__global__ void __launch_bounds__(256) fa2_v_scale_kernel(const __nv_bfloat16* __restrict__ v,
                                                          __half* __restrict__ v16,
                                                          const unsigned long long* __restrict__ flags,
                                                          float* __restrict__ scales, unsigned long long call,
                                                          long long rows, int d, long long row_stride,
                                                          long long head_stride) {
  griddep_wait();
  griddep_launch_dependents();
  const int h = blockIdx.x;
  if (flags[h] != call) {
    if (threadIdx.x == 0) scales[h] = 1.f;
    return;
  }
  const long long n = rows * d;
  const long long base = static_cast<long long>(h) * head_stride;
  auto at = [&](long long e) { return base + (e / d) * row_stride + e % d; };
  float mx = 0.f;
  for (long long e = threadIdx.x; e < n; e += blockDim.x) {
    const float a = fabsf(__bfloat162float(v[at(e)]));
    if (a < INFINITY) mx = fmaxf(mx, a);
  }
  __shared__ float red[32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) mx = fmaxf(mx, red[i]);
  int k = 0;
  while (ldexpf(mx, -k) > 32768.f) ++k;
  const float inv = ldexpf(1.f, -k);
  for (long long e = threadIdx.x; e < n; e += blockDim.x) {
    const long long i = at(e);
    v16[i] = __float2half_rn(__bfloat162float(v[i]) * inv);
  }
  if (threadIdx.x == 0) scales[h] = ldexpf(1.f, k);
}

// Small heads (rows * d <= kVHeadSmall): both steps above in one kernel, one
// CTA per K/V head (copy, then rescale the head if it held a value beyond
// the fp16 range), saving a launch where launches dominate.
constexpr long long kVHeadSmall = 64 * 1024;
__global__ void __launch_bounds__(256) fa2_v_to_f16_head_kernel(const __nv_bfloat16* __restrict__ v,
                                                               __half* __restrict__ v16,
                                                               float* __restrict__ scales, long long rows, int d,
                                                               long long row_stride, long long head_stride) {
  griddep_wait();
  griddep_launch_dependents();
  const int h = blockIdx.x;
  const int per_row = d / 8;
  const long long n8 = rows * per_row;
  const long long base = static_cast<long long>(h) * head_stride;
  auto at8 = [&](long long e8) { return base + (e8 / per_row) * row_stride + (e8 % per_row) * 8; };
  bool big = false;
  for (long long e8 = threadIdx.x; e8 < n8; e8 += blockDim.x) {
    const long long i = at8(e8);
    const uint4 a = *reinterpret_cast<const uint4*>(v + i);
    const uint32_t w[4] = {a.x, a.y, a.z, a.w};
    uint32_t hv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
      big |= (fabsf(lo) > 65504.f && fabsf(lo) < INFINITY) || (fabsf(hi) > 65504.f && fabsf(hi) < INFINITY);
      hv[e] = pack_f16x2(lo, hi);
    }
    *reinterpret_cast<uint4*>(v16 + i) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
  }
  if (!__syncthreads_or(big)) {
    if (threadIdx.x == 0) scales[h] = 1.f;
    return;
  }
  // the rare head: the same rescaling as fa2_v_scale_kernel
  const long long n = rows * d;
  auto at = [&](long long e) { return base + (e / d) * row_stride + e % d; };
  float mx = 0.f;
  for (long long e = threadIdx.x; e < n; e += blockDim.x) {
    const float a = fabsf(__bfloat162float(v[at(e)]));
    if (a < INFINITY) mx = fmaxf(mx, a);
  }
  __shared__ float red[32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = 0.f;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) mx = fmaxf(mx, red[i]);
  int k = 0;
  while (ldexpf(mx, -k) > 32768.f) ++k;
  const float inv = ldexpf(1.f, -k);
  for (long long e = threadIdx.x; e < n; e += blockDim.x) {
    const long long i = at(e);
    v16[i] = __float2half_rn(__bfloat162float(v[i]) * inv);
  }
  if (threadIdx.x == 0) scales[h] = ldexpf(1.f, k);
}

// Merge per-split results: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
// One warp per row; lane l holds columns [l * D / 32, (l + 1) * D / 32).  The
// split LSEs are read by the lanes in parallel (lane l: splits l, l + 32, ...)
// and combined with warp shuffles; the weights are then broadcast one split at
// a time while every lane accumulates its columns.
template <int D>
__global__ void __launch_bounds__(256) fa2_splitkv_combine_kernel(const float* __restrict__ o_part,
                                                                  const float* __restrict__ lse_part,
                                                                  __nv_bfloat16* __restrict__ o,
                                                                  float* __restrict__ lse, long long rows,
                                                                  int splits) {
  constexpr int kPer = D >= 32 ? D / 32 : 1;  // columns per lane
  griddep_wait();
  griddep_launch_dependents();
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int s = lane; s < splits; s += 32) mx = fmaxf(mx, lse_part[static_cast<size_t>(s) * rows + row]);
#pragma unroll
  for (int sh = 16; sh > 0; sh >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  float total = -INFINITY;
  if (mx != -INFINITY) {
    float sum = 0.f;
    for (int s = lane; s < splits; s += 32) sum += expf(lse_part[static_cast<size_t>(s) * rows + row] - mx);
#pragma unroll
    for (int sh = 16; sh > 0; sh >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, sh);
    total = mx + logf(sum);
    const bool active = D >= 32 || lane < D;
    for (int base = 0; base < splits; base += 32) {
      const int s_l = base + lane;
      const float w_l = s_l < splits ? expf(lse_part[static_cast<size_t>(s_l) * rows + row] - total) : 0.f;
      const int n = min(32, splits - base);
#pragma unroll 4
      for (int i = 0; i < n; ++i) {
        const float w = __shfl_sync(0xffffffffu, w_l, i);
        if (w == 0.f || !active) continue;
        const float* src = o_part + (static_cast<size_t>(base + i) * rows + row) * D + lane * kPer;
#pragma unroll
        for (int k = 0; k < kPer; ++k) acc[k] = fmaf(w, src[k], acc[k]);
      }
    }
  }
  if (D >= 32 || lane < D) {
    __nv_bfloat16* dst = o + static_cast<size_t>(row) * D + lane * kPer;
#pragma unroll
    for (int k = 0; k < kPer; ++k) dst[k] = __float2bfloat16_rn(acc[k]);
  }
  if (lane == 0) lse[row] = total;
}

}  // namespace

int launch_fwd(const TmapSet& tm, const FwdProblem& p, int d, float scale, bool causal, cudaStream_t stream) {
  switch (d) {
    case 16: return causal ? launch_fwd_t<16, true>(tm, p, scale, stream) : launch_fwd_t<16, false>(tm, p, scale, stream);
    case 32: return causal ? launch_fwd_t<32, true>(tm, p, scale, stream) : launch_fwd_t<32, false>(tm, p, scale, stream);
    case 64: return causal ? launch_fwd_t<64, true>(tm, p, scale, stream) : launch_fwd_t<64, false>(tm, p, scale, stream);
    case 128:
      return causal ? launch_fwd_t<128, true>(tm, p, scale, stream) : launch_fwd_t<128, false>(tm, p, scale, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

int launch_v_to_f16(const void* v, void* v16, unsigned long long* v_flags, float* v_scale, unsigned long long call,
                    int heads, long long rows, int d, long long row_stride, long long head_stride, bool packed,
                    cudaStream_t stream) {
  if (rows * d <= kVHeadSmall)
    return launch_pdl(fa2_v_to_f16_head_kernel, dim3(static_cast<unsigned>(heads)), dim3(256), 0, stream,
                      static_cast<const __nv_bfloat16*>(v), static_cast<__half*>(v16), v_scale, rows, d, row_stride,
                      head_stride);
  const long long n8 = static_cast<long long>(heads) * rows * d / 8;
  long long blocks = (n8 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  const long long inner = packed ? d : rows * d;
  if (int e = launch_pdl(fa2_v_to_f16_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                         static_cast<const uint4*>(v), static_cast<uint4*>(v16), v_flags, call, n8, inner, heads))
    return e;
  return launch_pdl(fa2_v_scale_kernel, dim3(static_cast<unsigned>(heads)), dim3(256), 0, stream,
                    static_cast<const __nv_bfloat16*>(v), static_cast<__half*>(v16),
                    static_cast<const unsigned long long*>(v_flags), v_scale, call, rows, d, row_stride, head_stride);
}

int launch_splitkv_combine(const FwdProblem& p, int d, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.RH) * p.M;
  const unsigned blocks = static_cast<unsigned>((rows * 32 + 255) / 256);
  auto o = static_cast<__nv_bfloat16*>(p.o);
  switch (d) {
    case 16: return launch_pdl(fa2_splitkv_combine_kernel<16>, dim3(blocks), dim3(256), 0, stream, p.o_part, p.lse_part, o, p.lse, rows, p.splits);
    case 32: return launch_pdl(fa2_splitkv_combine_kernel<32>, dim3(blocks), dim3(256), 0, stream, p.o_part, p.lse_part, o, p.lse, rows, p.splits);
    case 64: return launch_pdl(fa2_splitkv_combine_kernel<64>, dim3(blocks), dim3(256), 0, stream, p.o_part, p.lse_part, o, p.lse, rows, p.splits);
    case 128: return launch_pdl(fa2_splitkv_combine_kernel<128>, dim3(blocks), dim3(256), 0, stream, p.o_part, p.lse_part, o, p.lse, rows, p.splits);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

int read_fwd_status(int* value, bool reset) {
  if (cudaError_t e = cudaMemcpyFromSymbol(value, g_fwd_status, sizeof(int))) return static_cast<int>(e);
  if (reset) {
    const int zero = 0;
    if (cudaError_t e = cudaMemcpyToSymbol(g_fwd_status, &zero, sizeof(int))) return static_cast<int>(e);
  }
  return 0;
}

}  // namespace fa2
