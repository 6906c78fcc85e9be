// FlashAttention-2 forward on sm_103a: TMA-fed tiles, tcgen05 MMAs with TMEM
// accumulators and an online softmax.  One CTA per (pair of 128-row query
// tiles, head).
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
//   warp  8    TMA producer: Q_A, Q_B once, then K_j / V_j into 2-stage rings
//   warp  9    MMA issuer for tile A (one thread) + TMEM owner
//   warp 10    MMA issuer for tile B (one thread)
// One issuer per tile, so that waiting on one tile's MMA never delays the
// other tile's; K/V stages are released once both issuers are done with them.
// TMEM columns: S_A [0,128), S_B [128,256), O_A and O_B after them.  The
// softmax overwrites the first 64 columns of S_X with P_X (bf16 pairs) and
// O_X += P_X V_j reads P_X straight from TMEM (A operand in TMEM), so P never
// touches shared memory.  S_X(j+1) is issued only after P_X(j) V_j has
// completed, because it overwrites the columns that MMA reads.
// O is rescaled in TMEM only when some row of the warp sees its max grow, so
// every row's largest weight is exactly 1.  The softmax arithmetic runs on
// packed fp32 pairs (f32x2 FMA/ADD/MUL) and 3-input max to halve its
// instruction count, which bounds this kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "tiles.cuh"

namespace fa2 {

__device__ int g_fwd_status;

namespace {

constexpr int kFwdThreads = 352;
constexpr uint32_t kTmemCols = 512;

enum FwdBar {
  kBarQ = 0,
  kBarKFull = 1,    // +stage (2)
  kBarKEmpty = 3,   // +stage
  kBarVFull = 5,    // +stage
  kBarVEmpty = 7,   // +stage
  kBarSFull = 9,    // +tile (A, B)
  kBarPFull = 11,   // +tile, 4 warp arrivals
  kBarPVDone = 13,  // +tile
  kBarDrain = 15,   // +tile
  kNumFwdBars = 17,
};

template <int D>
struct FwdCfg {
  using T = HeadDim<D>;
  static constexpr int kCols = D < 32 ? 32 : D;
  static constexpr uint32_t kColS0 = 0, kColS1 = 128;
  static constexpr uint32_t kColO0 = 256, kColO1 = 256 + kCols;
  static constexpr int kQ = 0;  // Q_A, Q_B
  static constexpr int kK = kQ + 2 * T::kTileBytes;
  static constexpr int kV = kK + 2 * T::kTileBytes;
  static constexpr int kBars = kV + 2 * T::kTileBytes;
  static constexpr int kTmemSlot = kBars + kNumFwdBars * 8;
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

template <int D, bool CAUSAL, int MODE>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa2_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const FwdProblem p, float scale_log2) {
  using T = HeadDim<D>;
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kTmemSlot);
  int* status = &g_fwd_status;

  const int warp = warp_id();
  const int lane = lane_id();

  // CTA = (key split or sequence, group of heads_per_group row-heads, pair
  // of 128-row tiles, row-head), slowest first: a group's K/V rows stay in L2
  // while its CTAs run, and inside a group the heaviest pairs go first
  // (causal work grows with the pair index).  Row r of row-head rh is query
  // r % Nq; the row-head reads K/V head rh / kvdiv.
  const int num_row_tiles = (p.M + kTileRows - 1) / kTileRows;
  const int num_pairs = (num_row_tiles + 1) / 2;
  const int per_split = num_pairs * p.RH;
  const int split = MODE == kVarlen ? 0 : static_cast<int>(blockIdx.x / per_split);
  const int local = static_cast<int>(blockIdx.x % per_split);
  const int per_group = p.heads_per_group * num_pairs;
  const int hg0 = local / per_group * p.heads_per_group;
  const int hg = min(p.heads_per_group, p.RH - hg0);
  const int pair = num_pairs - 1 - (local % per_group) / hg;
  const int rh = hg0 + (local % per_group) % hg;
  const int rh_kv = rh / p.kvdiv;
  const int q0 = pair * 2 * kTileRows;
  // Rows and keys of this CTA's problem, the causal offset (query i sees key
  // j iff j <= i + off) and the first TMA row of its queries and keys.
  int M = p.M, Nk = p.Nk, off = MODE == kGeneral ? p.Nk - p.Nq : 0, q_base = 0, k_base = 0;
  if constexpr (MODE == kVarlen) {
    const int b = static_cast<int>(blockIdx.x / per_split);
    const int sq = p.cu_q[b], eq = p.cu_q[b + 1], sk = p.cu_k[b], ek = p.cu_k[b + 1];
    if (!(0 <= sq && sq <= eq && eq <= p.total_q && eq - sq <= p.M && 0 <= sk && sk <= ek && ek <= p.total_k &&
          ek - sk <= p.Nk)) {
      if (threadIdx.x == 0) atomicCAS(status, kDevOk, kDevBadSeqlens);
      return;
    }
    M = eq - sq;
    Nk = ek - sk;
    off = Nk - M;
    q_base = sq;
    k_base = sk;
    if (q0 >= M) return;  // the whole CTA lies past this sequence's queries
  }
  const int num_kv_tiles = (Nk + kTileRows - 1) / kTileRows;
  const int jb = split * p.tiles_per_split;
  const int je = min(num_kv_tiles, jb + p.tiles_per_split);
  // Local K/V tiles (from jb) each row tile visits, and the smallest query
  // index among its rows (for the causal-mask test).
  int cnt[2], imin[2];
  if constexpr (MODE == kSquare) {
    // Square problem: tile A sees tiles 0..2*pair (causal), tile B one more.
    cnt[0] = CAUSAL ? 2 * pair + 1 : num_kv_tiles;
    cnt[1] = 2 * pair + 1 >= num_row_tiles ? 0 : (CAUSAL ? 2 * pair + 2 : num_kv_tiles);
    imin[0] = q0;
    imin[1] = q0 + kTileRows;
  } else {
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      const int rx0 = q0 + x * kTileRows;
      cnt[x] = 0;
      imin[x] = 0;
      if (rx0 < M) {
        const int rlast = min(rx0 + kTileRows - 1, M - 1);
        const bool one_head = MODE == kVarlen || rx0 / p.Nq == rlast / p.Nq;
        const int i_max = MODE == kVarlen ? rlast : (one_head ? rlast % p.Nq : p.Nq - 1);
        imin[x] = MODE == kVarlen ? rx0 : (one_head ? rx0 % p.Nq : 0);
        // causal: the last key any row of the tile sees is i_max + off (< 0: none)
        const int kv_end = !CAUSAL ? num_kv_tiles
                                   : (i_max + off < 0 ? 0 : min(num_kv_tiles, (i_max + off) / kTileRows + 1));
        cnt[x] = max(0, min(je, kv_end) - jb);
      }
    }
  }
  const int nA = cnt[0], nB = cnt[1];
  const int n_kv = nA > nB ? nA : nB;

  if (threadIdx.x == 8 * 32) {
    mbar_init(&bars[kBarQ], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kBarKFull + s], 1);
      mbar_init(&bars[kBarKEmpty + s], 2);
      mbar_init(&bars[kBarVFull + s], 1);
      mbar_init(&bars[kBarVEmpty + s], 2);
      mbar_init(&bars[kBarSFull + s], 1);
      mbar_init(&bars[kBarPFull + s], 4);
      mbar_init(&bars[kBarPVDone + s], 1);
      mbar_init(&bars[kBarDrain + s], 1);
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

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int n_q_tiles = (nA > 0) + (nB > 0);
      if (n_q_tiles > 0) mbar_arrive_expect_tx(&bars[kBarQ], n_q_tiles * T::kTileBytes);
      for (int x = 0; x < 2; ++x)
        if (cnt[x] > 0)
          for (int b = 0; b < T::kNumBoxes; ++b)
            tma_load_3d(smem + C::kQ + x * T::kTileBytes + b * T::kBoxBytes, &tm_q, &bars[kBarQ],
                        b * T::kBoxCols, q_base + q0 + x * kTileRows, rh);
      int last_k0 = -1, last_k1 = -1, last_v0 = -1, last_v1 = -1;
#pragma unroll 1
      for (int j = 0; j < n_kv; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(&bars[kBarKEmpty + st], ((j >> 1) - 1) & 1, status)) break;
        mbar_arrive_expect_tx(&bars[kBarKFull + st], T::kTileBytes);
        for (int b = 0; b < T::kNumBoxes; ++b)
          tma_load_3d(smem + C::kK + st * T::kTileBytes + b * T::kBoxBytes, &tm_k, &bars[kBarKFull + st],
                      b * T::kBoxCols, k_base + (jb + j) * kTileRows, rh_kv);
        (st ? last_k1 : last_k0) = j;
        if (j >= 2 && !mbar_wait(&bars[kBarVEmpty + st], ((j >> 1) - 1) & 1, status)) break;
        mbar_arrive_expect_tx(&bars[kBarVFull + st], T::kTileBytes);
        for (int b = 0; b < T::kNumBoxes; ++b)
          tma_load_3d(smem + C::kV + st * T::kTileBytes + b * T::kBoxBytes, &tm_v, &bars[kBarVFull + st],
                      b * T::kBoxCols, k_base + (jb + j) * kTileRows, rh_kv);
        (st ? last_v1 : last_v0) = j;
      }
      // Never leave the CTA with a TMA write still landing in shared memory.
      if (n_q_tiles > 0) mbar_wait(&bars[kBarQ], 0, status);
      if (last_k0 >= 0) mbar_wait(&bars[kBarKFull + 0], (last_k0 >> 1) & 1, status);
      if (last_k1 >= 0) mbar_wait(&bars[kBarKFull + 1], (last_k1 >> 1) & 1, status);
      if (last_v0 >= 0) mbar_wait(&bars[kBarVFull + 0], (last_v0 >> 1) & 1, status);
      if (last_v1 >= 0) mbar_wait(&bars[kBarVFull + 1], (last_v1 >> 1) & 1, status);
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issuer of tile x
    if (lane == 0) {
      const int x = warp - 9;
      const int nx = x == 0 ? nA : nB;
      constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false, false);  // Q (K-major) x K (K-major)
      constexpr uint32_t kIdescO = make_idesc_bf16(128, D, false, true);     // P (TMEM) x V (MN-major)
      const uint32_t sQ0 = smem_u32(smem + C::kQ), sK0 = smem_u32(smem + C::kK), sV0 = smem_u32(smem + C::kV);
      const uint32_t tSx = tmem + (x ? C::kColS1 : C::kColS0), tOx = tmem + (x ? C::kColO1 : C::kColO0);
      // S_x(j) = Q_x K_j^T into TMEM S_x.
      auto issue_s = [&](int j) {
        uint32_t sQ = sQ0, sK = sK0;
        opaque(sQ);
        opaque(sK);
        const uint32_t qb = sQ + x * T::kTileBytes, kb = sK + (j & 1) * T::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tSx, T::kmajor_desc(qb, kk), T::kmajor_desc(kb, kk), kIdescS, kk > 0 ? 1u : 0u);
        mma_commit(&bars[kBarSFull + x]);
        mma_commit(&bars[kBarKEmpty + (j & 1)]);
      };
      // O_x += P_x V_j with P_x read from the first 64 columns of S_x.
      auto issue_pv = [&](int j) {
        uint32_t sV = sV0;
        opaque(sV);
        const uint32_t vb = sV + (j & 1) * T::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileRows / 16; ++kk)
          mma_bf16_ts(tOx, tSx + kk * 8, T::mnmajor_desc(vb, kk), kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars[kBarPVDone + x]);
        mma_commit(&bars[kBarVEmpty + (j & 1)]);
      };
      bool ok = true;
      if (nx > 0) {
        ok = mbar_wait(&bars[kBarQ], 0, status) && mbar_wait(&bars[kBarKFull + 0], 0, status);
        if (ok) {
          tc_fence_after();
          issue_s(0);
        }
      }
#pragma unroll 1
      for (int j = 0; ok && j < nx; ++j) {
        const int st = j & 1;
        if (!(ok = mbar_wait(&bars[kBarVFull + st], (j >> 1) & 1, status))) break;
        if (!(ok = mbar_wait(&bars[kBarPFull + x], j & 1, status))) break;
        tc_fence_after();
        issue_pv(j);
        if (j + 1 < nx) {
          // S_x(j+1) overwrites the P_x columns the MMA above reads.
          if (!(ok = mbar_wait(&bars[kBarPVDone + x], j & 1, status))) break;
          if (!(ok = mbar_wait(&bars[kBarKFull + (st ^ 1)], ((j + 1) >> 1) & 1, status))) break;
          tc_fence_after();
          issue_s(j + 1);
        }
      }
      // K/V tiles this query tile does not visit: release them once, in
      // phase order (after the stage's previous use has been released).
#pragma unroll 1
      for (int j = nx; ok && j < n_kv; ++j) {
        const int st = j & 1;
        if (j >= 2 && !(ok = mbar_wait(&bars[kBarKEmpty + st], ((j >> 1) - 1) & 1, status))) break;
        mbar_arrive(&bars[kBarKEmpty + st]);
        if (j >= 2 && !(ok = mbar_wait(&bars[kBarVEmpty + st], ((j >> 1) - 1) & 1, status))) break;
        mbar_arrive(&bars[kBarVEmpty + st]);
      }
      // Wait for every MMA this thread issued before TMEM can be released.
      mma_commit(&bars[kBarDrain + x]);
      mbar_wait(&bars[kBarDrain + x], 0, status);
    }
  } else {
    // ------------------------------------------------------------ softmax (tile x)
    const int x = warp >> 2;
    const int r = threadIdx.x & 127;  // row within the tile = TMEM lane
    const int q_row = q0 + x * kTileRows + r;  // row in the row-head
    const int qi = MODE == kGeneral ? q_row % p.Nq : q_row;  // its query index
    const int imin_x = x ? imin[1] : imin[0];
    const int nx = x == 0 ? nA : nB;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (x ? C::kColS1 : C::kColS0);
    const uint32_t tO = tmem + lane_base + (x ? C::kColO1 : C::kColO0);
    float m = -INFINITY;  // running row max, log2 units (scores * scale * log2 e)
    float l = 0.f;        // running sum of 2^(x - m)
    const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
    bool ok = true;
#pragma unroll 1
    for (int j = 0; j < nx; ++j) {
      // S_x(j) was issued after O_x += P_x(j-1) V_{j-1} completed, so O_x is
      // stable once S_x(j) has landed.
      if (!(ok = mbar_wait(&bars[kBarSFull + x], j & 1, status))) break;
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, *reinterpret_cast<float(*)[32]>(s + 32 * c));
      tmem_wait_ld();

      const int kv0 = (jb + j) * kTileRows;
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
      for (int k = 0; k < 8; ++k) {
        // chain k covers columns k, k + 8, ..., k + 120
        float v = fmax3(s[k], s[k + 8], s[k + 16]);
#pragma unroll
        for (int i = 24; i <= 104; i += 16) v = fmax3(v, s[k + i], s[k + i + 8]);
        mx8[k] = fmaxf(v, s[k + 120]);
      }
      const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
      const float m_new = fmaxf(m, mx * scale_log2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const bool grow = m_use > m;  // always true on the first tile
      const float alpha = ex2_approx(m - m_use);

      // P = 2^(s * scale_log2 - m) on packed pairs; 4 independent pair sums.
      const uint64_t negm2 = f2_pack(-m_use, -m_use);
      // P goes to TMEM (bf16 pairs over the first 64 S columns, all of which
      // are already in registers) 16 columns at a time.
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
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16u(tS + 16 * c, pk);
      }
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
              const float2 r = f2_unpack(fmul2(f2_pack(o[e], o[e + 1]), alpha2));
              o[e] = r.x;
              o[e + 1] = r.y;
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
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarPFull + x]);
      l = l * alpha + rs;
      m = m_use;
    }
    // ------------------------------------------------------------ epilogue
    // One split: O / l in bf16 and LSE.  Several splits: this split's O / l
    // and LSE in fp32 for the combine kernel.  A row that sees no key gets
    // O = 0, LSE = -inf.
    const bool valid = q_row < M;
    const bool partial = MODE == kGeneral && p.splits > 1;
    const int vrow = valid ? q_row : 0;
    // o_row: row of o (or o_part) in units of D elements; lse_idx: index into lse.
    size_t o_row, lse_idx;
    if constexpr (MODE == kVarlen) {
      o_row = static_cast<size_t>(q_base + vrow) * p.RH + rh;
      lse_idx = static_cast<size_t>(rh) * p.total_q + q_base + vrow;
    } else {
      o_row = (partial ? static_cast<size_t>(split) * p.RH + rh : static_cast<size_t>(rh)) * p.M + vrow;
      lse_idx = o_row;
    }
    if (MODE != kSquare && nx == 0) {
      if (valid && ok) {
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
      }
    } else if (ok && mbar_wait(&bars[kBarPVDone + x], (nx - 1) & 1, status)) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      constexpr int kC = D >= 32 ? 32 : 16;
#pragma unroll
      for (int c = 0; c < D / kC; ++c) {
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
    }
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
  const bool general = p.splits > 1 || p.M != p.Nq || p.Nq != p.Nk;
  // Every row-head re-reads the K and V rows of its split.
  const int kv_rows = min(p.Nk, p.tiles_per_split * kTileRows);
  p.heads_per_group = heads_per_l2_group(static_cast<size_t>(kv_rows) * D * 4 / p.kvdiv, p.RH);
  auto kern = varlen    ? fa2_fwd_kernel<D, CAUSAL, kVarlen>
              : general ? fa2_fwd_kernel<D, CAUSAL, kGeneral>
                        : fa2_fwd_kernel<D, CAUSAL, kSquare>;
  if (int rc = ensure_max_smem(reinterpret_cast<const void*>(kern), C::kBytes)) return rc;
  const int num_row_tiles = (p.M + kTileRows - 1) / kTileRows;
  const int num_pairs = (num_row_tiles + 1) / 2;
  const unsigned outer = static_cast<unsigned>(varlen ? p.batches : p.splits);  // sequences or key splits
  const dim3 grid(static_cast<unsigned>(num_pairs) * static_cast<unsigned>(p.RH) * outer);
  const float scale_log2 = scale * 1.44269504088896341f;
  kern<<<grid, kFwdThreads, C::kBytes, stream>>>(tm.q, tm.k, tm.v, p, scale_log2);
  return static_cast<int>(cudaGetLastError());
}

// Merge per-split results: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
// One warp per row; lane l holds columns [l * D / 32, (l + 1) * D / 32).
template <int D>
__global__ void __launch_bounds__(256) fa2_splitkv_combine_kernel(const float* __restrict__ o_part,
                                                                  const float* __restrict__ lse_part,
                                                                  __nv_bfloat16* __restrict__ o,
                                                                  float* __restrict__ lse, long long rows,
                                                                  int splits) {
  constexpr int kPer = D >= 32 ? D / 32 : 1;  // columns per lane
  const long long row = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, lse_part[static_cast<size_t>(s) * rows + row]);
  float acc[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
  float total = -INFINITY;
  if (mx != -INFINITY) {
    float sum = 0.f;
    for (int s = 0; s < splits; ++s) sum += expf(lse_part[static_cast<size_t>(s) * rows + row] - mx);
    total = mx + logf(sum);
    const bool active = D >= 32 || lane < D;
    for (int s = 0; s < splits; ++s) {
      const float w = expf(lse_part[static_cast<size_t>(s) * rows + row] - total);
      if (w == 0.f || !active) continue;
      const float* src = o_part + (static_cast<size_t>(s) * rows + row) * D + lane * kPer;
#pragma unroll
      for (int k = 0; k < kPer; ++k) acc[k] = fmaf(w, src[k], acc[k]);
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

int launch_splitkv_combine(const FwdProblem& p, int d, cudaStream_t stream) {
  const long long rows = static_cast<long long>(p.RH) * p.M;
  const unsigned blocks = static_cast<unsigned>((rows * 32 + 255) / 256);
  auto o = static_cast<__nv_bfloat16*>(p.o);
  switch (d) {
    case 16: fa2_splitkv_combine_kernel<16><<<blocks, 256, 0, stream>>>(p.o_part, p.lse_part, o, p.lse, rows, p.splits); break;
    case 32: fa2_splitkv_combine_kernel<32><<<blocks, 256, 0, stream>>>(p.o_part, p.lse_part, o, p.lse, rows, p.splits); break;
    case 64: fa2_splitkv_combine_kernel<64><<<blocks, 256, 0, stream>>>(p.o_part, p.lse_part, o, p.lse, rows, p.splits); break;
    case 128: fa2_splitkv_combine_kernel<128><<<blocks, 256, 0, stream>>>(p.o_part, p.lse_part, o, p.lse, rows, p.splits); break;
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
  return static_cast<int>(cudaGetLastError());
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
