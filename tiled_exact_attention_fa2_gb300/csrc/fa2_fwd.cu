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
// The running max is updated lazily: O and l are rescaled only when a row's
// max grows by more than 8 (log2 units); otherwise the stale max is kept and
// P = 2^(s - m) stays <= 256, which is exact after the final O / l.
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
constexpr float kRescaleThreshold = 8.f;  // log2 units

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

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fa2_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out_o,
                   float* __restrict__ out_lse, int BH, int N, float scale_log2) {
  using T = HeadDim<D>;
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kTmemSlot);
  int* status = &g_fwd_status;

  const int warp = warp_id();
  const int lane = lane_id();

  // Heaviest query-tile pairs first (causal work grows with the pair index).
  const int num_tiles = (N + kTileRows - 1) / kTileRows;
  const int num_pairs = (num_tiles + 1) / 2;
  const int bh = blockIdx.x % BH;
  const int pair = num_pairs - 1 - static_cast<int>(blockIdx.x / BH);
  const int q0 = pair * 2 * kTileRows;
  // K/V tiles each query tile visits; a tile with no row < N visits none.
  const int nA = CAUSAL ? 2 * pair + 1 : num_tiles;
  const int nB = 2 * pair + 1 >= num_tiles ? 0 : (CAUSAL ? 2 * pair + 2 : num_tiles);
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
      const int n_q_tiles = nB > 0 ? 2 : 1;
      mbar_arrive_expect_tx(&bars[kBarQ], n_q_tiles * T::kTileBytes);
      for (int x = 0; x < n_q_tiles; ++x)
        for (int b = 0; b < T::kNumBoxes; ++b)
          tma_load_3d(smem + C::kQ + x * T::kTileBytes + b * T::kBoxBytes, &tm_q, &bars[kBarQ], b * T::kBoxCols,
                      q0 + x * kTileRows, bh);
      int last_k0 = -1, last_k1 = -1, last_v0 = -1, last_v1 = -1;
#pragma unroll 1
      for (int j = 0; j < n_kv; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(&bars[kBarKEmpty + st], ((j >> 1) - 1) & 1, status)) break;
        mbar_arrive_expect_tx(&bars[kBarKFull + st], T::kTileBytes);
        for (int b = 0; b < T::kNumBoxes; ++b)
          tma_load_3d(smem + C::kK + st * T::kTileBytes + b * T::kBoxBytes, &tm_k, &bars[kBarKFull + st],
                      b * T::kBoxCols, j * kTileRows, bh);
        (st ? last_k1 : last_k0) = j;
        if (j >= 2 && !mbar_wait(&bars[kBarVEmpty + st], ((j >> 1) - 1) & 1, status)) break;
        mbar_arrive_expect_tx(&bars[kBarVFull + st], T::kTileBytes);
        for (int b = 0; b < T::kNumBoxes; ++b)
          tma_load_3d(smem + C::kV + st * T::kTileBytes + b * T::kBoxBytes, &tm_v, &bars[kBarVFull + st],
                      b * T::kBoxCols, j * kTileRows, bh);
        (st ? last_v1 : last_v0) = j;
      }
      // Never leave the CTA with a TMA write still landing in shared memory.
      mbar_wait(&bars[kBarQ], 0, status);
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
    const int q_row = q0 + x * kTileRows + r;
    const int nx = x == 0 ? nA : nB;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + (x ? C::kColS1 : C::kColS0);
    const uint32_t tO = tmem + lane_base + (x ? C::kColO1 : C::kColO0);
    float m = -INFINITY;  // max used for P, log2 units (scores * scale * log2 e)
    float l = 0.f;        // running sum of 2^(x - m) in fp32 (gives LSE)
    float lr = 0.f;       // running sum of the bf16-rounded weights the PV MMA uses (normalises O)
    bool ok = true;
#pragma unroll 1
    for (int j = 0; j < nx; ++j) {
      // S_x(j) was issued after O_x += P_x(j-1) V_{j-1} completed, so O_x is
      // stable once S_x(j) has landed.
      if (!(ok = mbar_wait(&bars[kBarSFull + x], j & 1, status))) break;
      tc_fence_after();
      float s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, s[c]);
      tmem_wait_ld();

      const int kv0 = j * kTileRows;
      if ((CAUSAL && j == nx - 1) || kv0 + kTileRows > N) {
        int lim = N - kv0;                              // keys >= N do not exist
        if (CAUSAL) lim = min(lim, q_row - kv0 + 1);    // key j visible iff j <= query
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c * 32 + e >= lim) s[c][e] = -INFINITY;
      }
      // Row max as a tree (8 independent chains), not one 128-long chain.
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(s[0][k], s[0][k + 8]);
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(mx8[k], fmaxf(s[0][k + 16], s[0][k + 24]));
#pragma unroll
      for (int c = 1; c < 4; ++c)
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mx8[k] = fmaxf(mx8[k], fmaxf(fmaxf(s[c][k], s[c][k + 8]), fmaxf(s[c][k + 16], s[c][k + 24])));
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_tile = mx * scale_log2;
      const bool grow = m_tile > m + kRescaleThreshold;  // always true on the first tile
      const float m_use = grow ? m_tile : m;
      const float alpha = grow ? ex2_approx(m - m_use) : 1.f;

      // Row sums in 4 independent partial accumulators each.
      float rs4[4] = {0.f, 0.f, 0.f, 0.f}, rsr4[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = ex2_approx(fmaf(s[c][e], scale_log2, -m_use));
          const float p1 = ex2_approx(fmaf(s[c][e + 1], scale_log2, -m_use));
          rs4[(e >> 1) & 3] += p0 + p1;
          const uint32_t w = pack_bf16x2(p0, p1);
          const float2 pr = unpack_bf16x2(w);
          rsr4[(e >> 1) & 3] += pr.x + pr.y;
          pk[c * 16 + e / 2] = w;
        }
      const float rs = (rs4[0] + rs4[1]) + (rs4[2] + rs4[3]);
      const float rsr = (rsr4[0] + rsr4[1]) + (rsr4[2] + rsr4[3]);

      if (j >= 1 && __any_sync(0xffffffffu, grow)) {
        if constexpr (D >= 32) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
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
      tmem_st32u(tS, pk);
      tmem_st32u(tS + 32, pk + 32);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarPFull + x]);
      l = l * alpha + rs;
      lr = lr * alpha + rsr;
      m = m_use;
    }
    // ------------------------------------------------------------ epilogue
    if (nx > 0 && ok && mbar_wait(&bars[kBarPVDone + x], (nx - 1) & 1, status)) {
      tc_fence_after();
      // O = sum_j bf16(p_j) V_j / sum_j bf16(p_j): the weights' bf16 rounding
      // cancels in the ratio (the dominant weight need not be 1 under the
      // lazy max).  LSE uses the fp32 sum.
      const float inv_l = lr > 0.f ? 1.f / lr : 0.f;
      const bool valid = q_row < N;
      __nv_bfloat16* orow = out_o + (static_cast<size_t>(bh) * N + (valid ? q_row : 0)) * D;
      if constexpr (D >= 32) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tO + c * 32, o);
          tmem_wait_ld();
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pack_bf16x2(o[8 * q + 0] * inv_l, o[8 * q + 1] * inv_l),
                                  pack_bf16x2(o[8 * q + 2] * inv_l, o[8 * q + 3] * inv_l),
                                  pack_bf16x2(o[8 * q + 4] * inv_l, o[8 * q + 5] * inv_l),
                                  pack_bf16x2(o[8 * q + 6] * inv_l, o[8 * q + 7] * inv_l));
          }
        }
      } else {
        float o[16];
        tmem_ld16(tO, o);
        tmem_wait_ld();
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int q = 0; q < 2; ++q)
            dst[q] = make_uint4(pack_bf16x2(o[8 * q + 0] * inv_l, o[8 * q + 1] * inv_l),
                                pack_bf16x2(o[8 * q + 2] * inv_l, o[8 * q + 3] * inv_l),
                                pack_bf16x2(o[8 * q + 4] * inv_l, o[8 * q + 5] * inv_l),
                                pack_bf16x2(o[8 * q + 6] * inv_l, o[8 * q + 7] * inv_l));
        }
      }
      // LSE in natural log of the scaled scores: ln 2 * (m + log2 l).
      if (valid) out_lse[static_cast<size_t>(bh) * N + q_row] = (m + log2f(l)) * 0.69314718055994531f;
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
int launch_fwd_t(const TmapSet& tm, void* o, float* lse, int BH, int N, float scale, cudaStream_t stream) {
  using C = FwdCfg<D>;
  auto kern = fa2_fwd_kernel<D, CAUSAL>;
  if (int rc = ensure_max_smem(reinterpret_cast<const void*>(kern), C::kBytes)) return rc;
  const int num_tiles = (N + kTileRows - 1) / kTileRows;
  const int num_pairs = (num_tiles + 1) / 2;
  const dim3 grid(static_cast<unsigned>(num_pairs) * static_cast<unsigned>(BH));
  const float scale_log2 = scale * 1.44269504088896341f;
  kern<<<grid, kFwdThreads, C::kBytes, stream>>>(tm.q, tm.k, tm.v, static_cast<__nv_bfloat16*>(o), lse, BH, N,
                                                  scale_log2);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace

int launch_fwd(const TmapSet& tm, void* o, float* lse, int BH, int N, int d, float scale, bool causal,
               cudaStream_t stream) {
  switch (d) {
    case 16: return causal ? launch_fwd_t<16, true>(tm, o, lse, BH, N, scale, stream)
                           : launch_fwd_t<16, false>(tm, o, lse, BH, N, scale, stream);
    case 32: return causal ? launch_fwd_t<32, true>(tm, o, lse, BH, N, scale, stream)
                           : launch_fwd_t<32, false>(tm, o, lse, BH, N, scale, stream);
    case 64: return causal ? launch_fwd_t<64, true>(tm, o, lse, BH, N, scale, stream)
                           : launch_fwd_t<64, false>(tm, o, lse, BH, N, scale, stream);
    case 128: return causal ? launch_fwd_t<128, true>(tm, o, lse, BH, N, scale, stream)
                            : launch_fwd_t<128, false>(tm, o, lse, BH, N, scale, stream);
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
