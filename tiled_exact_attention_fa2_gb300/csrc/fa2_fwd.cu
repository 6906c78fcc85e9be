// FlashAttention-2 forward on sm_103a: TMA-fed tiles, tcgen05 MMAs with TMEM
// accumulators and an online softmax, one CTA per (128-row query tile, head).
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
// Warp roles (192 threads):
//   warps 0-3  softmax: thread t owns query row t of the tile (TMEM lane t);
//              reads S, masks, updates m/l, rescales O when m grows, writes
//              P (bf16) to shared memory, and runs the epilogue.
//   warp  4    TMA producer: Q once, then K_j / V_j into 2-stage rings.
//   warp  5    MMA issuer (one thread) + TMEM owner:
//              S_j = Q K_j^T into one of two TMEM S buffers (double buffered
//              so S_{j+1} is computed while the softmax works on S_j), and
//              O += P_j V_j into the TMEM O accumulator.
// TMEM columns: S0 [0,128), S1 [128,256), O [256, 256+D).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "tiles.cuh"

namespace fa2 {

__device__ int g_fwd_status;

namespace {

constexpr int kFwdThreads = 192;
constexpr uint32_t kTmemCols = 512;

enum FwdBar {
  kBarQ = 0,
  kBarKFull = 1,    // +stage (2)
  kBarKEmpty = 3,   // +stage
  kBarVFull = 5,    // +stage
  kBarVEmpty = 7,   // +stage
  kBarSFull = 9,    // +buffer (2)
  kBarSEmpty = 11,  // +buffer
  kBarPFull = 13,
  kBarPVDone = 14,
  kBarDrain = 15,
  kNumFwdBars = 16,
};

template <int D>
struct FwdSmem {
  using T = HeadDim<D>;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + T::kTileBytes;
  static constexpr int kV = kK + 2 * T::kTileBytes;
  static constexpr int kP = kV + 2 * T::kTileBytes;
  static constexpr int kBars = kP + Square::kTileBytes;
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
  using L = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlot);
  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);
  const uint32_t sP = smem_u32(smem + L::kP);
  int* status = &g_fwd_status;

  const int warp = warp_id();
  const int lane = lane_id();

  // Heaviest query tiles first (causal work grows with the tile index).
  const int num_q_tiles = (N + kTileRows - 1) / kTileRows;
  const int bh = blockIdx.x % BH;
  const int qt = num_q_tiles - 1 - static_cast<int>(blockIdx.x / BH);
  const int q0 = qt * kTileRows;
  const int n_kv = CAUSAL ? (qt + 1) : num_q_tiles;

  if (threadIdx.x == kFwdThreads - 64) {  // warp 4, lane 0
    mbar_init(&bars[kBarQ], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kBarKFull + s], 1);
      mbar_init(&bars[kBarKEmpty + s], 1);
      mbar_init(&bars[kBarVFull + s], 1);
      mbar_init(&bars[kBarVEmpty + s], 1);
      mbar_init(&bars[kBarSFull + s], 1);
      mbar_init(&bars[kBarSEmpty + s], 4);
    }
    mbar_init(&bars[kBarPFull], 4);
    mbar_init(&bars[kBarPVDone], 1);
    mbar_init(&bars[kBarDrain], 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_O = tmem + 256;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
      mbar_arrive_expect_tx(&bars[kBarQ], T::kTileBytes);
      for (int b = 0; b < T::kNumBoxes; ++b)
        tma_load_3d(smem + L::kQ + b * T::kBoxBytes, &tm_q, &bars[kBarQ], b * T::kBoxCols, q0, bh);
#pragma unroll 1
      for (int j = 0; j < n_kv; ++j) {
        const int st = j & 1;
        if (j >= 2 && !mbar_wait(&bars[kBarKEmpty + st], ((j >> 1) - 1) & 1, status)) break;
        mbar_arrive_expect_tx(&bars[kBarKFull + st], T::kTileBytes);
        for (int b = 0; b < T::kNumBoxes; ++b)
          tma_load_3d(smem + L::kK + st * T::kTileBytes + b * T::kBoxBytes, &tm_k, &bars[kBarKFull + st],
                      b * T::kBoxCols, j * kTileRows, bh);
        last_k[st] = j;
        if (j >= 2 && !mbar_wait(&bars[kBarVEmpty + st], ((j >> 1) - 1) & 1, status)) break;
        mbar_arrive_expect_tx(&bars[kBarVFull + st], T::kTileBytes);
        for (int b = 0; b < T::kNumBoxes; ++b)
          tma_load_3d(smem + L::kV + st * T::kTileBytes + b * T::kBoxBytes, &tm_v, &bars[kBarVFull + st],
                      b * T::kBoxCols, j * kTileRows, bh);
        last_v[st] = j;
      }
      // Never leave the CTA with a TMA write still landing in shared memory.
      mbar_wait(&bars[kBarQ], 0, status);
      for (int s = 0; s < 2; ++s) {
        if (last_k[s] >= 0) mbar_wait(&bars[kBarKFull + s], (last_k[s] >> 1) & 1, status);
        if (last_v[s] >= 0) mbar_wait(&bars[kBarVFull + s], (last_v[s] >> 1) & 1, status);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = make_idesc_bf16(128, 128, false, false);  // Q (K-major) x K (K-major)
      constexpr uint32_t kIdescO = make_idesc_bf16(128, D, false, true);     // P (K-major) x V (MN-major)
      auto issue_pv = [&](int t) -> bool {
        const int st = t & 1;
        if (!mbar_wait(&bars[kBarPFull], t & 1, status)) return false;
        if (!mbar_wait(&bars[kBarVFull + st], (t >> 1) & 1, status)) return false;
        tc_fence_after();
        const uint32_t vbase = sV + st * T::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kTileRows / 16; ++kk)
          mma_bf16_ss(tmem_O, Square::kmajor_desc(sP, kk), T::mnmajor_desc(vbase, kk), kIdescO,
                      (t > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars[kBarPVDone]);
        mma_commit(&bars[kBarVEmpty + st]);
        return true;
      };
      bool ok = mbar_wait(&bars[kBarQ], 0, status);
#pragma unroll 1
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j & 1;
        if (!(ok = mbar_wait(&bars[kBarKFull + st], (j >> 1) & 1, status))) break;
        if (j >= 2 && !(ok = mbar_wait(&bars[kBarSEmpty + st], ((j >> 1) - 1) & 1, status))) break;
        tc_fence_after();
        const uint32_t kbase = sK + st * T::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tmem + st * 128, T::kmajor_desc(sQ, kk), T::kmajor_desc(kbase, kk), kIdescS,
                      kk > 0 ? 1u : 0u);
        mma_commit(&bars[kBarSFull + st]);
        mma_commit(&bars[kBarKEmpty + st]);
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(n_kv - 1);
      // Wait for every MMA issued above before TMEM can be released.
      mma_commit(&bars[kBarDrain]);
      mbar_wait(&bars[kBarDrain], 0, status);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // 0..127 = TMEM lane = row in the tile
    const int q_row = q0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    float m = -INFINITY;  // running max, log2 units (scores * scale * log2 e)
    float l = 0.f;        // running sum of 2^(x - m)
    bool ok = true;
#pragma unroll 1
    for (int j = 0; j < n_kv; ++j) {
      const int st = j & 1;
      if (!(ok = mbar_wait(&bars[kBarSFull + st], (j >> 1) & 1, status))) break;
      tc_fence_after();
      float s[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + st * 128 + c * 32, s[c]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarSEmpty + st]);

      const int kv0 = j * kTileRows;
      if ((CAUSAL && j == n_kv - 1) || kv0 + kTileRows > N) {
        int lim = N - kv0;                              // keys >= N do not exist
        if (CAUSAL) lim = min(lim, q_row - kv0 + 1);    // key j visible iff j <= query
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c * 32 + e >= lim) s[c][e] = -INFINITY;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, s[c][e]);
      const float m_new = fmaxf(m, mx * scale_log2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float p = ex2_approx(fmaf(s[c][e], scale_log2, -m_use));
          s[c][e] = p;
          rs += p;
        }
      const float alpha = ex2_approx(m - m_use);

      if (j >= 1) {
        // O holds sum_{t<j} P_t V_t relative to the old max: rescale it
        // before P_j V_j is accumulated (only when some row's max grew).
        if (!(ok = mbar_wait(&bars[kBarPVDone], (j - 1) & 1, status))) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          if constexpr (D >= 32) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              float o[32];
              tmem_ld32(tmem_O + lane_base + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              tmem_st32(tmem_O + lane_base + c * 32, o);
            }
          } else {
            float o[16];
            tmem_ld16(tmem_O + lane_base, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= alpha;
            tmem_st16(tmem_O + lane_base, o);
          }
          tmem_wait_st();
        }
      }
      // P (bf16) -> shared memory, K-major 128B-swizzled for the PV MMA.
#pragma unroll
      for (int c16 = 0; c16 < 16; ++c16) {
        const float* v = &s[c16 >> 2][(c16 & 3) * 8];
        store_square_chunk(sP, r, c16, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                           pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarPFull]);
      l = l * alpha + rs;
      m = m_new;
    }
    // ------------------------------------------------------------ epilogue
    if (ok && mbar_wait(&bars[kBarPVDone], (n_kv - 1) & 1, status)) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool valid = q_row < N;
      __nv_bfloat16* orow = out_o + (static_cast<size_t>(bh) * N + (valid ? q_row : 0)) * D;
      if constexpr (D >= 32) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tmem_O + lane_base + c * 32, o);
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
        tmem_ld16(tmem_O + lane_base, o);
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
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool CAUSAL>
int launch_fwd_t(const TmapSet& tm, void* o, float* lse, int BH, int N, float scale, cudaStream_t stream) {
  using L = FwdSmem<D>;
  auto kern = fa2_fwd_kernel<D, CAUSAL>;
  if (int rc = ensure_max_smem(reinterpret_cast<const void*>(kern), L::kBytes)) return rc;
  const int num_q_tiles = (N + kTileRows - 1) / kTileRows;
  const dim3 grid(static_cast<unsigned>(num_q_tiles) * static_cast<unsigned>(BH));
  const float scale_log2 = scale * 1.44269504088896341f;
  kern<<<grid, kFwdThreads, L::kBytes, stream>>>(tm.q, tm.k, tm.v, static_cast<__nv_bfloat16*>(o), lse, BH, N,
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
