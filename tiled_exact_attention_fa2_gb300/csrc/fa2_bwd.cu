// FlashAttention-2 backward on sm_103a.
//
// Method: "Revolutionizing Web-Based AI: How a Plain JavaScript Prototype
// Paved the Way for High-Performance WebGPU Flash Attention 2", section
// "Translating to WGSL and Optimizing Passes" (backward-pass bullet): the
// attention weights are recomputed tile by tile from the saved Q, K and the
// per-row log-sum-exp instead of being read back from a stored matrix.  The
// same article's section "Numerical Stability and Loss Drift" names atomic
// reductions as a rounding source; dQ here is such a reduction (fp32 adds
// into a zeroed accumulator, performed in L2 by TMA reduce-add), the only
// step whose summation order varies between runs.
//
// Three kernels, enqueued in this order on the caller's stream (each
// launched with programmatic stream serialisation):
//   1. preprocess: D = rowsum(dO * O) (fp32) and zero the fp32 dQ accumulator
//      (HBM-bound, 16-byte coalesced loads).
//   2. main: one CTA per (128-row key/value tile, K/V head); loops over the
//      query tiles that can see it (all of them, or those at or after the
//      diagonal when causal) of every query head that shares the K/V head:
//         S^T  = K Q_i^T                   (TMEM)
//         P^T  = exp(scale S^T - LSE_i)    (registers -> bf16 pairs in TMEM)
//         dP^T = V dO_i^T                  (TMEM)
//         dV  += P^T dO_i                  (TMEM accumulator, P^T from TMEM)
//         dS^T = P^T * (dP^T - D_i)        (registers -> bf16 smem)
//         dK  += dS^T Q_i                  (TMEM accumulator)
//         dQ_i = dS K                      (TMEM) -> TMA reduce-add into dQacc
//      then writes dK * scale and dV as bf16.
//   3. convert: dQ = bf16(scale * dQacc).
//
// Warp roles of the main kernel (448 threads, see kBwdThreads): two P/dS
// warpgroups (query columns 0-63 and 64-127 of every tile; thread t owns key
// row t = TMEM lane t), the dQ drain / epilogue warpgroup, the TMA producer
// warp and the MMA issuer warp (also TMEM owner).
// TMEM columns: S^T [0,128) (P^T as bf16 pairs inside each warpgroup's half),
// dP^T [128,256) (reused by dQ_i once dS^T is formed), dV and dK after them.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "tiles.cuh"

namespace fa2 {

__device__ int g_bwd_status;

namespace {

// 14 warps: two P/dS warpgroups (0-3 for query columns 0-63 of each tile,
// 4-7 for columns 64-127), the dQ-drain / epilogue warpgroup (8-11), the TMA
// producer (12) and the MMA issuer (13).  Warps spread round-robin over the
// four SM sub-partitions (16K registers each), two of which then hold four
// warps: at most 128 registers per thread (launch bound 512 threads).
constexpr int kBwdThreads = 448;
constexpr int kWarpDrain = 8, kWarpProducer = 12, kWarpMma = 13;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.44269504088896341f;

enum BwdBar {
  kBarKV = 0,
  kBarQFull = 1,     // +stage (2)
  kBarQEmpty = 3,    // +stage: dK(i), the stage's last MMA, is done
  kBarDoFull = 5,    // +stage
  kBarDoEmpty = 7,   // +stage (two dO stages only; with one, dV(i) done frees it)
  kBarSFull = 9,     // S^T in TMEM
  kBarDpFull = 10,   // dP^T in TMEM
  kBarPFull = 11,    // P^T in TMEM (4 warp arrivals)
  kBarDvDone = 12,   // dV(i) MMA done: the P^T columns may be overwritten by S^T(i+1)
  kBarDsFull = 13,   // dS^T in shared memory, dP^T read out (8 warp arrivals)
  kBarDqFull = 15,   // dQ_i in TMEM
  kBarDqDrained = 16,  // dQ_i read out of TMEM (4 warp arrivals)
  kBarAccFull = 17,  // dK, dV complete
  kBarDrain = 18,
  kBarStageFull = 19,  // +buffer (2): dQ chunk staged in shared memory (4 warp arrivals)
  kBarStageFree = 21,  // +buffer (2): the TMA reduce of that chunk has read it
  kBarEpi = 23,        // the 4 drain warps have staged dK, dV for their TMA stores
  kNumBwdBars = 24,
};

template <int D, int DQM = kDqReduce>
struct BwdCfg {
  using T = HeadDim<D>;
  static constexpr int kQStages = 2;
  // Shared memory is full at D = 128 with the dQ staging buffers; without
  // them (atomics) dO gets its second stage back.
  static constexpr int kDoStages = (D == 128 && DQM != kDqAtomic) ? 1 : 2;
  // TMEM: S^T [0,128) (P^T, as bf16 pairs, overwrites columns [0,32) and
  // [64,96): each P/dS warpgroup writes inside its own half),
  // dP^T [128,256) (dQ_i reuses these columns once dS^T is formed), dV and dK
  // after them on 32-column boundaries.
  static constexpr int kCols = D < 32 ? 32 : D;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 128, kColDV = 256, kColDK = 256 + kCols;
  // shared memory
  static constexpr int kK = 0;
  static constexpr int kV = kK + T::kTileBytes;
  static constexpr int kQ = kV + T::kTileBytes;
  static constexpr int kDo = kQ + kQStages * T::kTileBytes;
  // dQ partials leave through two staging buffers of 128 rows x kChunk fp32
  // columns (128B-swizzled, or 64B for D = 16), reduced into the fp32
  // accumulator by TMA.
  static constexpr int kChunk = D < 32 ? D : 32;
  static constexpr int kChunks = D / kChunk;
  static constexpr int kStageBytes = DQM == kDqAtomic ? 0 : 128 * kChunk * 4;
  static constexpr int kDSt = kDo + kDoStages * T::kTileBytes;
  static constexpr int kStage = kDSt + Square::kTileBytes;
  // Per Q stage: -LSE_i * log2 e [128] then -D_i [128] (fp32), written by
  // the producer warp together with the Q_i tile (same full barrier).
  static constexpr int kStats = kStage + 2 * kStageBytes;
  static constexpr int kBars = kStats + kQStages * 256 * 4;
  static constexpr int kTmemSlot = kBars + kNumBwdBars * 8;
  static constexpr int kUsed = kTmemSlot + 16;
  // Request 1 KB of slack to round the base up to 1024 bytes when it fits;
  // otherwise the kernel requires (and checks) an aligned base.
  static constexpr int kMaxSmem = 232448;
  static constexpr int kBytes = kUsed + 1024 <= kMaxSmem ? (kUsed + 1024 > 116 * 1024 ? kUsed + 1024 : 116 * 1024)
                                                         : kUsed;
  static_assert(kUsed <= kMaxSmem, "backward tile does not fit in shared memory");
};

// ---------------------------------------------------------------- preprocess
// D[row] = sum_c dO[row, c] * O[row, c]; also zero the dQ accumulator.
// Blocks take rows from the end, so the rows of the first heads come last:
// the main kernel's first CTAs visit those heads and find their dO, D and
// zeroed dQ rows (and the forward's last O rows) still in L2.
template <int D>
__global__ void __launch_bounds__(256) fa2_bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                                 const __nv_bfloat16* __restrict__ dO,
                                                                 float* __restrict__ Dvec,
                                                                 float* __restrict__ dq_acc, long long rows) {
  constexpr int kTpr = D / 8;  // threads per row, 16 bytes each
  griddep_wait();
  griddep_launch_dependents();
  const long long rb = static_cast<long long>(gridDim.x) - 1 - blockIdx.x;
  const long long row = (rb * blockDim.x + threadIdx.x) / kTpr;
  const int sub = threadIdx.x % kTpr;
  float acc = 0.f;
  if (row < rows) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + sub);
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(dO + row * D) + sub);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa = __bfloat1622float2(pa[e]);
      const float2 fb = __bfloat1622float2(pb[e]);
      acc = fmaf(fa.x, fb.x, acc);
      acc = fmaf(fa.y, fb.y, acc);
    }
  }
#pragma unroll
  for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) Dvec[row] = acc;

  // Zero this row of dQacc (D fp32 = 2 * kTpr 16-byte stores; none when dQ
  // leaves as per-tile partials).
  if (dq_acc == nullptr || row >= rows) return;
  float4* acc4 = reinterpret_cast<float4*>(dq_acc) + row * (D / 4);
  acc4[sub] = make_float4(0.f, 0.f, 0.f, 0.f);
  acc4[sub + kTpr] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------- dQ convert
__global__ void __launch_bounds__(256) fa2_dq_convert_kernel(const float* __restrict__ dq_acc,
                                                             __nv_bfloat16* __restrict__ dq, long long n8,
                                                             float scale) {
  griddep_wait();
  griddep_launch_dependents();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  // From the end: the main kernel's last CTAs reduced into the last heads'
  // rows, which are still in L2 when this kernel starts.
  for (long long j = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; j < n8; j += stride) {
    const long long i = n8 - 1 - j;
    const float4 a = __ldg(reinterpret_cast<const float4*>(dq_acc) + 2 * i);
    const float4 b = __ldg(reinterpret_cast<const float4*>(dq_acc) + 2 * i + 1);
    reinterpret_cast<uint4*>(dq)[i] =
        make_uint4(pack_bf16x2(a.x * scale, a.y * scale), pack_bf16x2(a.z * scale, a.w * scale),
                   pack_bf16x2(b.x * scale, b.y * scale), pack_bf16x2(b.z * scale, b.w * scale));
  }
}

// ---------------------------------------------------------------- main
// VARLEN = true: packed variable-length batch (per-sequence lengths from
// p.cu_q / p.cu_k); otherwise the square [B * H, N, d] problem.
template <int D, bool CAUSAL, bool VARLEN, int DQM>
__global__ void __launch_bounds__(512, 1)
    fa2_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dqacc, const __grid_constant__ CUtensorMap tm_dk,
                   const __grid_constant__ CUtensorMap tm_dv, const BwdProblem p, float scale, float scale_log2) {
  using T = HeadDim<D>;
  using C = BwdCfg<D, DQM>;
  const float* __restrict__ lse = p.lse;
  const float* __restrict__ Dvec = p.Dvec;
  __nv_bfloat16* __restrict__ dk = static_cast<__nv_bfloat16*>(p.dk);
  __nv_bfloat16* __restrict__ dv = static_cast<__nv_bfloat16*>(p.dv);
  const int group = p.group;
  constexpr int SQ = C::kQStages, SD = C::kDoStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int* status = &g_bwd_status;
  if (smem + C::kUsed > smem_raw + C::kBytes) {  // base not 1024-aligned and no slack requested
    if (threadIdx.x == 0) atomicCAS(status, kDevOk, kDevSmemMisaligned);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kTmemSlot);
  float* sStats = reinterpret_cast<float*>(smem + C::kStats);
  const uint32_t sK = smem_u32(smem + C::kK);
  const uint32_t sV = smem_u32(smem + C::kV);
  const uint32_t sQ = smem_u32(smem + C::kQ);
  const uint32_t sDo = smem_u32(smem + C::kDo);
  const uint32_t sDSt = smem_u32(smem + C::kDSt);

  const int warp = warp_id();
  const int lane = lane_id();
  // One CTA per (key/value tile, K/V head) (per sequence when VARLEN); it
  // visits the query tiles of all `group` query heads that share the K/V
  // head, so dK and dV accumulate the group sum in TMEM.  Iteration it covers
  // query head g = it / n_q, query tile i = i_begin + it % n_q.
  // CTAs come in groups of `heads_per_group` K/V heads, so that the group's
  // Q, dO and fp32 dQ rows stay in L2 while its CTAs run; inside a group the
  // key/value tile index is the slow one (causal work shrinks with jt, so
  // heavy tiles go first).
  if constexpr (VARLEN) griddep_wait();  // the geometry below reads cu_seqlens
  const int kv_tiles_grid = ((VARLEN ? p.max_k : p.N) + kTileRows - 1) / kTileRows;
  const int BHkv = VARLEN ? p.Hkv : p.BH / group;
  const int per_batch = BHkv * kv_tiles_grid;
  const int local = VARLEN ? static_cast<int>(blockIdx.x % per_batch) : static_cast<int>(blockIdx.x);
  // Groups of heads_per_group heads; the last one also takes the heads left
  // over, so that its heavy tiles are not few against a short group.
  const int n_groups = max(1, BHkv / p.heads_per_group);
  const int gi = min(local / (p.heads_per_group * kv_tiles_grid), n_groups - 1);
  const int hg0 = gi * p.heads_per_group;
  const int hg = gi == n_groups - 1 ? BHkv - hg0 : p.heads_per_group;
  const int within = local - hg0 * kv_tiles_grid;
  const int jt = within / hg;  // key/value tile
  const int bh_kv = hg0 + within % hg;
  const int kv0 = jt * kTileRows;
  // Query rows, key rows, causal offset (query i sees key j iff j <= i + off)
  // and the first TMA row of the sequence's queries and keys.
  int Nq = p.N, Nk = p.N, off = 0, q_base = 0, k_base = 0;
  if constexpr (VARLEN) {
    const int b = static_cast<int>(blockIdx.x / per_batch);
    const int sq = p.cu_q[b], eq = p.cu_q[b + 1], sk = p.cu_k[b], ek = p.cu_k[b + 1];
    if (!(0 <= sq && sq <= eq && eq <= p.total_q && eq - sq <= p.max_q && 0 <= sk && sk <= ek &&
          ek <= p.total_k && ek - sk <= p.max_k)) {
      if (threadIdx.x == 0) atomicCAS(status, kDevOk, kDevBadSeqlens);
      return;
    }
    Nq = eq - sq;
    Nk = ek - sk;
    off = Nk - Nq;
    q_base = sq;
    k_base = sk;
    if (kv0 >= Nk) return;  // the tile lies past this sequence's keys
  }
  const int num_q_tiles = (Nq + kTileRows - 1) / kTileRows;
  // First query tile that can see a key of this tile (causal): i >= kv0 - off.
  const int i_begin = !CAUSAL ? 0 : (VARLEN ? (kv0 - off > 0 ? (kv0 - off) / kTileRows : 0) : jt);
  const int n_q = num_q_tiles - i_begin;
  const int n_iter = n_q * group;
  if (VARLEN && n_q <= 0) {
    // No query of the sequence sees these keys (Lq = 0): dK = dV = 0.
    const int rows = min(kTileRows, Nk - kv0);
    for (int e = threadIdx.x; e < rows * (D / 8); e += blockDim.x) {
      const size_t at = (static_cast<size_t>(k_base + kv0 + e / (D / 8)) * BHkv + bh_kv) * D + (e % (D / 8)) * 8;
      *reinterpret_cast<uint4*>(dk + at) = make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(dv + at) = make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }

  if (threadIdx.x == kWarpProducer * 32) {
    mbar_init(&bars[kBarKV], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kBarQFull + s], 1);
      mbar_init(&bars[kBarQEmpty + s], 1);
      mbar_init(&bars[kBarDoFull + s], 1);
      mbar_init(&bars[kBarDoEmpty + s], 1);
    }
    mbar_init(&bars[kBarSFull], 1);
    mbar_init(&bars[kBarDpFull], 1);
    mbar_init(&bars[kBarPFull], 8);
    mbar_init(&bars[kBarDvDone], 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kBarStageFull + s], 4);
      mbar_init(&bars[kBarStageFree + s], 1);
    }
    mbar_init(&bars[kBarDsFull], 8);
    mbar_init(&bars[kBarDqFull], 1);
    mbar_init(&bars[kBarDqDrained], 4);
    mbar_init(&bars[kBarAccFull], 1);
    mbar_init(&bars[kBarDrain], 1);
    mbar_init(&bars[kBarEpi], 4);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if constexpr (!VARLEN) griddep_wait();
  griddep_launch_dependents();

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    // Lane 0 issues the TMA loads; all 32 lanes stage -LSE*log2e and -D of
    // the query tile into the Q stage's stats slot before lane 0 arms the
    // stage's full barrier (__syncwarp orders the lanes' stores before it).
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(&bars[kBarKV], 2 * T::kTileBytes);
      for (int b = 0; b < T::kNumBoxes; ++b) {
        tma_load_3d(smem + C::kK + b * T::kBoxBytes, &tm_k, &bars[kBarKV], b * T::kBoxCols, k_base + kv0, bh_kv);
        tma_load_3d(smem + C::kV + b * T::kBoxBytes, &tm_v, &bars[kBarKV], b * T::kBoxCols, k_base + kv0, bh_kv);
      }
    }
    int last_q0 = -1, last_q1 = -1, last_do0 = -1, last_do1 = -1;
    bool ok = true;
#pragma unroll 1
    for (int it = 0; it < n_iter; ++it) {
      const int q0 = (i_begin + it % n_q) * kTileRows;
      const int bh = bh_kv * group + it / n_q;
      {
        const int st = it % SQ, u = it / SQ;
        if (it >= SQ && !(ok = mbar_wait_sleep(&bars[kBarQEmpty + st], (u - 1) & 1, status))) break;
        float* stats = sStats + st * 256;
#pragma unroll
        for (int r = lane; r < 128; r += 32) {
          const int q = q0 + r;
          const bool in = q < Nq;
          // lse [BH, N] and D [BH, N]; packed batches: lse [H, total_q], D [total_q, H]
          const size_t li = VARLEN ? static_cast<size_t>(bh) * p.total_q + q_base + q : static_cast<size_t>(bh) * Nq + q;
          const size_t di = VARLEN ? static_cast<size_t>(q_base + q) * p.H + bh : li;
          stats[r] = in ? -__ldg(lse + li) * kLog2e : -INFINITY;
          stats[128 + r] = in ? -__ldg(Dvec + di) : 0.f;
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[kBarQFull + st], T::kTileBytes);
          for (int b = 0; b < T::kNumBoxes; ++b)
            tma_load_3d(smem + C::kQ + st * T::kTileBytes + b * T::kBoxBytes, &tm_q, &bars[kBarQFull + st],
                        b * T::kBoxCols, q_base + q0, bh);
        }
        (st ? last_q1 : last_q0) = it;
      }
      {
        const int st = it % SD, u = it / SD;
        // (one dO stage: dV(it - 1), the stage's last reader, done frees it)
        if (it >= SD && !(ok = mbar_wait_sleep(&bars[SD == 1 ? kBarDvDone : kBarDoEmpty + st], (u - 1) & 1, status)))
          break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[kBarDoFull + st], T::kTileBytes);
          for (int b = 0; b < T::kNumBoxes; ++b)
            tma_load_3d(smem + C::kDo + st * T::kTileBytes + b * T::kBoxBytes, &tm_do, &bars[kBarDoFull + st],
                        b * T::kBoxCols, q_base + q0, bh);
        }
        (st ? last_do1 : last_do0) = it;
      }
    }
    // Never leave the CTA with a TMA write still landing in shared memory.
    if (lane == 0) {
      mbar_wait(&bars[kBarKV], 0, status);
      if (last_q0 >= 0) mbar_wait(&bars[kBarQFull + 0], (last_q0 / SQ) & 1, status);
      if (last_q1 >= 0) mbar_wait(&bars[kBarQFull + 1], (last_q1 / SQ) & 1, status);
      if (last_do0 >= 0) mbar_wait(&bars[kBarDoFull + 0], (last_do0 / SD) & 1, status);
      if (last_do1 >= 0) mbar_wait(&bars[kBarDoFull + 1], (last_do1 / SD) & 1, status);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdSq = make_idesc_bf16(128, 128, false, false);  // K x Q^T, V x dO^T
      constexpr uint32_t kIdKV = make_idesc_bf16(128, D, false, true);     // P^T x dO, dS^T x Q
      constexpr uint32_t kIdDQ = make_idesc_bf16(128, D, true, true);      // dS x K
      const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP, tDQ = tmem + C::kColDQ,
                     tDV = tmem + C::kColDV, tDK = tmem + C::kColDK;
      const uint32_t sK0 = sK, sV0 = sV, sDSt0 = sDSt, sQ0 = sQ, sDo0 = sDo;
      // Issue order per query tile i (S^T(i) is issued one tile ahead so the
      // compute warps find it ready when they finish dS(i-1)):
      //   dP^T(i), dV(i), S^T(i+1), dQ(i), dK(i)
      auto issue_s = [&](int it) -> bool {
        const int qs = it % SQ;
        if (!mbar_wait(&bars[kBarQFull + qs], (it / SQ) & 1, status)) return false;
        uint32_t sK = sK0, sQ = sQ0;
        opaque(sK);
        opaque(sQ);
        const uint32_t q_s = sQ + qs * T::kTileBytes;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tS, T::kmajor_desc(sK, kk), T::kmajor_desc(q_s, kk), kIdSq, kk > 0 ? 1u : 0u);
        mma_commit(&bars[kBarSFull]);
        return true;
      };
      bool ok = mbar_wait(&bars[kBarKV], 0, status) && issue_s(0);
#pragma unroll 1
      for (int it = 0; ok && it < n_iter; ++it) {
        const int qs = it % SQ, ds = it % SD, du = it / SD;
        // Rebuild each operand's base descriptor every iteration instead of
        // keeping ~40 hoisted 64-bit descriptors live; each K step then adds
        // its offset to the base (one 32-bit add, tiles.cuh).  The issuing
        // thread shares its SM sub-partition with three busy warps, so its
        // instruction count per MMA sets how fast it can feed the tensor
        // core: stepping the descriptors instead of rebuilding them per MMA
        // made this kernel 5-8 % faster.
        uint32_t sK = sK0, sV = sV0, sDSt = sDSt0, sQ = sQ0, sDo = sDo0;
        opaque(sK); opaque(sV); opaque(sDSt); opaque(sQ); opaque(sDo);
        const uint32_t q_s = sQ + qs * T::kTileBytes, do_s = sDo + ds * T::kTileBytes;
        // dP^T = V dO_i^T into the columns dQ(i-1) occupied.
        if (!(ok = it >= 1 ? mbar_wait2(&bars[kBarDoFull + ds], du & 1, &bars[kBarDqDrained], (it - 1) & 1, status)
                           : mbar_wait(&bars[kBarDoFull + ds], du & 1, status)))
          break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_bf16_ss(tDP, T::kmajor_desc(sV, kk), T::kmajor_desc(do_s, kk), kIdSq, kk > 0 ? 1u : 0u);
        mma_commit(&bars[kBarDpFull]);
        // dV += P^T dO_i, P^T read from TMEM: query columns [0, 64) as bf16
        // pairs in S^T columns [0, 32), columns [64, 128) in [64, 96).
        if (!(ok = mbar_wait(&bars[kBarPFull], it & 1, status))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTileRows / 16; ++kk)
          mma_bf16_ts(tDV, tS + (kk < 4 ? 8 * kk : 64 + 8 * (kk - 4)), T::mnmajor_desc(do_s, kk), kIdKV,
                      (it > 0 || kk > 0) ? 1u : 0u);
        if constexpr (SD > 1) mma_commit(&bars[kBarDoEmpty + ds]);
        mma_commit(&bars[kBarDvDone]);
        // dQ_i = dS K (dS read as the MN-major view of dS^T)
        auto issue_dq = [&]() {
        if constexpr (DQM == kDqAtomic) {
          // dQ_i^T = K^T dS^T: the same two MN-major tiles with their roles
          // swapped (D = 128, so both are 128 x 128 and the instruction
          // descriptor is unchanged).  TMEM lane = head dimension, column =
          // query row, so a warp's 32 lanes hold 32 consecutive elements of a
          // dQ row.
          static_assert(DQM != kDqAtomic || D == 128, "transposed dQ needs D = 128");
#pragma unroll
          for (int kk = 0; kk < kTileRows / 16; ++kk)
            mma_bf16_ss(tDQ, T::mnmajor_desc(sK, kk), Square::mnmajor_desc(sDSt, kk), kIdDQ, kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < kTileRows / 16; ++kk)
            mma_bf16_ss(tDQ, Square::mnmajor_desc(sDSt, kk), T::mnmajor_desc(sK, kk), kIdDQ, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars[kBarDqFull]);
        };
        // S^T(i+1) overwrites the P^T columns dV(i) reads: wait for dV(i).
        // If dS(i) is ready when three quarters of S^T(i+1) are issued, dQ(i)
        // goes out before the last quarter: dQ(i) is on the kernel's critical
        // loop (dQ -> drain -> dP^T(i+1) -> dS(i+1) -> dQ(i+1)), and the P/dS
        // warps, which need S^T(i+1) right after dS(i), lose less by the
        // delay.  (Checking earlier in S^T(i+1) was slower; +1.8-2.5 %.)
        bool dq_done = false;
        if (it + 1 < n_iter) {
          const int qn = (it + 1) % SQ;
          if (!(ok = mbar_wait2(&bars[kBarDvDone], it & 1, &bars[kBarQFull + qn], ((it + 1) / SQ) & 1, status))) break;
          const uint32_t q_n = sQ + qn * T::kTileBytes;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            if (kk == 3 * (D / 16) / 4 && !dq_done && mbar_test_wait(&bars[kBarDsFull], it & 1)) {
              tc_fence_after();
              issue_dq();
              dq_done = true;
            }
            mma_bf16_ss(tS, T::kmajor_desc(sK, kk), T::kmajor_desc(q_n, kk), kIdSq, kk > 0 ? 1u : 0u);
          }
          mma_commit(&bars[kBarSFull]);
        }
        if (!dq_done) {
          if (!(ok = mbar_wait(&bars[kBarDsFull], it & 1, status))) break;
          tc_fence_after();
          issue_dq();
        }
        // dK += dS^T Q_i
#pragma unroll
        for (int kk = 0; kk < kTileRows / 16; ++kk)
          mma_bf16_ss(tDK, Square::kmajor_desc(sDSt, kk), T::mnmajor_desc(q_s, kk), kIdKV,
                      (it > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars[kBarQEmpty + qs]);
      }
      if (ok) mma_commit(&bars[kBarAccFull]);
      mma_commit(&bars[kBarDrain]);
      mbar_wait(&bars[kBarDrain], 0, status);
    }
  } else if (warp < kWarpDrain) {
    // ------------------------------------------------------------ P / dS warps
    // Warpgroup hh handles query columns [64 hh, 64 hh + 64) of every tile;
    // thread t owns key row kv0 + t (TMEM lane t).
    const int hh = warp >> 2;
    const int t = (warp & 3) * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int kv_row = kv0 + t;
    const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
    bool ok = true;
#pragma unroll 1
    for (int it = 0; it < n_iter; ++it) {
      const int i = i_begin + it % n_q;
      const int q0 = i * kTileRows;
      const int qs = it % SQ;
      // The Q stage's full barrier also covers the -LSE / -D the producer
      // staged for this query tile.
      if (!(ok = mbar_wait(&bars[kBarQFull + qs], (it / SQ) & 1, status))) break;
      const float* nlse2 = sStats + qs * 256;  // -LSE_i * log2 e
      const float* nd = nlse2 + 128;           // -D_i

      // P^T = 2^(scale log2e S^T - log2e LSE), masked, kept as packed bf16.
      if (!(ok = mbar_wait(&bars[kBarSFull], it & 1, status))) break;
      tc_fence_after();
      uint32_t pk[32];  // this half's 64 weights as bf16 pairs
      const bool row_dead = kv_row >= Nk;
      // queries q0 + c with c < first cannot see this key
      const int first = !CAUSAL ? 0 : (VARLEN ? kv_row - off - q0 : (i == jt ? kv_row - q0 : 0));
      // P^T goes back to TMEM as bf16 pairs inside this warpgroup's own S^T
      // columns (the other warpgroup may still be reading its half): the 64
      // weights of columns [64 hh, 64 hh + 64) land in TMEM columns
      // [64 hh, 64 hh + 32), 16 per 32 scores, over S columns already read.
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col0 = 64 * hh + 32 * c;
        float sv[32];
        tmem_ld32(tmem + lane_base + C::kColS + col0, sv);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          // one 16-byte broadcast load of -LSE log2 e for four columns
          const ulonglong2 nl = *reinterpret_cast<const ulonglong2*>(nlse2 + col0 + e);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = col0 + e + 2 * h;
            const float2 xx = f2_unpack(ffma2(f2_pack(sv[e + 2 * h], sv[e + 2 * h + 1]), scale2, h ? nl.y : nl.x));
            float p0 = ex2_approx(xx.x);
            float p1 = ex2_approx(xx.y);
            if (row_dead || col < first) p0 = 0.f;
            if (row_dead || col + 1 < first) p1 = 0.f;
            pk[16 * c + (e + 2 * h) / 2] = pack_bf16x2(p0, p1);
          }
        }
        tmem_st16u(tmem + lane_base + C::kColS + 64 * hh + 16 * c, pk + 16 * c);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarPFull]);

      // dS^T = P^T * (dP^T - D).  The dS^T buffer is free: its last reader,
      // dK(i-1), was issued before dP^T(i) by the same thread, and the
      // commit that completes dP-full tracks every MMA issued before it.
      if (!(ok = mbar_wait(&bars[kBarDpFull], it & 1, status))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col0 = 64 * hh + 32 * c;
        float dp[32];
        tmem_ld32(tmem + lane_base + C::kColDP + col0, dp);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint32_t w[4];
          // -D for these eight columns: two 16-byte broadcast loads
          const ulonglong2 nd01 = *reinterpret_cast<const ulonglong2*>(nd + col0 + e);
          const ulonglong2 nd23 = *reinterpret_cast<const ulonglong2*>(nd + col0 + e + 4);
          const uint64_t ndx[4] = {nd01.x, nd01.y, nd23.x, nd23.y};
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            const uint64_t diff = fadd2(f2_pack(dp[e + 2 * x], dp[e + 2 * x + 1]), ndx[x]);
            const float2 pp = unpack_bf16x2(pk[16 * c + (e + 2 * x) / 2]);
            const float2 ds = f2_unpack(fmul2(f2_pack(pp.x, pp.y), diff));
            w[x] = pack_bf16x2(ds.x, ds.y);
          }
          store_square_chunk(sDSt, t, (col0 + e) / 8, w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarDsFull]);
    }
    tc_fence_before();
  } else if (warp < kWarpProducer) {
    // ------------------------------------------------------------ dQ drain + epilogue warps
    const int t = (warp - kWarpDrain) * 32 + lane;  // TMEM lane: query row q0 + t (dQ), key row kv0 + t (dK, dV)
    const uint32_t lane_base = static_cast<uint32_t>((warp - kWarpDrain) * 32) << 16;
    // dQ_i goes out in kChunk-column pieces: each is read from TMEM (the
    // columns are released after the last piece), written to a swizzled
    // staging buffer and reduce-added (fp32) into dQacc by one TMA bulk tensor
    // op, issued by lane 0 of the first drain warp.  Rows past N fall outside
    // the tensor map and are dropped by TMA.
    const bool issuer = warp == kWarpDrain && lane == 0;
    const uint32_t sStage = smem_u32(smem + C::kStage);
    bool ok = true;
#pragma unroll 1
    for (int it = 0; it < n_iter; ++it) {
      const int i = i_begin + it % n_q;
      const int q0 = i * kTileRows;
      const int bh = bh_kv * group + it / n_q;
      if (!(ok = mbar_wait_sleep(&bars[kBarDqFull], it & 1, status))) break;
      tc_fence_after();
      if constexpr (DQM == kDqAtomic) {
        // dQ_i^T in TMEM: thread t holds head dimension t of every query row
        // (one row per column).  fp32 reductions straight from registers:
        // for each row the warp's 32 lanes add 32 consecutive floats, one
        // 128-byte line per instruction.  Two 32-row pieces at a time; the
        // TMEM columns are released right after the last read.
        const int rows = Nq - q0;  // rows of this tile that exist (>= 1)
        float* dst = p.dq_buf + (static_cast<size_t>(bh) * Nq + q0) * D + t;
        float g2[2][32];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          tmem_ld32(tmem + lane_base + C::kColDQ + 64 * h2, g2[0]);
          tmem_ld32(tmem + lane_base + C::kColDQ + 64 * h2 + 32, g2[1]);
          tmem_wait_ld();
          if (h2 == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kBarDqDrained]);
          }
          if (rows >= kTileRows) {
#pragma unroll
            for (int pc = 0; pc < 2; ++pc)
#pragma unroll
              for (int j = 0; j < 32; ++j) red_add_f32(dst + static_cast<size_t>(64 * h2 + 32 * pc + j) * D, g2[pc][j]);
          } else {
#pragma unroll
            for (int pc = 0; pc < 2; ++pc)
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (64 * h2 + 32 * pc + j < rows) red_add_f32(dst + static_cast<size_t>(64 * h2 + 32 * pc + j) * D, g2[pc][j]);
          }
        }
        continue;
      }
      // The first three pieces are read from TMEM at once (96 registers),
      // the fourth as soon as the first is staged, and the columns are
      // released right after that read (before the first reduce-add is
      // issued, which waits for the previous one to have read its source):
      // dP^T(i+1) reuses them, so only one piece's staging lies between dQ
      // landing and the release (+2 % over releasing after that reduce).
      constexpr int kFirst = C::kChunks < 3 ? C::kChunks : 3;
      float g[3][C::kChunk];
#pragma unroll
      for (int k = 0; k < kFirst; ++k) {
        if constexpr (C::kChunk == 32)
          tmem_ld32(tmem + lane_base + C::kColDQ + k * 32, g[k]);
        else
          tmem_ld16(tmem + lane_base + C::kColDQ, g[k]);
      }
      tmem_wait_ld();
      if (C::kChunks == kFirst) {  // every dQ column has been read: release the TMEM columns
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarDqDrained]);
      }
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c) {
        const int gi = it * C::kChunks + c, bsel = gi & 1, u = gi >> 1;
        const int slot = c == 3 ? 0 : c;
        if (gi >= 2 && !(ok = mbar_wait_sleep(&bars[kBarStageFree + bsel], (u - 1) & 1, status))) break;
        const uint32_t sb = sStage + bsel * C::kStageBytes;
#pragma unroll
        for (int j = 0; j < C::kChunk / 4; ++j) {
          const float* v4 = g[slot] + 4 * j;
          st_shared_v4(sb + swizzle_offset<C::kChunk * 4>(t, j), __float_as_uint(v4[0]), __float_as_uint(v4[1]),
                       __float_as_uint(v4[2]), __float_as_uint(v4[3]));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kBarStageFull + bsel]);
        if constexpr (C::kChunks == 4) {
          if (c == 0) {  // piece 3 into piece 0's registers (just staged), then release
            tmem_ld32(tmem + lane_base + C::kColDQ + 3 * 32, g[0]);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kBarDqDrained]);
          }
        }
        if (issuer) {
          if ((ok = mbar_wait(&bars[kBarStageFull + bsel], u & 1, status))) {
            if constexpr (DQM == kDqSplit) {
              // this (query tile, key tile) pair's own partial slot
              const int nq_t = num_q_tiles;
              const long long pair = CAUSAL ? static_cast<long long>(bh) * nq_t * (nq_t + 1) / 2 +
                                                  static_cast<long long>(i) * (i + 1) / 2 + jt
                                            : (static_cast<long long>(bh) * nq_t + i) * kv_tiles_grid + jt;
              tma_store_3d(&tm_dqacc, sb, c * C::kChunk, 0, static_cast<int>(pair));
            } else {
              tma_reduce_add_3d(&tm_dqacc, sb, c * C::kChunk, q_base + q0, bh);
            }
            bulk_commit_group();
            // The previous chunk's reduce (other buffer) has read its source
            // once at most this one is still pending: release that buffer.
            if (gi >= 1) {
              bulk_wait_group_read1();
              mbar_arrive(&bars[kBarStageFree + (bsel ^ 1)]);
            }
          }
        }
        __syncwarp();
        if (!ok) break;
      }
      if (!ok) break;
    }
    if (issuer) bulk_wait_group0();  // every reduce / store has landed before the CTA exits
    // ------------------------------------------------------------ epilogue: dV, dK * scale -> bf16
    // dK, dV (D >= 64) leave by TMA stores; in a packed batch only a key
    // tile that lies inside its sequence does so (the rows past a sequence
    // belong to the next one), the others store directly.
    const bool tma_kv = D >= 64 && (!VARLEN || kv0 + kTileRows <= Nk);
    if (ok && mbar_wait_sleep(&bars[kBarAccFull], 0, status)) {
      tc_fence_after();
      if (tma_kv) {
      // Every MMA has completed, so the Q stages are free: dV goes to stage 0
      // and dK to stage 1 in the layout a TMA load of a K tile produces, and
      // leaves by TMA stores (rows past N are dropped).  The CTA exits once
      // the stores have read shared memory; the writes drain while the next
      // CTA on this SM starts.
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? C::kColDV : C::kColDK;
        const float mul = which == 0 ? 1.f : scale;
        const uint32_t tile = smem_u32(smem + C::kQ + which * T::kTileBytes);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float g[32];
          tmem_ld32(tmem + lane_base + col + c * 32, g);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int chunk = c * 4 + q;  // 8 columns
            st_shared_v4(tile + (chunk >> 3) * T::kBoxBytes + sw128_offset(t, chunk & 7),
                         pack_bf16x2(g[8 * q + 0] * mul, g[8 * q + 1] * mul),
                         pack_bf16x2(g[8 * q + 2] * mul, g[8 * q + 3] * mul),
                         pack_bf16x2(g[8 * q + 4] * mul, g[8 * q + 5] * mul),
                         pack_bf16x2(g[8 * q + 6] * mul, g[8 * q + 7] * mul));
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarEpi]);
      if (issuer && mbar_wait(&bars[kBarEpi], 0, status)) {
#pragma unroll
        for (int which = 0; which < 2; ++which)
#pragma unroll
          for (int b = 0; b < T::kNumBoxes; ++b)
            tma_store_3d(which == 0 ? &tm_dv : &tm_dk, smem_u32(smem + C::kQ + which * T::kTileBytes) + b * T::kBoxBytes,
                         b * T::kBoxCols, k_base + kv0, bh_kv);
        bulk_commit_group();
        bulk_wait_group_read0();
      }
      } else {
      const int kv_row = kv0 + t;
      const bool valid = kv_row < Nk;
      const int vrow = valid ? kv_row : 0;
      const size_t off = VARLEN ? (static_cast<size_t>(k_base + vrow) * BHkv + bh_kv) * D
                                : (static_cast<size_t>(bh_kv) * Nk + vrow) * D;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col = which == 0 ? C::kColDV : C::kColDK;
        const float mul = which == 0 ? 1.f : scale;
        uint4* dst = reinterpret_cast<uint4*>((which == 0 ? dv : dk) + off);
        if constexpr (D >= 32) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float g[32];
            tmem_ld32(tmem + lane_base + col + c * 32, g);
            tmem_wait_ld();
            if (valid) {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                dst[c * 4 + q] = make_uint4(pack_bf16x2(g[8 * q + 0] * mul, g[8 * q + 1] * mul),
                                            pack_bf16x2(g[8 * q + 2] * mul, g[8 * q + 3] * mul),
                                            pack_bf16x2(g[8 * q + 4] * mul, g[8 * q + 5] * mul),
                                            pack_bf16x2(g[8 * q + 6] * mul, g[8 * q + 7] * mul));
            }
          }
        } else {
          float g[16];
          tmem_ld16(tmem + lane_base + col, g);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int q = 0; q < 2; ++q)
              dst[q] = make_uint4(pack_bf16x2(g[8 * q + 0] * mul, g[8 * q + 1] * mul),
                                  pack_bf16x2(g[8 * q + 2] * mul, g[8 * q + 3] * mul),
                                  pack_bf16x2(g[8 * q + 4] * mul, g[8 * q + 5] * mul),
                                  pack_bf16x2(g[8 * q + 6] * mul, g[8 * q + 7] * mul));
          }
        }
      }
      }
    }
    tc_fence_before();
  }

  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
int launch_preprocess_t(const void* o, const void* dO, float* Dvec, float* dq_acc, long long rows,
                        cudaStream_t stream) {
  constexpr int kTpr = D / 8;
  const long long threads = rows * kTpr;
  const long long blocks = (threads + 255) / 256;
  return launch_pdl(fa2_bwd_preprocess_kernel<D>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                    static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), Dvec, dq_acc, rows);
}

template <int D, bool CAUSAL, bool VARLEN, int DQM>
int launch_bwd_main_k(const TmapSet& tm, BwdProblem p, float scale, cudaStream_t stream) {
  using C = BwdCfg<D, DQM>;
  const bool varlen = VARLEN;
  auto kern = fa2_bwd_kernel<D, CAUSAL, VARLEN, DQM>;
  if (int rc = ensure_max_smem(reinterpret_cast<const void*>(kern), C::kBytes)) return rc;
  const int rows_q = varlen ? p.max_q : p.N;
  const int num_kv_tiles = ((varlen ? p.max_k : p.N) + kTileRows - 1) / kTileRows;
  const int kv_heads = varlen ? p.Hkv : p.BH / p.group;
  const dim3 grid(static_cast<unsigned>(num_kv_tiles) * static_cast<unsigned>(kv_heads) *
                  static_cast<unsigned>(varlen ? p.batches : 1));
  // Bytes one K/V head's CTAs keep re-reading: Q, dO (bf16), the fp32 dQ
  // accumulator and LSE, D of its `group` query heads.
  const size_t per_head = static_cast<size_t>(p.group) * rows_q * (static_cast<size_t>(D) * 8 + 8);
  p.heads_per_group = heads_per_l2_group(per_head, kv_heads, kL2GroupBytesBwd);
  return launch_pdl(kern, grid, dim3(kBwdThreads), C::kBytes, stream, tm.q, tm.k, tm.v, tm.dO, tm.dqacc, tm.dk, tm.dv, p,
                    scale, scale * kLog2e);
}

// The atomic and split dQ modes are compiled for d = 128 square problems only.
template <int D, bool CAUSAL>
int launch_bwd_main_t(const TmapSet& tm, const BwdProblem& p, float scale, cudaStream_t stream) {
  if (p.cu_q != nullptr) {
    if (p.dq_mode != kDqReduce) return static_cast<int>(cudaErrorInvalidValue);
    return launch_bwd_main_k<D, CAUSAL, true, kDqReduce>(tm, p, scale, stream);
  }
  if constexpr (D == 128) {
    if (p.dq_mode == kDqAtomic) return launch_bwd_main_k<D, CAUSAL, false, kDqAtomic>(tm, p, scale, stream);
    if (p.dq_mode == kDqSplit) return launch_bwd_main_k<D, CAUSAL, false, kDqSplit>(tm, p, scale, stream);
  }
  if (p.dq_mode != kDqReduce) return static_cast<int>(cudaErrorInvalidValue);
  return launch_bwd_main_k<D, CAUSAL, false, kDqReduce>(tm, p, scale, stream);
}

// dQ = bf16(scale * sum over key tiles jt, in increasing jt, of the partial
// of (query tile, jt)); thread = 8 columns of one row.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(256) fa2_dq_reduce_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ dq,
                                                            int BH, int N, float scale) {
  griddep_wait();
  griddep_launch_dependents();
  constexpr int kTpr = D / 8;
  const int nq = (N + kTileRows - 1) / kTileRows;
  const long long total = static_cast<long long>(BH) * N * kTpr;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < total; e += stride) {
    const int c8 = static_cast<int>(e % kTpr);
    const long long row = e / kTpr;  // bh * N + n
    const int bh = static_cast<int>(row / N), n = static_cast<int>(row % N);
    const int i = n / kTileRows, r = n % kTileRows;
    const long long first = CAUSAL ? static_cast<long long>(bh) * nq * (nq + 1) / 2 + static_cast<long long>(i) * (i + 1) / 2
                                   : (static_cast<long long>(bh) * nq + i) * nq;
    const int count = CAUSAL ? i + 1 : nq;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int jt = 0; jt < count; ++jt) {
      const float4* src = reinterpret_cast<const float4*>(part + ((first + jt) * kTileRows + r) * D + c8 * 8);
      const float4 a = __ldg(src), b = __ldg(src + 1);
      acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
      acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
    }
    reinterpret_cast<uint4*>(dq + row * D + c8 * 8)[0] =
        make_uint4(pack_bf16x2(acc[0] * scale, acc[1] * scale), pack_bf16x2(acc[2] * scale, acc[3] * scale),
                   pack_bf16x2(acc[4] * scale, acc[5] * scale), pack_bf16x2(acc[6] * scale, acc[7] * scale));
  }
}

int launch_dq_convert(const float* dq_acc, void* dq, long long elems, float scale, cudaStream_t stream) {
  const long long n8 = elems / 8;
  long long blocks = (n8 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  return launch_pdl(fa2_dq_convert_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, dq_acc,
                    static_cast<__nv_bfloat16*>(dq), n8, scale);
}

}  // namespace

int launch_bwd_preprocess(const void* o, const void* dO, float* Dvec, float* dq_acc, int BH, int N, int d,
                          cudaStream_t stream) {
  const long long rows = static_cast<long long>(BH) * N;
  switch (d) {
    case 16: return launch_preprocess_t<16>(o, dO, Dvec, dq_acc, rows, stream);
    case 32: return launch_preprocess_t<32>(o, dO, Dvec, dq_acc, rows, stream);
    case 64: return launch_preprocess_t<64>(o, dO, Dvec, dq_acc, rows, stream);
    case 128: return launch_preprocess_t<128>(o, dO, Dvec, dq_acc, rows, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

int launch_bwd_main(const TmapSet& tm, const BwdProblem& p, int d, float scale, bool causal, cudaStream_t stream) {
  switch (d) {
    case 16: return causal ? launch_bwd_main_t<16, true>(tm, p, scale, stream) : launch_bwd_main_t<16, false>(tm, p, scale, stream);
    case 32: return causal ? launch_bwd_main_t<32, true>(tm, p, scale, stream) : launch_bwd_main_t<32, false>(tm, p, scale, stream);
    case 64: return causal ? launch_bwd_main_t<64, true>(tm, p, scale, stream) : launch_bwd_main_t<64, false>(tm, p, scale, stream);
    case 128:
      return causal ? launch_bwd_main_t<128, true>(tm, p, scale, stream) : launch_bwd_main_t<128, false>(tm, p, scale, stream);
    default: return static_cast<int>(cudaErrorInvalidValue);
  }
}

long long bwd_dq_pairs(int BH, int N, bool causal) {
  const long long nq = (static_cast<long long>(N) + kTileRows - 1) / kTileRows;
  return causal ? BH * (nq * (nq + 1) / 2) : BH * nq * nq;
}

int launch_bwd_dq_reduce(const float* dq_part, void* dq, int BH, int N, int d, float scale, bool causal,
                         cudaStream_t stream) {
  if (d != 128) return static_cast<int>(cudaErrorInvalidValue);
  const long long threads = static_cast<long long>(BH) * N * (128 / 8);
  long long blocks = (threads + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  auto kern = causal ? fa2_dq_reduce_kernel<128, true> : fa2_dq_reduce_kernel<128, false>;
  return launch_pdl(kern, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, dq_part,
                    static_cast<__nv_bfloat16*>(dq), BH, N, scale);
}

int launch_bwd_dq_convert(const float* dq_acc, void* dq, int BH, int N, int d, float scale, cudaStream_t stream) {
  return launch_dq_convert(dq_acc, dq, static_cast<long long>(BH) * N * d, scale, stream);
}

int read_bwd_status(int* value, bool reset) {
  if (cudaError_t e = cudaMemcpyFromSymbol(value, g_bwd_status, sizeof(int))) return static_cast<int>(e);
  if (reset) {
    const int zero = 0;
    if (cudaError_t e = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(int))) return static_cast<int>(e);
  }
  return 0;
}

}  // namespace fa2
