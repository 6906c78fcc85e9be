// Internal interface between the C-ABI entry points (api.cu) and the kernel
// translation units.  Not part of the public header.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa2 {

// TMA descriptors of the [B*H, N, d] views of the operands (bf16), of the
// fp16 copy of V the forward pass reads, and of the fp32 dQ accumulator.
struct TmapSet {
  CUtensorMap q, k, v, v16, dO, dqacc;
  CUtensorMap o;       // forward output (bf16), 32-row boxes
  CUtensorMap dk, dv;  // backward outputs, 128-row boxes
};

// Launch `kern` on `stream` with programmatic stream serialisation (the
// kernel calls griddep_wait() before its first global memory access).
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...));
}

// Every function below returns 0 or the cudaError_t value of the failure.

// Raise a kernel's dynamic shared-memory limit once per (kernel, device).
int ensure_max_smem(const void* kernel, int bytes);

// The attention kernels order their CTAs head-group-major: all CTAs of a
// group of heads run before the next group's, so the rows every CTA of a head
// re-reads (K/V in the forward pass, Q/dO/dQ in the backward pass) are read
// from HBM about once per group instead of once per wave of CTAs.  A group's
// re-read set is kept to about a quarter of the L2 in the forward pass and
// about half of it in the backward pass (measured: at N = 4096 the larger
// backward groups are 3 % faster, the forward is 1 % slower with them).
constexpr size_t kL2GroupBytes = size_t(32) << 20;
constexpr size_t kL2GroupBytesBwd = size_t(64) << 20;
inline int heads_per_l2_group(size_t bytes_per_head, int heads, size_t group_bytes = kL2GroupBytes) {
  size_t g = bytes_per_head ? group_bytes / bytes_per_head : static_cast<size_t>(heads);
  if (g < 1) g = 1;
  if (g > static_cast<size_t>(heads)) g = static_cast<size_t>(heads);
  return static_cast<int>(g);
}

// Forward problem in row-head form.  The query / output tensors are viewed
// as [RH, M, d]; row r of row-head rh is query r % Nq and reads K/V head
// rh / kvdiv ([B * H_kv, Nk, d] view).  Plain attention: RH = B * H, M = Nq,
// kvdiv = H / H_kv.  Packed grouped decoding: RH = B * H_kv, M = (H / H_kv) *
// Nq, kvdiv = 1 (all query heads of a group share one 128-row tile).  With
// causal masking query i sees key j iff j <= i + Nk - Nq.  The keys are cut
// into `splits` ranges of tiles_per_split 128-key tiles; with one split the
// kernel writes bf16 o and lse, with more it writes per-split fp32 results
// to o_part [splits, RH, M, d] / lse_part [splits, RH, M] for
// launch_splitkv_combine.
//
// Variable-length batch (cu_q != nullptr): q, o are packed [total_q, RH, d]
// (RH = H query heads), k, v [total_k, H_kv, d], lse [RH, total_q];
// sequence b owns query rows cu_q[b] .. cu_q[b+1] - 1 and key rows
// cu_k[b] .. cu_k[b+1] - 1 (device arrays of batches + 1 ints), M = max
// query length, Nk = max key length, one split.  Query i of a sequence with
// Lq queries and Lk keys sees key j iff j <= i + Lk - Lq when causal.
//
// Square and variable-length problems run P V on fp16 operands: tm.v16
// describes an fp16 copy of V (same layout) written by launch_v_to_f16, in
// which K/V head h (index along the K/V map's head coordinate) is scaled by
// 1 / v_scale[h] (a power of two, 1 unless the head holds a finite value
// beyond the fp16 range); O of that head is multiplied by v_scale[h].  The
// general (split-KV) form runs P V in bf16 on V itself.
struct FwdProblem {
  int RH, M, Nq, Nk, kvdiv, splits, tiles_per_split;
  int heads_per_group;  // row-heads per CTA group (set by launch_fwd)
  void* o;
  float* lse;
  float* o_part;
  float* lse_part;
  const int* cu_q;
  const int* cu_k;
  int batches, total_q, total_k;
  const float* v_scale;
};

int launch_fwd(const TmapSet& tm, const FwdProblem& p, int d, float scale, bool causal, cudaStream_t stream);
// The fp16 copy of V for the forward pass, in two kernels: (1) v16[e] =
// fp16(v[e]) for the `elems` bf16 values of V, and for every finite value
// beyond the fp16 range v_flags[(e / inner) % heads] = call (the K/V head of
// element e: [heads, N, d] -> inner = N d; packed [total, heads, d] -> inner
// = d); (2) one CTA per K/V head writes v_scale[h] = 1, or, for a flagged
// head, the power of two 2^k that brings its largest finite magnitude into
// the fp16 range and rewrites the head's copy as fp16(v / 2^k).  Element
// (row r, column c) of head h is v[r * row_stride + h * head_stride + c],
// r < rows.  Flags holding another call's number count as clear.  Heads of
// at most 64K elements (rows * d) take one kernel instead: one CTA per head
// copies it and, if it holds such a value, rescales it and sets v_scale[h].
int launch_v_to_f16(const void* v, void* v16, unsigned long long* v_flags, float* v_scale, unsigned long long call,
                    int heads, long long rows, int d, long long row_stride, long long head_stride, bool packed,
                    cudaStream_t stream);
int launch_splitkv_combine(const FwdProblem& p, int d, cudaStream_t stream);
int launch_bwd_preprocess(const void* o, const void* dO, float* Dvec, float* dq_acc, int BH, int N, int d,
                          cudaStream_t stream);
// Backward main-kernel problem.  Square form: BH query heads ([B * H, N, d]
// views, lse and D [B * H, N]); one CTA per (key/value tile, K/V head) loops
// over the `group` query heads that share it, so dk / dv ([B * H / group, N,
// d]) hold the group sums.
//
// Variable-length batch (cu_q != nullptr): q, dO packed [total_q, H, d], k,
// v, dk, dv [total_k, Hkv, d], lse [H, total_q], D [total_q, H] (the
// preprocess kernel's row order); sequence b owns query rows cu_q[b] ..
// cu_q[b+1] - 1 and key rows cu_k[b] .. cu_k[b+1] - 1, at most max_q / max_k
// of each; causal: query i sees key j iff j <= i + Lk - Lq.
//
// dQ leaves the main kernel in one of three ways (dq_mode): kDqReduce, TMA
// bulk reduce-add of each query tile's fp32 partial into the zeroed
// accumulator (tm.dqacc); kDqAtomic, fp32 vector atomics (red.global.add)
// from registers into dq_buf, the zeroed accumulator [B*H, N, d]; kDqSplit,
// TMA store of each (query tile, key tile) partial into its own 128 x d
// slot of dq_buf (tm.dqacc describes [pairs, 128, d]), summed afterwards in
// a fixed order by launch_bwd_dq_reduce (deterministic).  The last two exist
// for d = 128 square problems only.
enum DqMode : int { kDqReduce = 0, kDqAtomic = 1, kDqSplit = 2 };

struct BwdProblem {
  const float* lse;
  const float* Dvec;
  void* dk;
  void* dv;
  int BH, N, group;
  int heads_per_group;  // K/V heads per CTA group (set by launch_bwd_main)
  const int* cu_q;
  const int* cu_k;
  int batches, H, Hkv, total_q, total_k, max_q, max_k;
  int dq_mode;
  float* dq_buf;
};
int launch_bwd_main(const TmapSet& tm, const BwdProblem& p, int d, float scale, bool causal, cudaStream_t stream);
int launch_bwd_dq_convert(const float* dq_acc, void* dq, int BH, int N, int d, float scale, cudaStream_t stream);
// kDqSplit: number of (query tile, key tile) partial slots and the bf16 dQ
// = scale * (sum over key tiles, in increasing order) of the partials.
long long bwd_dq_pairs(int BH, int N, bool causal);
int launch_bwd_dq_reduce(const float* dq_part, void* dq, int BH, int N, int d, float scale, bool causal,
                         cudaStream_t stream);

int read_fwd_status(int* value, bool reset);

// The argument checks of fa2_bwd_gqa_ws (pointers, sizes, head grouping,
// scale, alignment, overlaps): FA2_OK or the fa2_status of the first failure.
int validate_bwd_args(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d, float scale);
// Record a CUDA failure for fa2_last_error_detail; returns FA2_ERR_CUDA.
int record_cuda_failure(int cuda_code, const char* where);
// Unique id of the calling thread's current CUDA context, 0 if none or
// unreadable (changes after cudaDeviceReset).
unsigned long long current_context_id();
int read_bwd_status(int* value, bool reset);

}  // namespace fa2
