// Internal interface between the C-ABI entry points (api.cu) and the kernel
// translation units.  Not part of the public header.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa2 {

// TMA descriptors of the [B*H, N, d] views of the operands (bf16) and of
// the fp32 dQ accumulator.
struct TmapSet {
  CUtensorMap q, k, v, dO, dqacc;
};

// Every function below returns 0 or the cudaError_t value of the failure.

// Raise a kernel's dynamic shared-memory limit once per (kernel, device).
int ensure_max_smem(const void* kernel, int bytes);

// BH counts query heads (B * H); query head bh reads K/V head bh / group
// (group = H / H_kv, 1 for ordinary attention).
int launch_fwd(const TmapSet& tm, void* o, float* lse, int BH, int N, int d, int group, float scale, bool causal,
               cudaStream_t stream);
int launch_bwd_preprocess(const void* o, const void* dO, float* Dvec, float* dq_acc, int BH, int N, int d,
                          cudaStream_t stream);
// BH counts query heads; one CTA per (key/value tile, K/V head) loops over the
// `group` query heads that share it, so dk / dv ([B * H / group, N, d]) hold
// the group sums.
int launch_bwd_main(const TmapSet& tm, const float* lse, const float* Dvec, void* dk, void* dv, int BH, int N, int d,
                    int group, float scale, bool causal, cudaStream_t stream);
int launch_bwd_dq_convert(const float* dq_acc, void* dq, int BH, int N, int d, float scale, cudaStream_t stream);

int read_fwd_status(int* value, bool reset);
int read_bwd_status(int* value, bool reset);

}  // namespace fa2
