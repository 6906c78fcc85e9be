/*
 * fa2.h - C ABI of the GB300 (sm_103a) FlashAttention-2 library.
 *
 * Operation.  Exact scaled-dot-product attention, forward and backward, as
 * described by the article "Revolutionizing Web-Based AI: How a Plain
 * JavaScript Prototype Paved the Way for High-Performance WebGPU Flash
 * Attention 2", section "Translating to WGSL and Optimizing Passes":
 *   - forward: per (batch, head, query tile), walk K and V in blocks with an
 *     online softmax (running max m, running sum l) and never store the
 *     N x N score matrix;
 *   - backward: recompute the attention weights tile by tile from the saved
 *     Q, K and the per-row log-sum-exp (LSE).
 * With S = scale * Q K^T (S[i][j] = -inf for j > i when causal):
 *   LSE_i = ln sum_j exp(S_ij)          O = softmax(S) V
 *   D_i = sum_c dO_ic O_ic              dS = P * (dO V^T - D)
 *   dQ = scale dS K   dK = scale dS^T Q   dV = P^T dO,  P = exp(S - LSE).
 *
 * Layout.  q, k, v, o, dO, dq, dk, dv: bf16 (raw 16-bit storage), row-major
 * contiguous [B, H, N, d].  lse: fp32 [B, H, N], natural log of the scaled,
 * masked scores.  Queries and keys have the same length N.  causal != 0
 * means key j is visible to query i iff j <= i.
 *
 * Pointers.  Every tensor pointer is a DEVICE pointer on the current CUDA
 * device.  bf16 tensors must be 16-byte aligned; lse 4-byte aligned.
 * Outputs must not overlap inputs or each other.  The caller owns all
 * memory; the library keeps no state except one-time kernel attributes.
 *
 * Streams.  `stream` is a cudaStream_t (NULL = legacy default stream).
 * Calls only enqueue work and return; results are valid once the stream
 * has been synchronised.
 *
 * Errors.  Every argument is checked before anything is enqueued; on a bad
 * argument nothing is launched and a nonzero fa2_status is returned.  No
 * entry point aborts, traps or prints.  Kernels bound every internal wait
 * (2 s); a wait that runs out sets a device status word that
 * fa2_device_status() reads.
 */
#ifndef FA2_GB300_H
#define FA2_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA2_OK = 0,
  FA2_ERR_NULL = 1,      /* a required pointer is NULL                      */
  FA2_ERR_SHAPE = 2,     /* B, H or N < 1, or a size beyond the index range */
  FA2_ERR_HEADDIM = 3,   /* d not in {16, 32, 64, 128}                      */
  FA2_ERR_ALIGN = 4,     /* a pointer is not aligned as stated above        */
  FA2_ERR_SCALE = 5,     /* scale not finite or not > 0                     */
  FA2_ERR_ALLOC = 6,     /* stream-ordered workspace allocation failed      */
  FA2_ERR_CUDA = 7,      /* a CUDA runtime / driver call or launch failed   */
  FA2_ERR_WORKSPACE = 8, /* caller workspace NULL, too small or misaligned  */
  FA2_ERR_ALIAS = 9,     /* an output overlaps an input or another output   */
  FA2_ERR_SCRATCH_CAPACITY = 10 /* fa2_bwd_noalloc: problem exceeds its fixed scratch */
} fa2_status;

/*
 * Forward pass.  Writes o [B,H,N,d] bf16 and lse [B,H,N] fp32.
 * Source: the article's forward-pass bullet (blocked K/V walk, online
 * softmax state, no stored score matrix) and backward-pass bullet (the
 * saved log-sum-exp).  Two kernel launches: one writes an fp16 copy of V,
 * the attention kernel then multiplies the weights P with it in fp16 (the
 * weights carry 11 significant bits instead of bf16's 8, which keeps O's
 * error under the parity bound on sharply peaked rows).  A K/V head holding
 * a value of V outside the fp16 range (|v| > 65504) keeps bf16 V and
 * weights.  The scratch (fa2_fwd_workspace_bytes bytes) is obtained with
 * cudaMallocAsync and released with cudaFreeAsync on `stream`.
 */
int fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
            float scale, int causal, void* stream);

/*
 * fa2_fwd with caller-owned scratch: `workspace` (device, 256-byte aligned,
 * not overlapping any argument) of at least fa2_fwd_workspace_bytes(B, H, N,
 * d) bytes (H_kv in place of H for fa2_fwd_gqa_ws); FA2_ERR_WORKSPACE if it
 * is NULL, misaligned or too small, FA2_ERR_ALIAS if it overlaps an input or
 * output.  fa2_fwd_workspace_bytes returns 0 for invalid sizes.
 */
size_t fa2_fwd_workspace_bytes(int B, int H_kv, int N, int d);
int fa2_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
               float scale, int causal, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward pass for L with dL/dO = dO.  Reads q, k, v, the forward's o and
 * lse and dO; writes dq, dk, dv [B,H,N,d] bf16.  Source: the article's
 * backward-pass bullet (recompute P from Q, K and LSE) plus the standard
 * D = rowsum(dO * O) identity.  Enqueues three kernels (D preprocess, main,
 * dQ convert).  Scratch (fa2_bwd_workspace_bytes bytes) is obtained with
 * cudaMallocAsync and released with cudaFreeAsync on `stream`.
 */
int fa2_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
            void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * Grouped-query attention (GQA; multi-query attention when H_kv = 1), named
 * as a next primitive in the article's section "Next Frontiers in WebGPU ML".
 * q, o, dO, dq: [B, H, N, d]; k, v, dk, dv: [B, H_kv, N, d]; lse: [B, H, N];
 * H must be a multiple of H_kv, and query head h attends to key/value head
 * h / (H / H_kv).  dk and dv are the sums over each group of query heads.
 * Same rules and errors as fa2_fwd / fa2_bwd / fa2_bwd_ws (FA2_ERR_SHAPE if
 * H_kv < 1 or H % H_kv != 0); fa2_fwd(...) is fa2_fwd_gqa(..., H_kv = H, ...).
 * The workspace is fa2_bwd_workspace_bytes(B, H, N, d) (query heads).
 */
int fa2_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                int d, float scale, int causal, void* stream);
int fa2_fwd_gqa_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                   int d, float scale, int causal, void* workspace, size_t workspace_bytes, void* stream);
int fa2_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int d, float scale, int causal,
                void* stream);
int fa2_bwd_gqa_ws(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int d, float scale, int causal,
                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * Split-KV forward ("flash-decoding", named as a next primitive in the
 * article's section "Next Frontiers in WebGPU ML"), for queries shorter than
 * the key/value sequence (decoding against a key-value cache).
 * q, o: [B, H, Nq, d]; k, v: [B, H_kv, Nk, d]; lse: [B, H, Nq]; H a multiple
 * of H_kv.  With causal != 0 the Nq queries are the last Nq positions of the
 * Nk-long sequence: query i sees key j iff j <= i + Nk - Nq (Nk >= Nq
 * required).  The G = H / H_kv query heads of a K/V head are packed into the
 * rows of one 128-row tile (G * Nq rows per K/V head), so K and V are read
 * once per group.  The keys are cut into at most num_splits ranges of whole
 * 128-key tiles processed by separate CTAs; each writes its fp32 partial O
 * and LSE to the workspace and a combine kernel merges them with
 * LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
 * workspace: device pointer, 256-byte aligned, of at least
 * fa2_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits) bytes (may be
 * NULL when that is 0, i.e. a single split).  Two launches (one if a single
 * split).  Other rules as fa2_fwd, except that P V runs in bf16 here (no
 * fp16 copy of V: this path's time is the single read of the cache).
 */
size_t fa2_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits);
/*
 * A split count for fa2_fwd_splitkv on a GPU with sm_count SMs: the
 * smallest that gives at least 0.8 * sm_count work units (a unit is one
 * 256-row pair of packed query rows of one K/V head, for one key range), at
 * most one per 128-key tile.  Fewer, longer key ranges stream the cache
 * more efficiently than many short ones once the SMs are busy (measured on
 * GB300, 8 sequences x 8 K/V heads x 16K keys: 2 splits 5.7 TB/s, 4: 5.2,
 * 16: 5.0, 64: 3.0).  Pure arithmetic, no device access.  Returns 0 for
 * invalid arguments (any size < 1, H not a multiple of H_kv).
 */
int fa2_fwd_splitkv_suggest_splits(int sm_count, int B, int H, int H_kv, int Nq, int Nk);
int fa2_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int Nq,
                    int Nk, int d, float scale, int causal, int num_splits, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Variable-length batches (packed sequences).  The pages treat one sequence
 * length per call; this is the usual packed form of the same attention, in
 * the plainest reading: B sequences of different lengths are stored back to
 * back without padding.  q, o, dO, dq: [total_q, H, d]; k, v, dk, dv:
 * [total_k, H_kv, d] (bf16, row-major); lse: fp32 [H, total_q].
 * cu_seqlens_q / cu_seqlens_k: DEVICE int32 arrays of B + 1 offsets, 0 first,
 * non-decreasing, last = total_q / total_k: sequence b owns query rows
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1] - 1 and key rows cu_seqlens_k[b] ..
 * cu_seqlens_k[b+1] - 1 and never sees another sequence.  max_seqlen_q /
 * max_seqlen_k bound every sequence's lengths (they size the grid).  Query
 * head h reads key/value head h / (H / H_kv).  With causal != 0 a sequence's
 * Lq queries are its last Lq positions (key-value-cache alignment): query i
 * sees key j iff j <= i + Lk - Lq; a query that sees no key (Lk = 0, or
 * Lk < Lq when causal) gets o = 0 and lse = -inf and contributes nothing to
 * the gradients.  Rows outside every sequence are not written.
 * The host cannot read the device offsets without a synchronisation, so the
 * kernels check them: a sequence whose offsets are out of order, outside
 * [0, total] or longer than the stated maximum is skipped and the device
 * status word (fa2_device_status) is set to 3.
 * Sizes: B >= 1, total_q, total_k >= 0 (<= 2^30), 0 <= max_seqlen <= total,
 * max_seqlen >= 1 when its total is > 0.  Pointers of tensors with zero rows
 * may be NULL.  fa2_fwd_varlen: two kernel launches (the fp16 copy of V,
 * as in fa2_fwd, in a cudaMallocAsync workspace on `stream`, then the
 * attention kernel; one if total_k is 0).  fa2_bwd_varlen: the same
 * three stages as fa2_bwd_ws with caller scratch of
 * fa2_bwd_varlen_workspace_bytes(H, total_q, d) bytes (256-byte aligned; may
 * be NULL when total_q or total_k is 0, which only zeroes dk, dv or dq).
 */
int fa2_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                   const int* cu_seqlens_k, int B, int H, int H_kv, int total_q, int total_k, int max_seqlen_q,
                   int max_seqlen_k, int d, float scale, int causal, void* stream);
size_t fa2_bwd_varlen_workspace_bytes(int H, int total_q, int d);
int fa2_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                   int H_kv, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d, float scale,
                   int causal, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device scratch fa2_bwd needs: D (fp32 [B,H,N]) and the fp32 dQ
 * accumulator [B,H,N,d], each 256-byte aligned.  0 on invalid sizes. */
size_t fa2_bwd_workspace_bytes(int B, int H, int N, int d);

/* fa2_bwd with caller-provided scratch: `workspace` is a device pointer,
 * 256-byte aligned, of at least fa2_bwd_workspace_bytes(B,H,N,d) bytes,
 * owned by the caller and not used by anything else until the stream has
 * passed this call.  Allocates nothing.  FA2_ERR_WORKSPACE if it is NULL,
 * misaligned or too small, FA2_ERR_ALIAS if its first
 * fa2_bwd_workspace_bytes bytes overlap any tensor of the call. */
int fa2_bwd_ws(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
               void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three stages fa2_bwd / fa2_bwd_ws enqueue, exposed separately so that a
 * caller can time, reorder or overlap them.  Running the three in this order
 * on one stream is exactly fa2_bwd_ws.
 *
 * fa2_bwd_preprocess: Dvec[r] = sum_c dO[r,c] * o[r,c] (fp32 [B,H,N]) and
 *   dq_acc (fp32 [B,H,N,d], 16-byte aligned) set to zero; dq_acc may be NULL
 *   (D only, for FA2_DQ_SPLIT below).  The D identity is the standard FA2
 *   backward identity (the pages do not state it).
 * fa2_bwd_main: recomputes P from q, k and lse tile by tile (the article's
 *   backward-pass bullet), writes dk and dv (bf16) and ADDS the unscaled
 *   dS K into dq_acc with fp32 reduce-adds performed in L2 (TMA bulk
 *   reduce; the order of that sum varies from run to run; the article's
 *   "Numerical Stability and Loss Drift" section notes atomic reductions as
 *   a rounding source).
 * fa2_bwd_dq_convert: dq = bf16(scale * dq_acc).
 * Same pointer, alignment and error rules as above; Dvec and dq_acc are
 * device pointers owned by the caller.
 */
int fa2_bwd_preprocess(const void* o, const void* dO, float* Dvec, float* dq_acc, int B, int H, int N, int d,
                       void* stream);
int fa2_bwd_main(const void* q, const void* k, const void* v, const void* dO, const float* lse, const float* Dvec,
                 float* dq_acc, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                 void* stream);
int fa2_bwd_dq_convert(const float* dq_acc, void* dq, int B, int H, int N, int d, float scale, void* stream);

/*
 * How dQ leaves the main backward kernel (the pages name atomic reductions
 * as a rounding source, section "Numerical Stability and Loss Drift"; the
 * choice among these was made by measurement):
 *   FA2_DQ_REDUCE (0): each (query tile, key tile) partial is reduce-added in
 *     fp32 into the zeroed accumulator by TMA (cp.reduce.async.bulk): the
 *     default of fa2_bwd / fa2_bwd_ws / fa2_bwd_main;
 *   FA2_DQ_ATOMIC (1): the same sums by fp32 vector atomics
 *     (red.global.add.v4.f32) from registers;
 *   FA2_DQ_SPLIT (2): each partial is stored to its own slot and
 *     fa2_bwd_dq_reduce sums the slots in a fixed order (deterministic).
 * fa2_bwd_main_dq is fa2_bwd_main with the mode chosen (modes 1 and 2: d =
 * 128 only, else FA2_ERR_HEADDIM; an unknown mode gives FA2_ERR_SHAPE).
 * dq_buf: the zeroed fp32 accumulator [B,H,N,d] (modes 0 and 1), or
 * fa2_bwd_dq_partials_bytes(B, H, N, d, causal) bytes of partial slots
 * (mode 2; 0 for invalid sizes or d != 128), 16-byte aligned.
 * fa2_bwd_dq_reduce: dq (bf16 [B,H,N,d]) = scale * sum of the slots.
 */
enum { FA2_DQ_REDUCE = 0, FA2_DQ_ATOMIC = 1, FA2_DQ_SPLIT = 2 };
int fa2_bwd_main_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse, const float* Dvec,
                    float* dq_buf, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, int dq_mode,
                    void* stream);
size_t fa2_bwd_dq_partials_bytes(int B, int H, int N, int d, int causal);
int fa2_bwd_dq_reduce(const float* dq_part, void* dq, int B, int H, int N, int d, float scale, int causal,
                      void* stream);

/*
 * Deterministic backward pass (d = 128): the same results as fa2_bwd except
 * that dQ is summed over key tiles in a fixed order (FA2_DQ_SPLIT), so every
 * output is bitwise reproducible run to run.  Caller-owned workspace of
 * fa2_bwd_deterministic_workspace_bytes(B, H, N, d, causal) bytes (256-byte
 * aligned): D plus one 128 x d fp32 slot per (query tile, key tile) pair,
 * i.e. B H (N/128)(N/128 + 1)/2 x 64 KB causal -- gigabytes at N = 16384.
 * Three launches (D, main, ordered reduction).  Other rules as fa2_bwd_ws.
 */
size_t fa2_bwd_deterministic_workspace_bytes(int B, int H, int N, int d, int causal);
int fa2_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                          void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa2_bwd without any device allocation.  The pages describe no such call; it
 * exists for callers that may not allocate device memory themselves (a host
 * framework whose allocator owns all GPU memory, a plugin handed fixed
 * buffers, a latency-critical loop that cannot risk an allocation).  Same
 * arguments, results and errors as fa2_bwd, checked in the same order
 * (pointers, sizes, scale, alignment, overlaps) before anything else; the
 * backward scratch (D and the fp32 dQ accumulator) lives in one statically
 * allocated device array of fa2_noalloc_scratch_capacity() bytes (64 MiB)
 * that every GPU loading this library holds until the process exits.  Valid
 * problems needing more scratch than that (fa2_bwd_workspace_bytes) return
 * FA2_ERR_SCRATCH_CAPACITY before anything is enqueued.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, with
 * that device current), so make that first call before any stream capture.
 * The address belongs to the device's CUDA context: after cudaDeviceReset
 * (or under another context) the next call sees the context change and
 * looks the address up again, so that call too should come before any
 * capture.  Every call shares the array: calls whose GPU work overlaps in
 * time on one device race and give wrong results.  Each call zeroes what
 * must start at zero, so nothing carries over between calls.
 */
int fa2_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                    void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                    void* stream);

/* Bytes of the fixed scratch array fa2_bwd_noalloc uses. */
size_t fa2_noalloc_scratch_capacity(void);

/*
 * One forward and one backward pass whose tensors live in HOST memory: the
 * end-to-end form of fa2_fwd followed by fa2_bwd on the same problem, with
 * the same results (o, lse, dk, dv bit for bit; dq up to the order of its
 * fp32 reduction).  Every (batch, head) is an independent problem (the
 * article's forward-pass bullet: one work unit per batch, head and query
 * tile), so the B*H heads run as a pipeline over groups of heads: while a
 * group's kernels run, later groups upload and earlier ones download.
 *   q, k, v, dO      host bf16 [B,H,N,d] inputs
 *   o, dq, dk, dv    host bf16 [B,H,N,d] outputs; lse host fp32 [B,H,N]
 *   group_heads      host array of num_groups head counts (>= 1, at most 64
 *                    groups) summing to B*H, or NULL for the default plan:
 *                    B*H/8, three groups of B*H/4 and the rest (small first
 *                    and last groups shorten the first upload and the last
 *                    download), or min(B*H, 4) equal groups below 8 heads
 *   compute_streams  1 to 4: groups take turns on `stream` and up to three
 *                    library streams, so that one group's kernels overlap
 *                    the next group's
 *   workspace        device scratch, 256-byte aligned, of at least
 *                    fa2_step_from_host_workspace_bytes(...) bytes with the
 *                    same group plan and stream count: device copies of the
 *                    ten tensors and each compute stream's forward and
 *                    backward scratch; owned by the caller, untouched by
 *                    anything else until `stream` has passed this call.
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to overlap the kernels; pageable memory works but serialises.
 * Copies are plain stream-ordered copies, one per tensor and group, on two
 * library streams (host to device, device to host); the library's streams
 * and events are created on a device's first call and kept (created again
 * after cudaDeviceReset, which gives the device a new context).  The work starts
 * after everything enqueued on `stream` before the call, and `stream` waits
 * for the last download: synchronise it before reading the outputs.  Calls
 * on one device from several host threads are enqueued one at a time.
 * Errors (checked before anything is enqueued): FA2_ERR_NULL for a NULL
 * pointer, FA2_ERR_HEADDIM, FA2_ERR_SHAPE for sizes, an invalid group plan
 * or stream count, FA2_ERR_SCALE, FA2_ERR_WORKSPACE; then FA2_ERR_CUDA if a
 * copy, event or launch fails, or an error of fa2_fwd_ws / fa2_bwd_ws.
 * The workspace size function returns 0 for invalid arguments.
 */
size_t fa2_step_from_host_workspace_bytes(int B, int H, int N, int d, const int* group_heads, int num_groups,
                                          int compute_streams);
int fa2_step_from_host(const void* q, const void* k, const void* v, const void* dO, void* o, float* lse, void* dq,
                       void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                       const int* group_heads, int num_groups, int compute_streams, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Static description of a status code (never NULL). */
const char* fa2_status_string(int status);

/* Read (and if `reset` != 0, clear) the kernels' device status word on the
 * current device: 0 = every wait completed, 1 = some wait timed out,
 * 2 = shared memory base misaligned, 3 = invalid cu_seqlens (varlen calls).
 * Synchronous with respect to the device. Returns an fa2_status. */
int fa2_device_status(int* value, int reset);

/* Text describing the last CUDA failure (FA2_ERR_CUDA / FA2_ERR_ALLOC) an
 * entry point saw on the calling host thread: "where: cudaErrorName (text)".
 * Empty if none.  Valid until the next failing call on the same thread. */
const char* fa2_last_error_detail(void);

/* Failure-detection self-test (no counterpart on the pages): launches a
 * one-CTA kernel that waits on an mbarrier nothing arrives at, bounded by
 * timeout_us (1 .. 5e6) microseconds, synchronises, and stores the kernel's
 * status word in *status_out (1 = the wait timed out and was reported, as
 * every wait in the attention kernels does after 2 s).  Faults nothing. */
int fa2_check_wait_timeout(int timeout_us, int* status_out);

/* ABI version of this header (major * 100 + minor). */
int fa2_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA2_GB300_H */
