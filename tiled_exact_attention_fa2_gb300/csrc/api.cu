// C-ABI entry points declared in include/fa2.h: argument validation, TMA
// descriptor construction and kernel dispatch.  Host code only.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <set>
#include <utility>

#include "fa2.h"
#include "launch.h"

namespace fa2 {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled comes from the driver; fetching it through the
// runtime keeps the library free of a link-time libcuda dependency.
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

constexpr int kRowsPerTile = 128;

// (heads, rows, d) view of a bf16 or fp32 tensor for TMA: coordinates are
// (column, row, head); consecutive rows of a head are row_stride elements
// apart, heads head_stride elements apart.  [B*H, N, d]: row_stride = d,
// head_stride = N d.  Packed [total, H, d]: row_stride = H d, head_stride = d.
// Box = [1, 128 rows, box_cols columns] with the swizzle as wide as the box
// row; rows past `rows` read as zero and are dropped by reduce-adds.
enum class Elem { kBf16, kF16, kF32 };

// Recently encoded tensor maps.  A map is a pure function of the address and
// the layout, so a cached one is exact for the same (address, layout); the
// cache only saves the host time of encoding (a few per call, on the launch
// path of small problems).
struct TmapKey {
  const void* base;
  Elem type;
  int heads, d, box_rows;
  long long rows, row_stride, head_stride;
  bool operator==(const TmapKey& o) const {
    return base == o.base && type == o.type && heads == o.heads && d == o.d && box_rows == o.box_rows &&
           rows == o.rows && row_stride == o.row_stride && head_stride == o.head_stride;
  }
};
constexpr int kTmapCacheSize = 64;
std::mutex g_tmap_mu;
TmapKey g_tmap_keys[kTmapCacheSize];
CUtensorMap g_tmap_vals[kTmapCacheSize];
int g_tmap_count = 0, g_tmap_next = 0;

bool encode_rows_uncached(CUtensorMap* out, const void* base, Elem type, int heads, long long rows, int d,
                          long long row_stride, long long head_stride, int box_rows);

bool encode_rows(CUtensorMap* out, const void* base, Elem type, int heads, long long rows, int d,
                 long long row_stride, long long head_stride, int box_rows = kRowsPerTile) {
  const TmapKey key{base, type, heads, d, box_rows, rows, row_stride, head_stride};
  {
    std::lock_guard<std::mutex> lock(g_tmap_mu);
    for (int i = 0; i < g_tmap_count; ++i)
      if (g_tmap_keys[i] == key) {
        *out = g_tmap_vals[i];
        return true;
      }
  }
  if (!encode_rows_uncached(out, base, type, heads, rows, d, row_stride, head_stride, box_rows)) return false;
  std::lock_guard<std::mutex> lock(g_tmap_mu);
  g_tmap_keys[g_tmap_next] = key;
  g_tmap_vals[g_tmap_next] = *out;
  g_tmap_next = (g_tmap_next + 1) % kTmapCacheSize;
  if (g_tmap_count < kTmapCacheSize) ++g_tmap_count;
  return true;
}

bool encode_rows_uncached(CUtensorMap* out, const void* base, Elem type, int heads, long long rows, int d,
                          long long row_stride, long long head_stride, int box_rows) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const bool f32 = type == Elem::kF32;
  const int esz = f32 ? 4 : 2;
  const int box_cols = f32 ? (d >= 32 ? 32 : d) : (d >= 64 ? 64 : d);
  const int row_bytes = box_cols * esz;
  const CUtensorMapSwizzle swz = row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                   : CU_TENSOR_MAP_SWIZZLE_32B;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_stride) * esz, static_cast<cuuint64_t>(head_stride) * esz};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : (type == Elem::kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
  return enc(out, dt, 3,
             const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [B*H, N, d] bf16 view, box = [1, 128 rows, min(d, 64) columns].
bool make_tmap(CUtensorMap* out, const void* base, int BH, int N, int d, Elem type = Elem::kBf16) {
  return encode_rows(out, base, type, BH, N, d, d, static_cast<long long>(N) * d);
}

// [heads, rows, d] bf16 view of the forward output for its TMA stores: box =
// [1, 32 rows, min(d, 64) columns] (one softmax warp's rows).
bool make_tmap_out(CUtensorMap* out, const void* base, int heads, int rows, int d) {
  return encode_rows(out, base, Elem::kBf16, heads, rows, d, d, static_cast<long long>(rows) * d, 32);
}

// Packed [total, heads, d] bf16 view of the forward output for its TMA
// stores, box = [1, 32 rows, min(d, 64) columns].
bool make_tmap_out_packed(CUtensorMap* out, const void* base, int heads, int total, int d) {
  return encode_rows(out, base, Elem::kBf16, heads, total, d, static_cast<long long>(heads) * d, d, 32);
}

// Packed [total, heads, d] bf16 view (variable-length batches).
bool make_tmap_packed(CUtensorMap* out, const void* base, int heads, int total, int d, Elem type = Elem::kBf16) {
  return encode_rows(out, base, type, heads, total, d, static_cast<long long>(heads) * d, d);
}

// Text of the last CUDA failure seen by an entry point on this host thread.
thread_local char g_last_error[256] = "";

int cuda_fail(int cuda_code, const char* where) {
  const cudaError_t e = static_cast<cudaError_t>(cuda_code);
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return FA2_ERR_CUDA;
}

// [B*H, N, d] fp32 view of the dQ accumulator for TMA reduce-add, box =
// [1, 128 rows, min(d, 32) columns], swizzle = box row width.
bool make_tmap_f32(CUtensorMap* out, const void* base, int BH, int N, int d) {
  return encode_rows(out, base, Elem::kF32, BH, N, d, d, static_cast<long long>(N) * d);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

struct Range {
  uintptr_t lo, hi;
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }
Range range_of(const void* p, size_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return {lo, lo + bytes};
}

int check_sizes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1) return FA2_ERR_SHAPE;
  if (d != 16 && d != 32 && d != 64 && d != 128) return FA2_ERR_HEADDIM;
  const long long BH = static_cast<long long>(B) * H;
  const long long tiles = (static_cast<long long>(N) + kRowsPerTile - 1) / kRowsPerTile;
  // grid = tiles * B * H CTAs (32-bit); TMA dims < 2^32; row indices in int.
  if (BH > 0x7fffffffLL || tiles * BH > 0x7fffffffLL || N > (1 << 30)) return FA2_ERR_SHAPE;
  return FA2_OK;
}

int check_scale(float scale) { return (std::isfinite(scale) && scale > 0.f) ? FA2_OK : FA2_ERR_SCALE; }

constexpr size_t kWsAlign = 256;
size_t round_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

size_t workspace_bytes(int B, int H, int N, int d) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  return round_up(rows * sizeof(float)) + round_up(rows * d * sizeof(float));
}

// Forward workspace: the fp16 copy of V (kv_elems values), then per K/V head
// a 64-bit range flag and the fp32 scale of the head's copy.
size_t fwd_workspace(size_t kv_elems, size_t kv_heads) {
  return round_up(kv_elems * 2) + round_up(kv_heads * sizeof(unsigned long long)) + round_up(kv_heads * sizeof(float));
}

// A number no earlier forward call of this process used: a head's range
// flag counts as set only if it holds the current call's number, so the
// flags need no clearing between calls.
unsigned long long next_fwd_call() {
  static std::atomic<unsigned long long> calls{0};
  return ++calls;
}

// Write the fp16 copy of V (and the per-head scales) into the workspace and
// point p / tm.v16 at it.  V is [heads, rows, d] or packed [rows, heads, d].
int prepare_v16(TmapSet* tm, FwdProblem* p, const void* v, int heads, int rows, int d, bool packed, void* ws,
                cudaStream_t st) {
  const size_t kv_elems = static_cast<size_t>(heads) * rows * d;
  char* w = static_cast<char*>(ws);
  void* v16 = w;
  auto* flags = reinterpret_cast<unsigned long long*>(w + round_up(kv_elems * 2));
  auto* scales = reinterpret_cast<float*>(w + round_up(kv_elems * 2) + round_up(heads * sizeof(unsigned long long)));
  const bool ok = packed ? make_tmap_packed(&tm->v16, v16, heads, rows, d, Elem::kF16)
                         : make_tmap(&tm->v16, v16, heads, rows, d, Elem::kF16);
  if (!ok) return cuda_fail(static_cast<int>(cudaErrorInvalidValue), "tensor map encode");
  p->v_scale = scales;
  const long long row_stride = packed ? static_cast<long long>(heads) * d : d;
  const long long head_stride = packed ? d : static_cast<long long>(rows) * d;
  if (int e = launch_v_to_f16(v, v16, flags, scales, next_fwd_call(), heads, rows, d, row_stride, head_stride, packed,
                              st))
    return cuda_fail(e, "v to f16 launch");
  return FA2_OK;
}

// Query heads H, key/value heads Hkv (H a multiple of Hkv).
int check_heads(int H, int Hkv) { return (Hkv >= 1 && Hkv <= H && H % Hkv == 0) ? FA2_OK : FA2_ERR_SHAPE; }

int validate_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d, float scale) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return FA2_ERR_NULL;
  if (int rc = check_sizes(B, H, N, d)) return rc;
  if (int rc = check_heads(H, Hkv)) return rc;
  if (int rc = check_scale(scale)) return rc;
  const void* bf[] = {q, k, v, o, dO, dq, dk, dv};
  for (const void* p : bf)
    if (!aligned(p, 16)) return FA2_ERR_ALIGN;
  if (!aligned(lse, 4)) return FA2_ERR_ALIGN;
  const size_t tb = static_cast<size_t>(B) * H * N * d * 2;
  const size_t kb = static_cast<size_t>(B) * Hkv * N * d * 2;
  const size_t lb = static_cast<size_t>(B) * H * N * 4;
  const Range outs[] = {range_of(dq, tb), range_of(dk, kb), range_of(dv, kb)};
  const Range ins[] = {range_of(q, tb), range_of(k, kb), range_of(v, kb), range_of(o, tb), range_of(dO, tb),
                       range_of(lse, lb)};
  for (int a = 0; a < 3; ++a) {
    for (const Range& r : ins)
      if (overlap(outs[a], r)) return FA2_ERR_ALIAS;
    for (int b = a + 1; b < 3; ++b)
      if (overlap(outs[a], outs[b])) return FA2_ERR_ALIAS;
  }
  return FA2_OK;
}

int make_tmaps(TmapSet* tm, const void* q, const void* k, const void* v, const void* dO, const float* dq_acc,
               const void* dk, const void* dv, int BH, int BHkv, int N, int d) {
  return (make_tmap(&tm->q, q, BH, N, d) && make_tmap(&tm->k, k, BHkv, N, d) && make_tmap(&tm->v, v, BHkv, N, d) &&
          make_tmap(&tm->dO, dO, BH, N, d) && make_tmap_f32(&tm->dqacc, dq_acc, BH, N, d) &&
          make_tmap(&tm->dk, dk, BHkv, N, d) && make_tmap(&tm->dv, dv, BHkv, N, d))
             ? FA2_OK
             : cuda_fail(static_cast<int>(cudaErrorInvalidValue), "tensor map encode");
}

int run_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse, void* dq,
            void* dk, void* dv, int B, int H, int Hkv, int N, int d, float scale, int causal, void* ws,
            cudaStream_t st) {
  const int BH = B * H;
  const size_t rows = static_cast<size_t>(BH) * N;
  float* Dvec = static_cast<float*>(ws);
  float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(ws) + round_up(rows * sizeof(float)));
  TmapSet tm;
  if (int rc = make_tmaps(&tm, q, k, v, dO, dq_acc, dk, dv, BH, B * Hkv, N, d)) return rc;
  if (int e = launch_bwd_preprocess(o, dO, Dvec, dq_acc, BH, N, d, st)) return cuda_fail(e, "bwd preprocess launch");
  BwdProblem p{};
  p.lse = lse;
  p.Dvec = Dvec;
  p.dk = dk;
  p.dv = dv;
  p.BH = BH;
  p.N = N;
  p.group = H / Hkv;
  if (int e = launch_bwd_main(tm, p, d, scale, causal != 0, st)) return cuda_fail(e, "bwd main launch");
  if (int e = launch_bwd_dq_convert(dq_acc, dq, BH, N, d, scale, st)) return cuda_fail(e, "dq convert launch");
  return FA2_OK;
}

}  // namespace

int validate_bwd_args(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      void* dq, void* dk, void* dv, int B, int H, int Hkv, int N, int d, float scale) {
  return validate_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, Hkv, N, d, scale);
}

int record_cuda_failure(int cuda_code, const char* where) { return cuda_fail(cuda_code, where); }

int ensure_max_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return static_cast<int>(e);
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({kernel, dev})) return 0;
  if (cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes))
    return static_cast<int>(e);
  done.insert({kernel, dev});
  return 0;
}

}  // namespace fa2

using namespace fa2;

extern "C" {

}  // extern "C" (reopened below)

namespace {

int validate_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                 int d, float scale) {
  if (!q || !k || !v || !o || !lse) return FA2_ERR_NULL;
  if (int rc = check_sizes(B, H, N, d)) return rc;
  if (int rc = check_heads(H, H_kv)) return rc;
  if (int rc = check_scale(scale)) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA2_ERR_ALIGN;
  const size_t tb = static_cast<size_t>(B) * H * N * d * 2;
  const size_t kb = static_cast<size_t>(B) * H_kv * N * d * 2;
  const size_t lb = static_cast<size_t>(B) * H * N * 4;
  const Range ro = range_of(o, tb), rl = range_of(lse, lb);
  const Range ins[] = {range_of(q, tb), range_of(k, kb), range_of(v, kb)};
  for (const Range& r : ins)
    if (overlap(ro, r) || overlap(rl, r)) return FA2_ERR_ALIAS;
  if (overlap(ro, rl)) return FA2_ERR_ALIAS;
  return FA2_OK;
}

// The workspace must not overlap any input or output.
bool fwd_ws_overlaps(const void* ws, size_t ws_bytes, const void* q, const void* k, const void* v, const void* o,
                     const float* lse, int B, int H, int H_kv, int N, int d) {
  const size_t tb = static_cast<size_t>(B) * H * N * d * 2;
  const size_t kb = static_cast<size_t>(B) * H_kv * N * d * 2;
  const size_t lb = static_cast<size_t>(B) * H * N * 4;
  const Range rw = range_of(ws, ws_bytes);
  const Range all[] = {range_of(q, tb), range_of(k, kb), range_of(v, kb), range_of(o, tb), range_of(lse, lb)};
  for (const Range& r : all)
    if (overlap(rw, r)) return true;
  return false;
}

// Caller scratch of the backward pass against every tensor of the call.
bool bwd_ws_overlaps(const void* ws, size_t ws_bytes, const void* q, const void* k, const void* v, const void* o,
                     const void* dO, const float* lse, const void* dq, const void* dk, const void* dv, int B, int H,
                     int H_kv, int N, int d) {
  const size_t tb = static_cast<size_t>(B) * H * N * d * 2;
  const size_t kb = static_cast<size_t>(B) * H_kv * N * d * 2;
  const size_t lb = static_cast<size_t>(B) * H * N * 4;
  const Range rw = range_of(ws, ws_bytes);
  const Range all[] = {range_of(q, tb),  range_of(k, kb),  range_of(v, kb),  range_of(o, tb),  range_of(dO, tb),
                       range_of(lse, lb), range_of(dq, tb), range_of(dk, kb), range_of(dv, kb)};
  for (const Range& r : all)
    if (overlap(rw, r)) return true;
  return false;
}

int run_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N, int d,
            float scale, int causal, void* ws, cudaStream_t st) {
  const int BH = B * H;
  TmapSet tm;
  if (!make_tmap(&tm.q, q, BH, N, d) || !make_tmap(&tm.k, k, B * H_kv, N, d) || !make_tmap(&tm.v, v, B * H_kv, N, d) ||
      !make_tmap_out(&tm.o, o, BH, N, d))
    return cuda_fail(static_cast<int>(cudaErrorInvalidValue), "tensor map encode");
  FwdProblem p{};
  p.RH = BH;
  p.M = N;
  p.Nq = N;
  p.Nk = N;
  p.kvdiv = H / H_kv;
  p.splits = 1;
  p.tiles_per_split = (N + kRowsPerTile - 1) / kRowsPerTile;
  p.o = o;
  p.lse = lse;
  if (int rc = prepare_v16(&tm, &p, v, B * H_kv, N, d, false, ws, st)) return rc;
  if (int e = launch_fwd(tm, p, d, scale, causal != 0, st)) return cuda_fail(e, "fwd launch");
  return FA2_OK;
}

}  // namespace

extern "C" {

size_t fa2_fwd_workspace_bytes(int B, int H_kv, int N, int d) {
  if (check_sizes(B, H_kv, N, d) != FA2_OK) return 0;
  return fwd_workspace(static_cast<size_t>(B) * H_kv * N * d, static_cast<size_t>(B) * H_kv);
}

int fa2_fwd_gqa_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                   int d, float scale, int causal, void* workspace, size_t workspace_bytes_given, void* stream) {
  if (int rc = validate_fwd(q, k, v, o, lse, B, H, H_kv, N, d, scale)) return rc;
  const size_t need = fa2_fwd_workspace_bytes(B, H_kv, N, d);
  if (!workspace || !aligned(workspace, kWsAlign) || workspace_bytes_given < need) return FA2_ERR_WORKSPACE;
  if (fwd_ws_overlaps(workspace, need, q, k, v, o, lse, B, H, H_kv, N, d)) return FA2_ERR_ALIAS;
  return run_fwd(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, workspace, static_cast<cudaStream_t>(stream));
}

int fa2_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
               float scale, int causal, void* workspace, size_t workspace_bytes_given, void* stream) {
  return fa2_fwd_gqa_ws(q, k, v, o, lse, B, H, H, N, d, scale, causal, workspace, workspace_bytes_given, stream);
}

int fa2_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int N,
                int d, float scale, int causal, void* stream) {
  if (int rc = validate_fwd(q, k, v, o, lse, B, H, H_kv, N, d, scale)) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = fa2_fwd_workspace_bytes(B, H_kv, N, d);
  void* ws = nullptr;
  if (cudaError_t e = cudaMallocAsync(&ws, bytes, st)) {
    cudaGetLastError();
    cuda_fail(static_cast<int>(e), "cudaMallocAsync");
    return FA2_ERR_ALLOC;
  }
  const int rc = run_fwd(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, ws, st);
  if (cudaError_t e = cudaFreeAsync(ws, st)) return cuda_fail(static_cast<int>(e), "cudaFreeAsync");
  return rc;
}

int fa2_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
            float scale, int causal, void* stream) {
  return fa2_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, scale, causal, stream);
}

}  // extern "C" (reopened below)

namespace {

// Split plan for fa2_fwd_splitkv: at most `requested` ranges of whole
// 128-key tiles, none empty.
void splitkv_plan(int Nk, int requested, int* splits, int* tiles_per_split) {
  const int tiles = (Nk + kRowsPerTile - 1) / kRowsPerTile;
  const int want = requested < 1 ? 1 : (requested > tiles ? tiles : requested);
  *tiles_per_split = (tiles + want - 1) / want;
  *splits = (tiles + *tiles_per_split - 1) / *tiles_per_split;
}

int check_splitkv_sizes(int B, int H, int H_kv, int Nq, int Nk, int d, int causal, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || num_splits < 1) return FA2_ERR_SHAPE;
  if (d != 16 && d != 32 && d != 64 && d != 128) return FA2_ERR_HEADDIM;
  if (int rc = check_heads(H, H_kv)) return rc;
  if (causal && Nk < Nq) return FA2_ERR_SHAPE;
  const long long rows = static_cast<long long>(H / H_kv) * Nq;  // packed rows per K/V head
  const long long rh = static_cast<long long>(B) * H_kv;
  const long long pairs = (rows + 2 * kRowsPerTile - 1) / (2 * kRowsPerTile);
  if (rows > (1 << 30) || Nk > (1 << 30) || rh * pairs * num_splits > 0x7fffffffLL) return FA2_ERR_SHAPE;
  return FA2_OK;
}

}  // namespace

extern "C" {

int fa2_fwd_splitkv_suggest_splits(int sm_count, int B, int H, int H_kv, int Nq, int Nk) {
  if (sm_count < 1 || B < 1 || H < 1 || H_kv < 1 || Nq < 1 || Nk < 1 || H % H_kv != 0) return 0;
  const long long rows = static_cast<long long>(H / H_kv) * Nq;  // packed rows per K/V head
  const long long pairs = ((rows + kRowsPerTile - 1) / kRowsPerTile + 1) / 2;
  const long long units = static_cast<long long>(B) * H_kv * pairs;  // work units per key range
  const long long tiles = (static_cast<long long>(Nk) + kRowsPerTile - 1) / kRowsPerTile;
  const long long want = (4LL * sm_count + 5 * units - 1) / (5 * units);  // ceil(0.8 * sm_count / units)
  return static_cast<int>(want < 1 ? 1 : (want > tiles ? tiles : want));
}

size_t fa2_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || num_splits < 1) return 0;
  if (d != 16 && d != 32 && d != 64 && d != 128) return 0;
  int splits = 0, tps = 0;
  splitkv_plan(Nk, num_splits, &splits, &tps);
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(splits) * B * H * Nq;
  return round_up(rows * d * sizeof(float)) + round_up(rows * sizeof(float));
}

int fa2_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int H_kv, int Nq,
                    int Nk, int d, float scale, int causal, int num_splits, void* workspace,
                    size_t workspace_bytes_given, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA2_ERR_NULL;
  if (int rc = check_splitkv_sizes(B, H, H_kv, Nq, Nk, d, causal, num_splits)) return rc;
  if (int rc = check_scale(scale)) return rc;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return FA2_ERR_ALIGN;
  const size_t qb = static_cast<size_t>(B) * H * Nq * d * 2;
  const size_t kb = static_cast<size_t>(B) * H_kv * Nk * d * 2;
  const size_t lb = static_cast<size_t>(B) * H * Nq * 4;
  const Range ro = range_of(o, qb), rl = range_of(lse, lb);
  const Range ins[] = {range_of(q, qb), range_of(k, kb), range_of(v, kb)};
  for (const Range& r : ins)
    if (overlap(ro, r) || overlap(rl, r)) return FA2_ERR_ALIAS;
  if (overlap(ro, rl)) return FA2_ERR_ALIAS;
  const size_t need = fa2_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits);
  if (need > 0 && (!workspace || !aligned(workspace, kWsAlign) || workspace_bytes_given < need))
    return FA2_ERR_WORKSPACE;

  // Packed grouped rows: the G query heads of a K/V head and their Nq rows
  // form one row-head of G * Nq rows ([B * H_kv, G * Nq, d] view of q / o).
  const int G = H / H_kv;
  FwdProblem p{};
  p.RH = B * H_kv;
  p.M = G * Nq;
  p.Nq = Nq;
  p.Nk = Nk;
  p.kvdiv = 1;
  splitkv_plan(Nk, num_splits, &p.splits, &p.tiles_per_split);
  p.o = o;
  p.lse = lse;
  if (p.splits > 1) {
    const size_t rows = static_cast<size_t>(p.splits) * B * H * Nq;
    p.o_part = static_cast<float*>(workspace);
    p.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + round_up(rows * d * sizeof(float)));
  }
  TmapSet tm;
  if (!make_tmap(&tm.q, q, p.RH, p.M, d) || !make_tmap(&tm.k, k, B * H_kv, Nk, d) ||
      !make_tmap(&tm.v, v, B * H_kv, Nk, d) || !make_tmap_out(&tm.o, o, p.RH, p.M, d))
    return cuda_fail(static_cast<int>(cudaErrorInvalidValue), "tensor map encode");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (int e = launch_fwd(tm, p, d, scale, causal != 0, st)) return cuda_fail(e, "split-kv fwd launch");
  if (p.splits > 1)
    if (int e = launch_splitkv_combine(p, d, st)) return cuda_fail(e, "split-kv combine launch");
  return FA2_OK;
}

size_t fa2_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (check_sizes(B, H, N, d) != FA2_OK) return 0;
  return workspace_bytes(B, H, N, d);
}

int fa2_bwd_gqa_ws(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int d, float scale, int causal,
                   void* workspace, size_t workspace_bytes_given, void* stream) {
  if (int rc = validate_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, H_kv, N, d, scale)) return rc;
  const size_t need = workspace_bytes(B, H, N, d);
  if (!workspace || !aligned(workspace, kWsAlign) || workspace_bytes_given < need) return FA2_ERR_WORKSPACE;
  if (bwd_ws_overlaps(workspace, need, q, k, v, o, dO, lse, dq, dk, dv, B, H, H_kv, N, d)) return FA2_ERR_ALIAS;
  return run_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, H_kv, N, d, scale, causal, workspace,
                 static_cast<cudaStream_t>(stream));
}

int fa2_bwd_ws(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
               void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
               void* workspace, size_t workspace_bytes_given, void* stream) {
  return fa2_bwd_gqa_ws(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, N, d, scale, causal, workspace,
                        workspace_bytes_given, stream);
}

int fa2_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                void* dq, void* dk, void* dv, int B, int H, int H_kv, int N, int d, float scale, int causal,
                void* stream) {
  if (int rc = validate_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, H_kv, N, d, scale)) return rc;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t bytes = workspace_bytes(B, H, N, d);
  void* ws = nullptr;
  if (cudaError_t e = cudaMallocAsync(&ws, bytes, st)) {
    cudaGetLastError();
    cuda_fail(static_cast<int>(e), "cudaMallocAsync");
    return FA2_ERR_ALLOC;
  }
  const int rc = run_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, H_kv, N, d, scale, causal, ws, st);
  if (cudaError_t e = cudaFreeAsync(ws, st)) return cuda_fail(static_cast<int>(e), "cudaFreeAsync");
  return rc;
}

int fa2_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
            void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, void* stream) {
  return fa2_bwd_gqa(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, N, d, scale, causal, stream);
}

int fa2_bwd_preprocess(const void* o, const void* dO, float* Dvec, float* dq_acc, int B, int H, int N, int d,
                       void* stream) {
  if (!o || !dO || !Dvec) return FA2_ERR_NULL;  // dq_acc == NULL: D only
  if (int rc = check_sizes(B, H, N, d)) return rc;
  if (!aligned(o, 16) || !aligned(dO, 16) || !aligned(Dvec, 4) || !aligned(dq_acc, 16)) return FA2_ERR_ALIGN;
  const size_t tb = static_cast<size_t>(B) * H * N * d * 2;
  const Range rd = range_of(Dvec, static_cast<size_t>(B) * H * N * 4);
  const Range ra = range_of(dq_acc, dq_acc ? static_cast<size_t>(B) * H * N * d * 4 : 0);
  const Range ins[] = {range_of(o, tb), range_of(dO, tb)};
  for (const Range& r : ins)
    if (overlap(rd, r) || overlap(ra, r)) return FA2_ERR_ALIAS;
  if (overlap(rd, ra)) return FA2_ERR_ALIAS;
  if (int e = launch_bwd_preprocess(o, dO, Dvec, dq_acc, B * H, N, d, static_cast<cudaStream_t>(stream)))
    return cuda_fail(e, "bwd preprocess launch");
  return FA2_OK;
}

}  // extern "C" (reopened below)

namespace {

// The main backward kernel as a stage: dq_buf is the zeroed fp32 accumulator
// [B, H, N, d] (kDqReduce, kDqAtomic) or the partial slots of
// fa2_bwd_dq_partials_bytes bytes (kDqSplit).
int bwd_main_stage(const void* q, const void* k, const void* v, const void* dO, const float* lse, const float* Dvec,
                   float* dq_buf, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, int dq_mode,
                   cudaStream_t st) {
  if (!q || !k || !v || !dO || !lse || !Dvec || !dq_buf || !dk || !dv) return FA2_ERR_NULL;
  if (int rc = check_sizes(B, H, N, d)) return rc;
  if (int rc = check_scale(scale)) return rc;
  if (dq_mode != kDqReduce && dq_mode != kDqAtomic && dq_mode != kDqSplit) return FA2_ERR_SHAPE;
  if (dq_mode != kDqReduce && d != 128) return FA2_ERR_HEADDIM;
  const void* bf[] = {q, k, v, dO, dk, dv};
  for (const void* p : bf)
    if (!aligned(p, 16)) return FA2_ERR_ALIGN;
  if (!aligned(lse, 4) || !aligned(Dvec, 4) || !aligned(dq_buf, 16)) return FA2_ERR_ALIGN;
  const size_t tb = static_cast<size_t>(B) * H * N * d * 2;
  const size_t lb = static_cast<size_t>(B) * H * N * 4;
  const long long pairs = bwd_dq_pairs(B * H, N, causal != 0);
  const size_t qb = dq_mode == kDqSplit ? static_cast<size_t>(pairs) * kRowsPerTile * d * 4 : tb * 2;
  const Range outs[] = {range_of(dk, tb), range_of(dv, tb), range_of(dq_buf, qb)};
  const Range ins[] = {range_of(q, tb), range_of(k, tb), range_of(v, tb), range_of(dO, tb), range_of(lse, lb),
                       range_of(Dvec, lb)};
  for (int a = 0; a < 3; ++a) {
    for (const Range& r : ins)
      if (overlap(outs[a], r)) return FA2_ERR_ALIAS;
    for (int b = a + 1; b < 3; ++b)
      if (overlap(outs[a], outs[b])) return FA2_ERR_ALIAS;
  }
  TmapSet tm;
  if (int rc = make_tmaps(&tm, q, k, v, dO, dq_buf, dk, dv, B * H, B * H, N, d)) return rc;
  if (dq_mode == kDqSplit &&
      !encode_rows(&tm.dqacc, dq_buf, Elem::kF32, static_cast<int>(pairs), kRowsPerTile, d, d,
                   static_cast<long long>(kRowsPerTile) * d))
    return cuda_fail(static_cast<int>(cudaErrorInvalidValue), "tensor map encode");
  BwdProblem p{};
  p.lse = lse;
  p.Dvec = Dvec;
  p.dk = dk;
  p.dv = dv;
  p.BH = B * H;
  p.N = N;
  p.group = 1;
  p.dq_mode = dq_mode;
  p.dq_buf = dq_buf;
  if (int e = launch_bwd_main(tm, p, d, scale, causal != 0, st)) return cuda_fail(e, "bwd main launch");
  return FA2_OK;
}

}  // namespace

extern "C" {

int fa2_bwd_main(const void* q, const void* k, const void* v, const void* dO, const float* lse, const float* Dvec,
                 float* dq_acc, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                 void* stream) {
  return bwd_main_stage(q, k, v, dO, lse, Dvec, dq_acc, dk, dv, B, H, N, d, scale, causal, kDqReduce,
                        static_cast<cudaStream_t>(stream));
}

size_t fa2_bwd_dq_partials_bytes(int B, int H, int N, int d, int causal) {
  if (check_sizes(B, H, N, d) != FA2_OK || d != 128) return 0;
  return static_cast<size_t>(bwd_dq_pairs(B * H, N, causal != 0)) * kRowsPerTile * d * sizeof(float);
}

int fa2_bwd_main_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse, const float* Dvec,
                    float* dq_buf, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal, int dq_mode,
                    void* stream) {
  return bwd_main_stage(q, k, v, dO, lse, Dvec, dq_buf, dk, dv, B, H, N, d, scale, causal, dq_mode,
                        static_cast<cudaStream_t>(stream));
}

int fa2_bwd_dq_reduce(const float* dq_part, void* dq, int B, int H, int N, int d, float scale, int causal,
                      void* stream) {
  if (!dq_part || !dq) return FA2_ERR_NULL;
  if (int rc = check_sizes(B, H, N, d)) return rc;
  if (d != 128) return FA2_ERR_HEADDIM;
  if (int rc = check_scale(scale)) return rc;
  if (!aligned(dq_part, 16) || !aligned(dq, 16)) return FA2_ERR_ALIGN;
  const size_t pb = fa2_bwd_dq_partials_bytes(B, H, N, d, causal);
  if (overlap(range_of(dq_part, pb), range_of(dq, static_cast<size_t>(B) * H * N * d * 2))) return FA2_ERR_ALIAS;
  if (int e = launch_bwd_dq_reduce(dq_part, dq, B * H, N, d, scale, causal != 0, static_cast<cudaStream_t>(stream)))
    return cuda_fail(e, "dq reduce launch");
  return FA2_OK;
}

size_t fa2_bwd_deterministic_workspace_bytes(int B, int H, int N, int d, int causal) {
  const size_t pb = fa2_bwd_dq_partials_bytes(B, H, N, d, causal);
  if (pb == 0) return 0;
  return round_up(static_cast<size_t>(B) * H * N * sizeof(float)) + round_up(pb);
}

int fa2_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                          void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                          void* workspace, size_t workspace_bytes_given, void* stream) {
  if (int rc = validate_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, H, N, d, scale)) return rc;
  if (d != 128) return FA2_ERR_HEADDIM;
  const size_t need = fa2_bwd_deterministic_workspace_bytes(B, H, N, d, causal);
  if (!workspace || !aligned(workspace, kWsAlign) || workspace_bytes_given < need) return FA2_ERR_WORKSPACE;
  if (bwd_ws_overlaps(workspace, need, q, k, v, o, dO, lse, dq, dk, dv, B, H, H, N, d)) return FA2_ERR_ALIAS;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* Dvec = static_cast<float*>(workspace);
  float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                         round_up(static_cast<size_t>(B) * H * N * sizeof(float)));
  // D only: the partial slots are written whole, nothing to zero.
  if (int e = launch_bwd_preprocess(o, dO, Dvec, nullptr, B * H, N, d, st)) return cuda_fail(e, "bwd preprocess launch");
  if (int rc = bwd_main_stage(q, k, v, dO, lse, Dvec, part, dk, dv, B, H, N, d, scale, causal, kDqSplit, st))
    return rc;
  if (int e = launch_bwd_dq_reduce(part, dq, B * H, N, d, scale, causal != 0, st)) return cuda_fail(e, "dq reduce launch");
  return FA2_OK;
}

int fa2_bwd_dq_convert(const float* dq_acc, void* dq, int B, int H, int N, int d, float scale, void* stream) {
  if (!dq_acc || !dq) return FA2_ERR_NULL;
  if (int rc = check_sizes(B, H, N, d)) return rc;
  if (int rc = check_scale(scale)) return rc;
  if (!aligned(dq_acc, 16) || !aligned(dq, 16)) return FA2_ERR_ALIGN;
  const size_t n = static_cast<size_t>(B) * H * N * d;
  if (overlap(range_of(dq_acc, n * 4), range_of(dq, n * 2))) return FA2_ERR_ALIAS;
  if (int e = launch_bwd_dq_convert(dq_acc, dq, B * H, N, d, scale, static_cast<cudaStream_t>(stream)))
    return cuda_fail(e, "dq convert launch");
  return FA2_OK;
}

}  // extern "C" (reopened below)

namespace {

// Sizes of a packed variable-length batch (see fa2_fwd_varlen).
int check_varlen_sizes(int B, int H, int H_kv, int total_q, int total_k, int max_q, int max_k, int d) {
  if (B < 1 || H < 1 || total_q < 0 || total_k < 0 || max_q < 0 || max_k < 0) return FA2_ERR_SHAPE;
  if (d != 16 && d != 32 && d != 64 && d != 128) return FA2_ERR_HEADDIM;
  if (int rc = check_heads(H, H_kv)) return rc;
  if (max_q > total_q || max_k > total_k || total_q > (1 << 30) || total_k > (1 << 30)) return FA2_ERR_SHAPE;
  if ((total_q > 0 && max_q < 1) || (total_k > 0 && max_k < 1)) return FA2_ERR_SHAPE;
  const long long pairs = (static_cast<long long>(max_q) + 2 * kRowsPerTile - 1) / (2 * kRowsPerTile);
  const long long kt = (static_cast<long long>(max_k) + kRowsPerTile - 1) / kRowsPerTile;
  if (static_cast<long long>(B) * H * pairs > 0x7fffffffLL || static_cast<long long>(B) * H_kv * kt > 0x7fffffffLL)
    return FA2_ERR_SHAPE;
  return FA2_OK;
}

size_t varlen_bwd_workspace(int H, int total_q, int d) {
  const size_t rows = static_cast<size_t>(total_q) * H;
  return round_up(rows * sizeof(float)) + round_up(rows * d * sizeof(float));
}

}  // namespace

extern "C" {

int fa2_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                   const int* cu_seqlens_k, int B, int H, int H_kv, int total_q, int total_k, int max_seqlen_q,
                   int max_seqlen_k, int d, float scale, int causal, void* stream) {
  if (int rc = check_varlen_sizes(B, H, H_kv, total_q, total_k, max_seqlen_q, max_seqlen_k, d)) return rc;
  if (int rc = check_scale(scale)) return rc;
  if (total_q == 0) return FA2_OK;  // no query rows: nothing to write
  if (!q || !o || !lse || !cu_seqlens_q || !cu_seqlens_k || (total_k > 0 && (!k || !v))) return FA2_ERR_NULL;
  if (!aligned(q, 16) || !aligned(o, 16) || !aligned(lse, 4) || !aligned(cu_seqlens_q, 4) ||
      !aligned(cu_seqlens_k, 4) || (total_k > 0 && (!aligned(k, 16) || !aligned(v, 16))))
    return FA2_ERR_ALIGN;
  const size_t qb = static_cast<size_t>(total_q) * H * d * 2;
  const size_t kb = static_cast<size_t>(total_k) * H_kv * d * 2;
  const size_t lb = static_cast<size_t>(total_q) * H * 4;
  const size_t cb = static_cast<size_t>(B + 1) * 4;
  const Range ro = range_of(o, qb), rl = range_of(lse, lb);
  const Range ins[] = {range_of(q, qb), range_of(k, kb), range_of(v, kb), range_of(cu_seqlens_q, cb),
                       range_of(cu_seqlens_k, cb)};
  for (const Range& r : ins)
    if (overlap(ro, r) || overlap(rl, r)) return FA2_ERR_ALIAS;
  if (overlap(ro, rl)) return FA2_ERR_ALIAS;

  FwdProblem p{};
  p.RH = H;
  p.M = max_seqlen_q;
  p.Nq = max_seqlen_q;
  p.Nk = max_seqlen_k;
  p.kvdiv = H / H_kv;
  p.splits = 1;
  p.tiles_per_split = (max_seqlen_k + kRowsPerTile - 1) / kRowsPerTile;
  p.o = o;
  p.lse = lse;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.batches = B;
  p.total_q = total_q;
  p.total_k = total_k;
  if (max_seqlen_q == 0) return FA2_OK;  // every sequence is empty
  TmapSet tm;
  // With no keys at all the K/V maps are never read; they describe q instead.
  const void* kb_ptr = total_k > 0 ? k : q;
  const void* vb_ptr = total_k > 0 ? v : q;
  const int tk = total_k > 0 ? total_k : 1;
  if (!make_tmap_packed(&tm.q, q, H, total_q, d) || !make_tmap_packed(&tm.k, kb_ptr, H_kv, tk, d) ||
      !make_tmap_packed(&tm.v, vb_ptr, H_kv, tk, d))
    return cuda_fail(static_cast<int>(cudaErrorInvalidValue), "tensor map encode");
  if (!make_tmap_out_packed(&tm.o, o, H, total_q, d))
    return cuda_fail(static_cast<int>(cudaErrorInvalidValue), "tensor map encode");
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (total_k == 0) {  // no keys: V is never read (its maps describe q)
    tm.v16 = tm.v;
    if (int e = launch_fwd(tm, p, d, scale, causal != 0, st)) return cuda_fail(e, "varlen fwd launch");
    return FA2_OK;
  }
  // fp16 copy of the packed V ([total_k, H_kv, d]) in a stream-ordered workspace.
  const size_t kv_elems = static_cast<size_t>(total_k) * H_kv * d;
  void* ws = nullptr;
  if (cudaError_t e = cudaMallocAsync(&ws, fwd_workspace(kv_elems, H_kv), st)) {
    cudaGetLastError();
    cuda_fail(static_cast<int>(e), "cudaMallocAsync");
    return FA2_ERR_ALLOC;
  }
  int rc = prepare_v16(&tm, &p, v, H_kv, total_k, d, true, ws, st);
  if (rc == FA2_OK)
    if (int e = launch_fwd(tm, p, d, scale, causal != 0, st)) rc = cuda_fail(e, "varlen fwd launch");
  if (cudaError_t e = cudaFreeAsync(ws, st)) return cuda_fail(static_cast<int>(e), "cudaFreeAsync");
  return rc;
}

size_t fa2_bwd_varlen_workspace_bytes(int H, int total_q, int d) {
  if (H < 1 || total_q < 0 || total_q > (1 << 30)) return 0;
  if (d != 16 && d != 32 && d != 64 && d != 128) return 0;
  return varlen_bwd_workspace(H, total_q, d);
}

int fa2_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                   void* dq, void* dk, void* dv, const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                   int H_kv, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d, float scale,
                   int causal, void* workspace, size_t workspace_bytes_given, void* stream) {
  if (int rc = check_varlen_sizes(B, H, H_kv, total_q, total_k, max_seqlen_q, max_seqlen_k, d)) return rc;
  if (int rc = check_scale(scale)) return rc;
  const bool has_q = total_q > 0, has_k = total_k > 0;
  if (!cu_seqlens_q || !cu_seqlens_k) return FA2_ERR_NULL;
  if (has_q && (!q || !o || !dO || !lse || !dq)) return FA2_ERR_NULL;
  if (has_k && (!k || !v || !dk || !dv)) return FA2_ERR_NULL;
  if ((has_q && (!aligned(q, 16) || !aligned(o, 16) || !aligned(dO, 16) || !aligned(dq, 16) || !aligned(lse, 4))) ||
      (has_k && (!aligned(k, 16) || !aligned(v, 16) || !aligned(dk, 16) || !aligned(dv, 16))))
    return FA2_ERR_ALIGN;
  const size_t qb = static_cast<size_t>(total_q) * H * d * 2;
  const size_t kb = static_cast<size_t>(total_k) * H_kv * d * 2;
  const size_t lb = static_cast<size_t>(total_q) * H * 4;
  const size_t cb = static_cast<size_t>(B + 1) * 4;
  const Range outs[] = {range_of(dq, qb), range_of(dk, kb), range_of(dv, kb)};
  const Range ins[] = {range_of(q, qb), range_of(k, kb), range_of(v, kb), range_of(o, qb), range_of(dO, qb),
                       range_of(lse, lb), range_of(cu_seqlens_q, cb), range_of(cu_seqlens_k, cb)};
  for (int a = 0; a < 3; ++a) {
    for (const Range& r : ins)
      if (overlap(outs[a], r)) return FA2_ERR_ALIAS;
    for (int b = a + 1; b < 3; ++b)
      if (overlap(outs[a], outs[b])) return FA2_ERR_ALIAS;
  }
  const size_t need = varlen_bwd_workspace(H, total_q, d);
  if (has_q && has_k && (!workspace || !aligned(workspace, kWsAlign) || workspace_bytes_given < need))
    return FA2_ERR_WORKSPACE;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Degenerate batches: no queries means dK = dV = 0, no keys means dQ = 0.
  if (!has_q || !has_k) {
    if (has_k) {
      if (cudaError_t e = cudaMemsetAsync(dk, 0, kb, st)) return cuda_fail(static_cast<int>(e), "memset dk");
      if (cudaError_t e = cudaMemsetAsync(dv, 0, kb, st)) return cuda_fail(static_cast<int>(e), "memset dv");
    }
    if (has_q)
      if (cudaError_t e = cudaMemsetAsync(dq, 0, qb, st)) return cuda_fail(static_cast<int>(e), "memset dq");
    return FA2_OK;
  }
  float* Dvec = static_cast<float*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           round_up(static_cast<size_t>(total_q) * H * sizeof(float)));
  TmapSet tm;
  if (!make_tmap_packed(&tm.q, q, H, total_q, d) || !make_tmap_packed(&tm.k, k, H_kv, total_k, d) ||
      !make_tmap_packed(&tm.v, v, H_kv, total_k, d) || !make_tmap_packed(&tm.dO, dO, H, total_q, d) ||
      !encode_rows(&tm.dqacc, dq_acc, Elem::kF32, H, total_q, d, static_cast<long long>(H) * d, d))
    return cuda_fail(static_cast<int>(cudaErrorInvalidValue), "tensor map encode");
  if (!make_tmap_packed(&tm.dk, dk, H_kv, total_k, d) || !make_tmap_packed(&tm.dv, dv, H_kv, total_k, d))
    return cuda_fail(static_cast<int>(cudaErrorInvalidValue), "tensor map encode");
  // D and the zeroed accumulator in the packed row order ([total_q, H]).
  if (int e = launch_bwd_preprocess(o, dO, Dvec, dq_acc, H, total_q, d, st)) return cuda_fail(e, "bwd preprocess launch");
  BwdProblem p{};
  p.lse = lse;
  p.Dvec = Dvec;
  p.dk = dk;
  p.dv = dv;
  p.BH = H;
  p.N = 0;
  p.group = H / H_kv;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.batches = B;
  p.H = H;
  p.Hkv = H_kv;
  p.total_q = total_q;
  p.total_k = total_k;
  p.max_q = max_seqlen_q;
  p.max_k = max_seqlen_k;
  if (max_seqlen_k > 0)
    if (int e = launch_bwd_main(tm, p, d, scale, causal != 0, st)) return cuda_fail(e, "varlen bwd main launch");
  if (int e = launch_bwd_dq_convert(dq_acc, dq, H, total_q, d, scale, st)) return cuda_fail(e, "dq convert launch");
  return FA2_OK;
}

const char* fa2_status_string(int status) {
  switch (status) {
    case FA2_OK: return "ok";
    case FA2_ERR_NULL: return "a required pointer is NULL";
    case FA2_ERR_SHAPE: return "B, H or N < 1 or beyond the supported index range";
    case FA2_ERR_HEADDIM: return "head dim must be 16, 32, 64 or 128";
    case FA2_ERR_ALIGN: return "pointer misaligned (bf16 tensors need 16 bytes, lse 4)";
    case FA2_ERR_SCALE: return "scale must be finite and > 0";
    case FA2_ERR_ALLOC: return "stream-ordered workspace allocation failed";
    case FA2_ERR_CUDA: return "CUDA call or kernel launch failed";
    case FA2_ERR_WORKSPACE: return "workspace NULL, too small or not 256-byte aligned";
    case FA2_ERR_ALIAS: return "an output overlaps an input or another output";
    case FA2_ERR_SCRATCH_CAPACITY: return "problem needs more scratch than fa2_bwd_noalloc's fixed array holds";
    default: return "unknown fa2 status";
  }
}

int fa2_device_status(int* value, int reset) {
  if (!value) return FA2_ERR_NULL;
  int a = 0, b = 0;
  if (int e = read_fwd_status(&a, reset != 0)) return cuda_fail(e, "read status");
  if (int e = read_bwd_status(&b, reset != 0)) return cuda_fail(e, "read status");
  *value = a > b ? a : b;
  return FA2_OK;
}

int fa2_abi_version(void) { return 101; }

const char* fa2_last_error_detail(void) { return g_last_error; }

}  // extern "C"
