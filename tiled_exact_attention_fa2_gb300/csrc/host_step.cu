// fa2_step_from_host: one forward and backward pass whose tensors live in
// host memory, pipelined over groups of heads.
//
// Every (batch, head) is an independent attention problem (the article's
// forward-pass bullet: one work unit per batch, head and query tile), so the
// B * H heads are split into groups that flow through three stages on their
// own streams: upload (q, k, v, then dO), compute (fa2_fwd_ws, fa2_bwd_ws),
// download (o and lse once the group's forward is done, dq, dk, dv after its
// backward).  Groups take turns on the compute streams, so one group's
// kernels overlap the copies of its neighbours and the causal tail of one
// group overlaps the start of the next.  Only public entry points of this
// library and plain stream-ordered copies are used; the host side only
// enqueues.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa2.h"
#include "launch.h"

namespace {

constexpr int kMaxGroups = 64;
constexpr int kMaxComputeStreams = 4;
constexpr int kMaxDevices = 64;
constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool valid_sizes(int B, int H, int N, int d) {
  return fa2_bwd_workspace_bytes(B, H, N, d) != 0 && fa2_fwd_workspace_bytes(B, H, N, d) != 0;
}

// Group sizes in heads: the caller's, or a ramp (B*H/8, three of B*H/4, the
// rest) whose small first and last groups shorten the first upload and the
// last download while the large middle ones keep the kernels efficient; with
// fewer than 8 heads, min(B*H, 4) equal groups.  Returns the group count, or
// 0 if the caller's list is invalid.
int plan_groups(int BH, const int* group_heads, int num_groups, int* sizes) {
  if (group_heads != nullptr) {
    if (num_groups < 1 || num_groups > kMaxGroups) return 0;
    long long sum = 0;
    for (int c = 0; c < num_groups; ++c) {
      if (group_heads[c] < 1) return 0;
      sizes[c] = group_heads[c];
      sum += group_heads[c];
    }
    return sum == BH ? num_groups : 0;
  }
  if (BH < 8) {
    const int n = std::min(BH, 4);
    for (int c = 0; c < n; ++c) sizes[c] = BH * (c + 1) / n - BH * c / n;
    return n;
  }
  sizes[0] = BH / 8;
  sizes[1] = sizes[2] = sizes[3] = BH / 4;
  sizes[4] = BH - sizes[0] - 3 * (BH / 4);
  return 5;
}

struct Layout {
  size_t tensor, lse, fwd_ws, bwd_ws, total;
};

Layout layout_of(int B, int H, int N, int d, int max_group, int compute_streams) {
  Layout L;
  const size_t BH = static_cast<size_t>(B) * H;
  L.tensor = round_up(BH * N * d * 2);
  L.lse = round_up(BH * N * 4);
  L.fwd_ws = round_up(fa2_fwd_workspace_bytes(1, max_group, N, d));
  L.bwd_ws = round_up(fa2_bwd_workspace_bytes(1, max_group, N, d));
  L.total = 8 * L.tensor + L.lse + static_cast<size_t>(compute_streams) * (L.fwd_ws + L.bwd_ws);
  return L;
}

// Side streams (upload, download, extra compute) and the events that link
// the stages, created once per device and CUDA context (again after a device
// reset, which changes the context id; kept when the id cannot be read).  The
// mutex serialises the enqueue of concurrent calls on one device, which share
// these.
struct DeviceState {
  std::mutex mu;
  bool ready = false;
  unsigned long long ctx_id = 0;
  cudaStream_t up = nullptr, down = nullptr;
  cudaStream_t comp[kMaxComputeStreams - 1] = {};
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t qkv_in[kMaxGroups] = {}, do_in[kMaxGroups] = {}, fwd_done[kMaxGroups] = {},
              bwd_done[kMaxGroups] = {};
};
DeviceState g_state[kMaxDevices];

int init_state(DeviceState& s) {
  const unsigned long long ctx = fa2::current_context_id();
  if (s.ready && (ctx == 0 || ctx == s.ctx_id)) return FA2_OK;
  // (handles of an earlier context are invalid now; they are dropped)
  s.ready = false;
  s.ctx_id = ctx;
  cudaError_t e = cudaStreamCreateWithFlags(&s.up, cudaStreamNonBlocking);
  if (!e) e = cudaStreamCreateWithFlags(&s.down, cudaStreamNonBlocking);
  for (int i = 0; !e && i < kMaxComputeStreams - 1; ++i) e = cudaStreamCreateWithFlags(&s.comp[i], cudaStreamNonBlocking);
  if (!e) e = cudaEventCreateWithFlags(&s.start, cudaEventDisableTiming);
  if (!e) e = cudaEventCreateWithFlags(&s.done, cudaEventDisableTiming);
  for (int c = 0; !e && c < kMaxGroups; ++c) {
    e = cudaEventCreateWithFlags(&s.qkv_in[c], cudaEventDisableTiming);
    if (!e) e = cudaEventCreateWithFlags(&s.do_in[c], cudaEventDisableTiming);
    if (!e) e = cudaEventCreateWithFlags(&s.fwd_done[c], cudaEventDisableTiming);
    if (!e) e = cudaEventCreateWithFlags(&s.bwd_done[c], cudaEventDisableTiming);
  }
  if (e) return fa2::record_cuda_failure(static_cast<int>(e), "host step: stream / event creation");
  s.ready = true;
  return FA2_OK;
}

}  // namespace

extern "C" {

size_t fa2_step_from_host_workspace_bytes(int B, int H, int N, int d, const int* group_heads, int num_groups,
                                          int compute_streams) {
  if (!valid_sizes(B, H, N, d) || compute_streams < 1 || compute_streams > kMaxComputeStreams) return 0;
  if (static_cast<long long>(B) * H > (1LL << 30)) return 0;
  int sizes[kMaxGroups];
  const int n = plan_groups(B * H, group_heads, num_groups, sizes);
  if (n == 0) return 0;
  const int max_group = *std::max_element(sizes, sizes + n);
  return layout_of(B, H, N, d, max_group, compute_streams).total;
}

int fa2_step_from_host(const void* q, const void* k, const void* v, const void* dO, void* o, float* lse, void* dq,
                       void* dk, void* dv, int B, int H, int N, int d, float scale, int causal,
                       const int* group_heads, int num_groups, int compute_streams, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !dO || !o || !lse || !dq || !dk || !dv) return FA2_ERR_NULL;
  if (d != 16 && d != 32 && d != 64 && d != 128) return FA2_ERR_HEADDIM;
  if (!valid_sizes(B, H, N, d)) return FA2_ERR_SHAPE;
  if (!(std::isfinite(scale) && scale > 0.f)) return FA2_ERR_SCALE;
  if (compute_streams < 1 || compute_streams > kMaxComputeStreams) return FA2_ERR_SHAPE;
  int sizes[kMaxGroups];
  const int n = plan_groups(B * H, group_heads, num_groups, sizes);
  if (n == 0) return FA2_ERR_SHAPE;
  const int max_group = *std::max_element(sizes, sizes + n);
  const Layout L = layout_of(B, H, N, d, max_group, compute_streams);
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % kAlign != 0 || workspace_bytes < L.total)
    return FA2_ERR_WORKSPACE;

  int dev = 0;
  if (cudaError_t e = cudaGetDevice(&dev)) return fa2::record_cuda_failure(static_cast<int>(e), "host step: device");
  if (dev < 0 || dev >= kMaxDevices) return FA2_ERR_SHAPE;
  DeviceState& S = g_state[dev];
  std::lock_guard<std::mutex> lock(S.mu);
  if (int rc = init_state(S)) return rc;

  // Device copies of the ten tensors, then per compute stream its forward and
  // backward scratch.
  char* base = static_cast<char*>(workspace);
  char* t_dev[8];  // q, k, v, dO, o, dq, dk, dv: L.tensor bytes each
  for (int i = 0; i < 8; ++i) t_dev[i] = base + static_cast<size_t>(i) * L.tensor;
  float* lse_dev = reinterpret_cast<float*>(base + 8 * L.tensor);
  char* scratch = base + 8 * L.tensor + L.lse;
  const void* t_host_in[4] = {q, k, v, dO};
  void* t_host_out[4] = {o, dq, dk, dv};

  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t comp[kMaxComputeStreams];
  comp[0] = st;
  for (int i = 1; i < compute_streams; ++i) comp[i] = S.comp[i - 1];
  const size_t row_bytes = static_cast<size_t>(N) * d * 2;  // one head of one bf16 tensor
  const size_t lse_row = static_cast<size_t>(N) * 4;

  cudaError_t e = cudaEventRecord(S.start, st);
  // The device buffers and host outputs are free once earlier work on
  // `stream` is done.
  if (!e) e = cudaStreamWaitEvent(S.up, S.start, 0);
  if (!e) e = cudaStreamWaitEvent(S.down, S.start, 0);
  for (int i = 1; !e && i < compute_streams; ++i) e = cudaStreamWaitEvent(comp[i], S.start, 0);
  if (e) return fa2::record_cuda_failure(static_cast<int>(e), "host step: stream join");

  // Uploads: a group's q, k, v (all its forward needs), then its dO.
  int first[kMaxGroups + 1];
  first[0] = 0;
  for (int c = 0; c < n; ++c) first[c + 1] = first[c] + sizes[c];
  for (int c = 0; c < n && !e; ++c) {
    const size_t off = static_cast<size_t>(first[c]) * row_bytes, bytes = static_cast<size_t>(sizes[c]) * row_bytes;
    for (int i = 0; i < 3 && !e; ++i)
      e = cudaMemcpyAsync(t_dev[i] + off, static_cast<const char*>(t_host_in[i]) + off, bytes, cudaMemcpyDefault, S.up);
    if (!e) e = cudaEventRecord(S.qkv_in[c], S.up);
    if (!e) e = cudaMemcpyAsync(t_dev[3] + off, static_cast<const char*>(t_host_in[3]) + off, bytes, cudaMemcpyDefault, S.up);
    if (!e) e = cudaEventRecord(S.do_in[c], S.up);
  }
  if (e) return fa2::record_cuda_failure(static_cast<int>(e), "host step: upload");

  // Kernels: group c on compute stream c % compute_streams, with that
  // stream's scratch (stream order keeps group c + compute_streams behind it).
  for (int c = 0; c < n; ++c) {
    const int s = c % compute_streams;
    const cudaStream_t cs = comp[s];
    void* fws = scratch + static_cast<size_t>(s) * (L.fwd_ws + L.bwd_ws);
    void* bws = static_cast<char*>(fws) + L.fwd_ws;
    const size_t off = static_cast<size_t>(first[c]) * row_bytes;
    float* lse_g = lse_dev + static_cast<size_t>(first[c]) * N;
    if ((e = cudaStreamWaitEvent(cs, S.qkv_in[c], 0))) break;
    int rc = fa2_fwd_ws(t_dev[0] + off, t_dev[1] + off, t_dev[2] + off, t_dev[4] + off, lse_g, 1, sizes[c], N, d,
                        scale, causal, fws, L.fwd_ws, cs);
    if (rc) return rc;
    if ((e = cudaEventRecord(S.fwd_done[c], cs))) break;
    if ((e = cudaStreamWaitEvent(cs, S.do_in[c], 0))) break;
    rc = fa2_bwd_ws(t_dev[0] + off, t_dev[1] + off, t_dev[2] + off, t_dev[4] + off, t_dev[3] + off, lse_g,
                    t_dev[5] + off, t_dev[6] + off, t_dev[7] + off, 1, sizes[c], N, d, scale, causal, bws, L.bwd_ws,
                    cs);
    if (rc) return rc;
    if ((e = cudaEventRecord(S.bwd_done[c], cs))) break;
  }
  if (e) return fa2::record_cuda_failure(static_cast<int>(e), "host step: kernels");

  // Downloads: a group's o and lse as soon as its forward is done, its
  // gradients after its backward.
  for (int c = 0; c < n && !e; ++c) {
    const size_t off = static_cast<size_t>(first[c]) * row_bytes, bytes = static_cast<size_t>(sizes[c]) * row_bytes;
    const size_t loff = static_cast<size_t>(first[c]) * lse_row, lbytes = static_cast<size_t>(sizes[c]) * lse_row;
    e = cudaStreamWaitEvent(S.down, S.fwd_done[c], 0);
    if (!e) e = cudaMemcpyAsync(static_cast<char*>(t_host_out[0]) + off, t_dev[4] + off, bytes, cudaMemcpyDefault, S.down);
    if (!e) e = cudaMemcpyAsync(reinterpret_cast<char*>(lse) + loff, reinterpret_cast<char*>(lse_dev) + loff, lbytes,
                                cudaMemcpyDefault, S.down);
    if (!e) e = cudaStreamWaitEvent(S.down, S.bwd_done[c], 0);
    for (int i = 1; i < 4 && !e; ++i)
      e = cudaMemcpyAsync(static_cast<char*>(t_host_out[i]) + off, t_dev[4 + i] + off, bytes, cudaMemcpyDefault,
                          S.down);
  }
  // `stream` waits for the last download (which waited for every group's
  // backward, and those for every upload).
  if (!e) e = cudaEventRecord(S.done, S.down);
  if (!e) e = cudaStreamWaitEvent(st, S.done, 0);
  if (e) return fa2::record_cuda_failure(static_cast<int>(e), "host step: download");
  return FA2_OK;
}

}  // extern "C"
