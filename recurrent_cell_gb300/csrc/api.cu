// api.cu -- the extern "C" entry points declared in include/cfc.h.
//
// Every entry point validates its arguments on the host before enqueuing
// anything, then enqueues kernels on the caller's stream.  No allocation, no
// synchronisation, no host read of device data.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "cfc_internal.cuh"

namespace cfc {

// Tracing state: records of (kernel name, start event, stop event).  Events
// come from a pool that only grows, so re-enabling does not re-create them.
namespace {
struct TraceRec { const char* name; cudaEvent_t start, stop; };
bool g_trace_on = false;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_pool;
size_t g_pool_next = 0;

cudaEvent_t pool_event() {
  if (g_pool_next == g_pool.size()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_pool.push_back(e);
  }
  return g_pool[g_pool_next++];
}
}  // namespace

void trace_begin(const char* name, cudaStream_t s) {
  if (!g_trace_on) return;
  TraceRec r{name, pool_event(), pool_event()};
  if (!r.start || !r.stop) return;
  cudaEventRecord(r.start, s);
  g_trace.push_back(r);
}

void trace_end(cudaStream_t s) {
  if (!g_trace_on || g_trace.empty()) return;
  cudaEventRecord(g_trace.back().stop, s);
}

int kernel_choice() {
  const char* v = getenv("CFC_KLOOP_KERNELS");
  if (!v) return kAuto;
  if (strcmp(v, "cluster") == 0) return kCluster;
  if (strcmp(v, "simt") == 0) return kSimt;
  if (strcmp(v, "tc") == 0) return kTc;
  if (strcmp(v, "tcs") == 0) return kTcStream;
  if (strcmp(v, "solo") == 0) return kSolo;
  return kAuto;
}

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

bool make_layout(int B, int K, int n_in, int n_hid, int math, int grad_path, Layout* L) {
  if (B < 1 || K < 1 || n_in < 1 || n_hid < 1) return false;
  if (n_hid > 1024 || n_in + n_hid > 1024) return false;
  if (math < CFC_MATH_FP32 || math > CFC_MATH_BF16) return false;
  if (grad_path != CFC_GRAD_SCRATCH && grad_path != CFC_GRAD_GEMM) return false;
  if ((long long)B * K > (1ll << 31)) return false;
  L->B = B; L->K = K; L->n_in = n_in; L->H = n_hid;
  L->Zc = n_in + n_hid; L->H3 = 3 * n_hid;
  L->math = math; L->grad_path = grad_path;
  L->elem = (math == CFC_MATH_BF16) ? 2 : 4;
  L->dA_elem = L->elem;
  L->N = 3ll * (n_in + n_hid + 1) * n_hid;
  L->R = (long long)B * K;
  if (grad_path == CFC_GRAD_SCRATCH) {
    L->n_split = B;
    L->rows_per_split = K;
  } else if (math == CFC_MATH_FP32) {
    // Fixed split of the B*K rows into row blocks: about four blocks of the
    // 64 x 64 SIMT output tiling per SM (the 3xTF32 contraction serves the
    // per-sample path, whose split is the batch).  Depends on the sizes only,
    // so results are reproducible for a given configuration.
    const long long tiles = (long long)((L->H3 + 63) / 64) * ((L->Zc + 1 + 63) / 64);
    long long split = (4ll * kNumSMs + tiles - 1) / tiles;
    split = std::max(1ll, std::min(split, std::min<long long>(L->R, 256)));
    L->rows_per_split = (L->R + split - 1) / split;
    L->n_split = (int)((L->R + L->rows_per_split - 1) / L->rows_per_split);
  } else if (const int tma_splits = tma_wgrad_splits(B, K, n_in, n_hid, math, grad_path)) {
    // TMA-fed tensor-core contraction (bf16, TF32): one block per SM,
    // (3H / 128) x splits.
    L->n_split = tma_splits;
    L->rows_per_split = (L->R + tma_splits - 1) / tma_splits;
  } else {
    // Tensor-core contraction: about two blocks per SM over its 128-row x
    // N-block tiling; row blocks are whole multiples of 64 rows (one bf16
    // chunk, two TF32 chunks).
    const long long tiles = tc_wgrad_blocks(n_in, n_hid);
    long long split = std::max(1ll, (2ll * kNumSMs) / tiles);   // one wave at 2 blocks per SM
    split = std::min(split, std::max(1ll, L->R / 64));
    long long rps = (L->R + split - 1) / split;
    rps = (rps + 63) / 64 * 64;
    L->rows_per_split = rps;
    L->n_split = (int)((L->R + rps - 1) / rps);
  }
  size_t off = 0;
  L->off_wt = off;   off = align256(off + (size_t)L->Zc * L->H3 * L->elem);
  L->off_act = off;  off = align256(off + (size_t)L->R * L->H3 * sizeof(float));
  L->off_dA = off;   off = align256(off + (size_t)L->R * L->H3 * L->dA_elem);
  L->off_part = off;
  if (grad_path == CFC_GRAD_GEMM) off = align256(off + (size_t)L->n_split * L->N * sizeof(float));
  L->off_wtt = off;  // pre-swizzled W_cat^T tiles of the tensor-core backward
  off = align256(off + tc_bwd_tiles_bytes(n_in, n_hid, math));
  L->total = off;
  return true;
}

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace cfc

using namespace cfc;

extern "C" {

const char* cfc_status_string(int status) {
  switch (status) {
    case CFC_OK: return "ok";
    case CFC_ERR_NULL: return "a required pointer is NULL";
    case CFC_ERR_SHAPE: return "invalid size (negative, zero where not allowed, or too large)";
    case CFC_ERR_ALIGN: return "pointer not 16-byte aligned";
    case CFC_ERR_WORKSPACE: return "workspace NULL or smaller than cfc_kloop_workspace_bytes()";
    case CFC_ERR_MODE: return "unknown math mode or gradient path";
    case CFC_ERR_LAUNCH: return "kernel launch failed";
    case CFC_ERR_DEVICE: return "no usable CUDA device";
    case CFC_ERR_TOO_LARGE: return "sizes need more workspace than CFC_STATIC_WORKSPACE_BYTES";
    default: return "unknown status";
  }
}

long long cfc_per_sample_length(int n_in, int n_hid) {
  if (n_in < 1 || n_hid < 1) return 0;
  return 3ll * (n_in + n_hid + 1) * n_hid;
}

int cfc_kloop_grad_splits(int B, int K, int n_in, int n_hid, int math, int grad_path) {
  Layout L;
  if (!make_layout(B, K, n_in, n_hid, math, grad_path, &L)) return 0;
  return L.n_split;
}

int cfc_device_error(int clear) {
  const int a = read_device_error(clear);
  const int b = read_tc_kloop_error(clear);
  const int c = read_tc_bwd_error(clear);
  const int d = read_tc_solo_error(clear);
  if (a < 0 || b < 0 || c < 0 || d < 0) return CFC_ERR_DEVICE;
  return (a || b || c || d) ? 1 : 0;
}

int cfc_selftest_timeout(int max_polls, void* stream) {
  if (max_polls < 1 || max_polls > (1 << 20)) return CFC_ERR_SHAPE;
  cudaError_t e = launch_selftest_wait_timeout((uint32_t)max_polls, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CFC_OK : CFC_ERR_LAUNCH;
}

size_t cfc_kloop_workspace_bytes(int B, int K, int n_in, int n_hid, int math, int grad_path) {
  Layout L;
  if (!make_layout(B, K, n_in, n_hid, math, grad_path, &L)) return 0;
  return L.total;
}

static int check_common(int B, int K, int n_in, int n_hid, int math, int grad_path, Layout* L) {
  if (math < CFC_MATH_FP32 || math > CFC_MATH_BF16) return CFC_ERR_MODE;
  if (grad_path != CFC_GRAD_SCRATCH && grad_path != CFC_GRAD_GEMM) return CFC_ERR_MODE;
  if (!make_layout(B, K, n_in, n_hid, math, grad_path, L)) return CFC_ERR_SHAPE;
  return CFC_OK;
}

int cfc_kloop_forward(const void* x, const void* h0, const void* W_in, const void* W_rec,
                      const float* b, const float* dt, int dt_stride,
                      int B, int K, int n_in, int n_hid, int math,
                      void* h_seq, void* workspace, size_t workspace_bytes, void* stream) {
  Layout L;
  int st = check_common(B, K, n_in, n_hid, math, CFC_GRAD_SCRATCH, &L);
  if (st != CFC_OK) return st;
  if (!x || !h0 || !W_in || !W_rec || !b || !dt || !h_seq) return CFC_ERR_NULL;
  if (dt_stride != 0 && dt_stride != 1) return CFC_ERR_SHAPE;
  if (!workspace || workspace_bytes < L.total) return CFC_ERR_WORKSPACE;
  const void* ptrs[] = {x, h0, W_in, W_rec, b, dt, h_seq, workspace};
  for (const void* p : ptrs)
    if (!al16(p)) return CFC_ERR_ALIGN;
  CfcArgs a{};
  a.x = x; a.h0 = h0; a.W_in = W_in; a.W_rec = W_rec; a.b = b; a.dt = dt; a.dt_stride = dt_stride;
  a.h_seq = h_seq; a.ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Input projection + single-block tensor-core kernel (n_hid <= 128, W_rec
  // resident in one block) while its grid fits one wave, else the tensor-core
  // cluster kernel (weights resident) while its grid fits one wave, else the
  // tensor-core kernel with streamed weights, else the SIMT cluster kernel
  // (FP32), else the plain SIMT kernel.
  cudaError_t e = launch_forward_solo_tc(L, a, s);
  if (e == cudaErrorNotSupported) e = launch_forward_tc(L, a, s);
  if (e == cudaErrorNotSupported) e = launch_forward_tc_stream(L, a, s);
  if (e == cudaErrorNotSupported) e = launch_forward_cluster(L, a, s);
  if (e == cudaErrorNotSupported) e = launch_forward_simt(L, a, s);
  return e == cudaSuccess ? CFC_OK : CFC_ERR_LAUNCH;
}

int cfc_kloop_backward(const void* x, const void* h0, const void* W_in, const void* W_rec,
                       const float* b, const float* dt, int dt_stride,
                       int B, int K, int n_in, int n_hid, int math,
                       const void* h_seq, const float* grad_h_seq, const float* grad_h_last,
                       const float* y,
                       float* grad_W_in, float* grad_W_rec, float* grad_b,
                       float* grad_h0, float* grad_x,
                       float* per_sample_scratch, int grad_path,
                       void* workspace, size_t workspace_bytes, void* stream) {
  Layout L;
  int st = check_common(B, K, n_in, n_hid, math, grad_path, &L);
  if (st != CFC_OK) return st;
  if (!x || !h0 || !W_in || !W_rec || !b || !dt || !h_seq) return CFC_ERR_NULL;
  if (!grad_W_in || !grad_W_rec || !grad_b) return CFC_ERR_NULL;
  if (!grad_h_seq && !grad_h_last && !y) return CFC_ERR_NULL;
  if (grad_path == CFC_GRAD_SCRATCH && !per_sample_scratch) return CFC_ERR_NULL;
  if (dt_stride != 0 && dt_stride != 1) return CFC_ERR_SHAPE;
  if (!workspace || workspace_bytes < L.total) return CFC_ERR_WORKSPACE;
  const void* ptrs[] = {x, h0, W_in, W_rec, b, dt, h_seq, grad_h_seq, grad_h_last, y,
                        grad_W_in, grad_W_rec, grad_b, grad_h0, grad_x,
                        grad_path == CFC_GRAD_SCRATCH ? per_sample_scratch : nullptr, workspace};
  for (const void* p : ptrs)
    if (p && !al16(p)) return CFC_ERR_ALIGN;
  CfcArgs a{};
  a.x = x; a.h0 = h0; a.W_in = W_in; a.W_rec = W_rec; a.b = b; a.dt = dt; a.dt_stride = dt_stride;
  a.h_seq = const_cast<void*>(h_seq);
  a.grad_h_seq = grad_h_seq; a.grad_h_last = grad_h_last; a.y = y;
  a.grad_W_in = grad_W_in; a.grad_W_rec = grad_W_rec; a.grad_b = grad_b;
  a.grad_h0 = grad_h0; a.grad_x = grad_x; a.per_sample_scratch = per_sample_scratch;
  a.ws = static_cast<char*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // TF32 / bf16: the single-block tensor-core kernel (n_hid <= 128, W_rec^T
  // resident in one block) while its grid fits one wave; then the tensor-core
  // cluster kernel while its grid fits one wave; then the CUDA-core cluster
  // kernel while its grid stays within ~2 waves (many steps, fewer samples),
  // else the tensor-core kernel with streamed weights, else SIMT.
  cudaError_t e = launch_backward_solo_tc(L, a, s);
  if (e == cudaErrorNotSupported) e = launch_backward_cluster_tc(L, a, s);
  if (e == cudaErrorNotSupported) e = launch_backward_cluster(L, a, s);
  if (e == cudaErrorNotSupported) e = launch_backward_tc(L, a, s);
  if (e == cudaErrorNotSupported) e = launch_backward_simt(L, a, s);
  if (e != cudaSuccess) return CFC_ERR_LAUNCH;
  float* part = (grad_path == CFC_GRAD_SCRATCH) ? per_sample_scratch
                                                : reinterpret_cast<float*>(a.ws + L.off_part);
  // FP32: the tensor-core contraction with 3xTF32 operands where it applies,
  // else the SIMT tiles.
  e = launch_wgrad_tc(L, a, part, s);
  if (e == cudaErrorNotSupported && math == CFC_MATH_FP32)
    e = launch_wgrad_simt(L, a, part, L.n_split, L.rows_per_split, s);
  if (e != cudaSuccess) return CFC_ERR_LAUNCH;
  ReduceOut out{};
  out.nseg = 3;
  out.ptr[0] = grad_W_in;  out.begin[0] = 0;
  out.ptr[1] = grad_W_rec; out.begin[1] = (long long)L.H3 * n_in;
  out.ptr[2] = grad_b;     out.begin[2] = (long long)L.H3 * L.Zc;
  e = launch_reduce(part, L.n_split, L.N, L.N, out, s);
  return e == cudaSuccess ? CFC_OK : CFC_ERR_LAUNCH;
}

int cfc_trace_enable(int on) {
  g_trace.clear();
  g_pool_next = 0;
  g_trace_on = (on != 0);
  return CFC_OK;
}

int cfc_trace_count(void) { return (int)g_trace.size(); }

int cfc_trace_get(int i, const char** name, float* ms) {
  if (i < 0 || i >= (int)g_trace.size()) return CFC_ERR_SHAPE;
  if (name) *name = g_trace[i].name;
  if (ms) {
    *ms = 0.f;
    if (cudaEventSynchronize(g_trace[i].stop) != cudaSuccess) return CFC_ERR_LAUNCH;
    if (cudaEventElapsedTime(ms, g_trace[i].start, g_trace[i].stop) != cudaSuccess) return CFC_ERR_LAUNCH;
  }
  return CFC_OK;
}

int reduce_axis0(const float* per_batch, int n_batch, long long n_tail, float* out, void* stream) {
  if (n_batch < 0 || n_tail < 0 || n_tail > (1ll << 35)) return CFC_ERR_SHAPE;
  if (n_tail == 0) return CFC_OK;
  if (!out || (n_batch > 0 && !per_batch)) return CFC_ERR_NULL;
  if (!al4(out) || (per_batch && !al4(per_batch))) return CFC_ERR_ALIGN;
  ReduceOut o{};
  o.nseg = 1;
  o.ptr[0] = out;
  o.begin[0] = 0;
  cudaError_t e = launch_reduce(per_batch, n_batch, n_tail, n_tail, o, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CFC_OK : CFC_ERR_LAUNCH;
}

long long cfc_tau_per_sample_length(int n_in, int n_hid) {
  if (!tau_shape_supported(n_in, n_hid)) return 0;
  return (long long)(n_in + n_hid + 2) * n_hid;
}

size_t cfc_tau_kloop_workspace_bytes(int B, int K, int n_in, int n_hid) {
  if (B < 1 || K < 1 || !tau_shape_supported(n_in, n_hid)) return 0;
  return align256((size_t)B * K * n_hid * sizeof(float));
}

static int tau_check(const void* const* ptrs, int n, int B, int K, int n_in, int n_hid, int dt_stride,
                     const void* workspace, size_t workspace_bytes) {
  if (B < 1 || K < 1 || !tau_shape_supported(n_in, n_hid)) return CFC_ERR_SHAPE;
  if ((long long)B * K * (n_in > n_hid ? n_in : n_hid) > (1ll << 40)) return CFC_ERR_SHAPE;
  if (dt_stride != 0 && dt_stride != 1) return CFC_ERR_SHAPE;
  for (int i = 0; i < n; ++i)
    if (!ptrs[i]) return CFC_ERR_NULL;
  for (int i = 0; i < n; ++i)
    if (!al16(ptrs[i])) return CFC_ERR_ALIGN;
  if (!workspace || workspace_bytes < cfc_tau_kloop_workspace_bytes(B, K, n_in, n_hid)) return CFC_ERR_WORKSPACE;
  if (!al16(workspace)) return CFC_ERR_ALIGN;
  return CFC_OK;
}

int cfc_tau_kloop_forward(const float* x, const float* h0, const float* W_in, const float* W_rec, const float* b,
                          const float* tau, const float* dt, int dt_stride, int B, int K, int n_in, int n_hid,
                          float* h_seq, void* workspace, size_t workspace_bytes, void* stream) {
  const void* ptrs[] = {x, h0, W_in, W_rec, b, tau, dt, h_seq};
  const int st = tau_check(ptrs, 8, B, K, n_in, n_hid, dt_stride, workspace, workspace_bytes);
  if (st != CFC_OK) return st;
  cudaError_t e = launch_tau_forward(x, h0, W_in, W_rec, b, tau, dt, dt_stride, B, K, n_in, n_hid, h_seq,
                                     static_cast<float*>(workspace), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CFC_OK : CFC_ERR_LAUNCH;
}

int cfc_tau_kloop_backward(const float* x, const float* h0, const float* W_in, const float* W_rec,
                           const float* b, const float* tau, const float* dt, int dt_stride, int B, int K,
                           int n_in, int n_hid, const float* h_seq, const float* grad_h_seq,
                           const float* grad_h_last, const float* y, float* grad_W_in, float* grad_W_rec,
                           float* grad_b, float* grad_tau, float* grad_h0, float* grad_x,
                           float* per_sample_scratch, void* workspace, size_t workspace_bytes, void* stream) {
  const void* ptrs[] = {x, h0, W_in, W_rec, b, tau, dt, h_seq, grad_W_in, grad_W_rec, grad_b, grad_tau,
                        per_sample_scratch};
  const int st = tau_check(ptrs, 13, B, K, n_in, n_hid, dt_stride, workspace, workspace_bytes);
  if (st != CFC_OK) return st;
  if (!grad_h_seq && !grad_h_last && !y) return CFC_ERR_NULL;
  const void* opt[] = {grad_h_seq, grad_h_last, y, grad_h0, grad_x};
  for (const void* p : opt)
    if (p && !al16(p)) return CFC_ERR_ALIGN;
  cudaError_t e = launch_tau_backward(x, h0, W_in, W_rec, tau, dt, dt_stride, B, K, n_in, n_hid, h_seq,
                                      static_cast<const float*>(workspace), grad_h_seq, grad_h_last, y,
                                      per_sample_scratch, grad_h0, grad_x, grad_W_in, grad_W_rec, grad_b,
                                      grad_tau, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CFC_OK : CFC_ERR_LAUNCH;
}

int reduce_axis0_multi(const float* const* per_batch, const int* n_batch, const long long* n_tail,
                       float* const* out, int count, void* stream) {
  if (count < 0 || count > 4096) return CFC_ERR_SHAPE;
  if (count == 0) return CFC_OK;
  if (!per_batch || !n_batch || !n_tail || !out) return CFC_ERR_NULL;
  for (int i = 0; i < count; ++i) {
    if (n_batch[i] < 0 || n_tail[i] < 0 || n_tail[i] > (1ll << 35)) return CFC_ERR_SHAPE;
    if (n_tail[i] == 0) continue;
    if (!out[i] || (n_batch[i] > 0 && !per_batch[i])) return CFC_ERR_NULL;
    if (!al4(out[i]) || (per_batch[i] && !al4(per_batch[i]))) return CFC_ERR_ALIGN;
  }
  cudaError_t e = launch_reduce_multi(per_batch, n_batch, n_tail, out, count, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CFC_OK : CFC_ERR_LAUNCH;
}

}  // extern "C"
