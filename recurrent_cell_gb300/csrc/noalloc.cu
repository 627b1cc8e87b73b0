// noalloc.cu -- forward + backward of the CfC K-loop without any allocation by
// the caller or by the library.
//
// Some callers cannot allocate device memory at the point where they run the
// K loop: code that runs under an allocator it does not own (a host
// framework whose device memory is all handed out up front), plugins that
// are not allowed to call cudaMalloc, or hard real-time loops where an
// allocation would stall.  cfc_kloop_forward/backward need a workspace the
// caller allocates; this entry point instead keeps that workspace in a
// file-scope device array of fixed size that is part of the library's module
// image.  The array exists once per device that loads the library and stays
// allocated until the process exits.
//
// The array's name in host code is only a host-side stand-in for the device
// symbol.  Its device address is looked up with cudaGetSymbolAddress once per
// device, on the first call made with that device current, and that address
// is what the kernels receive.  The address is kept for the life of the
// process, so a device reset (cudaDeviceReset) after the first call on that
// device is not supported.
//
// It always runs the CUDA-core (SIMT) kernels: the forward and backward K
// loops, the SIMT weight-gradient tiles and reduce_axis0.  Those need the
// smallest workspace (no tensor-core weight tiles), so the fixed array
// serves the widest range of sizes.  The regular entry points pick the
// cluster or tensor-core kernels instead, which sum in other orders, so the
// results of the two agree within the parity tolerances, not bit for bit.
#include <mutex>

#include "cfc_internal.cuh"

namespace cfc {
namespace {

static __device__ __align__(256) unsigned char g_static_workspace[CFC_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device (looked up once
// per device).  Returns nullptr on failure.
void* static_workspace_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return nullptr;
    g_static_ptr[dev] = p;
  }
  return g_static_ptr[dev];
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Workspace of the SIMT kernels in the fixed array: the W_cat^T copy, the
// saved activations, dA and the weight gradient's split partials, with the
// rows split by the FP32 rule (about four 64 x 64 output tiles per SM, at
// most 256 row blocks) in every precision mode.
bool static_layout(int B, int K, int n_in, int n_hid, int math, Layout* L) {
  if (!make_layout(B, K, n_in, n_hid, math, CFC_GRAD_GEMM, L)) return false;
  const long long tiles = (long long)((L->H3 + 63) / 64) * ((L->Zc + 1 + 63) / 64);
  long long split = (4ll * kNumSMs + tiles - 1) / tiles;
  split = std::max(1ll, std::min(split, std::min<long long>(L->R, 256)));
  L->rows_per_split = (L->R + split - 1) / split;
  L->n_split = (int)((L->R + L->rows_per_split - 1) / L->rows_per_split);
  size_t off = 0;
  L->off_wt = off;   off = align256(off + (size_t)L->Zc * L->H3 * L->elem);
  L->off_act = off;  off = align256(off + (size_t)L->R * L->H3 * sizeof(float));
  L->off_dA = off;   off = align256(off + (size_t)L->R * L->H3 * L->dA_elem);
  L->off_part = off; off = align256(off + (size_t)L->n_split * L->N * sizeof(float));
  L->off_wtt = off;
  L->total = off;
  return true;
}

}  // namespace
}  // namespace cfc

using namespace cfc;

extern "C" int cfc_kloop_forward_backward_static(
    const void* x, const void* h0, const void* W_in, const void* W_rec,
    const float* b, const float* dt, int dt_stride,
    int B, int K, int n_in, int n_hid, int math,
    const float* grad_h_seq, const float* grad_h_last, const float* y,
    void* h_seq, float* grad_W_in, float* grad_W_rec, float* grad_b,
    float* grad_h0, float* grad_x, void* stream) {
  if (math < CFC_MATH_FP32 || math > CFC_MATH_BF16) return CFC_ERR_MODE;
  Layout L;
  if (!static_layout(B, K, n_in, n_hid, math, &L)) return CFC_ERR_SHAPE;
  if (L.total > (size_t)CFC_STATIC_WORKSPACE_BYTES) return CFC_ERR_TOO_LARGE;
  if (!x || !h0 || !W_in || !W_rec || !b || !dt || !h_seq) return CFC_ERR_NULL;
  if (!grad_W_in || !grad_W_rec || !grad_b) return CFC_ERR_NULL;
  if (!grad_h_seq && !grad_h_last && !y) return CFC_ERR_NULL;
  if (dt_stride != 0 && dt_stride != 1) return CFC_ERR_SHAPE;
  const void* ptrs[] = {x, h0, W_in, W_rec, b, dt, grad_h_seq, grad_h_last, y, h_seq,
                        grad_W_in, grad_W_rec, grad_b, grad_h0, grad_x};
  for (const void* p : ptrs)
    if (p && !al16(p)) return CFC_ERR_ALIGN;
  void* ws = static_workspace_for_current_device();
  if (!ws) return CFC_ERR_DEVICE;

  CfcArgs a{};
  a.x = x; a.h0 = h0; a.W_in = W_in; a.W_rec = W_rec; a.b = b; a.dt = dt; a.dt_stride = dt_stride;
  a.h_seq = h_seq;
  a.grad_h_seq = grad_h_seq; a.grad_h_last = grad_h_last; a.y = y;
  a.grad_W_in = grad_W_in; a.grad_W_rec = grad_W_rec; a.grad_b = grad_b;
  a.grad_h0 = grad_h0; a.grad_x = grad_x; a.per_sample_scratch = nullptr;
  a.ws = static_cast<char*>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Every region of the array that a kernel reads (weight copy, activations,
  // dA, split partials) is fully written earlier in this same call, so no
  // clearing is needed between calls.
  if (launch_forward_simt(L, a, s) != cudaSuccess) return CFC_ERR_LAUNCH;
  if (launch_backward_simt(L, a, s) != cudaSuccess) return CFC_ERR_LAUNCH;
  float* part = reinterpret_cast<float*>(a.ws + L.off_part);
  if (launch_wgrad_simt(L, a, part, L.n_split, L.rows_per_split, s) != cudaSuccess)
    return CFC_ERR_LAUNCH;
  ReduceOut out{};
  out.nseg = 3;
  out.ptr[0] = grad_W_in;  out.begin[0] = 0;
  out.ptr[1] = grad_W_rec; out.begin[1] = (long long)L.H3 * n_in;
  out.ptr[2] = grad_b;     out.begin[2] = (long long)L.H3 * L.Zc;
  return launch_reduce(part, L.n_split, L.N, L.N, out, s) == cudaSuccess ? CFC_OK : CFC_ERR_LAUNCH;
}
