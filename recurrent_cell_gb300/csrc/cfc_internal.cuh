// cfc_internal.cuh -- internal declarations shared by the CUDA translation
// units of libcfc (not part of the public C ABI in include/cfc.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/cfc.h"

namespace cfc {

constexpr int kNumSMs = 152;  // GB300: 2 dies x 76 SMs

// ---------------------------------------------------------------------------
// Precision helpers.  The rounding points of each mode are part of the
// method's definition (see include/cfc.h); both the SIMT and the tensor-core
// kernels apply them at the same places.
// ---------------------------------------------------------------------------

// TF32 = binary32 with the low 13 significand bits cleared, rounded to nearest
// with ties away from zero (add half of the dropped range to the magnitude).
__device__ __forceinline__ float round_tf32(float v) {
  uint32_t u = __float_as_uint(v);
  u = (u + 0x1000u) & 0xFFFFE000u;
  return __uint_as_float(u);
}

__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// Value of a float as it enters a contraction in mode MODE.
template <int MODE>
__device__ __forceinline__ float to_operand(float v) {
  if constexpr (MODE == CFC_MATH_TF32) return round_tf32(v);
  else if constexpr (MODE == CFC_MATH_BF16) return round_bf16(v);
  else return v;
}

// Load an element of storage type T as float.
__device__ __forceinline__ float ldf(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// Load of a stored operand (x, h, W) already in the mode's operand form when
// stored as bf16; fp32 storage is rounded for TF32.
template <int MODE, typename T>
__device__ __forceinline__ float ld_operand(const T* p) {
  if constexpr (sizeof(T) == 2) return ldf(p);
  else return to_operand<MODE>(ldf(p));
}

__device__ __forceinline__ void stf(float* p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// The cell's three nonlinearities in the tensor-core modes, from
// tanh(a) = 1 - 2 / (1 + exp(2a)) and gate = 1 / (1 + exp(z)), z = A_f dt:
// with p1 = 1 + exp(2 A_g), p2 = 1 + exp(2 A_h~), p3 = 1 + exp(z) and one
// reciprocal r = 1 / (p1 p2 p3), 1/p1 = r p2 p3 and so on.  The exponent
// arguments are capped at 28 so the product stays finite (p^3 < e^85); at
// the cap tanh is 1 and the gate below 7e-13, both within an fp32 ulp of the
// uncapped values' contribution.  Absolute error: a few fp32 ulps of 1, far
// below the TF32 / bf16 rounding these modes apply.
struct CellAct {
  float gate, g, hh;
};
__device__ __forceinline__ CellAct cell_act(float a_f, float a_g, float a_h, float dt) {
  constexpr float kCap = 28.f;
  const float p1 = 1.f + __expf(fminf(2.f * a_g, kCap));
  const float p2 = 1.f + __expf(fminf(2.f * a_h, kCap));
  const float p3 = 1.f + __expf(fminf(a_f * dt, kCap));
  const float p12 = p1 * p2;
  const float r = __fdividef(1.f, p12 * p3);
  const float rp3 = r * p3;
  CellAct c;
  c.g = fmaf(-2.f, rp3 * p2, 1.f);
  c.hh = fmaf(-2.f, rp3 * p1, 1.f);
  c.gate = r * p12;
  return c;
}

// Distributed shared memory: 32-bit shared::cluster address of the variable at
// local shared address `local` in block `rank` of the cluster, and stores to it.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ void dsmem_st(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st(uint32_t addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void dsmem_st_bf16(uint32_t addr, float v) {
  const unsigned short b = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(addr), "h"(b) : "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Split cluster barrier: arrive with release semantics (orders this thread's
// earlier writes, e.g. distributed shared-memory stores, before the peers'
// acquire) and wait with acquire semantics.  Global stores issued between the
// two are not covered by the release, so the arrive does not wait for them.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Workspace layout (byte offsets, every region 256-byte aligned).
// ---------------------------------------------------------------------------
struct Layout {
  int B, K, n_in, H, Zc, H3, math, grad_path;
  size_t elem;          // bytes of a stored x/h/W element (4 or 2)
  size_t dA_elem;       // bytes of a stored dA element (4 or 2)
  long long N;          // packed per-sample gradient length
  long long R;          // B*K rows of the gradient contraction
  int n_split;          // row blocks of the GEMM-path contraction
  long long rows_per_split;
  size_t off_wt, off_act, off_dA, off_part, off_wtt, total;
};

bool make_layout(int B, int K, int n_in, int n_hid, int math, int grad_path, Layout* L);

// ---------------------------------------------------------------------------
// Optional kernel tracing (see cfc_trace_enable in include/cfc.h).
// ---------------------------------------------------------------------------
void trace_begin(const char* name, cudaStream_t s);
void trace_end(cudaStream_t s);

struct TraceScope {
  cudaStream_t s;
  TraceScope(const char* name, cudaStream_t st) : s(st) { trace_begin(name, s); }
  ~TraceScope() { trace_end(s); }
};

// ---------------------------------------------------------------------------
// Launchers (return cudaError_t of the launch).
// ---------------------------------------------------------------------------
struct ReduceOut {
  float* ptr[4];
  long long begin[4];
  int nseg;
};

cudaError_t launch_reduce(const float* in, int n_batch, long long n_tail, long long ld,
                          const ReduceOut& out, cudaStream_t stream);
// One bounded wait that runs out (max_polls polls) and sets the device error
// word (cfc_tc.cu); diagnostic for the timeout path.
cudaError_t launch_selftest_wait_timeout(uint32_t max_polls, cudaStream_t s);

// tau-cell K loop (cfc_tau.cu), FP32.
bool tau_shape_supported(int n_in, int n_hid);
cudaError_t launch_tau_forward(const float* x, const float* h0, const float* W_in, const float* W_rec,
                               const float* b, const float* tau, const float* dt, int dt_stride, int B, int K,
                               int n_in, int H, float* h_seq, float* s_ws, cudaStream_t s);
cudaError_t launch_tau_backward(const float* x, const float* h0, const float* W_in, const float* W_rec,
                                const float* tau, const float* dt, int dt_stride, int B, int K, int n_in, int H,
                                const float* h_seq, const float* s_ws, const float* grad_h_seq,
                                const float* grad_h_last, const float* y, float* per_sample, float* grad_h0,
                                float* grad_x, float* grad_W_in, float* grad_W_rec, float* grad_b,
                                float* grad_tau, cudaStream_t s);

// count matrices (host arrays of device pointers and sizes, already checked),
// one launch per kernel configuration and up to 32 matrices.
cudaError_t launch_reduce_multi(const float* const* in, const int* n_batch, const long long* n_tail,
                                float* const* out, int count, cudaStream_t stream);

struct CfcArgs {
  const void* x; const void* h0; const void* W_in; const void* W_rec;
  const float* b; const float* dt; int dt_stride;
  void* h_seq;
  const float* grad_h_seq; const float* grad_h_last; const float* y;
  float* grad_W_in; float* grad_W_rec; float* grad_b; float* grad_h0; float* grad_x;
  float* per_sample_scratch;
  char* ws;
};

cudaError_t launch_forward_simt(const Layout& L, const CfcArgs& a, cudaStream_t s);
// K-loop kernel family: CFC_KLOOP_KERNELS=tc | cluster | simt forces one
// family where it supports the sizes (read on every call); anything else
// selects automatically.
enum KernelChoice { kAuto = 0, kCluster = 1, kSimt = 2, kTc = 3, kTcStream = 4, kSolo = 5 };
int kernel_choice();

// Tensor-core forward (TF32 / bf16 modes); cudaErrorNotSupported, launching
// nothing, when the sizes do not fit its plan or another family is forced.
cudaError_t launch_forward_tc(const Layout& L, const CfcArgs& a, cudaStream_t s);
int read_tc_kloop_error(int clear);
// grad_x = dA W_in on CUDA cores after the cluster K loop (any mode).
cudaError_t launch_grad_x_simt(const Layout& L, const CfcArgs& a, cudaStream_t s);
// grad_x = dA W_in for the tensor-core K-loop kernels (which carry only
// W_rec^T dA): one TMA-fed tcgen05 GEMM over the B*K rows after the loop.
bool grad_x_gemm_applies(const Layout& L);
cudaError_t launch_grad_x_tc(const Layout& L, const CfcArgs& a, cudaStream_t s);
// Tensor-core backward, cluster split by units (TF32 / bf16 modes).
cudaError_t launch_backward_cluster_tc(const Layout& L, const CfcArgs& a, cudaStream_t s);
// W_rec^T as pre-swizzled shared-memory tiles (tile of K atom a, M tile m at
// ((a / 2) * nM + m) * 32 KB + (a % 2) * 16 KB; for nM = 1 the atoms follow
// one another), rounded to the operand: the backward kernels copy them.
cudaError_t launch_prep_wt_tiles(const Layout& L, int nM, int nAk, uint8_t* tiles, const void* W_rec, cudaStream_t s);

// Tensor-core forward and backward in one block per sample tile (TF32 / bf16,
// n_hid <= 128); the forward first runs the input projection over all rows.
cudaError_t launch_forward_solo_tc(const Layout& L, const CfcArgs& a, cudaStream_t s);
cudaError_t launch_backward_solo_tc(const Layout& L, const CfcArgs& a, cudaStream_t s);
int read_tc_solo_error(int clear);
// Tensor-core forward with streamed W_cat tiles (TF32 / bf16 modes).
cudaError_t launch_forward_tc_stream(const Layout& L, const CfcArgs& a, cudaStream_t s);
// Tensor-core backward (TF32 / bf16 modes), streamed W_cat^T tiles.
cudaError_t launch_backward_tc(const Layout& L, const CfcArgs& a, cudaStream_t s);
size_t tc_bwd_tiles_bytes(int n_in, int n_hid, int math);
int read_tc_bwd_error(int clear);

// Cluster kernels (weights resident in shared memory of a block cluster).
// Return cudaErrorNotSupported, launching nothing, when no cluster plan fits
// the sizes or (for kernel selection "auto") the plan would need more than
// about two waves of blocks.
cudaError_t launch_forward_cluster(const Layout& L, const CfcArgs& a, cudaStream_t s);
cudaError_t launch_backward_cluster(const Layout& L, const CfcArgs& a, cudaStream_t s);
cudaError_t launch_backward_simt(const Layout& L, const CfcArgs& a, cudaStream_t s);
// Tensor-core (tcgen05) gradient contraction of the TF32 / bf16 modes.
// Splits of the TMA-fed contraction (bf16, GEMM path) for these sizes, or 0
// when it does not apply (then the register-staged contraction is used).
int tma_wgrad_splits(int B, int K, int n_in, int n_hid, int math, int grad_path);
cudaError_t launch_wgrad_tc(const Layout& L, const CfcArgs& a, float* out, cudaStream_t s);
int tc_wgrad_blocks(int n_in, int n_hid);
// Reads (and optionally clears) the device-side error word of the
// tensor-core kernels; blocks until the device is idle.
int read_device_error(int clear);

cudaError_t launch_wgrad_simt(const Layout& L, const CfcArgs& a, float* out, int n_split,
                              long long rows_per_split, cudaStream_t s);

}  // namespace cfc
