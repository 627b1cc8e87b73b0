// cfc_tau.cu -- K loop of the pages' single-head tau-cell, forward and
// backward through time, FP32 ("K-loop Parallelization Implementation Plan",
// Task 2: cfc_step_batched, Task 3: cfc_step_backward_batched):
//
//   pre = b + W_in x_k + W_rec h_k,  s = tanh(pre),
//   decay = exp(-dt / max(tau, 1e-6)),  h_{k+1} = h_k decay + (1 - decay) s.
//
// One block per sample keeps W_cat = [W_in | W_rec] resident in shared memory
// for the whole K loop (rows padded to an odd number of floats: 32 threads
// reading 32 rows, or 32 columns, touch 32 distinct banks); Q threads share
// each hidden unit's dot products.  The forward saves s for the backward.  The backward keeps
// the sample's parameter gradient [W_in | W_rec] in shared memory (same padded
// layout), accumulates it over the K steps in registers / shared memory and
// writes the packed per-sample row [gW_in | gW_rec | gb | gtau] once; the
// rows are then summed by reduce_axis0 (canonical order) into the four
// outputs.  The pages accumulate into global scratch with += at every step;
// here every gradient element is written once per call.
#include "cfc_internal.cuh"

namespace cfc {
namespace {

constexpr float kTauEps = 1e-6f;
constexpr size_t kTauSmemMax = 227 * 1024;

// Q threads per hidden unit (thread t: part p = t / Hr, unit u = t % Hr with
// Hr = H rounded up to 32, so a warp holds 32 units of one part and its
// shared-memory rows / columns fall on 32 distinct banks).  Part p of a dot
// product covers a contiguous Zc / Q (or H / Q) range; the Q partial sums
// meet in shared memory and unit u's part-0 thread adds them in the fixed
// order ((q0 + q1) + (q2 + q3)).
__host__ __device__ inline int tau_round32(int v) { return (v + 31) / 32 * 32; }
__host__ __device__ inline int tau_parts(int H) {
  const int hr = tau_round32(H);
  return hr <= 256 ? 4 : (hr <= 512 ? 2 : 1);
}
__host__ __device__ inline int tau_threads(int H) { return tau_parts(H) * tau_round32(H); }

__device__ __forceinline__ float sum_parts(const float* part, int Q, int H, int u) {
  if (Q == 4) return (part[u] + part[H + u]) + (part[2 * H + u] + part[3 * H + u]);
  if (Q == 2) return part[u] + part[H + u];
  return part[u];
}

__global__ void __launch_bounds__(1024) k_tau_fwd(const float* __restrict__ x, const float* __restrict__ h0,
                          const float* __restrict__ W_in, const float* __restrict__ W_rec,
                          const float* __restrict__ bias, const float* __restrict__ tau,
                          const float* __restrict__ dt, int dt_stride, int K, int n_in, int H,
                          float* __restrict__ h_seq, float* __restrict__ s_out) {
  extern __shared__ float sm[];
  const int Zc = n_in + H, ld = Zc | 1;
  const int Q = tau_parts(H), Hr = tau_round32(H);
  float* W = sm;                       // [H][ld]
  float* z = W + (size_t)H * ld;       // [Zc]: x_k, then h_k
  float* part = z + Zc;                // [Q][H] partial dot products
  const long long bi = blockIdx.x;
  const int tid = threadIdx.x, T = blockDim.x;
  const int p = tid / Hr, u = tid - p * Hr;
  const int j0 = (int)((long long)p * Zc / Q), j1 = (int)((long long)(p + 1) * Zc / Q);
  for (int e = tid; e < H * Zc; e += T) {
    const int uu = e / Zc, j = e - uu * Zc;
    W[uu * ld + j] = (j < n_in) ? W_in[(long long)uu * n_in + j] : W_rec[(long long)uu * H + (j - n_in)];
  }
  for (int uu = tid; uu < H; uu += T) z[n_in + uu] = h0[bi * H + uu];
  const float dtb = dt[dt_stride ? bi : 0];
  float bu = 0.f, du = 0.f;
  if (tid < H) {
    bu = bias[tid];
    du = expf(-dtb / fmaxf(tau[tid], kTauEps));
  }
  // x of the next step is loaded one step ahead (n_in <= 1024 <= 8 T)
  constexpr int kXR = 8;
  float xr[kXR];
  auto load_x = [&](int kk) {
#pragma unroll
    for (int q = 0; q < kXR; ++q) {
      const int j = tid + q * T;
      xr[q] = (kk < K && j < n_in) ? x[(bi * K + kk) * n_in + j] : 0.f;
    }
  };
  load_x(0);
  for (int k = 0; k < K; ++k) {
    const long long row = bi * K + k;
#pragma unroll
    for (int q = 0; q < kXR; ++q)
      if (tid + q * T < n_in) z[tid + q * T] = xr[q];
    load_x(k + 1);
    __syncthreads();
    if (u < H) {
      const float* __restrict__ w = W + u * ld;
      const float* __restrict__ zz = z;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
      int j = j0;
      for (; j + 3 < j1; j += 4) {
        a0 = fmaf(w[j], zz[j], a0);
        a1 = fmaf(w[j + 1], zz[j + 1], a1);
        a2 = fmaf(w[j + 2], zz[j + 2], a2);
        a3 = fmaf(w[j + 3], zz[j + 3], a3);
      }
      for (; j < j1; ++j) a0 = fmaf(w[j], zz[j], a0);
      part[p * H + u] = (a0 + a1) + (a2 + a3);
    }
    __syncthreads();
    if (tid < H) {
      const float s = tanhf(bu + sum_parts(part, Q, H, tid));
      const float hn = z[n_in + tid] * du + (1.f - du) * s;
      h_seq[row * H + tid] = hn;
      s_out[row * H + tid] = s;
      z[n_in + tid] = hn;      // every read of z of this step is behind the barrier above
    }
  }
}

// REG: each thread keeps its kGReg-or-fewer gradient entries of row u in
// registers (no shared-memory G); used when they fit.
constexpr int kGReg = 64;

template <bool REG>
__global__ void __launch_bounds__(REG ? 512 : 1024) k_tau_bwd(const float* __restrict__ x, const float* __restrict__ h0,
                          const float* __restrict__ W_in, const float* __restrict__ W_rec,
                          const float* __restrict__ tau, const float* __restrict__ dt, int dt_stride, int K,
                          int n_in, int H, const float* __restrict__ h_seq, const float* __restrict__ s_in,
                          const float* __restrict__ grad_h_seq, const float* __restrict__ grad_h_last,
                          const float* __restrict__ y, float* __restrict__ per_sample,
                          float* __restrict__ grad_h0, float* __restrict__ grad_x) {
  extern __shared__ float sm[];
  const int Zc = n_in + H, ld = Zc | 1;
  const int Q = tau_parts(H), Hr = tau_round32(H);
  float* W = sm;                      // [H][ld]
  float* G = W + (size_t)H * ld;      // [H][ld]: gradient of [W_in | W_rec] (not REG)
  float* z = G + (REG ? 0 : (size_t)H * ld);   // [Zc]: x_k, then h_k
  float* dpre = z + Zc;               // [H]
  float* part = dpre + H;             // [Q][H] partial carries
  const long long bi = blockIdx.x;
  const int tid = threadIdx.x, T = blockDim.x;
  const int p = tid / Hr, u = tid - p * Hr;
  const int j0 = (int)((long long)p * Zc / Q), j1 = (int)((long long)(p + 1) * Zc / Q);
  const int i0 = (int)((long long)p * H / Q), i1 = (int)((long long)(p + 1) * H / Q);
  for (int e = tid; e < H * Zc; e += T) {
    const int uu = e / Zc, j = e - uu * Zc;
    W[uu * ld + j] = (j < n_in) ? W_in[(long long)uu * n_in + j] : W_rec[(long long)uu * H + (j - n_in)];
    if (!REG) G[uu * ld + j] = 0.f;
  }
  float greg[REG ? kGReg : 1];
#pragma unroll
  for (int i = 0; i < (REG ? kGReg : 1); ++i) greg[i] = 0.f;
  const float dtb = dt[dt_stride ? bi : 0];
  float du = 0.f, tau_eff = 1.f, carry = 0.f, gb = 0.f, gtau = 0.f, dh = 0.f;
  bool live = false;
  if (tid < H) {
    tau_eff = fmaxf(tau[tid], kTauEps);
    live = tau[tid] > kTauEps;
    du = expf(-dtb / tau_eff);
  }
  // Inputs of step k (s, h_k, the per-step seed, x_k) are loaded one step
  // ahead (n_in <= 1024 <= 8 T).
  constexpr int kXR = 8;
  float xr[kXR], ps = 0.f, php = 0.f, pup = 0.f;
  auto load_step = [&](int kk) {
    const long long rr = bi * K + kk;
    if (kk >= 0 && tid < H) {
      ps = s_in[rr * H + tid];
      php = (kk == 0) ? h0[bi * H + tid] : h_seq[(rr - 1) * H + tid];
      pup = grad_h_seq ? grad_h_seq[rr * H + tid] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < kXR; ++q) {
      const int j = tid + q * T;
      xr[q] = (kk >= 0 && j < n_in) ? x[rr * n_in + j] : 0.f;
    }
  };
  load_step(K - 1);
  for (int k = K - 1; k >= 0; --k) {
    const long long row = bi * K + k;
    const float s = ps, hp = php, up = pup;
#pragma unroll
    for (int q = 0; q < kXR; ++q)
      if (tid + q * T < n_in) z[tid + q * T] = xr[q];
    load_step(k - 1);
    // phase A (one thread per unit): dh, d_pre, gb, gtau, h_k into z
    if (tid < H) {
      dh = carry + up;
      if (k == K - 1) {
        if (grad_h_last) dh += grad_h_last[bi * H + tid];
        if (y) dh += h_seq[row * H + tid] - y[bi * H + tid];
      }
      const float dp = dh * (1.f - du) * (1.f - s * s);
      dpre[tid] = dp;
      gb += dp;
      if (live) gtau += dh * (hp - s) * du * dtb / (tau_eff * tau_eff);
      z[n_in + tid] = hp;
    }
    __syncthreads();
    // phase B (Q threads per unit): part p of the gradient row and of the carry
    if (u < H) {
      const float dp = dpre[u];
      const float* __restrict__ zz = z;
      if constexpr (REG) {
#pragma unroll
        for (int i = 0; i < kGReg; ++i)
          if (j0 + i < j1) greg[i] = fmaf(dp, zz[j0 + i], greg[i]);
      } else {
        float* __restrict__ g = G + u * ld;
#pragma unroll 4
        for (int j = j0; j < j1; ++j) g[j] = fmaf(dp, zz[j], g[j]);
      }
      const float* __restrict__ wc = W + n_in + u;
      const float* __restrict__ dpr = dpre;
      float c0 = 0.f, c1 = 0.f;
      int i = i0;
      for (; i + 1 < i1; i += 2) {
        c0 = fmaf(dpr[i], wc[i * ld], c0);
        c1 = fmaf(dpr[i + 1], wc[(i + 1) * ld], c1);
      }
      if (i < i1) c0 = fmaf(dpr[i], wc[i * ld], c0);
      part[p * H + u] = c0 + c1;
    }
    if (grad_x) {
      for (int j = tid; j < n_in; j += T) {
        const float* wc = W + j;
        float c0 = 0.f, c1 = 0.f;
        int i = 0;
        for (; i + 1 < H; i += 2) {
          c0 = fmaf(dpre[i], wc[i * ld], c0);
          c1 = fmaf(dpre[i + 1], wc[(i + 1) * ld], c1);
        }
        if (i < H) c0 = fmaf(dpre[i], wc[i * ld], c0);
        grad_x[row * n_in + j] = c0 + c1;
      }
    }
    __syncthreads();
    // phase C: carry of step k-1 = W_rec^T d_pre + dh * decay
    if (tid < H) carry = sum_parts(part, Q, H, tid) + dh * du;
  }
  __syncthreads();
  if (tid < H && grad_h0) grad_h0[bi * H + tid] = carry;
  // packed row [gW_in (u, j) | gW_rec (u, j) | gb (u) | gtau (u)]
  float* out = per_sample + bi * (long long)(Zc + 2) * H;
  if constexpr (REG) {
    if (u < H) {
#pragma unroll
      for (int i = 0; i < kGReg; ++i) {
        const int j = j0 + i;
        if (j < j1) {
          const long long off = (j < n_in) ? (long long)u * n_in + j : (long long)H * n_in + (long long)u * H + (j - n_in);
          out[off] = greg[i];
        }
      }
    }
  } else {
    for (int e = tid; e < H * Zc; e += T) {
      const int uu = e / Zc, j = e - uu * Zc;
      const long long off =
          (j < n_in) ? (long long)uu * n_in + j : (long long)H * n_in + (long long)uu * H + (j - n_in);
      out[off] = G[uu * ld + j];
    }
  }
  if (tid < H) {
    out[(long long)H * Zc + tid] = gb;
    out[(long long)H * Zc + H + tid] = gtau;
  }
}

size_t fwd_smem(int n_in, int H) {
  return ((size_t)H * ((n_in + H) | 1) + (n_in + H) + (size_t)tau_parts(H) * H) * sizeof(float);
}
size_t bwd_smem(int n_in, int H) {
  return ((size_t)2 * H * ((n_in + H) | 1) + (n_in + H) + H + (size_t)tau_parts(H) * H) * sizeof(float);
}
// A thread's share of a gradient row fits kGReg registers, with at most 512
// threads (128 registers each).
bool bwd_reg(int n_in, int H) {
  const int Q = tau_parts(H);
  return tau_threads(H) <= 512 && (n_in + H + Q - 1) / Q <= kGReg;
}
size_t bwd_smem_reg(int n_in, int H) {
  return ((size_t)H * ((n_in + H) | 1) + (n_in + H) + H + (size_t)tau_parts(H) * H) * sizeof(float);
}

}  // namespace

bool tau_shape_supported(int n_in, int H) {
  return n_in >= 1 && H >= 1 && n_in <= 1024 && H <= 1024 && bwd_smem(n_in, H) <= kTauSmemMax;
}

cudaError_t launch_tau_forward(const float* x, const float* h0, const float* W_in, const float* W_rec,
                               const float* b, const float* tau, const float* dt, int dt_stride, int B, int K,
                               int n_in, int H, float* h_seq, float* s_ws, cudaStream_t s) {
  const size_t smem = fwd_smem(n_in, H);
  cudaError_t e = cudaFuncSetAttribute(k_tau_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  TraceScope trace("tau_fwd", s);
  k_tau_fwd<<<B, tau_threads(H), smem, s>>>(x, h0, W_in, W_rec, b, tau, dt, dt_stride, K, n_in, H, h_seq,
                                                   s_ws);
  return cudaGetLastError();
}

cudaError_t launch_tau_backward(const float* x, const float* h0, const float* W_in, const float* W_rec,
                                const float* tau, const float* dt, int dt_stride, int B, int K, int n_in, int H,
                                const float* h_seq, const float* s_ws, const float* grad_h_seq,
                                const float* grad_h_last, const float* y, float* per_sample, float* grad_h0,
                                float* grad_x, float* grad_W_in, float* grad_W_rec, float* grad_b,
                                float* grad_tau, cudaStream_t s) {
  const bool reg = bwd_reg(n_in, H);
  const size_t smem = reg ? bwd_smem_reg(n_in, H) : bwd_smem(n_in, H);
  auto kern = reg ? k_tau_bwd<true> : k_tau_bwd<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  {
    TraceScope trace("tau_bwd", s);
    kern<<<B, tau_threads(H), smem, s>>>(x, h0, W_in, W_rec, tau, dt, dt_stride, K, n_in, H, h_seq, s_ws,
                                         grad_h_seq, grad_h_last, y, per_sample, grad_h0, grad_x);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const long long N = (long long)(n_in + H + 2) * H;
  ReduceOut o{};
  o.nseg = 4;
  o.ptr[0] = grad_W_in;
  o.begin[0] = 0;
  o.ptr[1] = grad_W_rec;
  o.begin[1] = (long long)H * n_in;
  o.ptr[2] = grad_b;
  o.begin[2] = (long long)H * (n_in + H);
  o.ptr[3] = grad_tau;
  o.begin[3] = (long long)H * (n_in + H + 1);
  return launch_reduce(per_sample, B, N, N, o, s);
}

}  // namespace cfc
