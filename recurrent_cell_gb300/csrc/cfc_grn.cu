// cfc_grn.cu -- multi-horizon GRN heads on every K position of the trunk
// state, forward and backward, FP32.
//
// Per horizon j of a trunk row h (length Hd; the ml-alpha commit history,
// commit "wire TFT GRN heads into PerceptionTrainer (Phase 1.7)"):
//   z1 = W1[j] h + b1[j],  a1 = GELU(z1) = z1 Phi(z1),  z2 = W2[j] a1 + b2[j],
//   gate = w_gate[j].z2 + b_gate[j],  main = w_main[j].z2 + b_main[j],
//   skip = w_skip[j].h + b_skip[j],  p = sigmoid(skip + sigmoid(gate) main).
// The backward ("K-loop Parallelization Implementation Plan", Commit 2 /
// Task 11: inputs probs, grad_probs, the saved z1 / a1 / z2 / gate / main, h,
// grad_h_carry and a per-horizon lambda on the trunk gradient only; ten
// parameter gradients accumulated per sample over the K positions; grad_h
// written whole) is the chain rule of that forward.
//
// The pages run one launch per K position.  The heads do not feed the
// recurrence, so here all B*K rows (r = b*K + k, the K loop's h_seq layout)
// go through one forward launch and one backward launch:
//   k_grn_fwd      grid (rows / 32, J): a 32-row tile, one horizon; W1[j],
//                  W2[j] and the row tile staged in shared memory (rows
//                  padded by 16 bytes), 2 rows x 4 units per thread.
//   k_grn_bwd_rows grid (rows / 16): all J horizons of a 16-row tile in turn
//                  (fixed order, so grad_h sums the horizons in order j = 0..J-1),
//                  dz2, dz1 = (W2^T dz2) GELU'(z1) and the trunk gradient
//                  W1^T dz1 + dskip w_skip, scaled by lambda_j, in registers;
//                  dz1, dz2, dgate, dmain, dskip go to the workspace.
//   k_grn_wgrad    grid (tiles, B): each packed gradient block is a product
//                  (left factors)^T x (right factors) over a sample's K rows;
//                  a block computes one tile of <= 64 x 64 outputs from the
//                  sample's rows staged in shared memory, every output summed
//                  over k = K-1 .. 0 (the pages' loop order) and written once
//                  (no += into scratch).
// reduce_axis0 then sums the B rows into the packed parameter gradient.
//
// The extern "C" entry points of the heads (declared in cfc.h) are at the end
// of this file; they validate the arguments before anything is launched.
#include <algorithm>

#include "cfc_internal.cuh"

namespace cfc {
namespace {

constexpr int kGrnRows = 32;          // rows per block
constexpr int kGrnThreads = 256;
constexpr int kGrnBwdRows = 16;       // rows per block of the backward (4 warps x 4 rows)
constexpr int kGrnBwdThreads = 128;
constexpr int kGrnBwdLdT = kGrnBwdRows + 4;   // row stride of the transposed dz tiles

struct GrnDims {
  int Hd, M, J;
  long long oW1, ob1, oW2, ob2, owg, obg, owm, obm, ows, obs, N;
  long long sv, sw;   // floats per row of the saved intermediates / of the workspace
};

__host__ __device__ inline GrnDims grn_dims(int Hd, int M, int J) {
  GrnDims d;
  d.Hd = Hd; d.M = M; d.J = J;
  const long long JM = (long long)J * M;
  d.oW1 = 0;
  d.ob1 = d.oW1 + JM * Hd;
  d.oW2 = d.ob1 + JM;
  d.ob2 = d.oW2 + JM * M;
  d.owg = d.ob2 + JM;
  d.obg = d.owg + JM;
  d.owm = d.obg + J;
  d.obm = d.owm + JM;
  d.ows = d.obm + J;
  d.obs = d.ows + (long long)J * Hd;
  d.N = d.obs + J;
  d.sv = 3 * JM + 2 * J;   // [z1 | a1 | z2 | gate | main]
  d.sw = 2 * JM + 3 * J;   // [dz1 | dz2 | dgate | dmain | dskip]
  return d;
}

// Asynchronous global -> shared copies (no register round trip, so a thread's
// copies are all in flight at once); src_bytes 0 writes zeros instead.
__device__ __forceinline__ void cpa16(float* dst, const float* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(valid ? 16u : 0u)
               : "memory");
}
__device__ __forceinline__ void cpa4(float* dst, const float* src, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src), "r"(valid ? 4u : 0u)
               : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cpa_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ float gelu_f(float z) { return 0.5f * z * (1.f + erff(z * 0.70710678118654752f)); }
__device__ __forceinline__ float gelu_grad_f(float z) {
  return 0.5f * (1.f + erff(z * 0.70710678118654752f)) + z * expf(-0.5f * z * z) * 0.39894228040143268f;
}
__device__ __forceinline__ float sigmoid_f(float z) { return 1.f / (1.f + expf(-z)); }

size_t fwd_smem_floats(int Hd, int M) {
  const int ldh = Hd + 4, ldm = M + 4;
  return (size_t)M * ldh + (size_t)kGrnRows * ldh + (size_t)M * ldm + 2 * (size_t)kGrnRows * ldm + 4 * (size_t)M +
         Hd;
}
size_t bwd_smem_floats(int Hd, int M) {
  const int ldh = Hd + 4, ldm = M + 4;
  return 2 * ((size_t)M * ldh + (size_t)M * ldm + 2 * (size_t)M + Hd) + 2 * (size_t)M * kGrnBwdLdT +
         3 * kGrnBwdRows;
}

__global__ void __launch_bounds__(kGrnThreads)
k_grn_fwd(const float* __restrict__ h, long long R, int Hd, int M, int J, const float* __restrict__ params,
          float* __restrict__ probs, float* __restrict__ saved) {
  extern __shared__ __align__(16) float sm[];
  const GrnDims d = grn_dims(Hd, M, J);
  const int j = blockIdx.y;
  const long long r0 = (long long)blockIdx.x * kGrnRows;
  const int ldh = Hd + 4, ldm = M + 4, tid = threadIdx.x;
  float* W1s = sm;                                  // [M][ldh]
  float* hs = W1s + (size_t)M * ldh;                // [32][ldh]
  float* W2s = hs + (size_t)kGrnRows * ldh;         // [M][ldm]
  float* as = W2s + (size_t)M * ldm;                // [32][ldm]  a1
  float* zs = as + (size_t)kGrnRows * ldm;          // [32][ldm]  z2
  float* b1s = zs + (size_t)kGrnRows * ldm;         // [M]
  float* b2s = b1s + M;                             // [M]
  float* wgs = b2s + M;                             // [M]
  float* wms = wgs + M;                             // [M]
  float* wss = wms + M;                             // [Hd]

  const float* W1 = params + d.oW1 + (long long)j * M * Hd;
  const float* W2 = params + d.oW2 + (long long)j * M * M;
  const int hq = Hd / 4, mq4 = M / 4;
  for (int e = tid; e < M * hq; e += kGrnThreads) {
    const int m = e / hq, q = e - m * hq;
    cpa16(W1s + (size_t)m * ldh + 4 * q, W1 + (size_t)m * Hd + 4 * q, true);
  }
  for (int e = tid; e < kGrnRows * hq; e += kGrnThreads) {
    const int rr = e / hq, q = e - rr * hq;
    const long long row = r0 + rr;
    cpa16(hs + (size_t)rr * ldh + 4 * q, row < R ? h + row * Hd + 4 * q : h, row < R);   // rows past R: zeros
  }
  for (int e = tid; e < M * mq4; e += kGrnThreads) {
    const int m = e / mq4, q = e - m * mq4;
    cpa16(W2s + (size_t)m * ldm + 4 * q, W2 + (size_t)m * M + 4 * q, true);
  }
  for (int e = tid; e < M; e += kGrnThreads) {
    cpa4(b1s + e, params + d.ob1 + (long long)j * M + e, true);
    cpa4(b2s + e, params + d.ob2 + (long long)j * M + e, true);
    cpa4(wgs + e, params + d.owg + (long long)j * M + e, true);
    cpa4(wms + e, params + d.owm + (long long)j * M + e, true);
  }
  for (int e = tid; e < Hd; e += kGrnThreads) cpa4(wss + e, params + d.ows + (long long)j * Hd + e, true);
  cpa_commit();
  cpa_wait<0>();
  __syncthreads();

  // thread -> rows 2rp, 2rp+1 and units m = mq + 16 t (t = 0..3)
  const int rp = tid / 16, mq = tid % 16;
  {
    float acc[2][4] = {};
    for (int i = 0; i < Hd; i += 4) {
      const float4 x0 = *reinterpret_cast<const float4*>(hs + (size_t)(2 * rp) * ldh + i);
      const float4 x1 = *reinterpret_cast<const float4*>(hs + (size_t)(2 * rp + 1) * ldh + i);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int m = mq + 16 * t;
        if (m < M) {
          const float4 w = *reinterpret_cast<const float4*>(W1s + (size_t)m * ldh + i);
          acc[0][t] = fmaf(w.x, x0.x, acc[0][t]);
          acc[0][t] = fmaf(w.y, x0.y, acc[0][t]);
          acc[0][t] = fmaf(w.z, x0.z, acc[0][t]);
          acc[0][t] = fmaf(w.w, x0.w, acc[0][t]);
          acc[1][t] = fmaf(w.x, x1.x, acc[1][t]);
          acc[1][t] = fmaf(w.y, x1.y, acc[1][t]);
          acc[1][t] = fmaf(w.z, x1.z, acc[1][t]);
          acc[1][t] = fmaf(w.w, x1.w, acc[1][t]);
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int lr = 2 * rp + rr;
      const long long row = r0 + lr;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int m = mq + 16 * t;
        if (m >= M) continue;
        const float z = acc[rr][t] + b1s[m];
        const float a = gelu_f(z);
        as[(size_t)lr * ldm + m] = a;
        if (row < R) {
          saved[row * d.sv + (long long)j * M + m] = z;
          saved[row * d.sv + (long long)J * M + (long long)j * M + m] = a;
        }
      }
    }
  }
  __syncthreads();
  {
    float acc[2][4] = {};
    for (int n = 0; n < M; n += 4) {
      const float4 x0 = *reinterpret_cast<const float4*>(as + (size_t)(2 * rp) * ldm + n);
      const float4 x1 = *reinterpret_cast<const float4*>(as + (size_t)(2 * rp + 1) * ldm + n);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int m = mq + 16 * t;
        if (m < M) {
          const float4 w = *reinterpret_cast<const float4*>(W2s + (size_t)m * ldm + n);
          acc[0][t] = fmaf(w.x, x0.x, acc[0][t]);
          acc[0][t] = fmaf(w.y, x0.y, acc[0][t]);
          acc[0][t] = fmaf(w.z, x0.z, acc[0][t]);
          acc[0][t] = fmaf(w.w, x0.w, acc[0][t]);
          acc[1][t] = fmaf(w.x, x1.x, acc[1][t]);
          acc[1][t] = fmaf(w.y, x1.y, acc[1][t]);
          acc[1][t] = fmaf(w.z, x1.z, acc[1][t]);
          acc[1][t] = fmaf(w.w, x1.w, acc[1][t]);
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int lr = 2 * rp + rr;
      const long long row = r0 + lr;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int m = mq + 16 * t;
        if (m >= M) continue;
        const float z = acc[rr][t] + b2s[m];
        zs[(size_t)lr * ldm + m] = z;
        if (row < R) saved[row * d.sv + 2ll * J * M + (long long)j * M + m] = z;
      }
    }
  }
  __syncthreads();
  // gate, main, skip and p: one warp per row (lane partial sums, then a
  // fixed xor tree)
  const int warp = tid / 32, lane = tid % 32;
  const float bg = params[d.obg + j], bm = params[d.obm + j], bsk = params[d.obs + j];
  for (int lr = warp * 4; lr < warp * 4 + 4; ++lr) {
    const long long row = r0 + lr;
    float g = 0.f, mn = 0.f, sk = 0.f;
    for (int m = lane; m < M; m += 32) {
      const float z = zs[(size_t)lr * ldm + m];
      g = fmaf(wgs[m], z, g);
      mn = fmaf(wms[m], z, mn);
    }
    for (int i = lane; i < Hd; i += 32) sk = fmaf(wss[i], hs[(size_t)lr * ldh + i], sk);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, off);
      mn += __shfl_xor_sync(0xffffffffu, mn, off);
      sk += __shfl_xor_sync(0xffffffffu, sk, off);
    }
    if (lane == 0 && row < R) {
      const float gate = g + bg, main = mn + bm, skip = sk + bsk;
      const float logit = skip + sigmoid_f(gate) * main;
      probs[row * J + j] = sigmoid_f(logit);
      saved[row * d.sv + 3ll * J * M + j] = gate;
      saved[row * d.sv + 3ll * J * M + J + j] = main;
    }
  }
}

__global__ void __launch_bounds__(kGrnBwdThreads)
k_grn_bwd_rows(long long R, int Hd, int M, int J, const float* __restrict__ params,
               const float* __restrict__ probs, const float* __restrict__ saved,
               const float* __restrict__ grad_probs, const float* __restrict__ lambda,
               const float* __restrict__ grad_h_carry, float* __restrict__ grad_h, float* __restrict__ ws) {
  extern __shared__ __align__(16) float sm[];
  const GrnDims d = grn_dims(Hd, M, J);
  const long long r0 = (long long)blockIdx.x * kGrnBwdRows;
  const int ldh = Hd + 4, ldm = M + 4, tid = threadIdx.x;
  // two buffers of one horizon's weights {W1 [M][ldh], W2 [M][ldm], w_gate,
  // w_main [M], w_skip [Hd]}: horizon j + 1 is copied in while j computes
  const size_t bufsz = (size_t)M * ldh + (size_t)M * ldm + 2 * (size_t)M + Hd;
  float* dz2T = sm + 2 * bufsz;                     // [M][kGrnBwdLdT]
  float* dz1T = dz2T + (size_t)M * kGrnBwdLdT;      // [M][kGrnBwdLdT]
  float* sc = dz1T + (size_t)M * kGrnBwdLdT;        // [16][3]: dgate, dmain, dskip
  const int hq = Hd / 4, mq4 = M / 4;
  const long long JM = (long long)J * M;
  const int rg = tid / 32, lane = tid % 32;         // rows 4rg..4rg+3; columns 4 (lane + 32 c) ..
  float acc[4][8] = {};                             // lambda-weighted trunk gradient, c = 0, 1

  auto stage = [&](int jj) {
    float* W1b = sm + (size_t)(jj & 1) * bufsz;
    float* W2b = W1b + (size_t)M * ldh;
    float* wgb = W2b + (size_t)M * ldm;
    const float* W1 = params + d.oW1 + (long long)jj * M * Hd;
    const float* W2 = params + d.oW2 + (long long)jj * M * M;
    for (int e = tid; e < M * hq; e += kGrnBwdThreads) {
      const int m = e / hq, q = e - m * hq;
      cpa16(W1b + (size_t)m * ldh + 4 * q, W1 + (size_t)m * Hd + 4 * q, true);
    }
    for (int e = tid; e < M * mq4; e += kGrnBwdThreads) {
      const int m = e / mq4, q = e - m * mq4;
      cpa16(W2b + (size_t)m * ldm + 4 * q, W2 + (size_t)m * M + 4 * q, true);
    }
    for (int e = tid; e < M; e += kGrnBwdThreads) {
      cpa4(wgb + e, params + d.owg + (long long)jj * M + e, true);
      cpa4(wgb + M + e, params + d.owm + (long long)jj * M + e, true);
    }
    for (int e = tid; e < Hd; e += kGrnBwdThreads) cpa4(wgb + 2 * M + e, params + d.ows + (long long)jj * Hd + e, true);
  };
  stage(0);
  cpa_commit();
  for (int j = 0; j < J; ++j) {
    __syncthreads();                                // the previous horizon's readers are done
    if (j + 1 < J) stage(j + 1);                    // into the buffer horizon j - 1 used
    cpa_commit();
    cpa_wait<1>();                                  // this thread's copies of horizon j have landed
    const float* W1s = sm + (size_t)(j & 1) * bufsz;
    const float* W2s = W1s + (size_t)M * ldh;
    const float* wgs = W2s + (size_t)M * ldm;
    const float* wms = wgs + M;
    const float* wss = wms + M;
    if (tid < kGrnBwdRows) {
      const long long row = r0 + tid;
      float dgate = 0.f, dmain = 0.f, dskip = 0.f;
      if (row < R) {
        const float p = probs[row * J + j], gp = grad_probs[row * J + j];
        const float gate = saved[row * d.sv + 3 * JM + j], main = saved[row * d.sv + 3 * JM + J + j];
        const float dl = gp * p * (1.f - p);
        const float sg = sigmoid_f(gate);
        dmain = dl * sg;
        dgate = dl * main * sg * (1.f - sg);
        dskip = dl;
        ws[row * d.sw + 2 * JM + j] = dgate;
        ws[row * d.sw + 2 * JM + J + j] = dmain;
        ws[row * d.sw + 2 * JM + 2 * J + j] = dskip;
      }
      sc[3 * tid] = dgate;
      sc[3 * tid + 1] = dmain;
      sc[3 * tid + 2] = dskip;
    }
    __syncthreads();
    // dz2 = dmain w_main + dgate w_gate (rows past R are zero)
    for (int e = tid; e < kGrnBwdRows * M; e += kGrnBwdThreads) {
      const int lr = e / M, m = e - lr * M;
      const long long row = r0 + lr;
      const float v = fmaf(sc[3 * lr + 1], wms[m], sc[3 * lr] * wgs[m]);
      dz2T[(size_t)m * kGrnBwdLdT + lr] = v;
      if (row < R) ws[row * d.sw + JM + (long long)j * M + m] = v;
    }
    __syncthreads();
    // dz1 = (W2^T dz2) GELU'(z1): thread -> rows 4rg.., units n = lane + 32 t
    {
      float a2[4][2] = {};
      for (int m = 0; m < M; ++m) {
        const float4 dz = *reinterpret_cast<const float4*>(dz2T + (size_t)m * kGrnBwdLdT + 4 * rg);
        const float w0 = (lane < M) ? W2s[(size_t)m * ldm + lane] : 0.f;
        const float w1 = (lane + 32 < M) ? W2s[(size_t)m * ldm + lane + 32] : 0.f;
        a2[0][0] = fmaf(w0, dz.x, a2[0][0]);
        a2[1][0] = fmaf(w0, dz.y, a2[1][0]);
        a2[2][0] = fmaf(w0, dz.z, a2[2][0]);
        a2[3][0] = fmaf(w0, dz.w, a2[3][0]);
        a2[0][1] = fmaf(w1, dz.x, a2[0][1]);
        a2[1][1] = fmaf(w1, dz.y, a2[1][1]);
        a2[2][1] = fmaf(w1, dz.z, a2[2][1]);
        a2[3][1] = fmaf(w1, dz.w, a2[3][1]);
      }
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int lr = 4 * rg + rr;
        const long long row = r0 + lr;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int n = lane + 32 * t;
          if (n >= M) continue;
          float v = 0.f;
          if (row < R) {
            v = a2[rr][t] * gelu_grad_f(saved[row * d.sv + (long long)j * M + n]);
            ws[row * d.sw + (long long)j * M + n] = v;
          }
          dz1T[(size_t)n * kGrnBwdLdT + lr] = v;
        }
      }
    }
    __syncthreads();
    // trunk gradient W1^T dz1 + dskip w_skip, scaled by lambda_j
    {
      float t[4][8] = {};
      for (int m = 0; m < M; ++m) {
        const float4 dz = *reinterpret_cast<const float4*>(dz1T + (size_t)m * kGrnBwdLdT + 4 * rg);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int cq = lane + 32 * c;
          if (4 * cq >= Hd) continue;
          const float4 w = *reinterpret_cast<const float4*>(W1s + (size_t)m * ldh + 4 * cq);
          const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            t[0][4 * c + e] = fmaf(wv[e], dz.x, t[0][4 * c + e]);
            t[1][4 * c + e] = fmaf(wv[e], dz.y, t[1][4 * c + e]);
            t[2][4 * c + e] = fmaf(wv[e], dz.z, t[2][4 * c + e]);
            t[3][4 * c + e] = fmaf(wv[e], dz.w, t[3][4 * c + e]);
          }
        }
      }
      const float lam = lambda[j];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const float dskip = sc[3 * (4 * rg + rr) + 2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int cq = lane + 32 * c;
          if (4 * cq >= Hd) continue;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float v = fmaf(dskip, wss[4 * cq + e], t[rr][4 * c + e]);
            acc[rr][4 * c + e] = fmaf(lam, v, acc[rr][4 * c + e]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const long long row = r0 + 4 * rg + rr;
    if (row >= R) continue;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int cq = lane + 32 * c;
      if (4 * cq >= Hd) continue;
      float4 v = make_float4(acc[rr][4 * c], acc[rr][4 * c + 1], acc[rr][4 * c + 2], acc[rr][4 * c + 3]);
      if (grad_h_carry) {
        const float4 cr = *reinterpret_cast<const float4*>(grad_h_carry + row * Hd + 4 * cq);
        v.x += cr.x; v.y += cr.y; v.z += cr.z; v.w += cr.w;
      }
      *reinterpret_cast<float4*>(grad_h + row * Hd + 4 * cq) = v;
    }
  }
}

// Per-sample parameter gradients as small contractions over the sample's K
// rows.  Every packed block is a product (left factors)^T x (right factors):
//   W1[j][m][i]   = sum_k dz1[j][m] h[i]        w_skip[j][i] = sum_k dskip[j] h[i]
//   W2[j][m][q]   = sum_k dz2[j][m] a1[j][q]
//   w_gate[j][m]  = sum_k dgate[j] z2[j][m]     w_main[j][m] = sum_k dmain[j] z2[j][m]
//   b1, b2, b_gate, b_main, b_skip = sum_k of the left factor (right factor 1)
// A task is one tile of at most 64 left x 64 right columns of one such
// product; block (task, b) stages the sample's rows of both factors in shared
// memory, 64 rows at a time, and each thread accumulates 4 x 4 outputs.  Each
// output is one fmaf chain over k = K-1 .. 0 (the pages' loop order), so the
// result is exactly the per-element sum.
constexpr int kWgTile = 64;
constexpr int kWgLd = kWgTile + 4;          // padded row of the staged tiles
constexpr int kWgMaxTasks = 96;

struct GrnWgTask {
  int Lbase, Lcs, nL;       // left column c of row r: ws[r * sw + Lbase + c * Lcs]
  int Rsel, Rbase, nR;      // right column i of row r: 0 -> 1.0; 1 -> h[r * Hd + Rbase + i];
                            // 2 -> saved[r * sv + Rbase + i]
  long long Obase;          // output (c, i) -> per_sample[b * N + Obase + c * Ocs + i]
  int Ocs;
};
struct GrnWgTable {
  int count;
  GrnWgTask t[kWgMaxTasks];
};

__global__ void __launch_bounds__(256)
k_grn_wgrad(const __grid_constant__ GrnWgTable tab, const float* __restrict__ h, const float* __restrict__ saved,
            const float* __restrict__ ws, int K, int Hd, int M, int J, float* __restrict__ per_sample) {
  __shared__ __align__(16) float Ls[kWgTile][kWgLd];
  __shared__ __align__(16) float Rs[kWgTile][kWgLd];
  const GrnDims d = grn_dims(Hd, M, J);
  const GrnWgTask T = tab.t[blockIdx.x];
  const long long b = blockIdx.y;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const float* Rsrc = T.Rsel == 1 ? h : saved;
  const long long rrs = T.Rsel == 1 ? Hd : d.sv;
  float acc[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[a][c] = 0.f;
  // row chunks from the last one down, rows in a chunk from the last one down
  for (int k1 = K; k1 > 0; k1 -= kWgTile) {
    const int k0 = k1 > kWgTile ? k1 - kWgTile : 0, nk = k1 - k0;
    __syncthreads();
    for (int e = tid; e < kWgTile * kWgTile; e += 256) {
      const int kk = e >> 6, c = e & 63;
      const long long r = b * K + k0 + kk;
      const bool lv = kk < nk && c < T.nL, rv = kk < nk && c < T.nR;
      cpa4(&Ls[kk][c], lv ? ws + r * d.sw + T.Lbase + (long long)c * T.Lcs : ws, lv);   // zeros outside
      if (T.Rsel == 0) Rs[kk][c] = rv ? 1.f : 0.f;
      else cpa4(&Rs[kk][c], rv ? Rsrc + r * rrs + T.Rbase + c : Rsrc, rv);
    }
    cpa_commit();
    cpa_wait<0>();
    __syncthreads();
    for (int kk = nk - 1; kk >= 0; --kk) {
      const float4 l4 = *reinterpret_cast<const float4*>(&Ls[kk][4 * ty]);
      const float4 r4 = *reinterpret_cast<const float4*>(&Rs[kk][4 * tx]);
      const float lf[4] = {l4.x, l4.y, l4.z, l4.w}, rf[4] = {r4.x, r4.y, r4.z, r4.w};
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[a][c] = fmaf(lf[a], rf[c], acc[a][c]);
    }
  }
  float* out = per_sample + b * d.N + T.Obase;
#pragma unroll
  for (int a = 0; a < 4; ++a) {
    const int c = 4 * ty + a;
    if (c >= T.nL) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = 4 * tx + q;
      if (i < T.nR) out[(long long)c * T.Ocs + i] = acc[a][q];
    }
  }
}

// The task table of the packed gradient (at most kWgMaxTasks tiles for the
// supported shapes: J <= 8, M <= 64, Hd <= 256).
bool build_wgrad_tasks(const GrnDims& d, GrnWgTable* tab) {
  const int Hd = d.Hd, M = d.M, J = d.J, JM = J * M;
  tab->count = 0;
  auto add = [&](int Lbase, int Lcs, int nL, int Rsel, int Rbase, int nR, long long Obase, int Ocs) {
    for (int c0 = 0; c0 < nL; c0 += kWgTile)
      for (int i0 = 0; i0 < nR; i0 += kWgTile) {
        if (tab->count == kWgMaxTasks) return false;
        GrnWgTask& t = tab->t[tab->count++];
        t.Lbase = Lbase + c0 * Lcs;
        t.Lcs = Lcs;
        t.nL = std::min(kWgTile, nL - c0);
        t.Rsel = Rsel;
        t.Rbase = Rbase + i0;
        t.nR = std::min(kWgTile, nR - i0);
        t.Obase = Obase + (long long)c0 * Ocs + i0;
        t.Ocs = Ocs;
      }
    return true;
  };
  bool ok = true;
  ok = ok && add(0, 1, JM, 1, 0, Hd, d.oW1, Hd);                                  // W1
  ok = ok && add(2 * JM + 2 * J, 1, J, 1, 0, Hd, d.ows, Hd);                      // w_skip
  for (int j = 0; j < J && ok; ++j)
    ok = add(JM + j * M, 1, M, 2, JM + j * M, M, d.oW2 + (long long)j * M * M, M);   // W2[j]
  for (int j = 0; j < J && ok; ++j)                                               // w_gate[j], w_main[j]
    ok = add(2 * JM + j, J, 2, 2, 2 * JM + j * M, M, d.owg + (long long)j * M, (int)(d.owm - d.owg));
  ok = ok && add(0, 1, JM, 0, 0, 1, d.ob1, 1);                                    // b1
  ok = ok && add(JM, 1, JM, 0, 0, 1, d.ob2, 1);                                   // b2
  ok = ok && add(2 * JM, 1, J, 0, 0, 1, d.obg, 1);                                // b_gate
  ok = ok && add(2 * JM + J, 1, J, 0, 0, 1, d.obm, 1);                            // b_main
  ok = ok && add(2 * JM + 2 * J, 1, J, 0, 0, 1, d.obs, 1);                        // b_skip
  return ok;
}

}  // namespace

bool grn_shape_supported(int Hd, int M, int J) {
  return Hd >= 4 && Hd <= 256 && Hd % 4 == 0 && M >= 4 && M <= 64 && M % 4 == 0 && J >= 1 && J <= 8;
}

long long grn_param_length(int Hd, int M, int J) { return grn_dims(Hd, M, J).N; }
long long grn_saved_per_row(int M, int J) { return grn_dims(4, M, J).sv; }
long long grn_ws_per_row(int M, int J) { return grn_dims(4, M, J).sw; }

cudaError_t launch_grn_forward(const float* h, long long R, int Hd, int M, int J, const float* params,
                               float* probs, float* saved, cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const size_t smem = fwd_smem_floats(Hd, M) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_grn_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((R + kGrnRows - 1) / kGrnRows), (unsigned)J);
  TraceScope trace("grn_fwd", s);
  k_grn_fwd<<<grid, kGrnThreads, smem, s>>>(h, R, Hd, M, J, params, probs, saved);
  return cudaGetLastError();
}

cudaError_t launch_grn_backward(const float* h, int B, int K, int Hd, int M, int J, const float* params,
                                const float* probs, const float* saved, const float* grad_probs,
                                const float* lambda, const float* grad_h_carry, float* grad_h, float* ws,
                                float* per_sample, float* grad_params, cudaStream_t s) {
  const long long R = (long long)B * K;
  const GrnDims d = grn_dims(Hd, M, J);
  {
    const size_t smem = bwd_smem_floats(Hd, M) * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_grn_bwd_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    TraceScope trace("grn_bwd_rows", s);
    k_grn_bwd_rows<<<(unsigned)((R + kGrnBwdRows - 1) / kGrnBwdRows), kGrnBwdThreads, smem, s>>>(
        R, Hd, M, J, params, probs, saved, grad_probs, lambda, grad_h_carry, grad_h, ws);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  {
    GrnWgTable tab;
    if (!build_wgrad_tasks(d, &tab)) return cudaErrorInvalidValue;
    TraceScope trace("grn_wgrad", s);
    dim3 grid((unsigned)tab.count, (unsigned)B);
    k_grn_wgrad<<<grid, 256, 0, s>>>(tab, h, saved, ws, K, Hd, M, J, per_sample);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  ReduceOut o{};
  o.nseg = 1;
  o.ptr[0] = grad_params;
  o.begin[0] = 0;
  return launch_reduce(per_sample, B, d.N, d.N, o, s);
}

}  // namespace cfc

// ---------------------------------------------------------------------------
// C entry points
// ---------------------------------------------------------------------------

namespace {
bool grn_al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t grn_align256(size_t v) { return (v + 255) & ~size_t(255); }
}  // namespace

using namespace cfc;

extern "C" {

long long cfc_grn_param_length(int hidden, int head_mid, int n_horizons) {
  return grn_shape_supported(hidden, head_mid, n_horizons) ? grn_param_length(hidden, head_mid, n_horizons) : 0;
}

long long cfc_grn_saved_per_row(int head_mid, int n_horizons) {
  return grn_shape_supported(4, head_mid, n_horizons) ? grn_saved_per_row(head_mid, n_horizons) : 0;
}

size_t cfc_grn_workspace_bytes(int B, int K, int hidden, int head_mid, int n_horizons) {
  if (B < 1 || K < 1 || !grn_shape_supported(hidden, head_mid, n_horizons)) return 0;
  return grn_align256((size_t)B * K * grn_ws_per_row(head_mid, n_horizons) * sizeof(float));
}

int cfc_grn_forward(const float* h, long long rows, int hidden, int head_mid, int n_horizons,
                    const float* params, float* probs, float* saved, void* stream) {
  if (rows < 0 || rows > (1ll << 31) || !grn_shape_supported(hidden, head_mid, n_horizons)) return CFC_ERR_SHAPE;
  if (rows == 0) return CFC_OK;
  const void* ptrs[] = {h, params, probs, saved};
  for (const void* p : ptrs)
    if (!p) return CFC_ERR_NULL;
  for (const void* p : ptrs)
    if (!grn_al16(p)) return CFC_ERR_ALIGN;
  cudaError_t e = launch_grn_forward(h, rows, hidden, head_mid, n_horizons, params, probs, saved,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CFC_OK : CFC_ERR_LAUNCH;
}

int cfc_grn_backward(const float* h, int B, int K, int hidden, int head_mid, int n_horizons, const float* params,
                     const float* probs, const float* saved, const float* grad_probs, const float* lambda,
                     const float* grad_h_carry, float* grad_h, float* per_sample_scratch, float* grad_params,
                     void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 1 || K < 1 || (long long)B * K > (1ll << 31) || !grn_shape_supported(hidden, head_mid, n_horizons))
    return CFC_ERR_SHAPE;
  const void* ptrs[] = {h, params, probs, saved, grad_probs, lambda, grad_h, per_sample_scratch, grad_params};
  for (const void* p : ptrs)
    if (!p) return CFC_ERR_NULL;
  for (const void* p : ptrs)
    if (!grn_al16(p)) return CFC_ERR_ALIGN;
  if (grad_h_carry && !grn_al16(grad_h_carry)) return CFC_ERR_ALIGN;
  if (!workspace || workspace_bytes < cfc_grn_workspace_bytes(B, K, hidden, head_mid, n_horizons))
    return CFC_ERR_WORKSPACE;
  if (!grn_al16(workspace)) return CFC_ERR_ALIGN;
  cudaError_t e = launch_grn_backward(h, B, K, hidden, head_mid, n_horizons, params, probs, saved, grad_probs,
                                      lambda, grad_h_carry, grad_h, static_cast<float*>(workspace),
                                      per_sample_scratch, grad_params, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CFC_OK : CFC_ERR_LAUNCH;
}

}  // extern "C"
