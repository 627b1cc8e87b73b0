// cfc_simt.cu -- CUDA-core (FFMA) kernels of the batched CfC K-loop.
//
//   k_prep_wt      W_cat^T [Zc, 3H] (Zc = n_in + H): transposed, mode-rounded
//                  copy of [W_in | W_rec] so that a thread per hidden unit reads
//                  weights with coalesced loads in the forward.
//   k_cfc_fwd      persistent forward: one block per tile of BT samples, one
//                  thread per hidden unit, the K loop inside the kernel.  The
//                  operand vector z = [x_k; h_k] of the tile lives in shared
//                  memory; h_{k+1} never leaves the block between steps.
//   k_cfc_bwd      persistent reverse-K loop: one thread per hidden unit for
//                  the elementwise dA, one thread per column of z for
//                  dz = W_cat^T dA (grad_x | carry); writes dA of every step.
//   k_wgrad        gradient contraction out[s] = sum_{rows r in block s}
//                  dA[r]^T (x) [x_r; h_r; 1] written in the packed per-sample
//                  layout (one row block per sample for the scratch path, or
//                  a fixed split of all B*K rows for the GEMM path).
//
// Samples are independent through the whole K loop, so blocks never wait on
// one another.  The pages' kernels ("K-loop Parallelization Implementation
// Plan", Tasks 2-3) launch one block per sample per step and accumulate the
// per-sample gradients with += in global scratch at every step; here the K
// loop runs inside one launch and every gradient element is written once.
#include <algorithm>

#include "cfc_internal.cuh"

namespace cfc {
namespace {

template <typename T, int MODE>
__global__ void k_prep_wt(const T* __restrict__ W_in, const T* __restrict__ W_rec,
                          int n_in, int H, T* __restrict__ WT) {
  const int H3 = 3 * H, Zc = n_in + H;
  const long long total = (long long)H3 * Zc;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int j = (int)(e / H3);
    const int r = (int)(e - (long long)j * H3);
    const float v = (j < n_in) ? ld_operand<MODE>(W_in + (long long)r * n_in + j)
                               : ld_operand<MODE>(W_rec + (long long)r * H + (j - n_in));
    stf(WT + e, v);
  }
}

constexpr int kMaxThreads = 512;

// Forward.  blockDim.x = min(512, round_up(H, 32)); dynamic smem = 2 * BT * Zc
// floats: two copies of the operand tile z = [x_k; h_k] used alternately, so
// step k reads one copy while h_{k+1} and x_{k+1} are written to the other and
// a single barrier per step orders them.
template <typename T, int MODE, int BT>
__global__ void __launch_bounds__(kMaxThreads)
k_cfc_fwd(const T* __restrict__ x, const T* __restrict__ h0, const T* __restrict__ WT,
          const float* __restrict__ bias, const float* __restrict__ dt, int dt_stride,
          int B, int K, int n_in, int H, T* __restrict__ h_seq, float* __restrict__ act) {
  extern __shared__ float zbuf[];  // [2][BT][Zc]
  const int Zc = n_in + H, H3 = 3 * H;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int b0 = blockIdx.x * BT;

  for (int e = tid; e < BT * H; e += nthr) {
    const int n = e / H, u = e - n * H, bb = b0 + n;
    zbuf[n * Zc + n_in + u] = (bb < B) ? ld_operand<MODE>(h0 + (long long)bb * H + u) : 0.f;
  }
  for (int e = tid; e < BT * n_in; e += nthr) {
    const int n = e / n_in, j = e - n * n_in, bb = b0 + n;
    zbuf[n * Zc + j] = (bb < B) ? ld_operand<MODE>(x + (long long)bb * K * n_in + j) : 0.f;
  }
  float dtn[BT];
#pragma unroll
  for (int n = 0; n < BT; ++n) dtn[n] = (b0 + n < B) ? dt[dt_stride ? b0 + n : 0] : 0.f;
  __syncthreads();

  for (int k = 0; k < K; ++k) {
    const float* zs = zbuf + (k & 1) * BT * Zc;
    float* zn = zbuf + ((k + 1) & 1) * BT * Zc;
    for (int i = tid; i < H; i += nthr) {
      float af[BT], ag[BT], ah[BT];
      const float bf = bias[i], bg = bias[H + i], bh = bias[2 * H + i];
#pragma unroll
      for (int n = 0; n < BT; ++n) { af[n] = bf; ag[n] = bg; ah[n] = bh; }
      const T* w = WT + i;
#pragma unroll 4
      for (int j = 0; j < Zc; ++j) {
        const float wf = ldf(w + (long long)j * H3);
        const float wg = ldf(w + (long long)j * H3 + H);
        const float wh = ldf(w + (long long)j * H3 + 2 * H);
#pragma unroll
        for (int n = 0; n < BT; ++n) {
          const float z = zs[n * Zc + j];
          af[n] = fmaf(wf, z, af[n]);
          ag[n] = fmaf(wg, z, ag[n]);
          ah[n] = fmaf(wh, z, ah[n]);
        }
      }
#pragma unroll
      for (int n = 0; n < BT; ++n) {
        const int bb = b0 + n;
        const float g = tanhf(ag[n]);
        const float hh = tanhf(ah[n]);
        const float gate = 1.f / (1.f + expf(af[n] * dtn[n]));
        const float h = gate * g + (1.f - gate) * hh;
        if (bb < B) {
          const long long row = (long long)bb * K + k;
          act[row * H3 + i] = gate;
          act[row * H3 + H + i] = g;
          act[row * H3 + 2 * H + i] = hh;
          stf(h_seq + row * H + i, h);
        }
        float hop;
        if constexpr (sizeof(T) == 2) hop = round_bf16(h);   // the stored bf16 state
        else hop = to_operand<MODE>(h);
        zn[n * Zc + n_in + i] = (bb < B) ? hop : 0.f;
      }
    }
    if (k + 1 < K) {
      for (int e = tid; e < BT * n_in; e += nthr) {
        const int n = e / n_in, j = e - n * n_in, bb = b0 + n;
        zn[n * Zc + j] = (bb < B) ? ld_operand<MODE>(x + ((long long)bb * K + k + 1) * n_in + j) : 0.f;
      }
    }
    __syncthreads();
  }
}

// Backward.  blockDim.x = min(512, round_up(Zc, 32)); dynamic smem = BT * 4H floats.
template <typename T, typename DT, int MODE, int BT>
__global__ void __launch_bounds__(kMaxThreads)
k_cfc_bwd(const T* __restrict__ W_in, const T* __restrict__ W_rec,
          const float* __restrict__ dt, int dt_stride, int B, int K, int n_in, int H,
          const T* __restrict__ h_seq, const float* __restrict__ grad_h_seq,
          const float* __restrict__ grad_h_last, const float* __restrict__ y,
          const float* __restrict__ act, DT* __restrict__ dA_out,
          float* __restrict__ grad_h0, float* __restrict__ grad_x) {
  extern __shared__ float sm[];
  const int Zc = n_in + H, H3 = 3 * H;
  float* dAs = sm;               // [BT][3H] operand values of dA
  float* carry = sm + BT * H3;   // [BT][H]   gradient reaching h_{k+1} through step k+1
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int b0 = blockIdx.x * BT;

  for (int e = tid; e < BT * H; e += nthr) carry[e] = 0.f;
  float dtn[BT];
#pragma unroll
  for (int n = 0; n < BT; ++n) dtn[n] = (b0 + n < B) ? dt[dt_stride ? b0 + n : 0] : 0.f;
  __syncthreads();

  for (int k = K - 1; k >= 0; --k) {
    for (int i = tid; i < H; i += nthr) {
#pragma unroll
      for (int n = 0; n < BT; ++n) {
        const int bb = b0 + n;
        float d0 = 0.f, d1 = 0.f, d2 = 0.f;
        if (bb < B) {
          const long long row = (long long)bb * K + k;
          float delta = carry[n * H + i];
          if (grad_h_seq) delta += grad_h_seq[row * H + i];
          if (k == K - 1) {
            if (grad_h_last) delta += grad_h_last[(long long)bb * H + i];
            if (y) delta += ldf(h_seq + row * H + i) - y[(long long)bb * H + i];
          }
          const float gate = act[row * H3 + i];
          const float g = act[row * H3 + H + i];
          const float hh = act[row * H3 + 2 * H + i];
          d1 = delta * gate * (1.f - g * g);
          d2 = delta * (1.f - gate) * (1.f - hh * hh);
          d0 = -dtn[n] * delta * (g - hh) * gate * (1.f - gate);
          d0 = to_operand<MODE>(d0);
          d1 = to_operand<MODE>(d1);
          d2 = to_operand<MODE>(d2);
          stf(dA_out + row * H3 + i, d0);
          stf(dA_out + row * H3 + H + i, d1);
          stf(dA_out + row * H3 + 2 * H + i, d2);
        }
        dAs[n * H3 + i] = d0;
        dAs[n * H3 + H + i] = d1;
        dAs[n * H3 + 2 * H + i] = d2;
      }
    }
    __syncthreads();
    // dz[j] = sum_r W_cat[r, j] dA[r]: column j of W_cat = [W_in | W_rec]
    // (coalesced over j).  carry is not read in this phase, so it is
    // overwritten in place.
    for (int j = tid; j < Zc; j += nthr) {
      const T* wcol = (j < n_in) ? (W_in + j) : (W_rec + (j - n_in));
      const int ldw = (j < n_in) ? n_in : H;
      float acc[BT];
#pragma unroll
      for (int n = 0; n < BT; ++n) acc[n] = 0.f;
#pragma unroll 4
      for (int r = 0; r < H3; ++r) {
        const float w = ld_operand<MODE>(wcol + (long long)r * ldw);
#pragma unroll
        for (int n = 0; n < BT; ++n) acc[n] = fmaf(w, dAs[n * H3 + r], acc[n]);
      }
#pragma unroll
      for (int n = 0; n < BT; ++n) {
        const int bb = b0 + n;
        if (j < n_in) {
          if (grad_x && bb < B) grad_x[((long long)bb * K + k) * n_in + j] = acc[n];
        } else {
          carry[n * H + (j - n_in)] = acc[n];
        }
      }
    }
    __syncthreads();
  }
  if (grad_h0) {
    for (int e = tid; e < BT * H; e += nthr) {
      const int n = e / H, u = e - n * H;
      if (b0 + n < B) grad_h0[(long long)(b0 + n) * H + u] = carry[e];
    }
  }
}

// Gradient contraction, 64 x 64 output tile per block, 4 x 4 per thread.
constexpr int kTM = 64, kTN = 64, kTR = 16;

template <typename T, typename DT, int MODE>
__global__ void __launch_bounds__(256, 5)
k_wgrad(const DT* __restrict__ dA, const T* __restrict__ x, const T* __restrict__ h0,
        const T* __restrict__ h_seq, int K, int n_in, int H, long long R,
        long long rows_per_split, float* __restrict__ out) {
  // Thread (ty, tx) owns outputs m = m0 + 4*ty + p, j = j0 + 4*tx + q (p, q < 4):
  // per row one 128-bit shared load of dA and one of z feed 16 FMAs.  The
  // next row chunk is loaded into registers while the current one is used.
  __shared__ __align__(16) float sA[2][kTR][kTM];
  __shared__ __align__(16) float sZ[2][kTR][kTN];
  const int H3 = 3 * H, Zc = n_in + H, Zb = Zc + 1;
  const long long N = (long long)H3 * Zb;
  const int m0 = blockIdx.x * kTM, j0 = blockIdx.y * kTN;
  const long long s = blockIdx.z;
  const int r_begin = (int)(s * rows_per_split);            // B*K < 2^31
  const int r_end = (int)min(R, (long long)r_begin + rows_per_split);
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  constexpr int kPer = (kTR * kTM) / 256;                   // elements per thread per chunk

  // Row of element q of a chunk: r + tid/kTM + q*(256/kTM).  Its step index
  // (row mod K) and sample (row / K) advance by kTR rows per chunk, kept
  // incrementally (no integer division in the loop).
  constexpr int kRowStep = 256 / kTM;
  int kq[kPer], bq[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int row = r_begin + tid / kTM + q * kRowStep;
    bq[q] = row / K;
    kq[q] = row - bq[q] * K;
  }
  float ra[kPer], rz[kPer];
  const int cc = tid % kTM;
  const int m = m0 + cc, j = j0 + cc;
  auto load_chunk = [&](int r) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int row = r + tid / kTM + q * kRowStep;
      float a = 0.f, z = 0.f;
      if (row < r_end) {
        if (m < H3) a = ldf(dA + (long long)row * H3 + m);
        if (j < n_in) {
          z = ld_operand<MODE>(x + (long long)row * n_in + j);
        } else if (j < Zc) {
          const int u = j - n_in;
          z = (kq[q] == 0) ? ld_operand<MODE>(h0 + (long long)bq[q] * H + u)
                           : ld_operand<MODE>(h_seq + (long long)(row - 1) * H + u);
        } else if (j == Zc) {
          z = 1.f;
        }
      }
      ra[q] = a;
      rz[q] = z;
      // the same element of the next chunk: kTR rows further
      kq[q] += kTR;
      while (kq[q] >= K) {
        kq[q] -= K;
        ++bq[q];
      }
    }
  };

  // When Zc is a multiple of kTN the bias column would be a tile of its own;
  // the block whose tile ends at Zc sums it instead (accb, one per m row).
  const bool fold_bias = (Zc % kTN == 0) && (j0 + kTN == Zc);
  float acc[4][4], accb[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    accb[p] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[p][q] = 0.f;
  }

  if (r_begin < r_end) load_chunk(r_begin);
  int buf = 0;
  for (int r = r_begin; r < r_end; r += kTR, buf ^= 1) {
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int rr = tid / kTM + q * kRowStep;
      sA[buf][rr][cc] = ra[q];
      sZ[buf][rr][cc] = rz[q];
    }
    __syncthreads();
    if (r + kTR < r_end) load_chunk(r + kTR);
#pragma unroll
    for (int rr = 0; rr < kTR; ++rr) {
      const float4 av = *reinterpret_cast<const float4*>(&sA[buf][rr][4 * ty]);
      const float4 zv = *reinterpret_cast<const float4*>(&sZ[buf][rr][4 * tx]);
      const float a4[4] = {av.x, av.y, av.z, av.w}, z4[4] = {zv.x, zv.y, zv.z, zv.w};
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(a4[p], z4[q], acc[p][q]);
      if (fold_bias) {
#pragma unroll
        for (int p = 0; p < 4; ++p) accb[p] += a4[p];
      }
    }
    // The buffer written next iteration is the other one; the barrier at the
    // top of the iteration after that orders its reuse.
  }
  float* o = out + s * N;
  const long long off_rec = (long long)H3 * n_in;
  const long long off_b = (long long)H3 * Zc;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const int m = m0 + 4 * ty + p;
    if (m >= H3) continue;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + 4 * tx + q;
      if (j < n_in) o[(long long)m * n_in + j] = acc[p][q];
      else if (j < Zc) o[off_rec + (long long)m * H + (j - n_in)] = acc[p][q];
      else if (j == Zc) o[off_b + m] = acc[p][q];
    }
    if (fold_bias && tx == 0) o[off_b + m] = accb[p];
  }
}

// Samples per block: the smallest tile that keeps the grid within about two
// blocks per SM, limited so that the tile's shared memory (smem_per_sample
// bytes per sample) stays within 200 KB.
int pick_bt(int B, size_t smem_per_sample) {
  const int bts[5] = {1, 2, 4, 8, 16};
  int pick = 16;
  for (int t : bts)
    if ((B + t - 1) / t <= 2 * kNumSMs) { pick = t; break; }
  while (pick > 1 && (size_t)pick * smem_per_sample > 200 * 1024) pick /= 2;
  return pick;
}

template <typename T, int MODE, int BT>
cudaError_t fwd_bt(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  const int threads = std::min(kMaxThreads, (L.H + 31) / 32 * 32);
  const size_t smem = 2 * (size_t)BT * L.Zc * sizeof(float);
  auto kern = k_cfc_fwd<T, MODE, BT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int grid = (L.B + BT - 1) / BT;
  TraceScope trace("cfc_fwd_simt", s);
  kern<<<grid, threads, smem, s>>>(
      static_cast<const T*>(a.x), static_cast<const T*>(a.h0),
      reinterpret_cast<const T*>(a.ws + L.off_wt), a.b, a.dt, a.dt_stride,
      L.B, L.K, L.n_in, L.H, static_cast<T*>(a.h_seq), reinterpret_cast<float*>(a.ws + L.off_act));
  return cudaGetLastError();
}

template <typename T, typename DT, int MODE, int BT>
cudaError_t bwd_bt(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  const int threads = std::min(kMaxThreads, (L.Zc + 31) / 32 * 32);
  const size_t smem = (size_t)BT * 4 * L.H * sizeof(float);
  auto kern = k_cfc_bwd<T, DT, MODE, BT>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int grid = (L.B + BT - 1) / BT;
  TraceScope trace("cfc_bwd_simt", s);
  kern<<<grid, threads, smem, s>>>(
      static_cast<const T*>(a.W_in), static_cast<const T*>(a.W_rec), a.dt, a.dt_stride,
      L.B, L.K, L.n_in, L.H, static_cast<const T*>(a.h_seq), a.grad_h_seq, a.grad_h_last, a.y,
      reinterpret_cast<const float*>(a.ws + L.off_act), reinterpret_cast<DT*>(a.ws + L.off_dA),
      a.grad_h0, a.grad_x);
  return cudaGetLastError();
}

template <typename T, int MODE>
cudaError_t forward_mode(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  {
    const long long total = (long long)L.H3 * L.Zc;
    const int threads = 256;
    const int blocks = (int)std::min<long long>((total + threads - 1) / threads, 4 * kNumSMs);
    TraceScope trace("prep_wt", s);
    k_prep_wt<T, MODE><<<blocks, threads, 0, s>>>(static_cast<const T*>(a.W_in),
                                                  static_cast<const T*>(a.W_rec), L.n_in, L.H,
                                                  reinterpret_cast<T*>(a.ws + L.off_wt));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  switch (pick_bt(L.B, 2 * (size_t)L.Zc * sizeof(float))) {
    case 1: return fwd_bt<T, MODE, 1>(L, a, s);
    case 2: return fwd_bt<T, MODE, 2>(L, a, s);
    case 4: return fwd_bt<T, MODE, 4>(L, a, s);
    case 8: return fwd_bt<T, MODE, 8>(L, a, s);
    default: return fwd_bt<T, MODE, 16>(L, a, s);
  }
}

template <typename T, typename DT, int MODE>
cudaError_t backward_mode(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  switch (pick_bt(L.B, 4 * (size_t)L.H * sizeof(float))) {
    case 1: return bwd_bt<T, DT, MODE, 1>(L, a, s);
    case 2: return bwd_bt<T, DT, MODE, 2>(L, a, s);
    case 4: return bwd_bt<T, DT, MODE, 4>(L, a, s);
    case 8: return bwd_bt<T, DT, MODE, 8>(L, a, s);
    default: return bwd_bt<T, DT, MODE, 16>(L, a, s);
  }
}

template <typename T, typename DT, int MODE>
cudaError_t wgrad_mode(const Layout& L, const CfcArgs& a, float* out, int n_split,
                       long long rows_per_split, cudaStream_t s) {
  // Column tiles of z = [x; h; 1]; a bias column alone in a last tile is
  // folded into the tile before it.
  const int ntn = (L.Zc % kTN == 0) ? L.Zc / kTN : (L.Zc + 1 + kTN - 1) / kTN;
  dim3 grid((L.H3 + kTM - 1) / kTM, ntn, n_split);
  TraceScope trace("wgrad_simt", s);
  k_wgrad<T, DT, MODE><<<grid, 256, 0, s>>>(
      reinterpret_cast<const DT*>(a.ws + L.off_dA), static_cast<const T*>(a.x),
      static_cast<const T*>(a.h0), static_cast<const T*>(a.h_seq), L.K, L.n_in, L.H, L.R,
      rows_per_split, out);
  return cudaGetLastError();
}

// grad_x[r][i] = sum_m dA[r][m] * W_in[m][i] over the B*K rows r (W_in stacked
// as [3H][n_in], operand-rounded), for the K-loop kernels that leave grad_x
// out of the recurrence.  64 x 64 output tiles, m in chunks of 32 through
// shared memory, 4 x 4 outputs per thread; every output sums m in ascending
// order (deterministic).
constexpr int kGxTile = 64, kGxK = 32;

template <typename T, typename DT, int MODE>
__global__ void __launch_bounds__(256)
k_grad_x_simt(const DT* __restrict__ dA, const T* __restrict__ W_in, long long R, int H3, int n_in,
              float* __restrict__ grad_x) {
  __shared__ float As[kGxK][kGxTile + 1];     // [m][row]
  __shared__ float Bs[kGxK][kGxTile];         // [m][col]
  const long long r0 = (long long)blockIdx.x * kGxTile;
  const int c0 = blockIdx.y * kGxTile;
  const int tid = threadIdx.x, tr = tid / 16, tc = tid % 16;
  float acc[4][4] = {};
  for (int m0 = 0; m0 < H3; m0 += kGxK) {
    for (int e = tid; e < kGxTile * kGxK; e += 256) {
      const int rr = e / kGxK, mm = e - rr * kGxK;
      const long long row = r0 + rr;
      As[mm][rr] = (row < R && m0 + mm < H3) ? ldf(dA + row * H3 + m0 + mm) : 0.f;
    }
    for (int e = tid; e < kGxTile * kGxK; e += 256) {
      const int mm = e / kGxTile, cc = e - mm * kGxTile;
      Bs[mm][cc] = (m0 + mm < H3 && c0 + cc < n_in) ? ld_operand<MODE>(W_in + (long long)(m0 + mm) * n_in + c0 + cc)
                                                      : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int mm = 0; mm < kGxK; ++mm) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = As[mm][tr * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[mm][tc * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long row = r0 + tr * 4 + i;
    if (row >= R) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = c0 + tc * 4 + j;
      if (col < n_in) grad_x[row * n_in + col] = acc[i][j];
    }
  }
}

// Staged form for float dA and W_in (FP32 / TF32) when a 32-row tile of dA and
// a 64-column slice of W_in fit in shared memory together: every copy of the
// block is issued up front with cp.async in four commit groups along m (one
// memory latency instead of one per m chunk), and the products of chunk c run
// while chunks c+1.. are still landing.  32 x 64 outputs per block of 128
// threads, 4 x 4 per thread; every output sums m in ascending order with the
// same fmaf chain as k_grad_x_simt (identical results).
constexpr int kGxsRows = 32, kGxsCols = 64, kGxsThreads = 128, kGxsChunks = 4;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

size_t grad_x_staged_smem(int H3) {
  return sizeof(float) * ((size_t)kGxsRows * (H3 + 4) + (size_t)H3 * kGxsCols);
}

template <int MODE>
__global__ void __launch_bounds__(kGxsThreads)
k_grad_x_staged(const float* __restrict__ dA, const float* __restrict__ W_in, long long R, int H3, int n_in,
                float* __restrict__ grad_x) {
  extern __shared__ __align__(16) float gsm[];
  const int lda = H3 + 4;                        // row stride of the dA tile (16-byte rows)
  float* As = gsm;                               // [32][lda]
  float* Bs = As + (size_t)kGxsRows * lda;       // [H3][64]
  const long long r0 = (long long)blockIdx.x * kGxsRows;
  const int c0 = blockIdx.y * kGxsCols;
  const int tid = threadIdx.x;
  const int nq = H3 / 4;                         // 16-byte units along m (H3 % 4 == 0)

#pragma unroll
  for (int c = 0; c < kGxsChunks; ++c) {
    const int q0 = c * nq / kGxsChunks, q1 = (c + 1) * nq / kGxsChunks, w = q1 - q0;
    for (int e = tid; e < kGxsRows * w; e += kGxsThreads) {
      const int rr = e / w, q = q0 + (e - rr * w);
      const long long row = r0 + rr;
      const bool in = row < R;                   // rows past R are zero-filled
      cp_async16(smem_addr(As + (size_t)rr * lda + 4 * q), dA + (in ? row : 0) * H3 + 4 * q, in ? 16u : 0u);
    }
    for (int e = tid; e < 4 * w * (kGxsCols / 4); e += kGxsThreads) {
      const int m = 4 * q0 + e / (kGxsCols / 4), cq = e % (kGxsCols / 4);
      const int col = c0 + 4 * cq;
      const bool in = col < n_in;                // n_in % 4 == 0: a unit is all in or all out
      cp_async16(smem_addr(Bs + (size_t)m * kGxsCols + 4 * cq), W_in + (long long)m * n_in + (in ? col : 0),
                 in ? 16u : 0u);
    }
    cp_async_commit();
  }

  const int tr = tid / 16, tc = tid % 16;        // rows 4tr..4tr+3, columns 4tc..4tc+3
  float acc[4][4] = {};
  auto products = [&](int c) {
    const int q0 = c * nq / kGxsChunks, q1 = (c + 1) * nq / kGxsChunks;
    for (int q = q0; q < q1; ++q) {
      float a[4][4], b[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 v = *reinterpret_cast<const float4*>(As + (size_t)(4 * tr + i) * lda + 4 * q);
        a[i][0] = v.x; a[i][1] = v.y; a[i][2] = v.z; a[i][3] = v.w;
      }
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const float4 v = *reinterpret_cast<const float4*>(Bs + (size_t)(4 * q + t) * kGxsCols + 4 * tc);
        b[t][0] = to_operand<MODE>(v.x); b[t][1] = to_operand<MODE>(v.y);
        b[t][2] = to_operand<MODE>(v.z); b[t][3] = to_operand<MODE>(v.w);
      }
#pragma unroll
      for (int t = 0; t < 4; ++t)                // m = 4q + t, ascending
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i][t], b[t][j], acc[i][j]);
    }
  };
  static_assert(kGxsChunks == 4, "one wait per commit group");
  cp_async_wait<3>();
  __syncthreads();
  products(0);
  cp_async_wait<2>();
  __syncthreads();
  products(1);
  cp_async_wait<1>();
  __syncthreads();
  products(2);
  cp_async_wait<0>();
  __syncthreads();
  products(3);

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const long long row = r0 + 4 * tr + i;
    if (row >= R) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = c0 + 4 * tc + j;
      if (col < n_in) grad_x[row * n_in + col] = acc[i][j];
    }
  }
}

template <typename T, typename DT, int MODE>
cudaError_t grad_x_mode(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  if constexpr (sizeof(T) == 4 && sizeof(DT) == 4) {
    const float* dA = reinterpret_cast<const float*>(a.ws + L.off_dA);
    const size_t smem = grad_x_staged_smem(L.H3);
    const bool aligned = ((reinterpret_cast<uintptr_t>(dA) | reinterpret_cast<uintptr_t>(a.W_in)) & 15) == 0;
    if (L.H3 % 4 == 0 && L.n_in % 4 == 0 && aligned && smem <= 200 * 1024) {
      auto kern = k_grad_x_staged<MODE>;
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      dim3 grid((unsigned)((L.R + kGxsRows - 1) / kGxsRows), (unsigned)((L.n_in + kGxsCols - 1) / kGxsCols));
      TraceScope trace("grad_x_simt", s);
      kern<<<grid, kGxsThreads, smem, s>>>(dA, static_cast<const float*>(a.W_in), L.R, L.H3, L.n_in, a.grad_x);
      return cudaGetLastError();
    }
  }
  dim3 grid((unsigned)((L.R + kGxTile - 1) / kGxTile), (unsigned)((L.n_in + kGxTile - 1) / kGxTile));
  TraceScope trace("grad_x_simt", s);
  k_grad_x_simt<T, DT, MODE><<<grid, 256, 0, s>>>(reinterpret_cast<const DT*>(a.ws + L.off_dA),
                                                  static_cast<const T*>(a.W_in), L.R, L.H3, L.n_in, a.grad_x);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward_simt(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  switch (L.math) {
    case CFC_MATH_FP32: return forward_mode<float, CFC_MATH_FP32>(L, a, s);
    case CFC_MATH_TF32: return forward_mode<float, CFC_MATH_TF32>(L, a, s);
    default: return forward_mode<__nv_bfloat16, CFC_MATH_BF16>(L, a, s);
  }
}

cudaError_t launch_backward_simt(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  switch (L.math) {
    case CFC_MATH_FP32: return backward_mode<float, float, CFC_MATH_FP32>(L, a, s);
    case CFC_MATH_TF32: return backward_mode<float, float, CFC_MATH_TF32>(L, a, s);
    default: return backward_mode<__nv_bfloat16, __nv_bfloat16, CFC_MATH_BF16>(L, a, s);
  }
}

cudaError_t launch_wgrad_simt(const Layout& L, const CfcArgs& a, float* out, int n_split,
                              long long rows_per_split, cudaStream_t s) {
  switch (L.math) {
    case CFC_MATH_FP32: return wgrad_mode<float, float, CFC_MATH_FP32>(L, a, out, n_split, rows_per_split, s);
    case CFC_MATH_TF32: return wgrad_mode<float, float, CFC_MATH_TF32>(L, a, out, n_split, rows_per_split, s);
    default: return wgrad_mode<__nv_bfloat16, __nv_bfloat16, CFC_MATH_BF16>(L, a, out, n_split, rows_per_split, s);
  }
}

cudaError_t launch_grad_x_simt(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  if (!a.grad_x) return cudaSuccess;
  switch (L.math) {
    case CFC_MATH_FP32: return grad_x_mode<float, float, CFC_MATH_FP32>(L, a, s);
    case CFC_MATH_TF32: return grad_x_mode<float, float, CFC_MATH_TF32>(L, a, s);
    default: return grad_x_mode<__nv_bfloat16, __nv_bfloat16, CFC_MATH_BF16>(L, a, s);
  }
}

}  // namespace cfc
