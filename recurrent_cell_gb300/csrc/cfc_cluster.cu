// cfc_cluster.cu -- K-loop forward/backward with the weights resident in the
// shared memory of a thread-block cluster.
//
// A cluster of C blocks owns a tile of BT samples for the whole K loop.
//
// Forward: block r of the cluster owns hidden units [r*Hc, (r+1)*Hc)
// (Hc = H / C) and keeps the rows of W_cat = [W_in | W_rec] of those units
// (all three heads) in shared memory, [3][Hc][ldw]: a unit's row is
// contiguous (16-byte reads of four columns) and the row stride
// ldw = 4 (mod 8) floats puts eight consecutive units' 16-byte reads on
// distinct bank groups.  Each step it computes the three
// pre-activations of its units (the Zc-long dot products split over S thread
// groups, summed in a fixed order), applies the cell, and writes its slice of
// h_{k+1} into the next operand buffer of EVERY block of the cluster
// (distributed shared memory).  One cluster barrier per step publishes the
// slices; the operand buffer is double-buffered so that no second barrier is
// needed.
//
// Backward: block r owns the same units for the elementwise dA and the
// matching columns of the carry W_rec^T dA (the carry of its own units, which
// it needs next step).  It keeps those columns of W_rec in shared memory,
// [3H][Hc].  Each step it computes dA of its units, broadcasts it to every
// block of the cluster (distributed shared memory, double-buffered), and after
// the cluster barrier contracts the full dA vector with its columns.  grad_x =
// dA W_in does not feed the recurrence and is one GEMM after the loop.
//
// Every kernel here reads the weights from HBM once per block per launch; the
// K loop runs on chip.  No spin waits: the only synchronisation is the
// hardware cluster barrier (barrier.cluster via cooperative groups).
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <cooperative_groups.h>

#include "cfc_internal.cuh"

namespace cg = cooperative_groups;

namespace cfc {
namespace {

// Threads a block and thread groups a dot product is split over: the
// backward's contraction gains from 16 groups on 512 threads, the forward
// measured slower so (its cell adds the groups' partial sums).
constexpr int kFwdClusterThreads = 256, kBwdClusterThreads = 512;
constexpr int kXPerThread = 8;     // forward: x elements per thread prefetched one step ahead
// (sample, unit) items per thread kept in registers, by samples per cluster.
__host__ __device__ constexpr int items_per_thread(int bt) { return bt <= 4 ? 2 : (bt <= 8 ? 4 : 8); }
constexpr int kFwdMaxSplit = 8, kBwdMaxSplit = 16;
// Row stride (floats) of the forward's weight rows: Zc rounded up to 8, + 4.
__host__ __device__ constexpr int fwd_ldw(int Zc) { return (Zc + 7) / 8 * 8 + 4; }

struct ClusterPlan {
  int C = 0, BT = 0, S = 0, threads = 0;
  size_t smem = 0;
};

// ---------------------------------------------------------------------------
// Forward
// ---------------------------------------------------------------------------
template <typename T, int MODE, int BT>
__global__ void __launch_bounds__(kFwdClusterThreads)
k_cfc_fwd_cluster(const T* __restrict__ x, const T* __restrict__ h0, const T* __restrict__ W_in,
                  const T* __restrict__ W_rec, const float* __restrict__ bias,
                  const float* __restrict__ dt, int dt_stride, int B, int K, int n_in, int H, int S,
                  T* __restrict__ h_seq, float* __restrict__ act) {
  constexpr int kItemsPerThread = items_per_thread(BT);
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int r = (int)cluster.block_rank();
  const int Hc = H / C, Zc = n_in + H, H3 = 3 * H;
  const int b0 = (int)(blockIdx.x / C) * BT;
  const int tid = threadIdx.x, nthr = blockDim.x;

  const int ldw = fwd_ldw(Zc);
  extern __shared__ float sm[];
  float* Ws = sm;                              // [3][Hc][ldw] operand values
  float* zb = Ws + (size_t)3 * Hc * ldw;       // [2][BT][Zc]
  float* part = zb + 2 * BT * Zc;              // [S][BT][3][Hc]
  float* bs = part + (size_t)S * BT * 3 * Hc;  // [3][Hc] bias of the owned units
  float* dts = bs + 3 * Hc;                    // [BT] dt of the tile's samples

  for (int e = tid; e < 3 * Hc * Zc; e += nthr) {
    const int cu = e / Zc, j = e - cu * Zc, c = cu / Hc, u = cu - c * Hc;
    const long long row = (long long)c * H + r * Hc + u;
    Ws[(size_t)cu * ldw + j] = (j < n_in) ? ld_operand<MODE>(W_in + row * n_in + j)
                                          : ld_operand<MODE>(W_rec + row * H + (j - n_in));
  }
  for (int e = tid; e < BT * Zc; e += nthr) {
    const int n = e / Zc, j = e - n * Zc, bb = b0 + n;
    float v = 0.f;
    if (bb < B) v = (j < n_in) ? ld_operand<MODE>(x + (long long)bb * K * n_in + j)
                               : ld_operand<MODE>(h0 + (long long)bb * H + (j - n_in));
    zb[e] = v;
  }
  for (int e = tid; e < 3 * Hc; e += nthr) bs[e] = bias[(e / Hc) * H + r * Hc + (e % Hc)];
  for (int e = tid; e < BT; e += nthr) dts[e] = (b0 + e < B) ? dt[dt_stride ? b0 + e : 0] : 0.f;

  // x of the next step, loaded one step ahead so that its latency overlaps
  // the current step (the plan guarantees BT*n_in <= kXPerThread * threads).
  float xr[kXPerThread];
  auto load_x = [&](int kk) {
#pragma unroll
    for (int q = 0; q < kXPerThread; ++q) {
      const int e = tid + q * nthr;
      const int n = e / n_in, j = e - n * n_in, bb = b0 + n;
      xr[q] = (e < BT * n_in && kk < K && bb < B)
                  ? ld_operand<MODE>(x + ((long long)bb * K + kk) * n_in + j) : 0.f;
    }
  };
  load_x(1);
  // Every block of the cluster must be running before any block writes into
  // its shared memory.
  cluster.sync();

  uint32_t peer_zb[8];                // shared::cluster address of zb in every block
#pragma unroll
  for (int p = 0; p < 8; ++p) peer_zb[p] = (p < C) ? dsmem_map(smem_addr(zb), (uint32_t)p) : 0u;

  // thread -> (unit u, column group s) of the dot products; with Zc a
  // multiple of 4 the groups are whole 4-column quads (16-byte reads)
  const int u = tid % Hc, s = tid / Hc;
  const bool dot = s < S;
  const bool quads = (Zc & 3) == 0;
  const int nq = Zc / 4;
  const int j0 = quads ? 4 * (int)((long long)s * nq / S) : (int)((long long)s * Zc / S);
  const int j1 = quads ? 4 * (int)((long long)(s + 1) * nq / S) : (int)((long long)(s + 1) * Zc / S);
  const float* wrow0 = Ws + (size_t)u * ldw;             // head f, unit u
  const float* wrow1 = wrow0 + (size_t)Hc * ldw;          // head g
  const float* wrow2 = wrow1 + (size_t)Hc * ldw;          // head h~

  for (int k = 0; k < K; ++k) {
    const float* zs = zb + (k & 1) * BT * Zc;
    float* zn = zb + ((k + 1) & 1) * BT * Zc;
    if (dot) {
      float a0[BT], a1[BT], a2[BT];
#pragma unroll
      for (int n = 0; n < BT; ++n) { a0[n] = 0.f; a1[n] = 0.f; a2[n] = 0.f; }
      if (quads) {
        // four columns a read, added in ascending column order
#pragma unroll 2
        for (int j = j0; j < j1; j += 4) {
          const float4 wf = *reinterpret_cast<const float4*>(wrow0 + j);
          const float4 wg = *reinterpret_cast<const float4*>(wrow1 + j);
          const float4 wh = *reinterpret_cast<const float4*>(wrow2 + j);
#pragma unroll
          for (int n = 0; n < BT; ++n) {
            const float4 z = *reinterpret_cast<const float4*>(zs + n * Zc + j);
            a0[n] = fmaf(wf.x, z.x, a0[n]); a0[n] = fmaf(wf.y, z.y, a0[n]);
            a0[n] = fmaf(wf.z, z.z, a0[n]); a0[n] = fmaf(wf.w, z.w, a0[n]);
            a1[n] = fmaf(wg.x, z.x, a1[n]); a1[n] = fmaf(wg.y, z.y, a1[n]);
            a1[n] = fmaf(wg.z, z.z, a1[n]); a1[n] = fmaf(wg.w, z.w, a1[n]);
            a2[n] = fmaf(wh.x, z.x, a2[n]); a2[n] = fmaf(wh.y, z.y, a2[n]);
            a2[n] = fmaf(wh.z, z.z, a2[n]); a2[n] = fmaf(wh.w, z.w, a2[n]);
          }
        }
      } else {
#pragma unroll 4
        for (int j = j0; j < j1; ++j) {
          const float wf = wrow0[j], wg = wrow1[j], wh = wrow2[j];
#pragma unroll
          for (int n = 0; n < BT; ++n) {
            const float z = zs[n * Zc + j];
            a0[n] = fmaf(wf, z, a0[n]);
            a1[n] = fmaf(wg, z, a1[n]);
            a2[n] = fmaf(wh, z, a2[n]);
          }
        }
      }
#pragma unroll
      for (int n = 0; n < BT; ++n) {
        float* p = part + ((size_t)(s * BT + n) * 3) * Hc + u;
        p[0] = a0[n];
        p[Hc] = a1[n];
        p[2 * Hc] = a2[n];
      }
    }
    if (k + 1 < K) {
#pragma unroll
      for (int q = 0; q < kXPerThread; ++q) {
        const int e = tid + q * nthr;
        if (e < BT * n_in) zn[(e / n_in) * Zc + (e % n_in)] = xr[q];
      }
    }
    __syncthreads();
    // Cell of (sample n, unit u) pairs; partial sums added in the fixed order
    // s = 0..S-1.  Results stay in registers until after the barrier arrive.
    float rg[kItemsPerThread], rgg[kItemsPerThread], rhh[kItemsPerThread], rh[kItemsPerThread];
#pragma unroll
    for (int it = 0; it < kItemsPerThread; ++it) {
      const int e = tid + it * nthr;
      if (e >= BT * Hc) break;
      const int n = e / Hc, uu = e - n * Hc, bb = b0 + n;
      const int unit = r * Hc + uu;
      float A[3];
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        float pv[kFwdMaxSplit];
#pragma unroll
        for (int q = 0; q < kFwdMaxSplit; ++q)
          pv[q] = (q < S) ? part[((size_t)(q * BT + n) * 3 + c) * Hc + uu] : 0.f;
        float v = bs[c * Hc + uu];
#pragma unroll
        for (int q = 0; q < kFwdMaxSplit; ++q)
          if (q < S) v += pv[q];
        A[c] = v;
      }
      const float g = tanhf(A[1]);
      const float hh = tanhf(A[2]);
      const float gate = 1.f / (1.f + expf(A[0] * dts[n]));
      const float h = gate * g + (1.f - gate) * hh;
      rg[it] = gate; rgg[it] = g; rhh[it] = hh; rh[it] = h;
      float hop = 0.f;
      if (bb < B) {
        if constexpr (sizeof(T) == 2) hop = round_bf16(h);   // the stored bf16 state
        else hop = to_operand<MODE>(h);
      }
      const uint32_t off = (uint32_t)((((k + 1) & 1) * BT * Zc + n * Zc + n_in + unit) * 4);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < C) dsmem_st(peer_zb[q] + off, hop);
    }
    cluster_arrive_release();
    // x of step k+2, issued after the arrive: a release waits for the
    // thread's outstanding loads too
    if (k + 1 < K) load_x(k + 2);
#pragma unroll
    for (int it = 0; it < kItemsPerThread; ++it) {
      const int e = tid + it * nthr;
      if (e >= BT * Hc) break;
      const int n = e / Hc, uu = e - n * Hc, bb = b0 + n;
      if (bb < B) {
        const int unit = r * Hc + uu;
        const long long row = (long long)bb * K + k;
        act[row * H3 + unit] = rg[it];
        act[row * H3 + H + unit] = rgg[it];
        act[row * H3 + 2 * H + unit] = rhh[it];
        stf(h_seq + row * H + unit, rh[it]);
      }
    }
    cluster_wait_acquire();
  }
}

// ---------------------------------------------------------------------------
// Backward
// ---------------------------------------------------------------------------
template <typename T, typename DT, int MODE, int BT>
__global__ void __launch_bounds__(kBwdClusterThreads)
k_cfc_bwd_cluster(const T* __restrict__ W_in, const T* __restrict__ W_rec,
                  const float* __restrict__ dt, int dt_stride, int B, int K, int n_in, int H, int S,
                  const T* __restrict__ h_seq, const float* __restrict__ grad_h_seq,
                  const float* __restrict__ grad_h_last, const float* __restrict__ y,
                  const float* __restrict__ act, DT* __restrict__ dA_out,
                  float* __restrict__ grad_h0) {
  constexpr int kItemsPerThread = items_per_thread(BT);
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int r = (int)cluster.block_rank();
  const int Hc = H / C, H3 = 3 * H;
  const int nJ = Hc, nJmax = Hc;
  const int b0 = (int)(blockIdx.x / C) * BT;
  const int tid = threadIdx.x, nthr = blockDim.x;

  const int H3p = (H3 + 3) & ~3;                // dA row length, zero-padded
  const int ldw = (H3p % 8 == 0) ? H3p + 4 : H3p;  // weight row stride (ldw/4 odd)
  extern __shared__ float sm[];
  float* Wc = sm;                              // [Hc][ldw]: W_rec columns owned here, transposed
  float* dAf = Wc + (size_t)Hc * ldw;          // [2][BT][H3p] dA of all units (operand values)
  float* part = dAf + 2 * BT * H3p;            // [S][BT][nJmax] partial column sums
  float* dts = part + (size_t)S * BT * nJmax;  // [BT]

  for (int e = tid; e < Hc * ldw; e += nthr) {
    const int jj = e / ldw, row = e - jj * ldw;
    Wc[e] = (row < H3) ? ld_operand<MODE>(W_rec + (long long)row * H + r * Hc + jj) : 0.f;
  }
  for (int e = tid; e < 2 * BT * H3p; e += nthr) dAf[e] = 0.f;   // padding stays zero
  for (int e = tid; e < BT; e += nthr) dts[e] = (b0 + e < B) ? dt[dt_stride ? b0 + e : 0] : 0.f;
  cluster.sync();

  uint32_t peer_dA[8];                // shared::cluster address of dAf in every block
#pragma unroll
  for (int p = 0; p < 8; ++p) peer_dA[p] = (p < C) ? dsmem_map(smem_addr(dAf), (uint32_t)p) : 0u;
  const int jj = tid % nJmax, s = tid / nJmax;
  const bool dot = (s < S) && (jj < nJ);
  const int nq = H3p / 4;
  const int q0 = (int)((long long)s * nq / S), q1 = (int)((long long)(s + 1) * nq / S);
  const float4* wc4 = reinterpret_cast<const float4*>(Wc + (size_t)jj * ldw);

  // Saved activations (and per-step upstream gradient) of this thread's
  // (sample, unit) items, loaded one step ahead (the plan guarantees
  // BT*Hc <= kItemsPerThread * threads).
  float pg[kItemsPerThread], pgg[kItemsPerThread], phh[kItemsPerThread], pup[kItemsPerThread];
  auto load_act = [&](int kk) {
#pragma unroll
    for (int q = 0; q < kItemsPerThread; ++q) {
      const int e = tid + q * nthr;
      const int n = e / Hc, uu = e - n * Hc, bb = b0 + n, unit = r * Hc + uu;
      pg[q] = pgg[q] = phh[q] = pup[q] = 0.f;
      if (e < BT * Hc && kk >= 0 && bb < B) {
        const long long row = (long long)bb * K + kk;
        pg[q] = act[row * H3 + unit];
        pgg[q] = act[row * H3 + H + unit];
        phh[q] = act[row * H3 + 2 * H + unit];
        if (grad_h_seq) pup[q] = grad_h_seq[row * H + unit];
      }
    }
  };
  load_act(K - 1);

  // Sum of the S partial column sums of the previous contraction (fixed order).
  auto column_sum = [&](int n, int c) {
    float pv[kBwdMaxSplit];
#pragma unroll
    for (int q = 0; q < kBwdMaxSplit; ++q) pv[q] = (q < S) ? part[(size_t)(q * BT + n) * nJmax + c] : 0.f;
    float v = 0.f;
#pragma unroll
    for (int q = 0; q < kBwdMaxSplit; ++q)
      if (q < S) v += pv[q];
    return v;
  };
  // Per step: (A) dA of the owned units from the previous step's carry
  // (summed from part), broadcast to every block; cluster barrier; (B)
  // contract the full dA with the owned columns into part; block barrier.
  for (int k = K - 1; k >= 0; --k) {
    float* buf = dAf + (k & 1) * BT * H3p;
    float cg_[kItemsPerThread], cgg[kItemsPerThread], chh[kItemsPerThread], cup[kItemsPerThread];
#pragma unroll
    for (int q = 0; q < kItemsPerThread; ++q) { cg_[q] = pg[q]; cgg[q] = pgg[q]; chh[q] = phh[q]; cup[q] = pup[q]; }
    float rd0[kItemsPerThread], rd1[kItemsPerThread], rd2[kItemsPerThread];
#pragma unroll
    for (int q = 0; q < kItemsPerThread; ++q) {
      const int e = tid + q * nthr;
      if (e >= BT * Hc) break;
      const int n = e / Hc, u = e - n * Hc, bb = b0 + n;
      const int unit = r * Hc + u;
      float d0 = 0.f, d1 = 0.f, d2 = 0.f;
      if (bb < B) {
        const long long row = (long long)bb * K + k;
        float delta = ((k < K - 1) ? column_sum(n, u) : 0.f) + cup[q];
        if (k == K - 1) {
          if (grad_h_last) delta += grad_h_last[(long long)bb * H + unit];
          if (y) delta += ldf(h_seq + row * H + unit) - y[(long long)bb * H + unit];
        }
        const float gate = cg_[q], g = cgg[q], hh = chh[q];
        d1 = to_operand<MODE>(delta * gate * (1.f - g * g));
        d2 = to_operand<MODE>(delta * (1.f - gate) * (1.f - hh * hh));
        d0 = to_operand<MODE>(-dts[n] * delta * (g - hh) * gate * (1.f - gate));
      }
      rd0[q] = d0; rd1[q] = d1; rd2[q] = d2;
      const uint32_t off = (uint32_t)(((k & 1) * BT * H3p + n * H3p + unit) * 4);
#pragma unroll
      for (int q2 = 0; q2 < 8; ++q2) {
        if (q2 < C) {
          dsmem_st(peer_dA[q2] + off, d0);
          dsmem_st(peer_dA[q2] + off + 4 * H, d1);
          dsmem_st(peer_dA[q2] + off + 8 * H, d2);
        }
      }
    }
    cluster_arrive_release();
    // activations of step k-1, issued after the arrive: a release waits for
    // the thread's outstanding loads too
    load_act(k - 1);
#pragma unroll
    for (int q = 0; q < kItemsPerThread; ++q) {
      const int e = tid + q * nthr;
      if (e >= BT * Hc) break;
      const int n = e / Hc, u = e - n * Hc, bb = b0 + n;
      if (bb < B) {
        const int unit = r * Hc + u;
        const long long row = (long long)bb * K + k;
        stf(dA_out + row * H3 + unit, rd0[q]);
        stf(dA_out + row * H3 + H + unit, rd1[q]);
        stf(dA_out + row * H3 + 2 * H + unit, rd2[q]);
      }
    }
    cluster_wait_acquire();
    if (dot) {
      // two interleaved accumulator chains (even / odd rows), added at the end
      float acc0[BT], acc1[BT];
#pragma unroll
      for (int n = 0; n < BT; ++n) { acc0[n] = 0.f; acc1[n] = 0.f; }
      constexpr int kUnroll = BT <= 4 ? 2 : 1;   // larger tiles: registers go to the BT chains
#pragma unroll(kUnroll)
      for (int q = q0; q < q1; ++q) {
        const float4 w = wc4[q];
#pragma unroll
        for (int n = 0; n < BT; ++n) {
          const float4 d = reinterpret_cast<const float4*>(buf + n * H3p)[q];
          acc0[n] = fmaf(w.x, d.x, acc0[n]);
          acc1[n] = fmaf(w.y, d.y, acc1[n]);
          acc0[n] = fmaf(w.z, d.z, acc0[n]);
          acc1[n] = fmaf(w.w, d.w, acc1[n]);
        }
      }
#pragma unroll
      for (int n = 0; n < BT; ++n) part[(size_t)(s * BT + n) * nJmax + jj] = acc0[n] + acc1[n];
    }
    __syncthreads();
  }
  if (grad_h0) {
    for (int e = tid; e < BT * Hc; e += nthr) {
      const int n = e / Hc, u = e - n * Hc, bb = b0 + n;
      const float v = column_sum(n, u);
      if (bb < B) grad_h0[(long long)bb * H + r * Hc + u] = v;
    }
  }
}

// ---------------------------------------------------------------------------
// Planning and launch
// ---------------------------------------------------------------------------
constexpr size_t kSmemLimit = 200 * 1024;

size_t fwd_smem(const Layout& L, int C, int BT, int S) {
  const int Hc = L.H / C;
  return sizeof(float) * ((size_t)3 * Hc * fwd_ldw(L.Zc) + 2 * (size_t)BT * L.Zc + (size_t)S * BT * 3 * Hc +
                          3 * (size_t)Hc + BT);
}

size_t bwd_smem(const Layout& L, int C, int BT, int S) {
  const int Hc = L.H / C;
  const int nJmax = Hc;
  const int H3p = (L.H3 + 3) & ~3, ldw = (H3p % 8 == 0) ? H3p + 4 : H3p;
  return sizeof(float) * ((size_t)Hc * ldw + 2 * (size_t)BT * H3p + (size_t)S * BT * nJmax + BT);
}

// Cluster size from the hidden size alone (so a sample's arithmetic does not
// depend on the batch size): about 32 units per block, i.e. the smallest C in
// {1, 2, 4, 8} with C >= H/32 that divides H and whose slices fit; failing
// that, the largest C that fits.  Samples per cluster: the smallest BT that
// keeps the grid within about two blocks per SM.
bool plan(const Layout& L, bool forward, ClusterPlan* p) {
  const int Cs[4] = {1, 2, 4, 8};
  const int max_threads = forward ? kFwdClusterThreads : kBwdClusterThreads;
  const int max_split = forward ? kFwdMaxSplit : kBwdMaxSplit;
  auto valid = [&](int c) {
    if (L.H % c) return false;
    const int Hc = L.H / c;
    if (Hc > max_threads) return false;
    return (forward ? fwd_smem(L, c, 1, 1) : bwd_smem(L, c, 1, 1)) <= kSmemLimit;
  };
  const int target = (L.H + 31) / 32;
  int C = 0, largest = 0;
  for (int c : Cs) {
    if (!valid(c)) continue;
    largest = c;
    if (!C && c >= target) C = c;
  }
  if (!C) C = largest;
  if (!C) return false;
  const int Hc = L.H / C;
  const int width = Hc;
  const int S = std::max(1, std::min(max_split, max_threads / width));
  const int threads = std::min(max_threads, (width * S + 31) / 32 * 32);
  auto smem = [&](int bt) { return forward ? fwd_smem(L, C, bt, S) : bwd_smem(L, C, bt, S); };
  auto fits = [&](int bt) {
    const long long items = forward ? (long long)bt * L.n_in : (long long)bt * Hc;
    const int per = forward ? kXPerThread : items_per_thread(bt);
    return smem(bt) <= kSmemLimit && items <= (long long)per * threads &&
           (long long)bt * Hc <= (long long)items_per_thread(bt) * threads;
  };
  // Samples per cluster: the smallest BT whose grid fits in one wave (blocks
  // per SM from the shared-memory size); else the largest that fits.
  const int bts[6] = {1, 2, 4, 8, 16, 32};
  const int nbt = forward ? 5 : 6;
  int BT = 0;
  for (int i = 0; i < nbt; ++i) {
    const int t = bts[i];
    if (!fits(t)) break;
    BT = t;
    const long long per_sm = std::max<long long>(1, (long long)(227 * 1024) / (long long)smem(t));
    if ((long long)(L.B + t - 1) / t * C <= per_sm * kNumSMs) break;
  }
  if (!BT) return false;
  p->C = C;
  p->BT = BT;
  p->S = S;
  p->threads = threads;
  p->smem = smem(BT);
  return true;
}

template <typename Kern, typename... Args>
cudaError_t launch_cluster(Kern kern, const ClusterPlan& p, int B, cudaStream_t s, Args... args) {
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(((B + p.BT - 1) / p.BT) * p.C), 1, 1);
  cfg.blockDim = dim3((unsigned)p.threads, 1, 1);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename T, int MODE, int BT>
cudaError_t fwd_bt(const Layout& L, const ClusterPlan& p, const CfcArgs& a, cudaStream_t s) {
  TraceScope trace("cfc_fwd_cluster", s);
  return launch_cluster(k_cfc_fwd_cluster<T, MODE, BT>, p, L.B, s,
                        static_cast<const T*>(a.x), static_cast<const T*>(a.h0),
                        static_cast<const T*>(a.W_in), static_cast<const T*>(a.W_rec), a.b, a.dt,
                        a.dt_stride, L.B, L.K, L.n_in, L.H, p.S, static_cast<T*>(a.h_seq),
                        reinterpret_cast<float*>(a.ws + L.off_act));
}

template <typename T, typename DT, int MODE, int BT>
cudaError_t bwd_bt(const Layout& L, const ClusterPlan& p, const CfcArgs& a, cudaStream_t s) {
  cudaError_t e;
  {
    TraceScope trace("cfc_bwd_cluster", s);
    e = launch_cluster(k_cfc_bwd_cluster<T, DT, MODE, BT>, p, L.B, s,
                       static_cast<const T*>(a.W_in), static_cast<const T*>(a.W_rec), a.dt,
                       a.dt_stride, L.B, L.K, L.n_in, L.H, p.S, static_cast<const T*>(a.h_seq),
                       a.grad_h_seq, a.grad_h_last, a.y,
                       reinterpret_cast<const float*>(a.ws + L.off_act),
                       reinterpret_cast<DT*>(a.ws + L.off_dA), a.grad_h0);
  }
  if (e != cudaSuccess) return e;
  return launch_grad_x_simt(L, a, s);
}

template <typename T, int MODE>
cudaError_t fwd_mode(const Layout& L, const ClusterPlan& p, const CfcArgs& a, cudaStream_t s) {
  switch (p.BT) {
    case 1: return fwd_bt<T, MODE, 1>(L, p, a, s);
    case 2: return fwd_bt<T, MODE, 2>(L, p, a, s);
    case 4: return fwd_bt<T, MODE, 4>(L, p, a, s);
    case 8: return fwd_bt<T, MODE, 8>(L, p, a, s);
    default: return fwd_bt<T, MODE, 16>(L, p, a, s);
  }
}

template <typename T, typename DT, int MODE>
cudaError_t bwd_mode(const Layout& L, const ClusterPlan& p, const CfcArgs& a, cudaStream_t s) {
  switch (p.BT) {
    case 1: return bwd_bt<T, DT, MODE, 1>(L, p, a, s);
    case 2: return bwd_bt<T, DT, MODE, 2>(L, p, a, s);
    case 4: return bwd_bt<T, DT, MODE, 4>(L, p, a, s);
    case 8: return bwd_bt<T, DT, MODE, 8>(L, p, a, s);
    case 16: return bwd_bt<T, DT, MODE, 16>(L, p, a, s);
    default: return bwd_bt<T, DT, MODE, 32>(L, p, a, s);
  }
}

}  // namespace

namespace {
bool use_cluster(const Layout& L, bool forward, ClusterPlan* p) {
  const int choice = kernel_choice();
  if (choice == kSimt || choice == kTc || choice == kTcStream || !plan(L, forward, p)) return false;
  if (choice == kCluster) return true;
  return (long long)(L.B + p->BT - 1) / p->BT * p->C <= 2 * kNumSMs;
}
}  // namespace

cudaError_t launch_forward_cluster(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  ClusterPlan p;
  if (!use_cluster(L, true, &p)) return cudaErrorNotSupported;
  switch (L.math) {
    case CFC_MATH_FP32: return fwd_mode<float, CFC_MATH_FP32>(L, p, a, s);
    case CFC_MATH_TF32: return fwd_mode<float, CFC_MATH_TF32>(L, p, a, s);
    default: return fwd_mode<__nv_bfloat16, CFC_MATH_BF16>(L, p, a, s);
  }
}

cudaError_t launch_backward_cluster(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  ClusterPlan p;
  if (!use_cluster(L, false, &p)) return cudaErrorNotSupported;
  switch (L.math) {
    case CFC_MATH_FP32: return bwd_mode<float, float, CFC_MATH_FP32>(L, p, a, s);
    case CFC_MATH_TF32: return bwd_mode<float, float, CFC_MATH_TF32>(L, p, a, s);
    default: return bwd_mode<__nv_bfloat16, __nv_bfloat16, CFC_MATH_BF16>(L, p, a, s);
  }
}

}  // namespace cfc
