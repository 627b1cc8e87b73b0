// cfc_tc_kloop.cu -- forward K loop of the TF32 / bf16 modes on the tcgen05
// tensor cores.
//
// A cluster of C = H/32 blocks owns a tile of Bt samples for the whole K loop;
// block r owns hidden units [32r, 32r+32).  Per step the block computes
//
//   D[128 x Bt] = Wr[128 x Zc] * Z^T          (one M=128, N=Bt MMA chain)
//
// where Wr stacks the W_cat = [W_in | W_rec] rows of its units for the three
// heads (rows 0-31 f, 32-63 g, 64-95 h~, 96-127 zero) and Z holds the operand
// rows z_n = [x_k; h_k] of the Bt samples.  Wr stays in shared memory for the
// whole launch (K-major, 128B-swizzled, 96 KB for Zc*element = 768 B).  Z is
// double-buffered: while step k reads Z[k&1], every block writes its slice of
// h_{k+1} (32 units x Bt samples) into Z[(k+1)&1] of every block of the cluster
// through distributed shared memory, and x_{k+1} (prefetched into registers)
// locally.  One cluster barrier per step publishes the slices.
//
// Epilogue per step: warps w and w+4 read TMEM lane quadrant w (w = 0, 1, 2:
// the f, g, h~ rows) with tcgen05.ld, stage the pre-activations in padded
// shared memory, and all threads apply the cell to (unit, sample) items.
//
// The MMA waits are bounded; a timeout records an error in the device error
// word and the launch keeps its barrier schedule so that no block of the
// cluster is left waiting.
#include <algorithm>
#include <cooperative_groups.h>

#include "cfc_internal.cuh"
#include "tc_common.cuh"

namespace cg = cooperative_groups;

namespace cfc {

namespace {

constexpr int kThreads = 256;
constexpr int kUnits = 32;                 // hidden units per block
constexpr uint32_t kMaxPolls = 1u << 24;
constexpr size_t kSmemMax = 227 * 1024;
constexpr int kXRegs = 32;                 // prefetched x values per thread (scalar path)
constexpr int kXUnits = 4;                 // prefetched 16-byte x units per thread

__device__ int g_tc_kloop_error = 0;

struct TcPlan {
  int C = 0, Bt = 0, nA = 0;
  size_t smem = 0, off_z = 0, off_ex = 0, off_bs = 0, off_dt = 0;
  uint32_t tmem_cols = 0;
};

template <typename ET>
__device__ __forceinline__ void st_elem(uint8_t* p, float v) {
  if constexpr (sizeof(ET) == 4) *reinterpret_cast<float*>(p) = v;
  else *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
}

// 16 bytes of consecutive K elements starting at p (4 fp32 or 8 bf16), with
// the mode's operand rounding, as a 16-byte swizzle unit.
template <int MODE>
__device__ __forceinline__ uint4 round_unit(uint4 u) {
  if constexpr (MODE == CFC_MATH_TF32) {
    u.x = __float_as_uint(round_tf32(__uint_as_float(u.x)));
    u.y = __float_as_uint(round_tf32(__uint_as_float(u.y)));
    u.z = __float_as_uint(round_tf32(__uint_as_float(u.z)));
    u.w = __float_as_uint(round_tf32(__uint_as_float(u.w)));
  }
  return u;
}
template <typename ET, int MODE>
__device__ __forceinline__ uint4 load_unit(const ET* p) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  if constexpr (MODE == CFC_MATH_TF32) {
    u.x = __float_as_uint(round_tf32(__uint_as_float(u.x)));
    u.y = __float_as_uint(round_tf32(__uint_as_float(u.y)));
    u.z = __float_as_uint(round_tf32(__uint_as_float(u.z)));
    u.w = __float_as_uint(round_tf32(__uint_as_float(u.w)));
  }
  return u;
}

// Byte offset of operand element (row, kk) in a stack of K atoms of `rows` rows.
template <typename ET>
__device__ __forceinline__ uint32_t kmajor_off(int row, int kk, int rows) {
  const uint32_t kb = (uint32_t)kk * sizeof(ET);
  return (kb >> 7) * (uint32_t)rows * 128u + tc::sw128_offset(row, kb & 127u);
}

template <typename ET, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
k_cfc_fwd_tc(const ET* __restrict__ x, const ET* __restrict__ h0, const ET* __restrict__ W_in,
             const ET* __restrict__ W_rec, const float* __restrict__ bias, const float* __restrict__ dt,
             int dt_stride, int B, int K, int n_in, int H, int Bt, int nA, uint32_t off_z,
             uint32_t off_ex, uint32_t off_bs, uint32_t off_dt, uint32_t tmem_cols,
             ET* __restrict__ h_seq, float* __restrict__ act) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int r = (int)cluster.block_rank();
  const int Zc = n_in + H, H3 = 3 * H;
  const int Kpad = nA * (128 / (int)sizeof(ET));
  const int b0 = (int)(blockIdx.x / C) * Bt;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ex_ld = Bt + 1;

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* Ws = sm;                                  // nA x [128 rows][128 B]
  uint8_t* Zs = sm + off_z;                          // 2 x nA x [Bt rows][128 B]
  float* ex = reinterpret_cast<float*>(sm + off_ex); // [3][32][Bt+1]
  float* bs = reinterpret_cast<float*>(sm + off_bs); // [3][32]
  float* dts = reinterpret_cast<float*>(sm + off_dt);// [Bt]
  const uint32_t zbuf_bytes = (uint32_t)nA * Bt * 128;
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int err;

  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, tmem_cols);

  // Resident A operand: rows (head c, unit u) of W_cat, zero rows 96..127 and
  // zero K padding.  vec: n_in and H are multiples of one 16-byte unit, so a
  // unit never straddles W_in / W_rec or x / h and is 16-byte aligned.
  constexpr int EPU = 16 / (int)sizeof(ET);        // elements per 16-byte unit
  const bool vec = (n_in % EPU == 0) && (H % EPU == 0);
  const int upr = Kpad / EPU;                      // units per row
  if (vec) {
    for (int e = tid; e < 128 * upr; e += kThreads) {
      const int i = e / upr, kk = (e - i * upr) * EPU;
      const int c = i >> 5, u = i & 31;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (c < 3 && kk < Zc) {
        const long long row = (long long)c * H + r * kUnits + u;
        v = (kk < n_in) ? load_unit<ET, MODE>(W_in + row * n_in + kk)
                        : load_unit<ET, MODE>(W_rec + row * H + (kk - n_in));
      }
      *reinterpret_cast<uint4*>(Ws + kmajor_off<ET>(i, kk, 128)) = v;
    }
    for (int e = tid; e < Bt * upr; e += kThreads) {
      const int n = e / upr, kk = (e - n * upr) * EPU, bb = b0 + n;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (bb < B && kk < Zc)
        v = (kk < n_in) ? load_unit<ET, MODE>(x + (long long)bb * K * n_in + kk)
                        : load_unit<ET, MODE>(h0 + (long long)bb * H + (kk - n_in));
      *reinterpret_cast<uint4*>(Zs + kmajor_off<ET>(n, kk, Bt)) = v;
    }
  } else {
    for (int e = tid; e < 128 * Kpad; e += kThreads) {
      const int i = e / Kpad, kk = e - i * Kpad;
      const int c = i >> 5, u = i & 31;
      float v = 0.f;
      if (c < 3 && kk < Zc) {
        const long long row = (long long)c * H + r * kUnits + u;
        v = (kk < n_in) ? ld_operand<MODE>(W_in + row * n_in + kk)
                        : ld_operand<MODE>(W_rec + row * H + (kk - n_in));
      }
      st_elem<ET>(Ws + kmajor_off<ET>(i, kk, 128), v);
    }
    // Operand rows of step 0: z_n = [x_0; h0], zero padding.
    for (int e = tid; e < Bt * Kpad; e += kThreads) {
      const int n = e / Kpad, kk = e - n * Kpad, bb = b0 + n;
      float v = 0.f;
      if (bb < B && kk < Zc)
        v = (kk < n_in) ? ld_operand<MODE>(x + (long long)bb * K * n_in + kk)
                        : ld_operand<MODE>(h0 + (long long)bb * H + (kk - n_in));
      st_elem<ET>(Zs + kmajor_off<ET>(n, kk, Bt), v);
    }
  }
  // The second buffer's padding columns stay zero for the whole launch.
  for (int e = tid; e < Bt * Kpad; e += kThreads) {
    const int n = e / Kpad, kk = e - n * Kpad;
    if (kk >= Zc) st_elem<ET>(Zs + zbuf_bytes + kmajor_off<ET>(n, kk, Bt), 0.f);
  }
  for (int e = tid; e < 3 * kUnits; e += kThreads) bs[e] = bias[(e >> 5) * H + r * kUnits + (e & 31)];
  for (int e = tid; e < Bt; e += kThreads) dts[e] = (b0 + e < B) ? dt[dt_stride ? b0 + e : 0] : 0.f;

  asm volatile("fence.proxy.async;" ::: "memory");
  tc::fence_before_sync();
  cluster.sync();               // also: every block is running before DSMEM writes
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t id = tc::idesc(128, (uint32_t)Bt, sizeof(ET) == 4 ? tc::kFmtTF32 : tc::kFmtBF16);
  uint32_t peer_z[8];                 // shared::cluster address of Zs in every block
#pragma unroll
  for (int p = 0; p < 8; ++p) peer_z[p] = (p < C) ? dsmem_map(smem_addr(Zs), (uint32_t)p) : 0u;
  const int nx = Bt * n_in;     // x values staged per step

  // Cell results of (unit u, sample n) items; lanes of a warp take the 32
  // units of one sample (n is warp-uniform).  Step k's results are written to
  // global memory while step k+1's MMAs run.
  constexpr int kItems = 8;                    // items per thread (plan: 32*Bt <= 8*256)
  float ig[kItems], igg[kItems], ihh[kItems], ih[kItems];
  auto store_results = [&](int kk) {
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      const int e = tid + q * kThreads;
      if (e >= kUnits * Bt) break;
      const int u = e & 31, n = e >> 5, bb = b0 + n;
      if (bb < B) {
        const int unit = r * kUnits + u;
        const long long row = (long long)bb * K + kk;
        act[row * H3 + unit] = ig[q];
        act[row * H3 + H + unit] = igg[q];
        act[row * H3 + 2 * H + unit] = ihh[q];
        stf(h_seq + row * H + unit, ih[q]);
      }
    }
  };

  for (int k = 0; k < K; ++k) {
    uint8_t* zc = Zs + (k & 1) * zbuf_bytes;
    uint8_t* zn = Zs + ((k + 1) & 1) * zbuf_bytes;
    // x of the next step into registers while the MMAs run (16-byte units when
    // vec, else single elements); raw bits, rounded when stored.
    uint4 xu[kXUnits];
    float xr[kXRegs];
    if (vec) {
      const int xupr = n_in / EPU;
#pragma unroll
      for (int q = 0; q < kXUnits; ++q) {
        const int e = tid + q * kThreads;
        const int n = e / xupr, kk = (e - n * xupr) * EPU, bb = b0 + n;
        xu[q] = (e < Bt * xupr && k + 1 < K && bb < B)
                    ? __ldg(reinterpret_cast<const uint4*>(x + ((long long)bb * K + k + 1) * n_in + kk))
                    : make_uint4(0u, 0u, 0u, 0u);
      }
    } else {
#pragma unroll
      for (int q = 0; q < kXRegs; ++q) {
        const int e = tid + q * kThreads;
        const int n = e / n_in, kk = e - n * n_in, bb = b0 + n;
        xr[q] = (e < nx && k + 1 < K && bb < B) ? ldf(x + ((long long)bb * K + k + 1) * n_in + kk) : 0.f;
      }
    }
    if (warp == 0) {  // operands from the converged warp, one elected lane issues
      uint64_t ad = tc::sdesc_k_sw128(tc::smem_u32(Ws)), bd = tc::sdesc_k_sw128(tc::smem_u32(zc));
      const uint32_t b_step = (uint32_t)Bt * 128;
      if (tc::elect_one()) {
        for (int a = 0; a < nA; ++a) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if constexpr (sizeof(ET) == 4) tc::mma_tf32(tmem, ad + 2 * j, bd + 2 * j, id, (a | j) != 0);
            else tc::mma_bf16(tmem, ad + 2 * j, bd + 2 * j, id, (a | j) != 0);
          }
          ad = tc::sdesc_advance(ad, 128 * 128);
          bd = tc::sdesc_advance(bd, b_step);
        }
        tc::mma_commit(&bar);
      }
      __syncwarp();
    }
    if (k > 0) store_results(k - 1);
    // One thread waits for the MMAs; the others meet it at the block barrier.
    if (tid == 0 && !tc::mbar_wait(&bar, k & 1, kMaxPolls)) err = 1;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // TMEM -> shared: pre-activations of head w (lane quadrant w), columns split
    // between warps w and w+4.
    if ((warp & 3) < 3) {
      const int c = warp & 3;
      for (int q = warp >> 2; q < Bt / 16; q += 2) {
        float v[16];
        tc::tmem_ld16(tmem + ((uint32_t)(32 * c) << 16) + (uint32_t)(16 * q), v);
#pragma unroll
        for (int i = 0; i < 16; ++i) ex[(c * kUnits + lane) * ex_ld + 16 * q + i] = v[i];
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    float hop[kItems];
    // pass 1: cell math of all items
#pragma unroll
    for (int q = 0; q < kItems; ++q) {
      const int e = tid + q * kThreads;
      hop[q] = 0.f;
      if (e >= kUnits * Bt) break;
      const int u = e & 31, n = e >> 5, bb = b0 + n;
      const float af = ex[(0 * kUnits + u) * ex_ld + n] + bs[u];
      const float ag = ex[(1 * kUnits + u) * ex_ld + n] + bs[kUnits + u];
      const float ah = ex[(2 * kUnits + u) * ex_ld + n] + bs[2 * kUnits + u];
      const CellAct ca = cell_act(af, ag, ah, dts[n]);
      const float gate = ca.gate, g = ca.g, hh = ca.hh;
      const float h = fmaf(gate, g - hh, hh);
      ig[q] = gate; igg[q] = g; ihh[q] = hh; ih[q] = h;
      if (bb < B) {
        if constexpr (sizeof(ET) == 2) hop[q] = round_bf16(h);
        else hop[q] = round_tf32(h);
      }
    }
    // pass 2: this block's h slice into its own next Z buffer, then (vec) copied
    // to every other block of the cluster as whole 16-byte chunks.
    if (k + 1 < K) {
#pragma unroll
      for (int q = 0; q < kItems; ++q) {
        const int e = tid + q * kThreads;
        if (e >= kUnits * Bt) break;
        const int u = e & 31, n = e >> 5;
        const uint32_t off = kmajor_off<ET>(n, n_in + r * kUnits + u, Bt);
        if (vec) {
          st_elem<ET>(zn + off, hop[q]);
        } else {
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            if (p < C) {
              if constexpr (sizeof(ET) == 4) dsmem_st(peer_z[p] + ((k + 1) & 1) * zbuf_bytes + off, hop[q]);
              else dsmem_st_bf16(peer_z[p] + ((k + 1) & 1) * zbuf_bytes + off, hop[q]);
            }
          }
        }
      }
      if (vec) {
        __syncthreads();
        constexpr int kChunksPerRow = kUnits * (int)sizeof(ET) / 16;   // 8 (TF32) or 4 (bf16)
        for (int c = tid; c < Bt * kChunksPerRow; c += kThreads) {
          const int n = c / kChunksPerRow, cc = c - n * kChunksPerRow;
          const uint32_t off = kmajor_off<ET>(n, n_in + r * kUnits + cc * EPU, Bt);
          const uint4 val = *reinterpret_cast<const uint4*>(zn + off);
          const uint32_t roff = ((k + 1) & 1) * zbuf_bytes + off;
#pragma unroll
          for (int p = 0; p < 8; ++p)
            if (p < C && p != r) dsmem_st(peer_z[p] + roff, val);
        }
      }
    }
    if (k + 1 < K) {
      if (vec) {
        const int xupr = n_in / EPU;
#pragma unroll
        for (int q = 0; q < kXUnits; ++q) {
          const int e = tid + q * kThreads;
          if (e < Bt * xupr) {
            const int n = e / xupr, kk = (e - n * xupr) * EPU;
            *reinterpret_cast<uint4*>(zn + kmajor_off<ET>(n, kk, Bt)) = round_unit<MODE>(xu[q]);
          }
        }
      } else {
#pragma unroll
        for (int q = 0; q < kXRegs; ++q) {
          const int e = tid + q * kThreads;
          if (e < nx) st_elem<ET>(zn + kmajor_off<ET>(e / n_in, e % n_in, Bt), to_operand<MODE>(xr[q]));
        }
      }
    }
    asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
    tc::fence_before_sync();
    cluster_arrive_release();
    cluster_wait_acquire();
    tc::fence_after_sync();
  }
  store_results(K - 1);
  if (err && tid == 0) atomicExch(&g_tc_kloop_error, 1);
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, tmem_cols);
}

bool plan_fwd(const Layout& L, TcPlan* p) {
  if (L.math == CFC_MATH_FP32) return false;
  if (L.H % kUnits || L.H / kUnits > 8) return false;
  const int es = (L.math == CFC_MATH_TF32) ? 4 : 2;
  const int C = L.H / kUnits;
  const int nA = (L.Zc * es + 127) / 128;
  auto smem_for = [&](int Bt, TcPlan* q) {
    size_t off = (size_t)nA * 128 * 128;
    q->off_z = off;
    off += 2ull * nA * Bt * 128;
    q->off_ex = off;
    off += 3ull * kUnits * (Bt + 1) * 4;
    q->off_bs = off;
    off += 3 * kUnits * 4;
    q->off_dt = off;
    off += (size_t)Bt * 4;
    q->smem = off + 1024;  // alignment slack
    return q->smem;
  };
  // Smallest Bt (multiple of 16) whose grid fits in one wave of blocks, or
  // failing that the largest that fits in shared memory.
  int best = 0;
  for (int Bt = 16; Bt <= 128; Bt += 16) {
    TcPlan q;
    if (smem_for(Bt, &q) > kSmemMax) break;
    if ((long long)kUnits * Bt > 8ll * kThreads) break;
    const int epu = 16 / es;
    const bool vec = (L.n_in % epu == 0) && (L.H % epu == 0);
    if (vec ? ((long long)Bt * (L.n_in / epu) > (long long)kXUnits * kThreads)
            : ((long long)Bt * L.n_in > (long long)kXRegs * kThreads)) break;
    best = Bt;
    if ((long long)(L.B + Bt - 1) / Bt * C <= kNumSMs) break;
  }
  if (!best) return false;
  p->C = C;
  p->Bt = best;
  p->nA = nA;
  smem_for(best, p);
  uint32_t cols = 32;
  while (cols < (uint32_t)best) cols <<= 1;
  p->tmem_cols = cols;
  return true;
}

template <typename ET, int MODE>
cudaError_t launch_fwd(const Layout& L, const TcPlan& p, const CfcArgs& a, cudaStream_t s) {
  auto kern = k_cfc_fwd_tc<ET, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(((L.B + p.Bt - 1) / p.Bt) * p.C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  TraceScope trace("cfc_fwd_tc", s);
  return cudaLaunchKernelEx(&cfg, kern, static_cast<const ET*>(a.x), static_cast<const ET*>(a.h0),
                            static_cast<const ET*>(a.W_in), static_cast<const ET*>(a.W_rec), a.b, a.dt,
                            a.dt_stride, L.B, L.K, L.n_in, L.H, p.Bt, p.nA, (uint32_t)p.off_z,
                            (uint32_t)p.off_ex, (uint32_t)p.off_bs, (uint32_t)p.off_dt, p.tmem_cols,
                            static_cast<ET*>(a.h_seq), reinterpret_cast<float*>(a.ws + L.off_act));
}

// ---------------------------------------------------------------------------
// Backward K loop on the tensor cores, the cluster split by hidden units.
//
// Block r of the cluster owns units U_r = [32r, 32r+32).  Per step k
// (reverse) it
//   1. forms dA of its units for the Bt samples from its carry (the gradient
//      reaching its units' h columns, summed at the end of the previous step),
//      the saved activations (loaded one step ahead) and the upstream seeds;
//      writes dA to global memory (operand type) and into the K-major B tile
//      (rows = samples, K = (head, unit) = 96);
//   2. computes its partial carry^T [H x Bt] = W_rec[rows of U_r]^T dA_r^T:
//      nMt M=128 MMA chains, A = its 96 columns of W_rec^T resident in shared
//      memory (K-major, 128B swizzle), accumulators in TMEM;
//   3. sends each partial unit column j to the block that owns unit j through
//      distributed shared memory: receive buffer [source block][unit][sample],
//      double-buffered by step parity;
//   4. after one cluster barrier, sums the C partials of its own units in
//      block order (deterministic): the carry of step k-1, or grad_h0 after
//      step 0.
// Only partial sums cross the cluster; dA never leaves the block that made it.
// grad_x = dA W_in does not feed the recurrence: it is one GEMM over all B*K
// rows after the loop (launch_grad_x_tc).
// ---------------------------------------------------------------------------
constexpr int kBwdMaxItems = 8;         // (unit, sample) items per thread: 32*Bt <= 8*256

struct TcBwdPlan {
  int C = 0, Bt = 0, nMt = 0, nAk = 0;
  size_t smem = 0, off_da = 0, off_recv = 0, off_carry = 0, off_dt = 0;
  uint32_t tmem_cols = 0;
};

template <typename ET, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
k_cfc_bwd_tc(const ET* __restrict__ W_in, const ET* __restrict__ W_rec, const float* __restrict__ dt,
             int dt_stride, int B, int K, int H, int Bt, int nMt, int nAk, uint32_t off_da, uint32_t off_recv,
             uint32_t off_carry, uint32_t off_dt, uint32_t tmem_cols, const ET* __restrict__ h_seq,
             const float* __restrict__ grad_h_seq, const float* __restrict__ grad_h_last,
             const float* __restrict__ y, const float* __restrict__ act, ET* __restrict__ dA_out,
             float* __restrict__ grad_h0) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int r = (int)cluster.block_rank();
  const int H3 = 3 * H;
  const int Mrows = nMt * 128;
  const int Kpad = nAk * (128 / (int)sizeof(ET));
  constexpr int cpo = kUnits;                        // columns owned by one block
  const int b0 = (int)(blockIdx.x / C) * Bt;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nitems = kUnits * Bt;

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* Wt = sm;                                        // nAk x [Mrows][128 B]
  uint8_t* dAs = sm + off_da;                              // nAk x [Bt][128 B]
  float* recv = reinterpret_cast<float*>(sm + off_recv);   // [2][C][32][Bt]
  float* carry = reinterpret_cast<float*>(sm + off_carry); // [Bt][33]
  float* dts = reinterpret_cast<float*>(sm + off_dt);      // [Bt]
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int err;

  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, tmem_cols);
  // A operand: row j (unit), K index kap = c*32 + u -> W_rec[c*H + 32r + u][j].
  for (int e = tid; e < Mrows * Kpad; e += kThreads) {
    const int kap = e / Mrows, j = e - kap * Mrows;
    float v = 0.f;
    if (j < H && kap < 3 * kUnits) {
      const long long row = (long long)(kap >> 5) * H + r * kUnits + (kap & 31);
      v = ld_operand<MODE>(W_rec + row * H + j);
    }
    st_elem<ET>(Wt + kmajor_off<ET>(j, kap, Mrows), v);
  }
  for (int e = tid; e < nAk * Bt * 32; e += kThreads) reinterpret_cast<float*>(dAs)[e] = 0.f;
  for (int e = tid; e < Bt * 33; e += kThreads) carry[e] = 0.f;
  for (int e = tid; e < Bt; e += kThreads) dts[e] = (b0 + e < B) ? dt[dt_stride ? b0 + e : 0] : 0.f;
  const uint32_t recv_addr = smem_addr(recv);

  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc::fence_before_sync();
  cluster.sync();               // every block is running before DSMEM writes
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t id = tc::idesc(128, (uint32_t)Bt, sizeof(ET) == 4 ? tc::kFmtTF32 : tc::kFmtBF16);

  // Saved activations of step k (items: lanes = the 32 units of one sample).
  float pa[3][kBwdMaxItems], pu[kBwdMaxItems];
  auto load_step = [&](int k) {
#pragma unroll
    for (int q = 0; q < kBwdMaxItems; ++q) {
      const int e = tid + q * kThreads;
      pa[0][q] = pa[1][q] = pa[2][q] = pu[q] = 0.f;
      if (e < nitems && k >= 0) {
        const int u = e & 31, n = e >> 5, bb = b0 + n;
        if (bb < B) {
          const long long row = (long long)bb * K + k;
          const int unit = r * kUnits + u;
          pa[0][q] = act[row * H3 + unit];
          pa[1][q] = act[row * H3 + H + unit];
          pa[2][q] = act[row * H3 + 2 * H + unit];
          if (grad_h_seq) pu[q] = grad_h_seq[row * H + unit];
        }
      }
    }
  };
  load_step(K - 1);

  for (int step = 0; step < K; ++step) {
    const int k = K - 1 - step;
    const int buf = k & 1;
    {
      // ---- 1. dA of this block's units -> global dA and the B tile
#pragma unroll
      for (int q = 0; q < kBwdMaxItems; ++q) {
        const int e = tid + q * kThreads;
        if (e >= nitems) break;
        const int u = e & 31, n = e >> 5, bb = b0 + n;
        float d0 = 0.f, d1 = 0.f, d2 = 0.f;
        if (bb < B) {
          const int unit = r * kUnits + u;
          float delta = carry[n * 33 + u] + pu[q];
          if (k == K - 1) {
            if (grad_h_last) delta += grad_h_last[(long long)bb * H + unit];
            if (y) delta += ldf(h_seq + ((long long)bb * K + k) * H + unit) - y[(long long)bb * H + unit];
          }
          const float gate = pa[0][q], g = pa[1][q], hh = pa[2][q];
          d1 = to_operand<MODE>(delta * gate * (1.f - g * g));
          d2 = to_operand<MODE>(delta * (1.f - gate) * (1.f - hh * hh));
          d0 = to_operand<MODE>(-dts[n] * delta * (g - hh) * gate * (1.f - gate));
          const long long row = (long long)bb * K + k;
          stf(dA_out + row * H3 + unit, d0);
          stf(dA_out + row * H3 + H + unit, d1);
          stf(dA_out + row * H3 + 2 * H + unit, d2);
        }
        st_elem<ET>(dAs + kmajor_off<ET>(n, u, Bt), d0);
        st_elem<ET>(dAs + kmajor_off<ET>(n, kUnits + u, Bt), d1);
        st_elem<ET>(dAs + kmajor_off<ET>(n, 2 * kUnits + u, Bt), d2);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      // ---- 2. partial dz (thread 0 issues; the next step's activations load meanwhile)
      if (warp == 0) {  // operands from the converged warp, one elected lane issues
        const uint64_t a0 = tc::sdesc_k_sw128(tc::smem_u32(Wt)), b0d = tc::sdesc_k_sw128(tc::smem_u32(dAs));
        if (tc::elect_one()) {
          for (int mt = 0; mt < nMt; ++mt) {
            for (int a = 0; a < nAk; ++a) {
              const uint64_t ad = tc::sdesc_advance(a0, (uint32_t)(a * Mrows + mt * 128) * 128u);
              const uint64_t bd = tc::sdesc_advance(b0d, (uint32_t)(a * Bt) * 128u);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                if constexpr (sizeof(ET) == 4)
                  tc::mma_tf32(tmem + (uint32_t)(mt * Bt), ad + 2 * j, bd + 2 * j, id, (a | j) != 0);
                else tc::mma_bf16(tmem + (uint32_t)(mt * Bt), ad + 2 * j, bd + 2 * j, id, (a | j) != 0);
              }
            }
          }
          tc::mma_commit(&bar);
        }
        __syncwarp();
      }
      load_step(k - 1);
      if (tid == 0 && !tc::mbar_wait(&bar, (uint32_t)(step & 1), kMaxPolls)) err = 1;
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
      // ---- 3. partial unit column j -> its owner's receive buffer [buf][r][jl][n]
      const int qd = warp & 3, half = warp >> 2, nch = Bt / 16;
      for (int pidx = half; pidx < nMt * nch; pidx += 2) {
        const int mt = pidx / nch, n0 = (pidx - mt * nch) * 16;
        const int j = mt * 128 + qd * 32 + lane;
        float v[16];
        tc::tmem_ld16(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(mt * Bt + n0), v);
        if (j < H) {
          const int owner = j >> 5, jl = j & 31;
          const uint32_t off = (uint32_t)((((buf * C + r) * cpo + jl) * Bt + n0) * 4);
          const uint32_t dst = (owner == r) ? 0u : dsmem_map(recv_addr, (uint32_t)owner);
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const uint4 w = make_uint4(__float_as_uint(v[i]), __float_as_uint(v[i + 1]), __float_as_uint(v[i + 2]),
                                       __float_as_uint(v[i + 3]));
            if (owner == r) *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(recv) + off + 4 * i) = w;
            else dsmem_st(dst + off + 4 * i, w);
          }
        }
      }
    }
    // ---- 4. one barrier publishes the partials; owners sum them
    tc::fence_before_sync();
    cluster_arrive_release();
    cluster_wait_acquire();
    tc::fence_after_sync();
    for (int e = tid; e < cpo * Bt; e += kThreads) {
      const int u = e / Bt, n = e - u * Bt, bb = b0 + n;
      float sum = 0.f;
      for (int src = 0; src < C; ++src) sum += recv[((buf * C + src) * cpo + u) * Bt + n];
      if (k > 0) carry[n * 33 + u] = sum;
      else if (grad_h0 && bb < B) grad_h0[(long long)bb * H + r * kUnits + u] = sum;
    }
    __syncthreads();
  }
  if (err && tid == 0) atomicExch(&g_tc_kloop_error, 1);
  tc::fence_before_sync();
  cluster.sync();               // no block leaves while peers may still write its buffers
  if (warp == 0) tc::tmem_dealloc(tmem, tmem_cols);
}

bool plan_bwd_cluster(const Layout& L, TcBwdPlan* p) {
  if (L.math == CFC_MATH_FP32) return false;
  if (L.H % kUnits || L.H / kUnits > 8) return false;
  const int C = L.H / kUnits;
  const int es = (L.math == CFC_MATH_TF32) ? 4 : 2;
  const int nMt = (L.H + 127) / 128;
  const int nAk = (3 * kUnits * es + 127) / 128;
  const int cpo = kUnits;
  auto smem_for = [&](int Bt, TcBwdPlan* q) {
    size_t off = (size_t)nAk * nMt * 128 * 128;
    q->off_da = off;
    off += (size_t)nAk * Bt * 128;
    q->off_recv = off;
    off += 2ull * C * cpo * Bt * 4;
    q->off_carry = off;
    off += (size_t)Bt * 33 * 4;
    q->off_dt = off;
    off += (size_t)Bt * 4;
    q->smem = off + 1024;
    return q->smem;
  };
  // Smallest Bt (multiple of 16) whose grid fits one wave of blocks.
  int best = 0;
  for (int Bt = 16; Bt <= 128; Bt += 16) {
    TcBwdPlan q;
    if (smem_for(Bt, &q) > kSmemMax) break;
    if ((long long)kUnits * Bt > (long long)kBwdMaxItems * kThreads) break;
    if ((long long)nMt * Bt > 512) break;
    best = Bt;
    if ((long long)(L.B + Bt - 1) / Bt * C <= kNumSMs) break;
  }
  if (!best) return false;
  p->C = C;
  p->Bt = best;
  p->nMt = nMt;
  p->nAk = nAk;
  smem_for(best, p);
  uint32_t cols = 32;
  while (cols < (uint32_t)(nMt * best)) cols <<= 1;
  p->tmem_cols = cols;
  return true;
}

template <typename ET, int MODE>
cudaError_t launch_bwd_cluster(const Layout& L, const TcBwdPlan& p, const CfcArgs& a, cudaStream_t s) {
  auto kern = k_cfc_bwd_tc<ET, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(((L.B + p.Bt - 1) / p.Bt) * p.C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  {
    TraceScope trace("cfc_bwd_cluster_tc", s);
    e = cudaLaunchKernelEx(&cfg, kern, static_cast<const ET*>(a.W_in), static_cast<const ET*>(a.W_rec), a.dt,
                           a.dt_stride, L.B, L.K, L.H, p.Bt, p.nMt, p.nAk, (uint32_t)p.off_da,
                           (uint32_t)p.off_recv, (uint32_t)p.off_carry, (uint32_t)p.off_dt, p.tmem_cols,
                           static_cast<const ET*>(a.h_seq), a.grad_h_seq, a.grad_h_last, a.y,
                           reinterpret_cast<const float*>(a.ws + L.off_act), reinterpret_cast<ET*>(a.ws + L.off_dA),
                           a.grad_h0);
  }
  if (e != cudaSuccess || !a.grad_x) return e;
  return launch_grad_x_tc(L, a, s);
}

}  // namespace

int read_tc_kloop_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_kloop_error, sizeof(int)) != cudaSuccess) return CFC_ERR_DEVICE;
  if (clear && v) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_tc_kloop_error, &zero, sizeof(int)) != cudaSuccess) return CFC_ERR_DEVICE;
  }
  return v;
}

cudaError_t launch_forward_tc(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  const int choice = kernel_choice();
  if (choice == kCluster || choice == kSimt || choice == kTcStream) return cudaErrorNotSupported;
  TcPlan p;
  if (!plan_fwd(L, &p)) return cudaErrorNotSupported;
  // Beyond one wave of clusters the streamed-weight kernel is faster.
  if (choice == kAuto && (long long)(L.B + p.Bt - 1) / p.Bt * p.C > kNumSMs) return cudaErrorNotSupported;
  if (L.math == CFC_MATH_TF32) return launch_fwd<float, CFC_MATH_TF32>(L, p, a, s);
  return launch_fwd<__nv_bfloat16, CFC_MATH_BF16>(L, p, a, s);
}

cudaError_t launch_backward_cluster_tc(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  const int choice = kernel_choice();
  if (choice == kCluster || choice == kSimt || choice == kTcStream) return cudaErrorNotSupported;
  TcBwdPlan p;
  if (!plan_bwd_cluster(L, &p)) return cudaErrorNotSupported;
  if (a.grad_x && !grad_x_gemm_applies(L)) return cudaErrorNotSupported;
  if (choice == kAuto && (long long)(L.B + p.Bt - 1) / p.Bt * p.C > kNumSMs) return cudaErrorNotSupported;
  if (L.math == CFC_MATH_TF32) return launch_bwd_cluster<float, CFC_MATH_TF32>(L, p, a, s);
  return launch_bwd_cluster<__nv_bfloat16, CFC_MATH_BF16>(L, p, a, s);
}

}  // namespace cfc
