// cfc_tc_bwd.cu -- backward K loop of the TF32 / bf16 modes on the tcgen05
// tensor cores, one block per tile of Bt samples (no cluster).
//
// Per step k (reverse) the block computes the gradient reaching z_k = [x_k; h_k]
//
//   dz^T [Zc x Bt] = W_cat^T [Zc x 3H] * dA_k^T [3H x Bt]
//
// as nM = ceil(Zc/128) MMA row tiles (M = 128 z-columns, N = Bt samples,
// K = 3H).  The A operand, W_cat^T, is the same for every step and every
// block: it is prepared once per call as pre-swizzled 16 KB tiles (128 rows x
// 128 bytes of K) in the workspace and streamed through a ring of shared-memory
// stages with TMA bulk copies (cp.async.bulk, mbarrier transaction counts).
// The tile sequence repeats every step, so the copies for the next step's
// first tiles run while the block computes the next dA.  The B operand, dA_k
// of the Bt samples, is computed by the block itself into a K-major swizzled
// shared-memory tile.
//
// Elementwise phase of step k: thread <-> z-column j = 128*mt + 32*(warp%4) +
// lane (the TMEM lane quadrant rule).  It reads dz of step k+1 for its column
// from TMEM: x columns become grad_x[:, k+1], h columns the carry of unit
// j - n_in, from which (with the saved activations) it forms the three dA
// values of that unit for every sample of the tile.  After step 0 the same
// read gives grad_x[:, 0] and grad_h0.
//
// Waits are bounded; a timeout records an error in the device error word.
#include <algorithm>

#include "cfc_internal.cuh"
#include "tc_common.cuh"

namespace cfc {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxStages = 6;    // ring of streamed A tiles (runtime count: nst)
constexpr uint32_t kTile = 128 * 128;      // bytes of one streamed A tile
constexpr uint32_t kMaxPolls = 1u << 24;
constexpr size_t kSmemMax = 227 * 1024;

__device__ int g_tc_bwd_error = 0;

__device__ __forceinline__ void expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}

template <typename ET>
__device__ __forceinline__ void st_elem(uint8_t* p, float v) {
  if constexpr (sizeof(ET) == 4) *reinterpret_cast<float*>(p) = v;
  else *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
}

template <typename ET>
__device__ __forceinline__ uint32_t kmajor_off(int row, int kk, int rows) {
  const uint32_t kb = (uint32_t)kk * sizeof(ET);
  return (kb >> 7) * (uint32_t)rows * 128u + tc::sw128_offset(row, kb & 127u);
}

// W_cat^T tiles: tile (mt, a) holds rows j = 128*mt .. 128*mt+127 (z columns)
// and K elements a*EPA .. a*EPA+EPA-1 (EPA = 128 bytes / element), at byte
// offset ((a * nM) + mt) * kTile, swizzled exactly as in shared memory.
template <typename ET, int MODE>
__global__ void k_prep_wt_tiles(const ET* __restrict__ W_in, const ET* __restrict__ W_rec, int n_in,
                                int H, int nM, int nAk, uint8_t* __restrict__ tiles) {
  constexpr int EPA = 128 / sizeof(ET);
  const int Zc = n_in + H, H3 = 3 * H;
  const long long total = (long long)nM * nAk * 128 * EPA;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int kl = (int)(e % EPA);
    const long long rest = e / EPA;
    const int i = (int)(rest % 128);
    const long long t = rest / 128;            // tile index = a * nM + mt
    const int mt = (int)(t % nM), a = (int)(t / nM);
    const int j = mt * 128 + i, kk = a * EPA + kl;
    float v = 0.f;
    if (j < Zc && kk < H3)
      v = (j < n_in) ? ld_operand<MODE>(W_in + (long long)kk * n_in + j)
                     : ld_operand<MODE>(W_rec + (long long)kk * H + (j - n_in));
    st_elem<ET>(tiles + t * kTile + tc::sw128_offset(i, kl * sizeof(ET)), v);
  }
}

template <typename ET, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
k_cfc_bwd_tcb(const uint8_t* __restrict__ wtiles, const float* __restrict__ dt, int dt_stride, int B,
              int K, int n_in, int H, int Bt, int nM, int nAk, int nst, uint32_t tmem_cols,
              const ET* __restrict__ h_seq, const float* __restrict__ grad_h_seq,
              const float* __restrict__ grad_h_last, const float* __restrict__ y,
              const float* __restrict__ act, ET* __restrict__ dA_out, float* __restrict__ grad_h0,
              float* __restrict__ grad_x) {
  const int Zc = n_in + H, H3 = 3 * H;
  const int b0 = blockIdx.x * Bt;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3;
  const int T = nAk * nM;                       // streamed tiles per step
  const long long total_tiles = (long long)K * T;

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage = sm;                                   // nst x 16 KB
  uint8_t* dAs = sm + (size_t)nst * kTile;               // nAk x [Bt rows][128 B]
  float* dts = reinterpret_cast<float*>(dAs + (size_t)nAk * Bt * 128);   // [Bt]
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], done;
  __shared__ uint32_t tmem_base;
  __shared__ int err;

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    tc::mbar_init(&done, 1);
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, tmem_cols);
  for (int e = tid; e < Bt; e += kThreads) dts[e] = (b0 + e < B) ? dt[dt_stride ? b0 + e : 0] : 0.f;
  // dA tile padding (K beyond 3H) stays zero for the whole launch.
  {
    constexpr int EPA = 128 / sizeof(ET);
    const int Kpad = nAk * EPA;
    for (int e = tid; e < Bt * (Kpad - H3); e += kThreads) {
      const int n = e / (Kpad - H3), kk = H3 + e % (Kpad - H3);
      st_elem<ET>(dAs + kmajor_off<ET>(n, kk, Bt), 0.f);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t id = tc::idesc(128, (uint32_t)Bt, sizeof(ET) == 4 ? tc::kFmtTF32 : tc::kFmtBF16);

  // Producer state (thread 0): next tile sequence number to copy.
  long long next_copy = 0;
  auto issue_copy = [&](long long g) {
    const int st = (int)(g % nst);
    if (g >= nst) {
      // stage reuse: the MMAs of tile g - nst must be complete
      if (!tc::mbar_wait(&empty[st], (uint32_t)(((g - nst) / nst) & 1), kMaxPolls)) err = 1;
    }
    const int t = (int)(g % T);
    expect_tx(&full[st], kTile);
    bulk_g2s(stage + st * kTile, wtiles + (size_t)t * kTile, kTile, &full[st]);
  };
  if (tid == 0) {
    for (; next_copy < std::min<long long>(nst - 2, total_tiles); ++next_copy) issue_copy(next_copy);
  }

  // rows of z handled by this thread: j = 128*mt + 32*quad + lane for mt = warp/4, warp/4 + 2, ...
  for (int step = 0; step <= K; ++step) {
    const int k = K - 1 - step;                  // step == K: final read-out only
    // ---- elementwise phase: dz of step k+1 from TMEM -> grad_x / carry -> dA_k
    for (int mt = warp >> 2; mt < nM; mt += kThreads / 128) {
      const int j = mt * 128 + quad * 32 + lane;
      for (int n0 = 0; n0 < Bt; n0 += 16) {
        float dz[16];
        if (step > 0) {
          tc::tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(mt * Bt + n0), dz);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) dz[i] = 0.f;
        }
        if (j < n_in) {
          if (step > 0 && grad_x) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int bb = b0 + n0 + i;
              if (bb < B) grad_x[((long long)bb * K + (k + 1)) * n_in + j] = dz[i];
            }
          }
        } else if (j < Zc) {
          const int u = j - n_in;
          if (k < 0) {                           // after step 0: grad_h0
            if (grad_h0) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int bb = b0 + n0 + i;
                if (bb < B) grad_h0[(long long)bb * H + u] = dz[i];
              }
            }
          } else {
            float ga[16], gg[16], gh[16], up[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int bb = b0 + n0 + i;
              ga[i] = gg[i] = gh[i] = up[i] = 0.f;
              if (bb < B) {
                const long long row = (long long)bb * K + k;
                ga[i] = act[row * H3 + u];
                gg[i] = act[row * H3 + H + u];
                gh[i] = act[row * H3 + 2 * H + u];
                if (grad_h_seq) up[i] = grad_h_seq[row * H + u];
                if (k == K - 1) {
                  if (grad_h_last) up[i] += grad_h_last[(long long)bb * H + u];
                  if (y) up[i] += ldf(h_seq + row * H + u) - y[(long long)bb * H + u];
                }
              }
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int n = n0 + i, bb = b0 + n;
              float d0 = 0.f, d1 = 0.f, d2 = 0.f;
              if (bb < B) {
                const float delta = dz[i] + up[i];
                const float gate = ga[i], g = gg[i], hh = gh[i];
                d1 = to_operand<MODE>(delta * gate * (1.f - g * g));
                d2 = to_operand<MODE>(delta * (1.f - gate) * (1.f - hh * hh));
                d0 = to_operand<MODE>(-dts[n] * delta * (g - hh) * gate * (1.f - gate));
                const long long row = (long long)bb * K + k;
                stf(dA_out + row * H3 + u, d0);
                stf(dA_out + row * H3 + H + u, d1);
                stf(dA_out + row * H3 + 2 * H + u, d2);
              }
              st_elem<ET>(dAs + kmajor_off<ET>(n, u, Bt), d0);
              st_elem<ET>(dAs + kmajor_off<ET>(n, H + u, Bt), d1);
              st_elem<ET>(dAs + kmajor_off<ET>(n, 2 * H + u, Bt), d2);
            }
          }
        }
      }
    }
    if (k < 0) break;
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // ---- MMA phase (thread 0): stream W_cat^T tiles, dz_k = W^T dA_k into TMEM
    if (tid == 0) {
      const uint32_t da = tc::smem_u32(dAs);
      for (int t = 0; t < T; ++t) {
        const long long g = (long long)step * T + t;
        const int st = (int)(g % nst);
        if (!tc::mbar_wait(&full[st], (uint32_t)((g / nst) & 1), kMaxPolls)) err = 1;
        tc::fence_after_sync();
        const int a = t / nM, mt = t % nM;
        const uint32_t sa = tc::smem_u32(stage + st * kTile);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint64_t ad = tc::sdesc_k_sw128(sa + 32 * q);
          const uint64_t bd = tc::sdesc_k_sw128(da + (uint32_t)a * Bt * 128 + 32 * q);
          if constexpr (sizeof(ET) == 4) tc::mma_tf32(tmem + (uint32_t)(mt * Bt), ad, bd, id, (a | q) != 0);
          else tc::mma_bf16(tmem + (uint32_t)(mt * Bt), ad, bd, id, (a | q) != 0);
        }
        tc::mma_commit(&empty[st]);
        if (next_copy < total_tiles) issue_copy(next_copy++);
      }
      tc::mma_commit(&done);
      // Only this thread waits on the MMA completion; the others wait at the
      // block barrier (polling threads would compete with the barrier traffic
      // of the tile stream).
      if (!tc::mbar_wait(&done, (uint32_t)(step & 1), kMaxPolls)) err = 1;
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  }
  if (err) atomicExch(&g_tc_bwd_error, 1);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, tmem_cols);
}

struct BwdPlan {
  int Bt = 0, nM = 0, nAk = 0, nst = 0;
  uint32_t tmem_cols = 0;
  size_t smem = 0;
};

bool plan_bwd(const Layout& L, BwdPlan* p) {
  if (L.math == CFC_MATH_FP32) return false;
  const int es = (L.math == CFC_MATH_TF32) ? 4 : 2;
  const int nM = (L.Zc + 127) / 128;
  const int nAk = (L.H3 * es + 127) / 128;
  // Bt: samples per block, the MMA's N: about one block per SM, at least 32.
  int Bt = (int)(((long long)L.B + kNumSMs - 1) / kNumSMs);
  Bt = std::min(128, std::max(32, (Bt + 15) / 16 * 16));
  auto fixed_for = [&](int bt) { return 1024 + (size_t)nAk * bt * 128 + bt * 4 + 256; };
  while (Bt > 16 && (fixed_for(Bt) + 4 * (size_t)kTile > kSmemMax || (long long)nM * Bt > 512)) Bt -= 16;
  if (fixed_for(Bt) + 4 * (size_t)kTile > kSmemMax || (long long)nM * Bt > 512) return false;
  // as many stages as fit (the stream is latency-bound: more tiles in flight)
  const int nst = (int)std::min<size_t>(kMaxStages, (kSmemMax - fixed_for(Bt)) / kTile);
  p->Bt = Bt;
  p->nM = nM;
  p->nAk = nAk;
  p->nst = nst;
  uint32_t cols = 32;
  while (cols < (uint32_t)(nM * Bt)) cols <<= 1;
  p->tmem_cols = cols;
  p->smem = fixed_for(Bt) + (size_t)nst * kTile;
  return true;
}

template <typename ET, int MODE>
cudaError_t launch_bwd(const Layout& L, const BwdPlan& p, const CfcArgs& a, cudaStream_t s) {
  uint8_t* tiles = reinterpret_cast<uint8_t*>(a.ws + L.off_wtt);
  {
    const long long total = (long long)p.nM * p.nAk * 128 * (128 / sizeof(ET));
    const int blocks = (int)std::min<long long>((total + 255) / 256, 4 * kNumSMs);
    TraceScope trace("prep_wt_tiles", s);
    k_prep_wt_tiles<ET, MODE><<<blocks, 256, 0, s>>>(static_cast<const ET*>(a.W_in),
                                                     static_cast<const ET*>(a.W_rec), L.n_in, L.H, p.nM,
                                                     p.nAk, tiles);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  auto kern = k_cfc_bwd_tcb<ET, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  const int grid = (L.B + p.Bt - 1) / p.Bt;
  TraceScope trace("cfc_bwd_tc", s);
  kern<<<grid, kThreads, p.smem, s>>>(tiles, a.dt, a.dt_stride, L.B, L.K, L.n_in, L.H, p.Bt, p.nM, p.nAk,
                                      p.nst, p.tmem_cols, static_cast<const ET*>(a.h_seq), a.grad_h_seq,
                                      a.grad_h_last, a.y, reinterpret_cast<const float*>(a.ws + L.off_act),
                                      reinterpret_cast<ET*>(a.ws + L.off_dA), a.grad_h0, a.grad_x);
  return cudaGetLastError();
}

}  // namespace

size_t tc_bwd_tiles_bytes(int n_in, int n_hid, int math) {
  if (math == CFC_MATH_FP32) return 0;
  const int es = (math == CFC_MATH_TF32) ? 4 : 2;
  const int nM = (n_in + n_hid + 127) / 128;
  const int nAk = (3 * n_hid * es + 127) / 128;
  return (size_t)nM * nAk * kTile;
}

int read_tc_bwd_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_bwd_error, sizeof(int)) != cudaSuccess) return CFC_ERR_DEVICE;
  if (clear && v) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_tc_bwd_error, &zero, sizeof(int)) != cudaSuccess) return CFC_ERR_DEVICE;
  }
  return v;
}

cudaError_t launch_backward_tc(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  const int choice = kernel_choice();
  if (choice == kCluster || choice == kSimt) return cudaErrorNotSupported;
  BwdPlan p;
  if (!plan_bwd(L, &p)) return cudaErrorNotSupported;
  if (L.math == CFC_MATH_TF32) return launch_bwd<float, CFC_MATH_TF32>(L, p, a, s);
  return launch_bwd<__nv_bfloat16, CFC_MATH_BF16>(L, p, a, s);
}

}  // namespace cfc
