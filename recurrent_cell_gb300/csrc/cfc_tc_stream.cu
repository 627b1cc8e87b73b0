// cfc_tc_stream.cu -- forward and backward K loops of the TF32 / bf16 modes on
// the tcgen05 tensor cores with streamed weights, one block per tile of Bt
// samples (no cluster).
//
// Forward, per step k:  D [3H x Bt] = W_cat [3H x Zc] * Z_k^T  with M tiles of
// 128 rows ordered (f, g, h~) per block of 128 units, so the three
// pre-activations of a unit sit in the same TMEM lane of three consecutive
// tiles and the thread that reads them applies the whole cell.  W_cat is
// streamed as pre-swizzled 16 KB tiles (like W_cat^T below); Z_k = [x_k; h_k]
// of the block's samples is a K-major swizzled shared-memory tile that the
// epilogue overwrites with h_{k+1} once the step's MMAs are complete.
//
// Backward, per step k (reverse): the block computes the gradient reaching
// h_k (the carry)
//
//   carry^T [H x Bt] = W_rec^T [H x 3H] * dA_k^T [3H x Bt]
//
// as nM = ceil(H/128) MMA row tiles (M = 128 units, N = Bt samples, K = 3H).
// (grad_x = dA W_in does not feed the recurrence; it is one GEMM over all B*K
// rows after the loop.)  The A operand, W_rec^T, is the same for every step
// and every block: it is prepared once per call as pre-swizzled 16 KB tiles
// (128 rows x 128 bytes of K) in the workspace and streamed through a ring of
// shared-memory stages with TMA bulk copies (cp.async.bulk, mbarrier
// transaction counts).
// The B operand, dA_k of the Bt samples, is computed by the block itself
// into a K-major swizzled shared-memory tile.
//
// Both kernels are warp-specialised: a producer warp streams the tiles, an
// MMA warp issues the MMAs, eight warps do the cell / elementwise work.  The
// units are split into two halves with their own TMEM accumulators, and the
// stages of a step are ordered so that each half's elementwise work overlaps
// MMAs of the other half (TileSchedule).  Thread <-> unit 128*mt +
// 32*(warp%4) + lane (the TMEM lane quadrant rule).  After step 0 the
// backward's carry read gives grad_h0.
//
// Waits are bounded; a timeout records an error in the device error word.
#include <algorithm>
#include <climits>
#include <vector>

#include "cfc_internal.cuh"
#include "tc_common.cuh"

namespace cfc {
namespace {

constexpr uint32_t kTile = 128 * 128;      // bytes of one A tile (128 rows x one 128-byte K atom)
// A stage holds the tiles of two consecutive K atoms of one M tile (32 KB):
// one full-barrier wait and one commit per 8 MMAs.
constexpr uint32_t kStage = 2 * kTile;
// Byte offset of the tile of K atom a, M tile m in the streamed sequence
// (stage (a/2, m), in stage order a/2-major).
__host__ __device__ __forceinline__ size_t tile_offset(int a, int m, int nM) {
  return ((size_t)(a >> 1) * nM + m) * kStage + (size_t)(a & 1) * kTile;
}
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

// Store EPU = 16 / sizeof(ET) consecutive K elements as one 16-byte unit of
// a swizzled tile row.
template <typename ET>
__device__ __forceinline__ void st_unit(uint8_t* p, const float* v) {
  uint4 w;
  if constexpr (sizeof(ET) == 4) {
    w = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
  } else {
    uint32_t r[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
      r[q] = *reinterpret_cast<const uint32_t*>(&b2);
    }
    w = make_uint4(r[0], r[1], r[2], r[3]);
  }
  *reinterpret_cast<uint4*>(p) = w;
}

// Both tile builders run one thread per 16-byte unit (row i of the tile,
// unit u of its 128-byte K row): 128 x 8 units per tile, 32-bit indices
// (the launchers check the unit count).

// W_rec^T tiles: tile (mt, a) holds rows j = 128*mt .. 128*mt+127 (units)
// and K elements a*EPA .. a*EPA+EPA-1 (EPA = 128 bytes / element), at byte
// offset tile_offset(a, mt, nM), swizzled exactly as in shared memory.
// Consecutive threads take consecutive rows j, so each of a thread's EPU
// loads (one row kk of W_rec each) is coalesced across the warp.
template <typename ET, int MODE>
__global__ void k_prep_wt_tiles(const ET* __restrict__ W_rec, int H, int nM, int nAk, uint8_t* __restrict__ tiles) {
  constexpr int EPU = 16 / sizeof(ET);
  const int H3 = 3 * H;
  const int total = nM * nAk * 1024;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
    const int i = e & 127, u = (e >> 7) & 7, t = e >> 10;   // t = a * nM + mt
    const int mt = t % nM, a = t / nM;
    const int j = mt * 128 + i, k0 = a * (8 * EPU) + u * EPU;
    float v[EPU];
#pragma unroll
    for (int q = 0; q < EPU; ++q)
      v[q] = (j < H && k0 + q < H3) ? ld_operand<MODE>(W_rec + (size_t)(k0 + q) * H + j) : 0.f;
    st_unit<ET>(tiles + tile_offset(a, mt, nM) + tc::sw128_offset(i, u * 16), v);
  }
}

// W_cat tiles of the forward: tile (a, m), m = 3*ub + c, holds the rows of
// head c for units 128*ub + i (i = 0..127) and K elements a*EPA .. +EPA-1 of z,
// at byte offset tile_offset(a, m, nM), swizzled as in shared memory.
// Consecutive threads take consecutive units u of one row, so a warp reads
// four 128-byte runs of [W_in | W_rec] rows and writes four whole tile rows.
template <typename ET, int MODE>
__global__ void k_prep_w_tiles_fwd(const ET* __restrict__ W_in, const ET* __restrict__ W_rec, int n_in,
                                   int H, int nM, int nAk, uint8_t* __restrict__ tiles) {
  constexpr int EPU = 16 / sizeof(ET);
  const int Zc = n_in + H;
  const int total = nM * nAk * 1024;
  for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < total; e += gridDim.x * blockDim.x) {
    const int u = e & 7, i = (e >> 3) & 127, t = e >> 10;     // t = a * nM + m
    const int m = t % nM, a = t / nM;
    const int c = m % 3, ub = m / 3;
    const int unit = ub * 128 + i, k0 = a * (8 * EPU) + u * EPU;
    const size_t row = (size_t)c * H + unit;
    float v[EPU];
#pragma unroll
    for (int q = 0; q < EPU; ++q) {
      const int kk = k0 + q;
      v[q] = 0.f;
      if (unit < H && kk < Zc)
        v[q] = (kk < n_in) ? ld_operand<MODE>(W_in + row * n_in + kk) : ld_operand<MODE>(W_rec + row * H + (kk - n_in));
    }
    st_unit<ET>(tiles + tile_offset(a, m, nM) + tc::sw128_offset(i, u * 16), v);
  }
}

constexpr int kXUnits = 4;                 // prefetched 16-byte x units per epilogue thread
constexpr int kFwdConsumers = 512;         // cell epilogue: warps 0..15 (4 sample groups)
constexpr int kFwdGroups = kFwdConsumers / 128;
constexpr int kFwdProducerWarp = 16;       // W_cat tile stream
constexpr int kFwdMmaWarp = 17;            // MMA issue
constexpr int kFwdThreads = kFwdConsumers + 64;
constexpr int kFwdMaxStages = 12;
constexpr int kMaxSched = 256;             // streamed stages per step

// Order of the streamed stages of one step.  The units are split into two
// halves U0 (unit blocks ub < nU0) and U1 (the rest), each with its own TMEM
// accumulators, so that the epilogue of one half overlaps the MMAs of the
// other:
//   epilogue(k): [acc0] U0 cell, h(U0) -> Z  --zlo-->  [acc1] x_{k+1} -> Z
//                --zx-->  U1 cell, h(U1) -> Z  --zhi-->
//   MMAs(k+1):   U0 stages ordered by the signal their Z atoms need (zlo, zx,
//                zhi), then U1 stages (which also need U1's accumulators
//                read, i.e. zhi); the U1 stages that read atoms holding h(U0)
//                come first, and acc0 is committed right after them, so the
//                U0 epilogue never overwrites Z atoms that an MMA of the step
//                still has to read.
// lvl: 1, 2, 3 = the stage waits for zlo, zx, zhi of the previous step;
// first: the stage is the first of its M tile in the step (the MMA
// overwrites the accumulator).
struct TileSchedule {
  int T = 0, nacc0 = 0, nU0 = 0;
  uint8_t pa[kMaxSched], m[kMaxSched], lvl[kMaxSched], first[kMaxSched];
};

// Named barrier of the epilogue warps only.
__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kFwdConsumers) : "memory");
}

// Bounded mbarrier wait executed by a whole warp: lane 0's observation
// decides for all lanes, so the warp stays converged.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, uint32_t max_polls) {
  for (uint32_t i = 0; i < max_polls; ++i) {
    const int ok = tc::mbar_try_wait(bar, parity) ? 1 : 0;
    if (__shfl_sync(0xffffffffu, ok, 0)) return true;
  }
  return false;
}
__device__ __forceinline__ void mbar_arrive1(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

template <typename ET, int MODE>
__global__ void __launch_bounds__(kFwdThreads, 1)
k_cfc_fwd_tcb(const __grid_constant__ TileSchedule sched, const uint8_t* __restrict__ wtiles,
              const ET* __restrict__ x, const ET* __restrict__ h0, const float* __restrict__ bias,
              const float* __restrict__ dt, int dt_stride, int B, int K, int n_in, int H, int Bt, int nUB,
              int nAk, int nst, uint32_t tmem_cols, ET* __restrict__ h_seq, float* __restrict__ act) {
  constexpr int EPU = 16 / (int)sizeof(ET);
  constexpr int EPA = 128 / (int)sizeof(ET);
  const int Zc = n_in + H, H3 = 3 * H;
  const int nM = 3 * nUB;
  const int Kpad = nAk * EPA;
  const int b0 = blockIdx.x * Bt;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, grp = warp >> 2;
  const int T = sched.T;
  const long long total_tiles = (long long)K * T;
  const bool vec = (n_in % EPU == 0) && (H % EPU == 0);
  const int nU0 = sched.nU0;

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage = sm;                                       // nst x 32 KB
  uint8_t* Zs = sm + (size_t)nst * kStage;                   // nAk x [Bt rows][128 B]
  float* bs = reinterpret_cast<float*>(Zs + (size_t)nAk * Bt * 128);   // [3H]
  float* dts = bs + H3;                                      // [Bt]
  __shared__ uint64_t full[kFwdMaxStages], empty[kFwdMaxStages];
  __shared__ uint64_t acc0, acc1, zsig[3];                   // zsig: zlo, zx, zhi
  __shared__ uint32_t tmem_base;
  __shared__ int err;

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    tc::mbar_init(&acc0, 1);
    tc::mbar_init(&acc1, 1);
    for (int i = 0; i < 3; ++i) tc::mbar_init(&zsig[i], kFwdConsumers / 32);
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, tmem_cols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  volatile int* err_flag = &err;
  if (warp != kFwdProducerWarp) {
    // While the producer starts the tile stream: bias, dt and the z rows of
    // step 0 = [x_0; h0] with zero K padding (16-byte units when vec), then
    // the epilogue and MMA warps meet at named barrier 2.
    constexpr int kPro = kFwdConsumers + 32;
    const int ptid = (warp == kFwdMmaWarp) ? kFwdConsumers + lane : tid;   // 0 .. kPro-1
    for (int e = ptid; e < H3; e += kPro) bs[e] = bias[e];
    for (int e = ptid; e < Bt; e += kPro) dts[e] = (b0 + e < B) ? dt[dt_stride ? b0 + e : 0] : 0.f;
    if (vec) {
      const int upr = Kpad / EPU;
      for (int e = ptid; e < Bt * upr; e += kPro) {
        const int n = e / upr, kk = (e - n * upr) * EPU, bb = b0 + n;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (bb < B && kk < Zc)
          v = __ldg(reinterpret_cast<const uint4*>((kk < n_in) ? x + (long long)bb * K * n_in + kk
                                                              : h0 + (long long)bb * H + (kk - n_in)));
        if constexpr (MODE == CFC_MATH_TF32) {
          v.x = __float_as_uint(round_tf32(__uint_as_float(v.x)));
          v.y = __float_as_uint(round_tf32(__uint_as_float(v.y)));
          v.z = __float_as_uint(round_tf32(__uint_as_float(v.z)));
          v.w = __float_as_uint(round_tf32(__uint_as_float(v.w)));
        }
        *reinterpret_cast<uint4*>(Zs + kmajor_off<ET>(n, kk, Bt)) = v;
      }
    } else {
      for (int e = ptid; e < Bt * Kpad; e += kPro) {
        const int n = e / Kpad, kk = e - n * Kpad, bb = b0 + n;
        float v = 0.f;
        if (bb < B && kk < Zc)
          v = (kk < n_in) ? ld_operand<MODE>(x + (long long)bb * K * n_in + kk)
                          : ld_operand<MODE>(h0 + (long long)bb * H + (kk - n_in));
        st_elem<ET>(Zs + kmajor_off<ET>(n, kk, Bt), v);
      }
    }
    tc::fence_proxy_async_smem();
    asm volatile("bar.sync 2, %0;" ::"n"(kPro) : "memory");
  }

  if (warp == kFwdProducerWarp) {
    // ---- producer warp: the W_cat stages of every step, in schedule order,
    // through the ring; a slot is refilled once the MMAs that read it have
    // committed to its `empty` barrier.
    int st = 0, t = 0;
    uint32_t wrap = 0;
    for (long long g = 0; g < total_tiles; ++g) {
      if (__shfl_sync(0xffffffffu, *err_flag, 0)) break;
      if (wrap > 0 && !mbar_wait_warp(&empty[st], (wrap - 1) & 1u, kMaxPolls)) {
        if (lane == 0) *err_flag = 1;
        break;
      }
      if (lane == 0) {
        expect_tx(&full[st], kStage);
        const uint8_t* src = wtiles + ((size_t)sched.pa[t] * nM + sched.m[t]) * kStage;
        bulk_g2s(stage + (size_t)st * kStage, src, kStage, &full[st]);
      }
      __syncwarp();
      if (++t == T) t = 0;
      if (++st == nst) {
        st = 0;
        ++wrap;
      }
    }
  } else if (warp == kFwdMmaWarp) {
    // ---- MMA warp: D[m] (TMEM columns m*Bt ..) += W_cat stage rows x Z_k^T.
    // After a timed-out wait nothing more is issued; the epilogue's own waits
    // then run out and the host sees the device error word.
    const uint32_t id = tc::idesc(128, (uint32_t)Bt, sizeof(ET) == 4 ? tc::kFmtTF32 : tc::kFmtBF16);
    const uint64_t a_desc0 = tc::sdesc_k_sw128(tc::smem_u32(stage));
    const uint64_t b_desc0 = tc::sdesc_k_sw128(tc::smem_u32(Zs));
    int cst = 0;
    uint32_t cwrap = 0;
    bool ok = true;
    for (int k = 0; k < K && ok; ++k) {
      int waited = (k == 0) ? 3 : 0;
      for (int t = 0; t < T && ok; ++t) {
        while (waited < sched.lvl[t]) {
          if (!mbar_wait_warp(&zsig[waited], (uint32_t)((k - 1) & 1), kMaxPolls)) ok = false;
          ++waited;
        }
        if (ok && !mbar_wait_warp(&full[cst], cwrap & 1u, kMaxPolls)) ok = false;
        if (!ok) {
          if (lane == 0) *err_flag = 1;
          break;
        }
        tc::fence_after_sync();
        {  // operands from the converged warp, one elected lane issues
          const int pa = sched.pa[t];
          const uint32_t d = tmem + (uint32_t)sched.m[t] * (uint32_t)Bt;
          const bool first = sched.first[t] != 0;
          if (tc::elect_one()) {
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              const int a = 2 * pa + sub;
              if (a < nAk) {
                const uint64_t ad = tc::sdesc_advance(a_desc0, (uint32_t)cst * kStage + (uint32_t)sub * kTile);
                const uint64_t bd = tc::sdesc_advance(b_desc0, (uint32_t)(a * Bt * 128));
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const uint32_t accum = (first && sub == 0 && q == 0) ? 0u : 1u;
                  if constexpr (sizeof(ET) == 4) tc::mma_tf32(d, ad + 2 * q, bd + 2 * q, id, accum);
                  else tc::mma_bf16(d, ad + 2 * q, bd + 2 * q, id, accum);
                }
              }
            }
            tc::mma_commit(&empty[cst]);
            if (t == sched.nacc0 - 1) tc::mma_commit(&acc0);
            if (t == T - 1) tc::mma_commit(&acc1);
          }
        }
        __syncwarp();
        if (++cst == nst) {
          cst = 0;
          ++cwrap;
        }
      }
    }
  } else {
    // ---- epilogue warps
    const int xupr = vec ? n_in / EPU : 0;
    const long long sample_stride_act = (long long)K * H3, sample_stride_h = (long long)K * H;
    constexpr int kP = 8;                        // samples per pass
    const int nchunk = Bt / kP;
    bool ok = true;
    // thread <-> unit 128*ub + 32*quad + lane, 8 samples per pass; (ub, sample
    // chunk) pairs of units [ub_lo, ub_hi) go round the sample groups of warps.
    auto cell_pass = [&](int k, int ub_lo, int ub_hi) {
      for (int pidx = ub_lo * nchunk + grp; pidx < ub_hi * nchunk; pidx += kFwdGroups) {
        const int ub = pidx / nchunk, n0 = (pidx - ub * nchunk) * kP;
        const int u = ub * 128 + quad * 32 + lane;
        float af[kP], ag[kP], ah[kP];
        const uint32_t t0 = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(3 * ub * Bt + n0);
        tc::tmem_ld8x3(t0, t0 + (uint32_t)Bt, t0 + 2u * (uint32_t)Bt, af, ag, ah);
        if (u < H) {
          const float bf = bs[u], bg = bs[H + u], bh = bs[2 * H + u];
          const int nvalid = min(kP, B - (b0 + n0));
          float* ap = act + ((long long)(b0 + n0) * K + k) * H3 + u;
          ET* hp = h_seq + ((long long)(b0 + n0) * K + k) * H + u;
          uint8_t* zp = Zs + (size_t)((n_in + u) * (int)sizeof(ET) >> 7) * Bt * 128;
          const uint32_t kb = (uint32_t)(((n_in + u) * (int)sizeof(ET)) & 127);
#pragma unroll
          for (int i = 0; i < kP; ++i) {
            const int n = n0 + i;
            const CellAct c = cell_act(af[i] + bf, ag[i] + bg, ah[i] + bh, dts[n]);
            const float gate = c.gate, g = c.g, hh = c.hh;
            const float h = fmaf(gate, g - hh, hh);
            float hop = 0.f;
            if (i < nvalid) {
              ap[0] = gate;
              ap[H] = g;
              ap[2 * H] = hh;
              stf(hp, h);
              if constexpr (sizeof(ET) == 2) hop = round_bf16(h);
              else hop = round_tf32(h);
            }
            ap += sample_stride_act;
            hp += sample_stride_h;
            if (k + 1 < K) st_elem<ET>(zp + tc::sw128_offset(n, kb), hop);
          }
        }
      }
    };
    // Z writes (generic proxy) become visible to the MMAs (async proxy), the
    // TMEM reads are ordered before the signal, then one arrival per warp.
    auto signal = [&](uint64_t* bar) {
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive1(bar);
    };
    // One warp polls the MMA completion (polling threads slow the tile
    // stream), the epilogue warps meet it at a named barrier.
    auto wait_acc = [&](uint64_t* bar, uint32_t parity) {
      if (warp == 0 && ok && !mbar_wait_warp(bar, parity, kMaxPolls) && lane == 0) *err_flag = 1;
      epi_sync();
      ok = ok && *err_flag == 0;
      tc::fence_after_sync();
    };
    for (int k = 0; k < K; ++k) {
      // x of the next step: raw 16-byte units, stored into Z after all MMAs of step k.
      uint4 xu[kXUnits];
      if (vec) {
#pragma unroll
        for (int q = 0; q < kXUnits; ++q) {
          const int e = tid + q * kFwdConsumers;
          const int n = (xupr > 0) ? e / xupr : 0, kk = (e - n * xupr) * EPU, bb = b0 + n;
          xu[q] = (e < Bt * xupr && k + 1 < K && bb < B)
                      ? __ldg(reinterpret_cast<const uint4*>(x + ((long long)bb * K + k + 1) * n_in + kk))
                      : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      // ---- first half of the units
      wait_acc(&acc0, (uint32_t)(k & 1));
      if (ok) cell_pass(k, 0, nU0);
      if (k + 1 < K) signal(&zsig[0]);
      // ---- all MMAs of step k done: x_{k+1}, then the second half
      wait_acc(&acc1, (uint32_t)(k & 1));
      if (k + 1 < K) {
        if (vec) {
#pragma unroll
          for (int q = 0; q < kXUnits; ++q) {
            const int e = tid + q * kFwdConsumers;
            if (e < Bt * xupr) {
              const int n = e / xupr, kk = (e - n * xupr) * EPU;
              uint4 v = xu[q];
              if constexpr (MODE == CFC_MATH_TF32) {
                v.x = __float_as_uint(round_tf32(__uint_as_float(v.x)));
                v.y = __float_as_uint(round_tf32(__uint_as_float(v.y)));
                v.z = __float_as_uint(round_tf32(__uint_as_float(v.z)));
                v.w = __float_as_uint(round_tf32(__uint_as_float(v.w)));
              }
              *reinterpret_cast<uint4*>(Zs + kmajor_off<ET>(n, kk, Bt)) = v;
            }
          }
        } else {
          for (int e = tid; e < Bt * n_in; e += kFwdConsumers) {
            const int n = e / n_in, kk = e - n * n_in, bb = b0 + n;
            const float v = (bb < B) ? ld_operand<MODE>(x + ((long long)bb * K + k + 1) * n_in + kk) : 0.f;
            st_elem<ET>(Zs + kmajor_off<ET>(n, kk, Bt), v);
          }
        }
        signal(&zsig[1]);
      }
      if (ok) cell_pass(k, nU0, nUB);
      if (k + 1 < K) signal(&zsig[2]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (err) atomicExch(&g_tc_bwd_error, 1);
  if (warp == 0) tc::tmem_dealloc(tmem, tmem_cols);
}

struct FwdPlan {
  int Bt = 0, nUB = 0, nAk = 0, nst = 0;
  uint32_t tmem_cols = 0;
  size_t smem = 0;
  TileSchedule sched;
};

// The stage order of one step (see TileSchedule).  Atom levels: x -> 2 (zx),
// h of U0 -> 1 (zlo), h of U1 -> 3 (zhi), K padding -> 0; a stage (atom
// pair) takes the highest level of its atoms.
bool make_fwd_schedule(int n_in, int H, int es, int nUB, int nAk, TileSchedule* s) {
  const int nP = (nAk + 1) / 2, nM = 3 * nUB;
  if (nP * nM > kMaxSched) return false;
  const int nU0 = std::max(1, nUB / 2);
  const int H0 = std::min(H, 128 * nU0);
  const int epa = 128 / es;
  int lvl[kMaxSched / 2 + 1];
  bool has_u0h[kMaxSched / 2 + 1];
  for (int pa = 0; pa < nP; ++pa) {
    lvl[pa] = 0;
    has_u0h[pa] = false;
    for (int kk = 2 * pa * epa; kk < std::min(2 * (pa + 1) * epa, n_in + H); ++kk) {
      const int l = kk < n_in ? 2 : (kk < n_in + H0 ? 1 : 3);
      lvl[pa] = std::max(lvl[pa], l);
      has_u0h[pa] = has_u0h[pa] || l == 1;
    }
  }
  int t = 0;
  bool seen[3 * 64] = {};
  auto push = [&](int pa, int m, int l) {
    s->pa[t] = (uint8_t)pa;
    s->m[t] = (uint8_t)m;
    s->lvl[t] = (uint8_t)l;
    s->first[t] = seen[m] ? 0 : 1;
    seen[m] = true;
    ++t;
  };
  if (nM > 3 * 64 || nP > 255) return false;
  for (int l = 0; l <= 3; ++l)
    for (int pa = 0; pa < nP; ++pa)
      if (lvl[pa] == l)
        for (int m = 0; m < 3 * nU0; ++m) push(pa, m, std::max(l, 1));
  for (int pa = 0; pa < nP; ++pa)
    if (has_u0h[pa])
      for (int m = 3 * nU0; m < nM; ++m) push(pa, m, 3);
  s->nacc0 = t;
  for (int pa = 0; pa < nP; ++pa)
    if (!has_u0h[pa])
      for (int m = 3 * nU0; m < nM; ++m) push(pa, m, 3);
  s->T = t;
  s->nU0 = nU0;
  return t == nP * nM;
}

bool plan_fwd_stream(const Layout& L, FwdPlan* p) {
  if (L.math == CFC_MATH_FP32) return false;
  const int es = (L.math == CFC_MATH_TF32) ? 4 : 2;
  const int epu = 16 / es;
  const int nUB = (L.H + 127) / 128, nM = 3 * nUB;
  const int nAk = (L.Zc * es + 127) / 128;
  int Bt = (int)(((long long)L.B + kNumSMs - 1) / kNumSMs);
  Bt = std::min(128, std::max(32, (Bt + 15) / 16 * 16));
  auto fixed_for = [&](int bt) { return 1024 + (size_t)nAk * bt * 128 + (size_t)(3 * L.H + bt) * 4 + 256; };
  auto ok = [&](int bt) {
    const bool vec = (L.n_in % epu == 0) && (L.H % epu == 0);
    return fixed_for(bt) + 3 * (size_t)kStage <= kSmemMax && (long long)nM * bt <= 512 &&
           (!vec || (long long)bt * (L.n_in / epu) <= (long long)kXUnits * kFwdConsumers);
  };
  while (Bt > 16 && !ok(Bt)) Bt -= 16;
  if (!ok(Bt)) return false;
  if (!make_fwd_schedule(L.n_in, L.H, es, nUB, nAk, &p->sched)) return false;
  int nst = (int)std::min<size_t>(kFwdMaxStages, (kSmemMax - fixed_for(Bt)) / kStage);
  p->Bt = Bt;
  p->nUB = nUB;
  p->nAk = nAk;
  p->nst = nst;
  uint32_t cols = 32;
  while (cols < (uint32_t)(nM * Bt)) cols <<= 1;
  p->tmem_cols = cols;
  p->smem = fixed_for(Bt) + (size_t)nst * kStage;
  return true;
}

// ---------------------------------------------------------------------------
// Backward K loop with streamed W_rec^T tiles (large batches): one CTA per
// tile of Bt samples.  Per step k (reverse) the elementwise warps turn the
// carry of step k+1 (TMEM) into dA_k of their units -- written to global
// memory and into the K-major B tile dAs (K index c*H + u) -- and the MMAs
// compute carry_k^T = W_rec^T dA_k^T (M tiles of 128 units, N = Bt, K = 3H)
// from the streamed tiles.
//
// Warp-specialised like the forward: warp 16 streams tiles, warp 17 issues
// the MMAs, warps 0..15 do the elementwise work, the units split into halves U0
// (M tiles < nU0) and U1 with their own accumulators:
//   elementwise(s): [acc0 of s-1] U0: carry -> dA_k(U0)  --dlo-->
//                   [acc1 of s-1] U1: carry -> dA_k(U1)  --dhi-->
//   MMAs(s):        U0 stages over atoms of U0 units only (dlo), the other U0
//                   stages (dhi), U1 stages over atoms holding U0 units, acc0,
//                   the remaining U1 stages, acc1.
// So U1's elementwise work overlaps the first U0 MMAs of the step, and U0's
// elementwise work of the next step overlaps the last U1 MMAs.
// ---------------------------------------------------------------------------
constexpr int kBwdElem = 512;              // elementwise warps 0..15 (4 sample groups)
constexpr int kBwdGroups = kBwdElem / 128;
constexpr int kBwdProducerWarp = 16;
constexpr int kBwdMmaWarp = 17;
constexpr int kBwdThreads = kBwdElem + 64;

template <typename ET, int MODE>
__global__ void __launch_bounds__(kBwdThreads, 1)
k_cfc_bwd_tcb(const __grid_constant__ TileSchedule sched, const uint8_t* __restrict__ wtiles,
              const float* __restrict__ dt, int dt_stride, int B, int K, int H, int Bt, int nM, int nAk, int nst,
              uint32_t tmem_cols, const ET* __restrict__ h_seq, const float* __restrict__ grad_h_seq,
              const float* __restrict__ grad_h_last, const float* __restrict__ y,
              const float* __restrict__ act, ET* __restrict__ dA_out, float* __restrict__ grad_h0) {
  const int H3 = 3 * H;
  const int b0 = blockIdx.x * Bt;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, grp = warp >> 2;
  const int T = sched.T;
  const long long total_tiles = (long long)K * T;
  const int nM0 = sched.nU0;

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage = sm;                                   // nst x 32 KB
  uint8_t* dAs = sm + (size_t)nst * kStage;              // nAk x [Bt rows][128 B]
  float* dts = reinterpret_cast<float*>(dAs + (size_t)nAk * Bt * 128);   // [Bt]
  __shared__ uint64_t full[kFwdMaxStages], empty[kFwdMaxStages];
  __shared__ uint64_t acc0, acc1, dsig[2];               // dsig: dlo, dhi
  __shared__ uint32_t tmem_base;
  __shared__ int err;

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    tc::mbar_init(&acc0, 1);
    tc::mbar_init(&acc1, 1);
    for (int i = 0; i < 2; ++i) tc::mbar_init(&dsig[i], kBwdElem / 32);
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, tmem_cols);
  for (int e = tid; e < Bt; e += kBwdThreads) dts[e] = (b0 + e < B) ? dt[dt_stride ? b0 + e : 0] : 0.f;
  // dA tile padding (K beyond 3H) stays zero for the whole launch.
  {
    constexpr int EPA = 128 / sizeof(ET);
    const int Kpad = nAk * EPA;
    for (int e = tid; e < Bt * (Kpad - H3); e += kBwdThreads) {
      const int n = e / (Kpad - H3), kk = H3 + e % (Kpad - H3);
      st_elem<ET>(dAs + kmajor_off<ET>(n, kk, Bt), 0.f);
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  volatile int* err_flag = &err;

  if (warp == kBwdProducerWarp) {
    int st = 0, t = 0;
    uint32_t wrap = 0;
    for (long long g = 0; g < total_tiles; ++g) {
      if (__shfl_sync(0xffffffffu, *err_flag, 0)) break;
      if (wrap > 0 && !mbar_wait_warp(&empty[st], (wrap - 1) & 1u, kMaxPolls)) {
        if (lane == 0) *err_flag = 1;
        break;
      }
      if (lane == 0) {
        expect_tx(&full[st], kStage);
        bulk_g2s(stage + (size_t)st * kStage, wtiles + ((size_t)sched.pa[t] * nM + sched.m[t]) * kStage, kStage,
                 &full[st]);
      }
      __syncwarp();
      if (++t == T) t = 0;
      if (++st == nst) {
        st = 0;
        ++wrap;
      }
    }
  } else if (warp == kBwdMmaWarp) {
    const uint32_t id = tc::idesc(128, (uint32_t)Bt, sizeof(ET) == 4 ? tc::kFmtTF32 : tc::kFmtBF16);
    const uint64_t a_desc0 = tc::sdesc_k_sw128(tc::smem_u32(stage));
    const uint64_t b_desc0 = tc::sdesc_k_sw128(tc::smem_u32(dAs));
    int cst = 0;
    uint32_t cwrap = 0;
    bool ok = true;
    for (int s = 0; s < K && ok; ++s) {
      int waited = 0;
      for (int t = 0; t < T && ok; ++t) {
        while (waited < sched.lvl[t]) {
          if (!mbar_wait_warp(&dsig[waited], (uint32_t)(s & 1), kMaxPolls)) ok = false;
          ++waited;
        }
        if (ok && !mbar_wait_warp(&full[cst], cwrap & 1u, kMaxPolls)) ok = false;
        if (!ok) {
          if (lane == 0) *err_flag = 1;
          break;
        }
        tc::fence_after_sync();
        {  // operands from the converged warp, one elected lane issues
          const int pa = sched.pa[t];
          const uint32_t d = tmem + (uint32_t)sched.m[t] * (uint32_t)Bt;
          const bool first = sched.first[t] != 0;
          if (tc::elect_one()) {
#pragma unroll
            for (int sub = 0; sub < 2; ++sub) {
              const int a = 2 * pa + sub;
              if (a < nAk) {
                const uint64_t ad = tc::sdesc_advance(a_desc0, (uint32_t)cst * kStage + (uint32_t)sub * kTile);
                const uint64_t bd = tc::sdesc_advance(b_desc0, (uint32_t)(a * Bt * 128));
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const uint32_t accum = (first && sub == 0 && q == 0) ? 0u : 1u;
                  if constexpr (sizeof(ET) == 4) tc::mma_tf32(d, ad + 2 * q, bd + 2 * q, id, accum);
                  else tc::mma_bf16(d, ad + 2 * q, bd + 2 * q, id, accum);
                }
              }
            }
            tc::mma_commit(&empty[cst]);
            if (t == sched.nacc0 - 1) tc::mma_commit(&acc0);
            if (t == T - 1) tc::mma_commit(&acc1);
          }
        }
        __syncwarp();
        if (++cst == nst) {
          cst = 0;
          ++cwrap;
        }
      }
    }
  } else {
    // ---- elementwise warps: thread <-> unit 128*mt + 32*quad + lane, 4
    // samples per pass; (M tile, sample chunk) pairs go round the four
    // sample groups of warps (warp >> 2).
    constexpr int kP = 4;                        // samples per pass
    const int nchunk = Bt / kP;
    bool ok = true;
    auto wait_acc = [&](uint64_t* bar, uint32_t parity) {
      if (warp == 0 && ok && !mbar_wait_warp(bar, parity, kMaxPolls) && lane == 0) *err_flag = 1;
      asm volatile("bar.sync 1, %0;" ::"n"(kBwdElem) : "memory");
      ok = ok && *err_flag == 0;
      tc::fence_after_sync();
    };
    auto signal = [&](uint64_t* bar) {
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive1(bar);
    };
    // Saved activations and upstream gradients of one pass, loaded one pass
    // ahead of their use (the first pass of a half before its accumulator
    // wait): none of them depends on the MMAs.
    using VP = float[kP];
    const long long sample_stride = (long long)K * H3;   // act / dA rows of one sample
    const long long up_stride = (long long)K * H;        // grad_h_seq rows of one sample
    auto load_pass = [&](int k, int pidx, VP& ga, VP& gg, VP& gh, VP& gu) {
      const int mt = pidx / nchunk, n0 = (pidx - mt * nchunk) * kP;
      const int u = mt * 128 + quad * 32 + lane;
      const float* ap = act + ((long long)(b0 + n0) * K + k) * H3 + u;
      const float* up = grad_h_seq ? grad_h_seq + ((long long)(b0 + n0) * K + k) * H + u : nullptr;
      const int nvalid = (u < H && k >= 0) ? min(kP, B - (b0 + n0)) : 0;
#pragma unroll
      for (int i = 0; i < kP; ++i) {
        ga[i] = gg[i] = gh[i] = gu[i] = 0.f;
        if (i < nvalid) {
          ga[i] = ap[0];
          gg[i] = ap[H];
          gh[i] = ap[2 * H];
          if (up) gu[i] = up[0];
        }
        ap += sample_stride;
        if (up) up += up_stride;
      }
    };
    auto run_pass = [&](int s, int pidx, const VP& ga, const VP& gg, const VP& gh, const VP& gu) {
      const int k = K - 1 - s;                   // k < 0: grad_h0 read-out
      const int mt = pidx / nchunk, n0 = (pidx - mt * nchunk) * kP;
      const int u = mt * 128 + quad * 32 + lane;
      float dz[kP];
      if (s > 0) {
        tc::tmem_ld4(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(mt * Bt + n0), dz);
      } else {
#pragma unroll
        for (int i = 0; i < kP; ++i) dz[i] = 0.f;
      }
      if (u >= H) return;
      const int nvalid = min(kP, B - (b0 + n0));
      if (k < 0) {
        if (grad_h0) {
#pragma unroll
          for (int i = 0; i < kP; ++i)
            if (i < nvalid) grad_h0[(long long)(b0 + n0 + i) * H + u] = dz[i];
        }
        return;
      }
      // upstream gradient of h_k (only the per-step seeds and the last step's)
      if (grad_h_seq || k == K - 1) {
#pragma unroll
        for (int i = 0; i < kP; ++i) {
          const int bb = b0 + n0 + i;
          if (i < nvalid) {
            const long long row = (long long)bb * K + k;
            float up = gu[i];
            if (k == K - 1) {
              if (grad_h_last) up += grad_h_last[(long long)bb * H + u];
              if (y) up += ldf(h_seq + row * H + u) - y[(long long)bb * H + u];
            }
            dz[i] += up;
          }
        }
      }
      ET* dp = dA_out + ((long long)(b0 + n0) * K + k) * H3 + u;
#pragma unroll
      for (int i = 0; i < kP; ++i) {
        const int n = n0 + i;
        float d0 = 0.f, d1 = 0.f, d2 = 0.f;
        if (i < nvalid) {
          const float delta = dz[i];
          const float gate = ga[i], g = gg[i], hh = gh[i];
          d1 = to_operand<MODE>(delta * gate * (1.f - g * g));
          d2 = to_operand<MODE>(delta * (1.f - gate) * (1.f - hh * hh));
          d0 = to_operand<MODE>(-dts[n] * delta * (g - hh) * gate * (1.f - gate));
          stf(dp, d0);
          stf(dp + H, d1);
          stf(dp + 2 * H, d2);
        }
        dp += sample_stride;
        st_elem<ET>(dAs + kmajor_off<ET>(n, u, Bt), d0);
        st_elem<ET>(dAs + kmajor_off<ET>(n, H + u, Bt), d1);
        st_elem<ET>(dAs + kmajor_off<ET>(n, 2 * H + u, Bt), d2);
      }
    };
    // This thread's passes of M tiles [mt_lo, mt_hi): pidx = mt_lo*nchunk +
    // grp, + kBwdGroups, ...; two input buffers, the next pass always in
    // flight.  Buffer 0 arrives holding the first pass (prefetch()).
    float ga0[kP], gg0[kP], gh0[kP], gu0[kP], ga1[kP], gg1[kP], gh1[kP], gu1[kP];
    auto prefetch = [&](int s, int mt_lo, int mt_hi) {
      const int p = mt_lo * nchunk + grp;
      if (p < mt_hi * nchunk) load_pass(K - 1 - s, p, ga0, gg0, gh0, gu0);
    };
    auto elem = [&](int s, int mt_lo, int mt_hi) {
      const int k = K - 1 - s;
      const int end = mt_hi * nchunk;
      for (int p = mt_lo * nchunk + grp; p < end; p += 2 * kBwdGroups) {
        if (p + kBwdGroups < end) load_pass(k, p + kBwdGroups, ga1, gg1, gh1, gu1);
        run_pass(s, p, ga0, gg0, gh0, gu0);
        if (p + 2 * kBwdGroups < end) load_pass(k, p + 2 * kBwdGroups, ga0, gg0, gh0, gu0);
        if (p + kBwdGroups < end) run_pass(s, p + kBwdGroups, ga1, gg1, gh1, gu1);
      }
    };
    for (int s = 0; s <= K; ++s) {
      prefetch(s, 0, nM0);
      if (s > 0) wait_acc(&acc0, (uint32_t)((s - 1) & 1));
      if (ok) elem(s, 0, nM0);
      if (s < K) signal(&dsig[0]);
      prefetch(s, nM0, nM);
      if (s > 0) wait_acc(&acc1, (uint32_t)((s - 1) & 1));
      if (ok) elem(s, nM0, nM);
      if (s < K) signal(&dsig[1]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (err) atomicExch(&g_tc_bwd_error, 1);
  if (warp == 0) tc::tmem_dealloc(tmem, tmem_cols);
}

// Stage order of one backward step (see k_cfc_bwd_tcb).  K index kk of dA is
// unit kk % H; an atom pair has level 1 if all its units are in U0, else 2.
bool make_bwd_schedule(int H, int es, int nM, int nAk, TileSchedule* s) {
  const int nP = (nAk + 1) / 2;
  if (nP * nM > kMaxSched || nM > 255 || nP > 255) return false;
  const int nM0 = std::max(1, nM / 2);
  const int H0 = std::min(H, 128 * nM0);
  const int epa = 128 / es;
  std::vector<int> lvl(nP, 0);
  std::vector<char> has_u0(nP, 0), seen(nM, 0);
  for (int pa = 0; pa < nP; ++pa)
    for (int kk = 2 * pa * epa; kk < std::min(2 * (pa + 1) * epa, 3 * H); ++kk) {
      const int l = (kk % H) < H0 ? 1 : 2;
      lvl[pa] = std::max(lvl[pa], l);
      if (l == 1) has_u0[pa] = 1;
    }
  int t = 0;
  auto push = [&](int pa, int m, int l) {
    s->pa[t] = (uint8_t)pa;
    s->m[t] = (uint8_t)m;
    s->lvl[t] = (uint8_t)l;
    s->first[t] = seen[m] ? 0 : 1;
    seen[m] = 1;
    ++t;
  };
  for (int l = 0; l <= 2; ++l)
    for (int pa = 0; pa < nP; ++pa)
      if (lvl[pa] == l)
        for (int m = 0; m < nM0; ++m) push(pa, m, std::max(l, 1));
  for (int pa = 0; pa < nP; ++pa)
    if (has_u0[pa])
      for (int m = nM0; m < nM; ++m) push(pa, m, 2);
  s->nacc0 = t;
  for (int pa = 0; pa < nP; ++pa)
    if (!has_u0[pa])
      for (int m = nM0; m < nM; ++m) push(pa, m, 2);
  s->T = t;
  s->nU0 = nM0;
  return t == nP * nM;
}

template <typename ET, int MODE>
cudaError_t launch_fwd_stream(const Layout& L, const FwdPlan& p, const CfcArgs& a, cudaStream_t s) {
  uint8_t* tiles = reinterpret_cast<uint8_t*>(a.ws + L.off_wtt);
  {
    const long long total = (long long)3 * p.nUB * p.nAk * 1024;   // 16-byte tile units
    if (total > INT_MAX) return cudaErrorInvalidValue;
    const int blocks = (int)std::min<long long>((total + 255) / 256, 4 * kNumSMs);
    TraceScope trace("prep_w", s);
    k_prep_w_tiles_fwd<ET, MODE><<<blocks, 256, 0, s>>>(static_cast<const ET*>(a.W_in),
                                                        static_cast<const ET*>(a.W_rec), L.n_in, L.H,
                                                        3 * p.nUB, p.nAk, tiles);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  auto kern = k_cfc_fwd_tcb<ET, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  const int blocks = (L.B + p.Bt - 1) / p.Bt;
  TraceScope trace("cfc_fwd_stream_tc", s);
  kern<<<blocks, kFwdThreads, p.smem, s>>>(p.sched, static_cast<const uint8_t*>(tiles), static_cast<const ET*>(a.x),
                                           static_cast<const ET*>(a.h0), a.b, a.dt, a.dt_stride, L.B, L.K, L.n_in,
                                           L.H, p.Bt, p.nUB, p.nAk, p.nst, p.tmem_cols,
                                           static_cast<ET*>(a.h_seq), reinterpret_cast<float*>(a.ws + L.off_act));
  return cudaGetLastError();
}


struct BwdPlan {
  int Bt = 0, nM = 0, nAk = 0, nst = 0;
  uint32_t tmem_cols = 0;
  size_t smem = 0;
  TileSchedule sched;
};

bool plan_bwd(const Layout& L, BwdPlan* p) {
  if (L.math == CFC_MATH_FP32) return false;
  const int es = (L.math == CFC_MATH_TF32) ? 4 : 2;
  const int nM = (L.H + 127) / 128;
  const int nAk = (L.H3 * es + 127) / 128;
  // Bt: samples per block, the MMA's N: about one block per SM, at least 32.
  int Bt = (int)(((long long)L.B + kNumSMs - 1) / kNumSMs);
  Bt = std::min(128, std::max(32, (Bt + 15) / 16 * 16));
  auto fixed_for = [&](int bt) { return 1024 + (size_t)nAk * bt * 128 + bt * 4 + 256; };
  while (Bt > 16 && (fixed_for(Bt) + 3 * (size_t)kStage > kSmemMax || (long long)nM * Bt > 512)) Bt -= 16;
  if (fixed_for(Bt) + 3 * (size_t)kStage > kSmemMax || (long long)nM * Bt > 512) return false;
  // as many stages as fit (the stream is latency-bound: more tiles in flight)
  const int nst = (int)std::min<size_t>(kFwdMaxStages, (kSmemMax - fixed_for(Bt)) / kStage);
  if (!make_bwd_schedule(L.H, es, nM, nAk, &p->sched)) return false;
  p->Bt = Bt;
  p->nM = nM;
  p->nAk = nAk;
  p->nst = nst;
  uint32_t cols = 32;
  while (cols < (uint32_t)(nM * Bt)) cols <<= 1;
  p->tmem_cols = cols;
  p->smem = fixed_for(Bt) + (size_t)nst * kStage;
  return true;
}

template <typename ET, int MODE>
cudaError_t launch_bwd(const Layout& L, const BwdPlan& p, const CfcArgs& a, cudaStream_t s) {
  uint8_t* tiles = reinterpret_cast<uint8_t*>(a.ws + L.off_wtt);
  cudaError_t e = launch_prep_wt_tiles(L, p.nM, p.nAk, tiles, a.W_rec, s);
  if (e != cudaSuccess) return e;
  auto kern = k_cfc_bwd_tcb<ET, MODE>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  const int grid = (L.B + p.Bt - 1) / p.Bt;
  {
    TraceScope trace("cfc_bwd_tc", s);
    kern<<<grid, kBwdThreads, p.smem, s>>>(p.sched, tiles, a.dt, a.dt_stride, L.B, L.K, L.H, p.Bt, p.nM, p.nAk, p.nst,
                                        p.tmem_cols, static_cast<const ET*>(a.h_seq), a.grad_h_seq, a.grad_h_last,
                                        a.y, reinterpret_cast<const float*>(a.ws + L.off_act),
                                        reinterpret_cast<ET*>(a.ws + L.off_dA), a.grad_h0);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess || !a.grad_x) return e;
  return launch_grad_x_tc(L, a, s);
}

}  // namespace

cudaError_t launch_prep_wt_tiles(const Layout& L, int nM, int nAk, uint8_t* tiles, const void* W_rec, cudaStream_t s) {
  const long long total = (long long)nM * nAk * 1024;   // 16-byte tile units
  if (total > INT_MAX) return cudaErrorInvalidValue;
  const int blocks = (int)std::min<long long>((total + 255) / 256, 4 * kNumSMs);
  TraceScope trace("prep_wt_tiles", s);
  if (L.math == CFC_MATH_TF32)
    k_prep_wt_tiles<float, CFC_MATH_TF32><<<blocks, 256, 0, s>>>(static_cast<const float*>(W_rec), L.H, nM, nAk, tiles);
  else
    k_prep_wt_tiles<__nv_bfloat16, CFC_MATH_BF16>
        <<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(W_rec), L.H, nM, nAk, tiles);
  return cudaGetLastError();
}

size_t tc_bwd_tiles_bytes(int n_in, int n_hid, int math) {
  if (math == CFC_MATH_FP32) return 0;
  const int es = (math == CFC_MATH_TF32) ? 4 : 2;
  // backward: W_rec^T tiles; forward: W_cat tiles (the two are never live at once)
  const size_t bwd = (size_t)((n_hid + 127) / 128) * (((3 * n_hid * es + 127) / 128 + 1) / 2) * kStage;
  const size_t fwd = (size_t)(3 * ((n_hid + 127) / 128)) * ((((n_in + n_hid) * es + 127) / 128 + 1) / 2) * kStage;
  return std::max(bwd, fwd);
}

cudaError_t launch_forward_tc_stream(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  const int choice = kernel_choice();
  if (choice == kCluster || choice == kSimt || choice == kTc) return cudaErrorNotSupported;
  FwdPlan p;
  if (!plan_fwd_stream(L, &p)) return cudaErrorNotSupported;
  if (L.math == CFC_MATH_TF32) return launch_fwd_stream<float, CFC_MATH_TF32>(L, p, a, s);
  return launch_fwd_stream<__nv_bfloat16, CFC_MATH_BF16>(L, p, a, s);
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
  if (a.grad_x && !grad_x_gemm_applies(L)) return cudaErrorNotSupported;
  if (L.math == CFC_MATH_TF32) return launch_bwd<float, CFC_MATH_TF32>(L, p, a, s);
  return launch_bwd<__nv_bfloat16, CFC_MATH_BF16>(L, p, a, s);
}

}  // namespace cfc
