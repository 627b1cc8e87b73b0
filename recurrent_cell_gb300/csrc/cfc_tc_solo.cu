// cfc_tc_solo.cu -- forward and backward K loops of the TF32 / bf16 modes in
// ONE block per tile of samples, for n_hid <= 128, with the recurrent weights
// resident in tensor memory (TMEM).
//
// For n_hid <= 128 the recurrent weights of all three heads fit one SM's TMEM
// (TF32, H = 128: 3 x 128 columns of 128 lanes), so a block can carry its own
// samples through all K steps with no exchange between blocks: no cluster,
// no distributed shared memory, no cluster barrier.  The weights are the A
// operand of every per-step product and are read from TMEM by the MMA (with
// 8 or 16 samples per block each MMA is small and its cost is the 4 KB of A
// it reads; from TMEM that measured faster than from shared memory).  They
// reach TMEM through shared memory and tcgen05.cp.
//
// Backward, per step k (reverse):
//   1. elementwise: thread (unit u = TMEM lane, a group of the samples) reads
//      the carry of step k+1 from TMEM (zero at k = K-1), adds the upstream
//      seeds, forms dA_k of its unit from the saved activations (loaded one
//      step ahead), writes dA to global memory (for the weight gradient) and
//      into the K-major B tile (rows = samples, K index c*H + u);
//   2. one elected lane of warp 0 issues the MMAs of carry_k^T =
//      W_rec^T dA_k^T (A = W_rec^T, K = 3H, in TMEM) into TMEM (N = 16 columns,
//      the tile's samples and zero rows) as one burst;
//   3. the block waits for them; after step 0 the carry is grad_h0.
// grad_x = dA W_in does not feed the recurrence: one GEMM after the loop.
//
// Forward, per step k: the pre-activations of head c are
// A_c = W_in[c] x_k + W_rec[c] h_k (+ b[c] in the epilogue).  The input part
// does not depend on the state, so it is issued one step ahead (W_in in
// shared memory, x_{k+1} staged K-major) into the second of two accumulator
// sets and runs on the tensor cores while the block computes the cell of
// step k; the recurrent part (W_rec in TMEM, h_k the B tile) then accumulates
// onto it.  The cell writes h_{k+1} (global, and the next B tile) and the
// saved activations (gate, g, h~).
// The MMA waits are bounded; a timeout sets the device error word and the
// block keeps its barrier schedule without issuing more work.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "cfc_internal.cuh"
#include "tc_common.cuh"

namespace cfc {

__device__ int g_tc_solo_error = 0;

namespace {

// Cell warps: lane quadrant (warp & 3) = TMEM lanes of the thread's unit,
// sample group (warp >> 2) of HALF samples.  Backward: 16 warps, warp 0 also
// issues the MMAs.  Forward: 8 cell warps and warp 8, which only issues them
// (more cell warps there slowed the issue, which shares warp 0's scheduler).
constexpr int kSoloThreads = 512;                 // backward block
constexpr int kFwdCell = 256;                     // forward cell threads
constexpr int kSoloFwdBlock = kFwdCell + 32;
constexpr int kSoloBt = 16;                       // MMA N: rows of the B tiles, TMEM columns per accumulator
// A block carries 8 or 16 samples (the B tile rows beyond them stay zero),
// so that a small batch still spreads over the SMs: HALF = samples a thread
// = samples a block / (cell warps / 4).
constexpr uint32_t kSoloPolls = 1u << 24;
constexpr size_t kSoloSmemMax = 227 * 1024;
// TMEM: all 512 columns per block; accumulators from column 0, the A operand
// (weights) from column kSoloColA.  The dynamic shared-memory request is at
// least kSoloSmemOne, which keeps a second block off the SM.
constexpr uint32_t kSoloTmemCols = 512;
constexpr uint32_t kSoloColA = 128;
constexpr size_t kSoloSmemOne = 116 * 1024;

template <typename ET>
__device__ __forceinline__ void st_el(uint8_t* p, float v) {
  if constexpr (sizeof(ET) == 4) *reinterpret_cast<float*>(p) = v;
  else *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
}
// Byte offset of operand element (row, kk) in a stack of K atoms of `rows` rows
// (128-byte swizzled K-major atoms).
template <typename ET>
__device__ __forceinline__ uint32_t kmaj(int row, int kk, int rows) {
  const uint32_t kb = (uint32_t)kk * sizeof(ET);
  return (kb >> 7) * (uint32_t)rows * 128u + tc::sw128_offset(row, kb & 127u);
}

// Four (or three) 32x32b TMEM loads of N = 2, 4 or 8 columns of this warp's
// lanes at columns taddr + stride * j, under one wait.
template <int N> struct TmemShape;
template <> struct TmemShape<2> {
  static __device__ __forceinline__ void ld4(uint32_t t, uint32_t st, uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%8];\n"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%2,%3}, [%9];\n"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%4,%5}, [%10];\n"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%6,%7}, [%11];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
        : "r"(t), "r"(t + st), "r"(t + 2 * st), "r"(t + 3 * st)
        : "memory");
  }
  static __device__ __forceinline__ void ld3(uint32_t t, uint32_t st, uint32_t (&r)[6]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%6];\n"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%2,%3}, [%7];\n"
        "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%4,%5}, [%8];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5])
        : "r"(t), "r"(t + st), "r"(t + 2 * st)
        : "memory");
  }
};
template <> struct TmemShape<4> {
  static __device__ __forceinline__ void ld4(uint32_t t, uint32_t st, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%16];\n"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4,%5,%6,%7}, [%17];\n"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%8,%9,%10,%11}, [%18];\n"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%12,%13,%14,%15}, [%19];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(t), "r"(t + st), "r"(t + 2 * st), "r"(t + 3 * st)
        : "memory");
  }
  static __device__ __forceinline__ void ld3(uint32_t t, uint32_t st, uint32_t (&r)[12]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%12];\n"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%4,%5,%6,%7}, [%13];\n"
        "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%8,%9,%10,%11}, [%14];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11])
        : "r"(t), "r"(t + st), "r"(t + 2 * st)
        : "memory");
  }
};
template <> struct TmemShape<8> {
  static __device__ __forceinline__ void ld4(uint32_t t, uint32_t st, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%32];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%33];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%34];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24,%25,%26,%27,%28,%29,%30,%31}, [%35];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(t), "r"(t + st), "r"(t + 2 * st), "r"(t + 3 * st)
        : "memory");
  }
  static __device__ __forceinline__ void ld3(uint32_t t, uint32_t st, uint32_t (&r)[24]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%24];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%25];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%26];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23])
        : "r"(t), "r"(t + st), "r"(t + 2 * st)
        : "memory");
  }
};
template <int N>
__device__ __forceinline__ void tmem_ldx4(uint32_t taddr, uint32_t stride, float (&v)[4][N]) {
  uint32_t r[4 * N];
  TmemShape<N>::ld4(taddr, stride, r);
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < N; ++i) v[j][i] = __uint_as_float(r[N * j + i]);
}
template <int N>
__device__ __forceinline__ void tmem_ldx3(uint32_t taddr, uint32_t stride, float (&v)[3][N]) {
  uint32_t r[3 * N];
  TmemShape<N>::ld3(taddr, stride, r);
#pragma unroll
  for (int j = 0; j < 3; ++j)
#pragma unroll
    for (int i = 0; i < N; ++i) v[j][i] = __uint_as_float(r[N * j + i]);
}

// The carry of this thread's lane and samples: the sum of the four partial
// chains (TMEM columns 16 j + n).
template <int HALF>
__device__ __forceinline__ void ld_carry(uint32_t taddr, float (&cz)[HALF]) {
  float p[4][HALF];
  tmem_ldx4<HALF>(taddr, (uint32_t)kSoloBt, p);
#pragma unroll
  for (int i = 0; i < HALF; ++i) cz[i] = (p[0][i] + p[1][i]) + (p[2][i] + p[3][i]);
}

// Stage rows [0, 128) x K [0, Kpad) of a row-major matrix (row r at
// src + r * ld; rows >= rows_valid and K >= k_valid are zero) as a K-major
// operand of Kpad / (128 B) atoms at dst, rounded to the operand.  All
// nthreads threads of the block take part: lanes run along K (coalesced
// loads, conflict-free stores) and each thread has eight loads in flight.
// Element-wise: the path for rows that are not 16-byte aligned.
template <typename ET, int MODE>
__device__ __forceinline__ void stage_kmajor(uint8_t* dst, const ET* __restrict__ src, int ld, int rows_valid,
                                             int k_valid, int Kpad, int tid, int nthreads) {
  const int tot = 128 * Kpad;
  for (int e0 = tid; e0 < tot; e0 += 8 * nthreads) {
    float v[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int e = e0 + t * nthreads, i = e / Kpad, kk = e - i * Kpad;
      v[t] = (e < tot && i < rows_valid && kk < k_valid) ? ldf(src + (long long)i * ld + kk) : 0.f;
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int e = e0 + t * nthreads, i = e / Kpad, kk = e - i * Kpad;
      if (e < tot) st_el<ET>(dst + kmaj<ET>(i, kk, 128), to_operand<MODE>(v[t]));
    }
  }
}

// The same staging with 16-byte asynchronous copies, for rows whose byte
// length ld * sizeof(ET) is a multiple of 16 (16-byte aligned rows): one
// copy per 16-byte chunk straight into its swizzled place, zero-filled
// where the chunk is partly or wholly outside the valid rows and K.  The
// caller waits (cp_async_wait_all) and, for TF32, rounds the staged values
// (round_staged_tf32) before the tensor cores read them.
template <typename ET>
__device__ __forceinline__ void stage_kmajor_async(uint8_t* dst, const ET* __restrict__ src, int ld, int rows_valid,
                                                   int k_valid, int nA, int tid, int nthreads) {
  constexpr int EPC = 16 / (int)sizeof(ET), EPA = 128 / (int)sizeof(ET);
  const uint32_t d0 = tc::smem_u32(dst);
  for (int q = tid; q < nA * 1024; q += nthreads) {
    const int a = q >> 10, i = (q >> 3) & 127, ch = q & 7, kk = a * EPA + ch * EPC;
    const int nvalid = (i < rows_valid && kk < k_valid) ? min(EPC, k_valid - kk) : 0;
    const ET* g = nvalid ? src + (long long)i * ld + kk : src;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d0 + (uint32_t)a * 16384u +
                                                                         tc::sw128_offset((uint32_t)i, (uint32_t)ch * 16u)),
                 "l"(g), "r"(nvalid * (int)sizeof(ET))
                 : "memory");
  }
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}
// Round nbytes (a multiple of 16) of staged fp32 values to TF32 in place.
__device__ __forceinline__ void round_staged_tf32(uint8_t* p, int nbytes, int tid, int nthreads) {
  for (int q = tid; q < nbytes / 16; q += nthreads) {
    float4 v = reinterpret_cast<float4*>(p)[q];
    v.x = round_tf32(v.x);
    v.y = round_tf32(v.y);
    v.z = round_tf32(v.z);
    v.w = round_tf32(v.w);
    reinterpret_cast<float4*>(p)[q] = v;
  }
}

// Copy the K-major operand staged at src (nA atoms of 128 rows) into TMEM
// columns from tcol (8 columns per K step), issued by the calling warp.
__device__ __forceinline__ void copy_operand_to_tmem(uint32_t tcol, const uint8_t* src, int nA) {
  const uint64_t d0 = tc::sdesc_k_sw128(tc::smem_u32(src));
  for (int a = 0; a < nA; ++a) {
    const uint64_t d = tc::sdesc_advance(d0, (uint32_t)a * 128u * 128u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (tc::elect_one()) tc::tmem_cp_128x256b(tcol + (uint32_t)(a * 4 + j) * 8u, d + 2 * j);
      __syncwarp();
    }
  }
}

template <typename ET, int MODE, int HALF>
__global__ void __launch_bounds__(kSoloThreads, 1)
k_cfc_bwd_solo(const uint8_t* __restrict__ wimg, const float* __restrict__ dt, int dt_stride, int B, int K, int H,
               int nAk, const ET* __restrict__ h_seq, const float* __restrict__ grad_h_seq,
               const float* __restrict__ grad_h_last, const float* __restrict__ y, const float* __restrict__ act,
               ET* __restrict__ dA_out, float* __restrict__ grad_h0) {
  const int H3 = 3 * H;
  constexpr int SPB = 4 * HALF;                    // samples of the block
  const int b0 = blockIdx.x * SPB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = (warp & 3) * 32 + lane;            // unit = TMEM lane of this thread
  const int n0 = (warp >> 2) * HALF;               // first sample of this thread's group
  const int Kpad = nAk * (128 / (int)sizeof(ET));

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* Wt = sm;                                // nAk x [128 rows (j)][128 B]
  uint8_t* dAs = sm + (size_t)nAk * 128 * 128;     // nAk x [kSoloBt rows (n)][128 B]
  __shared__ uint64_t bar, bar_cp, bar_ld;
  __shared__ uint32_t tmem_base;
  __shared__ float dts[kSoloBt];
  __shared__ int err;

  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init(&bar_cp, 1);
    tc::mbar_init(&bar_ld, 1);
    tc::mbar_init_fence();
    err = 0;
    // A operand: the W_rec^T image (row j = output unit, K index kap =
    // c*H + i, swizzled and rounded as in shared memory), 16 KB per atom
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(&bar_ld)),
                 "r"((uint32_t)nAk * 16384u)
                 : "memory");
    for (int a = 0; a < nAk; ++a)
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 16384, [%2];" ::"r"(
                       tc::smem_u32(Wt) + (uint32_t)a * 16384u),
                   "l"(wimg + (size_t)a * 16384), "r"(tc::smem_u32(&bar_ld))
                   : "memory");
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kSoloTmemCols);
  for (int e = tid; e < kSoloBt * Kpad; e += kSoloThreads) st_el<ET>(dAs + kmaj<ET>(e / Kpad, e % Kpad, kSoloBt), 0.f);
  if (tid < kSoloBt) dts[tid] = (tid < SPB && b0 + tid < B) ? dt[dt_stride ? b0 + tid : 0] : 0.f;
  if (tid == 0 && !tc::mbar_wait(&bar_ld, 0, kSoloPolls)) err = 1;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  const bool mine = u < H;
  const uint32_t taddr = tmem + lane_off + (uint32_t)n0;
  const uint32_t id = tc::idesc(128, (uint32_t)kSoloBt, sizeof(ET) == 4 ? tc::kFmtTF32 : tc::kFmtBF16);
  // The staged A operand into TMEM (columns kSoloColA + 8 s for K step s),
  // where the MMAs read it; the copies complete before the first MMA.
  if (warp == 0) {
    copy_operand_to_tmem(tmem + kSoloColA, Wt, nAk);
    tc::mma_commit_w(&bar_cp);
    if (!tc::mbar_wait(&bar_cp, 0, kSoloPolls) && lane == 0) err = 1;
    __syncwarp();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // Saved activations and per-step seeds of step k for this thread's samples,
  // loaded one step ahead of their use.
  float pg[HALF], pgg[HALF], phh[HALF], pu[HALF];
  auto load_step = [&](int k) {
#pragma unroll
    for (int i = 0; i < HALF; ++i) {
      pg[i] = pgg[i] = phh[i] = pu[i] = 0.f;
      const int bb = b0 + n0 + i;
      if (mine && k >= 0 && bb < B) {
        const long long row = (long long)bb * K + k;
        pg[i] = act[row * H3 + u];
        pgg[i] = act[row * H3 + H + u];
        phh[i] = act[row * H3 + 2 * H + u];
        if (grad_h_seq) pu[i] = grad_h_seq[row * H + u];
      }
    }
  };
  load_step(K - 1);

  for (int step = 0; step < K; ++step) {
    const int k = K - 1 - step;
    // ---- 1. dA_k of this thread's unit and samples
    float cz[HALF];
    if (step > 0 && !err) {
      ld_carry<HALF>(taddr, cz);
    } else {
#pragma unroll
      for (int i = 0; i < HALF; ++i) cz[i] = 0.f;
    }
    if (mine) {
#pragma unroll
      for (int i = 0; i < HALF; ++i) {
        const int n = n0 + i, bb = b0 + n;
        float d0 = 0.f, d1 = 0.f, d2 = 0.f;
        if (bb < B) {
          float delta = cz[i] + pu[i];
          if (k == K - 1) {
            if (grad_h_last) delta += grad_h_last[(long long)bb * H + u];
            if (y) delta += ldf(h_seq + ((long long)bb * K + k) * H + u) - y[(long long)bb * H + u];
          }
          const float gate = pg[i], g = pgg[i], hh = phh[i];
          d1 = to_operand<MODE>(delta * gate * (1.f - g * g));
          d2 = to_operand<MODE>(delta * (1.f - gate) * (1.f - hh * hh));
          d0 = to_operand<MODE>(-dts[n] * delta * (g - hh) * gate * (1.f - gate));
          const long long row = (long long)bb * K + k;
          stf(dA_out + row * H3 + u, d0);
          stf(dA_out + row * H3 + H + u, d1);
          stf(dA_out + row * H3 + 2 * H + u, d2);
        }
        st_el<ET>(dAs + kmaj<ET>(n, u, kSoloBt), d0);
        st_el<ET>(dAs + kmaj<ET>(n, H + u, kSoloBt), d1);
        st_el<ET>(dAs + kmaj<ET>(n, 2 * H + u, kSoloBt), d2);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // ---- 2. carry_k^T = W_rec^T dA_k^T (warp 0 issues; the next step's
    // activations load meanwhile)
    if (warp == 0 && !err) {
      // K step (a, j) accumulates into partial carry j: four independent
      // chains, summed by the elementwise step.  One elected lane issues the
      // step's MMAs back to back.
      const uint64_t bd0 = tc::sdesc_k_sw128(tc::smem_u32(dAs));
      if (tc::elect_one()) {
        for (int a = 0; a < nAk; ++a) {
          const uint64_t bd = tc::sdesc_advance(bd0, (uint32_t)a * (uint32_t)kSoloBt * 128u);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t at = tmem + kSoloColA + (uint32_t)(a * 4 + j) * 8u;
            const uint32_t d = tmem + (uint32_t)(j * kSoloBt);
            if constexpr (sizeof(ET) == 4) tc::mma_tf32_ts(d, at, bd + 2 * j, id, a != 0);
            else tc::mma_bf16_ts(d, at, bd + 2 * j, id, a != 0);
          }
        }
        tc::mma_commit(&bar);
      }
      __syncwarp();
    }
    load_step(k - 1);
    // ---- 3. wait for the carry
    if (tid == 0 && !err && !tc::mbar_wait(&bar, (uint32_t)(step & 1), kSoloPolls)) err = 1;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  }
  // grad_h0 = the carry after step 0
  {
    float cz[HALF];
    if (!err) {
      ld_carry<HALF>(taddr, cz);
    } else {
#pragma unroll
      for (int i = 0; i < HALF; ++i) cz[i] = 0.f;
    }
    if (mine && grad_h0) {
#pragma unroll
      for (int i = 0; i < HALF; ++i) {
        const int bb = b0 + n0 + i;
        if (bb < B) grad_h0[(long long)bb * H + u] = cz[i];
      }
    }
  }
  if (err && tid == 0) atomicExch(&g_tc_solo_error, 1);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kSoloTmemCols);
}

// ---------------------------------------------------------------------------
// Forward K loop in one block per tile of 8 or 16 samples (see the file
// comment).  TMEM columns: accumulator set s (s = k & 1) of head c at
// 48 s + 16 c (N = kSoloBt columns), W_rec[c] from kSoloColA + c * nAh * 32.
// Shared memory: W_in of the three heads (A, K-major, nAx atoms each), two
// x tiles (B, rows = samples), the h tile (B), the W_rec staging buffer.
// Warps 0-7 compute the cell (lane quadrant warp & 3, sample half
// warp >> 2); warp 8 only issues the MMAs (one elected lane), so that its
// stalls on the input part's MMAs (A from shared memory, slower to issue)
// delay no cell work.
// ---------------------------------------------------------------------------
template <typename ET, int MODE, int HALF>
__global__ void __launch_bounds__(kSoloFwdBlock, 1)
k_cfc_fwd_solo(const ET* __restrict__ x, const ET* __restrict__ h0, const ET* __restrict__ W_in,
               const ET* __restrict__ W_rec, const float* __restrict__ bias, const float* __restrict__ dt,
               int dt_stride, int B, int K, int n_in, int H, int nAx, int nAh, float* __restrict__ act,
               ET* __restrict__ h_seq) {
  const int H3 = 3 * H;
  constexpr int SPB = 2 * HALF;                    // samples of the block
  const int b0 = blockIdx.x * SPB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = (warp & 3) * 32 + lane;            // unit = TMEM lane of this thread
  const int n0 = (warp >> 2) * HALF;
  constexpr int kEl = 128 / (int)sizeof(ET);       // K elements per atom
  const int KpadX = nAx * kEl, KpadH = nAh * kEl;
  const bool cell = warp < kFwdCell / 32;
  const bool mine = cell && u < H;
  // x staging: thread -> sample row xn (rows < kSoloBt; samples < SPB are
  // loaded, the other rows stay zero), K indices xk0 + 16 q (q < nq)
  const int xn = tid >> 4, xk0 = tid & 15, nq = KpadX / 16;
  constexpr int kMaxQ = 16;

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* Wi = sm;                                           // head c: c * nAx * 16 KB
  uint8_t* Xs = Wi + (size_t)3 * nAx * 128 * 128;             // buffer s: s * nAx * 2 KB
  uint8_t* Zh = Xs + (size_t)2 * nAx * kSoloBt * 128;         // nAh x 2 KB
  uint8_t* Wst = Zh + (size_t)nAh * kSoloBt * 128;            // W_rec[c] staging: nAh x 16 KB
  __shared__ uint64_t bar, bar_cp;
  __shared__ uint32_t tmem_base;
  __shared__ float dts[kSoloBt];
  __shared__ int err;

  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init(&bar_cp, 1);
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kSoloTmemCols);

  // x rows are kept as stored (raw) in registers until they are staged, so
  // that the loads of step k+2 stay in flight through step k.
  auto load_x = [&](int k, ET (&r)[kMaxQ]) {
    const int bb = b0 + xn;
    const ET* src = x + ((long long)bb * K + k) * n_in;
#pragma unroll
    for (int q = 0; q < kMaxQ; ++q) {
      const int kk = xk0 + 16 * q;
      r[q] = (q < nq && k < K && xn < SPB && bb < B && kk < n_in) ? src[kk] : ET(0.f);
    }
  };
  auto store_x = [&](int s, const ET (&r)[kMaxQ]) {
    if (xn >= kSoloBt) return;                     // the tile has kSoloBt rows
    uint8_t* dst = Xs + (size_t)s * nAx * kSoloBt * 128;
#pragma unroll
    for (int q = 0; q < kMaxQ; ++q)
      if (q < nq) st_el<ET>(dst + kmaj<ET>(xn, xk0 + 16 * q, kSoloBt), to_operand<MODE>((float)r[q]));
  };

  // W_rec[c] (rows = units, K = state) goes to TMEM head by head through
  // one staging buffer (copy of head c overlaps the staging of what
  // follows); W_in[c] (rows = units, K = input features) stays in shared
  // memory; then x_0, x_1 and h_0.
  // 16-byte-aligned rows take the asynchronous 16-byte path
  const bool vrec = (H * (int)sizeof(ET)) % 16 == 0, vin = (n_in * (int)sizeof(ET)) % 16 == 0;
  constexpr bool kTf32 = MODE == CFC_MATH_TF32;
  tc::fence_before_sync();
  __syncthreads();                                   // TMEM address visible
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const bool issuer = warp == kFwdCell / 32;
  for (int c = 0; c < 3; ++c) {
    if (c > 0) {                                     // staging buffer free again
      if (tid == 0 && !tc::mbar_wait(&bar_cp, (uint32_t)((c - 1) & 1), kSoloPolls)) err = 1;
      tc::fence_before_sync();
      __syncthreads();
      tc::fence_after_sync();
    }
    const ET* wr = W_rec + (long long)c * H * H;
    if (vrec) stage_kmajor_async<ET>(Wst, wr, H, H, H, nAh, tid, kSoloFwdBlock);
    else stage_kmajor<ET, MODE>(Wst, wr, H, H, H, KpadH, tid, kSoloFwdBlock);
    if (c == 0)
      for (int cc = 0; cc < 3; ++cc) {
        uint8_t* wi = Wi + (size_t)cc * nAx * 128 * 128;
        const ET* gi = W_in + (long long)cc * H * n_in;
        if (vin) stage_kmajor_async<ET>(wi, gi, n_in, H, n_in, nAx, tid, kSoloFwdBlock);
        else stage_kmajor<ET, MODE>(wi, gi, n_in, H, n_in, KpadX, tid, kSoloFwdBlock);
      }
    cp_async_wait_all();
    if (kTf32 && (vrec || (c == 0 && vin))) {
      __syncthreads();
      if (vrec) round_staged_tf32(Wst, nAh * 16384, tid, kSoloFwdBlock);
      if (c == 0 && vin) round_staged_tf32(Wi, 3 * nAx * 16384, tid, kSoloFwdBlock);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (issuer) {
      copy_operand_to_tmem(tmem + kSoloColA + (uint32_t)(c * nAh * 32), Wst, nAh);
      tc::mma_commit_w(&bar_cp);
    }
  }
  if (cell) {
    ET r0[kMaxQ], r1[kMaxQ];
    load_x(0, r0);
    load_x(1, r1);
    store_x(0, r0);
    store_x(1, r1);
  }
  {
    const int tot = kSoloBt * KpadH;
    for (int e0 = tid; e0 < tot; e0 += 8 * kSoloFwdBlock) {
      float v[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int e = e0 + t * kSoloFwdBlock;
        const int n = e / KpadH, kk = e - n * KpadH, bb = b0 + n;
        v[t] = (e < tot && n < SPB && bb < B && kk < H) ? ldf(h0 + (long long)bb * H + kk) : 0.f;
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int e = e0 + t * kSoloFwdBlock;
        const int n = e / KpadH, kk = e - n * KpadH;
        if (e < tot) st_el<ET>(Zh + kmaj<ET>(n, kk, kSoloBt), to_operand<MODE>(v[t]));
      }
    }
  }
  if (tid < kSoloBt) dts[tid] = (tid < SPB && b0 + tid < B) ? dt[dt_stride ? b0 + tid : 0] : 0.f;
  if (tid == 0 && !tc::mbar_wait(&bar_cp, 0u, kSoloPolls)) err = 1;   // the copy of head 2
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t id = tc::idesc(128, (uint32_t)kSoloBt, sizeof(ET) == 4 ? tc::kFmtTF32 : tc::kFmtBF16);
  const uint64_t wd0 = tc::sdesc_k_sw128(tc::smem_u32(Wi));
  const uint64_t xd0 = tc::sdesc_k_sw128(tc::smem_u32(Xs));
  const uint64_t hd0 = tc::sdesc_k_sw128(tc::smem_u32(Zh));
  // input part of step k into accumulator set k & 1 (fresh); called by the
  // elected lane of the issuing warp
  auto issue_x = [&](int k) {
    const uint32_t d = tmem + (uint32_t)((k & 1) * 3 * kSoloBt);
    const uint64_t xd = tc::sdesc_advance(xd0, (uint32_t)((k & 1) * nAx * kSoloBt * 128));
    for (int a = 0; a < nAx; ++a) {
      const uint64_t bd = tc::sdesc_advance(xd, (uint32_t)(a * kSoloBt * 128));
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          const uint64_t ad = tc::sdesc_advance(wd0, (uint32_t)((c * nAx + a) * 128 * 128));
          if constexpr (sizeof(ET) == 4) tc::mma_tf32(d + c * kSoloBt, ad + 2 * j, bd + 2 * j, id, (a | j) != 0);
          else tc::mma_bf16(d + c * kSoloBt, ad + 2 * j, bd + 2 * j, id, (a | j) != 0);
        }
    }
  };
  if (issuer) {
    if (tc::elect_one()) issue_x(0);
    __syncwarp();
  }

  float bc[3];
#pragma unroll
  for (int c = 0; c < 3; ++c) bc[c] = mine ? bias[c * H + u] : 0.f;

  for (int k = 0; k < K; ++k) {
    // ---- recurrent part of step k onto its input part; then the input part
    // of step k+1 into the other accumulator set
    if (issuer && !err) {
      // the three heads' chains interleaved: consecutive MMAs are independent;
      // one elected lane issues the step's MMAs back to back
      const uint32_t d = tmem + (uint32_t)((k & 1) * 3 * kSoloBt);
      if (tc::elect_one()) {
        for (int a = 0; a < nAh; ++a) {
          const uint64_t bd = tc::sdesc_advance(hd0, (uint32_t)(a * kSoloBt * 128));
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int c = 0; c < 3; ++c) {
              const uint32_t at = tmem + kSoloColA + (uint32_t)(c * nAh * 32 + (a * 4 + j) * 8);
              if constexpr (sizeof(ET) == 4) tc::mma_tf32_ts(d + c * kSoloBt, at, bd + 2 * j, id, 1u);
              else tc::mma_bf16_ts(d + c * kSoloBt, at, bd + 2 * j, id, 1u);
            }
        }
        tc::mma_commit(&bar);
        if (k + 1 < K) issue_x(k + 1);
      }
      __syncwarp();
    }
    if (cell) {
    ET xr[kMaxQ];
    load_x(k + 2, xr);
    // one cell thread waits for the recurrent part of step k and releases
    // the cell warps at a barrier of their own (the issuing warp, still
    // issuing the next input part, is not held)
    if (tid == 0 && !err && !tc::mbar_wait(&bar, (uint32_t)(k & 1), kSoloPolls)) err = 1;
    tc::fence_before_sync();
    asm volatile("bar.sync 1, %0;" ::"n"(kFwdCell) : "memory");
    tc::fence_after_sync();
    const bool ok = !err;
    // ---- cell of this thread's unit for its samples
    float dd[3][HALF];
    if (ok) {
      tmem_ldx3<HALF>(tmem + lane_off + (uint32_t)((k & 1) * 3 * kSoloBt + n0), (uint32_t)kSoloBt, dd);
    } else {
#pragma unroll
      for (int i = 0; i < HALF; ++i) dd[0][i] = dd[1][i] = dd[2][i] = 0.f;
    }
    if (mine) {
#pragma unroll
      for (int i = 0; i < HALF; ++i) {
        const int n = n0 + i, bb = b0 + n;
        const CellAct ca = cell_act(dd[0][i] + bc[0], dd[1][i] + bc[1], dd[2][i] + bc[2], dts[n]);
        const float h = fmaf(ca.gate, ca.g - ca.hh, ca.hh);
        float hop = 0.f;
        if (bb < B) {
          const long long row = (long long)bb * K + k;
          act[row * H3 + u] = ca.gate;
          act[row * H3 + H + u] = ca.g;
          act[row * H3 + 2 * H + u] = ca.hh;
          stf(h_seq + row * H + u, h);
          if constexpr (sizeof(ET) == 2) hop = round_bf16(h);   // the stored bf16 state
          else hop = round_tf32(h);
        }
        if (k + 1 < K) st_el<ET>(Zh + kmaj<ET>(n, u, kSoloBt), hop);
      }
    }
    // x_{k+2} into the tile the input part of step k has finished reading
    if (k + 2 < K) store_x(k & 1, xr);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  }
  if (err && tid == 0) atomicExch(&g_tc_solo_error, 1);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kSoloTmemCols);
}

struct SoloPlan {
  int nAk = 0;
  size_t smem = 0;
};

// Samples a block: 8 while that grid fits one wave, else 16.
// CFC_SOLO_TILE=8 or 16 overrides the choice.
int solo_tile(int B) {
  if (const char* v = getenv("CFC_SOLO_TILE")) {
    if (strcmp(v, "8") == 0) return 8;
    if (strcmp(v, "16") == 0) return 16;
  }
  return (B + 7) / 8 <= kNumSMs ? 8 : 16;
}

bool plan_bwd_solo(const Layout& L, SoloPlan* p) {
  if (L.math == CFC_MATH_FP32 || L.H > 128) return false;
  const int es = (L.math == CFC_MATH_TF32) ? 4 : 2;
  p->nAk = (L.H3 * es + 127) / 128;
  p->smem = std::max(kSoloSmemOne, 1024 + (size_t)p->nAk * 128 * 128 + (size_t)p->nAk * kSoloBt * 128);
  return p->smem <= kSoloSmemMax && kSoloColA + (uint32_t)p->nAk * 32u <= kSoloTmemCols;
}

template <typename ET, int MODE, int HALF>
cudaError_t launch_bwd_solo(const Layout& L, const SoloPlan& p, const CfcArgs& a, cudaStream_t s) {
  // W_rec^T image (one M tile: nAk consecutive 16 KB atoms)
  uint8_t* wimg = reinterpret_cast<uint8_t*>(a.ws + L.off_wtt);
  cudaError_t e = launch_prep_wt_tiles(L, 1, p.nAk, wimg, a.W_rec, s);
  if (e != cudaSuccess) return e;
  auto kern = k_cfc_bwd_solo<ET, MODE, HALF>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  const int grid = (L.B + 4 * HALF - 1) / (4 * HALF);
  {
    TraceScope trace("cfc_bwd_solo_tc", s);
    kern<<<grid, kSoloThreads, p.smem, s>>>(wimg, a.dt, a.dt_stride, L.B, L.K, L.H,
                                            p.nAk, static_cast<const ET*>(a.h_seq), a.grad_h_seq,
                                            a.grad_h_last, a.y, reinterpret_cast<const float*>(a.ws + L.off_act),
                                            reinterpret_cast<ET*>(a.ws + L.off_dA), a.grad_h0);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess || !a.grad_x) return e;
  return launch_grad_x_tc(L, a, s);
}

struct SoloFwdPlan {
  int nAh = 0, nAx = 0;
  size_t smem = 0;
};

bool plan_fwd_solo(const Layout& L, SoloFwdPlan* p) {
  if (L.math == CFC_MATH_FP32 || L.H > 128) return false;
  const int es = (L.math == CFC_MATH_TF32) ? 4 : 2;
  p->nAh = (L.H * es + 127) / 128;
  p->nAx = (L.n_in * es + 127) / 128;
  // x staging: 16 samples x nAx atoms over 256 threads, at most 16 a thread
  if (p->nAx * (128 / es) / 16 > 16) return false;
  p->smem = std::max(kSoloSmemOne, 1024 + (size_t)3 * p->nAx * 128 * 128 + (size_t)2 * p->nAx * kSoloBt * 128 +
                                       (size_t)p->nAh * kSoloBt * 128 + (size_t)p->nAh * 128 * 128);
  return p->smem <= kSoloSmemMax && kSoloColA + 3u * (uint32_t)p->nAh * 32u <= kSoloTmemCols;
}

template <typename ET, int MODE, int HALF>
cudaError_t launch_fwd_solo(const Layout& L, const SoloFwdPlan& p, const CfcArgs& a, cudaStream_t s) {
  auto kern = k_cfc_fwd_solo<ET, MODE, HALF>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  const int grid = (L.B + 2 * HALF - 1) / (2 * HALF);
  TraceScope trace("cfc_fwd_solo_tc", s);
  kern<<<grid, kSoloFwdBlock, p.smem, s>>>(static_cast<const ET*>(a.x), static_cast<const ET*>(a.h0),
                                          static_cast<const ET*>(a.W_in), static_cast<const ET*>(a.W_rec), a.b, a.dt,
                                          a.dt_stride, L.B, L.K, L.n_in, L.H, p.nAx, p.nAh,
                                          reinterpret_cast<float*>(a.ws + L.off_act), static_cast<ET*>(a.h_seq));
  return cudaGetLastError();
}

}  // namespace

// Single-block tensor-core forward (TF32 / bf16, n_hid <= 128); with the
// automatic choice, while its grid fits one wave.
cudaError_t launch_forward_solo_tc(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  const int choice = kernel_choice();
  if (choice != kAuto && choice != kSolo) return cudaErrorNotSupported;
  SoloFwdPlan p;
  if (!plan_fwd_solo(L, &p)) return cudaErrorNotSupported;
  const int tile = solo_tile(L.B);
  if (choice == kAuto && (long long)(L.B + tile - 1) / tile > kNumSMs) return cudaErrorNotSupported;
  if (L.math == CFC_MATH_TF32)
    return tile == 8 ? launch_fwd_solo<float, CFC_MATH_TF32, 4>(L, p, a, s)
                     : launch_fwd_solo<float, CFC_MATH_TF32, 8>(L, p, a, s);
  return tile == 8 ? launch_fwd_solo<__nv_bfloat16, CFC_MATH_BF16, 4>(L, p, a, s)
                   : launch_fwd_solo<__nv_bfloat16, CFC_MATH_BF16, 8>(L, p, a, s);
}

// Single-block tensor-core backward (TF32 / bf16, n_hid <= 128); with the
// automatic choice, while its grid fits one wave.
cudaError_t launch_backward_solo_tc(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  const int choice = kernel_choice();
  if (choice != kAuto && choice != kSolo) return cudaErrorNotSupported;
  SoloPlan p;
  if (!plan_bwd_solo(L, &p)) return cudaErrorNotSupported;
  if (a.grad_x && !grad_x_gemm_applies(L)) return cudaErrorNotSupported;
  const int tile = solo_tile(L.B);
  if (choice == kAuto && (long long)(L.B + tile - 1) / tile > kNumSMs) return cudaErrorNotSupported;
  if (L.math == CFC_MATH_TF32)
    return tile == 8 ? launch_bwd_solo<float, CFC_MATH_TF32, 2>(L, p, a, s)
                     : launch_bwd_solo<float, CFC_MATH_TF32, 4>(L, p, a, s);
  return tile == 8 ? launch_bwd_solo<__nv_bfloat16, CFC_MATH_BF16, 2>(L, p, a, s)
                   : launch_bwd_solo<__nv_bfloat16, CFC_MATH_BF16, 4>(L, p, a, s);
}

int read_tc_solo_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_tc_solo_error, sizeof(int)) != cudaSuccess) return CFC_ERR_DEVICE;
  if (clear && v) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_tc_solo_error, &zero, sizeof(int)) != cudaSuccess) return CFC_ERR_DEVICE;
  }
  return v;
}

}  // namespace cfc
