// cfc_tc_solo.cu -- forward and backward K loops of the TF32 / bf16 modes in
// ONE block per tile of samples, for n_hid <= 128, with the recurrent weights
// resident in tensor memory (TMEM).
//
// For n_hid <= 128 the recurrent weights of all three heads fit one SM's TMEM
// (TF32, H = 128: 3 x 128 columns of 128 lanes), so a block can carry its own
// samples through all K steps with no exchange between blocks: no cluster,
// no distributed shared memory, no cluster barrier.  The weights are the A
// operand of every per-step product and are read from TMEM by the MMA, not
// from shared memory: with only 16 samples per block each MMA is small, and
// a 4 KB A tile re-read from shared memory per MMA is what bounds it.
//
// Backward, per step k (reverse):
//   1. elementwise: thread (unit u = TMEM lane, half of the samples) reads
//      the carry of step k+1 from TMEM (zero at k = K-1), adds the upstream
//      seeds, forms dA_k of its unit from the saved activations (loaded one
//      step ahead), writes dA to global memory (for the weight gradient) and
//      into the K-major B tile (rows = samples, K index c*H + u);
//   2. one thread issues the MMAs of carry_k^T = W_rec^T dA_k^T (A = W_rec^T,
//      K = 3H, in TMEM) into TMEM (N = the tile's samples);
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

#include "cfc_internal.cuh"
#include "tc_common.cuh"

namespace cfc {

__device__ int g_tc_solo_error = 0;

namespace {

constexpr int kSoloThreads = 256;          // 8 warps: lane quadrant (warp & 3), sample half (warp >> 2)
constexpr int kSoloBt = 16;                // samples per block (the MMA's N)
constexpr int kSoloHalf = kSoloBt / 2;     // samples per thread
constexpr uint32_t kSoloPolls = 1u << 24;
constexpr size_t kSoloSmemMax = 227 * 1024;
// TMEM: all 512 columns per block; accumulators from column 0, the A operand
// (weights) from column kSoloColA.  The dynamic shared-memory request is at
// least kSoloSmemOne, which keeps a second block off the SM.
constexpr uint32_t kSoloTmemCols = 512;
constexpr uint32_t kSoloColA = 128;
constexpr size_t kSoloSmemOne = 116 * 1024;

// Eight A-operand values of one TMEM lane as 32-bit columns: tf32 one value a
// column, bf16 two (lower K index in the low half).
template <typename ET>
__device__ __forceinline__ uint32_t pack_col(float lo, float hi) {
  if constexpr (sizeof(ET) == 4) {
    return __float_as_uint(lo);
  } else {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
  }
}

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

// The carry of this thread's lane and samples: the sum of the four partial
// chains (TMEM columns 16 j + n).
__device__ __forceinline__ void ld_carry(uint32_t taddr, float (&cz)[kSoloHalf]) {
  float p[4][kSoloHalf];
#pragma unroll
  for (int j = 0; j < 4; ++j) tc::tmem_ld8(taddr + (uint32_t)(j * kSoloBt), p[j]);
#pragma unroll
  for (int i = 0; i < kSoloHalf; ++i) cz[i] = (p[0][i] + p[1][i]) + (p[2][i] + p[3][i]);
}

template <typename ET, int MODE>
__global__ void __launch_bounds__(kSoloThreads, 1)
k_cfc_bwd_solo(const ET* __restrict__ W_rec, const float* __restrict__ dt, int dt_stride, int B, int K, int H,
               int nAk, const ET* __restrict__ h_seq, const float* __restrict__ grad_h_seq,
               const float* __restrict__ grad_h_last, const float* __restrict__ y, const float* __restrict__ act,
               ET* __restrict__ dA_out, float* __restrict__ grad_h0) {
  const int H3 = 3 * H;
  const int b0 = blockIdx.x * kSoloBt;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = (warp & 3) * 32 + lane;            // unit = TMEM lane of this thread
  const int n0 = (warp >> 2) * kSoloHalf;          // first sample of this thread's half
  const int Kpad = nAk * (128 / (int)sizeof(ET));

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* dAs = sm;                               // nAk x [kSoloBt rows (n)][128 B]
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ float dts[kSoloBt];
  __shared__ int err;

  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kSoloTmemCols);
  for (int e = tid; e < kSoloBt * Kpad; e += kSoloThreads) st_el<ET>(dAs + kmaj<ET>(e / Kpad, e % Kpad, kSoloBt), 0.f);
  if (tid < kSoloBt) dts[tid] = (b0 + tid < B) ? dt[dt_stride ? b0 + tid : 0] : 0.f;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  // A operand in TMEM: lane j (output unit), K index kap = c*H + i ->
  // W_rec[c][i][j]; lanes j >= H and K beyond 3H are zero.  The two warps of
  // a lane quadrant fill one half of the nAk*32 columns each, 8 at a time
  // (for a fixed K index the 32 lanes read 32 consecutive floats).
  {
    const int ncols = nAk * 32, half = ncols / 2;
    const int j = u;
    for (int col0 = (warp >> 2) * half; col0 < (warp >> 2) * half + half; col0 += 8) {
      uint32_t r[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int k0 = (sizeof(ET) == 4) ? col0 + t : 2 * (col0 + t);
        const float lo = (j < H && k0 < H3) ? ld_operand<MODE>(W_rec + (long long)k0 * H + j) : 0.f;
        float hi = 0.f;
        if constexpr (sizeof(ET) == 2) hi = (j < H && k0 + 1 < H3) ? ld_operand<MODE>(W_rec + (long long)(k0 + 1) * H + j) : 0.f;
        r[t] = pack_col<ET>(lo, hi);
      }
      tc::tmem_st8(tmem + lane_off + kSoloColA + (uint32_t)col0, r);
    }
    tc::tmem_st_wait();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t taddr = tmem + lane_off + (uint32_t)n0;
  const uint32_t id = tc::idesc(128, (uint32_t)kSoloBt, sizeof(ET) == 4 ? tc::kFmtTF32 : tc::kFmtBF16);
  const bool mine = u < H;

  // Saved activations and per-step seeds of step k for this thread's samples,
  // loaded one step ahead of their use.
  float pg[kSoloHalf], pgg[kSoloHalf], phh[kSoloHalf], pu[kSoloHalf];
  auto load_step = [&](int k) {
#pragma unroll
    for (int i = 0; i < kSoloHalf; ++i) {
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
    float cz[kSoloHalf];
    if (step > 0 && !err) {
      ld_carry(taddr, cz);
    } else {
#pragma unroll
      for (int i = 0; i < kSoloHalf; ++i) cz[i] = 0.f;
    }
    if (mine) {
#pragma unroll
      for (int i = 0; i < kSoloHalf; ++i) {
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
    // ---- 2. carry_k^T = W_rec^T dA_k^T (one thread issues; the next step's
    // activations load meanwhile)
    if (warp == 0 && !err) {
      // K step (a, j) accumulates into partial carry j: four independent
      // chains, summed by the elementwise step
      const uint64_t bd0 = tc::sdesc_k_sw128(tc::smem_u32(dAs));
      for (int a = 0; a < nAk; ++a) {
        const uint64_t bd = tc::sdesc_advance(bd0, (uint32_t)a * (uint32_t)kSoloBt * 128u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t at = tmem + kSoloColA + (uint32_t)(a * 4 + j) * 8u;
          const uint32_t d = tmem + (uint32_t)(j * kSoloBt);
          if constexpr (sizeof(ET) == 4) tc::mma_tf32_ts_w(d, at, bd + 2 * j, id, a != 0);
          else tc::mma_bf16_ts_w(d, at, bd + 2 * j, id, a != 0);
        }
      }
      tc::mma_commit_w(&bar);
    }
    load_step(k - 1);
    // ---- 3. wait for the carry
    if (tid == 0 && !err && !tc::mbar_wait(&bar, (uint32_t)(step & 1), kSoloPolls)) err = 1;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
  }
  // grad_h0 = the carry after step 0
  if (grad_h0) {
    float cz[kSoloHalf];
    if (!err) {
      ld_carry(taddr, cz);
    } else {
#pragma unroll
      for (int i = 0; i < kSoloHalf; ++i) cz[i] = 0.f;
    }
    if (mine) {
#pragma unroll
      for (int i = 0; i < kSoloHalf; ++i) {
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
// Forward K loop in one block per tile of kSoloBt samples (see the file
// comment).  TMEM columns: accumulator set s (s = k & 1) of head c at
// 48 s + 16 c (N = kSoloBt columns), W_rec[c] from kSoloColA + c * nAh * 32.
// Shared memory: W_in of the three heads (A, K-major, nAx atoms each), two
// x tiles (B, rows = samples), the h tile (B).  Warps 0-7 compute the cell
// (lane quadrant warp & 3, sample half warp >> 2); warp 8 only issues the
// MMAs, so that its stalls on a full MMA queue (the look-ahead input part)
// delay no cell work.
// ---------------------------------------------------------------------------
constexpr int kFwdThreads = kSoloThreads + 32;

template <typename ET, int MODE>
__global__ void __launch_bounds__(kFwdThreads, 1)
k_cfc_fwd_solo(const ET* __restrict__ x, const ET* __restrict__ h0, const ET* __restrict__ W_in,
               const ET* __restrict__ W_rec, const float* __restrict__ bias, const float* __restrict__ dt,
               int dt_stride, int B, int K, int n_in, int H, int nAx, int nAh, float* __restrict__ act,
               ET* __restrict__ h_seq) {
  const int H3 = 3 * H;
  const int b0 = blockIdx.x * kSoloBt;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = (warp & 3) * 32 + lane;            // unit = TMEM lane of this thread
  const int n0 = (warp >> 2) * kSoloHalf;
  constexpr int kEl = 128 / (int)sizeof(ET);       // K elements per atom
  const int KpadX = nAx * kEl, KpadH = nAh * kEl;
  const bool mine = u < H;
  // x staging: thread -> sample xn, K indices xk0 + 16 q (q < nq)
  const int xn = tid >> 4, xk0 = tid & 15, nq = KpadX / 16;
  constexpr int kMaxQ = 16;

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* Wi = sm;                                           // head c: c * nAx * 16 KB
  uint8_t* Xs = Wi + (size_t)3 * nAx * 128 * 128;             // buffer s: s * nAx * 2 KB
  uint8_t* Zh = Xs + (size_t)2 * nAx * kSoloBt * 128;         // nAh x 2 KB
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ float dts[kSoloBt];
  __shared__ int err;

  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kSoloTmemCols);

  auto load_x = [&](int k, float (&r)[kMaxQ]) {
    const int bb = b0 + xn;
    const ET* src = x + ((long long)bb * K + k) * n_in;
#pragma unroll
    for (int q = 0; q < kMaxQ; ++q) {
      const int kk = xk0 + 16 * q;
      r[q] = (q < nq && k < K && bb < B && kk < n_in) ? ld_operand<MODE>(src + kk) : 0.f;
    }
  };
  auto store_x = [&](int s, const float (&r)[kMaxQ]) {
    uint8_t* dst = Xs + (size_t)s * nAx * kSoloBt * 128;
#pragma unroll
    for (int q = 0; q < kMaxQ; ++q)
      if (q < nq) st_el<ET>(dst + kmaj<ET>(xn, xk0 + 16 * q, kSoloBt), r[q]);
  };

  // W_in[c] (A, rows = units, K = input features), x_0 and x_1, h_0
  for (int e = tid; e < 3 * 128 * KpadX; e += kFwdThreads) {
    const int c = e / (128 * KpadX), rem = e - c * 128 * KpadX, i = rem / KpadX, kk = rem - i * KpadX;
    const float v = (i < H && kk < n_in) ? ld_operand<MODE>(W_in + ((long long)c * H + i) * n_in + kk) : 0.f;
    st_el<ET>(Wi + (size_t)c * nAx * 128 * 128 + kmaj<ET>(i, kk, 128), v);
  }
  if (tid < kSoloThreads) {
    float r[kMaxQ];
    load_x(0, r);
    store_x(0, r);
    load_x(1, r);
    store_x(1, r);
  }
  for (int e = tid; e < kSoloBt * KpadH; e += kFwdThreads) {
    const int n = e / KpadH, kk = e - n * KpadH, bb = b0 + n;
    const float v = (bb < B && kk < H) ? ld_operand<MODE>(h0 + (long long)bb * H + kk) : 0.f;
    st_el<ET>(Zh + kmaj<ET>(n, kk, kSoloBt), v);
  }
  if (tid < kSoloBt) dts[tid] = (b0 + tid < B) ? dt[dt_stride ? b0 + tid : 0] : 0.f;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  // W_rec[c] into TMEM: lane i (unit), column c * nAh * 32 + kk (tf32) or
  // kk / 2 (bf16) -> W_rec[c][i][kk]; lanes i >= H and kk >= H are zero.  The
  // two warps of a lane quadrant take alternate 8-column chunks.
  if (tid < kSoloThreads) {
    const int ccols = nAh * 32;
    for (int chunk = warp >> 2; chunk < 3 * ccols / 8; chunk += 2) {
      const int col0 = chunk * 8, c = col0 / ccols, cc = col0 - c * ccols;
      const ET* row = W_rec + ((long long)c * H + u) * H;
      uint32_t r[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int k0 = (sizeof(ET) == 4) ? cc + t : 2 * (cc + t);
        const float lo = (mine && k0 < H) ? ld_operand<MODE>(row + k0) : 0.f;
        float hi = 0.f;
        if constexpr (sizeof(ET) == 2) hi = (mine && k0 + 1 < H) ? ld_operand<MODE>(row + k0 + 1) : 0.f;
        r[t] = pack_col<ET>(lo, hi);
      }
      tc::tmem_st8(tmem + lane_off + kSoloColA + (uint32_t)col0, r);
    }
    tc::tmem_st_wait();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t id = tc::idesc(128, (uint32_t)kSoloBt, sizeof(ET) == 4 ? tc::kFmtTF32 : tc::kFmtBF16);
  const uint64_t wd0 = tc::sdesc_k_sw128(tc::smem_u32(Wi));
  const uint64_t xd0 = tc::sdesc_k_sw128(tc::smem_u32(Xs));
  const uint64_t hd0 = tc::sdesc_k_sw128(tc::smem_u32(Zh));
  // input part of step k into accumulator set k & 1 (fresh)
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
          if constexpr (sizeof(ET) == 4) tc::mma_tf32_w(d + c * kSoloBt, ad + 2 * j, bd + 2 * j, id, (a | j) != 0);
          else tc::mma_bf16_w(d + c * kSoloBt, ad + 2 * j, bd + 2 * j, id, (a | j) != 0);
        }
    }
  };
  const bool issuer = warp == kSoloThreads / 32;
  if (issuer) issue_x(0);

  float bc[3];
#pragma unroll
  for (int c = 0; c < 3; ++c) bc[c] = (mine && tid < kSoloThreads) ? bias[c * H + u] : 0.f;

  for (int k = 0; k < K; ++k) {
    // ---- recurrent part of step k onto its input part; then the input part
    // of step k+1 into the other accumulator set
    if (issuer && !err) {
      // the three heads' chains interleaved: consecutive MMAs are independent
      const uint32_t d = tmem + (uint32_t)((k & 1) * 3 * kSoloBt);
      for (int a = 0; a < nAh; ++a) {
        const uint64_t bd = tc::sdesc_advance(hd0, (uint32_t)(a * kSoloBt * 128));
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            const uint32_t at = tmem + kSoloColA + (uint32_t)(c * nAh * 32 + (a * 4 + j) * 8);
            if constexpr (sizeof(ET) == 4) tc::mma_tf32_ts_w(d + c * kSoloBt, at, bd + 2 * j, id, 1u);
            else tc::mma_bf16_ts_w(d + c * kSoloBt, at, bd + 2 * j, id, 1u);
          }
      }
      tc::mma_commit_w(&bar);
      if (k + 1 < K) issue_x(k + 1);
    }
    if (warp < kSoloThreads / 32) {
    float xr[kMaxQ];
    load_x(k + 2, xr);
    // every cell thread waits for the recurrent part of step k itself
    bool ok = !err;
    if (ok && !tc::mbar_wait(&bar, (uint32_t)(k & 1), kSoloPolls)) {
      ok = false;
      err = 1;
    }
    ok = __all_sync(0xffffffffu, ok);
    tc::fence_after_sync();
    // ---- cell of this thread's unit for its samples
    float df[kSoloHalf], dg[kSoloHalf], dh[kSoloHalf];
    if (ok) {
      const uint32_t t0 = tmem + lane_off + (uint32_t)((k & 1) * 3 * kSoloBt + n0);
      tc::tmem_ld8(t0, df);
      tc::tmem_ld8(t0 + (uint32_t)kSoloBt, dg);
      tc::tmem_ld8(t0 + 2u * (uint32_t)kSoloBt, dh);
    } else {
#pragma unroll
      for (int i = 0; i < kSoloHalf; ++i) df[i] = dg[i] = dh[i] = 0.f;
    }
    if (mine) {
#pragma unroll
      for (int i = 0; i < kSoloHalf; ++i) {
        const int n = n0 + i, bb = b0 + n;
        const CellAct ca = cell_act(df[i] + bc[0], dg[i] + bc[1], dh[i] + bc[2], dts[n]);
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

bool plan_bwd_solo(const Layout& L, SoloPlan* p) {
  if (L.math == CFC_MATH_FP32 || L.H > 128) return false;
  const int es = (L.math == CFC_MATH_TF32) ? 4 : 2;
  p->nAk = (L.H3 * es + 127) / 128;
  p->smem = std::max(kSoloSmemOne, 1024 + (size_t)p->nAk * kSoloBt * 128);
  return kSoloColA + (uint32_t)p->nAk * 32u <= kSoloTmemCols;
}

template <typename ET, int MODE>
cudaError_t launch_bwd_solo(const Layout& L, const SoloPlan& p, const CfcArgs& a, cudaStream_t s) {
  auto kern = k_cfc_bwd_solo<ET, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  const int grid = (L.B + kSoloBt - 1) / kSoloBt;
  {
    TraceScope trace("cfc_bwd_solo_tc", s);
    kern<<<grid, kSoloThreads, p.smem, s>>>(static_cast<const ET*>(a.W_rec), a.dt, a.dt_stride, L.B, L.K, L.H,
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
                                       (size_t)p->nAh * kSoloBt * 128);
  return p->smem <= kSoloSmemMax && kSoloColA + 3u * (uint32_t)p->nAh * 32u <= kSoloTmemCols;
}

template <typename ET, int MODE>
cudaError_t launch_fwd_solo(const Layout& L, const SoloFwdPlan& p, const CfcArgs& a, cudaStream_t s) {
  auto kern = k_cfc_fwd_solo<ET, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  const int grid = (L.B + kSoloBt - 1) / kSoloBt;
  TraceScope trace("cfc_fwd_solo_tc", s);
  kern<<<grid, kFwdThreads, p.smem, s>>>(static_cast<const ET*>(a.x), static_cast<const ET*>(a.h0),
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
  if (choice == kAuto && (long long)(L.B + kSoloBt - 1) / kSoloBt > kNumSMs) return cudaErrorNotSupported;
  if (L.math == CFC_MATH_TF32) return launch_fwd_solo<float, CFC_MATH_TF32>(L, p, a, s);
  return launch_fwd_solo<__nv_bfloat16, CFC_MATH_BF16>(L, p, a, s);
}

// Single-block tensor-core backward (TF32 / bf16, n_hid <= 128); with the
// automatic choice, while its grid fits one wave.
cudaError_t launch_backward_solo_tc(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  const int choice = kernel_choice();
  if (choice != kAuto && choice != kSolo) return cudaErrorNotSupported;
  SoloPlan p;
  if (!plan_bwd_solo(L, &p)) return cudaErrorNotSupported;
  if (a.grad_x && !grad_x_gemm_applies(L)) return cudaErrorNotSupported;
  if (choice == kAuto && (long long)(L.B + kSoloBt - 1) / kSoloBt > kNumSMs) return cudaErrorNotSupported;
  if (L.math == CFC_MATH_TF32) return launch_bwd_solo<float, CFC_MATH_TF32>(L, p, a, s);
  return launch_bwd_solo<__nv_bfloat16, CFC_MATH_BF16>(L, p, a, s);
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
