// cfc_tc.cu -- tensor-core (tcgen05) gradient contraction of the TF32 and
// bf16 modes.
//
//   out[s][pack(m, j)] = sum_{rows r of block s} dA[r][m] * z[r][j]
//
// with z_r = [x_r; h_r; 1] (h_r the state entering row r's step) and m over
// the 3H stacked head rows.  As a GEMM: D[m, j] = A[m, r] B[j, r]^T with the
// reduction r as the MMA's K dimension.  Both operands live in HBM with r as
// the outer index (dA [R][3H], x [R][n_in], h_seq [R][H]), so each 128-byte
// K chunk (32 TF32 or 64 bf16 rows) is transposed by the staging threads
// into K-major, 128B-swizzled shared-memory tiles: 16-byte units of 4 (TF32)
// or 8 (bf16) consecutive rows of one column, read with warp-coalesced loads.
//
// Block = (M block of 128 rows of 3H, N block of NB columns of z, row block
// s).  Per chunk: all threads store the chunk that was loaded into registers
// during the previous iteration, issue the loads of the next chunk, and one
// thread issues 4 MMAs (K = 32 bytes each) into the fp32 accumulator in TMEM
// and commits them to the stage's mbarrier; a stage is refilled only after
// its mbarrier reports the MMAs that read it complete.  The epilogue reads the
// accumulator with tcgen05.ld (warp w -> lanes 32*(w%4) ...) and writes the
// packed per-sample layout.
//
// Every mbarrier wait is bounded; on timeout the kernel records an error in
// g_cfc_device_error, stops issuing work, waits (bounded) for MMAs already in
// flight and frees its TMEM.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "cfc_internal.cuh"
#include "tc_common.cuh"

namespace cfc {

__device__ int g_cfc_device_error = 0;

namespace {

constexpr int kTcThreads = 256;
constexpr int kStages = 2;
constexpr int kMaxNB = 208;               // N block (columns of z), multiple of 16
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kMaxPolls = 1u << 26;  // bounded mbarrier waits
constexpr int kATile = 128 * 128;         // bytes of one A stage
constexpr int kBTile = kMaxNB * 128;      // bytes of one B stage

template <typename ET>
struct Elem;
template <>
struct Elem<float> {                      // TF32 operands stored as fp32
  static constexpr int kPerUnit = 4;      // rows per 16-byte unit
  static constexpr uint32_t kFmt = tc::kFmtTF32;
};
template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kPerUnit = 8;
  static constexpr uint32_t kFmt = tc::kFmtBF16;
};


// Raw loaded words of one staging task: PU rows x 4 consecutive columns.
// fp32: w[i][q] = bits of element (row i, column q); bf16: w[i][0..1] hold
// the 4 bf16 of row i (2 per word).  Kept raw so that a load is only waited
// for when the task is stored.
template <typename ET, int PU>
struct Raw4 {
  static constexpr int W = sizeof(ET) == 4 ? 4 : 2;
  uint32_t w[PU][W];
};

__device__ __forceinline__ void ld4_raw(const float* p, uint32_t (&w)[4]) {
  const uint4 t = __ldg(reinterpret_cast<const uint4*>(p));
  w[0] = t.x; w[1] = t.y; w[2] = t.z; w[3] = t.w;
}
__device__ __forceinline__ void ld4_raw(const __nv_bfloat16* p, uint32_t (&w)[2]) {
  const uint2 t = __ldg(reinterpret_cast<const uint2*>(p));
  w[0] = t.x; w[1] = t.y;
}

// 16-byte swizzle unit of column q (0..3) of a task: PU consecutive rows.
template <typename ET, int MODE, int PU>
__device__ __forceinline__ uint4 unit_of(const Raw4<ET, PU>& r, int q) {
  if constexpr (sizeof(ET) == 4) {
    uint32_t v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i] = r.w[i][q];
      if constexpr (MODE == CFC_MATH_TF32) v[i] = __float_as_uint(round_tf32(__uint_as_float(v[i])));
    }
    return make_uint4(v[0], v[1], v[2], v[3]);
  } else {
    const int word = q >> 1, sh = (q & 1) * 16;
    uint32_t v[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      v[t] = ((r.w[2 * t][word] >> sh) & 0xFFFFu) | (((r.w[2 * t + 1][word] >> sh) & 0xFFFFu) << 16);
    return make_uint4(v[0], v[1], v[2], v[3]);
  }
}

template <typename ET>
__device__ __forceinline__ void set_row(uint32_t (&w)[Raw4<ET, 1>::W], float a, float b, float c, float d) {
  if constexpr (sizeof(ET) == 4) {
    w[0] = __float_as_uint(a); w[1] = __float_as_uint(b); w[2] = __float_as_uint(c); w[3] = __float_as_uint(d);
  } else {
    w[0] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
    w[1] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(c)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(d)) << 16);
  }
}

// VEC: n_in, n_hid multiples of 4, so every 4-column block lies in one
// segment of z (x, h, or the ones/padding block) and is 4-element aligned.
template <typename ET, int MODE, bool VEC>
__global__ void __launch_bounds__(kTcThreads)
k_wgrad_tc(const ET* __restrict__ dA, const ET* __restrict__ x, const ET* __restrict__ h0,
           const ET* __restrict__ h_seq, int K, int n_in, int H, long long R,
           long long rows_per_split, int NB, float* __restrict__ out) {
  constexpr int PU = Elem<ET>::kPerUnit;
  constexpr int KC = 128 / sizeof(ET);          // rows per chunk
  constexpr int G = KC / PU;                    // 8 row groups of PU rows per chunk
  const int H3 = 3 * H, Zc = n_in + H, Zb = Zc + 1;
  const long long N = (long long)H3 * Zb;
  const int m0 = blockIdx.x * 128, n0 = blockIdx.y * NB;
  const long long s = blockIdx.z;
  const long long r_begin = s * rows_per_split;
  const long long r_end = min(R, r_begin + rows_per_split);
  const int nchunks = (int)((r_end - r_begin + KC - 1) / KC);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* As = sm;                               // [kStages][128 rows][128 B]
  uint8_t* Bs = sm + kStages * kATile;            // [kStages][kMaxNB rows][128 B]
  __shared__ uint64_t bars[kStages];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) tc::mbar_init(&bars[i], 1);
    tc::mbar_init_fence();
    abort_flag = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  // Tasks of a chunk: A: 32 column quads x G row groups (= 256, one per
  // thread); B: NB/4 column quads x G row groups (<= 416, two per thread).
  const int nbq = NB / 4;
  const int b_tasks = nbq * G;
  constexpr int kBPer = (kMaxNB / 4 * G + kTcThreads - 1) / kTcThreads;  // 2
  Raw4<ET, PU> ra, rb[kBPer];

  auto load_chunk = [&](int c) {
    const long long rc = r_begin + (long long)c * KC;
    {  // A: dA rows (m contiguous)
      const int mq = tid & 31, g = tid >> 5;
      const int m = m0 + 4 * mq;
#pragma unroll
      for (int i = 0; i < PU; ++i) {
        const long long row = rc + g * PU + i;
        if (VEC) {
          if (row < r_end && m < H3) ld4_raw(dA + row * H3 + m, ra.w[i]);
          else set_row<ET>(ra.w[i], 0.f, 0.f, 0.f, 0.f);
        } else {
          float v[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) v[q] = (row < r_end && m + q < H3) ? ldf(dA + row * H3 + m + q) : 0.f;
          set_row<ET>(ra.w[i], v[0], v[1], v[2], v[3]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kBPer; ++t) {
      const int task = tid + t * kTcThreads;
      const int jq = (task < b_tasks) ? task % nbq : 0, g = (task < b_tasks) ? task / nbq : 0;
      const int j = (task < b_tasks) ? n0 + 4 * jq : Zb;   // j >= Zb: zeros
      const long long row0 = rc + g * PU;
      long long b = row0 / K;
      int k = (int)(row0 - b * K);
#pragma unroll
      for (int i = 0; i < PU; ++i) {
        const long long row = row0 + i;
        bool done_row = false;
        if (row < r_end) {
          const ET* hrow = (k == 0) ? (h0 + b * H) : (h_seq + (row - 1) * H);
          if (VEC) {
            if (j < n_in) { ld4_raw(x + row * n_in + j, rb[t].w[i]); done_row = true; }
            else if (j < Zc) { ld4_raw(hrow + (j - n_in), rb[t].w[i]); done_row = true; }
            else if (j == Zc) { set_row<ET>(rb[t].w[i], 1.f, 0.f, 0.f, 0.f); done_row = true; }
          } else {
            float v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int jj = j + q;
              float val = 0.f;
              if (jj < n_in) val = ld_operand<MODE>(x + row * n_in + jj);
              else if (jj < Zc) val = ld_operand<MODE>(hrow + (jj - n_in));
              else if (jj == Zc) val = 1.f;
              v[q] = val;
            }
            set_row<ET>(rb[t].w[i], v[0], v[1], v[2], v[3]);
            done_row = true;
          }
        }
        if (!done_row) set_row<ET>(rb[t].w[i], 0.f, 0.f, 0.f, 0.f);
        if (++k == K) { k = 0; ++b; }
      }
    }
  };
  auto store_chunk = [&](int st) {
    uint8_t* a = As + st * kATile;
    uint8_t* bb = Bs + st * kBTile;
    {
      const int mq = tid & 31, g = tid >> 5;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(a + tc::sw128_offset(4 * mq + q, 16 * g)) = unit_of<ET, CFC_MATH_FP32, PU>(ra, q);
    }
#pragma unroll
    for (int t = 0; t < kBPer; ++t) {
      const int task = tid + t * kTcThreads;
      if (task < b_tasks) {
        const int jq = task % nbq, g = task / nbq;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(bb + tc::sw128_offset(4 * jq + q, 16 * g)) = unit_of<ET, MODE, PU>(rb[t], q);
      }
    }
  };

  const uint32_t id = tc::idesc(128, NB, Elem<ET>::kFmt);
  if (nchunks > 0) load_chunk(0);
  for (int c = 0; c < nchunks; ++c) {
    const int st = c % kStages;
    if (c >= kStages) {
      // the MMAs of chunk c - kStages read this stage
      if (tid == 0 && !tc::mbar_wait(&bars[st], ((c - kStages) / kStages) & 1, kMaxPolls)) abort_flag = 1;
    }
    __syncthreads();
    if (abort_flag) break;
    store_chunk(st);
    if (c + 1 < nchunks) load_chunk(c + 1);
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) {  // operands from the converged warp, one elected lane issues
      const uint64_t ad = tc::sdesc_k_sw128(tc::smem_u32(As + st * kATile));
      const uint64_t bd = tc::sdesc_k_sw128(tc::smem_u32(Bs + st * kBTile));
      if (tc::elect_one()) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if constexpr (sizeof(ET) == 4) tc::mma_tf32(tmem, ad + 2 * k, bd + 2 * k, id, (c | k) != 0);
          else tc::mma_bf16(tmem, ad + 2 * k, bd + 2 * k, id, (c | k) != 0);
        }
        tc::mma_commit(&bars[st]);
      }
      __syncwarp();
    }
  }
  // Wait for the last committed chunk (MMAs complete in issue order).
  __syncthreads();
  bool ok = !abort_flag;
  if (nchunks > 0) {
    const int last = nchunks - 1;
    if (tid == 0 && !tc::mbar_wait(&bars[last % kStages], (last / kStages) & 1, kMaxPolls)) abort_flag = 1;
  }
  __syncthreads();
  ok = ok && !abort_flag;
  if (!ok && tid == 0) atomicExch(&g_cfc_device_error, 1);
  tc::fence_after_sync();

  if (ok) {
    float* o = out + s * N;
    const long long off_rec = (long long)H3 * n_in;
    const long long off_b = (long long)H3 * Zc;
    const int quad = warp & 3;                    // TMEM lane quadrant of this warp
    const int m = m0 + quad * 32 + lane;
    const int nchunk16 = NB / 16;
    for (int cc = warp >> 2; cc < nchunk16; cc += kTcThreads / 128) {
      float v[16];
      if (nchunks > 0) {
        tc::tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(cc * 16), v);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
      }
      if (m < H3) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = n0 + cc * 16 + i;
          if (j < n_in) o[(long long)m * n_in + j] = v[i];
          else if (j < Zc) o[off_rec + (long long)m * H + (j - n_in)] = v[i];
          else if (j == Zc) o[off_b + m] = v[i];
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

template <typename ET, int MODE>
cudaError_t launch_mode(const Layout& L, const CfcArgs& a, float* out, cudaStream_t s) {
  const int Zb = L.Zc + 1;
  const int nNB = (Zb + kMaxNB - 1) / kMaxNB;
  const int NB = ((Zb + nNB - 1) / nNB + 15) / 16 * 16;   // balanced N blocks, multiple of 16
  const size_t smem = 1024 + (size_t)kStages * (kATile + kBTile);
  const bool vec = (L.n_in % 4 == 0) && (L.H % 4 == 0);
  auto kern = vec ? k_wgrad_tc<ET, MODE, true> : k_wgrad_tc<ET, MODE, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((L.H3 + 127) / 128, nNB, L.n_split);
  TraceScope trace("wgrad_tc", s);
  kern<<<grid, kTcThreads, smem, s>>>(reinterpret_cast<const ET*>(a.ws + L.off_dA),
                                      static_cast<const ET*>(a.x), static_cast<const ET*>(a.h0),
                                      static_cast<const ET*>(a.h_seq), L.K, L.n_in, L.H, L.R,
                                      L.rows_per_split, NB, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// TMA-fed contraction (bf16 mode, GEMM path).
//
// The rows r = (b, k) are the contraction index and the outer index of every
// operand in HBM, so the operands are loaded as MN-major tiles: for a chunk of
// 64 rows, a 64-column block of dA, x or h_seq is one TMA box of 64 rows x
// 128 bytes, 128-byte swizzled, and the MMA reads it with an MN-major
// descriptor (leading byte offset = the next 64-column block, stride byte
// offset = the next 8 rows).  No staging threads, no transposition.
//
// Tensor maps are 3-D (columns, K, B) so a chunk is a box of kb steps x nb
// samples (whole samples when K <= 64, 64 steps of one sample when K is a
// multiple of 64).  The state entering row (b, k) is h_seq[b][k-1]: the h
// boxes are loaded at step coordinate k0 - 1, so the rows with k = 0 come back
// zero-filled (out of bounds) and a patch warp writes h0[b] into them before
// the MMAs read the stage.  The bias gradient is the contraction with a ones
// column: a constant 64-column block after the h blocks holds 1 in its first
// column, written once per stage (the TMA never touches it).
//
// Block = (M tile of 128 rows of 3H, split s of the chunk sequence).  Warp 0
// issues the TMA boxes of each chunk into a ring of stages, warp 2 patches the
// k = 0 rows, warp 1 issues the MMAs (N pieces of at most 256 columns; the
// accumulator D[128 x Ntot] lives in TMEM), and all eight warps write D into
// the packed partial row of split s at the end.  Waits are bounded.
// ---------------------------------------------------------------------------
constexpr int kTmaRows = 64;                    // rows (MMA K) per chunk
constexpr int kTmaBlock = kTmaRows * 128;       // one 64-column block of a chunk
constexpr int kTmaMaxStages = 4;
constexpr int kTmaWarpProducer = 0, kTmaWarpMma = 1, kTmaWarpPatch = 2;
constexpr uint32_t kTmaTmemCols = 512;

struct TmaWgradPlan {
  int nx = 0, nh = 0;    // 64-column blocks of x and of h
  int Ntot = 0;          // accumulator columns: Zc + 1 rounded up to 16
  int nMt = 0, S = 0, chunks = 0, stages = 0;
  int kb = 0, nb = 0;    // chunk = kb steps x nb samples
  size_t stage_bytes = 0, smem = 0;
};

__global__ void k_wgrad_tma(const __grid_constant__ CUtensorMap, const __grid_constant__ CUtensorMap,
                            const __grid_constant__ CUtensorMap, const __nv_bfloat16*, int, int, int, int, int,
                            int, int, int, int, float*);

bool plan_tma_wgrad(int B, int K, int n_in, int H, int math, int grad_path, TmaWgradPlan* p) {
  if (math != CFC_MATH_BF16 || grad_path != CFC_GRAD_GEMM) return false;
  if (n_in % 64 || H % 64) return false;
  int kb, nb;
  if (K <= kTmaRows && kTmaRows % K == 0) {
    kb = K;
    nb = kTmaRows / K;
    if (B % nb) return false;
  } else if (K % kTmaRows == 0) {
    kb = kTmaRows;
    nb = 1;
  } else {
    return false;
  }
  const int Zc = n_in + H;
  const int Ntot = (Zc + 1 + 15) / 16 * 16;
  if (Ntot > (int)kTmaTmemCols) return false;
  p->nx = n_in / 64;
  p->nh = H / 64;
  p->Ntot = Ntot;
  p->nMt = (3 * H + 127) / 128;
  p->chunks = (int)((long long)B * K / kTmaRows);
  p->kb = kb;
  p->nb = nb;
  p->stage_bytes = (size_t)(2 + p->nx + p->nh + 1) * kTmaBlock;
  p->stages = (int)std::min<size_t>(kTmaMaxStages, (227 * 1024 - 1024) / p->stage_bytes);
  if (p->stages < 2) return false;
  p->smem = 1024 + (size_t)p->stages * p->stage_bytes;
  // One wave: every M tile of every split resident at once.
  p->S = std::max(1, std::min(p->chunks, kNumSMs / p->nMt));
  return true;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(tc::smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void expect_tx_bytes(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}
// Bounded wait by a whole warp; lane 0's observation decides for all lanes.
__device__ __forceinline__ bool wait_warp(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kMaxPolls; ++i) {
    const int ok = tc::mbar_try_wait(bar, parity) ? 1 : 0;
    if (__shfl_sync(0xffffffffu, ok, 0)) return true;
  }
  return false;
}
// MN-major, 128-byte-swizzled operand: 64-column blocks kTmaBlock apart,
// 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((uint32_t)kTmaBlock >> 4) << 16;   // leading byte offset: next MN block
  d |= (uint64_t)(1024u >> 4) << 32;                 // stride byte offset: next 8 rows
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}
__device__ __forceinline__ void chunk_origin(int c, int K, int nb, int* b0, int* k0) {
  if (nb > 1) {
    *b0 = c * nb;
    *k0 = 0;
  } else {
    const int per = K / kTmaRows;
    *b0 = c / per;
    *k0 = (c - *b0 * per) * kTmaRows;
  }
}

__global__ void __launch_bounds__(kTcThreads, 1)
k_wgrad_tma(const __grid_constant__ CUtensorMap map_dA, const __grid_constant__ CUtensorMap map_x,
            const __grid_constant__ CUtensorMap map_h, const __nv_bfloat16* __restrict__ h0, int K, int n_in,
            int H, int chunks, int S, int stages, int kb, int nb, int Ntot, float* __restrict__ out) {
  const int mt = blockIdx.x, s = blockIdx.y;
  const int c_begin = (int)((long long)chunks * s / S), c_end = (int)((long long)chunks * (s + 1) / S);
  const int nx = n_in / 64, nh = H / 64;
  const int H3 = 3 * H, Zc = n_in + H;
  const uint32_t stage_bytes = (uint32_t)(2 + nx + nh + 1) * kTmaBlock;
  const uint32_t tx_bytes = (uint32_t)(2 + nx + nh) * kTmaBlock;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kTmaMaxStages], ready[kTmaMaxStages], empty[kTmaMaxStages], done;
  __shared__ uint32_t tmem_base;
  __shared__ int err;
  volatile int* errp = &err;

  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&ready[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    tc::mbar_init(&done, 1);
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kTmaTmemCols);
  // The ones block of every stage: element 0 of each row (logical 16-byte
  // chunk 0, stored at chunk position row % 8) is bf16 1.0.
  for (int st = 0; st < stages; ++st) {
    uint8_t* cb = sm + (size_t)st * stage_bytes + (size_t)(2 + nx + nh) * kTmaBlock;
    for (int e = tid; e < kTmaBlock / 16; e += kTcThreads) {
      const int r = e >> 3, q = e & 7;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (q == (r & 7)) v.x = 0x3F80u;
      *reinterpret_cast<uint4*>(cb + (size_t)e * 16) = v;
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  if (warp == kTmaWarpProducer) {
    int st = 0;
    uint32_t wrap = 0;
    for (int c = c_begin; c < c_end; ++c) {
      if (__shfl_sync(0xffffffffu, *errp, 0)) break;
      if (wrap > 0 && !wait_warp(&empty[st], (wrap - 1) & 1u)) {
        if (lane == 0) *errp = 1;
        break;
      }
      if (lane == 0) {
        int b0, k0;
        chunk_origin(c, K, nb, &b0, &k0);
        uint8_t* base = sm + (size_t)st * stage_bytes;
        expect_tx_bytes(&full[st], tx_bytes);
        tma_load_3d(base, &map_dA, mt * 128, k0, b0, &full[st]);
        tma_load_3d(base + kTmaBlock, &map_dA, mt * 128 + 64, k0, b0, &full[st]);
        for (int j = 0; j < nx + nh; ++j) {
          uint8_t* dst = base + (size_t)(2 + j) * kTmaBlock;
          const CUtensorMap* map = (j < nx) ? &map_x : &map_h;
          const int col = (j < nx) ? 64 * j : 64 * (j - nx);
          const int kc = (j < nx) ? k0 : k0 - 1;
          tma_load_3d(dst, map, col, kc, b0, &full[st]);
        }
      }
      __syncwarp();
      if (++st == stages) {
        st = 0;
        ++wrap;
      }
    }
  } else if (warp == kTmaWarpPatch) {
    // rows n*kb of a chunk starting at step 0 hold k = 0 of sample b0 + n:
    // h0[b0 + n] goes into the h blocks.  The h0 rows of the next chunk are
    // loaded while this chunk's stage is patched (up to kPatchRegs 16-byte
    // units per lane; the rest are loaded when needed).
    constexpr int kPatchRegs = 8;
    const int items = nb * nh * 8;
    uint4 pre[kPatchRegs];
    auto prefetch = [&](int c) {
      int b0, k0;
      chunk_origin(c, K, nb, &b0, &k0);
#pragma unroll
      for (int i = 0; i < kPatchRegs; ++i) {
        const int e = lane + 32 * i;
        const int q = e & 7, j = (e >> 3) % nh, n = (e >> 3) / nh;
        pre[i] = make_uint4(0u, 0u, 0u, 0u);
        if (c < c_end && k0 == 0 && e < items)
          asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(pre[i].x), "=r"(pre[i].y), "=r"(pre[i].z), "=r"(pre[i].w)
                       : "l"(h0 + (long long)(b0 + n) * H + 64 * j + 8 * q));
      }
    };
    prefetch(c_begin);
    int st = 0;
    uint32_t wrap = 0;
    for (int c = c_begin; c < c_end; ++c) {
      int b0, k0;
      chunk_origin(c, K, nb, &b0, &k0);
      if (!wait_warp(&full[st], wrap & 1u)) {
        if (lane == 0) *errp = 1;
        break;
      }
      if (k0 == 0) {
        uint8_t* hb = sm + (size_t)st * stage_bytes + (size_t)(2 + nx) * kTmaBlock;
        auto put = [&](int e, const uint4& v) {
          const int q = e & 7, j = (e >> 3) % nh, n = (e >> 3) / nh;
          const int r = n * kb;
          *reinterpret_cast<uint4*>(hb + (size_t)j * kTmaBlock + r * 128 + ((q ^ (r & 7)) << 4)) = v;
        };
#pragma unroll
        for (int i = 0; i < kPatchRegs; ++i)
          if (lane + 32 * i < items) put(lane + 32 * i, pre[i]);
        for (int e = lane + 32 * kPatchRegs; e < items; e += 32) {
          const int q = e & 7, j = (e >> 3) % nh, n = (e >> 3) / nh;
          put(e, *reinterpret_cast<const uint4*>(h0 + (long long)(b0 + n) * H + 64 * j + 8 * q));
        }
        tc::fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready[st]);
      prefetch(c + 1);
      if (++st == stages) {
        st = 0;
        ++wrap;
      }
    }
  } else if (warp == kTmaWarpMma) {
    const uint64_t a_desc = sdesc_mn_sw128(tc::smem_u32(sm));
    const uint64_t b_desc = sdesc_mn_sw128(tc::smem_u32(sm + 2 * kTmaBlock));
    const int n1 = Ntot > 256 ? 256 : Ntot, n2 = Ntot - n1;   // N pieces
    constexpr uint32_t kMN = (1u << 15) | (1u << 16);          // A and B MN-major
    const uint32_t id1 = tc::idesc(128, (uint32_t)n1, tc::kFmtBF16) | kMN;
    const uint32_t id2 = tc::idesc(128, (uint32_t)(n2 > 0 ? n2 : 16), tc::kFmtBF16) | kMN;
    int st = 0;
    uint32_t wrap = 0;
    bool ok = true;
    for (int c = c_begin; c < c_end; ++c) {
      if (!wait_warp(&ready[st], wrap & 1u)) {
        if (lane == 0) *errp = 1;
        ok = false;
        break;
      }
      tc::fence_after_sync();
      {  // operands from the converged warp, one elected lane issues
        const uint32_t so = (uint32_t)st * stage_bytes;
        if (tc::elect_one()) {
#pragma unroll
          for (int ks = 0; ks < kTmaRows / 16; ++ks) {
            const uint32_t acc = (c > c_begin || ks > 0) ? 1u : 0u;
            const uint64_t ad = tc::sdesc_advance(a_desc, so + ks * 2048);
            const uint64_t bd = tc::sdesc_advance(b_desc, so + ks * 2048);
            tc::mma_bf16(tmem, ad, bd, id1, acc);
            if (n2 > 0) tc::mma_bf16(tmem + 256, ad, tc::sdesc_advance(bd, 4 * kTmaBlock), id2, acc);
          }
          tc::mma_commit(&empty[st]);
        }
      }
      __syncwarp();
      if (++st == stages) {
        st = 0;
        ++wrap;
      }
    }
    if (ok && c_end > c_begin) tc::mma_commit_w(&done);
    __syncwarp();
  }

  // ---- epilogue: D[m][j] -> packed partial row of split s
  if (tid == 0 && c_end > c_begin && *errp == 0 && !tc::mbar_wait(&done, 0, kMaxPolls)) *errp = 1;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const bool have = (c_end > c_begin) && *errp == 0;
  float* o = out + (long long)s * (3ll * (Zc + 1) * H);
  const long long off_rec = (long long)H3 * n_in, off_b = (long long)H3 * Zc;
  const int quad = warp & 3, half = warp >> 2;
  const int m = mt * 128 + quad * 32 + lane;
  const int ng = Ntot / 16, gh = (ng + 1) / 2;
  for (int g = half * gh; g < ng && g < (half + 1) * gh; ++g) {
    float v[16];
    if (have) {
      tc::tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(g * 16), v);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.f;
    }
    if (m < H3) {
      const int j0 = g * 16;
      float* dst = nullptr;
      if (j0 + 16 <= n_in) dst = o + (long long)m * n_in + j0;
      else if (j0 >= n_in && j0 + 16 <= Zc) dst = o + off_rec + (long long)m * H + (j0 - n_in);
      if (dst) {
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      } else if (j0 == Zc) {
        o[off_b + m] = v[0];
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (*errp) atomicExch(&g_cfc_device_error, 1);
  if (warp == 0) tc::tmem_dealloc(tmem, kTmaTmemCols);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D bf16 map (columns, K, B) of a dense [B][K][cols] array; box 64 x kb x nb.
bool encode_bkc(CUtensorMap* m, const void* base, int cols, int K, int B, int kb, int nb) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)K, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * 2 * K};
  const cuuint32_t box[3] = {64u, (cuuint32_t)kb, (cuuint32_t)nb};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_wgrad_tma(const Layout& L, const TmaWgradPlan& p, const CfcArgs& a, float* out,
                             cudaStream_t s) {
  CUtensorMap mdA, mx, mh;
  if (!encode_bkc(&mdA, a.ws + L.off_dA, L.H3, L.K, L.B, p.kb, p.nb) ||
      !encode_bkc(&mx, a.x, L.n_in, L.K, L.B, p.kb, p.nb) ||
      !encode_bkc(&mh, a.h_seq, L.H, L.K, L.B, p.kb, p.nb))
    return cudaErrorNotSupported;
  cudaError_t e = cudaFuncSetAttribute(k_wgrad_tma, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  TraceScope trace("wgrad_tma_tc", s);
  k_wgrad_tma<<<dim3((unsigned)p.nMt, (unsigned)p.S, 1), kTcThreads, p.smem, s>>>(
      mdA, mx, mh, static_cast<const __nv_bfloat16*>(a.h0), L.K, L.n_in, L.H, p.chunks, p.S, p.stages, p.kb, p.nb,
      p.Ntot, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// TMA-fed contraction, TF32 mode (GEMM path).
//
// kind::tf32 MMAs read K-major operands only, while dA, x and h_seq keep the
// contraction index r outermost.  The operands arrive as in the bf16 kernel --
// 3-D TMA boxes of 32 rows x 128 bytes (32 fp32 columns), 128-byte swizzled --
// in a raw stage, and transposer warps turn each block of 4 rows x 4 columns
// (one 16-byte unit in each of 4 rows) into 4 units of the K-major tile (4
// columns x 4 rows), rounding x and h to TF32 on the way (dA is stored
// rounded).  A chunk is 32 rows: one 128-byte K atom, 4 MMAs with K = 8.
//
// A thread's block is (box, kq, mq): raw rows 4kq..4kq+3, unit mq.  16-byte
// shared accesses are served per quarter warp, so the 8 lanes l of a quarter
// q take mq = l ^ 2(q/2), kq = l/2 + 4(q%2): their raw reads (position
// mq ^ (row % 8)) and their K-major writes (position kq ^ (row % 8)) each hit 8
// distinct 16-byte positions, and the 8 quarters of a box cover its 64
// blocks once.
//
// Warps: 0 TMA producer, 1 MMA issue, 2 h0 patch (the rows with k = 0, as in
// the bf16 kernel), 3..9 transposers.  Raw stages go full (TMA) -> ready
// (patched) -> rfree (transposers done); K-major stages kfull (transposers
// done, after their proxy fences) -> kempty (MMA completion).  Block = (M
// tile of 128 rows of 3H, split s); accumulator D[128 x Ntot] in TMEM.
// ---------------------------------------------------------------------------
constexpr int kT32Rows = 32;                     // rows (MMA K) per chunk
constexpr int kT32Box = kT32Rows * 128;          // one 32-column box of a chunk
constexpr int kT32Threads = 480;
constexpr int kT32WarpProducer = 0, kT32WarpMma = 1, kT32WarpPatch = 2, kT32FirstTr = 3;
constexpr int kT32Tr = kT32Threads / 32 - kT32FirstTr;   // transposer warps
constexpr int kT32MaxRaw = 4, kT32KStages = 2;
constexpr uint32_t kT32TmemCols = 256;

struct Tf32WgradPlan {
  int nx = 0, nh = 0;    // 32-column boxes of x and of h
  int Ntot = 0;          // accumulator columns: Zc + 1 rounded up to 16
  int nMt = 0, S = 0, chunks = 0, raw_stages = 0, k_stages = 0;
  int kb = 0, nb = 0;    // chunk = kb steps x nb samples
  bool split = false;    // FP32 operands as TF32 high + low parts (three MMAs)
  size_t raw_bytes = 0, k_bytes = 0, smem = 0;
};

// TF32 mode: GEMM path.  FP32 mode ("3xTF32"): every operand a is split into
// a_hi = tf32(a) and a_lo = tf32(a - a_hi) and the products accumulate
// a_hi b_hi + a_hi b_lo + a_lo b_hi in fp32 (the dropped a_lo b_lo and the
// rounding of a_lo are below 2^-21 relative), on the GEMM path or, with one
// split per sample (K a multiple of 32), on the per-sample scratch path.
bool plan_tf32_wgrad(int B, int K, int n_in, int H, int math, int grad_path, Tf32WgradPlan* p) {
  const bool split = (math == CFC_MATH_FP32);
  if (math == CFC_MATH_TF32 ? grad_path != CFC_GRAD_GEMM : !split) return false;
  if (n_in % 32 || H % 32) return false;
  int kb, nb;
  if (K <= kT32Rows && kT32Rows % K == 0) {
    kb = K;
    nb = kT32Rows / K;
    if (B % nb) return false;
  } else if (K % kT32Rows == 0) {
    kb = kT32Rows;
    nb = 1;
  } else {
    return false;
  }
  if (grad_path == CFC_GRAD_SCRATCH && nb != 1) return false;   // a chunk must not span samples
  const int Zc = n_in + H;
  const int Ntot = (Zc + 1 + 15) / 16 * 16;
  if (Ntot > 256) return false;   // one MMA of N <= 256
  p->nx = n_in / 32;
  p->nh = H / 32;
  p->Ntot = Ntot;
  p->nMt = (3 * H + 127) / 128;
  p->chunks = (int)((long long)B * K / kT32Rows);
  p->kb = kb;
  p->nb = nb;
  p->split = split;
  p->raw_bytes = (size_t)(4 + p->nx + p->nh) * kT32Box;
  p->k_bytes = (split ? 2 : 1) * (128 * 128 + (size_t)Ntot * 128);
  p->k_stages = split ? 1 : kT32KStages;
  const size_t fixed = 1024 + p->k_stages * p->k_bytes;
  if (fixed + 2 * p->raw_bytes > 227 * 1024) return false;
  p->raw_stages = (int)std::min<size_t>(kT32MaxRaw, (227 * 1024 - fixed) / p->raw_bytes);
  p->smem = fixed + (size_t)p->raw_stages * p->raw_bytes;
  p->S = (grad_path == CFC_GRAD_SCRATCH) ? B : std::max(1, std::min(p->chunks, kNumSMs / p->nMt));
  return true;
}

__device__ __forceinline__ void chunk_origin_rows(int c, int K, int nb, int rows, int* b0, int* k0) {
  if (nb > 1) {
    *b0 = c * nb;
    *k0 = 0;
  } else {
    const int per = K / rows;
    *b0 = c / per;
    *k0 = (c - *b0 * per) * rows;
  }
}

__device__ __forceinline__ uint32_t tf32_bits(uint32_t u) { return (u + 0x1000u) & 0xFFFFE000u; }

template <bool SPLIT>
__global__ void __launch_bounds__(kT32Threads, 1)
k_wgrad_tma_tf32(const __grid_constant__ CUtensorMap map_dA, const __grid_constant__ CUtensorMap map_x,
                 const __grid_constant__ CUtensorMap map_h, const float* __restrict__ h0, int K, int n_in,
                 int H, int chunks, int S, int raw_stages, int k_stages, int kb, int nb, int Ntot,
                 float* __restrict__ out) {
  const int mt = blockIdx.x, s = blockIdx.y;
  const int c_begin = (int)((long long)chunks * s / S), c_end = (int)((long long)chunks * (s + 1) / S);
  const int nx = n_in / 32, nh = H / 32, nbox = 4 + nx + nh;
  const int H3 = 3 * H, Zc = n_in + H;
  const uint32_t raw_bytes = (uint32_t)nbox * kT32Box;
  const uint32_t tile_bytes = 128u * 128u + (uint32_t)Ntot * 128u;   // A tile + B tile
  const uint32_t k_bytes = (SPLIT ? 2u : 1u) * tile_bytes;            // SPLIT: high parts, then low parts
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = sm;                                        // [raw_stages][nbox][32 rows][128 B]
  uint8_t* kst = sm + (size_t)raw_stages * raw_bytes;       // [2][A 128 rows | B Ntot rows][128 B]
  __shared__ uint64_t full[kT32MaxRaw], ready[kT32MaxRaw], rfree[kT32MaxRaw];
  __shared__ uint64_t kfull[kT32KStages], kempty[kT32KStages], done;
  __shared__ uint32_t tmem_base;
  __shared__ int err;
  volatile int* errp = &err;

  if (tid == 0) {
    for (int i = 0; i < raw_stages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&ready[i], 1);
      tc::mbar_init(&rfree[i], kT32Tr);
    }
    for (int i = 0; i < k_stages; ++i) {
      tc::mbar_init(&kfull[i], kT32Tr);
      tc::mbar_init(&kempty[i], 1);
    }
    tc::mbar_init(&done, 1);
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kT32TmemCols);
  // Rows Zc .. Ntot-1 of every K-major B tile never change: row Zc is the ones
  // column of the bias gradient, the rest zero padding.
  for (int ks = 0; ks < k_stages; ++ks) {
    for (int part = 0; part < (SPLIT ? 2 : 1); ++part) {   // the low part of 1.0 is 0
      uint8_t* bt = kst + (size_t)ks * k_bytes + (size_t)part * tile_bytes + 128 * 128;
      for (int e = tid; e < (Ntot - Zc) * 8; e += kT32Threads) {
        const int row = Zc + (e >> 3), q = e & 7;
        const uint32_t one = (row == Zc && part == 0) ? 0x3F800000u : 0u;
        *reinterpret_cast<uint4*>(bt + row * 128 + ((q ^ (row & 7)) << 4)) = make_uint4(one, one, one, one);
      }
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  if (warp == kT32WarpProducer) {
    int st = 0;
    uint32_t wrap = 0;
    for (int c = c_begin; c < c_end; ++c) {
      if (__shfl_sync(0xffffffffu, *errp, 0)) break;
      if (wrap > 0 && !wait_warp(&rfree[st], (wrap - 1) & 1u)) {
        if (lane == 0) *errp = 1;
        break;
      }
      if (lane == 0) {
        int b0, k0;
        chunk_origin_rows(c, K, nb, kT32Rows, &b0, &k0);
        uint8_t* base = raw + (size_t)st * raw_bytes;
        expect_tx_bytes(&full[st], raw_bytes);
        for (int i = 0; i < 4; ++i) tma_load_3d(base + i * kT32Box, &map_dA, mt * 128 + 32 * i, k0, b0, &full[st]);
        for (int j = 0; j < nx; ++j) tma_load_3d(base + (4 + j) * kT32Box, &map_x, 32 * j, k0, b0, &full[st]);
        for (int j = 0; j < nh; ++j)
          tma_load_3d(base + (4 + nx + j) * kT32Box, &map_h, 32 * j, k0 - 1, b0, &full[st]);
      }
      __syncwarp();
      if (++st == raw_stages) {
        st = 0;
        ++wrap;
      }
    }
  } else if (warp == kT32WarpPatch) {
    // Rows n*kb of a chunk that starts at step 0 hold k = 0 of sample b0 + n:
    // h0[b0 + n] replaces the zero-filled h rows.  The next chunk's h0 units
    // are loaded while this chunk is patched (kPatchRegs per lane; any rest
    // is loaded when needed).
    constexpr int kPatchRegs = 4;
    const int items = nb * nh * 8;
    uint4 pre[kPatchRegs];
    auto prefetch = [&](int c) {
      int b0, k0;
      chunk_origin_rows(c, K, nb, kT32Rows, &b0, &k0);
#pragma unroll
      for (int i = 0; i < kPatchRegs; ++i) {
        const int e = lane + 32 * i;
        const int q = e & 7, j = (e >> 3) % nh, n = (e >> 3) / nh;
        pre[i] = make_uint4(0u, 0u, 0u, 0u);
        if (c < c_end && k0 == 0 && e < items)
          asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(pre[i].x), "=r"(pre[i].y), "=r"(pre[i].z), "=r"(pre[i].w)
                       : "l"(h0 + (long long)(b0 + n) * H + 32 * j + 4 * q));
      }
    };
    prefetch(c_begin);
    int st = 0;
    uint32_t wrap = 0;
    for (int c = c_begin; c < c_end; ++c) {
      int b0, k0;
      chunk_origin_rows(c, K, nb, kT32Rows, &b0, &k0);
      if (!wait_warp(&full[st], wrap & 1u)) {
        if (lane == 0) *errp = 1;
        break;
      }
      if (k0 == 0) {
        uint8_t* hb = raw + (size_t)st * raw_bytes + (size_t)(4 + nx) * kT32Box;
        auto put = [&](int e, const uint4& v) {
          const int q = e & 7, j = (e >> 3) % nh, n = (e >> 3) / nh;
          const int r = n * kb;
          *reinterpret_cast<uint4*>(hb + (size_t)j * kT32Box + r * 128 + ((q ^ (r & 7)) << 4)) = v;
        };
#pragma unroll
        for (int i = 0; i < kPatchRegs; ++i)
          if (lane + 32 * i < items) put(lane + 32 * i, pre[i]);
        for (int e = lane + 32 * kPatchRegs; e < items; e += 32) {
          const int q = e & 7, j = (e >> 3) % nh, n = (e >> 3) / nh;
          put(e, *reinterpret_cast<const uint4*>(h0 + (long long)(b0 + n) * H + 32 * j + 4 * q));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready[st]);
      prefetch(c + 1);
      if (++st == raw_stages) {
        st = 0;
        ++wrap;
      }
    }
  } else if (warp >= kT32FirstTr) {
    const int tw = warp - kT32FirstTr;
    const int ntask = nbox * 64;
    int rs = 0, ks = 0;
    uint32_t rwrap = 0, kwrap = 0;
    for (int c = c_begin; c < c_end; ++c) {
      if (!wait_warp(&ready[rs], rwrap & 1u) || (kwrap > 0 && !wait_warp(&kempty[ks], (kwrap - 1) & 1u))) {
        if (lane == 0) *errp = 1;
        break;
      }
      const uint8_t* rb = raw + (size_t)rs * raw_bytes;
      uint8_t* ka = kst + (size_t)ks * k_bytes;
      uint8_t* kbt = ka + 128 * 128;
      for (int task = tw * 32 + lane; task < ntask; task += kT32Tr * 32) {
        const int box = task >> 6, q4 = (task >> 3) & 7, l = task & 7;
        const int mq = l ^ (2 * (q4 >> 1)), kq = (l >> 1) + 4 * (q4 & 1);
        const uint8_t* src = rb + (size_t)box * kT32Box;
        uint32_t w[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * kq + i;
          const uint4 u = *reinterpret_cast<const uint4*>(src + r * 128 + ((mq ^ (r & 7)) << 4));
          w[i][0] = u.x; w[i][1] = u.y; w[i][2] = u.z; w[i][3] = u.w;
        }
        uint8_t* dst;
        int row0;
        const bool rnd = box >= 4;
        if (box < 4) {
          dst = ka;
          row0 = 32 * box + 4 * mq;
        } else if (box < 4 + nx) {
          dst = kbt;
          row0 = 32 * (box - 4) + 4 * mq;
        } else {
          dst = kbt;
          row0 = n_in + 32 * (box - 4 - nx) + 4 * mq;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int row = row0 + j;
          uint4 v = make_uint4(w[0][j], w[1][j], w[2][j], w[3][j]);
          const uint32_t off = row * 128 + ((kq ^ (row & 7)) << 4);
          if constexpr (SPLIT) {
            const uint4 hi = make_uint4(tf32_bits(v.x), tf32_bits(v.y), tf32_bits(v.z), tf32_bits(v.w));
            auto lo1 = [](uint32_t a, uint32_t h) {
              return tf32_bits(__float_as_uint(__uint_as_float(a) - __uint_as_float(h)));
            };
            const uint4 lo = make_uint4(lo1(v.x, hi.x), lo1(v.y, hi.y), lo1(v.z, hi.z), lo1(v.w, hi.w));
            *reinterpret_cast<uint4*>(dst + off) = hi;
            *reinterpret_cast<uint4*>(dst + tile_bytes + off) = lo;
          } else {
            if (rnd) v = make_uint4(tf32_bits(v.x), tf32_bits(v.y), tf32_bits(v.z), tf32_bits(v.w));
            *reinterpret_cast<uint4*>(dst + off) = v;
          }
        }
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&rfree[rs]);
        mbar_arrive(&kfull[ks]);
      }
      if (++rs == raw_stages) {
        rs = 0;
        ++rwrap;
      }
      if (++ks == k_stages) {
        ks = 0;
        ++kwrap;
      }
    }
  } else if (warp == kT32WarpMma) {
    const uint32_t id = tc::idesc(128, (uint32_t)Ntot, tc::kFmtTF32);
    const uint64_t a_desc = tc::sdesc_k_sw128(tc::smem_u32(kst));
    const uint64_t b_desc = tc::sdesc_k_sw128(tc::smem_u32(kst + 128 * 128));
    int ks = 0;
    uint32_t wrap = 0;
    bool ok = true;
    for (int c = c_begin; c < c_end; ++c) {
      if (!wait_warp(&kfull[ks], wrap & 1u)) {
        if (lane == 0) *errp = 1;
        ok = false;
        break;
      }
      tc::fence_after_sync();
      {  // operands from the converged warp, one elected lane issues
        const uint32_t so = (uint32_t)ks * k_bytes;
        if (tc::elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (c > c_begin || kk > 0) ? 1u : 0u;
            const uint64_t ah = tc::sdesc_advance(a_desc, so + 32 * kk), bh = tc::sdesc_advance(b_desc, so + 32 * kk);
            if constexpr (SPLIT) {   // small terms first: a_hi b_lo, a_lo b_hi, a_hi b_hi
              tc::mma_tf32(tmem, ah, tc::sdesc_advance(bh, tile_bytes), id, acc);
              tc::mma_tf32(tmem, tc::sdesc_advance(ah, tile_bytes), bh, id, 1u);
              tc::mma_tf32(tmem, ah, bh, id, 1u);
            } else {
              tc::mma_tf32(tmem, ah, bh, id, acc);
            }
          }
          tc::mma_commit(&kempty[ks]);
        }
      }
      __syncwarp();
      if (++ks == k_stages) {
        ks = 0;
        ++wrap;
      }
    }
    if (ok && c_end > c_begin) tc::mma_commit_w(&done);
    __syncwarp();
  }

  // ---- epilogue: D[m][j] -> packed partial row of split s (warps 0..7)
  if (tid == 0 && c_end > c_begin && *errp == 0 && !tc::mbar_wait(&done, 0, kMaxPolls)) *errp = 1;
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const bool have = (c_end > c_begin) && *errp == 0;
  if (warp < 8) {
    float* o = out + (long long)s * (3ll * (Zc + 1) * H);
    const long long off_rec = (long long)H3 * n_in, off_b = (long long)H3 * Zc;
    const int quad = warp & 3, half = warp >> 2;
    const int m = mt * 128 + quad * 32 + lane;
    const int ng = Ntot / 16, gh = (ng + 1) / 2;
    for (int g = half * gh; g < ng && g < (half + 1) * gh; ++g) {
      float v[16];
      if (have) {
        tc::tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(g * 16), v);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.f;
      }
      if (m < H3) {
        const int j0 = g * 16;
        float* dst = nullptr;
        if (j0 + 16 <= n_in) dst = o + (long long)m * n_in + j0;
        else if (j0 >= n_in && j0 + 16 <= Zc) dst = o + off_rec + (long long)m * H + (j0 - n_in);
        if (dst) {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else if (j0 == Zc) {
          o[off_b + m] = v[0];
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (*errp) atomicExch(&g_cfc_device_error, 1);
  if (warp == 0) tc::tmem_dealloc(tmem, kT32TmemCols);
}

// 3-D fp32 map (columns, K, B) of a dense [B][K][cols] array; box 32 x kb x nb.
bool encode_bkc_f32(CUtensorMap* m, const void* base, int cols, int K, int B, int kb, int nb) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)K, (cuuint64_t)B};
  const cuuint64_t strides[2] = {(cuuint64_t)cols * 4, (cuuint64_t)cols * 4 * K};
  const cuuint32_t box[3] = {32u, (cuuint32_t)kb, (cuuint32_t)nb};
  const cuuint32_t es[3] = {1u, 1u, 1u};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_wgrad_tma_tf32(const Layout& L, const Tf32WgradPlan& p, const CfcArgs& a, float* out,
                                  cudaStream_t s) {
  CUtensorMap mdA, mx, mh;
  if (!encode_bkc_f32(&mdA, a.ws + L.off_dA, L.H3, L.K, L.B, p.kb, p.nb) ||
      !encode_bkc_f32(&mx, a.x, L.n_in, L.K, L.B, p.kb, p.nb) ||
      !encode_bkc_f32(&mh, a.h_seq, L.H, L.K, L.B, p.kb, p.nb))
    return cudaErrorNotSupported;
  auto kern = p.split ? k_wgrad_tma_tf32<true> : k_wgrad_tma_tf32<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  TraceScope trace(p.split ? "wgrad_tma_3xtf32" : "wgrad_tma_tf32", s);
  kern<<<dim3((unsigned)p.nMt, (unsigned)p.S, 1), kT32Threads, p.smem, s>>>(
      mdA, mx, mh, static_cast<const float*>(a.h0), L.K, L.n_in, L.H, p.chunks, p.S, p.raw_stages, p.k_stages, p.kb,
      p.nb, p.Ntot, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// grad_x of the tensor-core backward kernels as one GEMM after the K loop:
//
//   grad_x[r][i] = sum_m dA[r][m] * W_in[m][i]      (r over B*K rows, m over 3H)
//
// grad_x does not feed the recurrence, so the K-loop kernels only carry
// W_rec^T dA and this kernel does the rest with the dA they saved.  A = dA
// rows (K-major: m is dA's contiguous index) arrive as 128-row x 128-byte TMA
// boxes (2-D map, 128B swizzle) through a ring of stages; B = W_in^T (the
// block's part of NW columns, K-major, mode-rounded) is staged once per block
// and stays resident.  Blocks are persistent over 128-row tiles; the
// accumulator is double-buffered in TMEM so the epilogue of one tile overlaps
// the MMAs of the next.  Warp 0: TMA producer, warp 1: MMA issue, warps 4-7:
// epilogue (TMEM lane quadrants), warps 2-3 idle after staging.
// ---------------------------------------------------------------------------
constexpr int kGxMaxStages = 8;

struct GradXPlan {
  int nAk = 0, NW = 0, nN = 0, G = 0, nst = 0, tiles = 0;
  uint32_t tmem_cols = 0;
  size_t smem = 0;
};

bool plan_grad_x(const Layout& L, GradXPlan* p) {
  if (L.math == CFC_MATH_FP32) return false;
  const int es = (L.math == CFC_MATH_TF32) ? 4 : 2;
  if ((L.H3 * es) % 16) return false;                  // TMA row stride
  p->nAk = (L.H3 * es + 127) / 128;
  const int nw_max = std::min(256, (int)((110 * 1024) / ((size_t)p->nAk * 128)) / 16 * 16);
  if (nw_max < 16) return false;
  p->nN = (L.n_in + nw_max - 1) / nw_max;
  p->NW = ((L.n_in + p->nN - 1) / p->nN + 15) / 16 * 16;
  const size_t b_bytes = (size_t)p->nAk * p->NW * 128;
  p->nst = (int)std::min<size_t>(kGxMaxStages, (227 * 1024 - 1024 - b_bytes) / (128 * 128));
  if (p->nst < 2) return false;
  p->smem = 1024 + b_bytes + (size_t)p->nst * 128 * 128;
  p->tiles = (int)((L.R + 127) / 128);
  p->G = std::max(1, std::min(p->tiles, kNumSMs / p->nN));
  uint32_t cols = 32;
  while (cols < (uint32_t)(2 * p->NW)) cols <<= 1;
  p->tmem_cols = cols;
  return true;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(tc::smem_u32(bar))
      : "memory");
}

template <typename ET, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
k_grad_x_tc(const __grid_constant__ CUtensorMap map_dA, const ET* __restrict__ W_in, int H3, int n_in, long long R,
            int nAk, int NW, int nN, int G, int nst, int tiles, uint32_t tmem_cols, float* __restrict__ grad_x) {
  constexpr int EPA = 128 / (int)sizeof(ET);
  const int np = blockIdx.x % nN, g = blockIdx.x / nN;
  const int n0 = np * NW;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  uint8_t* Bs = sm;                                             // nAk x [NW rows][128 B]
  uint8_t* As = sm + (size_t)nAk * NW * 128;                    // nst x [128 rows][128 B]
  __shared__ uint64_t full[kGxMaxStages], empty[kGxMaxStages], dfull[2], dempty[2];
  __shared__ uint32_t tmem_base;
  __shared__ int err;
  volatile int* errp = &err;

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&dfull[i], 1);
      tc::mbar_init(&dempty[i], 4);     // one arrival per epilogue warp
    }
    tc::mbar_init_fence();
    err = 0;
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, tmem_cols);
  // B[n][m] = W_in[m][n0 + n] (W_in stacked as [3H][n_in]), zero padding.
  const int Kpad = nAk * EPA;
  for (int e = tid; e < NW * Kpad; e += kTcThreads) {
    const int m = e / NW, n = e - m * NW;
    float v = 0.f;
    if (m < H3 && n0 + n < n_in) v = ld_operand<MODE>(W_in + (long long)m * n_in + n0 + n);
    const uint32_t kb = (uint32_t)m * sizeof(ET);
    uint8_t* dst = Bs + (kb >> 7) * (uint32_t)NW * 128u + tc::sw128_offset(n, kb & 127u);
    if constexpr (sizeof(ET) == 4) *reinterpret_cast<float*>(dst) = v;
    else *reinterpret_cast<__nv_bfloat16*>(dst) = __float2bfloat16_rn(v);
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    // ---- producer: the nAk boxes of every tile of this block
    int st = 0;
    uint32_t wrap = 0;
    for (int t = g; t < tiles; t += G) {
      for (int a = 0; a < nAk; ++a) {
        if (__shfl_sync(0xffffffffu, *errp, 0)) break;
        if (wrap > 0 && !wait_warp(&empty[st], (wrap - 1) & 1u)) {
          if (lane == 0) *errp = 1;
          break;
        }
        if (lane == 0) {
          expect_tx_bytes(&full[st], 128 * 128);
          tma_load_2d(As + (size_t)st * 128 * 128, &map_dA, a * EPA, t * 128, &full[st]);
        }
        __syncwarp();
        if (++st == nst) {
          st = 0;
          ++wrap;
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issue: D[buf] (columns buf*NW ...) = A tile x B part
    const uint32_t id = tc::idesc(128, (uint32_t)NW, sizeof(ET) == 4 ? tc::kFmtTF32 : tc::kFmtBF16);
    const uint64_t a0 = tc::sdesc_k_sw128(tc::smem_u32(As)), b0 = tc::sdesc_k_sw128(tc::smem_u32(Bs));
    int st = 0, i = 0;
    uint32_t wrap = 0;
    bool ok = true;
    for (int t = g; t < tiles && ok; t += G, ++i) {
      const int buf = i & 1;
      if (i >= 2 && !wait_warp(&dempty[buf], (uint32_t)(((i - 2) >> 1) & 1))) {
        if (lane == 0) *errp = 1;
        ok = false;
        break;
      }
      tc::fence_after_sync();
      for (int a = 0; a < nAk; ++a) {
        if (!wait_warp(&full[st], wrap & 1u)) {
          if (lane == 0) *errp = 1;
          ok = false;
          break;
        }
        tc::fence_after_sync();
        {  // operands from the converged warp, one elected lane issues
          const uint64_t ad = tc::sdesc_advance(a0, (uint32_t)st * 128 * 128);
          const uint64_t bd = tc::sdesc_advance(b0, (uint32_t)a * NW * 128);
          if (tc::elect_one()) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              if constexpr (sizeof(ET) == 4)
                tc::mma_tf32(tmem + (uint32_t)(buf * NW), ad + 2 * q, bd + 2 * q, id, (a | q) != 0);
              else tc::mma_bf16(tmem + (uint32_t)(buf * NW), ad + 2 * q, bd + 2 * q, id, (a | q) != 0);
            }
            tc::mma_commit(&empty[st]);
          }
        }
        __syncwarp();
        if (++st == nst) {
          st = 0;
          ++wrap;
        }
      }
      if (ok) tc::mma_commit_w(&dfull[buf]);
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ---- epilogue: lane quadrant = warp - 4, 16 columns per load
    const int qd = warp - 4;
    int i = 0;
    for (int t = g; t < tiles; t += G, ++i) {
      const int buf = i & 1;
      if (!wait_warp(&dfull[buf], (uint32_t)((i >> 1) & 1))) {
        if (lane == 0) *errp = 1;
        break;
      }
      tc::fence_after_sync();
      const long long row = (long long)t * 128 + qd * 32 + lane;
      for (int c0 = 0; c0 < NW; c0 += 16) {
        float v[16];
        tc::tmem_ld16(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(buf * NW + c0), v);
        if (row < R) {
          float* dst = grad_x + row * n_in + n0 + c0;
          const int left = n_in - (n0 + c0);
          if (left >= 16 && (n_in & 3) == 0) {
#pragma unroll
            for (int q = 0; q < 16; q += 4) *reinterpret_cast<float4*>(dst + q) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q)
              if (q < left) dst[q] = v[q];
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&dempty[buf]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (*errp) atomicExch(&g_cfc_device_error, 1);
  if (warp == 0) tc::tmem_dealloc(tmem, tmem_cols);
}

template <typename ET, int MODE>
cudaError_t launch_grad_x(const Layout& L, const GradXPlan& p, const CfcArgs& a, cudaStream_t s) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  CUtensorMap map;
  const cuuint64_t dims[2] = {(cuuint64_t)L.H3, (cuuint64_t)L.R};
  const cuuint64_t strides[1] = {(cuuint64_t)L.H3 * sizeof(ET)};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / sizeof(ET)), 128u};
  const cuuint32_t es[2] = {1u, 1u};
  if (fn(&map, sizeof(ET) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
         a.ws + L.off_dA, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorNotSupported;
  auto kern = k_grad_x_tc<ET, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
  if (e != cudaSuccess) return e;
  TraceScope trace("grad_x_tc", s);
  kern<<<p.nN * p.G, kTcThreads, p.smem, s>>>(map, static_cast<const ET*>(a.W_in), L.H3, L.n_in, L.R, p.nAk, p.NW,
                                               p.nN, p.G, p.nst, p.tiles, p.tmem_cols, a.grad_x);
  return cudaGetLastError();
}

}  // namespace

namespace {
// Waits, bounded by max_polls, on an mbarrier that nothing completes -- the
// wait helper and the error word of the K-loop kernels -- so that a test can
// see a timeout reported without any real kernel failing.
__global__ void k_selftest_wait_timeout(uint32_t max_polls) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, max_polls)) atomicExch(&g_cfc_device_error, 1);
}
}  // namespace

cudaError_t launch_selftest_wait_timeout(uint32_t max_polls, cudaStream_t s) {
  k_selftest_wait_timeout<<<1, 32, 0, s>>>(max_polls);
  return cudaGetLastError();
}

int read_device_error(int clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_cfc_device_error, sizeof(int)) != cudaSuccess) return CFC_ERR_DEVICE;
  if (clear && v) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_cfc_device_error, &zero, sizeof(int)) != cudaSuccess) return CFC_ERR_DEVICE;
  }
  return v;
}

int tc_wgrad_blocks(int n_in, int n_hid) {
  const int Zb = n_in + n_hid + 1;
  return ((3 * n_hid + 127) / 128) * ((Zb + kMaxNB - 1) / kMaxNB);
}

int tma_wgrad_splits(int B, int K, int n_in, int n_hid, int math, int grad_path) {
  if (getenv("CFC_WGRAD_STAGED")) return 0;   // force the register-staged contraction
  TmaWgradPlan p;
  if (plan_tma_wgrad(B, K, n_in, n_hid, math, grad_path, &p)) return p.S;
  Tf32WgradPlan q;
  if (plan_tf32_wgrad(B, K, n_in, n_hid, math, grad_path, &q)) return q.S;
  return 0;
}

cudaError_t launch_wgrad_tc(const Layout& L, const CfcArgs& a, float* out, cudaStream_t s) {
  const int splits = tma_wgrad_splits(L.B, L.K, L.n_in, L.H, L.math, L.grad_path);
  TmaWgradPlan p;
  if (splits == L.n_split && plan_tma_wgrad(L.B, L.K, L.n_in, L.H, L.math, L.grad_path, &p)) {
    cudaError_t e = launch_wgrad_tma(L, p, a, out, s);
    if (e != cudaErrorNotSupported) return e;
  }
  Tf32WgradPlan q;
  if (splits == L.n_split && plan_tf32_wgrad(L.B, L.K, L.n_in, L.H, L.math, L.grad_path, &q)) {
    cudaError_t e = launch_wgrad_tma_tf32(L, q, a, out, s);
    if (e != cudaErrorNotSupported) return e;
  }
  if (L.math == CFC_MATH_TF32) return launch_mode<float, CFC_MATH_TF32>(L, a, out, s);
  if (L.math == CFC_MATH_BF16) return launch_mode<__nv_bfloat16, CFC_MATH_BF16>(L, a, out, s);
  return cudaErrorNotSupported;
}

bool grad_x_gemm_applies(const Layout& L) {
  GradXPlan p;
  return plan_grad_x(L, &p) && encode_fn() != nullptr;
}

cudaError_t launch_grad_x_tc(const Layout& L, const CfcArgs& a, cudaStream_t s) {
  GradXPlan p;
  if (!a.grad_x || !plan_grad_x(L, &p)) return cudaErrorNotSupported;
  if (L.math == CFC_MATH_TF32) return launch_grad_x<float, CFC_MATH_TF32>(L, p, a, s);
  return launch_grad_x<__nv_bfloat16, CFC_MATH_BF16>(L, p, a, s);
}

}  // namespace cfc
