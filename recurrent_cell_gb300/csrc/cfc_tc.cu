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
#include <algorithm>

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
    if (tid == 0) {
      const uint64_t ad = tc::sdesc_k_sw128(tc::smem_u32(As + st * kATile));
      const uint64_t bd = tc::sdesc_k_sw128(tc::smem_u32(Bs + st * kBTile));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if constexpr (sizeof(ET) == 4) tc::mma_tf32(tmem, ad + 2 * k, bd + 2 * k, id, (c | k) != 0);
        else tc::mma_bf16(tmem, ad + 2 * k, bd + 2 * k, id, (c | k) != 0);
      }
      tc::mma_commit(&bars[st]);
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

}  // namespace

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

cudaError_t launch_wgrad_tc(const Layout& L, const CfcArgs& a, float* out, cudaStream_t s) {
  if (L.math == CFC_MATH_TF32) return launch_mode<float, CFC_MATH_TF32>(L, a, out, s);
  if (L.math == CFC_MATH_BF16) return launch_mode<__nv_bfloat16, CFC_MATH_BF16>(L, a, out, s);
  return cudaErrorNotSupported;
}

}  // namespace cfc
