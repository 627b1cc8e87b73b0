// reduce_axis0.cu -- deterministic, atomic-free column sum [B, N] -> [N].
//
// Summation order (bit-identical to the reference reducer of "K-loop
// Parallelization Implementation Plan", Task 1, which runs one 256-thread
// block per column): leaf t (t = 0..255) is the ordered float32 sum
//     p[t] = ((0.0f + in[t]) + in[t+256]) + in[t+512] + ...
// and the leaves are combined by the stride-halving tree p[t] += p[t+s],
// s = 128, 64, ..., 1.  The first tree level pairs leaves whose indices differ
// in bit 7, the last level in bit 0.  Ordered by the 8-bit bit reversal
// i = rev(t), that tree is the plain contiguous pairwise tree over i, so any
// aligned power-of-two range of i is a complete subtree.  This kernel uses
// that: warp w of a block owns the 32-leaf subtree i in [32w, 32w+32), every
// lane owns 1 (ragged N) or 4 (float4) adjacent columns, and the 8 subtree
// sums meet in shared memory for the last three levels.  Leaves are loaded
// and summed in batches of 8 (an 8-leaf subtree each).  Leaves with t >= B are
// +0.0f; adding +0.0f to a partial sum that is never -0.0f (every sum starts
// from 0.0f + value) changes nothing, so their loads are skipped.
//
// A warp splits its 32 leaves into LG = 4 groups of lanes (each group a
// complete subtree of 8 leaves over the same GW = 8 column groups), combined
// afterwards by shuffles in tree order: a lane loads all 8 leaves' rows at
// once (one memory round trip per 256 rows), and the small column tiles give
// many blocks.
//
// Memory access: a warp reads LG row segments of GW x 16 B (x 4 B for ragged
// N) per load, each element exactly once.  The grid has one block per GW*VEC
// columns and no inter-block communication.
//
// Build without fast-math / FTZ: denormal partial sums must round exactly like
// the IEEE float32 reference.
#include "cfc_internal.cuh"

namespace cfc {
namespace {

constexpr int kWarps = 8;      // subtrees per block
constexpr int kMultiMax = 32;  // matrices per launch of the multi-matrix kernel

template <int VEC> struct Vec;
template <> struct Vec<4> {
  using T = float4;
  static __device__ __forceinline__ float4 zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
  static __device__ __forceinline__ float4 load(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
  }
  static __device__ __forceinline__ float4 add(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
  }
};
template <> struct Vec<1> {
  using T = float;
  static __device__ __forceinline__ float zero() { return 0.f; }
  static __device__ __forceinline__ float load(const float* p) { return __ldcs(p); }
  static __device__ __forceinline__ float add(float a, float b) { return a + b; }
};

__device__ __forceinline__ float* seg_ptr(const ReduceOut& o, long long col) {
  int s = 0;
  if (o.nseg > 1 && col >= o.begin[1]) s = 1;
  if (o.nseg > 2 && col >= o.begin[2]) s = 2;
  if (o.nseg > 3 && col >= o.begin[3]) s = 3;
  return o.ptr[s] + (col - o.begin[s]);
}

__device__ __forceinline__ float shfl_down(float v, int d) { return __shfl_down_sync(0xffffffffu, v, d); }
__device__ __forceinline__ float4 shfl_down(float4 v, int d) {
  return make_float4(__shfl_down_sync(0xffffffffu, v.x, d), __shfl_down_sync(0xffffffffu, v.y, d),
                     __shfl_down_sync(0xffffffffu, v.z, d), __shfl_down_sync(0xffffffffu, v.w, d));
}

// Template parameters: LG lane groups per warp (1 or 4), LPG leaves per lane
// group, CPL column sets per lane.  The kernel visits NL = 8 * LG * LPG leaves
// i = LS * j (LS = 256 / NL, j = 0 .. NL-1): every leaf with t < NL.  When
// B <= NL the leaves it skips are all empty, and since each subtree of LS
// consecutive leaves then holds exactly one visited leaf (the others add
// +0.0f exactly), the pairwise tree over the visited leaves in order is the
// full 256-leaf tree.  Small batches therefore use small NL and spend the
// lanes on more columns instead.
template <int VEC, int LG, int LPG, int CPL>
__device__ __forceinline__ void reduce_block(const float* __restrict__ in, int B, long long N, long long ld,
                                             const ReduceOut& out, long long block) {
  using V = Vec<VEC>;
  using T = typename V::T;
  constexpr int GW = 32 / LG;                 // column groups per warp and column set
  constexpr int NL = kWarps * LG * LPG;       // visited leaves
  constexpr int LS = 256 / NL;                // leaf stride
  __shared__ T part[kWarps][32 * CPL];

  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const int cg = lane % GW, lg = lane / GW;

  T total[CPL];
  {
    T v[CPL][LPG];
    int t[LPG];
#pragma unroll
    for (int m = 0; m < LPG; ++m) t[m] = (int)(__brev((unsigned)(((w * LG + lg) * LPG + m) * LS)) >> 24);
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const long long col = ((block * CPL + c) * GW + cg) * VEC;
#pragma unroll
      for (int m = 0; m < LPG; ++m) {
        v[c][m] = V::zero();
        if (col < N && t[m] < B) v[c][m] = V::add(V::zero(), V::load(in + (long long)t[m] * ld + col));
      }
    }
    // Rows t + 256, t + 512, ... of every leaf, in ascending order per leaf
    // (only when all 256 leaves are visited).
    if (NL == 256) {
#pragma unroll 2
      for (int off = 256; off < B; off += 256) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const long long col = ((block * CPL + c) * GW + cg) * VEC;
#pragma unroll
          for (int m = 0; m < LPG; ++m)
            if (col < N && t[m] + off < B) v[c][m] = V::add(v[c][m], V::load(in + (long long)(t[m] + off) * ld + col));
        }
      }
    }
    // The lane group's contiguous pairwise subtree (static indices).
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
#pragma unroll
      for (int width = 1; width < LPG; width *= 2) {
#pragma unroll
        for (int m = 0; m + width < LPG; m += 2 * width) v[c][m] = V::add(v[c][m], v[c][m + width]);
      }
      total[c] = v[c][0];
    }
  }
  // Lane groups of the warp: (g0 + g1), or ((g0 + g1) + (g2 + g3)).
#pragma unroll
  for (int c = 0; c < CPL; ++c) {
    if constexpr (LG >= 2) {
      const T o = shfl_down(total[c], GW);
      if ((lg & 1) == 0) total[c] = V::add(total[c], o);
    }
    if constexpr (LG == 4) {
      const T o = shfl_down(total[c], 2 * GW);
      if (lg == 0) total[c] = V::add(total[c], o);
    }
    if (lg == 0) part[w][c * GW + cg] = total[c];
  }
  __syncthreads();
  // The 8 warps' subtrees.
  for (int e = threadIdx.x; e < GW * CPL; e += kWarps * 32) {
    const long long col = (block * CPL * GW + e) * VEC;
    if (col < N) {
      T s01 = V::add(part[0][e], part[1][e]);
      T s23 = V::add(part[2][e], part[3][e]);
      T s45 = V::add(part[4][e], part[5][e]);
      T s67 = V::add(part[6][e], part[7][e]);
      *reinterpret_cast<T*>(seg_ptr(out, col)) = V::add(V::add(s01, s23), V::add(s45, s67));
    }
  }
}

template <int VEC, int LG, int LPG, int CPL>
__global__ void __launch_bounds__(kWarps * 32, 3)
k_reduce_axis0(const float* __restrict__ in, int B, long long N, long long ld, ReduceOut out) {
  reduce_block<VEC, LG, LPG, CPL>(in, B, N, ld, out, blockIdx.x);
}

// Several matrices in one launch: block b belongs to the matrix i with
// block_begin[i] <= b < block_begin[i+1] and runs that matrix's block
// b - block_begin[i], exactly as a single-matrix launch would.
struct MultiTable {
  int count;
  long long block_begin[kMultiMax + 1];
  const float* in[kMultiMax];
  float* out[kMultiMax];
  long long N[kMultiMax];
  int B[kMultiMax];
};

template <int VEC, int LG, int LPG, int CPL>
__global__ void __launch_bounds__(kWarps * 32, 3)
k_reduce_axis0_multi(const __grid_constant__ MultiTable t) {
  const long long b = blockIdx.x;
  int i = 0;
  while (i + 1 < t.count && t.block_begin[i + 1] <= b) ++i;
  ReduceOut o{};
  o.nseg = 1;
  o.ptr[0] = t.out[i];
  o.begin[0] = 0;
  reduce_block<VEC, LG, LPG, CPL>(t.in[i], t.B[i], t.N[i], t.N[i], o, b - t.block_begin[i]);
}

template <int VEC, int LG, int LPG, int CPL>
cudaError_t launch_cfg(const float* in, int n_batch, long long n_tail, long long ld, const ReduceOut& out,
                       cudaStream_t stream) {
  constexpr int GW = 32 / LG;
  const long long groups = (n_tail + VEC - 1) / VEC;
  const long long blocks = (groups + (long long)GW * CPL - 1) / ((long long)GW * CPL);
  k_reduce_axis0<VEC, LG, LPG, CPL><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(in, n_batch, n_tail, ld, out);
  return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <int VEC_, int LG_, int LPG_, int CPL_>
struct Cfg {
  static constexpr int VEC = VEC_, LG = LG_, LPG = LPG_, CPL = CPL_;
};

// Kernel configuration for a batch of n_batch rows: visited leaves NL >= B
// (all 256 beyond 128 rows), 8 or more loads per lane in flight.  0-3: float4
// rows; 4-7: scalar loads for ragged or unaligned rows.  The ragged choices
// were measured (B = 1024, N = 40961: 4 lane groups of 8 leaves and 2 column
// sets, 58 us, against 67-82 us for one 32-leaf group or 2 groups of 16).
int reduce_config(int n_batch, bool vec) {
  const int band = n_batch > 128 ? 0 : n_batch > 64 ? 1 : n_batch > 32 ? 2 : 3;
  return (vec ? 0 : 4) + band;
}

template <typename F>
cudaError_t with_config(int cfg, F&& f) {
  switch (cfg) {
    case 0: return f(Cfg<4, 4, 8, 1>{});
    case 1: return f(Cfg<4, 4, 4, 2>{});
    case 2: return f(Cfg<4, 4, 2, 4>{});
    case 3: return f(Cfg<4, 4, 1, 8>{});
    case 4: return f(Cfg<1, 4, 8, 2>{});
    case 5: return f(Cfg<1, 1, 16, 1>{});
    case 6: return f(Cfg<1, 1, 8, 1>{});
    default: return f(Cfg<1, 1, 4, 2>{});
  }
}

}  // namespace

cudaError_t launch_reduce(const float* in, int n_batch, long long n_tail, long long ld,
                          const ReduceOut& out, cudaStream_t stream) {
  if (n_tail <= 0) return cudaSuccess;
  bool vec = (n_tail % 4 == 0) && (ld % 4 == 0) && aligned16(in);
  for (int s = 0; s < out.nseg; ++s) vec = vec && aligned16(out.ptr[s]) && (out.begin[s] % 4 == 0);
  TraceScope trace("reduce_axis0", stream);
  return with_config(reduce_config(n_batch, vec), [&](auto c) {
    using C = decltype(c);
    return launch_cfg<C::VEC, C::LG, C::LPG, C::CPL>(in, n_batch, n_tail, ld, out, stream);
  });
}

cudaError_t launch_reduce_multi(const float* const* in, const int* n_batch, const long long* n_tail,
                                float* const* out, int count, cudaStream_t stream) {
  // Matrices grouped by kernel configuration, in their given order; each group
  // in launches of up to kMultiMax matrices (and fewer than 2^31 blocks).
  TraceScope trace("reduce_axis0_multi", stream);
  for (int cfg = 0; cfg < 8; ++cfg) {
    cudaError_t e = with_config(cfg, [&](auto c) -> cudaError_t {
      using C = decltype(c);
      constexpr int GW = 32 / C::LG;
      MultiTable t{};
      auto flush = [&]() -> cudaError_t {
        if (t.count == 0) return cudaSuccess;
        const long long blocks = t.block_begin[t.count];
        k_reduce_axis0_multi<C::VEC, C::LG, C::LPG, C::CPL><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(t);
        t.count = 0;
        return cudaGetLastError();
      };
      for (int i = 0; i < count; ++i) {
        if (n_tail[i] <= 0) continue;
        const bool vec = (n_tail[i] % 4 == 0) && aligned16(in[i]) && aligned16(out[i]);
        if (reduce_config(n_batch[i], vec) != cfg) continue;
        const long long groups = (n_tail[i] + C::VEC - 1) / C::VEC;
        const long long blocks = (groups + (long long)GW * C::CPL - 1) / ((long long)GW * C::CPL);
        if (t.count == kMultiMax || t.block_begin[t.count] + blocks > 0x7fffffffll) {
          cudaError_t fe = flush();
          if (fe != cudaSuccess) return fe;
        }
        const int j = t.count++;
        t.in[j] = in[i];
        t.out[j] = out[i];
        t.N[j] = n_tail[i];
        t.B[j] = n_batch[i];
        t.block_begin[j + 1] = t.block_begin[j] + blocks;
      }
      return flush();
    });
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace cfc
