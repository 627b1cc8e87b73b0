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
// sums meet in shared memory for the last three levels.  Leaves with t >= B are
// +0.0f; adding +0.0f to a partial sum that is never -0.0f (every sum starts
// from 0.0f + value) changes nothing, so their loads are skipped.
//
// Memory access: a warp reads 32 x 16 B = 512 contiguous bytes of one row per
// load (128 B for ragged N), each element exactly once.  The grid has one
// block per 128 (or 32) columns and no inter-block communication.
//
// Build without fast-math / FTZ: denormal partial sums must round exactly like
// the IEEE float32 reference.
#include "cfc_internal.cuh"

namespace cfc {
namespace {

constexpr int kWarps = 8;      // subtrees per block
constexpr int kLeaves = 32;    // leaves per subtree (kWarps * kLeaves == 256)
constexpr int kBatch = 8;      // leaves loaded together (memory-level parallelism)

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
  return o.ptr[s] + (col - o.begin[s]);
}

template <int VEC>
__global__ void __launch_bounds__(kWarps * 32, 3)
k_reduce_axis0(const float* __restrict__ in, int B, long long N, long long ld, ReduceOut out) {
  using V = Vec<VEC>;
  using T = typename V::T;
  __shared__ T part[kWarps][32];

  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const long long col = ((long long)blockIdx.x * 32 + lane) * VEC;
  const bool active = col < N;

  T stk[5];
  T total = V::zero();
#pragma unroll
  for (int mb = 0; mb < kLeaves; mb += kBatch) {
    T v[kBatch];
    int t[kBatch];
#pragma unroll
    for (int m = 0; m < kBatch; ++m) {
      t[m] = (int)(__brev((unsigned)(w * kLeaves + mb + m)) >> 24);
      v[m] = V::zero();
      if (active && t[m] < B) v[m] = V::add(V::zero(), V::load(in + (long long)t[m] * ld + col));
    }
    // Rows t + 256, t + 512, ... of every leaf, in ascending order per leaf.
    for (int off = 256; off < B; off += 256) {
#pragma unroll
      for (int m = 0; m < kBatch; ++m) {
        if (active && t[m] + off < B)
          v[m] = V::add(v[m], V::load(in + (long long)(t[m] + off) * ld + col));
      }
    }
    // Merge the leaves into the running pairwise tree (binary counter).
#pragma unroll
    for (int m = 0; m < kBatch; ++m) {
      const int idx = mb + m;
      T cur = v[m];
#pragma unroll
      for (int l = 0; l < 5; ++l) {
        if ((idx >> l) & 1) {
          cur = V::add(stk[l], cur);
        } else {
          stk[l] = cur;
          break;
        }
      }
      if (idx == kLeaves - 1) total = cur;
    }
  }
  part[w][lane] = total;
  __syncthreads();
  if (w == 0 && active) {
    T s01 = V::add(part[0][lane], part[1][lane]);
    T s23 = V::add(part[2][lane], part[3][lane]);
    T s45 = V::add(part[4][lane], part[5][lane]);
    T s67 = V::add(part[6][lane], part[7][lane]);
    T r = V::add(V::add(s01, s23), V::add(s45, s67));
    *reinterpret_cast<T*>(seg_ptr(out, col)) = r;
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_reduce(const float* in, int n_batch, long long n_tail, long long ld,
                          const ReduceOut& out, cudaStream_t stream) {
  if (n_tail <= 0) return cudaSuccess;
  bool vec = (n_tail % 4 == 0) && (ld % 4 == 0) && aligned16(in);
  for (int s = 0; s < out.nseg; ++s) vec = vec && aligned16(out.ptr[s]) && (out.begin[s] % 4 == 0);
  TraceScope trace("reduce_axis0", stream);
  if (vec) {
    const long long blocks = (n_tail / 4 + 31) / 32;
    k_reduce_axis0<4><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(in, n_batch, n_tail, ld, out);
  } else {
    const long long blocks = (n_tail + 31) / 32;
    k_reduce_axis0<1><<<(unsigned)blocks, kWarps * 32, 0, stream>>>(in, n_batch, n_tail, ld, out);
  }
  return cudaGetLastError();
}

}  // namespace cfc
