// Standalone ArgCompare: argmax or argmin over each row of an [M][N] matrix
// of fp16, bf16 or fp32 values, int64 indices out.
//
// "[WIP] ArgCompare Benchmark Results and Performance Analysis" (IREE
// discussion #23609), sections "ArgMax/ArgMin Operations Analysis in
// real-world AI models" (the shapes: vocabulary argmax [1..32, 32K..256K],
// batched rows up to [4096, 32768], argmin over [32, 1M]) and "Benchmark
// Results" (a single pass per row leaves a 131K-262K reduction short of
// work; splitting the row over several workgroups and merging the partial
// results is what wins).  The reduction is HBM-bound: every element is
// read once and compared once.
//
// GB300 design:
//   * a CTA of 256 threads takes one slice of one row (rows are split so
//     that the grid covers every SM at least four times over, never below
//     4096 elements a slice); with many short rows, a warp takes a whole
//     row instead;
//   * 32-byte read-only loads with an evict-first L2 policy, four in flight
//     per thread before any compare (rows of any pitch: a scalar head up to
//     the first 32-byte boundary, a scalar ragged tail);
//   * each thread keeps its best (value, index) in registers with a strict
//     compare, so among equal values the first one it met -- its lowest
//     index -- survives; -0.0 == +0.0 under the IEEE compare;
//   * threads, warps and slices merge through one 64-bit key per candidate:
//     the value mapped to an order-preserving unsigned word (complemented
//     for argmin) in the high half, 0xFFFFFFFF - index in the low half, so
//     the maximum key is the best value at its lowest index;
//   * slices of a row meet in the caller's workspace: atomicMax on the
//     row's key, then an arrival counter; the last slice to arrive writes the
//     index and returns key and counter to zero.
#include <cstring>

#include "common.cuh"

namespace wobs {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr uint32_t kNoIndex = 0xFFFFFFFFu;

template <typename T> struct Elem;
template <> struct Elem<__half> {
  static constexpr int kPerVec = 8;
  __device__ static float get(const uint4& v, int i) {
    const uint32_t w = (&v.x)[i >> 1];
    return __half2float(__ushort_as_half(static_cast<unsigned short>(i & 1 ? w >> 16 : w & 0xFFFFu)));
  }
  __device__ static float get1(const __half* p) { return __half2float(*p); }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int kPerVec = 8;
  __device__ static float get(const uint4& v, int i) {
    const uint32_t w = (&v.x)[i >> 1];
    return __uint_as_float(i & 1 ? (w & 0xFFFF0000u) : (w << 16));
  }
  __device__ static float get1(const __nv_bfloat16* p) { return __bfloat162float(*p); }
};
template <> struct Elem<float> {
  static constexpr int kPerVec = 4;
  __device__ static float get(const uint4& v, int i) { return __uint_as_float((&v.x)[i]); }
  __device__ static float get1(const float* p) { return *p; }
};

// Strict improvement test.  `best` starts as NaN, against which both forms
// are true, so a thread's first element is always taken.
template <bool kMin>
__device__ __forceinline__ bool better(float v, float best) {
  return kMin ? !(v >= best) : !(v <= best);
}

template <bool kMin>
__device__ __forceinline__ uint64_t make_key(float best, uint32_t idx) {
  if (idx == kNoIndex) return 0ull;       // saw nothing: the identity of the max
  const uint64_t k = argmax_key(best, idx);
  if (!kMin) return k;
  // complement the value word: the smallest value gets the largest word
  return (static_cast<uint64_t>(~static_cast<uint32_t>(k >> 32)) << 32) | (k & 0xFFFFFFFFull);
}

// Scan elements [lo, hi) of `row` with `nt` threads (this one is `lt`), each
// thread in increasing index order: a scalar head up to the first 32-byte
// boundary, whole 32-byte vectors, a scalar tail.  `row` is aligned to its
// element size; any pitch works.
template <typename T, bool kMin>
__device__ __forceinline__ void scan(const T* __restrict__ row, int lo, int hi, int lt, int nt,
                                     uint64_t pol, float& best, uint32_t& bi) {
  constexpr int E = 2 * Elem<T>::kPerVec;  // elements per 32-byte vector
  const int a0 = static_cast<int>(((32u - (reinterpret_cast<uintptr_t>(row) & 31u)) & 31u) /
                                  sizeof(T));   // first element on a 32-byte boundary
  int vs = lo <= a0 ? a0 : a0 + (lo - a0 + E - 1) / E * E;
  if (vs > hi) vs = hi;
  for (int i = lo + lt; i < vs; i += nt) {
    const float x = Elem<T>::get1(row + i);
    if (better<kMin>(x, best)) { best = x; bi = static_cast<uint32_t>(i); }
  }
  const int nv = (hi - vs) / E;           // whole vectors from vs
  const uint4* rv = reinterpret_cast<const uint4*>(row + vs);
  for (int v = lt; v < nv; v += nt * kUnroll) {
    uint4 buf[kUnroll][2];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j)
      if (v + j * nt < nv) ld_stream32(rv + 2 * (v + j * nt), pol, buf[j][0], buf[j][1]);
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      if (v + j * nt < nv) {
        const uint32_t base = static_cast<uint32_t>(vs + (v + j * nt) * E);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < E / 2; ++i) {
            const float x = Elem<T>::get(buf[j][h], i);
            if (better<kMin>(x, best)) { best = x; bi = base + h * (E / 2) + i; }
          }
      }
    }
  }
  for (int i = vs + nv * E + lt; i < hi; i += nt) {
    const float x = Elem<T>::get1(row + i);
    if (better<kMin>(x, best)) { best = x; bi = static_cast<uint32_t>(i); }
  }
}

// One CTA per (row, slice).  S slices of `chunk` elements per row (the last
// may be shorter); S == 1 writes the index directly.
template <typename T, bool kMin>
__global__ void __launch_bounds__(kThreads) argcmp_cta_kernel(const T* __restrict__ X, int64_t ldx,
                                                              int N, int S, int chunk,
                                                              int64_t* __restrict__ out,
                                                              uint64_t* keys, unsigned* counters) {
  __shared__ uint64_t wkey[kThreads / 32];
  pdl_launch_dependents();
  const int m = static_cast<int>(blockIdx.x / static_cast<unsigned>(S));
  const int s = static_cast<int>(blockIdx.x % static_cast<unsigned>(S));
  const int lo = s * chunk;
  const int hi = lo + chunk < N ? lo + chunk : N;
  const uint64_t pol = l2_evict_first_policy();
  pdl_wait();

  float best = __uint_as_float(0x7FC00000u);
  uint32_t bi = kNoIndex;
  scan<T, kMin>(X + static_cast<int64_t>(m) * ldx, lo, hi, static_cast<int>(threadIdx.x), kThreads,
                pol, best, bi);
  uint64_t k = warp_max_u64(make_key<kMin>(best, bi));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) wkey[warp] = k;
  __syncthreads();
  if (warp != 0) return;
  k = lane < kThreads / 32 ? wkey[lane] : 0ull;
  k = warp_max_u64(k);
  if (S == 1) {
    if (lane == 0) out[m] = argmax_key_index(k);
    return;
  }
  if (lane == 0) {
    atomicMax(reinterpret_cast<unsigned long long*>(keys + m), static_cast<unsigned long long>(k));
    __threadfence();
    const unsigned prev = atomicAdd(counters + m, 1u);
    if (prev == static_cast<unsigned>(S) - 1u) {
      __threadfence();
      const uint64_t fin = atomicExch(reinterpret_cast<unsigned long long*>(keys + m), 0ull);
      out[m] = argmax_key_index(fin);
      counters[m] = 0u;
    }
  }
}

// Warp per row, 8 rows per CTA: many short rows.
template <typename T, bool kMin>
__global__ void __launch_bounds__(kThreads) argcmp_warp_kernel(const T* __restrict__ X, int64_t ldx,
                                                               int M, int N,
                                                               int64_t* __restrict__ out) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int m = static_cast<int>(blockIdx.x) * (kThreads / 32) + static_cast<int>(threadIdx.x >> 5);
  const uint64_t pol = l2_evict_first_policy();
  pdl_wait();
  if (m >= M) return;
  float best = __uint_as_float(0x7FC00000u);
  uint32_t bi = kNoIndex;
  scan<T, kMin>(X + static_cast<int64_t>(m) * ldx, 0, N, lane, 32, pol, best, bi);
  const uint64_t k = warp_max_u64(make_key<kMin>(best, bi));
  if (lane == 0) out[m] = argmax_key_index(k);
}

template <typename T, bool kMin>
cudaError_t run(const void* X, int64_t ldx, int M, int N, const ArgcmpPlan& p, int64_t* out,
                uint64_t* keys, unsigned* counters, cudaStream_t st, Launch* info) {
  const T* x = static_cast<const T*>(X);
  info->block = kThreads;
  info->smem = 0;
  if (p.warp_rows) {
    info->grid_x = (M + kThreads / 32 - 1) / (kThreads / 32);
    info->kernel = "argcmp_warp";
    return launch_k(argcmp_warp_kernel<T, kMin>, dim3(info->grid_x), dim3(kThreads), 0, st, true, x,
                    ldx, M, N, out);
  }
  info->grid_x = M * p.splits;
  info->kernel = "argcmp_cta";
  return launch_k(argcmp_cta_kernel<T, kMin>, dim3(info->grid_x), dim3(kThreads), 0, st, true, x,
                  ldx, N, p.splits, p.chunk, out, keys, counters);
}

}  // namespace

ArgcmpPlan plan_argcmp(int esize, int M, int N, int forced_splits) {
  ArgcmpPlan p;
  // whole rows per warp when a row is at most 8 KB and there are enough rows
  // to give every SM several warps without splitting
  if (!forced_splits && static_cast<int64_t>(N) * esize <= 8192 && M >= 2 * device_sm_count()) {
    p.warp_rows = true;
    return p;
  }
  int64_t s;
  if (forced_splits > 0) {
    s = forced_splits;
  } else {
    // at least 4 CTAs per SM in total, slices of at least 4096 elements
    const int64_t target = 4ll * device_sm_count();
    const int64_t need = (target + M - 1) / M;
    const int64_t most = (N + 4095) / 4096;
    s = need < most ? need : most;
  }
  if (s < 1) s = 1;
  const int64_t cap = (N + 63) / 64;      // slices are multiples of 64 elements
  if (s > cap) s = cap;
  int64_t chunk = (N + s - 1) / s;
  chunk = (chunk + 63) / 64 * 64;
  p.chunk = static_cast<int>(chunk);
  p.splits = static_cast<int>((N + chunk - 1) / chunk);
  return p;
}

cudaError_t launch_argcmp(int dtype, bool is_min, const void* X, int64_t ldx, int M, int N,
                          const ArgcmpPlan& p, int64_t* out, uint64_t* keys, unsigned* counters,
                          cudaStream_t st, Launch* info) {
  switch (dtype) {
    case 1:
      return is_min ? run<__half, true>(X, ldx, M, N, p, out, keys, counters, st, info)
                    : run<__half, false>(X, ldx, M, N, p, out, keys, counters, st, info);
    case 2:
      return is_min ? run<__nv_bfloat16, true>(X, ldx, M, N, p, out, keys, counters, st, info)
                    : run<__nv_bfloat16, false>(X, ldx, M, N, p, out, keys, counters, st, info);
    case 3:
      return is_min ? run<float, true>(X, ldx, M, N, p, out, keys, counters, st, info)
                    : run<float, false>(X, ldx, M, N, p, out, keys, counters, st, info);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace wobs
