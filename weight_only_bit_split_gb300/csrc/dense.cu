// Dense fp16 / bf16 decode GEMV, y = W x, fp32 accumulation.
//
// batch1-cdna README, "02-gemv": one wavefront per output row, lanes strided
// across the row so each load instruction is one contiguous transaction,
// several independent accumulators so loads are issued as a batch, and
// 16-byte loads instead of 4.  The sm_103a version keeps those three
// mechanisms: one warp per row, lane-strided 16-byte chunks (a warp reads
// 512 contiguous bytes per instruction), U chunks per lane issued before
// any is consumed, L1-no-allocate / L2-evict-first hints on the weight
// stream, and a persistent grid with the rows spread evenly over all warps.
//
// Several activation columns (M > 1, up to 32): each lane owns one row and
// walks along K; the activation tile is staged in shared memory and read by
// broadcast, so every weight chunk is reused for all M columns from
// registers.  K is split over CTAs when the rows alone cannot fill the GPU;
// the last CTA of a row group adds the partial sums in a fixed order.
#include "common.cuh"

namespace wobs {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;    // 16-byte chunks in flight per lane
constexpr int kTileK = 256;   // activation elements staged per K tile

// ------------------------------------------------------------- M = 1

template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads) dense_m1_kernel(const T* __restrict__ W, int64_t ldw,
                                                             const T* __restrict__ x,
                                                             TO* __restrict__ y, int N, int K,
                                                             ArgmaxArgs am) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total_warps = gridDim.x * kWarps;
  const int nch = K >> 3;  // 16-byte chunks per row
  const uint64_t pol = l2_evict_first_policy();
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  uint64_t best = 0;
  for (int row = blockIdx.x * kWarps + warp; row < N; row += total_warps) {
    const uint4* wr = reinterpret_cast<const uint4*>(W + static_cast<int64_t>(row) * ldw);
    float acc0 = 0.f, acc1 = 0.f;
    int c = lane;
    for (; c + 32 * (kUnroll - 1) < nch; c += 32 * kUnroll) {
      uint4 wv[kUnroll], xx[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) wv[u] = ld_stream16(wr + c + 32 * u, pol);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) xx[u] = ld_nc16(xv + c + 32 * u);
#pragma unroll
      for (int u = 0; u < kUnroll; u += 2) {
        acc0 = dot8x8<T>(wv[u], xx[u], acc0);
        acc1 = dot8x8<T>(wv[u + 1], xx[u + 1], acc1);
      }
    }
    for (; c < nch; c += 32) acc0 = dot8x8<T>(ld_stream16(wr + c, pol), ld_nc16(xv + c), acc0);
    const float s = warp_sum(acc0 + acc1);
    const TO out = from_float<TO>(s);
    if (lane == 0) y[row] = out;
    if (am.out) {
      const uint64_t k = argmax_key(to_float(out), static_cast<uint32_t>(row));
      best = k > best ? k : best;
    }
  }
  if (am.out) {
    __shared__ uint64_t s_best[kWarps];
    __shared__ uint64_t s_cta[1];
    if (lane == 0) s_best[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t b = 0;
      for (int i = 0; i < kWarps; ++i) b = s_best[i] > b ? s_best[i] : b;
      s_cta[0] = b;
    }
    __syncthreads();
    argmax_publish(s_cta, 1, am, gridDim.x);
  }
}

// --------------------------------------------------------- M columns

// Per-column best keys of the rows this CTA finalised, then publish.
template <int NC>
__device__ __forceinline__ void cta_argmax_cols(const float* v, bool valid, int row, int M,
                                                const ArgmaxArgs& am) {
  __shared__ uint64_t s_key[kWarps][NC];
  __shared__ uint64_t s_cta[NC];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = 0; m < NC; ++m) {
    uint64_t k = valid ? argmax_key(v[m], static_cast<uint32_t>(row)) : 0ull;
    k = warp_max_u64(k);
    if (lane == 0) s_key[warp][m] = k;
  }
  __syncthreads();
  if (threadIdx.x < NC) {
    uint64_t b = 0;
    for (int w = 0; w < kWarps; ++w) b = s_key[w][threadIdx.x] > b ? s_key[w][threadIdx.x] : b;
    s_cta[threadIdx.x] = b;
  }
  __syncthreads();
  argmax_publish(s_cta, M, am, gridDim.x);
}

template <typename T, typename TO, int NC>
__global__ void __launch_bounds__(kThreads) dense_mn_kernel(const T* __restrict__ W, int64_t ldw,
                                                             const T* __restrict__ X, int64_t ldx,
                                                             int M, TO* __restrict__ Y, int N,
                                                             int K, int kps, SplitArgs sk,
                                                             ArgmaxArgs am) {
  __shared__ __align__(16) float xs[NC][kTileK];
  const int row = blockIdx.x * kThreads + threadIdx.x;
  const bool valid = row < N;
  const int s = blockIdx.y;
  const int k0 = s * kps;
  const int k1 = min(K, k0 + kps);
  float acc[NC];
#pragma unroll
  for (int m = 0; m < NC; ++m) acc[m] = 0.f;
  const T* wr = W + static_cast<int64_t>(valid ? row : 0) * ldw;

  for (int kt = k0; kt < k1; kt += kTileK) {
    const int kn = min(kTileK, k1 - kt);
    __syncthreads();
    for (int i = threadIdx.x; i < NC * kn; i += kThreads) {
      const int m = i / kn, k = i - m * kn;
      xs[m][k] = m < M ? to_float(X[static_cast<int64_t>(m) * ldx + kt + k]) : 0.f;
    }
    __syncthreads();
    if (valid) {
      for (int c = 0; c < kn; c += 8) {
        const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wr + kt + c));
        const T* tag = nullptr;
        const float2 a = to_float2(wv.x, tag), b = to_float2(wv.y, tag);
        const float2 e = to_float2(wv.z, tag), f = to_float2(wv.w, tag);
#pragma unroll
        for (int m = 0; m < NC; ++m) {
          const float4 x0 = *reinterpret_cast<const float4*>(&xs[m][c]);
          const float4 x1 = *reinterpret_cast<const float4*>(&xs[m][c + 4]);
          float t = acc[m];
          t = fmaf(a.x, x0.x, t); t = fmaf(a.y, x0.y, t);
          t = fmaf(b.x, x0.z, t); t = fmaf(b.y, x0.w, t);
          t = fmaf(e.x, x1.x, t); t = fmaf(e.y, x1.y, t);
          t = fmaf(f.x, x1.z, t); t = fmaf(f.y, x1.w, t);
          acc[m] = t;
        }
      }
    }
  }

  if (sk.splits > 1) {
    if (valid) {
#pragma unroll
      for (int m = 0; m < NC; ++m)
        if (m < M) sk.partials[(static_cast<int64_t>(s) * M + m) * N + row] = acc[m];
    }
    if (!splitk_arrive_last(sk.counters, blockIdx.x, sk.splits)) return;
    if (valid) {
#pragma unroll
      for (int m = 0; m < NC; ++m) {
        float t = 0.f;
        if (m < M)
          for (int j = 0; j < sk.splits; ++j)
            t += __ldcg(sk.partials + (static_cast<int64_t>(j) * M + m) * N + row);
        acc[m] = t;
      }
    }
  }
  float out[NC];
#pragma unroll
  for (int m = 0; m < NC; ++m) {
    const TO o = from_float<TO>(acc[m]);
    out[m] = to_float(o);
    if (valid && m < M) Y[static_cast<int64_t>(m) * N + row] = o;
  }
  if (am.out) cta_argmax_cols<NC>(out, valid, row, M, am);
}

template <typename T, typename TO, int NC>
cudaError_t run_mn(const void* W, int64_t ldw, const void* X, int64_t ldx, int M, void* Y, int N,
                   int K, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                   Launch* info) {
  const int kps = (((K + sk.splits - 1) / sk.splits) + 7) / 8 * 8;
  const int splits = (K + kps - 1) / kps;
  dim3 grid((N + kThreads - 1) / kThreads, splits);
  SplitArgs s2 = sk;
  s2.splits = splits;
  info->grid_x = grid.x;
  info->grid_y = grid.y;
  info->block = kThreads;
  info->kernel = "dense_mn";
  dense_mn_kernel<T, TO, NC><<<grid, kThreads, 0, st>>>(
      static_cast<const T*>(W), ldw, static_cast<const T*>(X), ldx, M, static_cast<TO*>(Y), N, K,
      kps, s2, am);
  return cudaGetLastError();
}

template <typename T, typename TO>
cudaError_t dispatch_mn(const void* W, int64_t ldw, const void* X, int64_t ldx, int M, void* Y,
                        int N, int K, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                        Launch* info) {
  if (M <= 1) return run_mn<T, TO, 1>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  if (M <= 2) return run_mn<T, TO, 2>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  if (M <= 4) return run_mn<T, TO, 4>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  if (M <= 8) return run_mn<T, TO, 8>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  if (M <= 16) return run_mn<T, TO, 16>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  return run_mn<T, TO, 32>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
}

template <typename T, typename TO>
cudaError_t run_m1(const void* W, int64_t ldw, const void* x, void* y, int N, int K,
                   const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const void* fn = reinterpret_cast<const void*>(dense_m1_kernel<T, TO>);
  const int per_sm = max_resident_ctas(fn, kThreads, 0);
  int grid = device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int need = (N + kWarps - 1) / kWarps;
  if (grid > need) grid = need;
  info->grid_x = grid;
  info->block = kThreads;
  info->kernel = "dense_m1";
  dense_m1_kernel<T, TO><<<grid, kThreads, 0, st>>>(static_cast<const T*>(W), ldw,
                                                     static_cast<const T*>(x),
                                                     static_cast<TO*>(y), N, K, am);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_dense(int dtype, const void* W, int64_t ldw, const void* X, int64_t ldx,
                              int M, void* Y, int out_f32, int N, int K, const SplitArgs& sk,
                              const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const bool m1 = (M == 1 && sk.splits <= 1);
  if (dtype == 0) {
    if (out_f32) return cudaErrorInvalidValue;
    return m1 ? run_m1<__half, __half>(W, ldw, X, Y, N, K, am, st, info)
              : dispatch_mn<__half, __half>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  }
  if (!out_f32) return cudaErrorInvalidValue;
  return m1 ? run_m1<__nv_bfloat16, float>(W, ldw, X, Y, N, K, am, st, info)
            : dispatch_mn<__nv_bfloat16, float>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
}

}  // namespace wobs
