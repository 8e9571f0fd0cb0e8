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
constexpr int kUnroll = 8;    // 16-byte chunks per lane per pipeline stage
constexpr int kTileK = 256;   // activation elements staged per K tile

// ------------------------------------------------------------- M = 1

// Each warp walks the (row, stage) sequence of its rows; a stage is kUnroll
// lane-strided 16-byte chunks of one row.  Two register stages: the loads of
// stage t+1 are in flight while stage t is consumed, across row boundaries.
// The first stage is issued before pdl_wait() (weights only), overlapping
// the previous kernel on the stream; x is read after it.
template <typename T>
struct DenseStage {
  uint4 w[kUnroll];
};

template <typename T>
__device__ __forceinline__ void dense_load_stage(DenseStage<T>& st, const T* __restrict__ W,
                                                 int64_t ldw, int row, int it, int nch, int lane,
                                                 uint64_t pol) {
  const uint4* wr = reinterpret_cast<const uint4*>(W + static_cast<int64_t>(row) * ldw);
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int c = it * (32 * kUnroll) + 32 * u + lane;
    st.w[u] = c < nch ? ld_stream16(wr + c, pol) : make_uint4(0u, 0u, 0u, 0u);
  }
}

template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads) dense_m1_kernel(const T* __restrict__ W, int64_t ldw,
                                                             const T* __restrict__ x,
                                                             TO* __restrict__ y, int N, int K,
                                                             ArgmaxArgs am) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total_warps = gridDim.x * kWarps;
  const int wg = blockIdx.x * kWarps + warp;
  const int nch = K >> 3;  // 16-byte chunks per row
  const int n_it = (nch + 32 * kUnroll - 1) / (32 * kUnroll);
  const int rows_w = wg < N ? (N - 1 - wg) / total_warps + 1 : 0;
  const int T_ = rows_w * n_it;
  const uint64_t pol = l2_evict_first_policy();
  const uint4* xv = reinterpret_cast<const uint4*>(x);

  DenseStage<T> sa, sb;
  int lrow = wg, lit = 0;
  auto advance = [&](int& r, int& it) {
    if (++it == n_it) { it = 0; r += total_warps; }
  };
  if (T_ > 0) { dense_load_stage(sa, W, ldw, lrow, lit, nch, lane, pol); advance(lrow, lit); }
  pdl_launch_dependents();
  pdl_wait();

  int crow = wg, cit = 0;
  float acc0 = 0.f, acc1 = 0.f;
  uint64_t best = 0;
  auto consume = [&](const DenseStage<T>& st) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = cit * (32 * kUnroll) + 32 * u + lane;
      if (c < nch) {
        if (u & 1) acc1 = dot8x8<T>(st.w[u], ld_nc16(xv + c), acc1);
        else acc0 = dot8x8<T>(st.w[u], ld_nc16(xv + c), acc0);
      }
    }
    if (cit == n_it - 1) {
      const float s = warp_sum(acc0 + acc1);
      const TO out = from_float<TO>(s);
      if (lane == 0) y[crow] = out;
      if (am.out) {
        const uint64_t k = argmax_key(to_float(out), static_cast<uint32_t>(crow));
        best = k > best ? k : best;
      }
      acc0 = acc1 = 0.f;
    }
    advance(crow, cit);
  };
  for (int t = 0; t < T_; t += 2) {
    if (t + 1 < T_) { dense_load_stage(sb, W, ldw, lrow, lit, nch, lane, pol); advance(lrow, lit); }
    consume(sa);
    if (t + 1 < T_) {
      if (t + 2 < T_) { dense_load_stage(sa, W, ldw, lrow, lit, nch, lane, pol); advance(lrow, lit); }
      consume(sb);
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

// ------------------------------------------- M = 1, cp.async staging

// The warp-per-row computation with the weight stream staged through
// shared memory by 16-byte asynchronous copies: each warp owns a ring of
// kRing 2048-byte row segments (128 lane-strided chunks), all requested
// before pdl_wait and refilled as they are consumed; the activation vector
// is copied to shared memory once per CTA after pdl_wait.  16 warps per CTA,
// two CTAs per SM (the measured optimum for the Q4_0 kernel of the same
// structure).
constexpr int kCpWarps = 16;
constexpr int kCpThreads = kCpWarps * 32;
constexpr int kSeg = 2048;
constexpr int kRing = 2;
constexpr int kRingBytes = kCpWarps * kRing * kSeg;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
               :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

template <typename T, typename TO, bool kArgmax>
__global__ void __launch_bounds__(kCpThreads) dense_m1_cp_kernel(const T* __restrict__ W,
                                                                  int64_t ldw,
                                                                  const T* __restrict__ x,
                                                                  TO* __restrict__ y, int N, int K,
                                                                  ArgmaxArgs am) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint4* xs = reinterpret_cast<uint4*>(smem + kRingBytes);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total_warps = gridDim.x * kCpWarps;
  const int wg = blockIdx.x * kCpWarps + warp;
  const int row_bytes = K * 2;
  const int nseg = (row_bytes + kSeg - 1) / kSeg;
  const int rows_w = wg < N ? (N - 1 - wg) / total_warps + 1 : 0;
  const int T_ = rows_w * nseg;
  uint8_t* myring = smem + warp * (kRing * kSeg);
  const uint8_t* wbase = reinterpret_cast<const uint8_t*>(W);

  int prow = wg, pseg = 0;
  auto issue = [&](int slot) {
    uint8_t* st = myring + slot * kSeg;
    const int off = pseg * kSeg;
    const int n = min(kSeg, row_bytes - off) / 16;
    const uint8_t* src = wbase + static_cast<int64_t>(prow) * ldw * 2 + off;
#pragma unroll
    for (int u = 0; u < kSeg / 16 / 32; ++u) {
      const int c = 32 * u + lane;
      if (c < n) cp_async16(st + 16 * c, src + 16 * c);
    }
    if (++pseg == nseg) { pseg = 0; prow += total_warps; }
  };
#pragma unroll
  for (int i = 0; i < kRing - 1; ++i) {
    if (i < T_) issue(i);
    cp_async_commit();
  }
  pdl_launch_dependents();
  pdl_wait();
  const uint4* xg = reinterpret_cast<const uint4*>(x);
  for (int c = threadIdx.x; c < (K >> 3); c += kCpThreads) xs[c] = ld_nc16(xg + c);
  __syncthreads();

  int crow = wg, cseg = 0;
  float acc0 = 0.f, acc1 = 0.f;
  uint64_t best = 0;
  for (int t = 0; t < T_; ++t) {
    // request segment t+kRing-1 (into the slot consumed last), then wait for segment t
    if (t + kRing - 1 < T_) issue((t + kRing - 1) % kRing);
    cp_async_commit();
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint4* st = reinterpret_cast<const uint4*>(myring + (t % kRing) * kSeg);
    const int c0 = cseg * (kSeg / 16);
    const int n = min(kSeg, row_bytes - cseg * kSeg) / 16;
#pragma unroll
    for (int u = 0; u < kSeg / 16 / 32; ++u) {
      const int c = 32 * u + lane;
      if (c < n) {
        if (u & 1) acc1 = dot8x8<T>(st[c], xs[c0 + c], acc1);
        else acc0 = dot8x8<T>(st[c], xs[c0 + c], acc0);
      }
    }
    if (cseg == nseg - 1) {
      const float sum = warp_sum(acc0 + acc1);
      const TO out = from_float<TO>(sum);
      if (lane == 0) y[crow] = out;
      if (kArgmax) {
        const uint64_t k = argmax_key(to_float(out), static_cast<uint32_t>(crow));
        best = k > best ? k : best;
      }
      acc0 = acc1 = 0.f;
    }
    if (++cseg == nseg) { cseg = 0; crow += total_warps; }
    __syncwarp();
  }
  cp_async_wait<0>();
  if (kArgmax) {
    __shared__ uint64_t s_best[kCpWarps];
    __shared__ uint64_t s_cta[1];
    if (lane == 0) s_best[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t b = 0;
      for (int i = 0; i < kCpWarps; ++i) b = s_best[i] > b ? s_best[i] : b;
      s_cta[0] = b;
    }
    __syncthreads();
    argmax_publish(s_cta, 1, am, gridDim.x);
  }
}

template <typename T, typename TO, bool kArgmax>
cudaError_t run_m1_cp_t(const void* W, int64_t ldw, const void* x, void* y, int N, int K,
                        const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const int smem = kRingBytes + K * 2;
  cudaError_t e = cudaFuncSetAttribute(dense_m1_cp_kernel<T, TO, kArgmax>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int grid = 2 * device_sm_count();
  const int need = (N + kCpWarps - 1) / kCpWarps;
  if (grid > need) grid = need;
  info->grid_x = grid;
  info->block = kCpThreads;
  info->smem = smem;
  info->kernel = "dense_m1_cp";
  return launch_k(dense_m1_cp_kernel<T, TO, kArgmax>, dim3(grid), dim3(kCpThreads), smem, st, true,
                  static_cast<const T*>(W), ldw, static_cast<const T*>(x), static_cast<TO*>(y), N,
                  K, am);
}

template <typename T, typename TO>
cudaError_t run_m1_cp(const void* W, int64_t ldw, const void* x, void* y, int N, int K,
                      const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  return am.out ? run_m1_cp_t<T, TO, true>(W, ldw, x, y, N, K, am, st, info)
                : run_m1_cp_t<T, TO, false>(W, ldw, x, y, N, K, am, st, info);
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
  pdl_launch_dependents();
  pdl_wait();

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
  return launch_k(dense_mn_kernel<T, TO, NC>, grid, dim3(kThreads), 0, st, true,
                  static_cast<const T*>(W), ldw, static_cast<const T*>(X), ldx, M,
                  static_cast<TO*>(Y), N, K, kps, s2, am);
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
  return launch_k(dense_m1_kernel<T, TO>, dim3(grid), dim3(kThreads), 0, st, true,
                  static_cast<const T*>(W), ldw, static_cast<const T*>(x), static_cast<TO*>(y), N,
                  K, am);
}

}  // namespace

cudaError_t launch_gemv_dense(int dtype, const void* W, int64_t ldw, const void* X, int64_t ldx,
                              int M, void* Y, int out_f32, int N, int K, const SplitArgs& sk,
                              const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const bool m1 = (M == 1 && sk.splits <= 1);
  // asynchronous copies: 16-byte aligned rows (checked by the caller), x in smem
  const bool cp = m1 && !m1_ldg_forced() && (kRingBytes + K * 2 <= 200 * 1024);
  if (dtype == 0) {
    if (out_f32) return cudaErrorInvalidValue;
    if (cp) return run_m1_cp<__half, __half>(W, ldw, X, Y, N, K, am, st, info);
    return m1 ? run_m1<__half, __half>(W, ldw, X, Y, N, K, am, st, info)
              : dispatch_mn<__half, __half>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  }
  if (!out_f32) return cudaErrorInvalidValue;
  if (cp) return run_m1_cp<__nv_bfloat16, float>(W, ldw, X, Y, N, K, am, st, info);
  return m1 ? run_m1<__nv_bfloat16, float>(W, ldw, X, Y, N, K, am, st, info)
            : dispatch_mn<__nv_bfloat16, float>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
}

}  // namespace wobs
