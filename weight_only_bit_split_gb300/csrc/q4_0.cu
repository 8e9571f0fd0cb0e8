// Q4_0 weights x Q8_1 activations decode GEMV, 1 to 32 columns.
//
// "The kernel that waited for itself" (m12-db-gemm case study): the Q4_0 x
// Q8_1 matrix product for a few activation columns, where the time goes
// into streaming the 4-bit weights and, second, into the VALU work of nibble
// unpacking and block scaling ("The VALU floor").  Per weight block b and
// column m the integer block dot sumi = sum_i (q4_i - 8) q8_i is exact:
// it is formed as sum_i q4_i q8_i - 8 sum_i q8_i with 4-way byte dot
// products (dp4a), the nibbles unpacked with two mask/shift ops per word.
// Only the block scaling d4 * d8 * sumi is floating point.
//
// M = 1: one warp per weight row, lanes strided over the row's blocks so a
// warp reads 512 contiguous bytes of nibbles per instruction; the
// activation blocks are staged once per CTA in shared memory as separate
// planes (low 16 codes, high 16 codes, scale, exact code sum) so lanes read
// them without bank conflicts; persistent grid over all rows.
//
// M > 1: each lane owns one weight row and walks its blocks; the activation
// blocks of the CTA's K range are staged in shared memory and read by
// broadcast, so every unpacked weight block is reused for all M columns
// from registers.  K is split across CTAs when the rows alone cannot fill
// the GPU; the last CTA of a row group adds the partials in a fixed order.
#include "common.cuh"

namespace wobs {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint16_t ld_stream_u16(const void* p, uint64_t pol) {
  uint16_t r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.u16 %0, [%1], %2;" : "=h"(r) : "l"(p), "l"(pol));
  return r;
}

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}

// Exact 32-element dot: sum over the 16 low-nibble and 16 high-nibble codes.
__device__ __forceinline__ int q4_dot_u(uint4 q, int4 lo, int4 hi) {
  int s = 0;
  s = __dp4a(static_cast<int>(q.x & 0x0F0F0F0Fu), lo.x, s);
  s = __dp4a(static_cast<int>(q.y & 0x0F0F0F0Fu), lo.y, s);
  s = __dp4a(static_cast<int>(q.z & 0x0F0F0F0Fu), lo.z, s);
  s = __dp4a(static_cast<int>(q.w & 0x0F0F0F0Fu), lo.w, s);
  s = __dp4a(static_cast<int>((q.x >> 4) & 0x0F0F0F0Fu), hi.x, s);
  s = __dp4a(static_cast<int>((q.y >> 4) & 0x0F0F0F0Fu), hi.y, s);
  s = __dp4a(static_cast<int>((q.z >> 4) & 0x0F0F0F0Fu), hi.z, s);
  s = __dp4a(static_cast<int>((q.w >> 4) & 0x0F0F0F0Fu), hi.w, s);
  return s;
}

// Read one 36-byte Q8_1 block {half d; half s; int8 q[32]} (4-byte aligned).
struct XBlock {
  int4 lo, hi;  // codes 0..15, 16..31
  float d;      // fp16 scale widened
  int s;        // exact sum of the 32 codes
};
__device__ __forceinline__ XBlock load_xblock(const uint8_t* blk) {
  const uint32_t* w = reinterpret_cast<const uint32_t*>(blk);
  XBlock r;
  const uint32_t ds = __ldg(w);
  r.d = half_bits_to_float(static_cast<uint16_t>(ds & 0xFFFFu));
  r.lo = make_int4(__ldg(w + 1), __ldg(w + 2), __ldg(w + 3), __ldg(w + 4));
  r.hi = make_int4(__ldg(w + 5), __ldg(w + 6), __ldg(w + 7), __ldg(w + 8));
  int s = 0;
  s = __dp4a(r.lo.x, 0x01010101, s); s = __dp4a(r.lo.y, 0x01010101, s);
  s = __dp4a(r.lo.z, 0x01010101, s); s = __dp4a(r.lo.w, 0x01010101, s);
  s = __dp4a(r.hi.x, 0x01010101, s); s = __dp4a(r.hi.y, 0x01010101, s);
  s = __dp4a(r.hi.z, 0x01010101, s); s = __dp4a(r.hi.w, 0x01010101, s);
  r.s = s;
  return r;
}

// ------------------------------------------------------------- M = 1

template <int U>
__global__ void __launch_bounds__(kThreads) q4_m1_kernel(const uint8_t* __restrict__ qs,
                                                          const uint16_t* __restrict__ d4,
                                                          const uint8_t* __restrict__ xq,
                                                          float* __restrict__ y, int N, int K,
                                                          ArgmaxArgs am) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int nb = K >> 5;
  int4* x_lo = reinterpret_cast<int4*>(smem);
  int4* x_hi = x_lo + nb;
  float* x_d = reinterpret_cast<float*>(x_hi + nb);
  int* x_s = reinterpret_cast<int*>(x_d + nb);
  const uint64_t pol = l2_evict_first_policy();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total_warps = gridDim.x * kWarps;
  int row = blockIdx.x * kWarps + warp;

  // Weight loads of this warp's first row go out before the activation
  // staging, which only depends on a small L2-resident vector.
  uint4 q[U];
  uint16_t dh[U];
  const bool full = (nb % (32 * U)) == 0;
  if (full && row < N) {
    const uint4* qrow = reinterpret_cast<const uint4*>(qs + static_cast<int64_t>(row) * (K >> 1));
    const uint16_t* drow = d4 + static_cast<int64_t>(row) * nb;
#pragma unroll
    for (int u = 0; u < U; ++u) q[u] = ld_stream16(qrow + lane + 32 * u, pol);
#pragma unroll
    for (int u = 0; u < U; ++u) dh[u] = ld_stream_u16(drow + lane + 32 * u, pol);
  }
  for (int b = threadIdx.x; b < nb; b += kThreads) {
    const XBlock xb = load_xblock(xq + 36 * static_cast<int64_t>(b));
    x_lo[b] = xb.lo;
    x_hi[b] = xb.hi;
    x_d[b] = xb.d;
    x_s[b] = xb.s;
  }
  __syncthreads();

  uint64_t best = 0;
  for (; row < N; row += total_warps) {
    const uint4* qrow = reinterpret_cast<const uint4*>(qs + static_cast<int64_t>(row) * (K >> 1));
    const uint16_t* drow = d4 + static_cast<int64_t>(row) * nb;
    float acc0 = 0.f, acc1 = 0.f;
    int b = lane;
    if (full) {
      for (; b < nb; b += 32 * U) {
        if (b != lane) {
#pragma unroll
          for (int u = 0; u < U; ++u) q[u] = ld_stream16(qrow + b + 32 * u, pol);
#pragma unroll
          for (int u = 0; u < U; ++u) dh[u] = ld_stream_u16(drow + b + 32 * u, pol);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int bb = b + 32 * u;
          const int dot = q4_dot_u(q[u], x_lo[bb], x_hi[bb]) - 8 * x_s[bb];
          const float sc = half_bits_to_float(dh[u]) * x_d[bb];
          if (u & 1) acc1 = fmaf(static_cast<float>(dot), sc, acc1);
          else acc0 = fmaf(static_cast<float>(dot), sc, acc0);
        }
      }
      // prefetch the next row's first chunk before the reduction
      const int nrow = row + total_warps;
      if (nrow < N) {
        const uint4* nq = reinterpret_cast<const uint4*>(qs + static_cast<int64_t>(nrow) * (K >> 1));
        const uint16_t* nd = d4 + static_cast<int64_t>(nrow) * nb;
#pragma unroll
        for (int u = 0; u < U; ++u) q[u] = ld_stream16(nq + lane + 32 * u, pol);
#pragma unroll
        for (int u = 0; u < U; ++u) dh[u] = ld_stream_u16(nd + lane + 32 * u, pol);
      }
    } else {
      for (; b < nb; b += 32) {
        const uint4 qq = ld_stream16(qrow + b, pol);
        const uint16_t dd = ld_stream_u16(drow + b, pol);
        const int dot = q4_dot_u(qq, x_lo[b], x_hi[b]) - 8 * x_s[b];
        acc0 = fmaf(static_cast<float>(dot), half_bits_to_float(dd) * x_d[b], acc0);
      }
    }
    const float s = warp_sum(acc0 + acc1);
    if (lane == 0) y[row] = s;
    if (am.out) {
      const uint64_t k = argmax_key(s, static_cast<uint32_t>(row));
      best = k > best ? k : best;
    }
  }
  if (am.out) {
    __shared__ uint64_t s_best[kWarps];
    __shared__ uint64_t s_cta[1];
    if (lane == 0) s_best[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t bk = 0;
      for (int i = 0; i < kWarps; ++i) bk = s_best[i] > bk ? s_best[i] : bk;
      s_cta[0] = bk;
    }
    __syncthreads();
    argmax_publish(s_cta, 1, am, gridDim.x);
  }
}

// --------------------------------------------------------- M columns

struct __align__(16) XS {
  int4 lo, hi;
  float d;
  int s;
  int pad0, pad1;
};

template <int NC>
__global__ void __launch_bounds__(kThreads) q4_mn_kernel(const uint8_t* __restrict__ qs,
                                                          const uint16_t* __restrict__ d4,
                                                          const uint8_t* __restrict__ xq, int M,
                                                          float* __restrict__ Y, int N, int K,
                                                          int bps, SplitArgs sk, ArgmaxArgs am) {
  extern __shared__ __align__(16) uint8_t smem[];
  XS* xs = reinterpret_cast<XS*>(smem);   // [bps][NC]
  const int nb = K >> 5;
  const int row = blockIdx.x * kThreads + threadIdx.x;
  const bool valid = row < N;
  const int s = blockIdx.y;
  const int b0 = s * bps;
  const int b1 = min(nb, b0 + bps);
  for (int i = threadIdx.x; i < (b1 - b0) * NC; i += kThreads) {
    const int bl = i / NC, m = i - bl * NC;
    XS v;
    if (m < M) {
      const XBlock xb = load_xblock(xq + 36 * (static_cast<int64_t>(m) * nb + b0 + bl));
      v.lo = xb.lo; v.hi = xb.hi; v.d = xb.d; v.s = xb.s;
    } else {
      v.lo = make_int4(0, 0, 0, 0); v.hi = v.lo; v.d = 0.f; v.s = 0;
    }
    v.pad0 = v.pad1 = 0;
    xs[i] = v;
  }
  __syncthreads();

  float acc[NC];
#pragma unroll
  for (int m = 0; m < NC; ++m) acc[m] = 0.f;
  if (valid) {
    const uint4* qrow = reinterpret_cast<const uint4*>(qs + static_cast<int64_t>(row) * (K >> 1));
    const uint16_t* drow = d4 + static_cast<int64_t>(row) * nb;
    for (int b = b0; b < b1; ++b) {
      const uint4 q = __ldg(qrow + b);
      const float dw = half_bits_to_float(__ldg(drow + b));
      const XS* xb = xs + (b - b0) * NC;
#pragma unroll
      for (int m = 0; m < NC; ++m) {
        const int dot = q4_dot_u(q, xb[m].lo, xb[m].hi) - 8 * xb[m].s;
        acc[m] = fmaf(static_cast<float>(dot), dw * xb[m].d, acc[m]);
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
  if (valid) {
#pragma unroll
    for (int m = 0; m < NC; ++m)
      if (m < M) Y[static_cast<int64_t>(m) * N + row] = acc[m];
  }
  if (am.out) {
    __shared__ uint64_t s_key[kWarps][NC];
    __shared__ uint64_t s_cta[NC];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int m = 0; m < NC; ++m) {
      uint64_t k = valid ? argmax_key(acc[m], static_cast<uint32_t>(row)) : 0ull;
      k = warp_max_u64(k);
      if (lane == 0) s_key[warp][m] = k;
    }
    __syncthreads();
    if (threadIdx.x < NC) {
      uint64_t bk = 0;
      for (int w = 0; w < kWarps; ++w) bk = s_key[w][threadIdx.x] > bk ? s_key[w][threadIdx.x] : bk;
      s_cta[threadIdx.x] = bk;
    }
    __syncthreads();
    argmax_publish(s_cta, M, am, gridDim.x);
  }
}

template <int NC>
cudaError_t run_mn(const uint8_t* qs, const void* d, const void* xq, int M, float* Y, int N,
                   int K, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                   Launch* info) {
  const int nb = K / 32;
  const int bps = (nb + sk.splits - 1) / sk.splits;
  const int splits = (nb + bps - 1) / bps;
  const int smem = bps * NC * static_cast<int>(sizeof(XS));
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(q4_mn_kernel<NC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((N + kThreads - 1) / kThreads, splits);
  SplitArgs s2 = sk;
  s2.splits = splits;
  info->grid_x = grid.x;
  info->grid_y = grid.y;
  info->block = kThreads;
  info->smem = smem;
  info->kernel = "q4_0_q8_1_mn";
  q4_mn_kernel<NC><<<grid, kThreads, smem, st>>>(qs, static_cast<const uint16_t*>(d),
                                                  static_cast<const uint8_t*>(xq), M, Y, N, K,
                                                  bps, s2, am);
  return cudaGetLastError();
}

template <int U>
cudaError_t run_m1(const uint8_t* qs, const void* d, const void* xq, float* y, int N, int K,
                   const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const int nb = K / 32;
  const int smem = nb * 40;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(q4_m1_kernel<U>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  const int per_sm = max_resident_ctas(reinterpret_cast<const void*>(q4_m1_kernel<U>), kThreads, smem);
  int grid = device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int need = (N + kWarps - 1) / kWarps;
  if (grid > need) grid = need;
  info->grid_x = grid;
  info->block = kThreads;
  info->smem = smem;
  info->kernel = U == 4 ? "q4_0_q8_1_m1_u4" : (U == 2 ? "q4_0_q8_1_m1_u2" : "q4_0_q8_1_m1_u1");
  q4_m1_kernel<U><<<grid, kThreads, smem, st>>>(qs, static_cast<const uint16_t*>(d),
                                                 static_cast<const uint8_t*>(xq), y, N, K, am);
  return cudaGetLastError();
}

// ------------------------------------------------------- block dots

__global__ void __launch_bounds__(kThreads) q4_blockdots_kernel(const uint8_t* __restrict__ qs,
                                                                 const uint8_t* __restrict__ xq,
                                                                 int M, int N, int K,
                                                                 int32_t* __restrict__ out) {
  const int nb = K >> 5;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t total = static_cast<int64_t>(M) * N * nb;
  if (t >= total) return;
  const int b = static_cast<int>(t % nb);
  const int64_t mn = t / nb;
  const int n = static_cast<int>(mn % N);
  const int m = static_cast<int>(mn / N);
  const uint4 q = __ldg(reinterpret_cast<const uint4*>(qs + static_cast<int64_t>(n) * (K >> 1)) + b);
  const XBlock xb = load_xblock(xq + 36 * (static_cast<int64_t>(m) * nb + b));
  out[t] = q4_dot_u(q, xb.lo, xb.hi) - 8 * xb.s;
}

}  // namespace

cudaError_t launch_gemv_q4_0_q8_1(const uint8_t* qs, const void* d, const void* xq, int M,
                                  float* Y, int N, int K, const SplitArgs& sk,
                                  const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  if (M == 1 && sk.splits <= 1) {
    const int nb = K / 32;
    if (nb % 128 == 0) return run_m1<4>(qs, d, xq, Y, N, K, am, st, info);
    if (nb % 64 == 0) return run_m1<2>(qs, d, xq, Y, N, K, am, st, info);
    return run_m1<1>(qs, d, xq, Y, N, K, am, st, info);
  }
  if (M <= 1) return run_mn<1>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 2) return run_mn<2>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 4) return run_mn<4>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 8) return run_mn<8>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 12) return run_mn<12>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 16) return run_mn<16>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 24) return run_mn<24>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  return run_mn<32>(qs, d, xq, M, Y, N, K, sk, am, st, info);
}

cudaError_t launch_q4_0_q8_1_blockdots(const uint8_t* qs, const void* xq, int M, int N, int K,
                                       int32_t* out, cudaStream_t st, Launch* info) {
  const int64_t total = static_cast<int64_t>(M) * N * (K / 32);
  const int64_t grid = (total + kThreads - 1) / kThreads;
  info->grid_x = static_cast<int>(grid);
  info->block = kThreads;
  info->kernel = "q4_0_q8_1_blockdots";
  q4_blockdots_kernel<<<static_cast<unsigned>(grid), kThreads, 0, st>>>(
      qs, static_cast<const uint8_t*>(xq), M, N, K, out);
  return cudaGetLastError();
}

}  // namespace wobs
