// Q8_0 weights: the quantiser and the Q8_0 x Q8_1 decode GEMV, 1 to 32
// activation columns.
//
// "The kernel that waited for itself" (m12-db-gemm case study), section
// "What correctness was measured against": the decode matrix path is
// exercised on Q4_0 and Q8_0 weights.  A Q8_0 block is 32 int8 codes and
// one fp16 scale, 1.0625 bytes per weight.  Per weight block b and
// activation column m the block dot sumi = sum_i qw_i * q8_{m,i} is exact
// (eight signed 4-way byte dot products); only the scaling dw * d8 * sumi
// is floating point.
//
// GEMV design (sm_103a): one warp per weight row, lanes along K, rows
// round-robin over every CTA; each warp streams its rows through its own
// two-slot ring of 2176-byte segments (64 blocks: their 2048 code bytes as
// in memory, then their 64 scales) filled by 16-byte cp.async.  Shared and
// global addresses of every copy are both lane-contiguous: a copy whose
// shared side is scattered makes the L1 fetch each sector once per pass
// (measured on GB300: twice the DRAM bytes over the crossbar and half the
// streaming rate).  A lane takes 16-byte chunks, half a block each, dots
// the 16 codes with the matching half of the Q8_1 activation block (staged
// once per CTA in the same chunk order, so those reads are lane-contiguous
// too) and scales the exact half-block sum by dw * d8.  Up to eight columns
// share each weight chunk, read once; more are taken eight at a time.
#include "common.cuh"

namespace wobs {
namespace {

// ---------------------------------------------------------------- quantise

constexpr int kQThreads = 256;

// One warp per 32-element block, one element per lane; IEEE float32
// division and roundf, as the format defines.
__global__ void __launch_bounds__(kQThreads) q8_0_quant_kernel(const float* __restrict__ W,
                                                                int64_t ldw, int N, int K,
                                                                int8_t* __restrict__ qs,
                                                                __half* __restrict__ d) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * kQThreads + threadIdx.x) >> 5;
  const int nb = K >> 5;
  if (wid >= static_cast<int64_t>(N) * nb) return;   // whole warp
  const int n = static_cast<int>(wid / nb);
  const int b = static_cast<int>(wid - static_cast<int64_t>(n) * nb);
  const float w = W[static_cast<int64_t>(n) * ldw + 32 * b + lane];
  float amax = fabsf(w);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float dd = amax / 127.0f;
  const int q = dd != 0.0f ? static_cast<int>(roundf(w / dd)) : 0;
  qs[static_cast<int64_t>(n) * K + 32 * b + lane] = static_cast<int8_t>(q);
  if (lane == 0) d[static_cast<int64_t>(n) * nb + b] = __float2half_rn(dd);
}

// -------------------------------------------------------------------- GEMV

constexpr int kSegBlocks = 64;                  // blocks per ring segment
constexpr int kScaleOff = kSegBlocks * 32;      // codes, then the segment's scales
constexpr int kSegBytes = kScaleOff + kSegBlocks * 2;
constexpr int kRing = 2;

template <int MC>
struct Q8Shape {
  static constexpr int kWarps = MC >= 8 ? 12 : 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRingBytes = kWarps * kRing * kSegBytes;
};

template <int MC>
constexpr int q8_smem(int nb) {
  return Q8Shape<MC>::kRingBytes + MC * nb * 36;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
               :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// Signed dot of 16 weight codes with 16 activation codes (exact).
__device__ __forceinline__ int q8_dot16(uint4 w, int4 x) {
  int s = 0;
  s = __dp4a(static_cast<int>(w.x), x.x, s);
  s = __dp4a(static_cast<int>(w.y), x.y, s);
  s = __dp4a(static_cast<int>(w.z), x.z, s);
  s = __dp4a(static_cast<int>(w.w), x.w, s);
  return s;
}

// Q8_1 quantisation of one fp32 activation vector into this kernel's
// planes (code chunks in block order, fp16-rounded scales), every CTA the
// whole vector, taking the quantiser's decisions (q8_1_part_block: TPB lanes
// per 32-block, amax, d = amax / 127 in IEEE float32, q = roundf(x / d), 0
// when d = 0).  Block b's 36-byte Q8_1 block is also written to xq_out (when
// given) by CTA b mod grid.  All NT threads call this with the same trip
// count, so the group shuffles see whole warps.
template <int NT, int TPB>
__device__ __forceinline__ void q8_planes_tpb(const float* __restrict__ X, int nb, int4* x_c,
                                              float* x_d, uint8_t* __restrict__ xq_out) {
  constexpr int kPerPass = NT / TPB;
  constexpr int kW = 8 / TPB;
  const int j = threadIdx.x & (TPB - 1);
  const int passes = (nb + kPerPass - 1) / kPerPass;
  for (int p = 0; p < passes; ++p) {
    const int b = p * kPerPass + static_cast<int>(threadIdx.x) / TPB;
    const bool valid = b < nb;
    float4 v[kW];
    const float4* src = reinterpret_cast<const float4*>(X + 32 * b) + kW * j;
#pragma unroll
    for (int i = 0; i < kW; ++i) v[i] = valid ? __ldg(src + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    const Q81Part<TPB> h = q8_1_part_block<TPB>(v);
    if (!valid) continue;
    uint32_t* dst = reinterpret_cast<uint32_t*>(x_c) + 8 * b + kW * j;   // chunks 2b, 2b + 1
#pragma unroll
    for (int i = 0; i < kW; ++i) dst[i] = h.codes[i];
    if (j == 0) x_d[b] = __half2float(__float2half_rn(h.d));
    if (xq_out != nullptr && b % static_cast<int>(gridDim.x) == static_cast<int>(blockIdx.x))
      store_q8_1_part<TPB>(xq_out + 36 * static_cast<int64_t>(b), h, j);
  }
}

template <int NT>
__device__ __forceinline__ void q8_planes_from_f32(const float* __restrict__ X, int nb, int4* x_c,
                                                   float* x_d, uint8_t* __restrict__ xq_out) {
  const int tpb = q8_1_lanes_per_block<NT>(nb);
  if (tpb == 8) q8_planes_tpb<NT, 8>(X, nb, x_c, x_d, xq_out);
  else if (tpb == 4) q8_planes_tpb<NT, 4>(X, nb, x_c, x_d, xq_out);
  else q8_planes_tpb<NT, 2>(X, nb, x_c, x_d, xq_out);
}

// Columns [0, M) of this launch (M <= MC); xq, Y and the argmax state are
// already offset to the launch's first column.  kF32X (MC = 1): xq is the
// fp32 activation vector, quantised in the prologue; W warps per CTA.
template <int MC, bool kArgmax, bool kF32X = false, int W = Q8Shape<MC>::kWarps>
__global__ void __launch_bounds__(W * 32) q8_mc_cp_kernel(
    const int8_t* __restrict__ qs, const uint16_t* __restrict__ dw, const uint8_t* __restrict__ xq,
    int M, float* __restrict__ Y, int N, int K, ArgmaxArgs am, uint8_t* __restrict__ xq_out) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int nb = K >> 5;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total_warps = gridDim.x * W;
  const int wg = warp * gridDim.x + blockIdx.x;   // rows round-robin over the CTAs first
  const int nseg = (nb + kSegBlocks - 1) / kSegBlocks;
  const int rows_w = wg < N ? (N - 1 - wg) / total_warps + 1 : 0;
  const int T = rows_w * nseg;
  uint8_t* myring = smem + warp * (kRing * kSegBytes);
  int4* x_c = reinterpret_cast<int4*>(smem + W * kRing * kSegBytes);     // [MC][2 nb] code chunks
  float* x_d = reinterpret_cast<float*>(x_c + 2 * MC * nb);                 // [MC][nb] scales

  int prow = wg, pseg = 0;   // next segment to request
  auto issue = [&](int slot) {
    uint8_t* st = myring + slot * kSegBytes;
    const int b0 = pseg * kSegBlocks;
    const int n = min(kSegBlocks, nb - b0);
    const int8_t* qr = qs + static_cast<int64_t>(prow) * K + 32 * b0;
#pragma unroll
    for (int u = 0; u < 2 * kSegBlocks / 32; ++u) {
      const int c = 32 * u + lane;                 // 16-byte chunk of the segment's codes
      if (c < 2 * n) cp_async16(st + 16 * c, qr + 16 * c);
    }
    const uint16_t* dr = dw + static_cast<int64_t>(prow) * nb + b0;
    if (lane < n / 8) cp_async16(st + kScaleOff + 16 * lane, dr + 8 * lane);
    if (++pseg == nseg) { pseg = 0; prow += total_warps; }
  };
  // the first kRing-1 segments are requested before waiting for the
  // previous kernel: weights are never written by a decode-path kernel
#pragma unroll
  for (int i = 0; i < kRing - 1; ++i) {
    if (i < T) issue(i);
    cp_async_commit();
  }
  pdl_launch_dependents();
  pdl_wait();
  if constexpr (kF32X) {
    q8_planes_from_f32<W * 32>(reinterpret_cast<const float*>(xq), nb, x_c, x_d, xq_out);
  } else {
  for (int i = threadIdx.x; i < MC * nb; i += W * 32) {
    const int m = i / nb, b = i - m * nb;
    if (m < M) {
      const uint32_t* blk = reinterpret_cast<const uint32_t*>(xq + 36 * (static_cast<int64_t>(m) * nb + b));
      x_d[i] = __half2float(__ushort_as_half(static_cast<unsigned short>(__ldg(blk) & 0xFFFFu)));
      x_c[2 * i] = make_int4(__ldg(blk + 1), __ldg(blk + 2), __ldg(blk + 3), __ldg(blk + 4));
      x_c[2 * i + 1] = make_int4(__ldg(blk + 5), __ldg(blk + 6), __ldg(blk + 7), __ldg(blk + 8));
    } else {
      x_d[i] = 0.f;
      x_c[2 * i] = make_int4(0, 0, 0, 0);
      x_c[2 * i + 1] = make_int4(0, 0, 0, 0);
    }
  }
  }
  __syncthreads();

  int crow = wg, cseg = 0;
  float acc[MC];
#pragma unroll
  for (int m = 0; m < MC; ++m) acc[m] = 0.f;
  uint64_t best[MC];
#pragma unroll
  for (int m = 0; m < MC; ++m) best[m] = 0ull;
  for (int t = 0; t < T; ++t) {
    // request segment t+kRing-1 into the slot consumed last, wait for segment t
    if (t + kRing - 1 < T) issue((t + kRing - 1) % kRing);
    cp_async_commit();
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint8_t* st = myring + (t % kRing) * kSegBytes;
    const int b0 = cseg * kSegBlocks;
    const int n = min(kSegBlocks, nb - b0);
#pragma unroll
    for (int u = 0; u < 2 * kSegBlocks / 32; ++u) {
      const int c = 32 * u + lane;              // chunk: half (c & 1) of block b0 + (c >> 1)
      if (c < 2 * n) {
        const uint4 wc = *reinterpret_cast<const uint4*>(st + 16 * c);
        const float dwf = __half2float(__ushort_as_half(
            *reinterpret_cast<const unsigned short*>(st + kScaleOff + 2 * (c >> 1))));
        const int b = b0 + (c >> 1);
#pragma unroll
        for (int m = 0; m < MC; ++m) {
          const int dot = q8_dot16(wc, x_c[2 * (m * nb + b0) + c]);
          acc[m] = fmaf(static_cast<float>(dot), dwf * x_d[m * nb + b], acc[m]);
        }
      }
    }
    if (cseg == nseg - 1) {
#pragma unroll
      for (int m = 0; m < MC; ++m) {
        const float sum = warp_sum(acc[m]);
        if (m < M) {
          if (lane == m) Y[static_cast<int64_t>(m) * N + crow] = sum;
          if (kArgmax) {
            const uint64_t k = argmax_key(sum, static_cast<uint32_t>(crow));
            best[m] = k > best[m] ? k : best[m];
          }
        }
        acc[m] = 0.f;
      }
    }
    if (++cseg == nseg) { cseg = 0; crow += total_warps; }
    __syncwarp();
  }
  cp_async_wait<0>();
  if (kArgmax) {
    __shared__ uint64_t s_best[W][MC];
    __shared__ uint64_t s_cta[MC];
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < MC; ++m) s_best[warp][m] = best[m];
    }
    __syncthreads();
    if (threadIdx.x < MC) {
      uint64_t bk = 0;
      for (int i = 0; i < W; ++i) bk = s_best[i][threadIdx.x] > bk ? s_best[i][threadIdx.x] : bk;
      s_cta[threadIdx.x] = bk;
    }
    __syncthreads();
    argmax_publish(s_cta, M, am, gridDim.x);
  }
}

int optin_smem() {
  static int v = [] {
    int dev = 0, o = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&o, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return 0;
    return o;
  }();
  return v;
}

template <int MC, bool kArgmax>
cudaError_t run_t(const int8_t* qs, const uint16_t* d, const uint8_t* xq, int M, float* Y, int N,
                  int K, const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  constexpr int W = Q8Shape<MC>::kWarps;
  const int smem = q8_smem<MC>(K / 32);
  auto kern = q8_mc_cp_kernel<MC, kArgmax>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int per_sm = max_resident_ctas(reinterpret_cast<const void*>(kern), W * 32, smem);
  int grid = device_sm_count() * (per_sm > 0 ? per_sm : 1);
  if (grid > N) grid = N;
  info->grid_x = grid;
  info->block = W * 32;
  info->smem = smem;
  info->kernel = "q8_0_q8_1_mc_cp";
  return launch_k(kern, dim3(grid), dim3(W * 32), smem, st, true, qs, d, xq, M, Y, N, K, am,
                  static_cast<uint8_t*>(nullptr));
}

// The fused entry: 32 warps and one CTA per SM (each SM quantises x once)
// when the ring and planes fit, else 16 warps and two CTAs per SM.
template <bool kArgmax, int W>
cudaError_t run_fused_t(const int8_t* qs, const uint16_t* d, const float* x, uint8_t* xq_out,
                        float* Y, int N, int K, const ArgmaxArgs& am, cudaStream_t st,
                        Launch* info) {
  const int smem = W * kRing * kSegBytes + (K / 32) * 36;
  auto kern = q8_mc_cp_kernel<1, kArgmax, true, W>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int grid = (W >= 32 ? 1 : 2) * device_sm_count();
  if (grid > N) grid = N;
  info->grid_x = grid;
  info->block = W * 32;
  info->smem = smem;
  info->kernel = "q8_0_f32_m1_cp";
  return launch_k(kern, dim3(grid), dim3(W * 32), smem, st, true, qs, d,
                  reinterpret_cast<const uint8_t*>(x), 1, Y, N, K, am, xq_out);
}

int fused_warps(int K) {
  if (32 * kRing * kSegBytes + (K / 32) * 36 <= 220 * 1024) return 32;
  // 1 KB left for the kernel's static shared memory (argmax keys)
  if (16 * kRing * kSegBytes + (K / 32) * 36 <= optin_smem() - 1024) return 16;
  return 0;
}

template <int MC>
cudaError_t run(const int8_t* qs, const uint16_t* d, const uint8_t* xq, int M, float* Y, int N,
                int K, const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  return am.out ? run_t<MC, true>(qs, d, xq, M, Y, N, K, am, st, info)
                : run_t<MC, false>(qs, d, xq, M, Y, N, K, am, st, info);
}

}  // namespace

cudaError_t launch_quantize_q8_0(const float* W, int64_t ldw, int N, int K, int8_t* qs, void* d,
                                 cudaStream_t st, Launch* info) {
  const int64_t warps = static_cast<int64_t>(N) * (K / 32);
  const int64_t grid = (warps * 32 + kQThreads - 1) / kQThreads;
  info->grid_x = static_cast<int>(grid);
  info->block = kQThreads;
  info->kernel = "quantize_q8_0";
  q8_0_quant_kernel<<<static_cast<unsigned>(grid), kQThreads, 0, st>>>(W, ldw, N, K, qs,
                                                                        static_cast<__half*>(d));
  return cudaGetLastError();
}

bool q8_0_f32_fused_applies(int K) { return fused_warps(K) > 0; }

cudaError_t launch_gemv_q8_0_f32_fused(const int8_t* qs, const void* d, const float* x,
                                       void* xq_out, float* y, int N, int K, const ArgmaxArgs& am,
                                       cudaStream_t st, Launch* info) {
  const int w = fused_warps(K);
  if (w == 0) return cudaErrorNotSupported;
  const uint16_t* dp = static_cast<const uint16_t*>(d);
  uint8_t* xo = static_cast<uint8_t*>(xq_out);
  if (w == 32)
    return am.out ? run_fused_t<true, 32>(qs, dp, x, xo, y, N, K, am, st, info)
                  : run_fused_t<false, 32>(qs, dp, x, xo, y, N, K, am, st, info);
  return am.out ? run_fused_t<true, 16>(qs, dp, x, xo, y, N, K, am, st, info)
                : run_fused_t<false, 16>(qs, dp, x, xo, y, N, K, am, st, info);
}

int q8_0_columns_per_launch(int K) {
  const int nb = K / 32, lim = optin_smem();
  if (q8_smem<8>(nb) <= lim) return 8;
  if (q8_smem<4>(nb) <= lim) return 4;
  if (q8_smem<2>(nb) <= lim) return 2;
  if (q8_smem<1>(nb) <= lim) return 1;
  return 0;
}

cudaError_t launch_gemv_q8_0_q8_1(const int8_t* qs, const void* d, const void* xq, int M, float* Y,
                                  int N, int K, const ArgmaxArgs& am, cudaStream_t st,
                                  Launch* info) {
  const int cmax = q8_0_columns_per_launch(K);
  if (cmax == 0) return cudaErrorNotSupported;
  const uint16_t* dp = static_cast<const uint16_t*>(d);
  const uint8_t* xp = static_cast<const uint8_t*>(xq);
  const int64_t xcol = 36ll * (K / 32);
  // columns eight (or fewer, for long rows) at a time; each launch's argmax
  // state starts at its first column
  for (int m0 = 0; m0 < M; m0 += cmax) {
    const int mc = M - m0 < cmax ? M - m0 : cmax;
    ArgmaxArgs a = am;
    if (am.out) {
      a.out = am.out + m0;
      a.keys = am.keys + m0;
    }
    const uint8_t* xm = xp + m0 * xcol;
    float* ym = Y + static_cast<int64_t>(m0) * N;
    cudaError_t e;
    if (mc == 1) e = run<1>(qs, dp, xm, mc, ym, N, K, a, st, info);
    else if (mc == 2) e = run<2>(qs, dp, xm, mc, ym, N, K, a, st, info);
    else if (mc <= 4) e = run<4>(qs, dp, xm, mc, ym, N, K, a, st, info);
    else e = run<8>(qs, dp, xm, mc, ym, N, K, a, st, info);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace wobs
