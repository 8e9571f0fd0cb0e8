// Quantisers: Q8_1 activations (hot path, once per decode step) and the
// Q4_0 / NF4 weight formats (once per model load).
//
// Formats: "The kernel that waited for itself" (m12-db-gemm case study),
// section "Seven variants, one microbenchmark, many mistakes" -- Q4_0
// weights, Q8_1 activations; bitsandbytes issue #1842, "Minimal Repro" --
// NF4 blockwise (64) quantisation.  Every decision is taken in IEEE float32
// exactly as the format defines it (true division, roundf, no contraction),
// so the outputs are bit-identical to the definition.
#include "common.cuh"

namespace wobs {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------- Q8_1
// Eight threads per 32-element block, four elements each.
__global__ void __launch_bounds__(kThreads) q8_1_kernel(const float* __restrict__ X, int64_t ldx,
                                                         int M, int K, uint8_t* __restrict__ xq) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int per_col = K >> 2;
  const int64_t total = static_cast<int64_t>(M) * per_col;
  const bool valid = t < total;   // groups of 8 are either all valid or all not
  const int m = valid ? static_cast<int>(t / per_col) : 0;
  const int k4 = valid ? static_cast<int>(t - static_cast<int64_t>(m) * per_col) : 0;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  pdl_launch_dependents();
  pdl_wait();
  if (valid) v = *reinterpret_cast<const float4*>(X + static_cast<int64_t>(m) * ldx + 4 * k4);
  float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float d = amax / 127.0f;
  int q0 = 0, q1 = 0, q2 = 0, q3 = 0;
  if (d != 0.0f) {
    q0 = static_cast<int>(roundf(v.x / d));
    q1 = static_cast<int>(roundf(v.y / d));
    q2 = static_cast<int>(roundf(v.z / d));
    q3 = static_cast<int>(roundf(v.w / d));
  }
  int sum = q0 + q1 + q2 + q3;
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (!valid) return;
  uint8_t* blk = xq + (static_cast<int64_t>(m) * (K >> 5) + (k4 >> 3)) * 36;
  if ((k4 & 7) == 0) {
    const float s = d * static_cast<float>(sum);
    const __half2 ds = __halves2half2(__float2half_rn(d), __float2half_rn(s));
    *reinterpret_cast<__half2*>(blk) = ds;
  }
  const uint32_t packed = (static_cast<uint32_t>(q0) & 0xFFu) | ((static_cast<uint32_t>(q1) & 0xFFu) << 8) |
                          ((static_cast<uint32_t>(q2) & 0xFFu) << 16) | (static_cast<uint32_t>(q3) << 24);
  *reinterpret_cast<uint32_t*>(blk + 4 + 4 * (k4 & 7)) = packed;
}

// ---------------------------------------------------------------- Q4_0
// One warp per 32-element block, one element per lane.
__global__ void __launch_bounds__(kThreads) q4_0_quant_kernel(const float* __restrict__ W,
                                                               int64_t ldw, int N, int K,
                                                               uint8_t* __restrict__ qs,
                                                               __half* __restrict__ d) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int nb = K >> 5;
  if (wid >= static_cast<int64_t>(N) * nb) return;   // whole warp
  const int n = static_cast<int>(wid / nb);
  const int b = static_cast<int>(wid - static_cast<int64_t>(n) * nb);
  const float w = W[static_cast<int64_t>(n) * ldw + 32 * b + lane];
  // largest magnitude, lowest index on ties
  uint64_t key = (static_cast<uint64_t>(__float_as_uint(fabsf(w))) << 32) | static_cast<uint64_t>(31 - lane);
  key = warp_max_u64(key);
  const int src = 31 - static_cast<int>(key & 0xFFFFFFFFu);
  const float amax = __shfl_sync(0xffffffffu, w, src);
  const float dd = amax / -8.0f;
  int q = 8;
  if (dd != 0.0f) q = min(15, max(0, static_cast<int>(roundf(w / dd)) + 8));
  const int qhi = __shfl_down_sync(0xffffffffu, q, 16);
  if (lane < 16) qs[static_cast<int64_t>(n) * (K >> 1) + 16 * b + lane] = static_cast<uint8_t>(q | (qhi << 4));
  if (lane == 0) d[static_cast<int64_t>(n) * nb + b] = __float2half_rn(dd);
}

// ----------------------------------------------------------------- NF4
// One warp per 64-element block, two elements per lane.
__device__ __forceinline__ int nearest_level(float v, const Codebook16& cb) {
  float best = fabsf(cb.v[0] - v);
  int code = 0;
#pragma unroll
  for (int k = 1; k < 16; ++k) {
    const float dist = fabsf(cb.v[k] - v);
    if (dist < best) { best = dist; code = k; }
  }
  return code;
}

__global__ void __launch_bounds__(kThreads) nf4_quant_kernel(const __nv_bfloat16* __restrict__ W,
                                                              int64_t ldw, int N, int K,
                                                              Codebook16 cb,
                                                              uint8_t* __restrict__ qs,
                                                              float* __restrict__ absmax) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int nb = K >> 6;
  if (wid >= static_cast<int64_t>(N) * nb) return;
  const int n = static_cast<int>(wid / nb);
  const int b = static_cast<int>(wid - static_cast<int64_t>(n) * nb);
  const uint32_t pair = *reinterpret_cast<const uint32_t*>(W + static_cast<int64_t>(n) * ldw + 64 * b + 2 * lane);
  const float w0 = __uint_as_float(pair << 16), w1 = __uint_as_float(pair & 0xFFFF0000u);
  float amax = fmaxf(fabsf(w0), fabsf(w1));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  float v0 = 0.f, v1 = 0.f;
  if (amax != 0.0f) { v0 = w0 / amax; v1 = w1 / amax; }
  const int c0 = nearest_level(v0, cb), c1 = nearest_level(v1, cb);
  qs[static_cast<int64_t>(n) * (K >> 1) + 32 * b + lane] = static_cast<uint8_t>((c0 << 4) | c1);
  if (lane == 0) absmax[static_cast<int64_t>(n) * nb + b] = amax;
}

// ------------------------------------------------------ NF4 -> bf16
// Dequantisation for the dequantise-then-GEMM path (bitsandbytes issue
// #1842, "Benchmark Data": the dequantise + bf16 matrix-product row): one
// thread per code byte, w = absmax * codebook[code] as an fp32 product,
// rounded to bf16 (nearest even); element 2j from the high nibble.
__global__ void __launch_bounds__(kThreads) nf4_dequant_kernel(const uint8_t* __restrict__ qs,
                                                                const float* __restrict__ absmax,
                                                                Codebook16 cb, int N, int K,
                                                                __nv_bfloat16* __restrict__ W,
                                                                int64_t ldw) {
  __shared__ float lv[16];
  if (threadIdx.x < 16) lv[threadIdx.x] = cb.v[threadIdx.x];
  __syncthreads();
  const int kh = K >> 1;
  const int64_t total = static_cast<int64_t>(N) * kh;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; t < total;
       t += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int n = static_cast<int>(t / kh);
    const int j = static_cast<int>(t - static_cast<int64_t>(n) * kh);
    const uint32_t c = qs[t];
    const float a = absmax[static_cast<int64_t>(n) * (K >> 6) + (j >> 5)];
    const __nv_bfloat162 o = __floats2bfloat162_rn(__fmul_rn(a, lv[c >> 4]), __fmul_rn(a, lv[c & 15u]));
    *reinterpret_cast<__nv_bfloat162*>(W + static_cast<int64_t>(n) * ldw + 2 * j) = o;
  }
}

// The same dequantisation for 4-byte aligned code rows and a 16-byte
// aligned W with a pitch of whole 16-byte pieces: CTAs take rows, a thread
// takes 8 codes (4 bytes) per step and writes their 8 bf16 values as one
// 16-byte store (a warp: 128 bytes of codes in, 512 contiguous bytes out).
// The levels sit in shared memory once per lane (level e of lane l at e *
// 32 + l), so a warp's lookups never meet in a bank.
__global__ void __launch_bounds__(kThreads) nf4_dequant_rows_kernel(const uint8_t* __restrict__ qs,
                                                                     const float* __restrict__ absmax,
                                                                     Codebook16 cb, int N, int K,
                                                                     __nv_bfloat16* __restrict__ W,
                                                                     int64_t ldw) {
  __shared__ float lv[16 * 32];
  for (int i = threadIdx.x; i < 16 * 32; i += kThreads) {
    float v = cb.v[0];
#pragma unroll
    for (int e = 1; e < 16; ++e) v = (i >> 5) == e ? cb.v[e] : v;
    lv[i] = v;
  }
  __syncthreads();
  const float* mylv = lv + (threadIdx.x & 31);
  const int units = K >> 3;                  // 4-byte code units per row
  const int nb = K >> 6;
  for (int n = blockIdx.x; n < N; n += gridDim.x) {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(qs + static_cast<int64_t>(n) * (K >> 1));
    const float* arow = absmax + static_cast<int64_t>(n) * nb;
    uint4* wrow = reinterpret_cast<uint4*>(W + static_cast<int64_t>(n) * ldw);
    for (int u = threadIdx.x; u < units; u += kThreads) {
      const uint32_t w = __ldg(qrow + u);
      const float a = __ldg(arow + (u >> 3));
      uint32_t o[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t byte = (w >> (8 * b)) & 0xFFu;
        const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(a, mylv[(byte >> 4) * 32]),
                                                       __fmul_rn(a, mylv[(byte & 15u) * 32]));
        o[b] = *reinterpret_cast<const uint32_t*>(&h);
      }
      wrow[u] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_q8_1(const float* X, int64_t ldx, int M, int K, void* xq,
                                 cudaStream_t st, Launch* info) {
  const int64_t threads = static_cast<int64_t>(M) * (K / 4);
  const int grid = static_cast<int>((threads + kThreads - 1) / kThreads);
  info->grid_x = grid;
  info->block = kThreads;
  info->kernel = "quantize_q8_1";
  return launch_k(q8_1_kernel, dim3(grid), dim3(kThreads), 0, st, true, X, ldx, M, K,
                  static_cast<uint8_t*>(xq));
}

cudaError_t launch_quantize_q4_0(const float* W, int64_t ldw, int N, int K, uint8_t* qs, void* d,
                                 cudaStream_t st, Launch* info) {
  const int64_t warps = static_cast<int64_t>(N) * (K / 32);
  const int64_t grid = (warps * 32 + kThreads - 1) / kThreads;
  info->grid_x = static_cast<int>(grid);
  info->block = kThreads;
  info->kernel = "quantize_q4_0";
  q4_0_quant_kernel<<<static_cast<unsigned>(grid), kThreads, 0, st>>>(W, ldw, N, K, qs,
                                                                       static_cast<__half*>(d));
  return cudaGetLastError();
}

cudaError_t launch_quantize_nf4(const void* W, int64_t ldw, int N, int K, const Codebook16& cb,
                                uint8_t* qs, float* absmax, cudaStream_t st, Launch* info) {
  const int64_t warps = static_cast<int64_t>(N) * (K / 64);
  const int64_t grid = (warps * 32 + kThreads - 1) / kThreads;
  info->grid_x = static_cast<int>(grid);
  info->block = kThreads;
  info->kernel = "quantize_nf4";
  nf4_quant_kernel<<<static_cast<unsigned>(grid), kThreads, 0, st>>>(
      static_cast<const __nv_bfloat16*>(W), ldw, N, K, cb, qs, absmax);
  return cudaGetLastError();
}

cudaError_t launch_dequantize_nf4(const uint8_t* qs, const float* absmax, const Codebook16& cb, int N,
                                  int K, void* W, int64_t ldw, cudaStream_t st, Launch* info) {
  if (reinterpret_cast<uintptr_t>(qs) % 4 == 0 && reinterpret_cast<uintptr_t>(W) % 16 == 0 &&
      ldw % 8 == 0) {
    // rows over the CTAs, eight codes per thread and step
    int64_t grid = device_sm_count() * 8;
    if (grid > N) grid = N;
    info->grid_x = static_cast<int>(grid);
    info->block = kThreads;
    info->kernel = "dequantize_nf4_rows";
    nf4_dequant_rows_kernel<<<static_cast<unsigned>(grid), kThreads, 0, st>>>(
        qs, absmax, cb, N, K, static_cast<__nv_bfloat16*>(W), ldw);
    return cudaGetLastError();
  }
  const int64_t total = static_cast<int64_t>(N) * (K / 2);
  int64_t grid = (total + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(device_sm_count()) * 16;
  if (grid > cap) grid = cap;
  info->grid_x = static_cast<int>(grid);
  info->block = kThreads;
  info->kernel = "dequantize_nf4";
  nf4_dequant_kernel<<<static_cast<unsigned>(grid), kThreads, 0, st>>>(qs, absmax, cb, N, K,
                                                                       static_cast<__nv_bfloat16*>(W), ldw);
  return cudaGetLastError();
}

}  // namespace wobs
