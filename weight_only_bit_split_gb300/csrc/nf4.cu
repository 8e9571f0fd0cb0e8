// NF4 blockwise 4-bit decode GEMV, M = 1.
//
// bitsandbytes issue #1842 ("70B 4-bit LLM decode bottlenecked by HIP kernel
// (kgemm_4bit_inference_naive) efficiency"): the fused 4-bit inference GEMV
// for one decode token, 64-element blocks with a float absmax each, codes
// looked up in a 16-entry float codebook, float accumulation.  The issue and
// its comments locate the losses in narrow loads, bf16 <-> float conversions
// in the inner loop, and too little latency hiding; a later comment asks for
// consecutive threads reading consecutive 128-bit chunks.
//
// sm_103a design:
//   * a warp owns a 1024-element K slice (32 lanes x 32 codes = one 16-byte
//     load per lane per row, 512 contiguous bytes per warp instruction);
//   * the CTA processes rows in batches of 32: each lane keeps its 32
//     activation values in registers (converted to float once) and one
//     partial sum per row of the batch, so activations are never re-read
//     per row;
//   * codes are decoded two at a time through a 256-entry byte -> (level,
//     level) float table in shared memory, replicated 16 times so the 16
//     lanes of a half-warp never share a bank; the pair goes straight into
//     a packed two-wide fp32 FMA;
//   * at the end of a batch a 31-shuffle reduce-scatter leaves row r's warp
//     partial in lane r; warps combine through shared memory in a fixed
//     order, so the result does not depend on timing.
#include <cstdlib>
#include <cstring>

#include "common.cuh"

namespace wobs {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBatch = 32;        // rows per batch (one per lane after the reduction)
constexpr int kRowUnroll = 8;     // rows whose codes are in flight at once
constexpr int kLutCopies = 16;

__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n"
      " mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p, uint64_t pol) {
  uint32_t r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(r) : "l"(p), "l"(pol));
  return r;
}

template <bool kArgmax>
__global__ void __launch_bounds__(kThreads, 2) nf4_m1_kernel(const uint8_t* __restrict__ qs,
                                                              const float* __restrict__ absmax,
                                                              Codebook16 cb,
                                                              const __nv_bfloat16* __restrict__ x,
                                                              __nv_bfloat16* __restrict__ y,
                                                              int N, int K, ArgmaxArgs am) {
  extern __shared__ __align__(16) float smem_f[];
  float2* lut = reinterpret_cast<float2*>(smem_f);                 // [256][16]
  float* xsm = smem_f + 2 * 256 * kLutCopies;                        // permuted x, K floats
  __shared__ float red[kWarps][kBatch];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nsl = (K + 1023) >> 10;        // 1024-element slices
  const int kh = K >> 1;                   // code bytes per row
  const int nab = K >> 6;                  // absmax per row
  const uint64_t pol = l2_evict_first_policy();

  for (int i = threadIdx.x; i < 256 * kLutCopies; i += kThreads) {
    const int e = i / kLutCopies;
    lut[i] = make_float2(cb.v[e >> 4], cb.v[e & 15]);
  }
  pdl_launch_dependents();
  pdl_wait();
  // x element k = sl*1024 + l*32 + 4*j + t  ->  xsm[((sl*8 + j)*32 + l)*4 + t]
  for (int k = threadIdx.x; k < nsl * 1024; k += kThreads) {
    const int sl = k >> 10, l = (k >> 5) & 31, j = (k >> 2) & 7, t = k & 3;
    xsm[((sl * 8 + j) * 32 + l) * 4 + t] = k < K ? __bfloat162float(x[k]) : 0.f;
  }
  __syncthreads();

  const float2* lut_l = lut + (lane & (kLutCopies - 1));
  const int nbatch = (N + kBatch - 1) / kBatch;
  uint64_t best = 0;
  float2 xr[16];
  int loaded_slice = -1;
  for (int bt = blockIdx.x; bt < nbatch; bt += gridDim.x) {
    const int row0 = bt * kBatch;
    float p[kBatch];
#pragma unroll
    for (int r = 0; r < kBatch; ++r) p[r] = 0.f;
    for (int sl = warp; sl < nsl; sl += kWarps) {
      if (sl != loaded_slice) {
        const float4* xp = reinterpret_cast<const float4*>(xsm) + (sl * 8) * 32 + lane;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float4 v = xp[j * 32];
          xr[2 * j] = make_float2(v.x, v.y);
          xr[2 * j + 1] = make_float2(v.z, v.w);
        }
        loaded_slice = sl;
      }
      const int chunk = sl * 32 + lane;              // 16-byte chunk index within a row
      const bool lane_ok = chunk * 32 < K;
#pragma unroll
      for (int r0 = 0; r0 < kBatch; r0 += kRowUnroll) {
        uint4 q[kRowUnroll];
        float a[kRowUnroll];
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
          const int row = row0 + r0 + u;
          if (lane_ok && row < N) {
            q[u] = ld_stream16(qs + static_cast<int64_t>(row) * kh + chunk * 16, pol);
            a[u] = __uint_as_float(ld_stream_u32(absmax + static_cast<int64_t>(row) * nab + (chunk >> 1), pol));
          } else {
            q[u] = make_uint4(0u, 0u, 0u, 0u);
            a[u] = 0.f;
          }
        }
#pragma unroll
        for (int u = 0; u < kRowUnroll; ++u) {
          float2 acc = make_float2(0.f, 0.f);
          const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t e = (w[i] >> (8 * j)) & 0xFFu;
              acc = ffma2(lut_l[e * kLutCopies], xr[4 * i + j], acc);
            }
          }
          p[r0 + u] = fmaf(a[u], acc.x + acc.y, p[r0 + u]);
        }
      }
    }
    // reduce-scatter: lane r ends with the warp's sum for row r
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < off; ++i) {
        const float send = upper ? p[i] : p[i + off];
        const float keep = upper ? p[i + off] : p[i];
        p[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    red[warp][lane] = p[0];
    __syncthreads();
    if (warp == 0) {
      float t = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kWarps; ++w2) t += red[w2][lane];
      const int row = row0 + lane;
      if (row < N) {
        const __nv_bfloat16 o = __float2bfloat16_rn(t);
        y[row] = o;
        if (kArgmax) {
          const uint64_t k = argmax_key(__bfloat162float(o), static_cast<uint32_t>(row));
          best = k > best ? k : best;
        }
      }
    }
    __syncthreads();
  }
  if (kArgmax) {
    __shared__ uint64_t s_cta[1];
    if (warp == 0) {
      best = warp_max_u64(best);
      if (lane == 0) s_cta[0] = best;
    }
    __syncthreads();
    argmax_publish(s_cta, 1, am, gridDim.x);
  }
}

// ----------------------------------------------- cp.async staged variant
//
// Same decomposition (a warp owns a 1024-element K slice and keeps its 32
// activations per lane in registers; rows in batches of 32), with the code
// and scale stream staged through a per-warp ring of shared-memory stages
// by 16-byte asynchronous copies, requested one stage ahead and, for the
// first stage, before the programmatic-launch wait.  A stage holds 8 rows of
// the warp's slice: 8 x 512 bytes of codes and 8 x 64 bytes of block scales.
// When K has fewer than 8 slices, the CTA runs 8 / slices batches side by
// side (one group of warps each, synchronised by its own named barrier).
constexpr int kCpRows = 8;                      // rows per stage
constexpr int kCpStage = kCpRows * 512 + kCpRows * 64;
constexpr int kCpRing = 2;

__device__ __forceinline__ void group_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void cp_async16_nf4(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src),
                  "r"(valid ? 16 : 0) : "memory");
}

template <bool kArgmax>
__global__ void __launch_bounds__(kThreads, 2) nf4_m1_cp_kernel(const uint8_t* __restrict__ qs,
                                                                const float* __restrict__ absmax,
                                                                Codebook16 cb,
                                                                const __nv_bfloat16* __restrict__ x,
                                                                __nv_bfloat16* __restrict__ y,
                                                                int N, int K, ArgmaxArgs am) {
  extern __shared__ __align__(16) float smem_f[];
  float2* lut = reinterpret_cast<float2*>(smem_f);                                   // [256][16]
  uint8_t* rings = reinterpret_cast<uint8_t*>(smem_f + 2 * 256 * kLutCopies);         // [warps][ring][stage]
  __shared__ float red[kWarps][kBatch];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nsl = K >> 10;                 // 1, 2, 4 or 8 slices
  const int groups = kWarps / nsl;         // batches processed side by side
  const int grp = warp / nsl, sl = warp - grp * nsl;
  const int kh = K >> 1;
  const int nab = K >> 6;
  const int nbatch = (N + kBatch - 1) / kBatch;
  const int bstride = gridDim.x * groups;
  const int bfirst = blockIdx.x * groups + grp;
  const int my_batches = bfirst < nbatch ? (nbatch - 1 - bfirst) / bstride + 1 : 0;
  constexpr int kOct = kBatch / kCpRows;   // stages per batch
  const int T = my_batches * kOct;
  uint8_t* ring = rings + warp * (kCpRing * kCpStage);

  int pb = bfirst, po = 0;                 // next stage: batch, row octet
  auto issue = [&](int slot) {
    uint8_t* st = ring + slot * kCpStage;
    const int row0 = pb * kBatch + po * kCpRows;
#pragma unroll
    for (int r = 0; r < kCpRows; ++r) {
      const int row = min(row0 + r, N - 1);
      cp_async16_nf4(st + r * 512 + 16 * lane, qs + static_cast<int64_t>(row) * kh + sl * 512 + 16 * lane, true);
    }
    {
      const int r = lane >> 2, q = lane & 3;
      const int row = min(row0 + r, N - 1);
      cp_async16_nf4(st + kCpRows * 512 + r * 64 + 16 * q,
                     absmax + static_cast<int64_t>(row) * nab + sl * 16 + 4 * q, true);
    }
    if (++po == kOct) { po = 0; pb += bstride; }
  };
  if (T > 0) issue(0);
  asm volatile("cp.async.commit_group;" ::: "memory");

  for (int i = threadIdx.x; i < 256 * kLutCopies; i += kThreads) {
    const int e = i / kLutCopies;
    lut[i] = make_float2(cb.v[e >> 4], cb.v[e & 15]);
  }
  pdl_launch_dependents();
  pdl_wait();
  // this lane's 32 activations: element sl*1024 + lane*32 + 4*j + t -> xr[2j], xr[2j+1]
  float2 xr[16];
  {
    const uint4* xp = reinterpret_cast<const uint4*>(x + sl * 1024 + lane * 32);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint4 v = __ldg(xp + h);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) xr[4 * h + i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    }
  }
  __syncthreads();                         // the codebook table is complete

  // this lane's replica of the table; entry e starts e * 128 bytes further
  const uint32_t lut_b = static_cast<uint32_t>(__cvta_generic_to_shared(lut)) +
                         static_cast<uint32_t>(lane & (kLutCopies - 1)) * 8u;
  uint64_t best = 0;
  int cbt = bfirst;                        // batch being consumed
  for (int t = 0; t < T; t += kOct, cbt += bstride) {
    float p[kBatch];
#pragma unroll
    for (int r = 0; r < kBatch; ++r) p[r] = 0.f;
#pragma unroll
    for (int o = 0; o < kOct; ++o) {
      if (t + o + 1 < T) issue((t + o + 1) % kCpRing);
      asm volatile("cp.async.commit_group;" ::: "memory");
      asm volatile("cp.async.wait_group 1;" ::: "memory");
      __syncwarp();
      const uint8_t* st = ring + (o % kCpRing) * kCpStage;   // t is a multiple of kOct (even)
#pragma unroll
      for (int r = 0; r < kCpRows; ++r) {
        const uint4 q = *reinterpret_cast<const uint4*>(st + r * 512 + 16 * lane);
        const float a = *reinterpret_cast<const float*>(st + kCpRows * 512 + r * 64 + 4 * (lane >> 1));
        float2 acc = make_float2(0.f, 0.f);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            // byte j of the word -> table entry (byte * 16 + replica) * 8
            const uint32_t e = __byte_perm(w[i], 0u, 0x4440u | static_cast<uint32_t>(j));
            float2 v;
            asm("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(e * 128u + lut_b));
            acc = ffma2(v, xr[4 * i + j], acc);
          }
        }
        p[o * kCpRows + r] = a * (acc.x + acc.y);
      }
      __syncwarp();
    }
    // batch complete: reduce-scatter, then combine the group's slices
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const bool upper = (lane & off) != 0;
#pragma unroll
      for (int i = 0; i < off; ++i) {
        const float send = upper ? p[i] : p[i + off];
        const float keep = upper ? p[i + off] : p[i];
        p[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    red[warp][lane] = p[0];
    group_barrier(1 + grp, nsl * 32);
    if (sl == 0) {
      float tot = 0.f;
      for (int w2 = 0; w2 < nsl; ++w2) tot += red[grp * nsl + w2][lane];
      const int row = cbt * kBatch + lane;
      if (row < N) {
        const __nv_bfloat16 o = __float2bfloat16_rn(tot);
        y[row] = o;
        if (kArgmax) {
          const uint64_t k = argmax_key(__bfloat162float(o), static_cast<uint32_t>(row));
          best = k > best ? k : best;
        }
      }
    }
    group_barrier(1 + grp, nsl * 32);
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  if (kArgmax) {
    __shared__ uint64_t s_g[kWarps];
    __shared__ uint64_t s_cta[1];
    if (sl == 0) {
      const uint64_t b = warp_max_u64(best);
      if (lane == 0) s_g[grp] = b;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t bk = 0;
      for (int i = 0; i < groups; ++i) bk = s_g[i] > bk ? s_g[i] : bk;
      s_cta[0] = bk;
    }
    __syncthreads();
    argmax_publish(s_cta, 1, am, gridDim.x);
  }
}

template <bool kArgmax>
cudaError_t run_cp(const uint8_t* qs, const float* absmax, const Codebook16& cb, const void* x,
                   void* y, int N, int K, const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const int smem = 2 * 256 * kLutCopies * static_cast<int>(sizeof(float)) + kWarps * kCpRing * kCpStage;
  cudaError_t e = cudaFuncSetAttribute(nf4_m1_cp_kernel<kArgmax>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int per_sm = max_resident_ctas(reinterpret_cast<const void*>(nf4_m1_cp_kernel<kArgmax>),
                                       kThreads, smem);
  const int groups = kWarps / (K / 1024);
  int grid = device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int need = ((N + kBatch - 1) / kBatch + groups - 1) / groups;
  if (grid > need) grid = need;
  info->grid_x = grid;
  info->block = kThreads;
  info->smem = smem;
  info->kernel = "nf4_m1_cp";
  return launch_k(nf4_m1_cp_kernel<kArgmax>, dim3(grid), dim3(kThreads), smem, st, true, qs, absmax,
                  cb, static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), N, K,
                  am);
}

template <bool kArgmax>
cudaError_t run(const uint8_t* qs, const float* absmax, const Codebook16& cb, const void* x,
                void* y, int N, int K, const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const int nsl = (K + 1023) / 1024;
  const int smem = (2 * 256 * kLutCopies + nsl * 1024) * static_cast<int>(sizeof(float));
  cudaError_t e = cudaFuncSetAttribute(nf4_m1_kernel<kArgmax>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int per_sm = max_resident_ctas(reinterpret_cast<const void*>(nf4_m1_kernel<kArgmax>),
                                       kThreads, smem);
  int grid = device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int need = (N + kBatch - 1) / kBatch;
  if (grid > need) grid = need;
  info->grid_x = grid;
  info->block = kThreads;
  info->smem = smem;
  info->kernel = "nf4_m1";
  return launch_k(nf4_m1_kernel<kArgmax>, dim3(grid), dim3(kThreads), smem, st, true, qs, absmax,
                  cb, static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), N, K,
                  am);
}

// ------------------------------------------------- 2..32 columns, CUDA cores

// The fallback for several activation columns where the tensor-memory kernel
// does not apply (K not a multiple of 256, unaligned planes or activations):
// one thread per weight row, K in chunks of 256 whose activations (all
// columns, fp32) sit in shared memory; per 64-block the code sums
// sum_i codebook[c_i] * x_i of every column, then times the block's absmax,
// as the format defines the product.
constexpr int kMnChunk = 256;

template <int MC, bool kArgmax>
__global__ void __launch_bounds__(kThreads) nf4_mn_kernel(const uint8_t* __restrict__ qs,
                                                           const float* __restrict__ absmax,
                                                           Codebook16 cb,
                                                           const __nv_bfloat16* __restrict__ X,
                                                           int64_t ldx, int M,
                                                           __nv_bfloat16* __restrict__ Y, int N,
                                                           int K, ArgmaxArgs am) {
  __shared__ float xs[MC][kMnChunk];
  __shared__ float lv[16];
  const int row = blockIdx.x * kThreads + threadIdx.x;
  const bool valid = row < N;
  const int nb = K >> 6;
  if (threadIdx.x < 16) lv[threadIdx.x] = cb.v[threadIdx.x];
  pdl_launch_dependents();
  pdl_wait();
  float acc[MC];
#pragma unroll
  for (int m = 0; m < MC; ++m) acc[m] = 0.f;
  const uint8_t* qrow = qs + static_cast<int64_t>(valid ? row : 0) * (K >> 1);
  const float* arow = absmax + static_cast<int64_t>(valid ? row : 0) * nb;
  for (int k0 = 0; k0 < K; k0 += kMnChunk) {
    const int kc = min(kMnChunk, K - k0);
    __syncthreads();
    for (int i = threadIdx.x; i < MC * kMnChunk; i += kThreads) {
      const int m = i / kMnChunk, k = i - m * kMnChunk;
      xs[m][k] = (m < M && k < kc) ? __bfloat162float(X[m * ldx + k0 + k]) : 0.f;
    }
    __syncthreads();
    if (valid) {
      for (int b = 0; b < (kc >> 6); ++b) {
        const int gb = (k0 >> 6) + b;
        const float a = __ldg(arow + gb);
        float inner[MC];
#pragma unroll
        for (int m = 0; m < MC; ++m) inner[m] = 0.f;
        for (int by = 0; by < 32; ++by) {
          const uint32_t c = __ldg(qrow + 32 * gb + by);
          const float w0 = lv[c >> 4], w1 = lv[c & 15u];   // elements 2 by, 2 by + 1
          const int k = 64 * b + 2 * by;
#pragma unroll
          for (int m = 0; m < MC; ++m) inner[m] = fmaf(w1, xs[m][k + 1], fmaf(w0, xs[m][k], inner[m]));
        }
#pragma unroll
        for (int m = 0; m < MC; ++m) acc[m] = fmaf(a, inner[m], acc[m]);
      }
    }
  }
  __shared__ uint64_t s_key[kWarps][MC];
  __shared__ uint64_t s_cta[MC];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int m = 0; m < MC; ++m) {
    const __nv_bfloat16 o = __float2bfloat16_rn(acc[m]);
    if (valid && m < M) Y[static_cast<int64_t>(m) * N + row] = o;
    if (kArgmax) {
      uint64_t k = (valid && m < M) ? argmax_key(__bfloat162float(o), static_cast<uint32_t>(row)) : 0ull;
      k = warp_max_u64(k);
      if (lane == 0) s_key[warp][m] = k;
    }
  }
  if (kArgmax) {
    __syncthreads();
    if (threadIdx.x < MC) {
      uint64_t bk = 0;
      for (int w = 0; w < kWarps; ++w) bk = s_key[w][threadIdx.x] > bk ? s_key[w][threadIdx.x] : bk;
      s_cta[threadIdx.x] = bk;
    }
    __syncthreads();
    argmax_publish(s_cta, M, am, gridDim.x);
  }
}

template <int MC>
cudaError_t run_mn(const uint8_t* qs, const float* absmax, const Codebook16& cb, const void* X,
                   int64_t ldx, int M, void* Y, int N, int K, const ArgmaxArgs& am, cudaStream_t st,
                   Launch* info) {
  const int grid = (N + kThreads - 1) / kThreads;
  info->grid_x = grid;
  info->block = kThreads;
  info->kernel = "nf4_mn";
  if (am.out)
    return launch_k(nf4_mn_kernel<MC, true>, dim3(grid), dim3(kThreads), 0, st, true, qs, absmax, cb,
                    static_cast<const __nv_bfloat16*>(X), ldx, M, static_cast<__nv_bfloat16*>(Y), N, K, am);
  return launch_k(nf4_mn_kernel<MC, false>, dim3(grid), dim3(kThreads), 0, st, true, qs, absmax, cb,
                  static_cast<const __nv_bfloat16*>(X), ldx, M, static_cast<__nv_bfloat16*>(Y), N, K, am);
}

}  // namespace

// Several activation columns: the tensor-memory kernel where it applies,
// otherwise the CUDA-core kernel above (which takes no K split).
cudaError_t launch_gemv_nf4_mc(const uint8_t* qs, const float* absmax, const Codebook16& cb,
                               const void* X, int64_t ldx, int M, void* Y, int N, int K,
                               const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                               Launch* info) {
  // up to four columns: the one-column tensor-core kernel serves them all
  // (its B operand has eight columns; the decode is shared), unless
  // WOBS_NF4_MC=tc asks for the tensor-memory kernel
  const char* mcv = std::getenv("WOBS_NF4_MC");
  const bool tc_forced = mcv && std::strcmp(mcv, "tc") == 0;
  if (M <= 4 && !nf4_cp_forced() && !tc_forced && !m1_ldg_forced()) {
    cudaError_t e = launch_nf4_mma(qs, absmax, cb, X, ldx, M, Y, N, K, am, st, info);
    if (e != cudaErrorNotSupported) return e;
    cudaGetLastError();
  }
  if (!nf4_cp_forced()) {
    cudaError_t e = launch_nf4_tc(qs, absmax, cb, X, ldx, M, Y, N, K, sk, am, st, info);
    if (e != cudaErrorNotSupported) return e;
    cudaGetLastError();
  }
  if (M <= 2) return run_mn<2>(qs, absmax, cb, X, ldx, M, Y, N, K, am, st, info);
  if (M <= 4) return run_mn<4>(qs, absmax, cb, X, ldx, M, Y, N, K, am, st, info);
  if (M <= 8) return run_mn<8>(qs, absmax, cb, X, ldx, M, Y, N, K, am, st, info);
  if (M <= 16) return run_mn<16>(qs, absmax, cb, X, ldx, M, Y, N, K, am, st, info);
  return run_mn<32>(qs, absmax, cb, X, ldx, M, Y, N, K, am, st, info);
}


cudaError_t launch_gemv_nf4(const uint8_t* qs, const float* absmax, const Codebook16& cb,
                            const void* x, void* y, int N, int K, const ArgmaxArgs& am,
                            cudaStream_t st, Launch* info) {
  // tensor-core variant first (K of 1, 2, 4 or 8 thousand, an f16-exact
  // scaled codebook, 16-byte aligned planes); WOBS_NF4=cp selects the
  // CUDA-core staged variant instead
  if (!m1_ldg_forced() && !nf4_cp_forced()) {
    cudaError_t e = launch_nf4_mma(qs, absmax, cb, x, K, 1, y, N, K, am, st, info);
    if (e != cudaErrorNotSupported) return e;
    cudaGetLastError();
  }
  // staged variant: K of 1, 2, 4 or 8 whole 1024-element slices, 16-byte
  // aligned scale rows and activations
  const bool cp = (K == 1024 || K == 2048 || K == 4096 || K == 8192) &&
                  reinterpret_cast<uintptr_t>(absmax) % 16 == 0 &&
                  reinterpret_cast<uintptr_t>(x) % 16 == 0 && !m1_ldg_forced();
  if (cp) return am.out ? run_cp<true>(qs, absmax, cb, x, y, N, K, am, st, info)
                        : run_cp<false>(qs, absmax, cb, x, y, N, K, am, st, info);
  if (am.out) return run<true>(qs, absmax, cb, x, y, N, K, am, st, info);
  return run<false>(qs, absmax, cb, x, y, N, K, am, st, info);
}

}  // namespace wobs
