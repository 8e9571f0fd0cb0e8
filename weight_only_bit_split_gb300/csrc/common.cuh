// Device helpers shared by the GEMV kernels (sm_103a).
//
// Streaming loads with cache hints, warp reductions, the greedy-argmax key,
// and the "last arriving CTA finishes the job" epilogue used for split-K and
// for the fused argmax.  No spin-waits anywhere: cross-CTA completion is an
// arrival counter, never a barrier.
#pragma once

#include <cstdint>
#include <cstdlib>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <utility>

#include "internal.h"

namespace wobs {

// ------------------------------------------- programmatic dependent launch
//
// Decode-path kernels are launched with programmatic stream serialisation:
// a kernel may start while the previous kernel on the stream is finishing.
// Before pdl_wait() a kernel only reads its weight planes (never written by
// a decode-path kernel); activations, outputs and the workspace are touched
// only after pdl_wait(), which returns once the previous kernel has
// completed and its writes are visible.  Kernels that write weights (the
// Q4_0 / NF4 quantisers) never call pdl_launch_dependents, so a GEMV right
// after them starts only when they are done.

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

inline bool pdl_enabled() {
  const char* v = std::getenv("WOBS_PDL");
  return !(v && v[0] == '0');
}

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = (pdl && pdl_enabled()) ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// ---------------------------------------------------------------- loads

// L2 policy for bytes that are read exactly once (weights): evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 16-byte read-only load that does not allocate in L1 and is marked
// evict-first in L2: the weight stream.
__device__ __forceinline__ uint4 ld_stream16(const void* p, uint64_t pol) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "l"(pol));
  return r;
}

// 32-byte (256-bit) form of ld_stream16; the address must be 32-byte aligned.
__device__ __forceinline__ void ld_stream32(const void* p, uint64_t pol, uint4& a, uint4& b) {
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
      : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
      : "l"(p), "l"(pol));
}

// 16-byte read-only load through L1 (activations, re-read by many warps).
__device__ __forceinline__ uint4 ld_nc16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// --------------------------------------------------------- conversions

__device__ __forceinline__ float2 to_float2(uint32_t v, const __half*) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
__device__ __forceinline__ float2 to_float2(uint32_t v, const __nv_bfloat16*) {
  // bf16 is the upper half of a float32: widening is a shift / mask
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}
__device__ __forceinline__ float to_float(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_float(float v) { return v; }

template <typename TO> __device__ __forceinline__ TO from_float(float v);
template <> __device__ __forceinline__ float from_float<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_float<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_float<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// 8 packed 16-bit values (one 16-byte chunk) dotted with 8 floats.
template <typename T>
__device__ __forceinline__ float dot8(uint4 w, const float* x, float acc) {
  const T* tag = nullptr;
  float2 a = to_float2(w.x, tag), b = to_float2(w.y, tag);
  float2 c = to_float2(w.z, tag), d = to_float2(w.w, tag);
  acc = fmaf(a.x, x[0], acc); acc = fmaf(a.y, x[1], acc);
  acc = fmaf(b.x, x[2], acc); acc = fmaf(b.y, x[3], acc);
  acc = fmaf(c.x, x[4], acc); acc = fmaf(c.y, x[5], acc);
  acc = fmaf(d.x, x[6], acc); acc = fmaf(d.y, x[7], acc);
  return acc;
}

// Two 16-byte chunks of 16-bit values, element-wise products summed.
template <typename T>
__device__ __forceinline__ float dot8x8(uint4 w, uint4 x, float acc) {
  const T* tag = nullptr;
  float2 w0 = to_float2(w.x, tag), x0 = to_float2(x.x, tag);
  float2 w1 = to_float2(w.y, tag), x1 = to_float2(x.y, tag);
  float2 w2 = to_float2(w.z, tag), x2 = to_float2(x.z, tag);
  float2 w3 = to_float2(w.w, tag), x3 = to_float2(x.w, tag);
  acc = fmaf(w0.x, x0.x, acc); acc = fmaf(w0.y, x0.y, acc);
  acc = fmaf(w1.x, x1.x, acc); acc = fmaf(w1.y, x1.y, acc);
  acc = fmaf(w2.x, x2.x, acc); acc = fmaf(w2.y, x2.y, acc);
  acc = fmaf(w3.x, x3.x, acc); acc = fmaf(w3.y, x3.y, acc);
  return acc;
}

// ---------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    uint64_t t = __shfl_xor_sync(0xffffffffu, v, o);
    v = t > v ? t : v;
  }
  return v;
}

// ------------------------------------------------ Q8_1 codes in a prologue

// The IEEE float32 quotient, kept out of line: it is the rare fallback of
// q8_1_codes and must not be evaluated (predicated) on the fast path.
static __device__ __noinline__ float ieee_div(float x, float d) { return x / d; }

// q = roundf(x / d) for four elements of one block, as the Q8_1 format
// defines it (IEEE float32 quotient, then round half away from zero),
// without a full division for almost every element.  For 2^-126 <= d <
// 2^126, __fdividef(x, d) is within 2 ulp of the exact quotient (CUDA's
// documented bound) and the IEEE quotient is within 0.5 ulp of it; with
// |x / d| <= 127 (x is in the block whose maximum defines d) one ulp is at
// most 2^-17, so both lie within 2^-14 of each other.  roundf changes value
// only at the half-integers k + 1/2, so when the approximation is farther
// than 2^-14 from the nearest one, both quotients round to the same
// integer; otherwise (and for d outside the bound's range) the IEEE
// division decides.
__device__ __forceinline__ float q8_1_quotient(float x, float d, bool d_ok) {
  const float t = __fdividef(x, d);
  const float h = floorf(t) + 0.5f;
  return (d_ok && fabsf(t - h) > 0x1p-14f) ? t : __int_as_float(0x7fc00000);   // NaN: decide exactly
}
__device__ __forceinline__ void q8_1_codes(const float4& v, float d, int& q0, int& q1, int& q2,
                                           int& q3) {
  const bool d_ok = d >= 0x1p-126f && d < 0x1p126f;
  float t0 = q8_1_quotient(v.x, d, d_ok), t1 = q8_1_quotient(v.y, d, d_ok);
  float t2 = q8_1_quotient(v.z, d, d_ok), t3 = q8_1_quotient(v.w, d, d_ok);
  if (__builtin_expect(isnan(t0) || isnan(t1) || isnan(t2) || isnan(t3), 0)) {
    if (isnan(t0)) t0 = ieee_div(v.x, d);
    if (isnan(t1)) t1 = ieee_div(v.y, d);
    if (isnan(t2)) t2 = ieee_div(v.z, d);
    if (isnan(t3)) t3 = ieee_div(v.w, d);
  }
  q0 = static_cast<int>(roundf(t0));
  q1 = static_cast<int>(roundf(t1));
  q2 = static_cast<int>(roundf(t2));
  q3 = static_cast<int>(roundf(t3));
}

// ------------------------------------------------------- argmax key

// Greedy-argmax key: the float maps to an unsigned integer with the same
// order (-0.0 folded onto +0.0), in the high word; the low word holds
// 0xFFFFFFFF - index, so the maximum key is the largest value and, among
// equal values, the lowest index.  Every finite float maps above 0, so a
// zeroed key is the identity of the max.
__device__ __forceinline__ uint64_t argmax_key(float v, uint32_t idx) {
  uint32_t b = __float_as_uint(v);
  if (b == 0x80000000u) b = 0u;
  uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - idx);
}
__device__ __forceinline__ int64_t argmax_key_index(uint64_t key) {
  return static_cast<int64_t>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFu));
}

// ------------------------------------------------ cross-CTA epilogues

// Publish this CTA's per-column best keys (one per column, held in `cta_key`
// in shared memory) and count the CTA as finished; the CTA that arrives
// last writes the argmax indices and returns the keys and its counter to
// zero, so the workspace is clean for the next call.  Must be called by all
// threads of the CTA.  `expected` = number of CTAs that call it.
__device__ __forceinline__ void argmax_publish(const uint64_t* cta_key, int ncols,
                                               const ArgmaxArgs& am, unsigned expected) {
  __shared__ int s_last;
  if (threadIdx.x < 32) {
    if (static_cast<int>(threadIdx.x) < ncols) {
      atomicMax(reinterpret_cast<unsigned long long*>(am.keys + threadIdx.x),
                static_cast<unsigned long long>(cta_key[threadIdx.x]));
    }
    __threadfence();
    __syncwarp();
    if (threadIdx.x == 0) {
      unsigned prev = atomicAdd(am.counter, 1u);
      s_last = (prev == expected - 1u);
    }
  }
  __syncthreads();
  if (s_last) {
    __threadfence();
    if (static_cast<int>(threadIdx.x) < ncols) {
      uint64_t k = atomicExch(reinterpret_cast<unsigned long long*>(am.keys + threadIdx.x), 0ull);
      am.out[threadIdx.x] = argmax_key_index(k);
    }
    if (threadIdx.x == 0) *am.counter = 0u;
  }
}

// Split-K arrival for one row group: returns true (in every thread) for
// the CTA that arrives last among the `splits` CTAs of `group`; that CTA
// resets the counter.  Call after the partial stores, from all threads.
// Reads a split-K partial and leaves zero behind (the CUDA-core fallback
// does so; partials lie past the counter region, so other kernels leave
// them in place).
__device__ __forceinline__ float take_partial(float* p) {
  const float v = __ldcg(p);
  __stcg(p, 0.f);
  return v;
}

__device__ __forceinline__ bool splitk_arrive_last(unsigned* counters, int group, int splits) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned prev = atomicAdd(counters + group, 1u);
    s_last = (prev == static_cast<unsigned>(splits) - 1u);
    if (s_last) counters[group] = 0u;
  }
  __syncthreads();
  if (s_last) __threadfence();
  return s_last != 0;
}

}  // namespace wobs
