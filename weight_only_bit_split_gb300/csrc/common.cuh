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

// TPB lanes per 32-element block (TPB = 2, 4 or 8 consecutive lanes; lane j
// of the group holds elements 32/TPB * j ... 32/TPB * (j + 1) - 1), for the
// quantising prologues.  The decisions are the Q8_1 format's: amax over the
// block, d = amax / 127 as an IEEE float32 division, q = roundf(x / d) with
// the IEEE quotient (0 when d = 0).  The quotient is formed as t = x * r
// with r the hardware's approximate reciprocal of d (PTX rcp.approx: at most
// 1 ulp from 1/d), so |t - x/d| <= |x/d| * (2^-23 + 2^-24) < 2^-15.4 for
// |x/d| <= 127, while the IEEE quotient lies within half an ulp (<= 2^-18)
// of x/d: the two are within 2^-15 of each other.  roundf changes value only
// at the half-integers, so whenever t is farther than 2^-13 from every
// half-integer, roundf(IEEE quotient) equals the nearest integer to t, which
// is read off with the 1.5 * 2^23 addition (exact for |t| < 2^22: the sum's
// low mantissa bits are the integer, its low byte the two's-complement
// code).  Otherwise, and for d outside [2^-126, 2^126), the lane takes the
// IEEE division for its elements.  No conversion-unit instruction
// (float-to-int, rounding, division) is spent per element on the fast path.
__device__ __forceinline__ float rcp_approx_ftz(float d) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
  return r;
}

// Low bytes of four words, in order, as one word.
__device__ __forceinline__ uint32_t pack_low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040), __byte_perm(c, d, 0x0040), 0x5410);
}

template <int TPB>
struct Q81Part {
  static constexpr int kWords = 8 / TPB;   // code words (4 codes each) per lane
  uint32_t codes[kWords];                  // this lane's codes in element order
  float d;                                 // the block's scale (float32, before fp16 rounding)
  int sum;                                 // exact sum of all 32 codes of the block
};

// All 32 lanes of the warp must call this (the group exchange is a
// shuffle); lanes whose block does not exist pass zeros and discard the
// result.
template <int TPB>
__device__ __forceinline__ Q81Part<TPB> q8_1_part_block(const float4 (&v)[8 / TPB]) {
  constexpr int kW = 8 / TPB;
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kW; ++i)
    amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w))));
#pragma unroll
  for (int o = 1; o < TPB; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  Q81Part<TPB> h;
  h.d = amax / 127.0f;
  const float d = h.d;
  const bool d_ok = d >= 0x1p-126f && d < 0x1p126f;
  const float r = d_ok ? rcp_approx_ftz(d) : 0.0f;
  constexpr float kRound = 12582912.0f;        // 1.5 * 2^23
  float x[4 * kW];
#pragma unroll
  for (int i = 0; i < kW; ++i) {
    x[4 * i] = v[i].x; x[4 * i + 1] = v[i].y; x[4 * i + 2] = v[i].z; x[4 * i + 3] = v[i].w;
  }
  uint32_t bits[4 * kW];
  bool ok = d_ok || d == 0.0f;                 // d == 0: r = 0, every code 0
#pragma unroll
  for (int i = 0; i < 4 * kW; ++i) {
    const float t = __fmul_rn(x[i], r);
    const float tm = __fadd_rn(t, kRound);
    const float e = __fsub_rn(t, __fsub_rn(tm, kRound));
    ok = ok && fabsf(e) < 0.5f - 0x1p-13f;
    bits[i] = __float_as_uint(tm);
  }
  if (__builtin_expect(!ok, 0)) {
#pragma unroll
    for (int i = 0; i < 4 * kW; ++i)
      bits[i] = static_cast<uint32_t>(d != 0.0f ? static_cast<int>(roundf(x[i] / d)) : 0);
  }
  int s = 0;
#pragma unroll
  for (int i = 0; i < kW; ++i) {
    h.codes[i] = pack_low_bytes(bits[4 * i], bits[4 * i + 1], bits[4 * i + 2], bits[4 * i + 3]);
    s = __dp4a(static_cast<int>(h.codes[i]), 0x01010101, s);
  }
#pragma unroll
  for (int o = 1; o < TPB; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  h.sum = s;
  return h;
}

// The lane group's share of the 36-byte Q8_1 block {fp16 d, fp16 d * sum,
// int8 q[32]} (4-byte aligned stores); `j` is the lane's index in its group.
template <int TPB>
__device__ __forceinline__ void store_q8_1_part(uint8_t* blk, const Q81Part<TPB>& h, int j) {
  constexpr int kW = 8 / TPB;
  uint32_t* w = reinterpret_cast<uint32_t*>(blk + 4) + kW * j;
#pragma unroll
  for (int i = 0; i < kW; ++i) w[i] = h.codes[i];
  if (j == 0)
    *reinterpret_cast<__half2*>(blk) =
        __halves2half2(__float2half_rn(h.d), __float2half_rn(h.d * static_cast<float>(h.sum)));
}

// Lanes per block for a prologue of NT threads over nb blocks: eight (the
// shortest chain per lane) when that covers the vector in one pass, else
// four.  Measured in the fused Q4_0 step on GB300 at K = 14336 with 1024
// threads: four lanes in two passes 0.4 us faster than two lanes in one.
template <int NT>
__host__ __device__ constexpr int q8_1_lanes_per_block(int nb) {
  return nb * 8 <= NT ? 8 : 4;
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
