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
#include <cstdlib>
#include <cstring>


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
// Block dots may start from kDotBias - 8 s (s the block's Q8_1 code sum):
// the integer bits of float 1.5 * 2^23 plus the exact dot Sum (q4 - 8) q8,
// whose magnitude stays below 2^22, are the bits of the float 1.5 * 2^23 +
// dot, so one float subtraction yields the dot exactly, with no
// integer-to-float conversion (a quarter-rate unit).
constexpr int kDotBias = 0x4B400000;
constexpr float kDotBiasF = 12582912.0f;

// Sum of q4 * q8 over one block (codes 0..15, no offset), added to s0.
__device__ __forceinline__ int q4_dot_u(uint4 q, int4 lo, int4 hi, int s0 = 0) {
  int s = s0;
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

constexpr int kU = 4;   // 16-byte chunks per lane per pipeline stage

// One pipeline stage: kU blocks of one row (lane-strided) and their scales.
struct Q4Stage {
  uint4 q[kU];
  uint16_t d[kU];
};

__device__ __forceinline__ void q4_load_stage(Q4Stage& st, const uint8_t* __restrict__ qs,
                                              const uint16_t* __restrict__ d4, int row, int it,
                                              int nb, int kh, int lane, uint64_t pol) {
  const uint4* qr = reinterpret_cast<const uint4*>(qs + static_cast<int64_t>(row) * kh);
  const uint16_t* dr = d4 + static_cast<int64_t>(row) * nb;
#pragma unroll
  for (int u = 0; u < kU; ++u) {
    const int b = it * (32 * kU) + 32 * u + lane;
    if (b < nb) {
      st.q[u] = ld_stream16(qr + b, pol);
      st.d[u] = ld_stream_u16(dr + b, pol);
    } else {
      st.q[u] = make_uint4(0u, 0u, 0u, 0u);
      st.d[u] = 0;
    }
  }
}

// Each warp walks the (row, stage) sequence of its rows with two register
// stages: the loads of stage t+1 are in flight while stage t is consumed, so
// a warp always has 2 * kU * 16 bytes per lane outstanding, across row
// boundaries too.  The first stage is issued before pdl_wait(), so it
// overlaps the end of the previous kernel on the stream.
__global__ void __launch_bounds__(kThreads) q4_m1_kernel(const uint8_t* __restrict__ qs,
                                                          const uint16_t* __restrict__ d4,
                                                          const uint8_t* __restrict__ xq,
                                                          float* __restrict__ y, int N, int K,
                                                          ArgmaxArgs am) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int nb = K >> 5;
  const int kh = K >> 1;
  int4* x_lo = reinterpret_cast<int4*>(smem);
  int4* x_hi = x_lo + nb;
  float* x_d = reinterpret_cast<float*>(x_hi + nb);
  int* x_s = reinterpret_cast<int*>(x_d + nb);
  const uint64_t pol = l2_evict_first_policy();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total_warps = gridDim.x * kWarps;
  const int wg = blockIdx.x * kWarps + warp;
  const int n_it = (nb + 32 * kU - 1) / (32 * kU);
  const int rows_w = wg < N ? (N - 1 - wg) / total_warps + 1 : 0;
  const int T = rows_w * n_it;

  Q4Stage sa, sb;
  int lrow = wg, lit = 0;  // next stage to load
  auto advance = [&](int& r, int& it) {
    if (++it == n_it) { it = 0; r += total_warps; }
  };
  if (T > 0) { q4_load_stage(sa, qs, d4, lrow, lit, nb, kh, lane, pol); advance(lrow, lit); }
  pdl_launch_dependents();
  pdl_wait();
  for (int b = threadIdx.x; b < nb; b += kThreads) {
    const XBlock xb = load_xblock(xq + 36 * static_cast<int64_t>(b));
    x_lo[b] = xb.lo;
    x_hi[b] = xb.hi;
    x_d[b] = xb.d;
    x_s[b] = xb.s;
  }
  __syncthreads();

  int crow = wg, cit = 0;
  float acc0 = 0.f, acc1 = 0.f;
  uint64_t best = 0;
  auto consume = [&](const Q4Stage& st) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int b = cit * (32 * kU) + 32 * u + lane;
      if (b < nb) {
        const int dot = q4_dot_u(st.q[u], x_lo[b], x_hi[b]) - 8 * x_s[b];
        const float sc = half_bits_to_float(st.d[u]) * x_d[b];
        if (u & 1) acc1 = fmaf(static_cast<float>(dot), sc, acc1);
        else acc0 = fmaf(static_cast<float>(dot), sc, acc0);
      }
    }
    if (cit == n_it - 1) {
      const float s = warp_sum(acc0 + acc1);
      if (lane == 0) y[crow] = s;
      if (am.out) {
        const uint64_t k = argmax_key(s, static_cast<uint32_t>(crow));
        best = k > best ? k : best;
      }
      acc0 = acc1 = 0.f;
    }
    advance(crow, cit);
  };
  for (int t = 0; t < T; t += 2) {
    if (t + 1 < T) { q4_load_stage(sb, qs, d4, lrow, lit, nb, kh, lane, pol); advance(lrow, lit); }
    consume(sa);
    if (t + 1 < T) {
      if (t + 2 < T) { q4_load_stage(sa, qs, d4, lrow, lit, nb, kh, lane, pol); advance(lrow, lit); }
      consume(sb);
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

// ------------------------------------------- M = 1, cp.async staging

// The warp-per-row computation with the weight stream staged through
// shared memory by asynchronous copies (cp.async, 16 bytes per lane): each
// warp owns a ring of kRing segments of kSegBlocks blocks (2048 bytes of
// nibbles + 256 bytes of scales).  The first segment is requested before
// pdl_wait, so the stream starts while the previous kernel finishes; each
// iteration requests the next segment into the slot consumed last, then
// waits for the current one.  Reads from the ring are lane-contiguous
// 16-byte loads (no bank conflicts).  16 warps per CTA and two CTAs per SM
// for Q8_1 input (the measured optimum on GB300 between bytes in flight and
// warps available to consume them); 32 warps and one CTA per SM when the CTA
// quantises fp32 activations itself.
constexpr int kCpWarps = 16;
constexpr int kCpThreads = kCpWarps * 32;
constexpr int kSegBlocks = 128;
constexpr int kSegQs = kSegBlocks * 16;
constexpr int kSegBytes = kSegQs + kSegBlocks * 2;
constexpr int kRing = 2;
constexpr int kRingBytes = kCpWarps * kRing * kSegBytes;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
               :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// Q8_1 quantisation of one fp32 activation vector straight into the
// shared-memory planes of the M = 1 kernel (every CTA quantises the whole
// vector).  The decisions are the quantiser's (q8_1_part_block: TPB lanes
// per 32-block, amax, d = amax / 127 in IEEE float32, q = roundf(x / d), 0
// when d = 0), d widened back from its fp16 rounding, exact integer code
// sum -- so the planes hold exactly what staging the stored Q8_1 blocks
// would.  Every thread of the CTA (NT of them) calls this with the same
// trip count, so the group shuffles see whole warps.
template <int NT, int TPB>
__device__ __forceinline__ void q8_1_planes_tpb(const float* __restrict__ X, int nb, int4* x_lo,
                                                int4* x_hi, float* x_d, int* x_s,
                                                uint8_t* __restrict__ xq_out) {
  constexpr int kPerPass = NT / TPB;           // blocks per pass
  constexpr int kW = 8 / TPB;                  // code words per lane
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
    // word w of the block's eight code words: words 0..3 in x_lo, 4..7 in x_hi
#pragma unroll
    for (int i = 0; i < kW; ++i) {
      const int w = kW * j + i;
      reinterpret_cast<uint32_t*>(w < 4 ? &x_lo[b] : &x_hi[b])[w & 3] = h.codes[i];
    }
    if (j == 0) {
      x_d[b] = __half2float(__float2half_rn(h.d));
      x_s[b] = kDotBias - 8 * h.sum;
    }
    // each 36-byte Q8_1 block written by one CTA
    if (xq_out != nullptr && b % static_cast<int>(gridDim.x) == static_cast<int>(blockIdx.x))
      store_q8_1_part<TPB>(xq_out + 36 * static_cast<int64_t>(b), h, j);
  }
}

template <int NT>
__device__ __forceinline__ void q8_1_planes_from_f32(const float* __restrict__ X, int nb, int4* x_lo,
                                                     int4* x_hi, float* x_d, int* x_s,
                                                     uint8_t* __restrict__ xq_out) {
  const int tpb = q8_1_lanes_per_block<NT>(nb);
  if (tpb == 8) q8_1_planes_tpb<NT, 8>(X, nb, x_lo, x_hi, x_d, x_s, xq_out);
  else if (tpb == 4) q8_1_planes_tpb<NT, 4>(X, nb, x_lo, x_hi, x_d, x_s, xq_out);
  else q8_1_planes_tpb<NT, 2>(X, nb, x_lo, x_hi, x_d, x_s, xq_out);
}

// kF32X: xsrc is the fp32 activation vector, quantised to Q8_1 in the
// prologue; otherwise it holds the Q8_1 blocks.  W warps per CTA.
template <bool kArgmax, bool kF32X, int W = kCpWarps>
__global__ void __launch_bounds__(W * 32) q4_m1_cp_kernel(const uint8_t* __restrict__ qs,
                                                               const uint16_t* __restrict__ d4,
                                                               const void* __restrict__ xsrc,
                                                               float* __restrict__ y, int N, int K,
                                                               ArgmaxArgs am,
                                                               uint8_t* __restrict__ xq_out) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int nb = K >> 5;
  const int kh = K >> 1;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total_warps = gridDim.x * W;
  // rows spread round-robin over the CTAs first, so every SM gets an
  // equal share even when there are fewer rows than warps
  const int wg = warp * gridDim.x + blockIdx.x;
  const int nseg = (nb + kSegBlocks - 1) / kSegBlocks;
  const int rows_w = wg < N ? (N - 1 - wg) / total_warps + 1 : 0;
  const int T = rows_w * nseg;
  uint8_t* myring = smem + warp * (kRing * kSegBytes);
  int4* x_lo = reinterpret_cast<int4*>(smem + W * kRing * kSegBytes);
  int4* x_hi = x_lo + nb;
  float* x_d = reinterpret_cast<float*>(x_hi + nb);
  int* x_s = reinterpret_cast<int*>(x_d + nb);

  int prow = wg, pseg = 0;   // next segment to request
  auto issue = [&](int slot) {
    uint8_t* st = myring + slot * kSegBytes;
    const int b0 = pseg * kSegBlocks;
    const int n = min(kSegBlocks, nb - b0);
    const uint8_t* qr = qs + static_cast<int64_t>(prow) * kh + b0 * 16;
#pragma unroll
    for (int u = 0; u < kSegBlocks / 32; ++u) {
      const int bl = 32 * u + lane;
      if (bl < n) cp_async16(st + 16 * bl, qr + 16 * bl);
    }
    const uint8_t* dr = reinterpret_cast<const uint8_t*>(d4 + static_cast<int64_t>(prow) * nb + b0);
    if (lane < n / 8) cp_async16(st + kSegQs + 16 * lane, dr + 16 * lane);
    if (++pseg == nseg) { pseg = 0; prow += total_warps; }
  };
  // request the first kRing-1 segments before waiting for the previous kernel
#pragma unroll
  for (int i = 0; i < kRing - 1; ++i) {
    if (i < T) issue(i);
    cp_async_commit();
  }
  pdl_launch_dependents();
  pdl_wait();
  if constexpr (kF32X) {
    q8_1_planes_from_f32<W * 32>(static_cast<const float*>(xsrc), nb, x_lo, x_hi, x_d, x_s, xq_out);
  } else {
    const uint8_t* xq = static_cast<const uint8_t*>(xsrc);
    for (int b = threadIdx.x; b < nb; b += W * 32) {
      const XBlock xb = load_xblock(xq + 36 * static_cast<int64_t>(b));
      x_lo[b] = xb.lo;
      x_hi[b] = xb.hi;
      x_d[b] = xb.d;
      x_s[b] = kDotBias - 8 * xb.s;
    }
  }
  __syncthreads();

  int crow = wg, cseg = 0;
  float acc0 = 0.f, acc1 = 0.f;
  uint64_t best = 0;
  for (int t = 0; t < T; ++t) {
    // request segment t+kRing-1 (into the slot consumed last), then wait for segment t
    if (t + kRing - 1 < T) issue((t + kRing - 1) % kRing);
    cp_async_commit();
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint8_t* st = myring + (t % kRing) * kSegBytes;
    const int b0 = cseg * kSegBlocks;
    const int n = min(kSegBlocks, nb - b0);
#pragma unroll
    for (int u = 0; u < kSegBlocks / 32; ++u) {
      const int bl = 32 * u + lane;
      if (bl < n) {
        const uint4 q = *reinterpret_cast<const uint4*>(st + 16 * bl);
        const uint16_t dh = *reinterpret_cast<const uint16_t*>(st + kSegQs + 2 * bl);
        const int b = b0 + bl;
        const float dot = __int_as_float(q4_dot_u(q, x_lo[b], x_hi[b], x_s[b])) - kDotBiasF;
        const float sc = half_bits_to_float(dh) * x_d[b];
        if (u & 1) acc1 = fmaf(dot, sc, acc1);
        else acc0 = fmaf(dot, sc, acc0);
      }
    }
    if (cseg == nseg - 1) {
      const float sum = warp_sum(acc0 + acc1);
      if (lane == 0) y[crow] = sum;
      if (kArgmax) {
        const uint64_t k = argmax_key(sum, static_cast<uint32_t>(crow));
        best = k > best ? k : best;
      }
      acc0 = acc1 = 0.f;
    }
    if (++cseg == nseg) { cseg = 0; crow += total_warps; }
    __syncwarp();
  }
  cp_async_wait<0>();
  if (kArgmax) {
    __shared__ uint64_t s_best[W];
    __shared__ uint64_t s_cta[1];
    if (lane == 0) s_best[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t bk = 0;
      for (int i = 0; i < W; ++i) bk = s_best[i] > bk ? s_best[i] : bk;
      s_cta[0] = bk;
    }
    __syncthreads();
    argmax_publish(s_cta, 1, am, gridDim.x);
  }
}

template <bool kArgmax, bool kF32X>
cudaError_t run_m1_cp_t(const uint8_t* qs, const void* d, const void* xsrc, float* y, int N, int K,
                        const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const int nb = K / 32;
  const int smem = kRingBytes + nb * 40;
  auto kern = q4_m1_cp_kernel<kArgmax, kF32X>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int grid = 2 * device_sm_count();
  if (grid > N) grid = N;
  info->grid_x = grid;
  info->block = kCpThreads;
  info->smem = smem;
  info->kernel = kF32X ? "q4_0_f32_m1_cp" : "q4_0_q8_1_m1_cp";
  return launch_k(kern, dim3(grid), dim3(kCpThreads), smem, st, true, qs,
                  static_cast<const uint16_t*>(d), xsrc, y, N, K, am,
                  static_cast<uint8_t*>(nullptr));
}

cudaError_t run_m1_cp(const uint8_t* qs, const void* d, const void* xq, float* y, int N, int K,
                      const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  return am.out ? run_m1_cp_t<true, false>(qs, d, xq, y, N, K, am, st, info)
                : run_m1_cp_t<false, false>(qs, d, xq, y, N, K, am, st, info);
}

// The M = 1 cp.async kernel applies: whole 256-element scale segments,
// 16-byte aligned scale plane, ring and planes within 200 KB.
bool m1_cp_shape(const void* d, int K) {
  return (K % 256 == 0) && (reinterpret_cast<uintptr_t>(d) % 16 == 0) &&
         (kRingBytes + (K / 32) * 40 <= 200 * 1024);
}
bool m1_cp_applies(const void* d, int K) { return m1_cp_shape(d, K) && !m1_ldg_forced(); }

// ------------------------------------- 2..8 columns, cp.async staging

// The M = 1 structure (warp per row, lanes along K, per-warp cp.async ring,
// whole rows so no K split) for a few activation columns: each weight block
// is unpacked once and dotted with MC columns.  The activation planes
// ([MC][nb] each) stay in shared memory; columns past M are zero.
template <int MC>
struct McShape {
  static constexpr int kWarps = MC >= 8 ? 12 : 16;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kRingBytes = kWarps * kRing * kSegBytes;
};

template <int MC, bool kArgmax>
__global__ void __launch_bounds__(McShape<MC>::kThreads) q4_mc_cp_kernel(
    const uint8_t* __restrict__ qs, const uint16_t* __restrict__ d4, const uint8_t* __restrict__ xq,
    int M, float* __restrict__ Y, int N, int K, ArgmaxArgs am) {
  constexpr int W = McShape<MC>::kWarps;
  extern __shared__ __align__(16) uint8_t smem[];
  const int nb = K >> 5;
  const int kh = K >> 1;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total_warps = gridDim.x * W;
  const int wg = warp * gridDim.x + blockIdx.x;   // rows round-robin over the CTAs first
  const int nseg = (nb + kSegBlocks - 1) / kSegBlocks;
  const int rows_w = wg < N ? (N - 1 - wg) / total_warps + 1 : 0;
  const int T = rows_w * nseg;
  uint8_t* myring = smem + warp * (kRing * kSegBytes);
  int4* x_lo = reinterpret_cast<int4*>(smem + McShape<MC>::kRingBytes);   // [MC][nb]
  int4* x_hi = x_lo + MC * nb;
  float2* x_ds = reinterpret_cast<float2*>(x_hi + MC * nb);               // (d, exact sum)

  int prow = wg, pseg = 0;
  auto issue = [&](int slot) {
    uint8_t* st = myring + slot * kSegBytes;
    const int b0 = pseg * kSegBlocks;
    const int n = min(kSegBlocks, nb - b0);
    const uint8_t* qr = qs + static_cast<int64_t>(prow) * kh + b0 * 16;
#pragma unroll
    for (int u = 0; u < kSegBlocks / 32; ++u) {
      const int bl = 32 * u + lane;
      if (bl < n) cp_async16(st + 16 * bl, qr + 16 * bl);
    }
    const uint8_t* dr = reinterpret_cast<const uint8_t*>(d4 + static_cast<int64_t>(prow) * nb + b0);
    if (lane < n / 8) cp_async16(st + kSegQs + 16 * lane, dr + 16 * lane);
    if (++pseg == nseg) { pseg = 0; prow += total_warps; }
  };
#pragma unroll
  for (int i = 0; i < kRing - 1; ++i) {
    if (i < T) issue(i);
    cp_async_commit();
  }
  pdl_launch_dependents();
  pdl_wait();
  for (int i = threadIdx.x; i < MC * nb; i += W * 32) {
    const int m = i / nb, b = i - m * nb;
    if (m < M) {
      const XBlock xb = load_xblock(xq + 36 * (static_cast<int64_t>(m) * nb + b));
      x_lo[i] = xb.lo;
      x_hi[i] = xb.hi;
      x_ds[i] = make_float2(xb.d, __int_as_float(kDotBias - 8 * xb.s));
    } else {
      x_lo[i] = make_int4(0, 0, 0, 0);
      x_hi[i] = make_int4(0, 0, 0, 0);
      x_ds[i] = make_float2(0.f, __int_as_float(kDotBias));
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
    if (t + kRing - 1 < T) issue((t + kRing - 1) % kRing);
    cp_async_commit();
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint8_t* st = myring + (t % kRing) * kSegBytes;
    const int b0 = cseg * kSegBlocks;
    const int n = min(kSegBlocks, nb - b0);
#pragma unroll
    for (int u = 0; u < kSegBlocks / 32; ++u) {
      const int bl = 32 * u + lane;
      if (bl < n) {
        const uint4 q = *reinterpret_cast<const uint4*>(st + 16 * bl);
        const float dw = half_bits_to_float(*reinterpret_cast<const uint16_t*>(st + kSegQs + 2 * bl));
        const int b = b0 + bl;
        const int lo0 = static_cast<int>(q.x & 0x0F0F0F0Fu), lo1 = static_cast<int>(q.y & 0x0F0F0F0Fu);
        const int lo2 = static_cast<int>(q.z & 0x0F0F0F0Fu), lo3 = static_cast<int>(q.w & 0x0F0F0F0Fu);
        const int hi0 = static_cast<int>((q.x >> 4) & 0x0F0F0F0Fu), hi1 = static_cast<int>((q.y >> 4) & 0x0F0F0F0Fu);
        const int hi2 = static_cast<int>((q.z >> 4) & 0x0F0F0F0Fu), hi3 = static_cast<int>((q.w >> 4) & 0x0F0F0F0Fu);
#pragma unroll
        for (int m = 0; m < MC; ++m) {
          const int4 xl = x_lo[m * nb + b], xh = x_hi[m * nb + b];
          const float2 ds = x_ds[m * nb + b];
          int sdot = __float_as_int(ds.y);
          sdot = __dp4a(lo0, xl.x, sdot); sdot = __dp4a(lo1, xl.y, sdot);
          sdot = __dp4a(lo2, xl.z, sdot); sdot = __dp4a(lo3, xl.w, sdot);
          sdot = __dp4a(hi0, xh.x, sdot); sdot = __dp4a(hi1, xh.y, sdot);
          sdot = __dp4a(hi2, xh.z, sdot); sdot = __dp4a(hi3, xh.w, sdot);
          acc[m] = fmaf(__int_as_float(sdot) - kDotBiasF, dw * ds.x, acc[m]);
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

// The same stream for 2..4 columns with R = 2 or 4 rows per warp: lane l
// takes row R p + (l mod R) of the warp's row group p and block l / R of
// each group of 32 / R, and a segment is 128 / R blocks of the R rows.  In
// the segment each row keeps its codes and its scales contiguous (so every
// cp.async fills shared memory in global order), row r's planes 128 r / R
// bytes past a bank period so that the R rows' reads of one block fall in
// different banks.  The R lanes of one block sit in the same quarter-warp:
// every read of the activation planes is a broadcast serving R rows.
template <int R>
struct RowGroup {
  static constexpr int kBlocks = 128 / R;                           // blocks per segment
  static constexpr int kCodePitch = kBlocks * 16 + 128 / R;          // row r's codes at r * pitch
  static constexpr int kScale0 = (R - 1) * kCodePitch + kBlocks * 16;
  static constexpr int kScalePitch = ((kBlocks * 2 + 127) / 128) * 128 + 128 / R;
  static constexpr int kSegBytes = kScale0 + (R - 1) * kScalePitch + kBlocks * 2;   // 2432 / 2688
  static_assert(kCodePitch % 16 == 0 && kScale0 % 16 == 0 && kScalePitch % 16 == 0, "16-byte copies");
};

template <int MC, int R, bool kArgmax>
__global__ void __launch_bounds__(McShape<MC>::kThreads) q4_mc2_cp_kernel(
    const uint8_t* __restrict__ qs, const uint16_t* __restrict__ d4, const uint8_t* __restrict__ xq,
    int M, float* __restrict__ Y, int N, int K, ArgmaxArgs am) {
  constexpr int W = McShape<MC>::kWarps;
  extern __shared__ __align__(16) uint8_t smem[];
  const int nb = K >> 5;
  const int kh = K >> 1;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  using G = RowGroup<R>;
  constexpr int SB = G::kBlocks;
  const int h = lane % R, hl = lane / R;
  const int total_warps = gridDim.x * W;
  const int wg = warp * gridDim.x + blockIdx.x;   // row groups round-robin over the CTAs first
  const int ngroups = (N + R - 1) / R;
  const int nseg = (nb + SB - 1) / SB;
  const int groups_w = wg < ngroups ? (ngroups - 1 - wg) / total_warps + 1 : 0;
  const int T = groups_w * nseg;
  uint8_t* myring = smem + warp * (kRing * G::kSegBytes);
  int4* x_lo = reinterpret_cast<int4*>(smem + W * kRing * G::kSegBytes);    // [MC][nb]
  int4* x_hi = x_lo + MC * nb;
  float2* x_ds = reinterpret_cast<float2*>(x_hi + MC * nb);                 // (d, exact sum)

  int pp = wg, pseg = 0;
  auto issue = [&](int slot) {
    uint8_t* st = myring + slot * G::kSegBytes;
    const int b0 = pseg * SB;
    const int n = min(SB, nb - b0);
    const int r0 = R * pp;
    // codes: 16-byte chunk j of 128 is block b0 + (j mod SB) of row r0 + j / SB
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = 32 * u + lane, rr = j / SB, bl = j % SB;
      if (bl < n && r0 + rr < N)
        cp_async16(st + rr * G::kCodePitch + 16 * bl,
                   qs + static_cast<int64_t>(r0 + rr) * kh + (b0 + bl) * 16);
    }
    // scales: 16-byte chunk c (8 blocks) of row r0 + rr
    if (lane < 16) {
      const int rr = lane / (SB / 8), c = lane % (SB / 8);
      if (8 * c < n && r0 + rr < N)
        cp_async16(st + G::kScale0 + rr * G::kScalePitch + 16 * c,
                   reinterpret_cast<const uint8_t*>(d4 + static_cast<int64_t>(r0 + rr) * nb + b0) + 16 * c);
    }
    if (++pseg == nseg) { pseg = 0; pp += total_warps; }
  };
#pragma unroll
  for (int i = 0; i < kRing - 1; ++i) {
    if (i < T) issue(i);
    cp_async_commit();
  }
  pdl_launch_dependents();
  pdl_wait();
  for (int i = threadIdx.x; i < MC * nb; i += W * 32) {
    const int m = i / nb, b = i - m * nb;
    if (m < M) {
      const XBlock xb = load_xblock(xq + 36 * (static_cast<int64_t>(m) * nb + b));
      x_lo[i] = xb.lo;
      x_hi[i] = xb.hi;
      x_ds[i] = make_float2(xb.d, __int_as_float(kDotBias - 8 * xb.s));
    } else {
      x_lo[i] = make_int4(0, 0, 0, 0);
      x_hi[i] = make_int4(0, 0, 0, 0);
      x_ds[i] = make_float2(0.f, __int_as_float(kDotBias));
    }
  }
  __syncthreads();

  int cpair = wg, cseg = 0;
  float acc[MC];
#pragma unroll
  for (int m = 0; m < MC; ++m) acc[m] = 0.f;
  uint64_t best[MC];
#pragma unroll
  for (int m = 0; m < MC; ++m) best[m] = 0ull;
  for (int t = 0; t < T; ++t) {
    if (t + kRing - 1 < T) issue((t + kRing - 1) % kRing);
    cp_async_commit();
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint8_t* st = myring + (t % kRing) * G::kSegBytes;
    const int b0 = cseg * SB;
    const int n = min(SB, nb - b0);
    // a missing second row of the last pair computes on stale bytes and
    // writes nothing
#pragma unroll
    for (int u = 0; u < SB * R / 32; ++u) {
      const int bl = (32 / R) * u + hl;
      if (bl < n) {
        const uint4 q = *reinterpret_cast<const uint4*>(st + h * G::kCodePitch + 16 * bl);
        const float dw = half_bits_to_float(
            *reinterpret_cast<const uint16_t*>(st + G::kScale0 + h * G::kScalePitch + 2 * bl));
        const int b = b0 + bl;
        const int lo0 = static_cast<int>(q.x & 0x0F0F0F0Fu), lo1 = static_cast<int>(q.y & 0x0F0F0F0Fu);
        const int lo2 = static_cast<int>(q.z & 0x0F0F0F0Fu), lo3 = static_cast<int>(q.w & 0x0F0F0F0Fu);
        const int hi0 = static_cast<int>((q.x >> 4) & 0x0F0F0F0Fu), hi1 = static_cast<int>((q.y >> 4) & 0x0F0F0F0Fu);
        const int hi2 = static_cast<int>((q.z >> 4) & 0x0F0F0F0Fu), hi3 = static_cast<int>((q.w >> 4) & 0x0F0F0F0Fu);
#pragma unroll
        for (int m = 0; m < MC; ++m) {
          const int4 xl = x_lo[m * nb + b], xh = x_hi[m * nb + b];
          const float2 ds = x_ds[m * nb + b];
          int sdot = __float_as_int(ds.y);
          sdot = __dp4a(lo0, xl.x, sdot); sdot = __dp4a(lo1, xl.y, sdot);
          sdot = __dp4a(lo2, xl.z, sdot); sdot = __dp4a(lo3, xl.w, sdot);
          sdot = __dp4a(hi0, xh.x, sdot); sdot = __dp4a(hi1, xh.y, sdot);
          sdot = __dp4a(hi2, xh.z, sdot); sdot = __dp4a(hi3, xh.w, sdot);
          acc[m] = fmaf(__int_as_float(sdot) - kDotBiasF, dw * ds.x, acc[m]);
        }
      }
    }
    if (cseg == nseg - 1) {
      const int row = R * cpair + h;
#pragma unroll
      for (int m = 0; m < MC; ++m) {
        float sum = acc[m];
#pragma unroll
        for (int o = 16; o >= R; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);   // lanes of one row
        if (m < M && row < N) {
          if (hl == m) Y[static_cast<int64_t>(m) * N + row] = sum;
          if (kArgmax) {
            const uint64_t k = argmax_key(sum, static_cast<uint32_t>(row));
            best[m] = k > best[m] ? k : best[m];
          }
        }
        acc[m] = 0.f;
      }
    }
    if (++cseg == nseg) { cseg = 0; cpair += total_warps; }
    __syncwarp();
  }
  cp_async_wait<0>();
  if (kArgmax) {
    __shared__ uint64_t s_best[W][MC];
    __shared__ uint64_t s_cta[MC];
#pragma unroll
    for (int m = 0; m < MC; ++m)
#pragma unroll
      for (int o = 1; o < R; o <<= 1) {                               // the other rows of the group
        const uint64_t k = __shfl_xor_sync(0xffffffffu, best[m], o);
        best[m] = k > best[m] ? k : best[m];
      }
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

// Two CTAs of the few-column kernel fit on an SM with this much shared memory each.
constexpr int kMcSmemMax = 110 * 1024;

template <int MC>
int mc_smem(int K) {
  return McShape<MC>::kRingBytes + MC * (K / 32) * 40;
}
template <int MC, int R>
int mc_group_smem(int K) {
  return McShape<MC>::kWarps * kRing * RowGroup<R>::kSegBytes + MC * (K / 32) * 40;
}

template <int MC, bool kArgmax>
cudaError_t run_mc_t(const uint8_t* qs, const void* d, const void* xq, int M, float* y, int N,
                     int K, const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  constexpr int W = McShape<MC>::kWarps;
  // rows per warp (GB300, us per call back to back, 1 / 2 / 4 rows per
  // warp: M = 2 4096^2 4.04 / 3.64 / 4.93, 14336x4096 8.16 / 7.67 / 8.20;
  // M = 4 4096^2 5.45 / 4.74 / 5.13, 14336x4096 12.47 / 10.54 / 9.62): four
  // for 3..4 columns on tall matrices, else two; a group ring that would
  // leave one CTA per SM falls back to fewer rows.  WOBS_Q4MC=1, 2 or 4
  // forces the rows per warp.
  const char* v = std::getenv("WOBS_Q4MC");
  int R = (MC == 4 && N >= 8192) ? 4 : 2;
  if (v && (v[0] == '1' || v[0] == '2' || v[0] == '4')) R = v[0] - '0';
  if (R == 4 && mc_group_smem<MC, 4>(K) > kMcSmemMax) R = 2;
  if (R == 2 && mc_group_smem<MC, 2>(K) > kMcSmemMax) R = 1;
  const int smem = R == 4 ? mc_group_smem<MC, 4>(K) : R == 2 ? mc_group_smem<MC, 2>(K) : mc_smem<MC>(K);
  auto kern = R == 4 ? q4_mc2_cp_kernel<MC, 4, kArgmax>
            : R == 2 ? q4_mc2_cp_kernel<MC, 2, kArgmax> : q4_mc_cp_kernel<MC, kArgmax>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int per_sm = max_resident_ctas(reinterpret_cast<const void*>(kern), W * 32, smem);
  int grid = device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int units = (N + R - 1) / R;   // rows or row groups
  if (grid > units) grid = units;
  info->grid_x = grid;
  info->block = W * 32;
  info->smem = smem;
  info->kernel = "q4_0_q8_1_mc_cp";
  return launch_k(kern, dim3(grid), dim3(W * 32), smem, st, true, qs,
                  static_cast<const uint16_t*>(d), static_cast<const uint8_t*>(xq), M, y, N, K, am);
}

template <int MC>
cudaError_t run_mc(const uint8_t* qs, const void* d, const void* xq, int M, float* y, int N, int K,
                   const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  return am.out ? run_mc_t<MC, true>(qs, d, xq, M, y, N, K, am, st, info)
                : run_mc_t<MC, false>(qs, d, xq, M, y, N, K, am, st, info);
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
  pdl_launch_dependents();
  pdl_wait();
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
            t += take_partial(sk.partials + (static_cast<int64_t>(j) * M + m) * N + row);
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
  return launch_k(q4_mn_kernel<NC>, grid, dim3(kThreads), smem, st, true, qs,
                  static_cast<const uint16_t*>(d), static_cast<const uint8_t*>(xq), M, Y, N, K,
                  bps, s2, am);
}

cudaError_t run_m1(const uint8_t* qs, const void* d, const void* xq, float* y, int N, int K,
                   const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const int nb = K / 32;
  const int smem = nb * 40;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(q4_m1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  const int per_sm = max_resident_ctas(reinterpret_cast<const void*>(q4_m1_kernel), kThreads, smem);
  int grid = device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int need = (N + kWarps - 1) / kWarps;
  if (grid > need) grid = need;
  info->grid_x = grid;
  info->block = kThreads;
  info->smem = smem;
  info->kernel = "q4_0_q8_1_m1";
  return launch_k(q4_m1_kernel, dim3(grid), dim3(kThreads), smem, st, true, qs,
                  static_cast<const uint16_t*>(d), static_cast<const uint8_t*>(xq), y, N, K, am);
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

bool q4_mc_applies(int M, int K) {
  if (M < 2 || M > 4 || K % 256 != 0) return false;
  const int smem = M == 2 ? mc_smem<2>(K) : mc_smem<4>(K);
  return smem <= kMcSmemMax;
}

cudaError_t launch_gemv_q4_0_q8_1(const uint8_t* qs, const void* d, const void* xq, int M,
                                  float* Y, int N, int K, const SplitArgs& sk,
                                  const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  if (M == 1 && sk.splits <= 1) {
    // 16-byte asynchronous copies need 16-byte aligned scale segments
    if (m1_cp_applies(d, K)) return run_m1_cp(qs, d, xq, Y, N, K, am, st, info);
    return run_m1(qs, d, xq, Y, N, K, am, st, info);
  }
  const bool cp_shape = K % 256 == 0 && reinterpret_cast<uintptr_t>(d) % 16 == 0;
  // a few columns: whole rows per warp, no K split
  if (cp_shape && sk.splits <= 1 && q4_mc_applies(M, K)) {
    if (M == 2) return run_mc<2>(qs, d, xq, M, Y, N, K, am, st, info);
    return run_mc<4>(qs, d, xq, M, Y, N, K, am, st, info);
  }
  // tensor-core path: whole 8-block stages and 16-byte scale copies
  if (M >= 2 && cp_shape)
    return launch_q4_mma(qs, d, xq, M, Y, N, K, forced_splits(), sk, am, st, info);
  if (M <= 1) return run_mn<1>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 2) return run_mn<2>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 4) return run_mn<4>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 8) return run_mn<8>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 12) return run_mn<12>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 16) return run_mn<16>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  if (M <= 24) return run_mn<24>(qs, d, xq, M, Y, N, K, sk, am, st, info);
  return run_mn<32>(qs, d, xq, M, Y, N, K, sk, am, st, info);
}

bool q4_0_f32_fused_applies(const void* d, int M, int K) { return M == 1 && m1_cp_shape(d, K); }

// CTA-local quantisation: W warps per CTA, 2 CTAs per SM for W = 16, one
// for W = 32 (each SM then quantises x once).
template <bool kArgmax, int W>
cudaError_t run_m1_local_t(const uint8_t* qs, const void* d, const float* x, uint8_t* xq_out,
                           float* y, int N, int K, const ArgmaxArgs& am, cudaStream_t st,
                           Launch* info) {
  const int smem = W * kRing * kSegBytes + (K / 32) * 40;
  auto kern = q4_m1_cp_kernel<kArgmax, true, W>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int grid = (W >= 32 ? 1 : 2) * device_sm_count();
  if (grid > N) grid = N;
  info->grid_x = grid;
  info->block = W * 32;
  info->smem = smem;
  info->kernel = "q4_0_f32_m1_cp";
  return launch_k(kern, dim3(grid), dim3(W * 32), smem, st, true, qs,
                  static_cast<const uint16_t*>(d), static_cast<const void*>(x), y, N, K, am,
                  xq_out);
}

// 32 warps and one CTA per SM (each SM quantises x once) for long vectors
// or few rows; 16 warps and two CTAs per SM for K <= 4096 with at least
// 4096 rows, where the prologue is short and a CTA that finishes early
// hands its SM half to the next kernel sooner (GB300, per call back to
// back: 4096^2 3.83 against 3.96 us, 14336x4096 6.90 against 7.30 us;
// 1024x4096 and 4096x14336 are faster with 32 warps).  WOBS_Q4F32=16 or 32
// forces one of them.
template <bool kArgmax>
cudaError_t run_m1_fused(const uint8_t* qs, const void* d, const float* x, uint8_t* xq_out, float* y,
                         int N, int K, const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const char* v = std::getenv("WOBS_Q4F32");
  const bool fits32 = 32 * kRing * kSegBytes + (K / 32) * 40 <= 220 * 1024;
  bool use32 = fits32 && !(K <= 4096 && N >= 4096);
  if (v && std::strcmp(v, "16") == 0) use32 = false;
  if (v && std::strcmp(v, "32") == 0 && fits32) use32 = true;
  if (use32) return run_m1_local_t<kArgmax, 32>(qs, d, x, xq_out, y, N, K, am, st, info);
  return run_m1_local_t<kArgmax, 16>(qs, d, x, xq_out, y, N, K, am, st, info);
}

cudaError_t launch_gemv_q4_0_f32_fused(const uint8_t* qs, const void* d, const float* x,
                                       void* xq_out, float* y, int N, int K, const ArgmaxArgs& am,
                                       cudaStream_t st, Launch* info) {
  uint8_t* xo = static_cast<uint8_t*>(xq_out);
  return am.out ? run_m1_fused<true>(qs, d, x, xo, y, N, K, am, st, info)
                : run_m1_fused<false>(qs, d, x, xo, y, N, K, am, st, info);
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
