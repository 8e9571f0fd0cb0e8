// Q4_0 weights x Q8_1 activations for 2..32 columns on the tensor cores,
// with every block dot still an exact integer.
//
// "The kernel that waited for itself" (m12-db-gemm case study), sections
// "The VALU floor" and "A step at sixteen columns": once several activation
// columns share each unpacked weight block, the integer dot products and
// the per-block scaling, not the weight stream, set the time, and the
// CUDA-core kernel falls off the bandwidth roof as the column count grows.
// Here the block dots run on mma.sync (m16n8k16, f16 operands, f32
// accumulate), arranged so that the f32 result of each block is the exact
// integer sum_i (q4_i - 8) q8_i:
//
//   * a 4-bit code q becomes the f16 value 1024 + q by OR-ing it into the
//     mantissa of 1024.0 (low nibbles), or 1024 + 16 q (high nibbles, used
//     in place, without a shift);
//   * activation codes are exact f16 integers, divided by 16 for the high
//     half of the block (exact: a power-of-two scale of a 7-bit integer), so
//     every product (1024 + q) x or (1024 + 16 q) x / 16 is an integer;
//   * the accumulator of each block starts at -1032 s_lo - 72 s_hi, where
//     s_lo, s_hi are the exact sums of the block's low and high 16
//     activation codes, which removes both the 1024 / 64 bias and the
//     "- 8" offset of Q4_0;
//   * all partial sums stay below 2^23 in magnitude, so the f32 tensor-core
//     accumulation is exact and the block result equals the integer dot.
// Only the block scaling d4 * d8 * sumi is floating point, as in the
// format's definition.
//
// Layout.  A warp owns 16 weight rows (one m16 tile) at a time and streams
// them through a private ring of kRing shared-memory stages by 16-byte
// asynchronous copies; a stage holds 8 blocks of the 16 rows (128 bytes of
// codes and 16 bytes of scales per row; the 144-byte row pitch makes the
// per-lane 32-bit fragment reads bank-conflict free).  The CTA converts the
// activation blocks of its K range once, after the programmatic-launch
// wait, into f16 B fragments in shared memory (16 bytes per lane, read with
// one conflict-free 128-bit load per n8 tile) plus, per column, the
// accumulator start value and the activation scale.  The grid is row
// groups x K splits; a row tile whose K range is split adds the partials
// of all splits in a fixed order in the warp that arrives last.
#include "common.cuh"
#include "tma.cuh"

namespace wobs {
namespace {

constexpr int kQSB = 8;                 // blocks per stage
constexpr int kQPitch = 144;            // bytes per row in a stage (128 codes + 16 scales)
constexpr int kQStage = 16 * kQPitch;   // 2304 bytes
constexpr int kQKB = 32;                // most blocks in one CTA's K range
constexpr int kQXBytes = 576;           // shared bytes per block per n8 tile (512 B fragments + 64 B scales)

__device__ __forceinline__ float half_lo(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t f16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ float2 f32x2_mul(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 f32x2_fma(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ void mma_f16(float& c0, float& c1, float& c2, float& c3, uint32_t a0,
                                        uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c0), "+f"(c1), "+f"(c2), "+f"(c3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A.B + {s0, s1, s0, s1}: the accumulator starts from two values (one
// per output column of the lane) without copying them into four registers.
__device__ __forceinline__ void mma_f16_init(float& d0, float& d1, float& d2, float& d3, uint32_t a0,
                                             uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                             uint32_t b1, float s0, float s1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%10,%11};"
      : "=f"(d0), "=f"(d1), "=f"(d2), "=f"(d3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(s0), "f"(s1));
}

// Warp-level split-K arrival: true in the warp that brings the count to
// `splits` (it resets the counter, and then sees every split's partials).
__device__ __forceinline__ bool splitk_arrive_last_warp(unsigned* counters, int group, int splits) {
  __threadfence();
  __syncwarp();
  unsigned last = 0;
  if ((threadIdx.x & 31) == 0) {
    const unsigned prev = atomicAdd(counters + group, 1u);
    last = prev == static_cast<unsigned>(splits) - 1u;
    if (last) counters[group] = 0u;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) __threadfence();
  return last != 0;
}

// Rows one warp owns at a time: R m16 tiles share every activation fragment
// read from shared memory.
// With 9 or more columns a warp owns 32 rows, and the CTA runs 16 warps
// with 2-stage rings (more warps to hide the tensor-core and shared-memory
// latencies, the same bytes in flight); below that, 8 warps with 3-stage
// rings and two CTAs per SM.
template <int NT>
struct Q4Shape {
  static constexpr int R = NT >= 2 ? 2 : 1;
  static constexpr int kRows = 16 * R;
  static constexpr int kStage = kRows * kQPitch;
  static constexpr int kW = NT >= 2 ? 16 : 8;
  static constexpr int kThreads = kW * 32;
  static constexpr int kRing = NT >= 2 ? 2 : 3;
};

template <int NT, bool kArgmax>
__global__ void __launch_bounds__(Q4Shape<NT>::kThreads, NT == 1 ? 2 : 1) q4_mma_kernel(const uint8_t* __restrict__ qs,
                                                               const uint16_t* __restrict__ d4,
                                                               const uint8_t* __restrict__ xq, int M,
                                                               float* __restrict__ Y, int N, int K,
                                                               int kpb, int gpc, SplitArgs sk,
                                                               ArgmaxArgs am) {
  constexpr int R = Q4Shape<NT>::R;
  constexpr int RW = Q4Shape<NT>::kRows;
  constexpr int STG = Q4Shape<NT>::kStage;
  constexpr int kQW = Q4Shape<NT>::kW;
  constexpr int kQThreads = Q4Shape<NT>::kThreads;
  constexpr int kQRing = Q4Shape<NT>::kRing;
  extern __shared__ __align__(16) uint8_t smem[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int nb = K >> 5, kh = K >> 1;
  const int s = blockIdx.y;
  const int kb0 = s * kpb;
  const int nbl = min(nb, kb0 + kpb) - kb0;   // a positive multiple of kQSB
  const int nst = nbl / kQSB;
  const int ngr = (N + RW - 1) / RW;          // row groups of RW rows
  const int gr0 = blockIdx.x * gpc, gr1 = min(ngr, gr0 + gpc);
  const int my_groups = gr0 + warp < gr1 ? (gr1 - 1 - gr0 - warp) / kQW + 1 : 0;
  const int T = my_groups * nst;
  uint8_t* bfrag = smem;                          // [kpb][NT][8 cols][4 lanes][16 B]
  uint8_t* cdbuf = smem + kpb * NT * 512;         // [kpb][NT][4 lanes][C0, C1, d0, d1]
  uint8_t* ring = smem + kpb * NT * kQXBytes + warp * (kQRing * STG);

  // L2 prefetch of one row group's whole K range: long runs per row keep the
  // DRAM access pattern close to a streaming read while the shared-memory
  // stages stay small
  auto prefetch_group = [&](int grp) {
    if (lane < RW) {
      const int row = min(grp * RW + lane, N - 1);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                   :: "l"(qs + static_cast<int64_t>(row) * kh + 16 * kb0), "r"(nbl * 16) : "memory");
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                   :: "l"(d4 + static_cast<int64_t>(row) * nb + kb0), "r"(nbl * 2) : "memory");
    }
  };
  int pgr = gr0 + warp, pst = 0;                  // next stage to request
  auto issue = [&](int slot) {
    if (pst == 0 && pgr + kQW < gr1) prefetch_group(pgr + kQW);
    uint8_t* st = ring + slot * STG;
    const int b0 = kb0 + pst * kQSB;
    const int rbase = pgr * RW;
#pragma unroll
    for (int u = 0; u < 4 * R; ++u) {
      const int c = lane + 32 * u;                // RW rows x 8 chunks
      const int r = c >> 3, cb = c & 7;
      const int row = min(rbase + r, N - 1);
      cp_async16_zfill(st + r * kQPitch + 16 * cb, qs + static_cast<int64_t>(row) * kh + 16 * (b0 + cb), true);
    }
#pragma unroll
    for (int u = 0; u < (RW + 31) / 32; ++u) {
      const int r = lane + 32 * u;
      if (r < RW) {
        const int row = min(rbase + r, N - 1);
        cp_async16_zfill(st + r * kQPitch + 128, d4 + static_cast<int64_t>(row) * nb + b0, true);
      }
    }
    if (++pst == nst) { pst = 0; pgr += kQW; }
  };
#pragma unroll
  for (int i = 0; i < kQRing - 1; ++i) {
    if (i < T) issue(i);
    cp_async_commit_group();
  }
  pdl_launch_dependents();
  pdl_wait();

  // activation blocks of [kb0, kb0 + nbl) -> f16 fragments, start values and
  // scales; every thread's loads are issued before any is used
  {
    constexpr int kPer = (kQKB * NT * 8 + kQThreads - 1) / kQThreads;
    uint32_t w[kPer][9];
#pragma unroll
    for (int it = 0; it < kPer; ++it) {
      const int p = tid + it * kQThreads;
      const int blk = p / (NT * 8), col = p - blk * (NT * 8);
      const bool ok = blk < nbl && col < M;
      const uint32_t* src = reinterpret_cast<const uint32_t*>(
          xq + (static_cast<int64_t>(ok ? col : 0) * nb + kb0 + (ok ? blk : 0)) * 36);
#pragma unroll
      for (int i = 0; i < 9; ++i) w[it][i] = ok ? __ldg(src + i) : 0u;
    }
#pragma unroll
    for (int it = 0; it < kPer; ++it) {
      const int p = tid + it * kQThreads;
      const int blk = p / (NT * 8), col = p - blk * (NT * 8);
      if (blk < nbl) {
        int slo = 0, shi = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          slo = __dp4a(static_cast<int>(w[it][1 + i]), 0x01010101, slo);
          shi = __dp4a(static_cast<int>(w[it][5 + i]), 0x01010101, shi);
        }
        const int n = col >> 3, gg = col & 7;
        uint4* dst = reinterpret_cast<uint4*>(bfrag + ((blk * NT + n) * 8 + gg) * 64);
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          // code byte c -> f16 (1024 + (c + 128)); minus 1152 gives c, times
          // 1/16 minus 72 gives c / 16
          const uint32_t lo = w[it][1 + tt] ^ 0x80808080u, hi = w[it][5 + tt] ^ 0x80808080u;
          uint4 v;
          v.x = f16x2_sub(__byte_perm(lo, 0x64646464u, 0x4240), 0x64806480u);
          v.y = f16x2_sub(__byte_perm(lo, 0x64646464u, 0x4341), 0x64806480u);
          v.z = f16x2_fma(__byte_perm(hi, 0x64646464u, 0x4240), 0x2C002C00u, 0xD480D480u);
          v.w = f16x2_fma(__byte_perm(hi, 0x64646464u, 0x4341), 0x2C002C00u, 0xD480D480u);
          dst[tt] = v;
        }
        float* cd = reinterpret_cast<float*>(cdbuf + ((blk * NT + n) * 4 + (gg >> 1)) * 16);
        cd[gg & 1] = static_cast<float>(-1032 * slo - 72 * shi);
        cd[2 + (gg & 1)] = half_lo(w[it][0]);
      }
    }
  }
  __syncthreads();

  float acc[R][NT][4];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[r][n][0] = acc[r][n][1] = acc[r][n][2] = acc[r][n][3] = 0.f;
  uint64_t best[NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n) best[n][0] = best[n][1] = 0ull;

  // final values of a group: store, fold into the argmax candidates
  auto emit = [&](int grp, float (&v)[R][NT][4]) {
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int col = n * 8 + 2 * t + (h & 1), row = grp * RW + r * 16 + g + 8 * (h >> 1);
          if (col < M && row < N) {
            Y[static_cast<int64_t>(col) * N + row] = v[r][n][h];
            if (kArgmax) {
              const uint64_t k = argmax_key(v[r][n][h], static_cast<uint32_t>(row));
              best[n][h & 1] = k > best[n][h & 1] ? k : best[n][h & 1];
            }
          }
        }
  };

  int cgr = gr0 + warp, cst = 0;
  for (int i = 0; i < T; ++i) {
    if (i + kQRing - 1 < T) issue((i + kQRing - 1) % kQRing);
    cp_async_commit_group();
    cp_async_wait_group<kQRing - 1>();
    __syncwarp();
    const uint8_t* st = ring + (i % kQRing) * STG;
    uint4 sc[R][2];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      sc[r][0] = *reinterpret_cast<const uint4*>(st + (r * 16 + g) * kQPitch + 128);
      sc[r][1] = *reinterpret_cast<const uint4*>(st + (r * 16 + g + 8) * kQPitch + 128);
    }
    const int blk0 = cst * kQSB;
#pragma unroll
    for (int j = 0; j < kQSB; ++j) {
      const int blk = blk0 + j;
      uint4 xv[NT];
      float4 cd[NT];
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        xv[n] = *reinterpret_cast<const uint4*>(bfrag + ((blk * NT + n) * 8 + g) * 64 + 16 * t);
        cd[n] = *reinterpret_cast<const float4*>(cdbuf + ((blk * NT + n) * 4 + t) * 16);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint8_t* rowa = st + (r * 16 + g) * kQPitch + 16 * j + 4 * t;
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(rowa);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(rowa + 8 * kQPitch);
        const uint32_t sa = wa >> 8, sb = wb >> 8;
        const uint32_t a0 = (wa & 0x000F000Fu) | 0x64006400u, a1 = (wb & 0x000F000Fu) | 0x64006400u;
        const uint32_t a2 = (sa & 0x000F000Fu) | 0x64006400u, a3 = (sb & 0x000F000Fu) | 0x64006400u;
        const uint32_t h0 = (wa & 0x00F000F0u) | 0x64006400u, h1 = (wb & 0x00F000F0u) | 0x64006400u;
        const uint32_t h2 = (sa & 0x00F000F0u) | 0x64006400u, h3 = (sb & 0x00F000F0u) | 0x64006400u;
        const uint32_t swa = (j < 4 ? (j < 2 ? sc[r][0].x : sc[r][0].y) : (j < 6 ? sc[r][0].z : sc[r][0].w));
        const uint32_t swb = (j < 4 ? (j < 2 ? sc[r][1].x : sc[r][1].y) : (j < 6 ? sc[r][1].z : sc[r][1].w));
        const float dga = (j & 1) ? half_hi(swa) : half_lo(swa);
        const float dgb = (j & 1) ? half_hi(swb) : half_lo(swb);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          float c0, c1, c2, c3;
          mma_f16_init(c0, c1, c2, c3, a0, a1, a2, a3, xv[n].x, xv[n].y, cd[n].x, cd[n].y);
          mma_f16(c0, c1, c2, c3, h0, h1, h2, h3, xv[n].z, xv[n].w);
          const float2 d8 = make_float2(cd[n].z, cd[n].w);
          const float2 sa2 = f32x2_mul(make_float2(dga, dga), d8);
          const float2 sb2 = f32x2_mul(make_float2(dgb, dgb), d8);
          const float2 ra = f32x2_fma(make_float2(c0, c1), sa2, make_float2(acc[r][n][0], acc[r][n][1]));
          const float2 rb = f32x2_fma(make_float2(c2, c3), sb2, make_float2(acc[r][n][2], acc[r][n][3]));
          acc[r][n][0] = ra.x; acc[r][n][1] = ra.y; acc[r][n][2] = rb.x; acc[r][n][3] = rb.y;
        }
      }
    }
    __syncwarp();
    if (++cst == nst) {
      // row group cgr is complete for this K range
      if (sk.splits > 1) {
        // fragment order: one coalesced 512-byte store per (r, n)
        float4* pp = reinterpret_cast<float4*>(sk.partials) +
                     (static_cast<int64_t>(s) * ngr + cgr) * (R * NT * 32) + lane;
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int n = 0; n < NT; ++n)
            __stcg(pp + (r * NT + n) * 32,
                   make_float4(acc[r][n][0], acc[r][n][1], acc[r][n][2], acc[r][n][3]));
      } else {
        emit(cgr, acc);
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[r][n][0] = acc[r][n][1] = acc[r][n][2] = acc[r][n][3] = 0.f;
      cst = 0;
      cgr += kQW;
    }
  }
  cp_async_wait_group<0>();

  if (sk.splits > 1 && my_groups > 0) {
    // Arrivals after all of this warp's partials (no fence inside the
    // streaming loop): every lane arrives for one of the warp's groups at
    // once, then the warp adds up the groups it completed, all splits of a
    // group loaded together where registers allow, in split order.
    __threadfence();
    __syncwarp();
    for (int base = 0; base < my_groups; base += 32) {
      const int gi = base + lane;
      bool last = false;
      if (gi < my_groups) {
        const int grp = gr0 + warp + gi * kQW;
        const unsigned prev = atomicAdd(sk.counters + grp, 1u);
        last = prev == static_cast<unsigned>(sk.splits) - 1u;
        if (last) sk.counters[grp] = 0u;
      }
      unsigned mask = __ballot_sync(0xffffffffu, last);
      if (mask) __threadfence();
      while (mask) {
        const int gi2 = base + __ffs(mask) - 1;
        mask &= mask - 1;
        const int grp = gr0 + warp + gi2 * kQW;
        constexpr int kB = (16 / (R * NT)) > 0 ? 16 / (R * NT) : 1;
        for (int sp0 = 0; sp0 < sk.splits; sp0 += kB) {
          float4 v[kB][R][NT];
#pragma unroll
          for (int b = 0; b < kB; ++b) {
            const int sp = sp0 + b;
            const float4* pp = reinterpret_cast<const float4*>(sk.partials) +
                               (static_cast<int64_t>(sp < sk.splits ? sp : 0) * ngr + grp) * (R * NT * 32) + lane;
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
              for (int n = 0; n < NT; ++n)
                v[b][r][n] = sp < sk.splits ? __ldcg(pp + (r * NT + n) * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int b = 0; b < kB; ++b)
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
              for (int n = 0; n < NT; ++n) {
                acc[r][n][0] += v[b][r][n].x; acc[r][n][1] += v[b][r][n].y;
                acc[r][n][2] += v[b][r][n].z; acc[r][n][3] += v[b][r][n].w;
              }
        }
        // the partials are scratch (past the counter region): not cleared
        emit(grp, acc);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int n = 0; n < NT; ++n) acc[r][n][0] = acc[r][n][1] = acc[r][n][2] = acc[r][n][3] = 0.f;
      }
    }
  }

  if (kArgmax) {
    __shared__ uint64_t s_key[kQW][32];
    __shared__ uint64_t s_cta[32];
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint64_t k = best[n][hb];
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          const uint64_t other = __shfl_xor_sync(0xffffffffu, k, o);
          k = other > k ? other : k;
        }
        if (g == 0) s_key[warp][n * 8 + 2 * t + hb] = k;
      }
    __syncthreads();
    if (tid < 32) {
      uint64_t k = 0;
      if (tid < NT * 8)
        for (int w2 = 0; w2 < kQW; ++w2) k = s_key[w2][tid] > k ? s_key[w2][tid] : k;
      s_cta[tid] = k;
    }
    __syncthreads();
    argmax_publish(s_cta, M, am, gridDim.x * gridDim.y);
  }
}

// Launch plan shared by the workspace sizing and the launcher: n8 tiles,
// blocks per K range and the number of K ranges.  K ranges of up to 32
// blocks keep the converted activations in shared memory; shorter ranges
// are used when the row groups alone would leave the GPU short of
// independent warp streams.
struct Q4Plan {
  int nt, kpb, splits;
};
Q4Plan q4_plan(int M, int N, int K, int forced) {
  Q4Plan p;
  p.nt = M <= 8 ? 1 : (M <= 16 ? 2 : (M <= 24 ? 3 : 4));
  const int rows = p.nt >= 2 ? 32 : 16;
  const int nb = K / 32;
  const int ngr = (N + rows - 1) / rows;
  if (forced > 0) {
    int s = forced;
    const int smin = (nb + kQKB - 1) / kQKB;
    if (s < smin) s = smin;
    int kpb = (nb + s - 1) / s;
    kpb = (kpb + kQSB - 1) / kQSB * kQSB;
    p.kpb = kpb;
    p.splits = (nb + kpb - 1) / kpb;
    return p;
  }
  // (row group, K range) units to aim for: 4 per SM, 8 per SM for up to 8
  // columns (two CTAs of 8 warps per SM; GB300, 8 columns on 4096^2: 8 K
  // ranges 6.63 us against 4 ranges 7.13; 14336 x 4096 keeps 4 ranges,
  // 13.5 us against 14.9 with 8)
  const int want = (p.nt == 1 ? 8 : 4) * device_sm_count();
  for (int kpb = kQKB; kpb >= kQSB; kpb /= 2) {
    p.kpb = kpb;
    p.splits = (nb + kpb - 1) / kpb;
    if (static_cast<int64_t>(ngr) * p.splits >= want) break;
  }
  return p;
}

template <int NT, bool kArgmax>
cudaError_t run_t(const uint8_t* qs, const void* d, const void* xq, int M, float* Y, int N, int K,
                  const Q4Plan& plan, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                  Launch* info) {
  const int kpb = plan.kpb, splits = plan.splits;
  if (splits > 1 && splits > sk.splits) return cudaErrorInvalidValue;   // workspace too small
  constexpr int kQW = Q4Shape<NT>::kW, kQThreads = Q4Shape<NT>::kThreads;
  const int smem = kpb * NT * kQXBytes + kQW * Q4Shape<NT>::kRing * Q4Shape<NT>::kStage;
  auto kern = q4_mma_kernel<NT, kArgmax>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int per_sm = max_resident_ctas(reinterpret_cast<const void*>(kern), kQThreads, smem);
  const int slots = device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int ngr = (N + Q4Shape<NT>::kRows - 1) / Q4Shape<NT>::kRows;
  int groups = (slots + splits - 1) / splits;
  if (groups > ngr) groups = ngr;
  const int gpc = (ngr + groups - 1) / groups;
  groups = (ngr + gpc - 1) / gpc;
  SplitArgs s2 = sk;
  s2.splits = splits;
  info->grid_x = groups;
  info->grid_y = splits;
  info->block = kQThreads;
  info->smem = smem;
  info->kernel = "q4_0_q8_1_mma";
  return launch_k(kern, dim3(groups, splits), dim3(kQThreads), smem, st, true, qs,
                  static_cast<const uint16_t*>(d), static_cast<const uint8_t*>(xq), M, Y, N, K,
                  kpb, gpc, s2, am);
}

template <int NT>
cudaError_t run_nt(const uint8_t* qs, const void* d, const void* xq, int M, float* Y, int N, int K,
                   const Q4Plan& plan, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                   Launch* info) {
  return am.out ? run_t<NT, true>(qs, d, xq, M, Y, N, K, plan, sk, am, st, info)
                : run_t<NT, false>(qs, d, xq, M, Y, N, K, plan, sk, am, st, info);
}

}  // namespace

int q4_mma_splits(int M, int N, int K, int forced) {
  return q4_plan(M, N, K, forced).splits;
}

size_t q4_mma_partial_bytes(int M, int N, int K, int forced) {
  const Q4Plan p = q4_plan(M, N, K, forced);
  if (p.splits <= 1) return 0;
  const int rows = p.nt >= 2 ? 32 : 16;
  const size_t ngr = (N + rows - 1) / rows;
  return static_cast<size_t>(p.splits) * ngr * rows * (8 * p.nt) * sizeof(float);
}

cudaError_t launch_q4_mma(const uint8_t* qs, const void* d, const void* xq, int M, float* Y, int N,
                          int K, int forced, const SplitArgs& sk, const ArgmaxArgs& am,
                          cudaStream_t st, Launch* info) {
  const Q4Plan plan = q4_plan(M, N, K, forced);
  switch (plan.nt) {
    case 1: return run_nt<1>(qs, d, xq, M, Y, N, K, plan, sk, am, st, info);
    case 2: return run_nt<2>(qs, d, xq, M, Y, N, K, plan, sk, am, st, info);
    case 3: return run_nt<3>(qs, d, xq, M, Y, N, K, plan, sk, am, st, info);
    default: return run_nt<4>(qs, d, xq, M, Y, N, K, plan, sk, am, st, info);
  }
}

}  // namespace wobs
