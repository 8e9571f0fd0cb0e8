// NF4 blockwise 4-bit decode GEMV for one to four activation columns, with
// the products on the tensor cores.
//
// bitsandbytes issue #1842 ("70B 4-bit LLM decode bottlenecked by HIP kernel
// (kgemm_4bit_inference_naive) efficiency"): the fused 4-bit inference GEMV
// for one decode token, 64-element blocks with a float absmax each, codes
// looked up in a 16-entry codebook.  On this GPU the CUDA-core form of that
// kernel is bound by its codebook lookups, not by DRAM: one shared-memory
// table read per code pair, and the float FMAs behind it, for each half
// byte of weight stream.  This variant moves the multiply-adds to mma.sync
// and splits the lookups between two pipes:
//
//   * codes decode to f16 pairs.  The codebook is scaled by a power of two
//     (so its largest entry lies in [2^14, 2^15)) and rounded to f16 once:
//     each weight carries a relative rounding error of at most 2^-11 and the
//     scale comes back out exactly in f32.  The activations are scaled the
//     same way per warp slice and are exact in f16;
//   * half of the code words go through a 256-entry byte -> f16-pair table in
//     shared memory, laid out so lane l always reads bank l (one wavefront
//     per warp lookup, whatever the codes); the other half go through
//     byte-permute lookups in four registers of low bytes and four of high
//     bytes (21 integer instructions per 8 codes, no memory traffic);
//   * a decoded byte is already an A-fragment register (two consecutive
//     codes of one row), so one m16n8k16 MMA covers 16 rows x 16 codes.  The
//     four MMAs of a 64-element block accumulate in f32 and the block sum is
//     scaled by its absmax in f32, as in the format's definition;
//   * a CTA takes blocks of 64 rows and streams each through a ring of
//     shared-memory stages of 64 rows x 1024 codes plus their absmax, each
//     filled by five 2-D tensor copies (128-byte x 64-row code boxes in the
//     128-byte swizzle) that one producer warp issues.  Each of the 16
//     compute warps owns 32 rows and two 64-code blocks of every stage; the
//     activation fragments, converted once, sit in the unused halves of the
//     table's 256-byte entry strides.  When the last stage of a row block is
//     released, the producer adds the 8 K-group partials of each row in a
//     fixed order and writes the outputs;
//   * MMA row i of a row tile is box row 2i (i < 8) or 2(i - 8) + 1, so the
//     8-byte code reads of a half warp meet four distinct swizzle phases and
//     no bank twice;
//   * the table lives at shared-window address 0x20000, so the lookup
//     address of a byte is one byte permute of the code word and a constant
//     (0x20000 | lane * 4), with no add;
//   * two to four columns share every decoded code: the MMA's B operand
//     has eight columns, lane (g, t) supplies column g % M, and the sums of
//     columns 2t and 2t + 1 come back in lane (g, t).  Column 1 fits in the
//     table's unused gaps; columns 2 and 3 need shared memory beside it, so
//     the ring has four stages for two columns and three for four.  One column keeps its
//     own kernel: the column form instantiated for one column ran 2 us
//     slower on the 70B matrix (28.9 against 26.9 us).
#include <cmath>
#include <cstdlib>

#include "common.cuh"
#include "nf4_decode.cuh"
#include "tcgen05.cuh"

namespace wobs {
namespace {

constexpr int kCW = 16;                      // compute warps: 2 row halves x 8 K groups
constexpr int kThreads = (kCW + 1) * 32;     // + the producer warp
constexpr int kRB = 64;                      // rows per row block
constexpr int kKG = 8;                       // K groups (two 64-code blocks each per stage)
constexpr uint32_t kTabAddr = 0x20000;       // shared-window address of the table
constexpr int kTabBytes = 256 * 256;         // entry e: 64 words at e * 256, lane l reads word l;
                                             // bytes 128..255 of entry c hold activation block c
constexpr int kMaxStages = 4;
constexpr int kMiscBytes = 512;              // barriers, counters, codebook, scales, argmax keys
constexpr int kRedBytes = kMaxStages * kKG * kRB * 4;   // one-column partials
// A stage: 64 rows x 1024 codes (four 128-byte x 64-row code boxes in the
// 128-byte swizzle, 8 KB each) and their 16 absmax per row (4 KB).
constexpr int kKS = 1024;                    // codes per row per stage
constexpr int kStage = 4 * 8192 + kRB * 64;  // 36864 bytes, a multiple of 1024
constexpr uint32_t kStageTx = kStage;

// Shared loads as pure functions of their address, so the compiler may
// interleave them with the MMAs.  Stage reads stay between the stage's full
// wait and its release because their addresses come from a value produced
// after the wait (`launder`) and the release takes the accumulators they
// feed as inputs.
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t launder(uint32_t v) {
  uint32_t r;
  asm volatile("mov.b32 %0, %1;" : "=r"(r) : "r"(v) : "memory");
  return r;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
               :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" :: "r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cta(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D = A.B (accumulator from zero)
__device__ __forceinline__ void mma16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                           uint32_t b1) {
  const float z = 0.f;
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}
// Release of a stage once `dep` (the accumulators its reads feed) exists.
__device__ __forceinline__ void mbar_arrive_after(uint64_t* bar, float d0, float d1, float d2,
                                                  float d3) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];"
               :: "r"(smem_addr(bar)), "f"(d0), "f"(d1), "f"(d2), "f"(d3) : "memory");
}

// One code word (4 bytes, 8 codes; byte j = element 2j in its high nibble,
// element 2j + 1 in its low nibble) -> four f16 pairs, low half = the even
// element.  Table variant: one lookup per byte.
// `tl` = kTabAddr | lane * 4: byte e of the word addresses table word
// e * 64 + lane, i.e. kTabAddr | e << 8 | lane << 2.
__device__ __forceinline__ void decode_table(uint32_t w, uint32_t tl, uint32_t (&r)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) r[j] = lds32(prmt(w, tl, 0x7604u | (j << 4)));
}

// Power-of-two scale 2^(141 - E) for a positive float with biased exponent E
// (clamped to [15, 254]): brings the value into [2^14, 2^15); `inv` is its
// exact inverse.
__device__ __forceinline__ void pow2_scale(float m, float& scale, float& inv) {
  int e = static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu);
  e = e < 15 ? 15 : e;
  scale = __uint_as_float(static_cast<uint32_t>(268 - e) << 23);
  inv = __uint_as_float(static_cast<uint32_t>(e - 14) << 23);
}

// Shared-memory layout, from the dynamic base `base` (same in every CTA):
// [base, +lead) barriers, counters and extra activation columns, [+lead,
// +lead + red) warp partials, then 1024-byte aligned stage slots up to the
// table at 0x20000, the table [0x20000, 0x30000), then more stage slots up
// to the end of the allocation.
struct Layout {
  uint32_t base, red, a0, b0;
  int na, S;
};
__device__ __forceinline__ Layout make_layout(uint32_t base, uint32_t bytes,
                                              uint32_t lead = kMiscBytes,
                                              uint32_t red_bytes = kRedBytes) {
  Layout L;
  L.base = base;
  L.red = base + lead;
  L.a0 = (L.red + red_bytes + 1023u) & ~1023u;
  L.b0 = kTabAddr + kTabBytes;
  const uint32_t end = base + bytes;
  L.na = L.a0 <= kTabAddr ? static_cast<int>((kTabAddr - L.a0) / kStage) : -1;
  const int nb = end >= L.b0 ? static_cast<int>((end - L.b0) / kStage) : -1;
  L.S = (L.na < 0 || nb < 0) ? 0 : (L.na + nb < kMaxStages ? L.na + nb : kMaxStages);
  return L;
}
__device__ __forceinline__ uint32_t slot_addr(const Layout& L, int s) {
  return s < L.na ? L.a0 + s * kStage : L.b0 + (s - L.na) * kStage;
}

// Warps 0..15 compute (row half warp & 1, K group warp >> 1), warp 16
// produces.  A CTA takes row blocks blockIdx.x, + gridDim.x, ...; each row
// block streams K in stages of 1024 codes.
template <int P, bool kArgmax>
__global__ void __launch_bounds__(kThreads, 1) nf4_mma_kernel(const __grid_constant__ CUtensorMap tq,
                                                             const __grid_constant__ CUtensorMap ta,
                                                             Codebook16 cb, float cb_scale,
                                                             float cb_inv,
                                                             const __nv_bfloat16* __restrict__ x,
                                                             __nv_bfloat16* __restrict__ y, int N,
                                                             int K, uint32_t smem_bytes,
                                                             int max_stages, ArgmaxArgs am,
                                                             int* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = smem_addr(smem);
  const Layout L = make_layout(base, smem_bytes);
  auto gen = [&](uint32_t a) { return smem + (a - base); };
  uint64_t* full = reinterpret_cast<uint64_t*>(gen(base));              // [8]
  uint64_t* empty = full + kMaxStages;                                   // [8]
  unsigned* nissue = reinterpret_cast<unsigned*>(gen(base + 128));       // [8]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gen(base + 160));
  uint16_t* cbh = reinterpret_cast<uint16_t*>(gen(base + 192));          // [16]
  float* wmax = reinterpret_cast<float*>(gen(base + 224));               // [8] (16 halves)
  uint64_t* keys = reinterpret_cast<uint64_t*>(gen(base + 288));         // [17], to base + 424
  float* red = reinterpret_cast<float*>(gen(L.red));                     // [S][8 K groups][64 rows]
  const int S = L.S < max_stages ? L.S : max_stages;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int spb = K / kKS;                  // stages per row block
  const int nblk = (N + kRB - 1) / kRB;
  const int T = static_cast<int>(blockIdx.x) < nblk
                    ? (nblk - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                    : 0;
  const int total = T * spb;                // stages this CTA streams
  if (S < 2) {                              // the table cannot sit at 0x20000: refuse, touch nothing
    if (tid == 0 && err) atomicExch(err, kErrGemvWait);
    return;
  }

  // stage j (row block j / spb, K part j % spb) -> slot j % S; lane 0 of the
  // producer warp calls it
  auto issue = [&](int j) {
    const int s = j % S;
    const uint32_t st = slot_addr(L, s);
    const int row0 = (static_cast<int>(blockIdx.x) + (j / spb) * static_cast<int>(gridDim.x)) * kRB;
    const int k0 = (j % spb) * (kKS / 2);   // byte column of the codes
    nissue[s] += 1u;
    mbar_expect_tx(full + s, kStageTx);
#pragma unroll
    for (int bx = 0; bx < 4; ++bx) tma_load_2d(st + bx * 8192, &tq, k0 + bx * 128, row0, full + s);
    tma_load_2d(st + 4 * 8192, &ta, (j % spb) * (kKS / 64), row0, full + s);
  };

  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kCW);
    }
    mbar_fence_init();
    *abort_flag = 0;
  }
  if (tid < kMaxStages) nissue[tid] = 0u;
  if (tid < 16) {
    float v = cb.v[0];
#pragma unroll
    for (int i = 1; i < 16; ++i) v = tid == i ? cb.v[i] : v;
    cbh[tid] = __half_as_ushort(__float2half_rn(v * cb_scale));
  }
  __syncthreads();
  if (tid == kCW * 32)
    for (int j = 0; j < S && j < total; ++j) issue(j);
  pdl_launch_dependents();

  Planes pl;
  if (warp < kCW) {
    // the codebook as the shared table (every entry's 32 lane words) and as
    // byte planes
    for (int i = tid; i < 256 * 32; i += kCW * 32) {
      const int e = i >> 5, l = i & 31;
      sts32(kTabAddr + e * 256 + l * 4,
            static_cast<uint32_t>(cbh[e >> 4]) | (static_cast<uint32_t>(cbh[e & 15]) << 16));
    }
    auto lob = [&](int i) { return static_cast<uint32_t>(cbh[i] & 0xFFu); };
    auto hib = [&](int i) { return static_cast<uint32_t>(cbh[i] >> 8); };
    pl.la0 = lob(0) | lob(1) << 8 | lob(2) << 16 | lob(3) << 24;
    pl.la1 = lob(4) | lob(5) << 8 | lob(6) << 16 | lob(7) << 24;
    pl.lb0 = lob(8) | lob(9) << 8 | lob(10) << 16 | lob(11) << 24;
    pl.lb1 = lob(12) | lob(13) << 8 | lob(14) << 16 | lob(15) << 24;
    pl.ha0 = hib(0) | hib(1) << 8 | hib(2) << 16 | hib(3) << 24;
    pl.ha1 = hib(4) | hib(5) << 8 | hib(6) << 16 | hib(7) << 24;
    pl.hb0 = hib(8) | hib(9) << 8 | hib(10) << 16 | hib(11) << 24;
    pl.hb1 = hib(12) | hib(13) << 8 | hib(14) << 16 | hib(15) << 24;
  }
  pdl_wait();
  // activations -> f16 in the table's gaps, block c at kTabAddr + c * 256 +
  // 128 (elements in order), all scaled by one power of two that puts max|x|
  // in [2^14, 2^15): the maximum first (warp w takes blocks w, w + 16, ...),
  // then the conversion
  const int nbk = K / 64;
  if (warp < kCW) {
    float mx = 0.f;
    for (int c = warp; c < nbk; c += kCW) {
      const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(x + c * 64) + lane);
      mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(v << 16)), fabsf(__uint_as_float(v & 0xFFFF0000u))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) wmax[warp] = mx;
  }
  __syncthreads();
  float xs, xinv;
  {
    float mx = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kCW; ++w2) mx = fmaxf(mx, wmax[w2]);
    pow2_scale(mx, xs, xinv);
  }
  if (warp < kCW) {
    for (int c = warp; c < nbk; c += kCW) {
      const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(x + c * 64) + lane);
      const __half2 h2 = __floats2half2_rn(__uint_as_float(v << 16) * xs,
                                           __uint_as_float(v & 0xFFFF0000u) * xs);
      sts32(kTabAddr + c * 256 + 128 + 4 * lane, *reinterpret_cast<const uint32_t*>(&h2));
    }
  }
  __syncthreads();                          // table and activation blocks complete

  uint64_t best = 0;
  bool ok = true;
  if (warp < kCW) {
    // ------------------------------------------------------------ compute
    const int rh = warp & 1, q = warp >> 1;
    const uint32_t tl = kTabAddr | (static_cast<uint32_t>(lane) << 2);
    const float out_mul = xinv * cb_inv;
    // rows of MMA row g in row tile u: 32 rh + 16 u + 2g, and + 1 for MMA
    // row g + 8.  This lane's 8 code bytes of block b of a row: logical
    // 16-byte chunk 4 (q & 1) + 2b + t / 2 of box q / 2, stored at chunk ^
    // (row & 7); the odd row's chunk differs by one in bit 0.
    const int r0 = 32 * rh + 2 * g;
    const uint32_t swz = (2 * g) & 7;
    uint32_t co[2][2];                      // [block][row parity] byte offsets in the stage
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t c = 4 * (q & 1) + 2 * b + (t >> 1);
      co[b][0] = (q >> 1) * 8192 + r0 * 128 + ((c ^ swz) << 4) + 8 * (t & 1);
      co[b][1] = (q >> 1) * 8192 + (r0 + 1) * 128 + ((c ^ swz ^ 1u) << 4) + 8 * (t & 1);
    }
    // absmax box: 64-byte rows in the 64-byte swizzle (16-byte chunk index ^=
    // (row >> 1) & 3); this lane's pair of K group q is chunk q / 2, half q & 1
    const uint32_t abs_off = 4 * 8192 + r0 * 64 + ((((q >> 1) ^ g) & 3) << 4) + 8 * (q & 1);
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};   // [row tile][row parity]
    int s = 0, ks = 0;
    uint32_t ph = 0;
    uint32_t st = slot_addr(L, 0);
    for (int j = 0; j < total; ++j) {
      if (*abort_flag) break;
      if (!mbar_wait(full + s, ph)) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      st = launder(st);
      float am[2][2][2];                    // [row tile][row parity][block]
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int p2 = 0; p2 < 2; ++p2) {
          const uint2 a = lds64(st + abs_off + (16 * u + p2) * 64);
          am[u][p2][0] = __uint_as_float(a.x);
          am[u][p2][1] = __uint_as_float(a.y);
        }
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t xa = kTabAddr + (ks * 16 + 2 * q + b) * 256 + 128 + 32 * t;
        const uint4 xv0 = lds128(xa), xv1 = lds128(xa + 16);
        const uint32_t xf[8] = {xv0.x, xv0.y, xv0.z, xv0.w, xv1.x, xv1.y, xv1.z, xv1.w};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint2 wg = lds64(st + co[b][0] + u * 16 * 128);
          const uint2 wh = lds64(st + co[b][1] + u * 16 * 128);
          const uint32_t words[4] = {wg.x, wg.y, wh.x, wh.y};
          uint32_t r[4][4];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            // P of every 8 code words (two blocks) through the register planes
            if (4 * b + qq >= 8 - P) decode_planes(words[qq], pl, r[qq]);
            else decode_table(words[qq], tl, r[qq]);
          }
          float d[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            // MMA m: bytes 2m, 2m + 1 of the lane's 8 bytes of both rows
            const int wq = m >> 1, jj = 2 * (m & 1);
            const uint32_t a[4] = {r[wq][jj], r[2 + wq][jj], r[wq][jj + 1], r[2 + wq][jj + 1]};
            if (m == 0) mma16816_z(d, a, xf[0], xf[1]);
            else mma16816(d, a, xf[2 * m], xf[2 * m + 1]);
          }
          acc[u][0] = fmaf(am[u][0][b], d[0], acc[u][0]);
          acc[u][1] = fmaf(am[u][1][b], d[2], acc[u][1]);
        }
      }
      if (ks == spb - 1) {
        // row block complete for this warp: its row partials, then a fresh start
        if (t == 0) {
          float* rs = red + (s * kKG + q) * kRB + r0;
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            rs[16 * u] = acc[u][0] * out_mul;
            rs[16 * u + 1] = acc[u][1] * out_mul;
            acc[u][0] = acc[u][1] = 0.f;
          }
        } else {
          acc[0][0] = acc[0][1] = acc[1][0] = acc[1][1] = 0.f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_after(empty + s, acc[0][0], acc[0][1], acc[1][0], acc[1][1]);
      if (++ks == spb) ks = 0;
      if (++s == S) { s = 0; ph ^= 1u; }
      st = slot_addr(L, s);
    }
  } else {
    // ----------------------------------------------------------- produce
    int s = 0;
    uint32_t ph = 0;
    for (int j = 0; j < total; ++j) {
      if (*abort_flag) break;
      if (!mbar_wait(empty + s, ph)) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      if (j % spb == spb - 1) {
        // every compute warp has left its partials of this row block in slot s:
        // rows lane and lane + 32, K groups added in order
        const int row0 = (static_cast<int>(blockIdx.x) + (j / spb) * static_cast<int>(gridDim.x)) * kRB;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int rr = lane + 32 * hh, row = row0 + rr;
          if (row < N) {
            const float* rs = red + s * kKG * kRB + rr;
            float v = rs[0];
#pragma unroll
            for (int q2 = 1; q2 < kKG; ++q2) v += rs[q2 * kRB];
            const __nv_bfloat16 o = __float2bfloat16_rn(v);
            y[row] = o;
            if (kArgmax) {
              const uint64_t k = argmax_key(__bfloat162float(o), static_cast<uint32_t>(row));
              best = k > best ? k : best;
            }
          }
        }
        __syncwarp();
      }
      if (j + S < total && lane == 0) issue(j + S);
      __syncwarp();
      if (++s == S) { s = 0; ph ^= 1u; }
    }
  }
  if (!ok && lane == 0 && err) atomicExch(err, kErrGemvWait);
  __syncthreads();
  if (*abort_flag && tid == 0) {
    // let every issued copy land before the CTA's shared memory is released
    for (int s2 = 0; s2 < S; ++s2)
      if (nissue[s2] > 0u) mbar_wait(full + s2, (nissue[s2] - 1u) & 1u);
  }
  if (kArgmax) {
    best = warp_max_u64(best);
    if (lane == 0) keys[warp] = best;
    __syncthreads();
    if (tid == 0) {
      uint64_t k = 0;
      for (int w2 = 0; w2 <= kCW; ++w2) k = keys[w2] > k ? keys[w2] : k;
      keys[0] = k;
    }
    __syncthreads();
    argmax_publish(keys, 1, am, gridDim.x);
  }
}

// The same GEMV for MC activation columns (2 or 4; M <= MC of them exist),
// same warps, stages and decode: the B operand of
// m16n8k16 has eight columns, so lane (g, t) supplies activation column g %
// M and the decoded codes, the shared-memory lookups and the MMAs serve
// every column at once; lane (g, t) then holds the sums of columns 2t and 2t
// + 1.  Columns 0 and 1 sit in the table's gaps (entries 0..127 and
// 128..255; K <= 8192 is at most 128 blocks), columns 2.. M - 1 in their
// own region after the barriers ([column - 2][block][64 f16]); column 1's
// 16-byte pieces are stored rotated by one place.  Each column has its own
// power-of-two scale.  The K-group partials need one buffer
// when a row block spans more stages than the ring holds (no warp can then
// reach the next row block's end before the copy warp has read them), else
// one per slot.
template <int P, bool kArgmax, int MC>
__global__ void __launch_bounds__(kThreads, 1) nf4_mma_mc_kernel(const __grid_constant__ CUtensorMap tq,
                                                             const __grid_constant__ CUtensorMap ta,
                                                             Codebook16 cb, float cb_scale,
                                                             float cb_inv,
                                                             const __nv_bfloat16* __restrict__ x,
                                                             int64_t ldx, int M,
                                                             __nv_bfloat16* __restrict__ y, int N,
                                                             int K, uint32_t smem_bytes,
                                                             int max_stages, ArgmaxArgs am,
                                                             int* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t base = smem_addr(smem);
  const int nbk = K / 64;
  // activation columns 2.. right after the barriers, then the partials
  // [nred][8 K groups][64 rows][MC], for the deepest ring that fits
  const uint32_t xcol = base + kMiscBytes;
  static_assert(MC == 2 || MC == 4, "two or four columns");
  const int spb0 = K / kKS;
  const uint32_t xbytes = M > 2 ? static_cast<uint32_t>(M - 2) * nbk * 128u : 0u;
  Layout L{};
  int nred = 1;
  for (int s_try = kMaxStages; s_try >= 2; --s_try) {
    nred = spb0 > s_try ? 1 : s_try;
    L = make_layout(base, smem_bytes, kMiscBytes + xbytes,
                    static_cast<uint32_t>(nred) * kKG * kRB * 4 * MC);
    if (L.S >= s_try) {
      L.S = s_try;
      break;
    }
    L.S = 0;
  }
  auto gen = [&](uint32_t a) { return smem + (a - base); };
  uint64_t* full = reinterpret_cast<uint64_t*>(gen(base));              // [4]
  uint64_t* empty = full + kMaxStages;                                   // [4]
  uint64_t* keys = reinterpret_cast<uint64_t*>(gen(base + 64));          // [MC]
  unsigned* nissue = reinterpret_cast<unsigned*>(gen(base + 128));       // [4]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gen(base + 160));
  uint16_t* cbh = reinterpret_cast<uint16_t*>(gen(base + 192));          // [16]
  float* wmax = reinterpret_cast<float*>(gen(base + 224));               // [16 warps][MC], to base + 480
  float* red = reinterpret_cast<float*>(gen(L.red));                     // [S][8][64][MC]
  const int S = L.S < max_stages ? L.S : max_stages;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int spb = K / kKS;                  // stages per row block
  const int nblk = (N + kRB - 1) / kRB;
  const int T = static_cast<int>(blockIdx.x) < nblk
                    ? (nblk - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                    : 0;
  const int total = T * spb;                // stages this CTA streams
  if (S < 2) {                              // no room for two stages: refuse, touch nothing
    if (tid == 0 && err) atomicExch(err, kErrGemvWait);
    return;
  }

  // stage j (row block j / spb, K part j % spb) -> slot j % S; lane 0 of the
  // producer warp calls it
  auto issue = [&](int j) {
    const int s = j % S;
    const uint32_t st = slot_addr(L, s);
    const int row0 = (static_cast<int>(blockIdx.x) + (j / spb) * static_cast<int>(gridDim.x)) * kRB;
    const int k0 = (j % spb) * (kKS / 2);   // byte column of the codes
    nissue[s] += 1u;
    mbar_expect_tx(full + s, kStageTx);
#pragma unroll
    for (int bx = 0; bx < 4; ++bx) tma_load_2d(st + bx * 8192, &tq, k0 + bx * 128, row0, full + s);
    tma_load_2d(st + 4 * 8192, &ta, (j % spb) * (kKS / 64), row0, full + s);
  };

  if (tid == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, kCW);
    }
    mbar_fence_init();
    *abort_flag = 0;
  }
  if (tid < kMaxStages) nissue[tid] = 0u;
  if (tid < 16) {
    float v = cb.v[0];
#pragma unroll
    for (int i = 1; i < 16; ++i) v = tid == i ? cb.v[i] : v;
    cbh[tid] = __half_as_ushort(__float2half_rn(v * cb_scale));
  }
  __syncthreads();
  if (tid == kCW * 32)
    for (int j = 0; j < S && j < total; ++j) issue(j);
  pdl_launch_dependents();

  Planes pl;
  if (warp < kCW) {
    // the codebook as the shared table (every entry's 32 lane words) and as
    // byte planes
    for (int i = tid; i < 256 * 32; i += kCW * 32) {
      const int e = i >> 5, l = i & 31;
      sts32(kTabAddr + e * 256 + l * 4,
            static_cast<uint32_t>(cbh[e >> 4]) | (static_cast<uint32_t>(cbh[e & 15]) << 16));
    }
    auto lob = [&](int i) { return static_cast<uint32_t>(cbh[i] & 0xFFu); };
    auto hib = [&](int i) { return static_cast<uint32_t>(cbh[i] >> 8); };
    pl.la0 = lob(0) | lob(1) << 8 | lob(2) << 16 | lob(3) << 24;
    pl.la1 = lob(4) | lob(5) << 8 | lob(6) << 16 | lob(7) << 24;
    pl.lb0 = lob(8) | lob(9) << 8 | lob(10) << 16 | lob(11) << 24;
    pl.lb1 = lob(12) | lob(13) << 8 | lob(14) << 16 | lob(15) << 24;
    pl.ha0 = hib(0) | hib(1) << 8 | hib(2) << 16 | hib(3) << 24;
    pl.ha1 = hib(4) | hib(5) << 8 | hib(6) << 16 | hib(7) << 24;
    pl.hb0 = hib(8) | hib(9) << 8 | hib(10) << 16 | hib(11) << 24;
    pl.hb1 = hib(12) | hib(13) << 8 | hib(14) << 16 | hib(15) << 24;
  }
  pdl_wait();
  // activations -> f16: block c of column 0 at kTabAddr + c * 256 + 128, of
  // column 1 at kTabAddr + (128 + c) * 256 + 128, of column m >= 2 at xcol +
  // ((m - 2) * nbk + c) * 128 (elements in order),
  // each column scaled by one power of two that puts its max |x| in [2^14,
  // 2^15): the maxima first (warp w takes blocks w, w + 16, ...), then the
  // conversion
  auto xaddr = [&](int m, int c) -> uint32_t {
    return m < 2 ? kTabAddr + (128 * m + c) * 256 + 128 : xcol + ((m - 2) * nbk + c) * 128;
  };
  if (warp < kCW) {
    float mx[MC];
#pragma unroll
    for (int m = 0; m < MC; ++m) mx[m] = 0.f;
    for (int c = warp; c < nbk; c += kCW) {
#pragma unroll
      for (int m = 0; m < MC; ++m)
        if (m < M) {
          const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(x + m * ldx + c * 64) + lane);
          mx[m] = fmaxf(mx[m], fmaxf(fabsf(__uint_as_float(v << 16)), fabsf(__uint_as_float(v & 0xFFFF0000u))));
        }
    }
#pragma unroll
    for (int m = 0; m < MC; ++m) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx[m] = fmaxf(mx[m], __shfl_xor_sync(0xffffffffu, mx[m], o));
      if (lane == 0) wmax[warp * MC + m] = mx[m];
    }
  }
  __syncthreads();
  float xs[MC], xinv[MC];
#pragma unroll
  for (int m = 0; m < MC; ++m) {
    float mx = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kCW; ++w2) mx = fmaxf(mx, wmax[w2 * MC + m]);
    pow2_scale(mx, xs[m], xinv[m]);
  }
  if (warp < kCW) {
    for (int c = warp; c < nbk; c += kCW) {
#pragma unroll
      for (int m = 0; m < MC; ++m)
        if (m < M) {
          const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(x + m * ldx + c * 64) + lane);
          const __half2 h2 = __floats2half2_rn(__uint_as_float(v << 16) * xs[m],
                                               __uint_as_float(v & 0xFFFF0000u) * xs[m]);
          // column 1's 16-byte pieces rotated by one: its lanes then read
          // other banks than column 0's in the same load
          const uint32_t o = m == 1 ? ((((lane >> 2) + 1) & 7) << 4) | ((4 * lane) & 15) : 4 * lane;
          sts32(xaddr(m, c) + o, *reinterpret_cast<const uint32_t*>(&h2));
        }
    }
  }
  __syncthreads();                          // table and activation blocks complete

  uint64_t best[MC];
#pragma unroll
  for (int m = 0; m < MC; ++m) best[m] = 0;
  bool ok = true;
  if (warp < kCW) {
    // ------------------------------------------------------------ compute
    const int rh = warp & 1, q = warp >> 1;
    const uint32_t tl = kTabAddr | (static_cast<uint32_t>(lane) << 2);
    // this lane's activation column (B column g) and its block stride
    const int xm = g % M;
    const uint32_t xb = xaddr(xm, 0), xst = xm < 2 ? 256u : 128u;
    const uint32_t xo0 = xm == 1 ? ((2 * t + 1) & 7) << 4 : 32 * t;
    const uint32_t xo1 = xm == 1 ? ((2 * t + 2) & 7) << 4 : 32 * t + 16;
    // output scales of the two columns this lane's sums belong to
    // (lanes t = 0, 1 carry columns 0..3; the others' sums are not used)
    float om0 = xinv[0] * cb_inv, om1 = xinv[1] * cb_inv;
    if constexpr (MC == 4) {
      const float e0 = xinv[0] * cb_inv, e1 = xinv[1] * cb_inv;
      const float e2 = xinv[2] * cb_inv, e3 = xinv[3] * cb_inv;
      om0 = (t & 1) ? e2 : e0;
      om1 = (t & 1) ? e3 : e1;
    }
    // rows of MMA row g in row tile u: 32 rh + 16 u + 2g, and + 1 for MMA
    // row g + 8.  This lane's 8 code bytes of block b of a row: logical
    // 16-byte chunk 4 (q & 1) + 2b + t / 2 of box q / 2, stored at chunk ^
    // (row & 7); the odd row's chunk differs by one in bit 0.
    const int r0 = 32 * rh + 2 * g;
    const uint32_t swz = (2 * g) & 7;
    uint32_t co[2][2];                      // [block][row parity] byte offsets in the stage
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t c = 4 * (q & 1) + 2 * b + (t >> 1);
      co[b][0] = (q >> 1) * 8192 + r0 * 128 + ((c ^ swz) << 4) + 8 * (t & 1);
      co[b][1] = (q >> 1) * 8192 + (r0 + 1) * 128 + ((c ^ swz ^ 1u) << 4) + 8 * (t & 1);
    }
    // absmax box: 64-byte rows in the 64-byte swizzle (16-byte chunk index ^=
    // (row >> 1) & 3); this lane's pair of K group q is chunk q / 2, half q & 1
    const uint32_t abs_off = 4 * 8192 + r0 * 64 + ((((q >> 1) ^ g) & 3) << 4) + 8 * (q & 1);
    constexpr int NH = 2;                   // output columns per lane
    float acc[2][2][NH];                    // [row tile][row parity][column]
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int p2 = 0; p2 < 2; ++p2)
#pragma unroll
        for (int h = 0; h < NH; ++h) acc[u][p2][h] = 0.f;
    int s = 0, ks = 0;
    uint32_t ph = 0;
    uint32_t st = slot_addr(L, 0);
    for (int j = 0; j < total; ++j) {
      if (*abort_flag) break;
      if (!mbar_wait(full + s, ph)) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      st = launder(st);
      float amx[2][2][2];                   // [row tile][row parity][block]
#pragma unroll
      for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int p2 = 0; p2 < 2; ++p2) {
          const uint2 a = lds64(st + abs_off + (16 * u + p2) * 64);
          amx[u][p2][0] = __uint_as_float(a.x);
          amx[u][p2][1] = __uint_as_float(a.y);
        }
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const uint32_t xa = xb + (ks * 16 + 2 * q + b) * xst;
        const uint4 xv0 = lds128(xa + xo0), xv1 = lds128(xa + xo1);
        const uint32_t xf[8] = {xv0.x, xv0.y, xv0.z, xv0.w, xv1.x, xv1.y, xv1.z, xv1.w};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint2 wg = lds64(st + co[b][0] + u * 16 * 128);
          const uint2 wh = lds64(st + co[b][1] + u * 16 * 128);
          const uint32_t words[4] = {wg.x, wg.y, wh.x, wh.y};
          uint32_t r[4][4];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            // P of every 8 code words (two blocks) through the register planes
            if (4 * b + qq >= 8 - P) decode_planes(words[qq], pl, r[qq]);
            else decode_table(words[qq], tl, r[qq]);
          }
          float d[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            // MMA m: bytes 2m, 2m + 1 of the lane's 8 bytes of both rows
            const int wq = m >> 1, jj = 2 * (m & 1);
            const uint32_t a[4] = {r[wq][jj], r[2 + wq][jj], r[wq][jj + 1], r[2 + wq][jj + 1]};
            if (m == 0) mma16816_z(d, a, xf[0], xf[1]);
            else mma16816(d, a, xf[2 * m], xf[2 * m + 1]);
          }
#pragma unroll
          for (int h = 0; h < NH; ++h) {
            acc[u][0][h] = fmaf(amx[u][0][b], d[h], acc[u][0][h]);
            acc[u][1][h] = fmaf(amx[u][1][b], d[2 + h], acc[u][1][h]);
          }
        }
      }
      if (ks == spb - 1) {
        // row block complete for this warp: its row partials, then a fresh start
        if (2 * t < MC) {
          float* rs = red + (((nred == 1 ? 0 : s) * kKG + q) * kRB + r0) * MC + 2 * t;
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int p2 = 0; p2 < 2; ++p2) {
              rs[(16 * u + p2) * MC] = acc[u][p2][0] * om0;
              rs[(16 * u + p2) * MC + 1] = acc[u][p2][NH - 1] * om1;
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int p2 = 0; p2 < 2; ++p2)
#pragma unroll
            for (int h = 0; h < NH; ++h) acc[u][p2][h] = 0.f;
      }
      __syncwarp();
      if (lane == 0)
        mbar_arrive_after(empty + s, acc[0][0][0], acc[0][1][0], acc[1][0][0], acc[1][1][NH - 1]);
      if (++ks == spb) ks = 0;
      if (++s == S) { s = 0; ph ^= 1u; }
      st = slot_addr(L, s);
    }
  } else {
    // ----------------------------------------------------------- produce
    int s = 0;
    uint32_t ph = 0;
    for (int j = 0; j < total; ++j) {
      if (*abort_flag) break;
      if (!mbar_wait(empty + s, ph)) {
        ok = false;
        *abort_flag = 1;
        break;
      }
      if (j % spb == spb - 1) {
        // every compute warp has left its partials of this row block in slot s:
        // rows lane and lane + 32, K groups added in order
        const int row0 = (static_cast<int>(blockIdx.x) + (j / spb) * static_cast<int>(gridDim.x)) * kRB;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int rr = lane + 32 * hh, row = row0 + rr;
          if (row < N) {
#pragma unroll
            for (int m = 0; m < MC; ++m) {
              if (m < M) {
                const float* rs = red + ((nred == 1 ? 0 : s) * kKG * kRB + rr) * MC + m;
                float v = rs[0];
#pragma unroll
                for (int q2 = 1; q2 < kKG; ++q2) v += rs[q2 * kRB * MC];
                const __nv_bfloat16 o = __float2bfloat16_rn(v);
                y[static_cast<int64_t>(m) * N + row] = o;
                if (kArgmax) {
                  const uint64_t k = argmax_key(__bfloat162float(o), static_cast<uint32_t>(row));
                  best[m] = k > best[m] ? k : best[m];
                }
              }
            }
          }
        }
        __syncwarp();
      }
      if (j + S < total && lane == 0) issue(j + S);
      __syncwarp();
      if (++s == S) { s = 0; ph ^= 1u; }
    }
  }
  if (!ok && lane == 0 && err) atomicExch(err, kErrGemvWait);
  __syncthreads();
  if (*abort_flag && tid == 0) {
    // let every issued copy land before the CTA's shared memory is released
    for (int s2 = 0; s2 < S; ++s2)
      if (nissue[s2] > 0u) mbar_wait(full + s2, (nissue[s2] - 1u) & 1u);
  }
  if (kArgmax) {
    // only the producer warp folds outputs into the keys
    if (warp == kCW) {
#pragma unroll
      for (int m = 0; m < MC; ++m) {
        const uint64_t k = warp_max_u64(best[m]);
        if (lane == 0) keys[m] = k;
      }
    }
    __syncthreads();
    argmax_publish(keys, M, am, gridDim.x);
  }
}

// 2-D tensor map over a row-major [rows][cols] matrix (row pitch `ld`
// bytes), no fill beyond the edges other than zeros.
bool make_map(CUtensorMap* map, CUtensorMapDataType type, int esize, const void* ptr, int64_t cols,
              int64_t rows, int64_t ld, int box_cols, int box_rows, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  (void)esize;
  return fn(map, type, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int P, bool kArgmax, int MC>
cudaError_t run_p(const uint8_t* qs, const float* absmax, const Codebook16& cb, float cb_scale,
                  float cb_inv, const void* x, int64_t ldx, int M, void* y, int N, int K,
                  const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  auto kern = [] {
    if constexpr (MC == 1) return nf4_mma_kernel<P, kArgmax>;
    else return nf4_mma_mc_kernel<P, kArgmax, MC>;
  }();
  // all the opt-in shared memory the static part leaves, set up once (-1 if
  // the attribute calls fail)
  static const int smem = [&] {
    cudaFuncAttributes fa;
    int dev = 0, optin = 0;
    if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return -1;
    const int bytes = optin - static_cast<int>(fa.sharedSizeBytes);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
      return -1;
    return bytes;
  }();
  // the allocation must reach past the table at 0x20000 (two stages fit below it)
  if (smem < static_cast<int>(kTabAddr + kTabBytes)) {
    cudaGetLastError();
    return cudaErrorNotSupported;
  }
  CUtensorMap tq, ta;
  if (!make_map(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qs, K / 2, N, K / 2, 128, kRB,
                CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, absmax, K / 64, N, K / 16, 16, kRB,
                CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorNotSupported;
  const int nblk = (N + kRB - 1) / kRB;
  int grid = device_sm_count();
  if (grid > nblk) grid = nblk;
  info->grid_x = grid;
  info->block = kThreads;
  info->smem = smem;
  info->kernel = "nf4_mma";
  // ring depth: every stage the shared memory holds (WOBS_NF4_STAGES = 2..4
  // caps it, for measurements)
  const char* sv = std::getenv("WOBS_NF4_STAGES");
  const int max_stages = sv ? std::atoi(sv) : kMaxStages;
  const int ms = max_stages < 2 ? 2 : max_stages;
  if constexpr (MC == 1)
    return launch_k(kern, dim3(grid), dim3(kThreads), smem, st, true, tq, ta, cb, cb_scale, cb_inv,
                    static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), N, K,
                    static_cast<uint32_t>(smem), ms, am, error_word_ptr());
  else
    return launch_k(kern, dim3(grid), dim3(kThreads), smem, st, true, tq, ta, cb, cb_scale, cb_inv,
                    static_cast<const __nv_bfloat16*>(x), ldx, M, static_cast<__nv_bfloat16*>(y), N,
                    K, static_cast<uint32_t>(smem), ms, am, error_word_ptr());
}

template <bool kArgmax, int MC>
cudaError_t run(const uint8_t* qs, const float* absmax, const Codebook16& cb, float cb_scale,
                float cb_inv, const void* x, int64_t ldx, int M, void* y, int N, int K,
                const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  // code words per 8 decoded through the register planes instead of the
  // shared table (WOBS_NF4_P = 0..3 overrides the default)
  const char* v = std::getenv("WOBS_NF4_P");
  const int p = v ? std::atoi(v) : 1;
  if (p == 0)
    return run_p<0, kArgmax, MC>(qs, absmax, cb, cb_scale, cb_inv, x, ldx, M, y, N, K, am, st, info);
  if (p == 2)
    return run_p<2, kArgmax, MC>(qs, absmax, cb, cb_scale, cb_inv, x, ldx, M, y, N, K, am, st, info);
  if (p == 3)
    return run_p<3, kArgmax, MC>(qs, absmax, cb, cb_scale, cb_inv, x, ldx, M, y, N, K, am, st, info);
  return run_p<1, kArgmax, MC>(qs, absmax, cb, cb_scale, cb_inv, x, ldx, M, y, N, K, am, st, info);
}

template <int MC>
cudaError_t run_mc(const uint8_t* qs, const float* absmax, const Codebook16& cb, float cb_scale,
                   float cb_inv, const void* x, int64_t ldx, int M, void* y, int N, int K,
                   const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  return am.out ? run<true, MC>(qs, absmax, cb, cb_scale, cb_inv, x, ldx, M, y, N, K, am, st, info)
                : run<false, MC>(qs, absmax, cb, cb_scale, cb_inv, x, ldx, M, y, N, K, am, st, info);
}

}  // namespace

// The f16 codebook is usable when every entry is finite and every nonzero
// entry, after the power-of-two scale that puts the largest magnitude in
// [2^14, 2^15), is an f16 normal number (relative rounding error <= 2^-11).
bool nf4_codebook_scale(const Codebook16& cb, float* scale, float* inv) {
  float mx = 0.f;
  for (float v : cb.v) {
    if (!std::isfinite(v)) return false;
    mx = std::fmax(mx, std::fabs(v));
  }
  if (mx == 0.f) { *scale = 1.f; *inv = 1.f; return true; }
  int ex;
  std::frexp(mx, &ex);                    // mx in [2^(ex-1), 2^ex)
  if (ex < -100 || ex > 100) return false;
  const float sc = std::ldexp(1.f, 15 - ex);
  for (float v : cb.v)
    if (v != 0.f && std::fabs(v) * sc < std::ldexp(1.f, -14)) return false;
  *scale = sc;
  *inv = std::ldexp(1.f, ex - 15);
  return true;
}

cudaError_t launch_nf4_mma(const uint8_t* qs, const float* absmax, const Codebook16& cb,
                           const void* x, int64_t ldx, int M, void* y, int N, int K,
                           const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  float sc, inv;
  if (!nf4_codebook_scale(cb, &sc, &inv)) return cudaErrorNotSupported;
  if (reinterpret_cast<uintptr_t>(qs) % 16 || reinterpret_cast<uintptr_t>(absmax) % 16 ||
      reinterpret_cast<uintptr_t>(x) % 16)
    return cudaErrorNotSupported;
  // stages of 1024 codes per row; at most 128 blocks of 64, the activation
  // blocks the table's gaps hold; up to four columns, rows 16-byte aligned
  if (K % kKS != 0 || K > 8192 || M < 1 || M > 4) return cudaErrorNotSupported;
  if (M > 1 && (ldx % 8 != 0)) return cudaErrorNotSupported;
  if (M == 1) return run_mc<1>(qs, absmax, cb, sc, inv, x, K, 1, y, N, K, am, st, info);
  if (M == 2) return run_mc<2>(qs, absmax, cb, sc, inv, x, ldx, M, y, N, K, am, st, info);
  return run_mc<4>(qs, absmax, cb, sc, inv, x, ldx, M, y, N, K, am, st, info);
}

}  // namespace wobs
