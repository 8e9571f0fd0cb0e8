// NF4 blockwise 4-bit GEMV for 2..32 activation columns on the fifth-
// generation tensor cores (tcgen05), weights decoded into tensor memory.
//
// bitsandbytes issue #1842 ("70B 4-bit LLM decode bottlenecked by HIP
// kernel..."): the fused 4-bit GEMV y = W x with NF4 weights (64-element
// blocks, an fp32 absmax each, codes indexing a 16-entry codebook) against
// dequantising the whole matrix first.  With several activation columns the
// code lookups are shared by every column; here the multiply-adds go to the
// tensor cores and the decode happens once per weight:
//
//   * weights: the code c of block b of row n becomes the f16 value
//     absmax[n][b] * codebook[c] * 2^s (the fp32 product of the two
//     operands, rounded once to f16), s a power of two per row and work unit
//     that puts the unit's largest |absmax| * max|codebook| in [2^14, 2^15);
//     the sixteen values of a block are built once and held as byte planes
//     in registers, and each 4-byte code word (eight codes) is looked up by
//     byte permutes;
//   * activations: bf16 values times a power of two per column (max |x| of
//     the column over the CTA's K range into [2^14, 2^15)), exact in f16;
//   * y[m][n] = sum over K of the products, accumulated in fp32 by
//     tcgen05.mma (kind::f16, M = 128 rows, N = 16 or 32 columns), then both
//     powers of two are taken out exactly in fp32.
// Each weight is within 2^-11 (plus 2^-24) of its exact value relative to
// |w|, the activations are exact, inside the GEMV tolerance of
// 1e-3 * sum |w_i x_i|; y is rounded to bf16.
//
// Pipeline (one CTA per SM, warp-specialised, the Q4_0 tensor-memory
// kernel's structure):
//   * warp 0, one thread: 2-D TMA copies of 128 rows x 256 codes (128-byte
//     swizzle) into an 8-stage ring, and of the unit's absmax (128 rows x
//     R / 64 floats) into one of two buffers;
//   * warps 2..9: each thread owns one weight row (its tensor-memory lane)
//     and two of a stage's four blocks; it decodes them into f16 pairs in
//     tensor memory (three A buffers of 256 K) and publishes the row's scale
//     of each unit for the epilogue;
//   * warp 1, one thread: tcgen05.mma with A from tensor memory and B (the
//     activations of the CTA's K range, converted once, 128-byte swizzle)
//     from shared memory, fp32 accumulators in tensor memory (two buffers);
//   * warps 10..13: read the accumulator (one row per thread), remove the
//     scales, write bf16 y or fp32 split-K partials, fold the greedy argmax.
// Work units are (128-row tile, K range); every CTA keeps one K range.
// Split K ranges are added in split order by the CTA that completes a tile.
// Every wait is bounded: on expiry the CTA records the error word and stops.
#include <cmath>
#include <cstdlib>

#include "../../include/wobs.h"
#include "common.cuh"
#include "nf4_decode.cuh"
#include "tcgen05.cuh"

namespace wobs {
namespace {

constexpr int kRows = 128;                       // weight rows per tile (MMA M)
constexpr int kSK = 256;                         // codes per row per TMA stage (4 blocks of 64)
constexpr int kStageBytes = kRows * kSK / 2;     // 16384
constexpr int kMaxUnits = 256;                   // work units of one CTA at most
constexpr int kThreads = 448;                    // TMA, MMA, 8 decoder, 4 epilogue warps
constexpr int kAcols = kSK / 2;                  // tensor-memory columns of one A buffer
constexpr int kAbufs = 3;
constexpr int kDcol0 = kAbufs * kAcols;          // first accumulator column
constexpr int kTmemCols = 512;
constexpr int kSclSlots = 8;                     // row-scale slots (units in flight < 8)

static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");

template <int BN>
struct TcN {
  static constexpr int kMaxR = 1024;
  static constexpr int kStages = 8;
  static constexpr int kSBuf = kRows * (kMaxR / 16);   // R / 64 fp32 absmax per row
  static constexpr int kBoxBytes = BN * 128;           // one 64-element K box of B
  static constexpr int kBBytes = (kMaxR / 64) * kBoxBytes;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + 2 * kSBuf + kBBytes;
};

// kind::f16 instruction descriptor: f32 accumulator, f16 A and B, K-major,
// M = 128, N = BN.
template <int BN>
__device__ __forceinline__ uint32_t nf4tc_idesc() {
  return (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(kRows >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Power of two 2^(141 - E) for a positive float with biased exponent E
// (clamped to [15, 254]) that brings it into [2^14, 2^15), and its exact
// inverse; 1 and 1 for zero.
__device__ __forceinline__ void pow2_into_f16_top(float v, float& scale, float& inv) {
  if (!(v > 0.f)) {
    scale = inv = 1.f;
    return;
  }
  int e = static_cast<int>((__float_as_uint(v) >> 23) & 0xFFu);
  e = e < 15 ? 15 : e;
  scale = __uint_as_float(static_cast<uint32_t>(268 - e) << 23);
  inv = __uint_as_float(static_cast<uint32_t>(e - 14) << 23);
}

__device__ __forceinline__ void decoder_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

template <int BN, bool kArgmax>
__global__ void __launch_bounds__(kThreads, 1) nf4_tc_kernel(const __grid_constant__ CUtensorMap tq,
                                                             const __grid_constant__ CUtensorMap ta,
                                                             Codebook16 cb,
                                                             const __nv_bfloat16* __restrict__ X,
                                                             int64_t ldx, int M,
                                                             __nv_bfloat16* __restrict__ Y, int N,
                                                             int K, int R, int S, SplitArgs sk,
                                                             ArgmaxArgs am, int* err) {
  using Sh = TcN<BN>;
  constexpr int kStages = Sh::kStages;
  constexpr int kSBuf = Sh::kSBuf;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], afull[kAbufs], aempty[kAbufs], tfull[2],
      tempty[2], sfull[2], sempty[2], sclfull[kSclSlots], bready, done;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ unsigned char s_lastu[kMaxUnits];   // per unit: this CTA completed the tile
  __shared__ float s_scl[kSclSlots][kRows];      // per unit slot and row: 2^-s of the row's weights
  __shared__ float s_cb[16];
  __shared__ float s_cbmax;
  __shared__ unsigned s_colmax[32];              // max |x| per column (float bits)
  __shared__ float s_colinv[32];                 // per column: 2^-t of the activations
  __shared__ uint64_t s_key[4][32];
  __shared__ uint64_t s_kc[32];                  // split-K argmax keys per column
  __shared__ uint64_t s_cta[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t sbase = base + kStages * kStageBytes;     // two absmax buffers
  const uint32_t bbase = sbase + 2 * kSBuf;               // activation tile
  uint8_t* const gbase = smem_raw + (base - smem_addr(smem_raw));   // generic view of `base`
  const int ntiles = (N + kRows - 1) / kRows;
  const int split = static_cast<int>(blockIdx.x) % S;
  const int tile0 = static_cast<int>(blockIdx.x) / S, tstep = static_cast<int>(gridDim.x) / S;
  const int my_units = tile0 < ntiles ? (ntiles - 1 - tile0) / tstep + 1 : 0;
  const int su = R / kSK;                        // stages per unit
  const int total = my_units * su;
  const int k0 = split * R;                      // this CTA's K range [k0, k0 + R)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 8);
    }
    for (int a = 0; a < kAbufs; ++a) {
      mbar_init(&afull[a], 8);
      mbar_init(&aempty[a], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
      mbar_init(&sfull[a], 1);
      mbar_init(&sempty[a], 8);
    }
    for (int a = 0; a < kSclSlots; ++a) mbar_init(&sclfull[a], 8);
    mbar_init(&bready, 8);
    mbar_init(&done, 1);
    s_abort = 0;
    float mx = 0.f;
    for (int c = 0; c < 16; ++c) {
      s_cb[c] = cb.v[c];
      mx = fmaxf(mx, fabsf(cb.v[c]));
    }
    s_cbmax = mx;
    for (int c = 0; c < 32; ++c) {
      s_kc[c] = 0ull;
      s_colmax[c] = 0u;
      for (int w = 0; w < 4; ++w) s_key[w][c] = 0ull;
    }
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(&s_tmem)), "r"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- weight copies (weights are never written by a decode kernel)
    if (lane == 0) {
      int issued = 0, sissued = 0;
      for (int i = 0; i < total; ++i) {
        const int s = i % kStages;
        const int u = i / su, tile = tile0 + u * tstep;
        if (i % su == 0) {
          // the unit's absmax: R / 64 floats of each of the tile's rows
          const int sb = u & 1;
          if (u >= 2 && !mbar_wait(&sempty[sb], ((u >> 1) & 1) ^ 1)) { s_abort = 1; break; }
          mbar_expect_tx(&sfull[sb], kRows * (R >> 4));
          tma_load_2d(sbase + sb * kSBuf, &ta, k0 >> 6, tile * kRows, &sfull[sb]);
          sissued = u + 1;
        }
        if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1)) { s_abort = 1; break; }
        if (s_abort) break;
        const int kc = k0 + (i % su) * kSK;
        mbar_expect_tx(&full[s], kStageBytes);
        tma_load_2d(base + s * kStageBytes, &tq, kc >> 1, tile * kRows, &full[s]);
        issued = i + 1;
      }
      if (s_abort) {
        // copies still in flight land before the CTA's shared memory is released
        const int first = issued > kStages ? issued - kStages : 0;
        for (int i = first; i < issued; ++i) mbar_wait(&full[i % kStages], (i / kStages) & 1);
        const int sfirst = sissued > 2 ? sissued - 2 : 0;
        for (int u = sfirst; u < sissued; ++u) mbar_wait(&sfull[u & 1], (u >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issue
    if (lane == 0) {
      const uint32_t idesc = nf4tc_idesc<BN>();
      bool issued = false;
      if (!mbar_wait(&bready, 0)) s_abort = 1;
      for (int u = 0; u < my_units && !s_abort; ++u) {
        const int acc = u & 1;
        if (!mbar_wait(&tempty[acc], ((u >> 1) & 1) ^ 1)) { s_abort = 1; break; }
        tc_fence_after();
        const uint32_t d = tmem + kDcol0 + acc * BN;
        for (int j = 0; j < su; ++j) {
          const int i = u * su + j, a = i % kAbufs;
          if (!mbar_wait(&afull[a], (i / kAbufs) & 1)) { s_abort = 1; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kSK / 16; ++kk) {
            const int k = j * kSK + 16 * kk;     // K offset inside the unit
            const uint64_t bd = sw128_desc(bbase + (k >> 6) * Sh::kBoxBytes) + 2 * ((k & 63) >> 4);
            tc_mma_ta(d, tmem + a * kAcols + 8 * kk, bd, idesc, (j | kk) != 0);
          }
          tc_commit(&aempty[a]);
          issued = true;
        }
        if (s_abort) break;
        tc_commit(&tfull[acc]);
      }
      if (issued) {
        tc_commit(&done);
        if (!mbar_wait(&done, 0)) s_abort = 1;
      }
    }
    __syncwarp();
  } else if (warp < 10) {
    // ---------------- decoders: thread = weight row = tensor-memory lane
    const int dw = warp - 2, q = warp & 3, h = dw >> 2;
    const int r = 32 * q + lane;
    const int dt = dw * 32 + lane;               // 0..255
    pdl_wait();
    // activations of this CTA's K range -> f16 x * 2^t (t per column) in the
    // 128-byte swizzle layout (one 64-element box of BN rows per BN * 128
    // bytes); 8 elements (one 16-byte load) per item, columns past M zero
    {
      const int cpr = R >> 3;                    // items per column
      const int items = BN * cpr;
      for (int it = dt; it < items; it += 256) {
        const int m = it / cpr;
        if (m >= M) break;
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(X + m * ldx + k0 + 8 * (it - m * cpr)));
        float mx = 0.f;
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w4[e] << 16)), fabsf(__uint_as_float(w4[e] & 0xFFFF0000u))));
        if (mx > 0.f) atomicMax(&s_colmax[m], __float_as_uint(mx));
      }
      decoder_sync();
      for (int it = dt; it < items; it += 256) {
        const int m = it / cpr, c8 = it - m * cpr;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (m < M) {
          float sc, inv;
          pow2_into_f16_top(__uint_as_float(s_colmax[m]), sc, inv);
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(X + m * ldx + k0 + 8 * c8));
          o.x = pack_h2(__uint_as_float(v.x << 16) * sc, __uint_as_float(v.x & 0xFFFF0000u) * sc);
          o.y = pack_h2(__uint_as_float(v.y << 16) * sc, __uint_as_float(v.y & 0xFFFF0000u) * sc);
          o.z = pack_h2(__uint_as_float(v.z << 16) * sc, __uint_as_float(v.z & 0xFFFF0000u) * sc);
          o.w = pack_h2(__uint_as_float(v.w << 16) * sc, __uint_as_float(v.w & 0xFFFF0000u) * sc);
        }
        const int box = c8 >> 3, chunk = c8 & 7;
        *reinterpret_cast<uint4*>(gbase + (bbase - base) + box * Sh::kBoxBytes + m * 128 +
                                  ((chunk ^ (m & 7)) << 4)) = o;
      }
      if (dt < BN) {
        float sc, inv;
        pow2_into_f16_top(__uint_as_float(s_colmax[dt]), sc, inv);
        s_colinv[dt] = inv;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bready);
    }
    const float cbmax = s_cbmax;
    float rsc = 1.f;                             // this row's weight scale in the current unit
    for (int i = 0; i < total; ++i) {
      const int s = i % kStages, a = i % kAbufs;
      const int u = i / su, j = i % su, sb = u & 1;
      bool ok = mbar_wait(&full[s], (i / kStages) & 1);
      ok = ok && mbar_wait(&aempty[a], ((i / kAbufs) & 1) ^ 1);
      if (j == 0) ok = ok && mbar_wait(&sfull[sb], (u >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) { s_abort = 1; break; }
      if (s_abort) break;
      tc_fence_after();
      const float* arow = reinterpret_cast<const float*>(gbase + (sbase - base) + sb * kSBuf + r * (R >> 4));
      if (j == 0) {
        // the row's scale for this unit, from its largest |absmax|
        float amx = 0.f;
        for (int b = 0; b < (R >> 6); b += 4) {
          const float4 a4 = *reinterpret_cast<const float4*>(arow + b);
          amx = fmaxf(amx, fmaxf(fmaxf(fabsf(a4.x), fabsf(a4.y)), fmaxf(fabsf(a4.z), fabsf(a4.w))));
        }
        float inv;
        pow2_into_f16_top(amx * cbmax, rsc, inv);
        if (h == 0) s_scl[u & (kSclSlots - 1)][r] = inv;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sclfull[u & (kSclSlots - 1)]);
      }
      const uint8_t* st = gbase + s * kStageBytes;
#pragma unroll
      for (int jb = 0; jb < 2; ++jb) {
        const int b = 2 * h + jb;                // block of the stage (64 codes, 32 bytes)
        const float ab = arow[4 * j + b] * rsc;  // exact: a power of two
        uint32_t pw[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) pw[e] = pack_h2(ab * s_cb[2 * e], ab * s_cb[2 * e + 1]);
        const Planes pl = planes_from_pairs(pw);
        const uint4 c0 = *reinterpret_cast<const uint4*>(st + 128 * r + (((2 * b) ^ (r & 7)) << 4));
        const uint4 c1 = *reinterpret_cast<const uint4*>(st + 128 * r + (((2 * b + 1) ^ (r & 7)) << 4));
        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t out[16];
#pragma unroll
          for (int wq = 0; wq < 4; ++wq) {
            uint32_t rr[4];
            decode_planes(words[4 * hf + wq], pl, rr);
            out[4 * wq] = rr[0];
            out[4 * wq + 1] = rr[1];
            out[4 * wq + 2] = rr[2];
            out[4 * wq + 3] = rr[3];
          }
          tmem_store16(tmem + (static_cast<uint32_t>(32 * q) << 16) + a * kAcols + 32 * b + 16 * hf, out);
        }
      }
      tmem_store_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&afull[a]);
        mbar_arrive(&empty[s]);
        if (j == su - 1) mbar_arrive(&sempty[sb]);
      }
    }
  } else {
    // ---------------- epilogue: tensor-memory lanes 32q..32q+31 belong to warp q (mod 4)
    const int q = warp & 3, lr = 32 * q + lane;
    pdl_wait();
    uint64_t mybest = 0;
    if (!__all_sync(0xffffffffu, mbar_wait(&bready, 0))) s_abort = 1;
    float cinv[BN];
#pragma unroll
    for (int c = 0; c < BN; ++c) cinv[c] = s_colinv[c];
    for (int u = 0; u < my_units && !s_abort; ++u) {
      const int acc = u & 1;
      bool ok = mbar_wait(&tfull[acc], (u >> 1) & 1);
      ok = ok && mbar_wait(&sclfull[u & (kSclSlots - 1)], (u / kSclSlots) & 1);
      if (!__all_sync(0xffffffffu, ok)) { s_abort = 1; break; }
      if (s_abort) break;
      tc_fence_after();
      float v[BN];
      tmem_load_row<BN>(tmem + (static_cast<uint32_t>(32 * q) << 16) + kDcol0 + acc * BN, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      const float rinv = s_scl[u & (kSclSlots - 1)][lr];
      const int tile = tile0 + u * tstep;
      const int row = tile * kRows + lr;
      if (S == 1) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const __nv_bfloat16 o = __float2bfloat16_rn(v[c] * rinv * cinv[c]);
          if (c < M && row < N) Y[static_cast<int64_t>(c) * N + row] = o;
          if (kArgmax) {
            uint64_t k = (c < M && row < N) ? argmax_key(__bfloat162float(o), static_cast<uint32_t>(row)) : 0ull;
            k = warp_max_u64(k);
            if (lane == c) mybest = k > mybest ? k : mybest;
          }
        }
      } else {
        float* pp = sk.partials + static_cast<int64_t>(split * ntiles + tile) * (BN * kRows) + lr;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c < M) __stcg(pp + c * kRows, v[c] * rinv * cinv[c]);
      }
    }
    if (S > 1) __threadfence();                 // partials before the arrivals below
    if (kArgmax) s_key[q][lane] = mybest;
  }

  __syncthreads();
  if (S > 1 && !s_abort) {
    // Split K: one arrival per unit; the CTA that completes a tile adds its
    // splits in split order over the tile's M x 128 outputs and rounds them
    // to bf16.  The partials are scratch (written before they are read).
    for (int u = threadIdx.x; u < my_units; u += kThreads) {
      const int tile = tile0 + u * tstep;
      const unsigned prev = atomicAdd(sk.counters + tile, 1u);
      const bool last = prev == static_cast<unsigned>(S) - 1u;
      if (last) sk.counters[tile] = 0u;
      s_lastu[u] = last ? 1 : 0;
    }
    __syncthreads();
    __threadfence();
    constexpr int kE = (BN * kRows + kThreads - 1) / kThreads;
    const int64_t sstride = static_cast<int64_t>(ntiles) * (BN * kRows);
    for (int u = 0; u < my_units; ++u) {
      if (!s_lastu[u]) continue;
      const int tile = tile0 + u * tstep;
      const float* pt = sk.partials + static_cast<int64_t>(tile) * (BN * kRows);
      float v[kE];
#pragma unroll
      for (int i = 0; i < kE; ++i) v[i] = 0.f;
      for (int sp0 = 0; sp0 < S; sp0 += 4) {
        float t[4][kE];
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int i = 0; i < kE; ++i) {
            const int e = threadIdx.x + i * kThreads;
            t[b][i] = (sp0 + b < S && e < M * kRows) ? __ldcg(pt + (sp0 + b) * sstride + e) : 0.f;
          }
#pragma unroll
        for (int b = 0; b < 4; ++b)
#pragma unroll
          for (int i = 0; i < kE; ++i) v[i] += t[b][i];
      }
#pragma unroll
      for (int i = 0; i < kE; ++i) {
        const int e = threadIdx.x + i * kThreads;
        const int c = e / kRows, row = tile * kRows + (e - c * kRows);
        if (e < M * kRows && row < N) {
          const __nv_bfloat16 o = __float2bfloat16_rn(v[i]);
          Y[static_cast<int64_t>(c) * N + row] = o;
          if (kArgmax)
            atomicMax(reinterpret_cast<unsigned long long*>(&s_kc[c]),
                      static_cast<unsigned long long>(argmax_key(__bfloat162float(o), static_cast<uint32_t>(row))));
        }
      }
    }
  }
  if (s_abort && threadIdx.x == 0 && err) atomicExch(err, kErrGemvWait);
  if (kArgmax) {
    __syncthreads();
    if (threadIdx.x < 32) {
      uint64_t k = s_kc[threadIdx.x];
      if (static_cast<int>(threadIdx.x) < BN)
        for (int w = 0; w < 4; ++w) k = s_key[w][threadIdx.x] > k ? s_key[w][threadIdx.x] : k;
      s_cta[threadIdx.x] = k;
    }
    __syncthreads();
    argmax_publish(s_cta, M, am, gridDim.x);
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---- host ------------------------------------------------------------------

// 2-D map over a row-major [rows][cols] matrix (row pitch `ld` bytes), boxes
// of box_cols x kRows elements.
bool make_map(CUtensorMap* map, CUtensorMapDataType type, const void* ptr, int64_t cols, int rows,
              int64_t ld, int box_cols, bool swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(kRows)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, type, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, bool kArgmax>
cudaError_t run_t(const uint8_t* qs, const float* absmax, const Codebook16& cb, const void* X,
                  int64_t ldx, int M, void* Y, int N, int K, const Nf4TcPlan& p, const SplitArgs& sk,
                  const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  CUtensorMap tq, ta;
  if (!make_map(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, qs, K / 2, N, K / 2, kSK / 2, true) ||
      !make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, absmax, K / 64, N, K / 16, p.range / 64, false))
    return cudaErrorNotSupported;
  auto kern = nf4_tc_kernel<BN, kArgmax>;
  const int smem = TcN<BN>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  info->grid_x = p.grid;
  info->block = kThreads;
  info->smem = smem;
  info->kernel = "nf4_tc";
  return launch_k(kern, dim3(p.grid), dim3(kThreads), smem, st, true, tq, ta, cb,
                  static_cast<const __nv_bfloat16*>(X), ldx, M, static_cast<__nv_bfloat16*>(Y), N, K,
                  p.range, p.splits, sk, am, error_word_ptr());
}

}  // namespace

// Work plan: the K range of a unit is the largest of 1024, 768, 512, 256
// elements that divides K; the grid is a multiple of the split count so
// each CTA keeps one K range (and converts its activations once).
Nf4TcPlan nf4_tc_plan(int M, int N, int K) {
  Nf4TcPlan p;
  if (M < 2 || M > WOBS_MAX_M || N < 1 || K < kSK || K % kSK) return p;
  const int cand[4] = {1024, 768, 512, 256};
  for (int c : cand)
    if (K % c == 0) { p.range = c; break; }
  p.splits = K / p.range;
  const int sms = device_sm_count();
  if (p.splits > sms) return Nf4TcPlan{};
  const int ntiles = (N + kRows - 1) / kRows;
  const int per_split = sms / p.splits;
  const int groups = ntiles < per_split ? ntiles : per_split;
  p.grid = groups * p.splits;
  if ((ntiles + groups - 1) / groups > kMaxUnits) return Nf4TcPlan{};
  p.ok = true;
  return p;
}

size_t nf4_tc_partial_bytes(int M, int N, int K) {
  const Nf4TcPlan p = nf4_tc_plan(M, N, K);
  if (!p.ok || p.splits <= 1) return 0;
  const int bn = M <= 16 ? 16 : 32;
  return static_cast<size_t>(p.splits) * ((N + kRows - 1) / kRows) * kRows * bn * sizeof(float);
}

cudaError_t launch_nf4_tc(const uint8_t* qs, const float* absmax, const Codebook16& cb, const void* X,
                          int64_t ldx, int M, void* Y, int N, int K, const SplitArgs& sk,
                          const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const Nf4TcPlan p = nf4_tc_plan(M, N, K);
  if (!p.ok || p.splits != sk.splits) return cudaErrorNotSupported;
  for (float v : cb.v)
    if (!std::isfinite(v)) return cudaErrorNotSupported;
  if (reinterpret_cast<uintptr_t>(qs) % 16 || reinterpret_cast<uintptr_t>(absmax) % 16 ||
      reinterpret_cast<uintptr_t>(X) % 16 || ldx % 8)
    return cudaErrorNotSupported;
  if (M <= 16)
    return am.out ? run_t<16, true>(qs, absmax, cb, X, ldx, M, Y, N, K, p, sk, am, st, info)
                  : run_t<16, false>(qs, absmax, cb, X, ldx, M, Y, N, K, p, sk, am, st, info);
  return am.out ? run_t<32, true>(qs, absmax, cb, X, ldx, M, Y, N, K, p, sk, am, st, info)
                : run_t<32, false>(qs, absmax, cb, X, ldx, M, Y, N, K, p, sk, am, st, info);
}

}  // namespace wobs
