// Q4_0 weights x Q8_1 activations for 5..32 columns on the fifth-
// generation tensor cores (tcgen05), weights decoded into tensor memory.
//
// "The kernel that waited for itself" (m12-db-gemm case study), sections
// "The VALU floor" and "A step at sixteen columns": with many activation
// columns per weight block, the per-block integer dots and scaling, not
// the weight stream, set the time of a CUDA-core (or mma.sync) kernel.
// Here the block scales are folded into the operands, so one tensor-core
// accumulation runs over the whole K range of a tile:
//
//   * weights: each 4-bit code q of block b becomes the f16 value
//     (q - 8) * d4[n][b] (the small integer is exact, the product rounded
//     once to f16);
//   * activations: each Q8_1 code becomes d8[m][b] * q8 (exact in fp32,
//     rounded once to f16);
//   * y[m][n] = sum over K of the products, accumulated in fp32 by
//     tcgen05.mma (kind::f16, M = 128 rows, N = 16 or 32 columns).
// Each product is then within 2^-10 of its exact value relative to
// |w_i x_i|, inside the GEMV tolerance of 1e-3 * sum |w_i x_i|.
//
// Pipeline (one CTA per SM, warp-specialised):
//   * warp 0, one thread: 2-D TMA copies of 128 rows x 256 codes (128-byte
//     swizzle) into an 8-stage ring, and of the unit's scales (128 rows x
//     R / 32) into one of two scale buffers;
//   * warps 2..9: each thread owns one weight row (its tensor-memory lane);
//     it reads its codes and scales from the stage, decodes four blocks into
//     f16 pairs and stores them into tensor memory (three A buffers of 256 K);
//   * warp 1, one thread: tcgen05.mma with A read from tensor memory and B
//     (the activations, converted once per CTA for its K range into the
//     128-byte swizzle layout) from shared memory, fp32 accumulators in
//     tensor memory (two buffers);
//   * warps 10..13: read the accumulator (one row per thread), write y or
//     the split-K partials, fold the greedy argmax.
// Work units are (128-row tile, K range); every CTA keeps one K range, so
// its activation tile is converted once.  Split K ranges are added in split
// order by the CTA that finishes a tile last.  The K order inside each
// 32-block is permuted identically on both operands so that the decode is
// four mask-or operations per code word.  Every wait is bounded: on expiry
// the CTA records the error word and stops.
#include <cstdlib>
#include <cstring>

#include "../../include/wobs.h"
#include "common.cuh"
#include "tcgen05.cuh"

namespace wobs {
namespace {

constexpr int kRows = 128;                       // weight rows per tile (MMA M)
constexpr int kSK = 256;                         // K elements per TMA stage (8 blocks)
constexpr int kCodeBytes = kRows * kSK / 2;      // 16384
constexpr int kStageBytes = kCodeBytes;
constexpr int kMaxUnits = 256;                   // work units of one CTA at most
constexpr int kThreads = 448;                    // TMA, MMA, 8 decoder, 4 epilogue warps
constexpr int kAcols = kSK / 2;                  // tensor-memory columns of one A buffer
constexpr int kAbufs = 3;                        // A buffers in tensor memory
constexpr int kDcol0 = kAbufs * kAcols;          // first accumulator column
constexpr int kTmemCols = 512;

static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");

// The longest K range of a unit (its activation tile, BN x R f16, takes up
// to 64 KB), the copy ring depth and one unit's scales.  Ranges of 2048 for
// 16 columns were measured slower (8 columns: 13.8 / 21.5 us against
// 9.5 / 18.7 us on 4096^2 / 14336 x 4096): half the units, worse balance.
template <int BN>
struct TcQ {
  static constexpr int kMaxR = 1024;
  static constexpr int kStages = 8;
  static constexpr int kSBuf = kRows * (kMaxR / 16);   // fp16 per block and row
  static constexpr int kBoxBytes = BN * 128;     // one 64-element K box of B
  static constexpr int kBBytes = (kMaxR / 64) * kBoxBytes;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + 2 * kSBuf + kBBytes;
};

// kind::f16 instruction descriptor: f32 accumulator, f16 A and B, K-major,
// M = 128, N = BN.
template <int BN>
__device__ __forceinline__ uint32_t q4tc_idesc() {
  return (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(kRows >> 4) << 24);
}

__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t h2_mul(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Four code bytes of a block (bytes 4i..4i+3: elements 4i..4i+3 in the low
// nibbles, 4i+16..4i+19 in the high ones) -> four f16 pairs (q - 8) * d4 in
// the kernel's K order: (4i, 4i+2), (4i+16, 4i+18), (4i+1, 4i+3),
// (4i+17, 4i+19).  1024 + q is exact in f16 (q OR-ed into the mantissa of
// 1024), so is (1024 + q) - 1032; the multiply rounds once.
__device__ __forceinline__ void decode_word(uint32_t w, uint32_t dd, uint32_t* out) {
  const uint32_t kBias = 0x64086408u;          // 1032, 1032
  out[0] = h2_mul(h2_sub((w & 0x000F000Fu) | 0x64006400u, kBias), dd);
  out[1] = h2_mul(h2_sub(((w >> 4) & 0x000F000Fu) | 0x64006400u, kBias), dd);
  out[2] = h2_mul(h2_sub(((w >> 8) & 0x000F000Fu) | 0x64006400u, kBias), dd);
  out[3] = h2_mul(h2_sub(((w >> 12) & 0x000F000Fu) | 0x64006400u, kBias), dd);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int BN, bool kArgmax>
__global__ void __launch_bounds__(kThreads, 1) q4_tc_kernel(const __grid_constant__ CUtensorMap tq,
                                                            const __grid_constant__ CUtensorMap td,
                                                            const uint8_t* __restrict__ xq, int M,
                                                            float* __restrict__ Y, int N, int K, int R,
                                                            int S, SplitArgs sk, ArgmaxArgs am,
                                                            int* err) {
  using Sh = TcQ<BN>;
  constexpr int kStages = Sh::kStages;
  constexpr int kSBuf = Sh::kSBuf;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], afull[kAbufs], aempty[kAbufs], tfull[2],
      tempty[2], sfull[2], sempty[2], bready, done;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ unsigned char s_lastu[kMaxUnits];   // per unit: this CTA completed the tile
  __shared__ uint64_t s_key[4][32];
  __shared__ uint64_t s_kc[32];                 // split-K argmax keys per column
  __shared__ uint64_t s_cta[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t sbase = base + kStages * kStageBytes;     // two scale buffers
  const uint32_t bbase = sbase + 2 * kSBuf;               // activation tile
  uint8_t* const gbase = smem_raw + (base - smem_addr(smem_raw));   // generic view of `base`
  const int nb = K >> 5;
  const int ntiles = (N + kRows - 1) / kRows;
  const int split = static_cast<int>(blockIdx.x) % S;
  const int tile0 = static_cast<int>(blockIdx.x) / S, tstep = static_cast<int>(gridDim.x) / S;
  const int my_units = tile0 < ntiles ? (ntiles - 1 - tile0) / tstep + 1 : 0;
  const int su = R / kSK;                        // stages per unit
  const int total = my_units * su;
  const int kb0 = split * (R >> 5);              // first block of this CTA's K range

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
    mbar_init(&bready, 8);
    mbar_init(&done, 1);
    s_abort = 0;
    for (int c = 0; c < 32; ++c) {
      s_kc[c] = 0ull;
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
          // the unit's scales (the scale plane as bytes: block b at 2 b)
          const int sb = u & 1;
          if (u >= 2 && !mbar_wait(&sempty[sb], ((u >> 1) & 1) ^ 1)) { s_abort = 1; break; }
          mbar_expect_tx(&sfull[sb], kRows * (R >> 4));
          tma_load_2d(sbase + sb * kSBuf, &td, (split * R) >> 4, tile * kRows, &sfull[sb]);
          sissued = u + 1;
        }
        if (i >= kStages && !mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1)) { s_abort = 1; break; }
        if (s_abort) break;
        const int k0 = split * R + (i % su) * kSK;
        mbar_expect_tx(&full[s], kStageBytes);
        tma_load_2d(base + s * kStageBytes, &tq, k0 >> 1, tile * kRows, &full[s]);
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
      const uint32_t idesc = q4tc_idesc<BN>();
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
    pdl_wait();
    // activations of this CTA's K range -> f16 d8 * q8 in the 128-byte
    // swizzle layout (one 64-element box of BN rows per 4 KB), K order as
    // the weights'
    {
      // batches of eight items per thread: every load of a batch is issued
      // before any is used, so a batch costs one L2 round trip
      constexpr int kIt = 8;
      const int nbr = R >> 5;
      const int items = BN * nbr * 4;
      for (int it0 = 0; it0 < items; it0 += 256 * kIt) {
      uint32_t w[kIt][3];
#pragma unroll
      for (int j = 0; j < kIt; ++j) {
        const int it = it0 + dw * 32 + lane + 256 * j;
        const int m = it / (nbr * 4), rem = it - m * (nbr * 4);
        const int bl = rem >> 2, i = rem & 3;
        w[j][0] = w[j][1] = w[j][2] = 0u;
        if (it < items && m < M) {
          const uint32_t* blk =
              reinterpret_cast<const uint32_t*>(xq + (static_cast<int64_t>(m) * nb + kb0 + bl) * 36);
          w[j][0] = __ldg(blk);
          w[j][1] = __ldg(blk + 1 + i);
          w[j][2] = __ldg(blk + 5 + i);
        }
      }
#pragma unroll
      for (int j = 0; j < kIt; ++j) {
        const int it = it0 + dw * 32 + lane + 256 * j;
        if (it >= items) break;
        const int m = it / (nbr * 4), rem = it - m * (nbr * 4);
        const int bl = rem >> 2, i = rem & 3;
        const float d8 = __half2float(__ushort_as_half(static_cast<unsigned short>(w[j][0] & 0xFFFFu)));
        const uint32_t lo = w[j][1], hi = w[j][2];
        auto c = [](uint32_t v, int b) { return static_cast<float>(static_cast<int8_t>((v >> (8 * b)) & 0xFFu)); };
        uint4 v;
        v.x = pack_h2(d8 * c(lo, 0), d8 * c(lo, 2));
        v.y = pack_h2(d8 * c(hi, 0), d8 * c(hi, 2));
        v.z = pack_h2(d8 * c(lo, 1), d8 * c(lo, 3));
        v.w = pack_h2(d8 * c(hi, 1), d8 * c(hi, 3));
        const int chunk = 4 * (bl & 1) + i;
        *reinterpret_cast<uint4*>(gbase + (bbase - base) + (bl >> 1) * Sh::kBoxBytes + m * 128 +
                                  ((chunk ^ (m & 7)) << 4)) = v;
      }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bready);
    }
    for (int i = 0; i < total; ++i) {
      const int s = i % kStages, a = i % kAbufs;
      const int u = i / su, j = i % su, sb = u & 1;
      bool ok = mbar_wait(&full[s], (i / kStages) & 1);
      ok = ok && mbar_wait(&aempty[a], ((i / kAbufs) & 1) ^ 1);
      if (j == 0) ok = ok && mbar_wait(&sfull[sb], (u >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) { s_abort = 1; break; }
      if (s_abort) break;
      tc_fence_after();
      const uint8_t* st = gbase + s * kStageBytes;
      // this warp's four scales of stage j: blocks 8j + 4h .. 8j + 4h + 3 of
      // the unit, two fp16 per 32-bit word (rows R / 16 bytes apart)
      const uint2 sc = *reinterpret_cast<const uint2*>(gbase + (sbase - base) + sb * kSBuf +
                                                       r * (R >> 4) + 16 * j + 8 * h);
#pragma unroll
      for (int jb = 0; jb < 4; ++jb) {
        const int b = 4 * h + jb;
        const uint4 cw = *reinterpret_cast<const uint4*>(st + 128 * r + ((b ^ (r & 7)) << 4));
        const uint32_t sw = jb < 2 ? sc.x : sc.y;
        const uint32_t hw = (jb & 1) ? (sw >> 16) : (sw & 0xFFFFu);
        const uint32_t dd = hw | (hw << 16);
        uint32_t out[16];
        decode_word(cw.x, dd, out);
        decode_word(cw.y, dd, out + 4);
        decode_word(cw.z, dd, out + 8);
        decode_word(cw.w, dd, out + 12);
        tmem_store16(tmem + (static_cast<uint32_t>(32 * q) << 16) + a * kAcols + 16 * b, out);
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
    const int q = warp & 3, et = threadIdx.x - 320, lr = 32 * q + lane;
    pdl_wait();
    uint64_t mybest = 0;
    auto emit = [&](int tile, const float (&v)[BN]) {
      const int row = tile * kRows + lr;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        if (c < M && row < N) Y[static_cast<int64_t>(c) * N + row] = v[c];
        if (kArgmax) {
          uint64_t k = (c < M && row < N) ? argmax_key(v[c], static_cast<uint32_t>(row)) : 0ull;
          k = warp_max_u64(k);
          if (lane == c) mybest = k > mybest ? k : mybest;
        }
      }
    };
    for (int u = 0; u < my_units; ++u) {
      const int acc = u & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], (u >> 1) & 1));
      if (!ok) { s_abort = 1; break; }
      if (s_abort) break;
      tc_fence_after();
      float v[BN];
      tmem_load_row<BN>(tmem + (static_cast<uint32_t>(32 * q) << 16) + kDcol0 + acc * BN, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      const int tile = tile0 + u * tstep;
      if (S == 1) {
        emit(tile, v);
      } else {
        float* pp = sk.partials + static_cast<int64_t>(split * ntiles + tile) * (BN * kRows) + lr;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c < M) __stcg(pp + c * kRows, v[c]);
      }
    }
    if (S > 1) __threadfence();                 // partials before the arrivals below
    if (kArgmax) s_key[q][lane] = mybest;
  }

  __syncthreads();
  if (S > 1 && !s_abort) {
    // Split K: one arrival per unit; the CTA that completes a tile adds its
    // splits in split order, all 448 threads over the tile's M x 128
    // outputs (each with its splits' loads in flight).  The partials are
    // scratch (written before they are read, never taken for counters), so
    // they are not cleared.  s_abort no longer changes: every role is done.
    for (int u = threadIdx.x; u < my_units; u += kThreads) {
      const int tile = tile0 + u * tstep;
      const unsigned prev = atomicAdd(sk.counters + tile, 1u);
      const bool last = prev == static_cast<unsigned>(S) - 1u;
      if (last) sk.counters[tile] = 0u;
      s_lastu[u] = last ? 1 : 0;
    }
    __syncthreads();
    __threadfence();
    // per thread at most kE outputs of a tile; loads of four splits of all
    // of them are in flight together, then the outputs
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
          Y[static_cast<int64_t>(c) * N + row] = v[i];
          if (kArgmax)
            atomicMax(reinterpret_cast<unsigned long long*>(&s_kc[c]),
                      static_cast<unsigned long long>(argmax_key(v[i], static_cast<uint32_t>(row))));
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

bool make_map_u8(CUtensorMap* map, const void* ptr, int64_t row_bytes, int rows, int box_x,
                 bool swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_x), static_cast<cuuint32_t>(kRows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides,
                        box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, bool kArgmax>
cudaError_t run_t(const uint8_t* qs, const void* d, const void* xq, int M, float* Y, int N, int K,
                  const Q4TcPlan& p, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                  Launch* info) {
  CUtensorMap tq, td;
  if (!make_map_u8(&tq, qs, K / 2, N, kSK / 2, true) ||
      !make_map_u8(&td, d, K / 16, N, p.range / 16, false))
    return cudaErrorNotSupported;
  auto kern = q4_tc_kernel<BN, kArgmax>;
  const int smem = TcQ<BN>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  info->grid_x = p.grid;
  info->block = kThreads;
  info->smem = smem;
  info->kernel = "q4_0_q8_1_tc";
  return launch_k(kern, dim3(p.grid), dim3(kThreads), smem, st, true, tq, td,
                  static_cast<const uint8_t*>(xq), M, Y, N, K, p.range, p.splits, sk, am,
                  error_word_ptr());
}

}  // namespace

bool q4_tc_enabled() {
  const char* v = std::getenv("WOBS_Q4TC");
  return !(v && v[0] == '0');
}

bool q4_tc_forced() {
  const char* v = std::getenv("WOBS_Q4TC");
  return v && v[0] == '1';
}

// Work plan: the K range of a unit is the largest of 1024, 768, 512, 256
// elements that divides K; the grid is a multiple of the split count so
// each CTA keeps one K range.  By default the kernel takes 17 to 32 columns
// when the units can occupy at least half of the SMs.  Measured on GB300
// against the mma.sync kernel (4096 x 4096 / 14336 x 4096, us): 32 columns
// 10.9 / 20.9 against 16.4 / 29.0; 24 columns 10.7 / 20.2 against
// 12.8 / 22.8; 16 columns 9.2 / 17.8 against 9.8 / 17.2; 8 columns
// 8.8 / 17.3 against 7.5 / 13.7.  WOBS_Q4TC=1 takes it from 5 columns.
Q4TcPlan q4_tc_plan(int M, int N, int K) {
  Q4TcPlan p;
  if (M < 5 || M > WOBS_MAX_M || N < 1 || K < kSK || K % kSK) return p;
  const int cand[5] = {2048, 1024, 768, 512, 256};
  const int rmax = M <= 16 ? TcQ<16>::kMaxR : TcQ<32>::kMaxR;
  for (int c : cand)
    if (c <= rmax && K % c == 0) { p.range = c; break; }
  p.splits = K / p.range;
  const int sms = device_sm_count();
  if (p.splits > sms) return Q4TcPlan{};
  const int ntiles = (N + kRows - 1) / kRows;
  const int per_split = sms / p.splits;
  const int groups = ntiles < per_split ? ntiles : per_split;
  p.grid = groups * p.splits;
  if ((ntiles + groups - 1) / groups > kMaxUnits) return Q4TcPlan{};
  p.ok = q4_tc_forced() || (M > 16 && 2 * ntiles * p.splits >= sms);
  return p;
}

size_t q4_tc_partial_bytes(int M, int N, int K) {
  const Q4TcPlan p = q4_tc_plan(M, N, K);
  if (!p.ok || p.splits <= 1) return 0;
  const int bn = M <= 16 ? 16 : 32;
  return static_cast<size_t>(p.splits) * ((N + kRows - 1) / kRows) * kRows * bn * sizeof(float);
}

cudaError_t launch_q4_tc(const uint8_t* qs, const void* d, const void* xq, int M, float* Y, int N,
                         int K, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                         Launch* info) {
  const Q4TcPlan p = q4_tc_plan(M, N, K);
  if (!p.ok || p.splits != sk.splits) return cudaErrorInvalidValue;
  if (M <= 16)
    return am.out ? run_t<16, true>(qs, d, xq, M, Y, N, K, p, sk, am, st, info)
                  : run_t<16, false>(qs, d, xq, M, Y, N, K, p, sk, am, st, info);
  return am.out ? run_t<32, true>(qs, d, xq, M, Y, N, K, p, sk, am, st, info)
                : run_t<32, false>(qs, d, xq, M, Y, N, K, p, sk, am, st, info);
}

}  // namespace wobs
