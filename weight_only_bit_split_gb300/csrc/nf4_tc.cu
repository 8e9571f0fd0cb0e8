// NF4 blockwise 4-bit GEMV for 2..32 activation columns on the fifth-
// generation tensor cores (tcgen05), codes decoded into tensor memory.
//
// bitsandbytes issue #1842 ("70B 4-bit LLM decode bottlenecked by HIP
// kernel..."): the fused 4-bit GEMV y = W x with NF4 weights (64-element
// blocks, an fp32 absmax each, codes indexing a 16-entry codebook) against
// dequantising the whole matrix first.  With several activation columns the
// code lookups are shared by every column; here the multiply-adds go to the
// tensor cores, each code is decoded once, and the absmax is applied in
// fp32 as the format defines the product:
//
//   * weights: the code c becomes the f16 value codebook[c] * 2^g, g one
//     power of two for the whole codebook that puts its largest magnitude in
//     [2^14, 2^15) (each level then within 2^-11 of its exact value); a code
//     byte (two codes) is looked up in a 256-entry table of f16 pairs in
//     shared memory, laid out so lane l always reads bank l, or, for some of
//     the code words, by byte permutes of register planes;
//   * activations: bf16 values times a power of two per column (max |x| of
//     the column over the CTA's K range into [2^14, 2^15)), exact in f16;
//   * every 64-element block gets its own fp32 accumulator in tensor memory
//     (tcgen05.mma kind::f16, M = 128 rows, N = 16 or 32 columns, four
//     K = 16 steps per block); the epilogue adds absmax[n][b] * D_b in fp32,
//     block by block, and takes both powers of two out exactly.
// The weights' only rounding is the codebook's to f16, the activations are
// exact, so each product is within 2^-11 of |w_i x_i|, inside the GEMV
// tolerance of 1e-3 * sum |w_i x_i|; y is rounded to bf16.
//
// Pipeline (one CTA per SM, warp-specialised):
//   * warp 0, one thread: 2-D TMA copies of 128 rows x 256 codes (128-byte
//     swizzle) into a ring of shared-memory stages, and of each unit's absmax
//     (128 rows x R / 64 floats) into one of two buffers;
//   * warps 2..9: each thread owns one weight row (its tensor-memory lane)
//     and two of a stage's four blocks, decoded into tensor memory (A
//     buffers of 256 K);
//   * warp 1, one thread: tcgen05.mma with A from tensor memory and B (the
//     activations of the CTA's K range, converted once, 128-byte swizzle)
//     from shared memory, into four block accumulators per stage (two sets);
//   * warps 10..13: per stage read the four block accumulators (one row per
//     thread), add them times their absmax into registers; per unit remove
//     the scales and write bf16 y or fp32 split-K partials, fold the argmax.
// Work units are (128-row tile, K range); every CTA keeps one K range.
// Split K ranges are added in split order by the CTA that completes a tile.
// The lookup table sits at a fixed shared-window address (0x10000), so a
// lookup address is one byte permute and one shift of the code word; stages
// are placed below and above it.  Every wait is bounded: on expiry the CTA
// records the error word and stops.
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
constexpr int kTmemCols = 512;
constexpr int kMaxStages = 8;
constexpr uint32_t kTabAddr = 0x10000;           // shared-window address of the lookup table
constexpr int kTabBytes = 256 * 128;             // entry e: 32 lane words at e * 128
constexpr int kAbsBytes = kRows * 16;            // a stage's absmax: 4 floats per row
constexpr int kSlotBytes = kStageBytes + kAbsBytes;   // codes, then absmax (18 KB)

static_assert(kStageBytes % 1024 == 0 && kSlotBytes % 1024 == 0,
              "stages keep the 1024-byte swizzle alignment");

template <int BN>
struct TcN {
  static constexpr int kAbufs = BN <= 16 ? 3 : 2;       // A buffers beside 2 x 4 block accumulators
  static constexpr int kDcol0 = kAbufs * kAcols;        // first accumulator column
  static constexpr int kMaxR = BN <= 16 ? 2048 : 1024;  // longest K range (a 64 KB activation tile)
  static constexpr int kBoxBytes = BN * 128;            // one 64-element K box of B
  static constexpr int kBBytes = (kMaxR / 64) * kBoxBytes;
  static_assert(kDcol0 + 2 * 4 * BN <= kTmemCols, "tensor memory");
};

// Shared-memory placement around the table at kTabAddr: stages below it, the
// activation tile and more stages above it (stage slot s at lo0 + s *
// kSlotBytes for s < nlo, else hi0 + (s - nlo) * kSlotBytes).
struct Layout {
  uint32_t bt, lo0, hi0;
  int nlo, ns;
};
template <int BN>
__device__ __forceinline__ Layout make_layout(uint32_t base, uint32_t bytes) {
  using Sh = TcN<BN>;
  Layout L;
  const uint32_t end = base + bytes;
  L.lo0 = (base + 1023u) & ~1023u;
  L.bt = kTabAddr + kTabBytes;
  L.hi0 = L.bt + Sh::kBBytes;
  if (L.lo0 > kTabAddr || L.hi0 > end) { L.nlo = 0; L.ns = -1; return L; }
  L.nlo = static_cast<int>((kTabAddr - L.lo0) / kSlotBytes);
  if (L.nlo > kMaxStages) L.nlo = kMaxStages;
  const int nhi = static_cast<int>((end - L.hi0) / kSlotBytes);
  L.ns = L.nlo + nhi < kMaxStages ? L.nlo + nhi : kMaxStages;
  return L;
}
__device__ __forceinline__ uint32_t slot_addr(const Layout& L, int s) {
  return s < L.nlo ? L.lo0 + s * kSlotBytes : L.hi0 + (s - L.nlo) * kSlotBytes;
}

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
__device__ __forceinline__ void epilogue_sync() {
  asm volatile("bar.sync 2, 128;" ::: "memory");
}

// Shared load as a pure function of its address (free to interleave).
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// One code word (byte j = element 2j in the high nibble, 2j + 1 in the low)
// -> four f16 pairs through the table: `tl` = 0x20000 | lane << 3, so the
// byte permute gives 0x20000 | byte << 8 | lane << 3 and the shift the
// table word kTabAddr + byte * 128 + lane * 4 (lane l reads bank l).
__device__ __forceinline__ void decode_table(uint32_t w, uint32_t tl, uint32_t (&r)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) r[j] = lds32(prmt(w, tl, 0x7604u | (j << 4)) >> 1);
}

template <int BN, int P, bool kArgmax>
__global__ void __launch_bounds__(kThreads, 1) nf4_tc_kernel(const __grid_constant__ CUtensorMap tq,
                                                             const __grid_constant__ CUtensorMap ta,
                                                             Codebook16 cb, float cb_scale, float cb_inv,
                                                             const __nv_bfloat16* __restrict__ X,
                                                             int64_t ldx, int M,
                                                             __nv_bfloat16* __restrict__ Y, int N,
                                                             int K, int R, int S, uint32_t smem_bytes,
                                                             SplitArgs sk, ArgmaxArgs am, int* err) {
  using Sh = TcN<BN>;
  constexpr int kAbufs = Sh::kAbufs;
  constexpr int kDcol0 = Sh::kDcol0;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], afull[kAbufs], aempty[kAbufs],
      dfull[2], dempty[2], bready, done;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_last;                         // the epilogue's unit completed its tile
  __shared__ volatile int s_evote[2];            // epilogue warps' abort vote, per step parity
  __shared__ uint16_t s_cbh[16];                 // codebook * 2^g in f16
  __shared__ unsigned s_colmax[32];              // max |x| per column (float bits)
  __shared__ float s_colinv[32];                 // per column: 2^-t of the activations
  __shared__ uint64_t s_key[4][32];
  __shared__ uint64_t s_cta[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = smem_addr(smem_raw);
  const Layout L = make_layout<BN>(base, smem_bytes);
  auto gen = [&](uint32_t a) { return smem_raw + (a - base); };   // generic view
  const int ntiles = (N + kRows - 1) / kRows;
  const int split = static_cast<int>(blockIdx.x) % S;
  const int tile0 = static_cast<int>(blockIdx.x) / S, tstep = static_cast<int>(gridDim.x) / S;
  const int my_units = tile0 < ntiles ? (ntiles - 1 - tile0) / tstep + 1 : 0;
  const int su = R / kSK;                        // stages per unit
  const int total = my_units * su;
  const int k0 = split * R;                      // this CTA's K range [k0, k0 + R)
  if (L.ns < 2) {                                // the table cannot sit at kTabAddr: refuse
    if (threadIdx.x == 0 && err) atomicExch(err, kErrGemvWait);
    return;
  }
  const int NS = L.ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 12);                  // 8 decoder warps (codes), 4 epilogue warps (absmax)
    }
    for (int a = 0; a < kAbufs; ++a) {
      mbar_init(&afull[a], 8);
      mbar_init(&aempty[a], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&dfull[a], 1);
      mbar_init(&dempty[a], 4);
    }
    mbar_init(&bready, 8);
    mbar_init(&done, 1);
    s_abort = 0;
    s_evote[0] = s_evote[1] = 0;
    for (int c = 0; c < 16; ++c) s_cbh[c] = __half_as_ushort(__float2half_rn(cb.v[c] * cb_scale));
    for (int c = 0; c < 32; ++c) {
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
      int issued = 0;
      for (int i = 0; i < total; ++i) {
        const int s = i % NS;
        const int u = i / su, tile = tile0 + u * tstep;
        if (i >= NS && !mbar_wait(&empty[s], ((i / NS) & 1) ^ 1)) { s_abort = 1; break; }
        if (s_abort) break;
        const int kc = k0 + (i % su) * kSK;
        const uint32_t sa = slot_addr(L, s);
        mbar_expect_tx(&full[s], kSlotBytes);
        tma_load_2d(sa, &tq, kc >> 1, tile * kRows, &full[s]);
        tma_load_2d(sa + kStageBytes, &ta, kc >> 6, tile * kRows, &full[s]);
        issued = i + 1;
      }
      if (s_abort) {
        // copies still in flight land before the CTA's shared memory is released
        const int first = issued > NS ? issued - NS : 0;
        for (int i = first; i < issued; ++i) mbar_wait(&full[i % NS], (i / NS) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issue: per stage, four 64-element blocks into
    // their own accumulators (four K = 16 steps each)
    if (lane == 0) {
      const uint32_t idesc = nf4tc_idesc<BN>();
      bool issued = false;
      if (!mbar_wait(&bready, 0)) s_abort = 1;
      for (int i = 0; i < total && !s_abort; ++i) {
        const int a = i % kAbufs, db = i & 1, j = i % su;
        if (!mbar_wait(&dempty[db], ((i >> 1) & 1) ^ 1)) { s_abort = 1; break; }
        if (!mbar_wait(&afull[a], (i / kAbufs) & 1)) { s_abort = 1; break; }
        tc_fence_after();
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const uint32_t d = tmem + kDcol0 + (db * 4 + b) * BN;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const int k = j * kSK + 64 * b + 16 * kk;     // K offset inside the unit
            const uint64_t bd = sw128_desc(L.bt + (k >> 6) * Sh::kBoxBytes) + 2 * kk;
            tc_mma_ta(d, tmem + a * kAcols + 32 * b + 8 * kk, bd, idesc, kk != 0);
          }
        }
        tc_commit(&aempty[a]);
        tc_commit(&dfull[db]);
        issued = true;
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
    // the lookup table (entry e: f16 pair of levels e >> 4, e & 15, in every
    // lane's word) and the register planes
    for (int i = dt; i < 256 * 32; i += 256) {
      const int e = i >> 5;
      asm volatile("st.shared.b32 [%0], %1;"
                   :: "r"(kTabAddr + e * 128 + (i & 31) * 4),
                      "r"(static_cast<uint32_t>(s_cbh[e >> 4]) | (static_cast<uint32_t>(s_cbh[e & 15]) << 16))
                   : "memory");
    }
    uint32_t pw[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      pw[e] = static_cast<uint32_t>(s_cbh[2 * e]) | (static_cast<uint32_t>(s_cbh[2 * e + 1]) << 16);
    const Planes pl = planes_from_pairs(pw);
    const uint32_t tl = 0x20000u | (static_cast<uint32_t>(lane) << 3);
    pdl_wait();
    // activations of this CTA's K range -> f16 x * 2^t (t per column) in the
    // 128-byte swizzle layout (one 64-element box of BN rows per BN * 128
    // bytes); 8 elements (one 16-byte load) per item, every load of a thread
    // in flight at once, columns past M zero
    {
      const int cpr = R >> 3;                    // items per column
      constexpr int kIt = BN * Sh::kMaxR / 8 / 256;   // items per thread at the longest range
      const int items = BN * cpr;
      uint4 xv[kIt];
#pragma unroll
      for (int j = 0; j < kIt; ++j) {
        const int it = dt + 256 * j;
        const int m = it / cpr;
        xv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (it < items && m < M) xv[j] = __ldg(reinterpret_cast<const uint4*>(X + m * ldx + k0 + 8 * (it - m * cpr)));
      }
#pragma unroll
      for (int j = 0; j < kIt; ++j) {
        const int it = dt + 256 * j;
        const int m = it / cpr;
        if (it >= items || m >= M) continue;
        const uint32_t w4[4] = {xv[j].x, xv[j].y, xv[j].z, xv[j].w};
        float mx = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          mx = fmaxf(mx, fmaxf(fabsf(__uint_as_float(w4[e] << 16)), fabsf(__uint_as_float(w4[e] & 0xFFFF0000u))));
        if (mx > 0.f) atomicMax(&s_colmax[m], __float_as_uint(mx));
      }
      decoder_sync();                            // column maxima and the table complete
#pragma unroll
      for (int j = 0; j < kIt; ++j) {
        const int it = dt + 256 * j;
        if (it >= items) continue;
        const int m = it / cpr, c8 = it - m * cpr;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (m < M) {
          float sc, inv;
          pow2_into_f16_top(__uint_as_float(s_colmax[m]), sc, inv);
          const uint4 v = xv[j];
          o.x = pack_h2(__uint_as_float(v.x << 16) * sc, __uint_as_float(v.x & 0xFFFF0000u) * sc);
          o.y = pack_h2(__uint_as_float(v.y << 16) * sc, __uint_as_float(v.y & 0xFFFF0000u) * sc);
          o.z = pack_h2(__uint_as_float(v.z << 16) * sc, __uint_as_float(v.z & 0xFFFF0000u) * sc);
          o.w = pack_h2(__uint_as_float(v.w << 16) * sc, __uint_as_float(v.w & 0xFFFF0000u) * sc);
        }
        const int box = c8 >> 3, chunk = c8 & 7;
        *reinterpret_cast<uint4*>(gen(L.bt) + box * Sh::kBoxBytes + m * 128 + ((chunk ^ (m & 7)) << 4)) = o;
      }
      if (dt < BN) {
        float sc, inv;
        pow2_into_f16_top(__uint_as_float(s_colmax[dt]), sc, inv);
        s_colinv[dt] = inv * cb_inv;             // both scales of the product, removed together
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bready);
    }
    for (int i = 0; i < total; ++i) {
      const int s = i % NS, a = i % kAbufs;
      bool ok = mbar_wait(&full[s], (i / NS) & 1);
      ok = ok && mbar_wait(&aempty[a], ((i / kAbufs) & 1) ^ 1);
      if (!__all_sync(0xffffffffu, ok)) { s_abort = 1; break; }
      if (s_abort) break;
      tc_fence_after();
      const uint8_t* st = gen(slot_addr(L, s));
#pragma unroll
      for (int jb = 0; jb < 2; ++jb) {
        const int b = 2 * h + jb;                // block of the stage (64 codes, 32 bytes)
        const uint4 c0 = *reinterpret_cast<const uint4*>(st + 128 * r + (((2 * b) ^ (r & 7)) << 4));
        const uint4 c1 = *reinterpret_cast<const uint4*>(st + 128 * r + (((2 * b + 1) ^ (r & 7)) << 4));
        const uint32_t words[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t out[16];
#pragma unroll
          for (int wq = 0; wq < 4; ++wq) {
            uint32_t rr[4];
            // P of every 8 code words through the register planes, the rest
            // through the table
            if (4 * (2 * jb + hf) + wq >= 16 - 2 * P) decode_planes(words[4 * hf + wq], pl, rr);
            else decode_table(words[4 * hf + wq], tl, rr);
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
      }
    }
  } else {
    // ---------------- epilogue: tensor-memory lanes 32q..32q+31 belong to warp q (mod 4)
    const int q = warp & 3, lr = 32 * q + lane;
    pdl_wait();
    uint64_t mybest = 0;
    const bool ready = __all_sync(0xffffffffu, mbar_wait(&bready, 0));
    float cinv[BN], acc[BN];
#pragma unroll
    for (int c = 0; c < BN; ++c) {
      cinv[c] = s_colinv[c];
      acc[c] = 0.f;
    }
    const int64_t sstride = static_cast<int64_t>(ntiles) * (BN * kRows);
    for (int i = 0; i < total; ++i) {
      const int u = i / su, j = i % su, db = i & 1, s = i % NS;
      bool ok = ready && mbar_wait(&dfull[db], (i >> 1) & 1);
      ok = ok && mbar_wait(&full[s], (i / NS) & 1);      // the stage's absmax has landed
      // the four warps leave together (they meet at named barriers below):
      // a vote per step, in a slot that is not rewritten before every warp
      // has read it
      if (!__all_sync(0xffffffffu, ok) && lane == 0) s_evote[i & 1] = 1;
      epilogue_sync();
      if (s_evote[i & 1]) { s_abort = 1; break; }
      tc_fence_after();
      // this row's absmax of the stage's four blocks
      const float4 a4 = *reinterpret_cast<const float4*>(gen(slot_addr(L, s)) + kStageBytes + 16 * lr);
      const float ab[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float v[BN];
        tmem_load_row<BN>(tmem + (static_cast<uint32_t>(32 * q) << 16) + kDcol0 + (db * 4 + b) * BN, v);
#pragma unroll
        for (int c = 0; c < BN; ++c) acc[c] = fmaf(ab[b], v[c], acc[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&dempty[db]);
        mbar_arrive(&empty[s]);
      }
      if (j != su - 1) continue;
      const int tile = tile0 + u * tstep;
      const int row = tile * kRows + lr;
#pragma unroll
      for (int c = 0; c < BN; ++c) acc[c] *= cinv[c];
      bool emit = true;
      if (S > 1) {
        // split K: leave this range's partial, count the arrival; the CTA
        // that completes the tile adds the ranges in split order
        float* pt = sk.partials + static_cast<int64_t>(tile) * (BN * kRows) + lr;
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c < M) __stcg(pt + split * sstride + c * kRows, acc[c]);
        epilogue_sync();
        if (lr == 0) {
          __threadfence();
          const unsigned prev = atomicAdd(sk.counters + tile, 1u);
          s_last = prev == static_cast<unsigned>(S) - 1u;
          if (s_last) sk.counters[tile] = 0u;
        }
        epilogue_sync();
        emit = s_last != 0;
        if (emit) {
          __threadfence();
#pragma unroll
          for (int c = 0; c < BN; ++c) acc[c] = 0.f;
          constexpr int kG = BN <= 16 ? 4 : 2;    // splits whose loads are in flight together
          for (int sp0 = 0; sp0 < S; sp0 += kG) {
            float t[kG][BN];
#pragma unroll
            for (int g = 0; g < kG; ++g)
#pragma unroll
              for (int c = 0; c < BN; ++c)
                t[g][c] = (sp0 + g < S && c < M) ? __ldcg(pt + (sp0 + g) * sstride + c * kRows) : 0.f;
#pragma unroll
            for (int g = 0; g < kG; ++g)
#pragma unroll
              for (int c = 0; c < BN; ++c) acc[c] += t[g][c];
          }
        }
        epilogue_sync();                         // s_last is read before the next unit writes it
      }
      if (emit) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const __nv_bfloat16 o = __float2bfloat16_rn(acc[c]);
          if (c < M && row < N) Y[static_cast<int64_t>(c) * N + row] = o;
          if (kArgmax) {
            uint64_t k = (c < M && row < N) ? argmax_key(__bfloat162float(o), static_cast<uint32_t>(row)) : 0ull;
            k = warp_max_u64(k);
            if (lane == c) mybest = k > mybest ? k : mybest;
          }
        }
      }
#pragma unroll
      for (int c = 0; c < BN; ++c) acc[c] = 0.f;
    }
    if (kArgmax) s_key[q][lane] = mybest;
  }

  __syncthreads();
  if (s_abort && threadIdx.x == 0 && err) atomicExch(err, kErrGemvWait);
  if (kArgmax) {
    __syncthreads();
    if (threadIdx.x < 32) {
      uint64_t k = 0ull;
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

template <int BN, int P, bool kArgmax>
cudaError_t run_t(const uint8_t* qs, const float* absmax, const Codebook16& cb, float cb_scale,
                  float cb_inv, const void* X, int64_t ldx, int M, void* Y, int N, int K,
                  const Nf4TcPlan& p, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                  Launch* info) {
  CUtensorMap tq, ta;
  if (!make_map(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, qs, K / 2, N, K / 2, kSK / 2, true) ||
      !make_map(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, absmax, K / 64, N, K / 16, kSK / 64, false))
    return cudaErrorNotSupported;
  auto kern = nf4_tc_kernel<BN, P, kArgmax>;
  // all the opt-in shared memory the static part leaves (set up once; -1 if
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
  // the allocation must reach past the table and the activation tile above it
  if (smem < static_cast<int>(kTabAddr + kTabBytes + TcN<BN>::kBBytes + 2 * kSlotBytes)) {
    cudaGetLastError();
    return cudaErrorNotSupported;
  }
  info->grid_x = p.grid;
  info->block = kThreads;
  info->smem = smem;
  info->kernel = "nf4_tc";
  return launch_k(kern, dim3(p.grid), dim3(kThreads), smem, st, true, tq, ta, cb, cb_scale, cb_inv,
                  static_cast<const __nv_bfloat16*>(X), ldx, M, static_cast<__nv_bfloat16*>(Y), N, K,
                  p.range, p.splits, static_cast<uint32_t>(smem), sk, am, error_word_ptr());
}

template <int BN, bool kArgmax>
cudaError_t run_p(const uint8_t* qs, const float* absmax, const Codebook16& cb, float sc, float inv,
                  const void* X, int64_t ldx, int M, void* Y, int N, int K, const Nf4TcPlan& p,
                  const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  // code words per 8 decoded through the register planes instead of the
  // table (WOBS_NF4_P = 0..3 overrides the default, for measurements)
  const char* v = std::getenv("WOBS_NF4_P");
  const int pp = v ? std::atoi(v) : 1;
  if (pp == 0) return run_t<BN, 0, kArgmax>(qs, absmax, cb, sc, inv, X, ldx, M, Y, N, K, p, sk, am, st, info);
  if (pp == 2) return run_t<BN, 2, kArgmax>(qs, absmax, cb, sc, inv, X, ldx, M, Y, N, K, p, sk, am, st, info);
  if (pp == 3) return run_t<BN, 3, kArgmax>(qs, absmax, cb, sc, inv, X, ldx, M, Y, N, K, p, sk, am, st, info);
  return run_t<BN, 1, kArgmax>(qs, absmax, cb, sc, inv, X, ldx, M, Y, N, K, p, sk, am, st, info);
}

}  // namespace

// Work plan: the K range of a unit is the largest of 2048 (up to 16
// columns), 1024, 768, 512, 256 elements that divides K; the grid is a multiple of the split count so
// each CTA keeps one K range (and converts its activations once).
Nf4TcPlan nf4_tc_plan(int M, int N, int K) {
  Nf4TcPlan p;
  if (M < 2 || M > WOBS_MAX_M || N < 1 || K < kSK || K % kSK) return p;
  const int cand[5] = {2048, 1024, 768, 512, 256};
  const int rmax = M <= 16 ? TcN<16>::kMaxR : TcN<32>::kMaxR;
  for (int c : cand)
    if (c <= rmax && K % c == 0) { p.range = c; break; }
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
  float sc, inv;
  if (!nf4_codebook_scale(cb, &sc, &inv)) return cudaErrorNotSupported;
  if (reinterpret_cast<uintptr_t>(qs) % 16 || reinterpret_cast<uintptr_t>(absmax) % 16 ||
      reinterpret_cast<uintptr_t>(X) % 16 || ldx % 8)
    return cudaErrorNotSupported;
  if (M <= 16)
    return am.out ? run_p<16, true>(qs, absmax, cb, sc, inv, X, ldx, M, Y, N, K, p, sk, am, st, info)
                  : run_p<16, false>(qs, absmax, cb, sc, inv, X, ldx, M, Y, N, K, p, sk, am, st, info);
  return am.out ? run_p<32, true>(qs, absmax, cb, sc, inv, X, ldx, M, Y, N, K, p, sk, am, st, info)
                : run_p<32, false>(qs, absmax, cb, sc, inv, X, ldx, M, Y, N, K, p, sk, am, st, info);
}

}  // namespace wobs
