// Dense fp16 / bf16 decode GEMV, y = W x, fp32 accumulation.
//
// batch1-cdna README, "02-gemv": one wavefront per output row, lanes strided
// across the row so each load instruction is one contiguous transaction,
// several independent accumulators so loads are issued as a batch, and
// 16-byte loads instead of 4.  The sm_103a version keeps those three
// mechanisms: one warp per row, lane-strided 16-byte chunks (a warp reads
// 512 contiguous bytes per instruction), U chunks per lane issued before
// any is consumed, L1-no-allocate / L2-evict-first hints on the weight
// stream, and a persistent grid with the rows spread evenly over all warps.
//
// Several activation columns (M > 1, up to 32): each lane owns one row and
// walks along K; the activation tile is staged in shared memory and read by
// broadcast, so every weight chunk is reused for all M columns from
// registers.  K is split over CTAs when the rows alone cannot fill the GPU;
// the last CTA of a row group adds the partial sums in a fixed order.
#include "common.cuh"
#include "tma.cuh"

namespace wobs {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;    // 16-byte chunks per lane per pipeline stage

// ------------------------------------------------------------- M = 1

// Each warp walks the (row, stage) sequence of its rows; a stage is kUnroll
// lane-strided 16-byte chunks of one row.  Two register stages: the loads of
// stage t+1 are in flight while stage t is consumed, across row boundaries.
// The first stage is issued before pdl_wait() (weights only), overlapping
// the previous kernel on the stream; x is read after it.
template <typename T>
struct DenseStage {
  uint4 w[kUnroll];
};

template <typename T>
__device__ __forceinline__ void dense_load_stage(DenseStage<T>& st, const T* __restrict__ W,
                                                 int64_t ldw, int row, int it, int nch, int lane,
                                                 uint64_t pol) {
  const uint4* wr = reinterpret_cast<const uint4*>(W + static_cast<int64_t>(row) * ldw);
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int c = it * (32 * kUnroll) + 32 * u + lane;
    st.w[u] = c < nch ? ld_stream16(wr + c, pol) : make_uint4(0u, 0u, 0u, 0u);
  }
}

template <typename T, typename TO>
__global__ void __launch_bounds__(kThreads) dense_m1_kernel(const T* __restrict__ W, int64_t ldw,
                                                             const T* __restrict__ x,
                                                             TO* __restrict__ y, int N, int K,
                                                             ArgmaxArgs am) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total_warps = gridDim.x * kWarps;
  const int wg = blockIdx.x * kWarps + warp;
  const int nch = K >> 3;  // 16-byte chunks per row
  const int n_it = (nch + 32 * kUnroll - 1) / (32 * kUnroll);
  const int rows_w = wg < N ? (N - 1 - wg) / total_warps + 1 : 0;
  const int T_ = rows_w * n_it;
  const uint64_t pol = l2_evict_first_policy();
  const uint4* xv = reinterpret_cast<const uint4*>(x);

  DenseStage<T> sa, sb;
  int lrow = wg, lit = 0;
  auto advance = [&](int& r, int& it) {
    if (++it == n_it) { it = 0; r += total_warps; }
  };
  if (T_ > 0) { dense_load_stage(sa, W, ldw, lrow, lit, nch, lane, pol); advance(lrow, lit); }
  pdl_launch_dependents();
  pdl_wait();

  int crow = wg, cit = 0;
  float acc0 = 0.f, acc1 = 0.f;
  uint64_t best = 0;
  auto consume = [&](const DenseStage<T>& st) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int c = cit * (32 * kUnroll) + 32 * u + lane;
      if (c < nch) {
        if (u & 1) acc1 = dot8x8<T>(st.w[u], ld_nc16(xv + c), acc1);
        else acc0 = dot8x8<T>(st.w[u], ld_nc16(xv + c), acc0);
      }
    }
    if (cit == n_it - 1) {
      const float s = warp_sum(acc0 + acc1);
      const TO out = from_float<TO>(s);
      if (lane == 0) y[crow] = out;
      if (am.out) {
        const uint64_t k = argmax_key(to_float(out), static_cast<uint32_t>(crow));
        best = k > best ? k : best;
      }
      acc0 = acc1 = 0.f;
    }
    advance(crow, cit);
  };
  for (int t = 0; t < T_; t += 2) {
    if (t + 1 < T_) { dense_load_stage(sb, W, ldw, lrow, lit, nch, lane, pol); advance(lrow, lit); }
    consume(sa);
    if (t + 1 < T_) {
      if (t + 2 < T_) { dense_load_stage(sa, W, ldw, lrow, lit, nch, lane, pol); advance(lrow, lit); }
      consume(sb);
    }
  }
  if (am.out) {
    __shared__ uint64_t s_best[kWarps];
    __shared__ uint64_t s_cta[1];
    if (lane == 0) s_best[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t b = 0;
      for (int i = 0; i < kWarps; ++i) b = s_best[i] > b ? s_best[i] : b;
      s_cta[0] = b;
    }
    __syncthreads();
    argmax_publish(s_cta, 1, am, gridDim.x);
  }
}

// ------------------------------------------- M = 1, cp.async staging

// The warp-per-row computation with the weight stream staged through
// shared memory by 16-byte asynchronous copies: each warp owns a ring of
// kRing 2048-byte row segments (128 lane-strided chunks), requested ahead
// (the first before pdl_wait) and refilled as they are consumed; the
// activation vector is copied to shared memory once per CTA after pdl_wait.
// 16 warps per CTA, two CTAs per SM.  Three slots (two segments in flight
// per warp) measured 22 % faster than two on the 4096² fp16 GEMV, where
// each warp streams one whole 8 KB row.
constexpr int kCpWarps = 16;
constexpr int kCpThreads = kCpWarps * 32;
constexpr int kSeg = 2048;
constexpr int kRing = 3;
constexpr int kRingBytes = kCpWarps * kRing * kSeg;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
               :: "r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

template <typename T, typename TO, bool kArgmax>
__global__ void __launch_bounds__(kCpThreads) dense_m1_cp_kernel(const T* __restrict__ W,
                                                                  int64_t ldw,
                                                                  const T* __restrict__ x,
                                                                  TO* __restrict__ y, int N, int K,
                                                                  ArgmaxArgs am) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint4* xs = reinterpret_cast<uint4*>(smem + kRingBytes);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int total_warps = gridDim.x * kCpWarps;
  // rows spread round-robin over the CTAs first, so every SM gets an
  // equal share even when there are fewer rows than warps
  const int wg = warp * gridDim.x + blockIdx.x;
  const int row_bytes = K * 2;
  const int nseg = (row_bytes + kSeg - 1) / kSeg;
  const int rows_w = wg < N ? (N - 1 - wg) / total_warps + 1 : 0;
  const int T_ = rows_w * nseg;
  uint8_t* myring = smem + warp * (kRing * kSeg);
  const uint8_t* wbase = reinterpret_cast<const uint8_t*>(W);

  int prow = wg, pseg = 0;
  auto issue = [&](int slot) {
    uint8_t* st = myring + slot * kSeg;
    const int off = pseg * kSeg;
    const int n = min(kSeg, row_bytes - off) / 16;
    const uint8_t* src = wbase + static_cast<int64_t>(prow) * ldw * 2 + off;
#pragma unroll
    for (int u = 0; u < kSeg / 16 / 32; ++u) {
      const int c = 32 * u + lane;
      if (c < n) cp_async16(st + 16 * c, src + 16 * c);
    }
    if (++pseg == nseg) { pseg = 0; prow += total_warps; }
  };
#pragma unroll
  for (int i = 0; i < kRing - 1; ++i) {
    if (i < T_) issue(i);
    cp_async_commit();
  }
  pdl_launch_dependents();
  pdl_wait();
  const uint4* xg = reinterpret_cast<const uint4*>(x);
  for (int c = threadIdx.x; c < (K >> 3); c += kCpThreads) xs[c] = ld_nc16(xg + c);
  __syncthreads();

  int crow = wg, cseg = 0;
  float acc0 = 0.f, acc1 = 0.f;
  uint64_t best = 0;
  for (int t = 0; t < T_; ++t) {
    // request segment t+kRing-1 (into the slot consumed last), then wait for segment t
    if (t + kRing - 1 < T_) issue((t + kRing - 1) % kRing);
    cp_async_commit();
    cp_async_wait<kRing - 1>();
    __syncwarp();
    const uint4* st = reinterpret_cast<const uint4*>(myring + (t % kRing) * kSeg);
    const int c0 = cseg * (kSeg / 16);
    const int n = min(kSeg, row_bytes - cseg * kSeg) / 16;
#pragma unroll
    for (int u = 0; u < kSeg / 16 / 32; ++u) {
      const int c = 32 * u + lane;
      if (c < n) {
        if (u & 1) acc1 = dot8x8<T>(st[c], xs[c0 + c], acc1);
        else acc0 = dot8x8<T>(st[c], xs[c0 + c], acc0);
      }
    }
    if (cseg == nseg - 1) {
      const float sum = warp_sum(acc0 + acc1);
      const TO out = from_float<TO>(sum);
      if (lane == 0) y[crow] = out;
      if (kArgmax) {
        const uint64_t k = argmax_key(to_float(out), static_cast<uint32_t>(crow));
        best = k > best ? k : best;
      }
      acc0 = acc1 = 0.f;
    }
    if (++cseg == nseg) { cseg = 0; crow += total_warps; }
    __syncwarp();
  }
  cp_async_wait<0>();
  if (kArgmax) {
    __shared__ uint64_t s_best[kCpWarps];
    __shared__ uint64_t s_cta[1];
    if (lane == 0) s_best[warp] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
      uint64_t b = 0;
      for (int i = 0; i < kCpWarps; ++i) b = s_best[i] > b ? s_best[i] : b;
      s_cta[0] = b;
    }
    __syncthreads();
    argmax_publish(s_cta, 1, am, gridDim.x);
  }
}

template <typename T, typename TO, bool kArgmax>
cudaError_t run_m1_cp_t(const void* W, int64_t ldw, const void* x, void* y, int N, int K,
                        const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const int smem = kRingBytes + K * 2;
  cudaError_t e = cudaFuncSetAttribute(dense_m1_cp_kernel<T, TO, kArgmax>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int grid = 2 * device_sm_count();
  if (grid > N) grid = N;
  info->grid_x = grid;
  info->block = kCpThreads;
  info->smem = smem;
  info->kernel = "dense_m1_cp";
  return launch_k(dense_m1_cp_kernel<T, TO, kArgmax>, dim3(grid), dim3(kCpThreads), smem, st, true,
                  static_cast<const T*>(W), ldw, static_cast<const T*>(x), static_cast<TO*>(y), N,
                  K, am);
}

template <typename T, typename TO>
cudaError_t run_m1_cp(const void* W, int64_t ldw, const void* x, void* y, int N, int K,
                      const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  return am.out ? run_m1_cp_t<T, TO, true>(W, ldw, x, y, N, K, am, st, info)
                : run_m1_cp_t<T, TO, false>(W, ldw, x, y, N, K, am, st, info);
}

// --------------------------------------------------------- M columns

// M > 1: tensor cores (mma.sync m16n8k16, fp32 accumulate).  Each warp owns
// 16 weight rows, a CTA 256 rows; the activation columns (padded to
// multiples of 8, one n-tile each) are the MMA's N side.  The contraction
// order inside an MMA is free, so k-slots are permuted to make every
// fragment one contiguous 16-byte piece: for each 32-element chunk, lane
// (g, t) takes elements 8t..8t+7 of weight rows g and g+8 and of activation
// column g; the first four feed MMA 0, the last four MMA 1.
//
// Weights: every lane streams its own two 16-byte pieces per chunk through
// a private ring of kWS slots in shared memory with cp.async (zero-filled
// past K), kWS-1 chunks ahead, across K-tile and row-tile boundaries; the
// first kWS-1 are requested before pdl_wait.  Activations: K tiles of 512
// elements per column, brought in by 1-D bulk copies (TMA) into two
// alternating buffers completed on mbarriers (waits are bounded), one tile
// ahead.  Outputs go straight from the accumulator fragments to memory (8
// consecutive rows per column = one 32-byte sector).  K is split over CTAs
// when the row tiles alone cannot fill the GPU.
constexpr int kMW = 16;
constexpr int kMThreads = kMW * 32;
constexpr int kMRows = kMW * 16;             // rows per CTA tile
constexpr int kWS = 8;                       // weight ring slots per lane (32 bytes each)
constexpr int kKT = 512;                     // activation K tile (elements)
constexpr int kXStride = kKT * 2 + 64;       // bytes per staged column (bank-conflict free)

template <typename T>
__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__half>(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                                 uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float* d, uint32_t a0, uint32_t a1,
                                                        uint32_t a2, uint32_t a3, uint32_t b0,
                                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <typename T, typename TO, int NT>
__global__ void __launch_bounds__(kMThreads, 1) dense_mma_kernel(const T* __restrict__ W, int64_t ldw,
                                                                  const T* __restrict__ X, int64_t ldx,
                                                                  int M, TO* __restrict__ Y, int N,
                                                                  int K, int kps, SplitArgs sk,
                                                                  ArgmaxArgs am, int* err) {
  extern __shared__ __align__(128) uint8_t smem[];
  constexpr int kXBuf = NT * 8 * kXStride;
  uint8_t* xbuf = smem;                                  // [2][NT*8][kXStride]
  uint8_t* wring = smem + 2 * kXBuf;                     // [warps][kWS][2 rows][32 lanes][16 B]
  __shared__ __align__(8) uint64_t xbar[2];
  __shared__ uint64_t s_cta[NT * 8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int s = blockIdx.y;
  const int k0 = s * kps;
  const int k1 = min(K, k0 + kps);
  const int nch = (k1 - k0 + 31) / 32;
  const int nkt = (k1 - k0 + kKT - 1) / kKT;
  const int ntiles = (N + kMRows - 1) / kMRows;
  const int my_tiles = static_cast<int>(blockIdx.x) < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  // lane-contiguous 16-byte pieces: the copies and the 128-bit reads of a
  // warp touch 512 contiguous bytes each, free of bank conflicts
  uint8_t* myw = wring + warp * (kWS * 1024) + lane * 16;

  int ptile = blockIdx.x, pch = 0;        // weight chunk producer cursor
  auto wissue = [&](int slot) {
    const int r0 = ptile * kMRows + warp * 16;
    const int ra = min(r0 + g, N - 1), rb = min(r0 + g + 8, N - 1);
    const int e = k0 + 32 * pch + 8 * t;
    const bool v = e < k1;
    const T* pa = W + static_cast<int64_t>(ra) * ldw + (v ? e : 0);
    const T* pb = W + static_cast<int64_t>(rb) * ldw + (v ? e : 0);
    cp_async16_zfill(myw + slot * 1024, pa, v);
    cp_async16_zfill(myw + slot * 1024 + 512, pb, v);
    if (++pch == nch) { pch = 0; ptile += gridDim.x; }
  };
  const int TW = my_tiles * nch;
#pragma unroll
  for (int i = 0; i < kWS - 1; ++i) {
    if (i < TW) wissue(i);
    cp_async_commit_group();
  }
  for (int i = tid; i < 2 * kXBuf / 16; i += kMThreads)
    reinterpret_cast<uint4*>(xbuf)[i] = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    mbar_fence_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait();

  const int TX = my_tiles * nkt;
  auto xissue = [&](int q) {              // thread 0: activation tile q into buffer q & 1
    const int kb = k0 + (q % nkt) * kKT;
    const int kn = min(kKT, k1 - kb);
    uint64_t* bar = &xbar[q & 1];
    uint8_t* dst = xbuf + (q & 1) * kXBuf;
    mbar_expect_tx(bar, static_cast<uint32_t>(M * kn * 2));
    for (int col = 0; col < M; ++col)
      bulk_g2s(dst + col * kXStride, X + static_cast<int64_t>(col) * ldx + kb, kn * 2, bar);
  };
  if (tid == 0) {
    if (TX > 0) xissue(0);
    if (TX > 1) xissue(1);
  }

  bool ok = true;
  int q = 0, wi = 0;
  for (int j = 0; j < my_tiles; ++j) {
    const int tile = blockIdx.x + j * gridDim.x;
    float d[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) d[n][0] = d[n][1] = d[n][2] = d[n][3] = 0.f;
    for (int kt = 0; kt < nkt; ++kt, ++q) {
      if (ok) ok = mbar_wait(&xbar[q & 1], static_cast<uint32_t>((q >> 1) & 1));
      const uint8_t* xs = xbuf + (q & 1) * kXBuf + g * kXStride + 16 * t;
      const int kc = (min(kKT, k1 - k0 - kt * kKT) + 31) / 32;
      for (int cc = 0; cc < kc; ++cc, ++wi) {
        if (wi + kWS - 1 < TW) wissue((wi + kWS - 1) % kWS);
        cp_async_commit_group();
        cp_async_wait_group<kWS - 1>();
        const uint8_t* wsl = myw + (wi % kWS) * 1024;
        const uint4 a = *reinterpret_cast<const uint4*>(wsl);
        const uint4 b = *reinterpret_cast<const uint4*>(wsl + 512);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xs + n * 8 * kXStride + 64 * cc);
          mma16816<T>(d[n], a.x, b.x, a.y, b.y, xv.x, xv.y);
          mma16816<T>(d[n], a.z, b.z, a.w, b.w, xv.z, xv.w);
        }
      }
      __syncthreads();                     // everyone is done with buffer q & 1
      if (tid == 0 && q + 2 < TX) {
        fence_proxy_async_smem();
        xissue(q + 2);
      }
    }
    // outputs of this tile, straight from the fragments
    const int rbase = tile * kMRows;
    const int rg = rbase + warp * 16 + g;
    bool finish = true;
    if (sk.splits > 1) {
      // fragment order: one coalesced 512-byte store per n8 tile
      const int64_t fbase = ((static_cast<int64_t>(s) * ntiles + tile) * kMW + warp) * (NT * 32) + lane;
      float4* pp = reinterpret_cast<float4*>(sk.partials);
#pragma unroll
      for (int n = 0; n < NT; ++n) __stcg(pp + fbase + n * 32, make_float4(d[n][0], d[n][1], d[n][2], d[n][3]));
      finish = splitk_arrive_last(sk.counters, tile, sk.splits);
      if (finish) {
#pragma unroll
        for (int n = 0; n < NT; ++n) d[n][0] = d[n][1] = d[n][2] = d[n][3] = 0.f;
        // splits added in order, several loaded together
        constexpr int kB = 16 / NT;
        const int64_t tstride = static_cast<int64_t>(ntiles) * kMW * NT * 32;
        const int64_t f0 = (static_cast<int64_t>(tile) * kMW + warp) * (NT * 32) + lane;
        for (int sp0 = 0; sp0 < sk.splits; sp0 += kB) {
          float4 v[kB][NT];
#pragma unroll
          for (int b = 0; b < kB; ++b)
#pragma unroll
            for (int n = 0; n < NT; ++n)
              v[b][n] = sp0 + b < sk.splits ? __ldcg(pp + (sp0 + b) * tstride + f0 + n * 32)
                                             : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int b = 0; b < kB; ++b)
#pragma unroll
            for (int n = 0; n < NT; ++n) {
              d[n][0] += v[b][n].x; d[n][1] += v[b][n].y; d[n][2] += v[b][n].z; d[n][3] += v[b][n].w;
            }
        }
        // the partials are scratch (past the counter region): not cleared
      }
    }
    if (finish) {
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const int col = n * 8 + 2 * t + (h & 1), row = rg + 8 * (h >> 1);
          if (col < M && row < N) Y[static_cast<int64_t>(col) * N + row] = from_float<TO>(d[n][h]);
        }
      if (am.out) {
        __syncthreads();                   // this tile's outputs are written
        for (int col = warp; col < M; col += kMW) {
          uint64_t k = 0;
          for (int rl = lane; rl < kMRows; rl += 32) {
            const int row = rbase + rl;
            if (row < N) {
              const uint64_t kk = argmax_key(to_float(Y[static_cast<int64_t>(col) * N + row]),
                                             static_cast<uint32_t>(row));
              k = kk > k ? kk : k;
            }
          }
          k = warp_max_u64(k);
          if (lane == 0) s_cta[col] = k;
        }
        __syncthreads();
        argmax_publish(s_cta, M, am, ntiles);
      }
    }
  }
  cp_async_wait_group<0>();
  if (!ok && err) atomicExch(err, kErrGemvWait);
}

template <typename T, typename TO, int NT>
cudaError_t run_mma(const void* W, int64_t ldw, const void* X, int64_t ldx, int M, void* Y, int N,
                    int K, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                    Launch* info) {
  // K range per split: a multiple of the activation tile
  const int kps = (((K + sk.splits - 1) / sk.splits) + kKT - 1) / kKT * kKT;
  const int splits = (K + kps - 1) / kps;
  const int ntiles = (N + kMRows - 1) / kMRows;
  const int smem = 2 * NT * 8 * kXStride + kMThreads * kWS * 32;
  cudaError_t e = cudaFuncSetAttribute(dense_mma_kernel<T, TO, NT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int gx = device_sm_count();
  if (splits > 1 || gx > ntiles) gx = ntiles;   // split-K: one CTA per (tile, split)
  SplitArgs s2 = sk;
  s2.splits = splits;
  info->grid_x = gx;
  info->grid_y = splits;
  info->block = kMThreads;
  info->smem = smem;
  info->kernel = "dense_mma";
  return launch_k(dense_mma_kernel<T, TO, NT>, dim3(gx, splits), dim3(kMThreads), smem, st, true,
                  static_cast<const T*>(W), ldw, static_cast<const T*>(X), ldx, M,
                  static_cast<TO*>(Y), N, K, kps, s2, am, error_word_ptr());
}

template <typename T, typename TO>
cudaError_t dispatch_mn(const void* W, int64_t ldw, const void* X, int64_t ldx, int M, void* Y,
                        int N, int K, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                        Launch* info) {
  if (M <= 8) return run_mma<T, TO, 1>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  if (M <= 16) return run_mma<T, TO, 2>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  if (M <= 24) return run_mma<T, TO, 3>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  return run_mma<T, TO, 4>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
}

template <typename T, typename TO>
cudaError_t run_m1(const void* W, int64_t ldw, const void* x, void* y, int N, int K,
                   const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const void* fn = reinterpret_cast<const void*>(dense_m1_kernel<T, TO>);
  const int per_sm = max_resident_ctas(fn, kThreads, 0);
  int grid = device_sm_count() * (per_sm > 0 ? per_sm : 1);
  const int need = (N + kWarps - 1) / kWarps;
  if (grid > need) grid = need;
  info->grid_x = grid;
  info->block = kThreads;
  info->kernel = "dense_m1";
  return launch_k(dense_m1_kernel<T, TO>, dim3(grid), dim3(kThreads), 0, st, true,
                  static_cast<const T*>(W), ldw, static_cast<const T*>(x), static_cast<TO*>(y), N,
                  K, am);
}

}  // namespace

cudaError_t launch_gemv_dense(int dtype, const void* W, int64_t ldw, const void* X, int64_t ldx,
                              int M, void* Y, int out_f32, int N, int K, const SplitArgs& sk,
                              const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  const bool m1 = (M == 1 && sk.splits <= 1);
  // tensor-core streaming kernel: any column count, as long as its 128-row
  // tiles alone fill the GPU (it has no K split)
  if (sk.splits <= 1 && dense_tc_enabled() && (M >= 2 || (N + 127) / 128 >= device_sm_count())) {
    const cudaError_t e = launch_gemv_dense_tc(dtype, W, ldw, X, ldx, M, Y, N, K, am, st, info);
    if (e != cudaErrorNotSupported) return e;
    cudaGetLastError();
  }
  // asynchronous copies: 16-byte aligned rows (checked by the caller), x in smem
  const bool cp = m1 && !m1_ldg_forced() && (kRingBytes + K * 2 <= 200 * 1024);
  if (dtype == 0) {
    if (out_f32) return cudaErrorInvalidValue;
    if (cp) return run_m1_cp<__half, __half>(W, ldw, X, Y, N, K, am, st, info);
    return m1 ? run_m1<__half, __half>(W, ldw, X, Y, N, K, am, st, info)
              : dispatch_mn<__half, __half>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
  }
  if (!out_f32) return cudaErrorInvalidValue;
  if (cp) return run_m1_cp<__nv_bfloat16, float>(W, ldw, X, Y, N, K, am, st, info);
  return m1 ? run_m1<__nv_bfloat16, float>(W, ldw, X, Y, N, K, am, st, info)
            : dispatch_mn<__nv_bfloat16, float>(W, ldw, X, ldx, M, Y, N, K, sk, am, st, info);
}

}  // namespace wobs
