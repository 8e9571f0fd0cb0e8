// Dense fp16 / bf16 GEMV for 2..32 activation columns on the fifth-
// generation tensor cores (tcgen05), weights streamed by the tensor-memory
// accelerator.
//
// batch1-cdna README, "02-gemv": the decode product y = W x reads every
// weight byte once, so the work is to keep HBM busy; with several columns
// (the lm-head of a small decode batch) the multiply-adds grow with the
// column count while the bytes do not.  This kernel gives the weights the
// shortest route from HBM to the multipliers:
//
//   * one thread (warp 0) streams 128-row x 64-element weight boxes and the
//     matching activation boxes with 2-D TMA copies (128-byte swizzle) into
//     an 8-stage shared-memory ring, completion counted by mbarriers;
//   * one thread (warp 1) issues tcgen05.mma (kind::f16, M = 128, N = 16 or
//     32, K = 16; four per stage) reading both operands straight from shared
//     memory through matrix descriptors, accumulating in tensor memory, and
//     releases each stage with tcgen05.commit;
//   * four warps read the 128 x N fp32 accumulator out of tensor memory
//     (one row per thread), store the outputs and fold them into the greedy
//     argmax; two accumulator buffers let this overlap the next tile's MMAs.
//
// Persistent grid (one CTA per SM) over 128-row tiles.  Rows past N, columns
// past M and the K tail are zero-filled by the copies.  Every wait is
// bounded: on expiry the CTA records the error word and stops issuing.
#include <cstdlib>
#include <type_traits>

#include "common.cuh"
#include "tcgen05.cuh"

namespace wobs {
namespace {

constexpr int kTcRows = 128;                 // weight rows per tile (MMA M)
constexpr int kTcK = 64;                     // K elements per stage: one 128-byte swizzle row
constexpr int kTcStages = 8;
constexpr int kTcABytes = kTcRows * kTcK * 2;
constexpr int kTcThreads = 192;              // copy warp, MMA warp, four epilogue warps

template <int BN>
struct TcShape {
  static constexpr int kBBytes = BN * kTcK * 2;
  static constexpr int kStage = kTcABytes + kBBytes;        // multiple of 1024
  static constexpr int kSmem = 1024 + kTcStages * kStage;   // + alignment slack
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
};

// Instruction descriptor, kind::f16: f32 accumulator, A and B of one type
// (0 = f16, 1 = bf16), both K-major, M = 128.
template <typename T, int BN>
__device__ __forceinline__ uint32_t tc_idesc() {
  constexpr uint32_t fmt = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(kTcRows >> 4) << 24);
}

// ---- kernel --------------------------------------------------------------

template <typename T, typename TO, int BN, bool kArgmax>
__global__ void __launch_bounds__(kTcThreads, 1) dense_tc_kernel(const __grid_constant__ CUtensorMap tw,
                                                                  const __grid_constant__ CUtensorMap tx,
                                                                  int M, TO* __restrict__ Y, int N, int K,
                                                                  ArgmaxArgs am, int* err) {
  using S = TcShape<BN>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kTcStages], empty[kTcStages], tfull[2], tempty[2], done;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ uint64_t s_key[4][32];
  __shared__ uint64_t s_cta[32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = (smem_addr(smem_raw) + 1023u) & ~1023u;
  const int ntiles = (N + kTcRows - 1) / kTcRows;
  const int nk = (K + kTcK - 1) / kTcK;
  const int my_tiles = static_cast<int>(blockIdx.x) < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(&done, 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(&s_tmem)), "r"(S::kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  pdl_launch_dependents();

  if (warp == 0) {
    // ---------------- copies
    if (lane == 0) {
      const int total = my_tiles * nk;
      const int pre = total < kTcStages ? total : kTcStages;
      // weight boxes of the first stages do not depend on the previous kernel
      for (int i = 0; i < pre; ++i) {
        const int tile = blockIdx.x + (i / nk) * gridDim.x;
        mbar_expect_tx(&full[i], S::kStage);
        tma_load_2d(base + i * S::kStage, &tw, (i % nk) * kTcK, tile * kTcRows, &full[i]);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i)
        tma_load_2d(base + i * S::kStage + kTcABytes, &tx, (i % nk) * kTcK, 0, &full[i]);
      int issued = pre;
      for (int i = pre; i < total; ++i) {
        const int s = i % kTcStages;
        if (!mbar_wait(&empty[s], ((i / kTcStages) & 1) ^ 1)) { s_abort = 1; break; }
        if (s_abort) break;
        const int tile = blockIdx.x + (i / nk) * gridDim.x;
        const int k0 = (i % nk) * kTcK;
        mbar_expect_tx(&full[s], S::kStage);
        tma_load_2d(base + s * S::kStage, &tw, k0, tile * kTcRows, &full[s]);
        tma_load_2d(base + s * S::kStage + kTcABytes, &tx, k0, 0, &full[s]);
        issued = i + 1;
      }
      if (s_abort) {
        // copies still in flight must land before the CTA's shared memory is
        // released: wait (bounded) for the last round of stages issued
        const int first = issued > kTcStages ? issued - kTcStages : 0;
        for (int i = first; i < issued; ++i) mbar_wait(&full[i % kTcStages], (i / kTcStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issue
    if (lane == 0) {
      const uint32_t idesc = tc_idesc<T, BN>();
      bool issued = false;
      for (int t = 0; t < my_tiles && !s_abort; ++t) {
        const int acc = t & 1;
        if (!mbar_wait(&tempty[acc], ((t >> 1) & 1) ^ 1)) { s_abort = 1; break; }
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        for (int kb = 0; kb < nk; ++kb) {
          const int i = t * nk + kb;
          const int s = i % kTcStages;
          if (!mbar_wait(&full[s], (i / kTcStages) & 1)) { s_abort = 1; break; }
          tc_fence_after();
          const uint32_t a0 = base + s * S::kStage;
          const uint64_t ad = sw128_desc(a0), bd = sw128_desc(a0 + kTcABytes);
#pragma unroll
          for (int kk = 0; kk < kTcK / 16; ++kk)   // +32 bytes along K: +2 in the address field
            tc_mma(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          tc_commit(&empty[s]);
          issued = true;
        }
        if (s_abort) break;
        tc_commit(&tfull[acc]);
      }
      // every issued MMA has finished before tensor memory is released
      if (issued) {
        tc_commit(&done);
        if (!mbar_wait(&done, 0)) s_abort = 1;
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: TMEM lanes 32q..32q+31 belong to warp q (mod 4)
    const int q = warp & 3;
    pdl_wait();
    uint64_t mybest = 0;
    for (int t = 0; t < my_tiles; ++t) {
      const int acc = t & 1;
      const bool ok = __all_sync(0xffffffffu, mbar_wait(&tfull[acc], (t >> 1) & 1));
      if (!ok) { s_abort = 1; break; }
      if (s_abort) break;
      tc_fence_after();
      float v[BN];
      tmem_load_row<BN>(tmem + (static_cast<uint32_t>(32 * q) << 16) + acc * BN, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      const int tile = blockIdx.x + t * gridDim.x;
      const int row = tile * kTcRows + 32 * q + lane;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        if (c < M && row < N) Y[static_cast<int64_t>(c) * N + row] = from_float<TO>(v[c]);
        if (kArgmax) {
          uint64_t k = (c < M && row < N) ? argmax_key(to_float(from_float<TO>(v[c])), static_cast<uint32_t>(row)) : 0ull;
          k = warp_max_u64(k);
          if (lane == c) mybest = k > mybest ? k : mybest;
        }
      }
    }
    if (kArgmax) s_key[q][lane] = mybest;
  }

  __syncthreads();
  if (s_abort && threadIdx.x == 0 && err) atomicExch(err, kErrGemvWait);
  if (kArgmax) {
    if (threadIdx.x < 32) {
      uint64_t k = 0;
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
                 :: "r"(tmem), "r"(S::kTmemCols) : "memory");
  }
}

// ---- host ------------------------------------------------------------------

// 2-D map over a row-major [rows][ld] matrix of 16-bit elements, K extent
// `cols`, boxes of 64 elements x `box_rows` rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, bool bf16, const void* ptr, int64_t ld, int cols, int rows,
              int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTcK), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                        const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename T, typename TO, int BN, bool kArgmax>
cudaError_t run_tc_t(const void* W, int64_t ldw, const void* X, int64_t ldx, int M, void* Y, int N,
                     int K, const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  constexpr bool bf16 = std::is_same<T, __nv_bfloat16>::value;
  CUtensorMap tw, tx;
  if (!make_map(&tw, bf16, W, ldw, K, N, kTcRows) || !make_map(&tx, bf16, X, ldx, K, M, BN))
    return cudaErrorNotSupported;
  auto kern = dense_tc_kernel<T, TO, BN, kArgmax>;
  const int smem = TcShape<BN>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int ntiles = (N + kTcRows - 1) / kTcRows;
  int grid = device_sm_count();
  if (grid > ntiles) grid = ntiles;
  info->grid_x = grid;
  info->block = kTcThreads;
  info->smem = smem;
  info->kernel = "dense_tc";
  return launch_k(kern, dim3(grid), dim3(kTcThreads), smem, st, true, tw, tx, M,
                  static_cast<TO*>(Y), N, K, am, error_word_ptr());
}

template <typename T, typename TO>
cudaError_t run_tc(const void* W, int64_t ldw, const void* X, int64_t ldx, int M, void* Y, int N,
                   int K, const ArgmaxArgs& am, cudaStream_t st, Launch* info) {
  if (M <= 16)
    return am.out ? run_tc_t<T, TO, 16, true>(W, ldw, X, ldx, M, Y, N, K, am, st, info)
                  : run_tc_t<T, TO, 16, false>(W, ldw, X, ldx, M, Y, N, K, am, st, info);
  return am.out ? run_tc_t<T, TO, 32, true>(W, ldw, X, ldx, M, Y, N, K, am, st, info)
                : run_tc_t<T, TO, 32, false>(W, ldw, X, ldx, M, Y, N, K, am, st, info);
}

}  // namespace

bool dense_tc_enabled() {
  const char* v = std::getenv("WOBS_TC");
  return !(v && v[0] == '0');
}

cudaError_t launch_gemv_dense_tc(int dtype, const void* W, int64_t ldw, const void* X, int64_t ldx,
                                 int M, void* Y, int N, int K, const ArgmaxArgs& am, cudaStream_t st,
                                 Launch* info) {
  if (dtype == 0) return run_tc<__half, __half>(W, ldw, X, ldx, M, Y, N, K, am, st, info);
  return run_tc<__nv_bfloat16, float>(W, ldw, X, ldx, M, Y, N, K, am, st, info);
}

}  // namespace wobs
