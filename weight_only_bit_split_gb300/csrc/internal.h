// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Host and device visible; no torch types anywhere.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace wobs {

// Fused greedy-argmax epilogue state (all pointers device memory, inside
// the caller's workspace except `out`).
struct ArgmaxArgs {
  int64_t* out;        // [M] argmax indices (caller's output); null = off
  uint64_t* keys;      // [32] running best keys, zero between calls
  unsigned* counter;   // CTA arrival counter, zero between calls
};

// Split-K state: fp32 partial sums and one arrival counter per row group.
struct SplitArgs {
  float* partials;     // [splits][M][N]
  unsigned* counters;  // [row groups], zero between calls
  int splits;          // 1 = no split
};

struct Launch {
  int grid_x = 0, grid_y = 1, block = 0, smem = 0;
  const char* kernel = "";
};

// 16-entry codebook passed by value as a kernel parameter.
struct Codebook16 {
  float v[16];
};

// ---- launchers (each returns cudaGetLastError() after the launch) ----

cudaError_t launch_bw_probe(const void* buf, size_t bytes, int grid, int variant,
                            uint32_t* xor_out, cudaStream_t st, Launch* info);

// dense: T = 0 fp16 inputs, 1 bf16 inputs; out_f32 = 1 writes float, else
// the input type.
cudaError_t launch_gemv_dense(int dtype, const void* W, int64_t ldw, const void* X, int64_t ldx,
                              int M, void* Y, int out_f32, int N, int K, const SplitArgs& sk,
                              const ArgmaxArgs& am, cudaStream_t st, Launch* info);

// Dense 2..32 columns on tcgen05 / TMA (no K split); cudaErrorNotSupported
// when the driver offers no tensor-map encoder.  WOBS_TC=0 turns it off.
cudaError_t launch_gemv_dense_tc(int dtype, const void* W, int64_t ldw, const void* X, int64_t ldx,
                                 int M, void* Y, int N, int K, const ArgmaxArgs& am, cudaStream_t st,
                                 Launch* info);
bool dense_tc_enabled();

cudaError_t launch_quantize_q8_1(const float* X, int64_t ldx, int M, int K, void* xq,
                                 cudaStream_t st, Launch* info);
cudaError_t launch_quantize_q4_0(const float* W, int64_t ldw, int N, int K, uint8_t* qs,
                                 void* d, cudaStream_t st, Launch* info);
cudaError_t launch_quantize_nf4(const void* W, int64_t ldw, int N, int K, const Codebook16& cb,
                                uint8_t* qs, float* absmax, cudaStream_t st, Launch* info);

cudaError_t launch_gemv_q4_0_q8_1(const uint8_t* qs, const void* d, const void* xq, int M,
                                  float* Y, int N, int K, const SplitArgs& sk,
                                  const ArgmaxArgs& am, cudaStream_t st, Launch* info);
// Multi-column (M >= 2) tensor-core kernel; K % 256 == 0 and a 16-byte
// aligned scale plane.  q4_mma_splits gives the K split it launches with
// (forced > 0: the WOBS_SPLITK override), which sizes the workspace.
cudaError_t launch_q4_mma(const uint8_t* qs, const void* d, const void* xq, int M, float* Y, int N,
                          int K, int forced, const SplitArgs& sk, const ArgmaxArgs& am,
                          cudaStream_t st, Launch* info);
int q4_mma_splits(int M, int N, int K, int forced);
// Split-K partial bytes of its launch (fragment-ordered, padded columns).
size_t q4_mma_partial_bytes(int M, int N, int K, int forced);
// The few-column (2..8) whole-row kernel applies (it needs no K split).
bool q4_mc_applies(int M, int K);
// Q8_1 quantisation fused into the M = 1 cp.async kernel (one launch).
bool q4_0_f32_fused_applies(const void* d, int M, int K);
cudaError_t launch_gemv_q4_0_f32_fused(const uint8_t* qs, const void* d, const float* x,
                                       void* xq_out, float* y, int N, int K, const ArgmaxArgs& am,
                                       cudaStream_t st, Launch* info);
// Q8_1 quantisation fused into the Q8_0 M = 1 kernel (one launch).
bool q8_0_f32_fused_applies(int K);
cudaError_t launch_gemv_q8_0_f32_fused(const int8_t* qs, const void* d, const float* x,
                                       void* xq_out, float* y, int N, int K, const ArgmaxArgs& am,
                                       cudaStream_t st, Launch* info);
// Multi-column (5..32) tcgen05 kernel: weights decoded into tensor memory,
// block scales folded into f16 operands.  The plan fixes the K range of a
// work unit, the split count (K / range) and the grid.
struct Q4TcPlan {
  bool ok = false;
  int range = 0, splits = 1, grid = 0;
};
bool q4_tc_enabled();      // WOBS_Q4TC != 0
Q4TcPlan q4_tc_plan(int M, int N, int K);
size_t q4_tc_partial_bytes(int M, int N, int K);
cudaError_t launch_q4_tc(const uint8_t* qs, const void* d, const void* xq, int M, float* Y, int N,
                         int K, const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                         Launch* info);
// WOBS_SPLITK, or 0 when unset.
int forced_splits();
cudaError_t launch_q4_0_q8_1_blockdots(const uint8_t* qs, const void* xq, int M, int N, int K,
                                       int32_t* out, cudaStream_t st, Launch* info);

// Q8_0 weights: quantiser, and the GEMV (K % 256 == 0, 16-byte aligned
// planes; columns taken q8_0_columns_per_launch(K) at a time, 0 = K too long)
cudaError_t launch_quantize_q8_0(const float* W, int64_t ldw, int N, int K, int8_t* qs, void* d,
                                 cudaStream_t st, Launch* info);
cudaError_t launch_gemv_q8_0_q8_1(const int8_t* qs, const void* d, const void* xq, int M, float* Y,
                                  int N, int K, const ArgmaxArgs& am, cudaStream_t st,
                                  Launch* info);
int q8_0_columns_per_launch(int K);

cudaError_t launch_gemv_nf4(const uint8_t* qs, const float* absmax, const Codebook16& cb,
                            const void* x, void* y, int N, int K, const ArgmaxArgs& am,
                            cudaStream_t st, Launch* info);
// NF4 with 2..32 activation columns (X bf16 [M][ldx], Y bf16 [M][N]): the
// tcgen05 kernel (K % 256 == 0, 16-byte aligned planes and activation rows;
// its plan fixes the K split, which must equal sk.splits) or the CUDA-core
// kernel (no split).
// The codebook scaled by a power of two into f16 normal numbers (largest
// magnitude in [2^14, 2^15)); false when an entry is not finite or a nonzero
// entry would fall below the f16 normal range.
bool nf4_codebook_scale(const Codebook16& cb, float* scale, float* inv);
struct Nf4TcPlan {
  bool ok = false;
  int range = 0, splits = 1, grid = 0;
};
Nf4TcPlan nf4_tc_plan(int M, int N, int K);
size_t nf4_tc_partial_bytes(int M, int N, int K);
cudaError_t launch_nf4_tc(const uint8_t* qs, const float* absmax, const Codebook16& cb, const void* X,
                          int64_t ldx, int M, void* Y, int N, int K, const SplitArgs& sk,
                          const ArgmaxArgs& am, cudaStream_t st, Launch* info);
cudaError_t launch_gemv_nf4_mc(const uint8_t* qs, const float* absmax, const Codebook16& cb,
                               const void* X, int64_t ldx, int M, void* Y, int N, int K,
                               const SplitArgs& sk, const ArgmaxArgs& am, cudaStream_t st,
                               Launch* info);
// NF4 -> bf16 dequantisation: W[n][k] = bf16(absmax[n][k/64] * codebook[code])
cudaError_t launch_dequantize_nf4(const uint8_t* qs, const float* absmax, const Codebook16& cb, int N,
                                  int K, void* W, int64_t ldw, cudaStream_t st, Launch* info);

// Standalone argmax / argmin over the rows of [M][N] (dtype 1 fp16, 2 bf16,
// 3 fp32).  warp_rows: one warp per row, no workspace; otherwise one CTA per
// (row, slice of `chunk` elements), `splits` slices a row, and with more than
// one slice the rows' keys [M] and arrival counters [M] live in the caller's
// workspace.
struct ArgcmpPlan {
  bool warp_rows = false;
  int splits = 1;
  int chunk = 0;
};
ArgcmpPlan plan_argcmp(int esize, int M, int N, int forced_splits);
cudaError_t launch_argcmp(int dtype, bool is_min, const void* X, int64_t ldx, int M, int N,
                          const ArgcmpPlan& p, int64_t* out, uint64_t* keys, unsigned* counters,
                          cudaStream_t st, Launch* info);

cudaError_t read_and_clear_error_word(cudaStream_t st, int* host_out);
cudaError_t launch_wait_timeout(long long limit, cudaStream_t st, Launch* info);
// Device address of the error word on the current device (null if unknown).
int* error_word_ptr();

// Device error codes written to the error word.
constexpr int kErrProbeWait = 1;      // bw_probe bulk-copy wait gave up
constexpr int kErrGemvWait = 2;       // a GEMV bulk-copy wait gave up
constexpr int kErrSelfTestWait = 3;   // the failure-path self test's wait gave up (expected)

// Which M = 1 kernel family to use: bulk-copy rings (default where the
// shape allows) or direct 16-byte loads (WOBS_M1=ldg forces the latter).
bool m1_ldg_forced();
// WOBS_NF4=cp: NF4 GEMVs take the CUDA-core staged kernel, not the tensor-core one
bool nf4_cp_forced();
// NF4 for 1..4 activation columns (x [M][ldx] bf16, y [M][N]) on mma.sync;
// cudaErrorNotSupported when the shape, the alignment or the codebook rules
// it out (the caller then takes another kernel)
cudaError_t launch_nf4_mma(const uint8_t* qs, const float* absmax, const Codebook16& cb,
                           const void* x, int64_t ldx, int M, void* y, int N, int K,
                           const ArgmaxArgs& am, cudaStream_t st, Launch* info);

// ---- shared launch-shape helpers (api.cu) ----
int device_sm_count();                       // current device, cached
int max_resident_ctas(const void* kernel, int block, int smem);  // per SM

// Split factor chosen for an op (also sizes the workspace).
int choose_splits(int op, int M, int N, int K);

// Workspace bytes for (op, M, N, K); *zero_prefix_bytes receives how many
// leading bytes hold counters and keys that must be zero before a call.
size_t workspace_layout(int op, int M, int N, int K, size_t* zero_prefix_bytes);
// Validates a workspace and points the split-K / argmax state into it.
int prepare_workspace(int op, int M, int N, int K, int64_t* argmax, void* ws, size_t ws_bytes,
                      SplitArgs* sk, ArgmaxArgs* am);
int check_dense_args(const char* op, const void* W, int64_t ldw, const void* X, int64_t ldx, int M,
                     const void* Y, int N, int K);
int report_launch(cudaError_t e, const char* op, int M, int N, int K, const Launch& L, int splits);
int set_error(int code, const char* msg);

}  // namespace wobs
