/*
 * wobs.h -- C ABI of the weight-only low-bit decode GEMV library (sm_103a).
 *
 * The library computes the batch-1 (and small-batch, M <= 32) decode
 * matrix-vector product y = W x that the batch1-cdna README describes
 * ("Hand-written FP16 y = Wx, batch size one ... every weight is read once
 * and never reused, so token time is bytes divided by bandwidth"), over
 * three weight formats:
 *   - dense fp16 / bf16 (batch1-cdna README, "02-gemv");
 *   - Q4_0 weights x Q8_1 activations with integer block dots ("The kernel
 *     that waited for itself", m12-db-gemm case study, section "Seven
 *     variants, one microbenchmark, many mistakes"), and Q8_0 weights x
 *     Q8_1 activations (same page, "What correctness was measured against");
 *   - NF4 blockwise 4-bit codebook weights (bitsandbytes issue #1842,
 *     "Benchmark Data" and "Minimal Repro");
 * plus an optional fused greedy argmax over the outputs ("[WIP] ArgCompare
 * Benchmark Results and Performance Analysis", IREE discussion #23609).
 *
 * Conventions (every entry point):
 *   - Returns an int status: WOBS_OK (0) or a negative WOBS_ERR_* code.
 *     wobs_last_error() gives a message for the calling thread's last error.
 *     No exception, abort or trap crosses the ABI.
 *   - Pointers are DEVICE memory owned by the caller unless the argument
 *     says "host".  The library never allocates, frees or synchronises in
 *     these calls.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls are asynchronous: argument and launch errors are
 *     reported on return; results are ready when the stream reaches them.
 *   - Activations and outputs with M columns are row-major [M][...]: column
 *     m of the mathematical X is the contiguous row X + m*ldx.
 *   - Weight matrices are row-major [N][K] (one output per row).
 *   - Alignment: every weight pointer, activation pointer and row pitch must
 *     give 16-byte aligned rows; violations return WOBS_ERR_MISALIGNED.
 *   - Workspace: calls that take (ws, ws_bytes) need at least
 *     wobs_workspace_size(op, M, N, K) bytes, ZERO-FILLED before its first
 *     use.  Its first WOBS_WS_ZERO_BYTES bytes (or all of it, if smaller)
 *     hold arrival counters and argmax keys; every call that returns
 *     WOBS_OK leaves them zero again (reset by the last arrival).  Bytes
 *     past that offset are split-K partials: scratch that a call writes
 *     before it reads, which may be left non-zero.  So one zeroing serves
 *     any number of calls, whatever their shapes.  Split-K calls support
 *     N up to 1048576 rows (WOBS_ERR_UNSUPPORTED_SHAPE beyond).  Calls that
 *     overlap on the GPU must not share one workspace.  Size 0 means no
 *     workspace is needed (ws may be NULL).
 *   - Environment: WOBS_DEBUG=1 logs every dispatch (op, shape, kernel,
 *     grid, split) to stderr; WOBS_SPLITK=<s> overrides the split-K factor
 *     of the dense and Q4_0 multi-column kernels (testing only; the
 *     workspace must be sized for it with the same variable set);
 *     WOBS_TC=0 keeps dense GEMVs off the tcgen05 kernel and WOBS_M1=ldg
 *     selects the direct-load M = 1 kernels (both for testing).
 *     WOBS_SPLITK=<s> also forces <s> slices per row on wobs_argmax /
 *     wobs_argmin.  WOBS_NF4=cp selects the CUDA-core NF4 kernel,
 *     WOBS_NF4_P=0..3 sets how many code words in eight the tensor-core NF4
 *     kernel decodes in registers, and WOBS_NF4_STAGES=2..4 caps its copy
 *     ring (all three for measurements).  WOBS_Q4TC=1 takes Q4_0 calls with
 *     5..16 columns to the tcgen05 kernel as well (17..32 take it by
 *     default where its plan fills the GPU), WOBS_Q4TC=0 keeps every Q4_0
 *     call off it; WOBS_Q4F32=16 or 32 runs the fused quantise-and-GEMV
 *     kernel with 16 warps and two CTAs per SM or 32 warps and one (the
 *     default picks by shape; testing only).  WOBS_NF4_P=0..3 also applies
 *     to the NF4 tensor-memory kernel for several columns.  WOBS_Q4MC=1, 2
 *     or 4 runs the 2..4-column Q4_0 kernel with that many weight rows per
 *     warp (the default picks by shape; testing only).  WOBS_NF4_MC=tc
 *     takes NF4 calls with 2..4 columns to the tensor-memory kernel instead
 *     of the mma.sync kernel (testing only).  WOBS_PDL=0 launches every
 *     kernel without programmatic dependent launch (each then starts after
 *     its predecessor has finished; for measurements).
 */
#ifndef WOBS_H
#define WOBS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define WOBS_API __attribute__((visibility("default")))
#else
#define WOBS_API
#endif

/* ---- status codes ---- */
#define WOBS_OK 0
#define WOBS_ERR_INVALID_ARG (-1)         /* null pointer, bad enum, M out of range */
#define WOBS_ERR_MISALIGNED (-2)          /* pointer or pitch breaks 16-byte rows */
#define WOBS_ERR_UNSUPPORTED_SHAPE (-3)   /* K not a multiple of the block size, N < 1 */
#define WOBS_ERR_WORKSPACE_TOO_SMALL (-4)
#define WOBS_ERR_LAUNCH_FAILED (-5)       /* cudaGetLastError() after the launch */
#define WOBS_ERR_CUDA (-6)                /* other CUDA runtime error (device query) */
#define WOBS_ERR_DEVICE_TIMEOUT (-7)      /* wobs_error_word: a bounded device wait gave up */

/* ---- ops for wobs_workspace_size ---- */
#define WOBS_OP_GEMV_F16 1
#define WOBS_OP_GEMV_BF16 2
#define WOBS_OP_GEMV_Q4_0_Q8_1 3
#define WOBS_OP_GEMV_NF4 4
#define WOBS_OP_ARGCMP 5     /* wobs_argmax / wobs_argmin; K = element bytes */
#define WOBS_OP_GEMV_Q8_0_Q8_1 6
#define WOBS_OP_GEMV_Q4_0_F32 7   /* wobs_gemv_q4_0_f32 */
#define WOBS_OP_GEMV_Q8_0_F32 8   /* wobs_gemv_q8_0_f32 */

/* ---- element types of wobs_argmax / wobs_argmin ---- */
#define WOBS_DTYPE_F16 1
#define WOBS_DTYPE_BF16 2
#define WOBS_DTYPE_F32 3

/* Leading workspace bytes that hold counters and keys (zero between calls). */
#define WOBS_WS_ZERO_BYTES 262408

/* Largest activation-column count of the multi-column entry points. */
#define WOBS_MAX_M 32

/* Message for the calling thread's most recent error ("" if none). */
WOBS_API const char* wobs_last_error(void);

/* Library ABI version (integer, increases on incompatible change). */
WOBS_API int wobs_version(void);

/*
 * Streaming-read probe: the bandwidth ceiling used as the denominator of
 * every bandwidth-utilisation figure (batch1-cdna README, "01-ceiling": a
 * grid-stride read of a buffer far larger than the last-level cache, every
 * element folded into one scalar so no load can be dropped).
 *
 *   buf      device buffer, 16-byte aligned; bytes a multiple of 16
 *   grid     CTAs to launch; 0 = one wave of resident CTAs on every SM
 *   variant  0 = plain 16-byte read-only loads (L1-cached)
 *            1 = 16-byte loads, L1 no-allocate + L2 evict-first
 *            2 = 32-byte loads (one 256-bit vector per iteration), same hints;
 *                buf must be 32-byte aligned
 *            3 = bulk asynchronous copies (cp.async.bulk) into a shared-memory
 *                ring, completion tracked by mbarriers
 *   xor_out  device uint32: the XOR of every little-endian 32-bit word of
 *            buf is XOR-ed into it (zero it first to read the checksum)
 * Errors: INVALID_ARG (null, bad variant, grid < 0), MISALIGNED.  Variant 3
 * bounds every wait; a wait that gives up sets the device error word
 * (wobs_error_word) instead of hanging.
 */
WOBS_API int wobs_bw_probe(const void* buf, size_t bytes, int grid, int variant,
                           uint32_t* xor_out, void* stream);

/*
 * Dense fp16 GEMV, y[m][n] = sum_k W[n][k] * X[m][k], fp32 accumulation,
 * fp16 outputs rounded to nearest even (batch1-cdna README, "02-gemv":
 * fp16 weights and activations, fp32 accumulate).
 *
 *   W   fp16 [N][ldw] (ldw >= K, multiple of 8), X fp16 [M][ldx] (ldx >= K,
 *       multiple of 8), Y fp16 [M][N]; 1 <= M <= WOBS_MAX_M; K multiple of 8.
 *   ws  workspace (op WOBS_OP_GEMV_F16); may be NULL when the call does not
 *       split K (wobs_workspace_size(...) <= 512).
 */
WOBS_API int wobs_gemv_f16(const void* W, int64_t ldw, const void* X, int64_t ldx, int M,
                           void* Y, int N, int K, void* ws, size_t ws_bytes, void* stream);

/*
 * Dense bf16 GEMV with fp32 outputs (logits) and an optional fused greedy
 * argmax per activation column: argmax[m] = the n of the largest
 * logits[m][n], ties to the lowest n, -0.0 equal to +0.0 (ArgCompare
 * discussion, section "ArgMax/ArgMin Operations Analysis in real-world AI
 * models": LLaMA-3-8B argmax over [1,128000] and [32,128000], i64 out).
 *
 *   W  bf16 [N][ldw], X bf16 [M][ldx] (pitches multiples of 8, >= K),
 *   logits fp32 [M][N], argmax int64 [M] or NULL; 1 <= M <= WOBS_MAX_M,
 *   K multiple of 8.  Logits must be finite for the argmax to be defined.
 *   ws  workspace (op WOBS_OP_GEMV_BF16).
 */
WOBS_API int wobs_gemv_bf16(const void* W, int64_t ldw, const void* X, int64_t ldx, int M,
                            float* logits, int64_t* argmax, int N, int K, void* ws,
                            size_t ws_bytes, void* stream);

/*
 * wobs_gemv_bf16 for callers that cannot give the library a workspace: the
 * same computation, outputs and argmax rule, with the workspace taken from a
 * fixed scratch array of WOBS_NOALLOC_SCRATCH_BYTES that the library keeps
 * in device memory.  The pages have no counterpart to this entry point.
 * It serves callers that may not allocate device memory at the point of the
 * call: inference engines that reserve their whole memory budget once at
 * start-up and hand it out through their own allocator (a further
 * cudaMalloc can fail, or push them past the budget they planned for),
 * plugins loaded into a host process that owns and accounts every device
 * allocation, and latency-critical decode loops that cannot afford
 * cudaMalloc/cudaFree, which may synchronise the device.
 *
 *   Arguments as wobs_gemv_bf16, without (ws, ws_bytes).  No cudaMalloc,
 *   cudaFree or other allocating call is made.
 *   - Shapes whose workspace (wobs_workspace_size(WOBS_OP_GEMV_BF16, M, N,
 *     K)) exceeds WOBS_NOALLOC_SCRATCH_BYTES return
 *     WOBS_ERR_WORKSPACE_TOO_SMALL.
 *   - The first call made with a given device current looks up the scratch
 *     array's device address (cudaGetSymbolAddress) and keeps it for the
 *     life of the process; make that first call before any stream capture.
 *     A cudaDeviceReset (or anything else that unloads the library's module
 *     from the device) invalidates the kept address: do not call this entry
 *     point on that device afterwards.
 *   - Every call shares the one array and it keeps the last call's
 *     contents: each call clears the counters and keys on `stream` before
 *     its kernel, and calls that may overlap on the GPU (unordered streams
 *     or threads) race on the scratch and must not be issued.
 *   - Every GPU that loads the library holds the array until the process
 *     exits.
 */
#define WOBS_NOALLOC_SCRATCH_BYTES (4u << 20)
WOBS_API int wobs_gemv_bf16_noalloc(const void* W, int64_t ldw, const void* X, int64_t ldx,
                                    int M, float* logits, int64_t* argmax, int N, int K,
                                    void* stream);

/*
 * Q8_1 activation quantisation ("The kernel that waited for itself", section
 * "Seven variants, one microbenchmark, many mistakes": Q8_1 activations).
 * Per block of 32 consecutive elements of a column, IEEE float32:
 * d = max|x| / 127, q = round-half-away(x / d) (0 when d == 0),
 * s = d * sum(q); stored as {fp16 d; fp16 s; int8 q[32]} = 36 bytes,
 * fp16 by round-to-nearest-even.  Bit-exact with the definition.
 *
 *   X   fp32 [M][ldx] (ldx >= K, multiple of 4), xq  [M][K/32] blocks of 36
 *       bytes (4-byte aligned); 1 <= M <= WOBS_MAX_M; K multiple of 32.
 */
WOBS_API int wobs_quantize_q8_1(const float* X, int64_t ldx, int M, int K, void* xq,
                                void* stream);

/*
 * Q4_0 weight quantisation (same page and section: Q4_0 weights).  Per block
 * of 32 consecutive elements of a row, IEEE float32: amax = the signed
 * element of largest magnitude (first on ties), d = amax / -8,
 * q = clamp(round-half-away(w / d) + 8, 0, 15) (8 when d == 0).
 * Outputs the two planes the GEMV reads: qs [N][K/2] (byte j of a block =
 * element j in the low nibble, element j+16 in the high nibble) and
 * d fp16 [N][K/32].  Bit-exact with the definition.
 *
 *   W fp32 [N][ldw] (ldw >= K, multiple of 4); K multiple of 32.
 */
WOBS_API int wobs_quantize_q4_0(const float* W, int64_t ldw, int N, int K, uint8_t* qs,
                                void* d, void* stream);

/*
 * NF4 blockwise weight quantisation (bitsandbytes issue #1842, "Minimal
 * Repro": quantize_4bit with quant_type 'nf4', blocksize 64).  Per block of
 * 64 consecutive bf16 elements of a row, IEEE float32: absmax = max|w|,
 * v = w / absmax (0 when absmax == 0), code = the index k minimising
 * |codebook[k] - v| (lowest k on ties).  Outputs qs [N][K/2] (two codes per
 * byte, the first element in the HIGH nibble) and absmax fp32 [N][K/64].
 * Bit-exact with the definition.
 *
 *   W bf16 [N][ldw] (ldw >= K, multiple of 8); codebook: HOST pointer to 16
 *   floats (copied into the launch); K multiple of 64.
 */
WOBS_API int wobs_quantize_nf4(const void* W, int64_t ldw, int N, int K,
                               const float* codebook, uint8_t* qs, float* absmax,
                               void* stream);

/*
 * Q4_0 x Q8_1 GEMV ("The kernel that waited for itself": the decode matrix
 * product over Q4_0 weights and Q8_1 activations, 1 to 32 columns).  Per
 * weight block b and column m the exact integer block dot
 * sumi = sum_i (q4_i - 8) * q8_{m,i} is formed with 4-way byte dot
 * products, then y[m][n] += d4[n][b] * d8[m][b] * sumi in fp32.
 *
 *   qs  [N][K/2] nibble plane, d fp16 [N][K/32] (from wobs_quantize_q4_0 or
 *   repacked llama.cpp blocks); xq [M][K/32] Q8_1 blocks; y fp32 [M][N];
 *   argmax int64 [M] or NULL; 1 <= M <= WOBS_MAX_M; K multiple of 32.
 *   ws  workspace (op WOBS_OP_GEMV_Q4_0_Q8_1).
 */
WOBS_API int wobs_gemv_q4_0_q8_1(const uint8_t* qs, const void* d, const void* xq, int M,
                                 float* y, int64_t* argmax, int N, int K, void* ws,
                                 size_t ws_bytes, void* stream);

/*
 * Q4_0 GEMV on one fp32 activation vector, its Q8_1 quantisation fused into
 * the GEMV ("The kernel that waited for itself", section "Seven variants,
 * one microbenchmark, many mistakes": the decode product over Q4_0 weights
 * and Q8_1-quantised activations).  One kernel: every CTA quantises x into
 * shared memory itself, taking every decision of the quantiser (IEEE
 * float32 block scale and quotients, round half away from zero), and
 * y and argmax are bit-identical to wobs_quantize_q8_1(x) followed by
 * wobs_gemv_q4_0_q8_1 with M = 1.  When xq_out is not NULL the kernel also
 * writes the K/32 Q8_1 blocks there, bit-identical to wobs_quantize_q8_1
 * (for other GEMVs on the same activation vector).
 *
 *   qs, d, y, argmax, N: as wobs_gemv_q4_0_q8_1 with M = 1; x fp32 [K];
 *   xq_out [K/32] blocks of 36 bytes or NULL (must not overlap x).
 *   qs, d and x 16-byte aligned, y and xq_out 4-byte aligned; K a multiple
 *   of 256 and at most 104704 (the activation planes live in shared memory).
 *   ws  workspace (op WOBS_OP_GEMV_Q4_0_F32), needed only for the argmax.
 *   Errors: WOBS_ERR_UNSUPPORTED_SHAPE for another K (quantise with
 *   wobs_quantize_q8_1 and call wobs_gemv_q4_0_q8_1 instead),
 *   WOBS_ERR_MISALIGNED, WOBS_ERR_INVALID_ARG for a null pointer.
 */
WOBS_API int wobs_gemv_q4_0_f32(const uint8_t* qs, const void* d, const float* x, void* xq_out,
                                float* y, int64_t* argmax, int N, int K, void* ws,
                                size_t ws_bytes, void* stream);

/*
 * Q8_0 weight quantisation ("The kernel that waited for itself", section
 * "What correctness was measured against": the matrix path is tested on
 * Q4_0 and Q8_0 weights).  Per block of 32 consecutive elements of a row,
 * IEEE float32: d = max|w| / 127, q = round-half-away(w / d) (0 when
 * d == 0).  Outputs the two planes the GEMV reads: qs int8 [N][K] (codes in
 * element order) and d fp16 [N][K/32].  Bit-exact with the definition.
 *
 *   W fp32 [N][ldw] (ldw >= K, 4-byte aligned); K multiple of 32.
 */
WOBS_API int wobs_quantize_q8_0(const float* W, int64_t ldw, int N, int K, int8_t* qs, void* d,
                                void* stream);

/*
 * Q8_0 x Q8_1 GEMV (same page and section), 1 to 32 columns: per weight
 * block b and column m the exact integer block dot
 * sumi = sum_i qw_i * q8_{m,i} (signed 4-way byte dot products), then
 * y[m][n] += dw[n][b] * d8[m][b] * sumi in fp32.
 *
 *   qs int8 [N][K] and d fp16 [N][K/32] (both 16-byte aligned, from
 *   wobs_quantize_q8_0 or repacked llama.cpp blocks); xq [M][K/32] Q8_1
 *   blocks; y fp32 [M][N]; argmax int64 [M] or NULL; 1 <= M <= WOBS_MAX_M;
 *   K a multiple of 256 (UNSUPPORTED_SHAPE otherwise, also when K is so long
 *   that one column's activation blocks no longer fit in shared memory).
 *   Columns are processed eight at a time (fewer for very long rows), one
 *   kernel launch each, so the weights are read once per eight columns.
 *   ws  workspace (op WOBS_OP_GEMV_Q8_0_Q8_1), needed only for the argmax.
 */
WOBS_API int wobs_gemv_q8_0_q8_1(const int8_t* qs, const void* d, const void* xq, int M,
                                 float* y, int64_t* argmax, int N, int K, void* ws,
                                 size_t ws_bytes, void* stream);

/*
 * Q8_0 GEMV on one fp32 activation vector, its Q8_1 quantisation fused into
 * the GEMV (the case study's Q8_0 weights with Q8_1-quantised activations).
 * One kernel: every CTA quantises x into shared memory with the quantiser's
 * IEEE float32 decisions, and y and argmax are bit-identical to
 * wobs_quantize_q8_1(x) followed by wobs_gemv_q8_0_q8_1 with M = 1.  When
 * xq_out is not NULL the K/32 Q8_1 blocks are also written there,
 * bit-identical to wobs_quantize_q8_1.
 *
 *   qs, d, y, argmax, N: as wobs_gemv_q8_0_q8_1 with M = 1; x fp32 [K];
 *   xq_out [K/32] blocks of 36 bytes or NULL (must not overlap x).
 *   qs, d and x 16-byte aligned, y and xq_out 4-byte aligned; K a multiple
 *   of 256 whose activation planes (36 bytes per block) fit in shared memory
 *   beside the weight ring (K up to 143616 with 227 KB of shared memory per CTA).
 *   ws  workspace (op WOBS_OP_GEMV_Q8_0_F32), needed only for the argmax.
 *   Errors: WOBS_ERR_UNSUPPORTED_SHAPE for another K, WOBS_ERR_MISALIGNED,
 *   WOBS_ERR_INVALID_ARG for a null pointer.
 */
WOBS_API int wobs_gemv_q8_0_f32(const int8_t* qs, const void* d, const float* x, void* xq_out,
                                float* y, int64_t* argmax, int N, int K, void* ws,
                                size_t ws_bytes, void* stream);

/*
 * NF4 GEMV for 1..32 activation columns (bitsandbytes issue #1842: the
 * fused 4-bit inference GEMV; one decode token is M = 1, a small decode
 * batch M > 1): Y[m][n] = sum_b absmax[n][b] * sum_i codebook[code_i] *
 * X[m][i], fp32 accumulation, bf16 output (round to nearest even).
 * Optional fused argmax per column over the bf16 outputs (as stored).
 * M >= 2 runs on the tensor cores with every weight rounded once to f16
 * (relative error <= 2^-11, inside the GEMV tolerance): for 2..4 columns
 * the one-column mma.sync kernel, each code decoded once for all columns,
 * where K is a multiple of 1024 up to 8192, the planes and X 16-byte
 * aligned and ldx a multiple of 8; otherwise the tcgen05 kernel where K is
 * a multiple of 256 and the planes and activation rows are 16-byte aligned;
 * else the CUDA cores in fp32.
 *
 *   qs [N][K/2], absmax fp32 [N][K/64], codebook HOST pointer to 16 floats,
 *   X bf16 [M][ldx] (ldx >= K; ignored for M = 1), Y bf16 [M][N], argmax
 *   int64 [M] or NULL; 1 <= M <= WOBS_MAX_M; K multiple of 64, at most
 *   32768.  ws  workspace (op WOBS_OP_GEMV_NF4, with the same M).
 */
WOBS_API int wobs_gemv_nf4(const uint8_t* qs, const float* absmax, const float* codebook,
                           const void* X, int64_t ldx, int M, void* Y, int64_t* argmax, int N,
                           int K, void* ws, size_t ws_bytes, void* stream);

/*
 * NF4 -> bf16 dequantisation, the first half of the dequantise-then-GEMM
 * path (bitsandbytes issue #1842, "Benchmark Data": dequantise + bf16
 * matrix product, the alternative the fused GEMV is measured against, which
 * pays off when the dequantised matrix serves many activation columns):
 * W[n][k] = bf16(absmax[n][k/64] * codebook[code(n, k)]), the product taken
 * in IEEE float32 and rounded to nearest even.  Bit-exact with the
 * definition.  The dense GEMV entry points (wobs_gemv_bf16) then take W.
 *
 *   qs [N][K/2], absmax fp32 [N][K/64], codebook HOST pointer to 16 floats,
 *   W bf16 [N][ldw] (ldw >= K, even, 4-byte aligned); K multiple of 64.
 */
WOBS_API int wobs_dequantize_nf4(const uint8_t* qs, const float* absmax, const float* codebook,
                                 int N, int K, void* W, int64_t ldw, void* stream);

/*
 * Standalone ArgCompare over the rows of a matrix ("[WIP] ArgCompare
 * Benchmark Results and Performance Analysis", IREE discussion #23609:
 * argmax over the vocabulary axis, [1..32, 32K..256K] f16/bf16/f32 -> i64,
 * batched rows up to [4096, 32768], and argmin over [32, 1M] f32, section
 * "ArgMax/ArgMin Operations Analysis in real-world AI models").
 *
 *   wobs_argmax: out[m] = the n of the largest X[m][n]; wobs_argmin: of the
 *   smallest.  Among equal values the lowest n wins; -0.0 equals +0.0;
 *   infinities are ordered like other values; a row holding NaN gives an
 *   unspecified index in 0..N-1.
 *
 *   dtype  WOBS_DTYPE_F16, _BF16 or _F32
 *   X      [M][ldx] elements of dtype, aligned to the element size, any
 *          pitch ldx >= N (ignored when M == 1): rows need not start on a
 *          16-byte boundary (the exception to the library's alignment rule);
 *          N any value in 1..WOBS_ARGCMP_MAX_N; 1 <= M <= WOBS_ARGCMP_MAX_M
 *   out    int64 [M], 8-byte aligned
 *   ws     workspace of wobs_workspace_size(WOBS_OP_ARGCMP, M, N, element
 *          bytes): zero when one CTA or one warp covers a row (ws may then
 *          be NULL), else 12 bytes a row (per-row keys and arrival counters,
 *          zero-filled, left zero-filled after the call).
 * Errors: INVALID_ARG (null, dtype, M, ldx), UNSUPPORTED_SHAPE (N),
 * MISALIGNED, WORKSPACE_TOO_SMALL, LAUNCH_FAILED.
 */
#define WOBS_ARGCMP_MAX_M (1 << 24)
#define WOBS_ARGCMP_MAX_N (1 << 30)
WOBS_API int wobs_argmax(int dtype, const void* X, int64_t ldx, int M, int N, int64_t* out,
                         void* ws, size_t ws_bytes, void* stream);
WOBS_API int wobs_argmin(int dtype, const void* X, int64_t ldx, int M, int N, int64_t* out,
                         void* ws, size_t ws_bytes, void* stream);

/*
 * Workspace bytes needed by one call of `op` with this shape on the current
 * device (split-K partials and counters, argmax keys and counter).  Returns
 * 0 for an unknown op or a shape that needs none.  For WOBS_OP_ARGCMP, M
 * and N are the matrix shape and K the element size in bytes (2 or 4).
 */
WOBS_API size_t wobs_workspace_size(int op, int M, int N, int K);

/*
 * Test export: the exact int32 block dots sumi[m][n][b] =
 * sum_i (q4_i - 8) * q8_{m,i} that the Q4_0 x Q8_1 GEMV forms ("The kernel
 * that waited for itself", section "What correctness was measured against":
 * CPU calculation on the quantised values).  out int32 [M][N][K/32].
 */
WOBS_API int wobs_q4_0_q8_1_blockdots(const uint8_t* qs, const void* xq, int M, int N, int K,
                                      int32_t* out, void* stream);

/*
 * Device error word: kernels that give up a bounded wait record a nonzero
 * code here instead of hanging.  Copies the word to *host_out (host pointer)
 * and clears it; synchronises `stream` to do so.  0 = no error.
 * Returns WOBS_OK when the word was 0 and WOBS_ERR_DEVICE_TIMEOUT when it
 * held a code (still copied to *host_out): a launch returns before its
 * kernel runs, so a wait that gives up on the GPU can only be reported by
 * this later, synchronising call.
 */
WOBS_API int wobs_error_word(void* stream, int* host_out);

/*
 * Test export for the failure path (no counterpart on the pages): launches
 * one warp that waits on an mbarrier nothing arrives on, bounded by
 * `limit_cycles` (1 ... 1e9 SM clock cycles), so the wait gives up, writes
 * WOBS_DEVICE_WAIT_SELFTEST (3) to the device error word and the kernel
 * returns; the context stays usable.  Codes the kernels write: 1 = a
 * read-ceiling probe wait, 2 = a GEMV copy wait, 3 = this self test.
 */
WOBS_API int wobs_selftest_wait_timeout(long long limit_cycles, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* WOBS_H */
