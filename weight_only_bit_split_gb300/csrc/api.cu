// C ABI of the library: argument checks, workspace layout, split-K choice,
// dispatch logging, status codes.  Declarations and full contracts are in
// include/wobs.h.  No allocation, no synchronisation (except
// wobs_error_word, which says so), no exception crosses this file.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/wobs.h"
#include "internal.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where, int code) {
  return fail(code, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool debug_on() {
  const char* v = std::getenv("WOBS_DEBUG");
  return v && v[0] && v[0] != '0';
}

int env_splits() {
  const char* v = std::getenv("WOBS_SPLITK");
  if (!v || !v[0]) return 0;
  int s = std::atoi(v);
  return s > 0 ? s : 0;
}

void log_dispatch(const char* op, int M, int N, int K, const wobs::Launch& L, int splits) {
  if (!debug_on()) return;
  std::fprintf(stderr,
               "wobs: op=%s M=%d N=%d K=%d kernel=%s grid=(%d,%d) block=%d smem=%d splits=%d\n",
               op, M, N, K, L.kernel, L.grid_x, L.grid_y, L.block, L.smem, splits);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

constexpr int kRowsPerGroup = 16;    // smallest row group of the multi-column kernels
// Split-K counters live in a fixed region (room for N up to 16 * kMaxGroups
// rows) and every call's partials start past it, so no call's counters can
// fall where another call left partials: only the header and the counter
// region must stay zero between calls.
constexpr int kMaxGroups = 65536;

struct WsLayout {
  size_t counter = 0, keys = 0, groups = 0, partials = 0, total = 0;
  int splits = 1;
  int ngroups = 0;
};

WsLayout ws_layout(int op, int M, int N, int K) {
  WsLayout L;
  L.splits = wobs::choose_splits(op, M, N, K);
  L.ngroups = L.splits > 1 ? (N + kRowsPerGroup - 1) / kRowsPerGroup : 0;
  size_t off = 0;
  L.counter = off;
  off += 8;
  L.keys = off;
  off += 8 * WOBS_MAX_M;
  L.groups = off;
  off += 4 * static_cast<size_t>(L.splits > 1 ? kMaxGroups : 0);
  off = (off + 255) & ~static_cast<size_t>(255);
  L.partials = off;
  if (L.splits > 1) {
    size_t pb = 4ull * L.splits * M * N;
    if ((op == WOBS_OP_GEMV_F16 || op == WOBS_OP_GEMV_BF16) && M >= 1) {
      // fragment-ordered partials of the tensor-core kernel: 256-row tiles,
      // columns padded to n8 tiles
      const size_t tb = 4ull * L.splits * ((N + 255) / 256) * 256 * (8 * ((M + 7) / 8));
      if (tb > pb) pb = tb;
    }
    if (op == WOBS_OP_GEMV_NF4 && M >= 2) {
      const size_t tb = wobs::nf4_tc_partial_bytes(M, N, K);
      if (tb > pb) pb = tb;
    }
    if (op == WOBS_OP_GEMV_Q4_0_Q8_1 && M >= 2 && K % 256 == 0) {
      size_t tb = wobs::q4_mma_partial_bytes(M, N, K, env_splits());
      if (!env_splits() && M >= 5 && wobs::q4_tc_enabled()) {
        const size_t tc = wobs::q4_tc_partial_bytes(M, N, K);
        if (tc > tb) tb = tc;
      }
      if (tb > pb) pb = tb;
    }
    off += pb;
  }
  L.total = off;
  return L;
}

struct Prepared {
  wobs::SplitArgs sk;
  wobs::ArgmaxArgs am;
};

int prepare_ws(int op, int M, int N, int K, int64_t* argmax, void* ws, size_t ws_bytes,
               Prepared* out) {
  const WsLayout L = ws_layout(op, M, N, K);
  if (L.ngroups > kMaxGroups)
    return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "N=%d: split-K calls support at most %d rows", N,
                16 * kMaxGroups);
  const bool need = argmax != nullptr || L.splits > 1;
  out->sk = wobs::SplitArgs{nullptr, nullptr, L.splits};
  out->am = wobs::ArgmaxArgs{nullptr, nullptr, nullptr};
  if (!need) return WOBS_OK;
  if (!ws) return fail(WOBS_ERR_INVALID_ARG, "workspace required (%zu bytes) but ws is NULL", L.total);
  if (!aligned16(ws)) return fail(WOBS_ERR_MISALIGNED, "workspace must be 16-byte aligned");
  if (ws_bytes < L.total)
    return fail(WOBS_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", ws_bytes, L.total);
  uint8_t* base = static_cast<uint8_t*>(ws);
  out->sk.partials = reinterpret_cast<float*>(base + L.partials);
  out->sk.counters = reinterpret_cast<unsigned*>(base + L.groups);
  if (argmax) {
    out->am.out = argmax;
    out->am.keys = reinterpret_cast<uint64_t*>(base + L.keys);
    out->am.counter = reinterpret_cast<unsigned*>(base + L.counter);
  }
  return WOBS_OK;
}

int finish_launch(cudaError_t e, const char* op, int M, int N, int K, const wobs::Launch& L,
                  int splits) {
  if (e != cudaSuccess) return cuda_fail(e, op, WOBS_ERR_LAUNCH_FAILED);
  log_dispatch(op, M, N, K, L, splits);
  g_err[0] = '\0';
  return WOBS_OK;
}

}  // namespace

namespace wobs {

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

int max_resident_ctas(const void* kernel, int block, int smem) {
  struct Entry { const void* k; int dev, block, smem, n; };
  static Entry table[128];
  static int used = 0;
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (table[i].k == kernel && table[i].dev == dev && table[i].block == block && table[i].smem == smem)
      return table[i].n;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, block, smem) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  if (n <= 0) n = 1;
  if (used < 128) table[used++] = Entry{kernel, dev, block, smem, n};
  return n;
}

int forced_splits() { return env_splits(); }

bool nf4_cp_forced() {
  const char* v = std::getenv("WOBS_NF4");
  return v && std::strcmp(v, "cp") == 0;
}

bool m1_ldg_forced() {
  const char* v = std::getenv("WOBS_M1");
  return v && std::strcmp(v, "ldg") == 0;
}

int choose_splits(int op, int M, int N, int K) {
  const int forced = env_splits();
  // row groups of 128 for the split heuristics (the counters themselves are
  // sized per kRowsPerGroup rows)
  const int groups = (N + 127) / 128;
  const int target = 2 * device_sm_count();
  switch (op) {
    case WOBS_OP_GEMV_F16:
    case WOBS_OP_GEMV_BF16: {
      const int kmax = K / 8 > 0 ? K / 8 : 1;
      if (forced) return forced < kmax ? forced : kmax;
      if (M == 1) return 1;
      // one CTA per SM: no split when the tensor-core kernel's 128-row tiles
      // fill the GPU; otherwise split K for the 256-row mma.sync tiles, never
      // past one wave
      if ((N + 127) / 128 >= device_sm_count()) return 1;
      const int ntiles = (N + 255) / 256;
      int s = device_sm_count() / ntiles;
      const int cap = K / 512 > 0 ? K / 512 : 1;
      if (s > cap) s = cap;
      return s < 1 ? 1 : s;
    }
    case WOBS_OP_GEMV_Q4_0_Q8_1: {
      const int nb = K / 32 > 0 ? K / 32 : 1;
      if (M == 1 && !forced) return 1;
      if (!forced && M >= 5 && q4_tc_enabled()) {
        const Q4TcPlan tp = q4_tc_plan(M, N, K);
        if (tp.ok) return tp.splits;
      }
      int s;
      if (M == 1) return forced < nb ? forced : nb;
      if (!forced && q4_mc_applies(M, K)) return 1;
      if (K % 256 == 0) {
        // tensor-core kernel (its own plan); the CUDA-core fallback, taken
        // for a misaligned scale plane, accepts any split
        const int sm = q4_mma_splits(M, N, K, forced);
        s = forced ? (forced < nb ? forced : nb) : sm;
        return s > sm ? s : sm;
      }
      // CUDA-core kernel: 48 bytes of shared memory per block per padded
      // column, at most 144 KB
      int nc = 1;
      while (nc < M) nc = nc < 8 ? nc * 2 : (nc == 8 ? 12 : (nc == 12 ? 16 : (nc == 16 ? 24 : 32)));
      const int bps_max = (144 * 1024) / (48 * nc);
      const int smin = (nb + bps_max - 1) / bps_max;
      if (forced) s = forced < nb ? forced : nb;
      else {
        s = (target + groups - 1) / groups;
        const int cap = nb / 4 > 0 ? nb / 4 : 1;
        if (s > cap) s = cap;
      }
      if (s < smin) s = smin;
      return s < 1 ? 1 : s;
    }
    case WOBS_OP_GEMV_NF4: {
      // several columns: the tensor-memory kernel's own K split (the
      // CUDA-core fallback takes none)
      if (M < 2 || nf4_cp_forced()) return 1;
      const Nf4TcPlan p = nf4_tc_plan(M, N, K);
      return p.ok ? p.splits : 1;
    }
    default:
      return 1;
  }
}

// ---- helpers for entry points defined in other files ----

size_t workspace_layout(int op, int M, int N, int K, size_t* zero_prefix_bytes) {
  const WsLayout L = ws_layout(op, M, N, K);
  // the bytes this call needs zero: header and its own group counters
  if (zero_prefix_bytes) *zero_prefix_bytes = L.groups + 4 * static_cast<size_t>(L.ngroups);
  return L.total;
}

int prepare_workspace(int op, int M, int N, int K, int64_t* argmax, void* ws, size_t ws_bytes,
                      SplitArgs* sk, ArgmaxArgs* am) {
  Prepared p;
  const int rc = prepare_ws(op, M, N, K, argmax, ws, ws_bytes, &p);
  *sk = p.sk;
  *am = p.am;
  return rc;
}

int check_dense_args(const char* op, const void* W, int64_t ldw, const void* X, int64_t ldx, int M,
                     const void* Y, int N, int K);

int report_launch(cudaError_t e, const char* op, int M, int N, int K, const Launch& L, int splits) {
  return finish_launch(e, op, M, N, K, L, splits);
}

int set_error(int code, const char* msg) { return fail(code, "%s", msg); }

}  // namespace wobs

extern "C" {

const char* wobs_last_error(void) { return g_err; }

int wobs_version(void) { return 1; }

size_t wobs_workspace_size(int op, int M, int N, int K) {
  if (op == WOBS_OP_ARGCMP) {
    // K carries the element size in bytes (2 or 4)
    if (M < 1 || M > WOBS_ARGCMP_MAX_M || N < 1 || N > WOBS_ARGCMP_MAX_N || (K != 2 && K != 4))
      return 0;
    const wobs::ArgcmpPlan p = wobs::plan_argcmp(K, M, N, env_splits());
    if (p.warp_rows || p.splits == 1) return 0;
    return (12ull * M + 15ull) & ~15ull;   // keys [M] (8 bytes), then counters [M] (4 bytes)
  }
  const bool known = (op >= WOBS_OP_GEMV_F16 && op <= WOBS_OP_GEMV_NF4) ||
                     op == WOBS_OP_GEMV_Q8_0_Q8_1 || op == WOBS_OP_GEMV_Q4_0_F32 ||
                     op == WOBS_OP_GEMV_Q8_0_F32;
  if (!known || M < 1 || M > WOBS_MAX_M || N < 1 || K < 1) return 0;
  return ws_layout(op, M, N, K).total;
}

int wobs_bw_probe(const void* buf, size_t bytes, int grid, int variant, uint32_t* xor_out,
                  void* stream) {
  if (!buf || !xor_out) return fail(WOBS_ERR_INVALID_ARG, "bw_probe: null pointer");
  if (variant < 0 || variant > 3) return fail(WOBS_ERR_INVALID_ARG, "bw_probe: variant %d", variant);
  if (grid < 0) return fail(WOBS_ERR_INVALID_ARG, "bw_probe: grid %d", grid);
  if (!aligned16(buf) || (bytes & 15u)) return fail(WOBS_ERR_MISALIGNED, "bw_probe: buffer/bytes not 16-byte aligned");
  if (!aligned4(xor_out)) return fail(WOBS_ERR_MISALIGNED, "bw_probe: xor_out not 4-byte aligned");
  if (variant == 2 && (reinterpret_cast<uintptr_t>(buf) & 31u))
    return fail(WOBS_ERR_MISALIGNED, "bw_probe: variant 2 (32-byte loads) needs a 32-byte aligned buffer");
  wobs::Launch L;
  cudaError_t e = wobs::launch_bw_probe(buf, bytes, grid, variant, xor_out,
                                        static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "bw_probe", 0, static_cast<int>(bytes > 0x7fffffff ? 0x7fffffff : bytes), 0, L, 1);
}

static int check_dense(const char* op, const void* W, int64_t ldw, const void* X, int64_t ldx,
                       int M, const void* Y, int N, int K) {
  if (!W || !X || !Y) return fail(WOBS_ERR_INVALID_ARG, "%s: null pointer", op);
  if (M < 1 || M > WOBS_MAX_M) return fail(WOBS_ERR_INVALID_ARG, "%s: M=%d outside 1..%d", op, M, WOBS_MAX_M);
  if (N < 1 || K < 8 || (K % 8)) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "%s: N=%d K=%d (K must be a positive multiple of 8)", op, N, K);
  if (ldw < K || (M > 1 && ldx < K)) return fail(WOBS_ERR_INVALID_ARG, "%s: pitch smaller than K", op);
  if (!aligned16(W) || !aligned16(X) || (ldw % 8) || (M > 1 && (ldx % 8)))
    return fail(WOBS_ERR_MISALIGNED, "%s: W/X rows must be 16-byte aligned", op);
  if (!aligned4(Y)) return fail(WOBS_ERR_MISALIGNED, "%s: output not aligned", op);
  return WOBS_OK;
}

}  // extern "C"

namespace wobs {
int check_dense_args(const char* op, const void* W, int64_t ldw, const void* X, int64_t ldx, int M,
                     const void* Y, int N, int K) {
  return check_dense(op, W, ldw, X, ldx, M, Y, N, K);
}
}  // namespace wobs

extern "C" {

int wobs_gemv_f16(const void* W, int64_t ldw, const void* X, int64_t ldx, int M, void* Y, int N,
                  int K, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_dense("gemv_f16", W, ldw, X, ldx, M, Y, N, K);
  if (rc) return rc;
  Prepared p;
  rc = prepare_ws(WOBS_OP_GEMV_F16, M, N, K, nullptr, ws, ws_bytes, &p);
  if (rc) return rc;
  wobs::Launch L;
  cudaError_t e = wobs::launch_gemv_dense(0, W, ldw, X, ldx, M, Y, 0, N, K, p.sk, p.am,
                                          static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "gemv_f16", M, N, K, L, p.sk.splits);
}

int wobs_gemv_bf16(const void* W, int64_t ldw, const void* X, int64_t ldx, int M, float* logits,
                   int64_t* argmax, int N, int K, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_dense("gemv_bf16", W, ldw, X, ldx, M, logits, N, K);
  if (rc) return rc;
  if (argmax && (reinterpret_cast<uintptr_t>(argmax) & 7u))
    return fail(WOBS_ERR_MISALIGNED, "gemv_bf16: argmax not 8-byte aligned");
  Prepared p;
  rc = prepare_ws(WOBS_OP_GEMV_BF16, M, N, K, argmax, ws, ws_bytes, &p);
  if (rc) return rc;
  wobs::Launch L;
  cudaError_t e = wobs::launch_gemv_dense(1, W, ldw, X, ldx, M, logits, 1, N, K, p.sk, p.am,
                                          static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "gemv_bf16", M, N, K, L, p.sk.splits);
}

int wobs_quantize_q8_1(const float* X, int64_t ldx, int M, int K, void* xq, void* stream) {
  if (!X || !xq) return fail(WOBS_ERR_INVALID_ARG, "quantize_q8_1: null pointer");
  if (M < 1 || M > WOBS_MAX_M) return fail(WOBS_ERR_INVALID_ARG, "quantize_q8_1: M=%d outside 1..%d", M, WOBS_MAX_M);
  if (K < 32 || (K % 32)) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "quantize_q8_1: K=%d not a positive multiple of 32", K);
  if (ldx < K) return fail(WOBS_ERR_INVALID_ARG, "quantize_q8_1: ldx < K");
  if (!aligned16(X) || (ldx % 4)) return fail(WOBS_ERR_MISALIGNED, "quantize_q8_1: X rows must be 16-byte aligned");
  if (!aligned4(xq)) return fail(WOBS_ERR_MISALIGNED, "quantize_q8_1: xq not 4-byte aligned");
  wobs::Launch L;
  cudaError_t e = wobs::launch_quantize_q8_1(X, ldx, M, K, xq, static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "quantize_q8_1", M, 0, K, L, 1);
}

int wobs_quantize_q4_0(const float* W, int64_t ldw, int N, int K, uint8_t* qs, void* d,
                       void* stream) {
  if (!W || !qs || !d) return fail(WOBS_ERR_INVALID_ARG, "quantize_q4_0: null pointer");
  if (N < 1 || K < 32 || (K % 32)) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "quantize_q4_0: N=%d K=%d", N, K);
  if (ldw < K) return fail(WOBS_ERR_INVALID_ARG, "quantize_q4_0: ldw < K");
  if (!aligned4(W) || !aligned16(qs) || (reinterpret_cast<uintptr_t>(d) & 1u))
    return fail(WOBS_ERR_MISALIGNED, "quantize_q4_0: misaligned pointer");
  wobs::Launch L;
  cudaError_t e = wobs::launch_quantize_q4_0(W, ldw, N, K, qs, d, static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "quantize_q4_0", 0, N, K, L, 1);
}

int wobs_quantize_nf4(const void* W, int64_t ldw, int N, int K, const float* codebook,
                      uint8_t* qs, float* absmax, void* stream) {
  if (!W || !codebook || !qs || !absmax) return fail(WOBS_ERR_INVALID_ARG, "quantize_nf4: null pointer");
  if (N < 1 || K < 64 || (K % 64)) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "quantize_nf4: N=%d K=%d", N, K);
  if (ldw < K || (ldw % 2)) return fail(WOBS_ERR_INVALID_ARG, "quantize_nf4: ldw");
  if (!aligned4(W) || !aligned4(absmax)) return fail(WOBS_ERR_MISALIGNED, "quantize_nf4: misaligned pointer");
  wobs::Codebook16 cb;
  std::memcpy(cb.v, codebook, sizeof(cb.v));
  wobs::Launch L;
  cudaError_t e = wobs::launch_quantize_nf4(W, ldw, N, K, cb, qs, absmax, static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "quantize_nf4", 0, N, K, L, 1);
}

int wobs_gemv_q4_0_q8_1(const uint8_t* qs, const void* d, const void* xq, int M, float* y,
                        int64_t* argmax, int N, int K, void* ws, size_t ws_bytes, void* stream) {
  if (!qs || !d || !xq || !y) return fail(WOBS_ERR_INVALID_ARG, "gemv_q4_0_q8_1: null pointer");
  if (M < 1 || M > WOBS_MAX_M) return fail(WOBS_ERR_INVALID_ARG, "gemv_q4_0_q8_1: M=%d outside 1..%d", M, WOBS_MAX_M);
  if (N < 1 || K < 32 || (K % 32)) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "gemv_q4_0_q8_1: N=%d K=%d (K must be a positive multiple of 32)", N, K);
  if (!aligned16(qs) || (reinterpret_cast<uintptr_t>(d) & 1u) || !aligned4(xq) || !aligned4(y))
    return fail(WOBS_ERR_MISALIGNED, "gemv_q4_0_q8_1: misaligned pointer");
  if (argmax && (reinterpret_cast<uintptr_t>(argmax) & 7u))
    return fail(WOBS_ERR_MISALIGNED, "gemv_q4_0_q8_1: argmax not 8-byte aligned");
  Prepared p;
  int rc = prepare_ws(WOBS_OP_GEMV_Q4_0_Q8_1, M, N, K, argmax, ws, ws_bytes, &p);
  if (rc) return rc;
  wobs::Launch L;
  cudaError_t e;
  // 5..32 columns: the tcgen05 kernel where its plan applies (TMA needs a
  // 16-byte aligned scale plane); otherwise the CUDA-core / mma.sync kernels
  const bool tc = M >= 5 && !env_splits() && wobs::q4_tc_enabled() && aligned16(d) &&
                  wobs::q4_tc_plan(M, N, K).ok;
  if (tc)
    e = wobs::launch_q4_tc(qs, d, xq, M, y, N, K, p.sk, p.am, static_cast<cudaStream_t>(stream), &L);
  else
    e = wobs::launch_gemv_q4_0_q8_1(qs, d, xq, M, y, N, K, p.sk, p.am,
                                    static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "gemv_q4_0_q8_1", M, N, K, L, p.sk.splits);
}

int wobs_gemv_q4_0_f32(const uint8_t* qs, const void* d, const float* X, void* xq_out, float* y,
                       int64_t* argmax, int N, int K, void* ws, size_t ws_bytes, void* stream) {
  const int M = 1;
  if (!qs || !d || !X || !y) return fail(WOBS_ERR_INVALID_ARG, "gemv_q4_0_f32: null pointer");
  if (xq_out && !aligned4(xq_out)) return fail(WOBS_ERR_MISALIGNED, "gemv_q4_0_f32: xq_out not 4-byte aligned");
  if (N < 1 || K < 256 || (K % 256)) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "gemv_q4_0_f32: N=%d K=%d (K must be a positive multiple of 256)", N, K);
  if (!aligned16(X) || !aligned16(qs) || !aligned16(d) || !aligned4(y))
    return fail(WOBS_ERR_MISALIGNED, "gemv_q4_0_f32: X, qs and d must be 16-byte aligned, y 4-byte aligned");
  if (argmax && (reinterpret_cast<uintptr_t>(argmax) & 7u))
    return fail(WOBS_ERR_MISALIGNED, "gemv_q4_0_f32: argmax not 8-byte aligned");
  if (!wobs::q4_0_f32_fused_applies(d, M, K))
    return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "gemv_q4_0_f32: K=%d too long for the shared-memory activation planes", K);
  Prepared p;
  int rc = prepare_ws(WOBS_OP_GEMV_Q4_0_F32, M, N, K, argmax, ws, ws_bytes, &p);
  if (rc) return rc;
  wobs::Launch L;
  cudaError_t e = wobs::launch_gemv_q4_0_f32_fused(qs, d, X, xq_out, y, N, K, p.am,
                                                   static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "gemv_q4_0_f32", M, N, K, L, 1);
}

int wobs_gemv_q8_0_f32(const int8_t* qs, const void* d, const float* X, void* xq_out, float* y,
                       int64_t* argmax, int N, int K, void* ws, size_t ws_bytes, void* stream) {
  const int M = 1;
  if (!qs || !d || !X || !y) return fail(WOBS_ERR_INVALID_ARG, "gemv_q8_0_f32: null pointer");
  if (xq_out && !aligned4(xq_out)) return fail(WOBS_ERR_MISALIGNED, "gemv_q8_0_f32: xq_out not 4-byte aligned");
  if (N < 1 || K < 256 || (K % 256)) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "gemv_q8_0_f32: N=%d K=%d (K must be a positive multiple of 256)", N, K);
  if (!aligned16(X) || !aligned16(qs) || !aligned16(d) || !aligned4(y))
    return fail(WOBS_ERR_MISALIGNED, "gemv_q8_0_f32: X, qs and d must be 16-byte aligned, y 4-byte aligned");
  if (argmax && (reinterpret_cast<uintptr_t>(argmax) & 7u))
    return fail(WOBS_ERR_MISALIGNED, "gemv_q8_0_f32: argmax not 8-byte aligned");
  if (!wobs::q8_0_f32_fused_applies(K))
    return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "gemv_q8_0_f32: K=%d too long for the shared-memory activation planes", K);
  Prepared p;
  int rc = prepare_ws(WOBS_OP_GEMV_Q8_0_F32, M, N, K, argmax, ws, ws_bytes, &p);
  if (rc) return rc;
  wobs::Launch L;
  cudaError_t e = wobs::launch_gemv_q8_0_f32_fused(qs, d, X, xq_out, y, N, K, p.am,
                                                   static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "gemv_q8_0_f32", M, N, K, L, 1);
}

int wobs_quantize_q8_0(const float* W, int64_t ldw, int N, int K, int8_t* qs, void* d,
                       void* stream) {
  if (!W || !qs || !d) return fail(WOBS_ERR_INVALID_ARG, "quantize_q8_0: null pointer");
  if (N < 1 || K < 32 || (K % 32)) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "quantize_q8_0: N=%d K=%d", N, K);
  if (ldw < K) return fail(WOBS_ERR_INVALID_ARG, "quantize_q8_0: ldw < K");
  if (!aligned4(W) || (reinterpret_cast<uintptr_t>(d) & 1u))
    return fail(WOBS_ERR_MISALIGNED, "quantize_q8_0: misaligned pointer");
  wobs::Launch L;
  cudaError_t e = wobs::launch_quantize_q8_0(W, ldw, N, K, qs, d, static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "quantize_q8_0", 0, N, K, L, 1);
}

int wobs_gemv_q8_0_q8_1(const int8_t* qs, const void* d, const void* xq, int M, float* y,
                        int64_t* argmax, int N, int K, void* ws, size_t ws_bytes, void* stream) {
  if (!qs || !d || !xq || !y) return fail(WOBS_ERR_INVALID_ARG, "gemv_q8_0_q8_1: null pointer");
  if (M < 1 || M > WOBS_MAX_M) return fail(WOBS_ERR_INVALID_ARG, "gemv_q8_0_q8_1: M=%d outside 1..%d", M, WOBS_MAX_M);
  if (N < 1 || K < 256 || (K % 256))
    return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "gemv_q8_0_q8_1: N=%d K=%d (K must be a positive multiple of 256)", N, K);
  if (!aligned16(qs) || !aligned16(d) || !aligned4(xq) || !aligned4(y))
    return fail(WOBS_ERR_MISALIGNED, "gemv_q8_0_q8_1: misaligned pointer");
  if (argmax && (reinterpret_cast<uintptr_t>(argmax) & 7u))
    return fail(WOBS_ERR_MISALIGNED, "gemv_q8_0_q8_1: argmax not 8-byte aligned");
  Prepared p;
  int rc = prepare_ws(WOBS_OP_GEMV_Q8_0_Q8_1, M, N, K, argmax, ws, ws_bytes, &p);
  if (rc) return rc;
  if (wobs::q8_0_columns_per_launch(K) == 0)
    return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "gemv_q8_0_q8_1: K=%d: one column's activation blocks do not fit in shared memory", K);
  wobs::Launch L;
  cudaError_t e = wobs::launch_gemv_q8_0_q8_1(qs, d, xq, M, y, N, K, p.am,
                                              static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "gemv_q8_0_q8_1", M, N, K, L, 1);
}

int wobs_gemv_nf4(const uint8_t* qs, const float* absmax, const float* codebook, const void* X,
                  int64_t ldx, int M, void* Y, int64_t* argmax, int N, int K, void* ws,
                  size_t ws_bytes, void* stream) {
  if (!qs || !absmax || !codebook || !X || !Y) return fail(WOBS_ERR_INVALID_ARG, "gemv_nf4: null pointer");
  if (M < 1 || M > WOBS_MAX_M) return fail(WOBS_ERR_INVALID_ARG, "gemv_nf4: M=%d outside 1..%d", M, WOBS_MAX_M);
  if (N < 1 || K < 64 || (K % 64) || K > 32768)
    return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "gemv_nf4: N=%d K=%d (K a multiple of 64, at most 32768)", N, K);
  if (M > 1 && ldx < K) return fail(WOBS_ERR_INVALID_ARG, "gemv_nf4: ldx < K");
  if (!aligned16(qs) || !aligned4(absmax) || (reinterpret_cast<uintptr_t>(X) & 1u) ||
      (reinterpret_cast<uintptr_t>(Y) & 1u))
    return fail(WOBS_ERR_MISALIGNED, "gemv_nf4: misaligned pointer");
  if (argmax && (reinterpret_cast<uintptr_t>(argmax) & 7u))
    return fail(WOBS_ERR_MISALIGNED, "gemv_nf4: argmax not 8-byte aligned");
  Prepared p;
  int rc = prepare_ws(WOBS_OP_GEMV_NF4, M, N, K, argmax, ws, ws_bytes, &p);
  if (rc) return rc;
  wobs::Codebook16 cb;
  std::memcpy(cb.v, codebook, sizeof(cb.v));
  wobs::Launch L;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = M == 1 ? wobs::launch_gemv_nf4(qs, absmax, cb, X, Y, N, K, p.am, st, &L)
                         : wobs::launch_gemv_nf4_mc(qs, absmax, cb, X, M > 1 ? ldx : K, M, Y, N, K, p.sk,
                                                    p.am, st, &L);
  return finish_launch(e, "gemv_nf4", M, N, K, L, p.sk.splits);
}

int wobs_dequantize_nf4(const uint8_t* qs, const float* absmax, const float* codebook, int N, int K,
                        void* W, int64_t ldw, void* stream) {
  if (!qs || !absmax || !codebook || !W) return fail(WOBS_ERR_INVALID_ARG, "dequantize_nf4: null pointer");
  if (N < 1 || K < 64 || (K % 64)) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "dequantize_nf4: N=%d K=%d", N, K);
  if (ldw < K || (ldw % 2)) return fail(WOBS_ERR_INVALID_ARG, "dequantize_nf4: ldw");
  if (!aligned4(absmax) || !aligned4(W)) return fail(WOBS_ERR_MISALIGNED, "dequantize_nf4: misaligned pointer");
  wobs::Codebook16 cb;
  std::memcpy(cb.v, codebook, sizeof(cb.v));
  wobs::Launch L;
  cudaError_t e = wobs::launch_dequantize_nf4(qs, absmax, cb, N, K, W, ldw, static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "dequantize_nf4", 0, N, K, L, 1);
}

static int argcmp(const char* op, bool is_min, int dtype, const void* X, int64_t ldx, int M, int N,
                  int64_t* out, void* ws, size_t ws_bytes, void* stream) {
  if (!X || !out) return fail(WOBS_ERR_INVALID_ARG, "%s: null pointer", op);
  if (dtype < WOBS_DTYPE_F16 || dtype > WOBS_DTYPE_F32)
    return fail(WOBS_ERR_INVALID_ARG, "%s: dtype %d (1 fp16, 2 bf16, 3 fp32)", op, dtype);
  if (M < 1 || M > WOBS_ARGCMP_MAX_M) return fail(WOBS_ERR_INVALID_ARG, "%s: M=%d outside 1..%d", op, M, WOBS_ARGCMP_MAX_M);
  if (N < 1 || N > WOBS_ARGCMP_MAX_N) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "%s: N=%d outside 1..%d", op, N, WOBS_ARGCMP_MAX_N);
  const int es = dtype == WOBS_DTYPE_F32 ? 4 : 2;
  if (M > 1 && ldx < N) return fail(WOBS_ERR_INVALID_ARG, "%s: ldx < N", op);
  if (reinterpret_cast<uintptr_t>(X) % es)
    return fail(WOBS_ERR_MISALIGNED, "%s: X not aligned to its element size", op);
  if (reinterpret_cast<uintptr_t>(out) & 7u) return fail(WOBS_ERR_MISALIGNED, "%s: out not 8-byte aligned", op);
  const wobs::ArgcmpPlan p = wobs::plan_argcmp(es, M, N, env_splits());
  if (!p.warp_rows && static_cast<int64_t>(M) * p.splits > 0x7FFFFFFFll)
    return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "%s: M x slices exceeds the grid", op);
  uint64_t* keys = nullptr;
  unsigned* counters = nullptr;
  if (!p.warp_rows && p.splits > 1) {
    const size_t need = (12ull * M + 15ull) & ~15ull;
    if (!ws) return fail(WOBS_ERR_INVALID_ARG, "%s: workspace required (%zu bytes) but ws is NULL", op, need);
    if (!aligned16(ws)) return fail(WOBS_ERR_MISALIGNED, "%s: workspace must be 16-byte aligned", op);
    if (ws_bytes < need)
      return fail(WOBS_ERR_WORKSPACE_TOO_SMALL, "%s: workspace %zu bytes < %zu needed", op, ws_bytes, need);
    keys = static_cast<uint64_t*>(ws);
    counters = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(ws) + 8ull * M);
  }
  wobs::Launch L;
  cudaError_t e = wobs::launch_argcmp(dtype, is_min, X, M > 1 ? ldx : N, M, N, p, out, keys, counters,
                                      static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, op, M, N, 0, L, p.warp_rows ? 1 : p.splits);
}

int wobs_argmax(int dtype, const void* X, int64_t ldx, int M, int N, int64_t* out, void* ws,
                size_t ws_bytes, void* stream) {
  return argcmp("argmax", false, dtype, X, ldx, M, N, out, ws, ws_bytes, stream);
}

int wobs_argmin(int dtype, const void* X, int64_t ldx, int M, int N, int64_t* out, void* ws,
                size_t ws_bytes, void* stream) {
  return argcmp("argmin", true, dtype, X, ldx, M, N, out, ws, ws_bytes, stream);
}

int wobs_q4_0_q8_1_blockdots(const uint8_t* qs, const void* xq, int M, int N, int K, int32_t* out,
                             void* stream) {
  if (!qs || !xq || !out) return fail(WOBS_ERR_INVALID_ARG, "q4_0_q8_1_blockdots: null pointer");
  if (M < 1 || M > WOBS_MAX_M) return fail(WOBS_ERR_INVALID_ARG, "q4_0_q8_1_blockdots: M=%d", M);
  if (N < 1 || K < 32 || (K % 32)) return fail(WOBS_ERR_UNSUPPORTED_SHAPE, "q4_0_q8_1_blockdots: N=%d K=%d", N, K);
  if (!aligned16(qs) || !aligned4(xq) || !aligned4(out))
    return fail(WOBS_ERR_MISALIGNED, "q4_0_q8_1_blockdots: misaligned pointer");
  wobs::Launch L;
  cudaError_t e = wobs::launch_q4_0_q8_1_blockdots(qs, xq, M, N, K, out, static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "q4_0_q8_1_blockdots", M, N, K, L, 1);
}

int wobs_selftest_wait_timeout(long long limit_cycles, void* stream) {
  if (limit_cycles < 1 || limit_cycles > 1000000000ll)
    return fail(WOBS_ERR_INVALID_ARG, "selftest_wait_timeout: limit %lld outside 1..1e9 cycles", limit_cycles);
  wobs::Launch L;
  cudaError_t e = wobs::launch_wait_timeout(limit_cycles, static_cast<cudaStream_t>(stream), &L);
  return finish_launch(e, "selftest_wait_timeout", 0, 0, 0, L, 1);
}

int wobs_error_word(void* stream, int* host_out) {
  if (!host_out) return fail(WOBS_ERR_INVALID_ARG, "error_word: null pointer");
  cudaError_t e = wobs::read_and_clear_error_word(static_cast<cudaStream_t>(stream), host_out);
  if (e != cudaSuccess) return cuda_fail(e, "error_word", WOBS_ERR_CUDA);
  if (*host_out != 0)
    return fail(WOBS_ERR_DEVICE_TIMEOUT, "error_word: a bounded device wait gave up (code %d)",
                *host_out);
  g_err[0] = '\0';
  return WOBS_OK;
}

}  // extern "C"
