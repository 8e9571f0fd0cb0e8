// wobs_gemv_bf16_noalloc: the bf16 GEMV with fused argmax, its workspace
// taken from a fixed scratch array inside the library.
//
// Some callers cannot hand the library a workspace because they may not
// allocate device memory when they call it: inference engines that reserve
// their whole memory budget at start-up and carve it up with their own
// allocator, plugins inside a host process that owns every device
// allocation, and decode loops that cannot pay for a cudaMalloc/cudaFree
// (which may synchronise the device).  For them this entry point needs no
// workspace argument and calls no allocating routine.
//
// The scratch is a file-scope __device__ array of kScratchBytes: every GPU
// that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address, so the device address is
// looked up once per device with cudaGetSymbolAddress (on the first call
// made with that device current; make that first call before any stream
// capture) and kept: a cudaDeviceReset invalidates it.  All calls share the
// one array, which keeps the last call's contents: the counters and keys
// are cleared on the call's stream before every launch, and calls that
// overlap on the GPU (different streams, no ordering) race on it.
#include <mutex>

#include "../../include/wobs.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = WOBS_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size");

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once).
int scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return wobs::set_error(WOBS_ERR_CUDA, "gemv_bf16_noalloc: no usable current device");
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return wobs::set_error(WOBS_ERR_CUDA, "gemv_bf16_noalloc: cudaGetSymbolAddress failed");
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return WOBS_OK;
}

}  // namespace

extern "C" int wobs_gemv_bf16_noalloc(const void* W, int64_t ldw, const void* X, int64_t ldx,
                                      int M, float* logits, int64_t* argmax, int N, int K,
                                      void* stream) {
  int rc = wobs::check_dense_args("gemv_bf16_noalloc", W, ldw, X, ldx, M, logits, N, K);
  if (rc) return rc;
  if (argmax && (reinterpret_cast<uintptr_t>(argmax) & 7u))
    return wobs::set_error(WOBS_ERR_MISALIGNED, "gemv_bf16_noalloc: argmax not 8-byte aligned");
  size_t zero_prefix = 0;
  const size_t need = wobs::workspace_layout(WOBS_OP_GEMV_BF16, M, N, K, &zero_prefix);
  if (need > kScratchBytes)
    return wobs::set_error(WOBS_ERR_WORKSPACE_TOO_SMALL,
                           "gemv_bf16_noalloc: this shape needs more scratch than the library's "
                           "fixed WOBS_NOALLOC_SCRATCH_BYTES; use wobs_gemv_bf16 with a workspace");
  void* ws = nullptr;
  rc = scratch_on_current_device(&ws);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws, 0, zero_prefix, st);
  if (e != cudaSuccess) return wobs::report_launch(e, "gemv_bf16_noalloc", M, N, K, wobs::Launch{}, 1);
  wobs::SplitArgs sk;
  wobs::ArgmaxArgs am;
  rc = wobs::prepare_workspace(WOBS_OP_GEMV_BF16, M, N, K, argmax, ws, kScratchBytes, &sk, &am);
  if (rc) return rc;
  wobs::Launch L;
  e = wobs::launch_gemv_dense(1, W, ldw, X, ldx, M, logits, 1, N, K, sk, am, st, &L);
  return wobs::report_launch(e, "gemv_bf16_noalloc", M, N, K, L, sk.splits);
}
