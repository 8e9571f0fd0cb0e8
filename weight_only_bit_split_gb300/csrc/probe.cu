// Streaming-read ceiling probe.
//
// batch1-cdna README, "01-ceiling": a grid-stride read of a buffer much
// larger than the last-level cache, vectorised, with the result folded into
// a scalar so that no load can be removed; grid size and load type are
// swept and the best figure is the denominator of every bandwidth-
// utilisation number.  Here the fold is XOR (exactly checkable against the
// oracle) and the load types are the sm_103a ones: L1-cached 16-byte
// loads, 16- and 32-byte loads with L1 no-allocate + L2 evict-first, and
// bulk asynchronous copies into a shared-memory ring (the TMA engine).
#include <cstdio>

#include "common.cuh"
#include "tma.cuh"

namespace wobs {

__device__ int g_error_word = 0;

namespace {

constexpr int kProbeThreads = 256;
constexpr int kUnroll = 8;

__device__ __forceinline__ uint32_t xor4(uint4 v) { return v.x ^ v.y ^ v.z ^ v.w; }

__device__ __forceinline__ void publish_xor(uint32_t v, uint32_t* out) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v ^= __shfl_xor_sync(0xffffffffu, v, o);
  __shared__ uint32_t s[kProbeThreads / 32];
  if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int i = 0; i < kProbeThreads / 32; ++i) t ^= s[i];
    atomicXor(out, t);
  }
}

// Variants 0 and 1: one 16-byte load per thread-iteration, kUnroll in flight.
template <bool kStream>
__global__ void __launch_bounds__(kProbeThreads) probe16_kernel(const uint4* buf, size_t n16,
                                                                 uint32_t* out) {
  const uint64_t pol = l2_evict_first_policy();
  const size_t stride = static_cast<size_t>(gridDim.x) * kProbeThreads;
  size_t i = static_cast<size_t>(blockIdx.x) * kProbeThreads + threadIdx.x;
  uint32_t acc = 0;
  for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      v[u] = kStream ? ld_stream16(buf + i + u * stride, pol) : ld_nc16(buf + i + u * stride);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc ^= xor4(v[u]);
  }
  for (; i < n16; i += stride) acc ^= xor4(kStream ? ld_stream16(buf + i, pol) : ld_nc16(buf + i));
  publish_xor(acc, out);
}

// Variant 2: 32 bytes per thread-iteration (one 256-bit load, ld_stream32).
__global__ void __launch_bounds__(kProbeThreads) probe32_kernel(const uint4* buf, size_t n16,
                                                                 uint32_t* out) {
  const uint64_t pol = l2_evict_first_policy();
  const size_t n32 = n16 / 2;
  const size_t stride = static_cast<size_t>(gridDim.x) * kProbeThreads;
  size_t i = static_cast<size_t>(blockIdx.x) * kProbeThreads + threadIdx.x;
  uint32_t acc = 0;
  constexpr int U = kUnroll / 2;
  for (; i + (U - 1) * stride < n32; i += U * stride) {
    uint4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) ld_stream32(buf + 2 * (i + u * stride), pol, a[u], b[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) acc ^= xor4(a[u]) ^ xor4(b[u]);
  }
  for (; i < n32; i += stride) {
    uint4 a, b;
    ld_stream32(buf + 2 * i, pol, a, b);
    acc ^= xor4(a) ^ xor4(b);
  }
  // odd trailing 16-byte chunk
  if (blockIdx.x == 0 && threadIdx.x == 0 && (n16 & 1)) acc ^= xor4(ld_nc16(buf + n16 - 1));
  publish_xor(acc, out);
}

// Variant 3: cp.async.bulk (TMA, 1-D) into a ring of shared-memory stages.
constexpr int kBulkStages = 4;
constexpr int kBulkChunk = 32768;  // bytes per stage
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return smem_addr(p); }

__device__ __forceinline__ void bulk_issue(void* dst, const void* src, uint32_t bytes,
                                           uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__global__ void __launch_bounds__(kProbeThreads) probe_bulk_kernel(const uint8_t* buf,
                                                                    size_t bytes,
                                                                    uint32_t* out) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(8) uint64_t full[kBulkStages], empty[kBulkStages];
  __shared__ int s_abort;
  const size_t nchunks = bytes / kBulkChunk;
  // chunks of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
  const size_t mine = nchunks > blockIdx.x ? (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int nwarps = kProbeThreads / 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBulkStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(smem_u32(&full[s])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(&empty[s])), "r"(nwarps));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_abort = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (size_t i = 0; i < mine && i < kBulkStages; ++i)
      bulk_issue(ring + i * kBulkChunk, buf + (blockIdx.x + i * gridDim.x) * kBulkChunk,
                 kBulkChunk, &full[i]);
  }
  uint32_t acc = 0;
  size_t issued = mine < kBulkStages ? mine : kBulkStages;
  for (size_t i = 0; i < mine; ++i) {
    const int s = static_cast<int>(i % kBulkStages);
    const uint32_t ph = static_cast<uint32_t>((i / kBulkStages) & 1);
    const bool got = mbar_wait(&full[s], ph);
    if (!got) s_abort = 1;
    __syncwarp();
    if (__any_sync(0xffffffffu, !got || s_abort != 0)) break;   // warp-uniform exit
    const uint4* st = reinterpret_cast<const uint4*>(ring + s * kBulkChunk);
#pragma unroll
    for (int u = 0; u < kBulkChunk / 16 / kProbeThreads; ++u) acc ^= xor4(st[u * kProbeThreads + threadIdx.x]);
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(&empty[s])) : "memory");
    if (threadIdx.x == 0 && i + kBulkStages < mine) {
      if (!mbar_wait(&empty[s], ph)) { s_abort = 1; }
      if (!s_abort) {
        bulk_issue(ring + s * kBulkChunk,
                   buf + (blockIdx.x + (i + kBulkStages) * gridDim.x) * kBulkChunk, kBulkChunk,
                   &full[s]);
        ++issued;
      }
    }
  }
  if (threadIdx.x == 0 && s_abort) {
    atomicExch(&g_error_word, kErrProbeWait);
    // let copies still in flight land before the CTA's shared memory goes
    for (size_t i = 0; i < issued && i < kBulkStages; ++i) {
      size_t j = issued - 1 - i;
      mbar_wait(&full[j % kBulkStages], static_cast<uint32_t>((j / kBulkStages) & 1));
    }
  }
  // tail bytes beyond the last whole chunk: plain loads by CTA 0
  if (blockIdx.x == 0) {
    const uint4* t = reinterpret_cast<const uint4*>(buf + nchunks * kBulkChunk);
    const size_t nt = (bytes - nchunks * kBulkChunk) / 16;
    for (size_t k = threadIdx.x; k < nt; k += kProbeThreads) acc ^= xor4(ld_nc16(t + k));
  }
  publish_xor(acc, out);
}

}  // namespace

cudaError_t launch_bw_probe(const void* buf, size_t bytes, int grid, int variant,
                            uint32_t* xor_out, cudaStream_t st, Launch* info) {
  const size_t n16 = bytes / 16;
  const void* fn = nullptr;
  int smem = 0;
  switch (variant) {
    case 0: fn = reinterpret_cast<const void*>(probe16_kernel<false>); break;
    case 1: fn = reinterpret_cast<const void*>(probe16_kernel<true>); break;
    case 2: fn = reinterpret_cast<const void*>(probe32_kernel); break;
    default:
      fn = reinterpret_cast<const void*>(probe_bulk_kernel);
      smem = kBulkStages * kBulkChunk;
      break;
  }
  if (variant == 3) {
    cudaError_t e = cudaFuncSetAttribute(probe_bulk_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  if (grid <= 0) grid = device_sm_count() * max_resident_ctas(fn, kProbeThreads, smem);
  if (grid <= 0) grid = 1;
  info->grid_x = grid;
  info->block = kProbeThreads;
  info->smem = smem;
  switch (variant) {
    case 0:
      info->kernel = "probe16_l1";
      probe16_kernel<false><<<grid, kProbeThreads, 0, st>>>(static_cast<const uint4*>(buf), n16, xor_out);
      break;
    case 1:
      info->kernel = "probe16_stream";
      probe16_kernel<true><<<grid, kProbeThreads, 0, st>>>(static_cast<const uint4*>(buf), n16, xor_out);
      break;
    case 2:
      info->kernel = "probe32_stream";
      probe32_kernel<<<grid, kProbeThreads, 0, st>>>(static_cast<const uint4*>(buf), n16, xor_out);
      break;
    default:
      info->kernel = "probe_bulk";
      probe_bulk_kernel<<<grid, kProbeThreads, smem, st>>>(static_cast<const uint8_t*>(buf), bytes, xor_out);
      break;
  }
  return cudaGetLastError();
}

// Failure-path self test: one warp waits on an mbarrier that nothing
// arrives on, with a short bound; the wait gives up, the error word gets
// kErrSelfTestWait and the kernel returns normally (no trap, no hang).
__global__ void wait_timeout_kernel(long long limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0, limit);
  if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) atomicExch(&g_error_word, kErrSelfTestWait);
  // leave the barrier complete so nothing is pending at exit
  if (threadIdx.x == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_addr(&bar)) : "memory");
}

cudaError_t launch_wait_timeout(long long limit, cudaStream_t st, Launch* info) {
  info->grid_x = 1;
  info->block = 32;
  info->kernel = "wait_timeout";
  wait_timeout_kernel<<<1, 32, 0, st>>>(limit);
  return cudaGetLastError();
}

int* error_word_ptr() {
  static int* cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    cache[dev] = static_cast<int*>(p);
  }
  return cache[dev];
}

cudaError_t read_and_clear_error_word(cudaStream_t st, int* host_out) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(host_out, g_error_word, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyToSymbolAsync(g_error_word, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(st);
}

}  // namespace wobs
