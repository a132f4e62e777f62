// staging.cu -- moving the host-buffer entry point's inputs and outputs
// between page-locked host memory and the device with SM loads and stores.
//
// A page-locked (CUDA-registered) host buffer is mapped into the device's
// address space, so kernels read and write it in place over the CPU-GPU link.
// On GB300 an SM-driven copy of such a buffer held 211 GB/s run after run,
// while cudaMemcpyAsync of the same buffer, issued after some seconds of
// HBM-bound kernels, fell step by step to 15 GB/s (and came back only after an
// SM-driven pass had touched the buffer). The prompt phase is bound by this
// copy, so the library moves page-locked buffers with its own kernel.
#include "kvevict_internal.cuh"

namespace kvx {
namespace {

constexpr int kCopyThreads = 256;
// The background form: one 128-thread block per SM, at most 32 registers a
// thread and 24 KB of shared memory, so that a block fits beside two CTAs of
// the prompt scorer (2 x 320 threads at up to 96 registers, 99 KB of shared
// memory each) and the copy of the next prompt chunk runs under the scoring
// of the current one.
constexpr int kBgThreads = 128;

// dst[i] = src[i] for i < n, four independent loads in flight per thread.
template <typename W, int THREADS, int MIN_BLOCKS>
__global__ void __launch_bounds__(THREADS, MIN_BLOCKS) copy_words_kernel(const W* __restrict__ src,
                                                                        W* __restrict__ dst, size_t n) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const W a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

// Background copy of 16-byte words through a 3-stage shared-memory ring with
// asynchronous global->shared copies (cp.async): the bytes in flight are held
// in shared memory, not registers, so a 128-thread block keeps 16-24 KB of
// reads in flight instead of the 8 KB four registers' worth of loads a thread
// allows (the prompt from page-locked memory: 64-78 ms -> 57 ms on the
// large-context workload). Each thread copies and later stores its own words,
// so no barrier is needed; a stage is refilled only after the thread has
// stored what it read from it.
constexpr int kAsyncStages = 3;
constexpr int kAsyncPer = 4;                                   // words per thread per chunk
constexpr int kAsyncChunk = kBgThreads * kAsyncPer;            // words per chunk (8 KB)
__device__ __forceinline__ void cp_async16(uint32_t s, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(g) : "memory");
}
__global__ void __launch_bounds__(kBgThreads, 16) copy_async_kernel(const uint4* __restrict__ src,
                                                                  uint4* __restrict__ dst, size_t n) {
  extern __shared__ __align__(16) uint4 ring[];
  const size_t nchunks = (n + kAsyncChunk - 1) / kAsyncChunk;
  const size_t mine = nchunks > blockIdx.x ? (nchunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const uint32_t ring0 = (uint32_t)__cvta_generic_to_shared(ring);
  for (size_t k = 0; k < mine + kAsyncStages - 1; ++k) {
    if (k < mine) {
      const size_t c = blockIdx.x + k * gridDim.x;
      const int st = (int)(k % kAsyncStages);
#pragma unroll
      for (int u = 0; u < kAsyncPer; ++u) {
        const size_t i = c * kAsyncChunk + (size_t)u * kBgThreads + threadIdx.x;
        const uint32_t so = ring0 + (uint32_t)((st * kAsyncChunk + u * kBgThreads + threadIdx.x) * 16);
        if (i < n) cp_async16(so, src + i);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (k + 1 >= (size_t)kAsyncStages) {   // chunk k - (kAsyncStages - 1) has landed
      asm volatile("cp.async.wait_group %0;" ::"n"(kAsyncStages - 1) : "memory");
      const size_t kk = k + 1 - kAsyncStages;
      const size_t c = blockIdx.x + kk * gridDim.x;
      const int st = (int)(kk % kAsyncStages);
#pragma unroll
      for (int u = 0; u < kAsyncPer; ++u) {
        const size_t i = c * kAsyncChunk + (size_t)u * kBgThreads + threadIdx.x;
        if (i < n) dst[i] = ring[st * kAsyncChunk + u * kBgThreads + threadIdx.x];
      }
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
}

template <typename W>
cudaError_t launch_words(const void* src, void* dst, size_t bytes, int sms, bool background, cudaStream_t s) {
  const size_t n = bytes / sizeof(W);
  const int threads = background ? kBgThreads : kCopyThreads;
  const size_t want = (n + 4 * (size_t)threads - 1) / (4 * (size_t)threads);
  const size_t cap = (size_t)std::max(1, sms) * (background ? 1 : 4);
  const unsigned blocks = (unsigned)std::max<size_t>(1, std::min<size_t>(want, cap));
  if (background)
    copy_words_kernel<W, kBgThreads, 16><<<blocks, kBgThreads, 0, s>>>(static_cast<const W*>(src),
                                                                       static_cast<W*>(dst), n);
  else
    copy_words_kernel<W, kCopyThreads, 1><<<blocks, kCopyThreads, 0, s>>>(static_cast<const W*>(src),
                                                                          static_cast<W*>(dst), n);
  return cudaGetLastError();
}

}  // namespace

void* mapped_host(const void* p, size_t bytes) {
  if (!p || bytes == 0) return nullptr;
  cudaPointerAttributes a0{}, a1{};
  if (cudaPointerGetAttributes(&a0, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (a0.type != cudaMemoryTypeHost || !a0.devicePointer) return nullptr;
  const char* last = static_cast<const char*>(p) + (bytes - 1);
  if (cudaPointerGetAttributes(&a1, last) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (a1.type != cudaMemoryTypeHost ||
      static_cast<const char*>(a1.devicePointer) != static_cast<const char*>(a0.devicePointer) + (bytes - 1))
    return nullptr;
  return a0.devicePointer;
}

cudaError_t launch_copy(const void* src, void* dst, size_t bytes, int sms, bool background, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  const uintptr_t al = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | (uintptr_t)bytes;
  if (background && (al & 15) == 0) {
    const size_t smem = (size_t)kAsyncStages * kAsyncChunk * 16;
    copy_async_kernel<<<(unsigned)std::max(1, sms), kBgThreads, smem, s>>>(static_cast<const uint4*>(src),
                                                                          static_cast<uint4*>(dst), bytes / 16);
    return cudaGetLastError();
  }
  if ((al & 15) == 0) return launch_words<uint4>(src, dst, bytes, sms, background, s);
  if ((al & 7) == 0) return launch_words<uint2>(src, dst, bytes, sms, background, s);
  if ((al & 3) == 0) return launch_words<uint32_t>(src, dst, bytes, sms, background, s);
  if ((al & 1) == 0) return launch_words<uint16_t>(src, dst, bytes, sms, background, s);
  return launch_words<uint8_t>(src, dst, bytes, sms, background, s);
}

}  // namespace kvx
