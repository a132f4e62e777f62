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
// thread, so that a block fits beside two CTAs of the prompt scorer (2 x 320
// threads at up to 96 registers, about 100 KB of shared memory each) and the
// copy of the next prompt chunk runs under the scoring of the current one.
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
  if ((al & 15) == 0) return launch_words<uint4>(src, dst, bytes, sms, background, s);
  if ((al & 7) == 0) return launch_words<uint2>(src, dst, bytes, sms, background, s);
  if ((al & 3) == 0) return launch_words<uint32_t>(src, dst, bytes, sms, background, s);
  if ((al & 1) == 0) return launch_words<uint16_t>(src, dst, bytes, sms, background, s);
  return launch_words<uint8_t>(src, dst, bytes, sms, background, s);
}

}  // namespace kvx
