// hostio.cu -- the host copies of a decode step issued as kernels.
//
// A step that starts from host memory moves a few hundred KB each way (its
// packed inputs up, out and lse down).  At that size a copy-engine transfer
// costs several microseconds of fixed latency on each side of the decode; a
// kernel that reads or writes page-locked host memory directly over the host
// link costs about one link round trip, and, launched as a programmatic
// dependent like every libdsa kernel, it is scheduled while the previous kernel
// drains.  Only host memory the device can address (page-locked and mapped)
// takes this path; any other pointer goes through cudaMemcpyAsync.
#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

// dst[0, bytes) = src[0, bytes); 16-byte vectors when both are 16-byte aligned.
__global__ void __launch_bounds__(256)
    copy_kernel(unsigned char* dst, const unsigned char* src, size_t bytes, int vec) {
  griddep_wait();
  griddep_launch_dependents();
  const size_t tid = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nthreads = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t done = 0;
  if (vec) {
    const size_t n16 = bytes / 16;
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    for (size_t i = tid; i < n16; i += nthreads) d4[i] = s4[i];
    done = n16 * 16;
  }
  for (size_t i = done + tid; i < bytes; i += nthreads) dst[i] = src[i];
}

// The device's address of host memory p, or null when p is not page-locked
// memory the device can address.
void* device_view_of_host(const void* p) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
    cudaGetLastError();  // not an error of the call: take the copy engine
    return nullptr;
  }
  return attr.type == cudaMemoryTypeHost ? attr.devicePointer : nullptr;
}

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  const int vec =
      ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) % 16) == 0;
  const size_t items = vec ? bytes / 16 + bytes % 16 : bytes;
  size_t blocks = (items + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  return launch_pdl(copy_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                    static_cast<unsigned char*>(dst), static_cast<const unsigned char*>(src),
                    bytes, vec);
}

}  // namespace

#ifndef DSA_HOSTIO_KERNEL
#define DSA_HOSTIO_KERNEL 1  // 0: every host copy through cudaMemcpyAsync
#endif

cudaError_t copy_host_to_device(void* dev, const void* host, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  const void* view = DSA_HOSTIO_KERNEL ? device_view_of_host(host) : nullptr;
  return view != nullptr ? launch_copy(dev, view, bytes, s)
                         : cudaMemcpyAsync(dev, host, bytes, cudaMemcpyHostToDevice, s);
}

cudaError_t copy_device_to_host(void* host, const void* dev, size_t bytes, cudaStream_t s) {
  if (bytes == 0) return cudaSuccess;
  void* view = DSA_HOSTIO_KERNEL ? device_view_of_host(host) : nullptr;
  return view != nullptr ? launch_copy(view, dev, bytes, s)
                         : cudaMemcpyAsync(host, dev, bytes, cudaMemcpyDeviceToHost, s);
}

}  // namespace dsa
