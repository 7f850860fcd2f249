// residency.cuh -- where a pointer argument lives, as the kernels see it
// (host side only).
#pragma once

#include <cuda_runtime.h>

namespace rlscan {

// Where an argument lives, for the kernels: device (or managed) memory is
// staged with bulk asynchronous copies; page-locked host memory
// (cudaHostAlloc / cudaHostRegister) is read and written in place over the
// host link with plain loads and stores (zero copy), and so is pageable
// host memory on a device that reads it through the host's page tables;
// other pointers are refused before anything is launched.
enum class Residency { Device, Host, Unreachable };

inline bool pageable_access()
{
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrPageableMemoryAccess, dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return v != 0;
}

inline Residency residency(const void *ptr)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        a.type = cudaMemoryTypeUnregistered;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return Residency::Device;
    if (a.type == cudaMemoryTypeHost) return Residency::Host;
    return pageable_access() ? Residency::Host : Residency::Unreachable;
}

}  // namespace rlscan
