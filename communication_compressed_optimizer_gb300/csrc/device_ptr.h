// Host-side check that a pointer the GPU will dereference is memory of the
// current (or a given) device, so a host pointer becomes an argument error
// before anything is enqueued.
#pragma once
#include <cuda_runtime.h>

namespace lamb1b {

inline bool is_device_ptr(const void* p, int device)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == device;
}

inline bool is_current_device_ptr(const void* p)
{
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && is_device_ptr(p, dev);
}

}  // namespace lamb1b
