// ctx_key.cuh -- identity of the CUDA context the calling thread works in.
//
// The library keeps some set-up per device: kernel attributes, occupancy
// figures, the device address of its fixed scratch array, and the host-buffer
// path's copy streams.  All of these belong to one CUDA context.  A
// cudaDeviceReset destroys the device's primary context, and the next runtime
// call creates a new one in which those handles and addresses mean nothing.
// Each cache therefore records the unique id of the context it was built in
// (cuCtxGetId; ids are never reused within a process) and builds itself again
// when the current context's id differs.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace sg_ctx {

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

struct DriverFns {
    CtxGetCurrentFn get_current = nullptr;
    CtxGetIdFn get_id = nullptr;
};

inline const DriverFns &driver_fns() {
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fns.get_id = reinterpret_cast<CtxGetIdFn>(fn);
        (void)cudaGetLastError();
    });
    return fns;
}

// Id of the context current on this thread for device `dev` (made current by
// cudaSetDevice, which initialises the primary context, when no context is
// current yet).  Returns false when the driver offers no way to tell; callers
// then keep their set-up for the life of the process.
inline bool current_id(int dev, unsigned long long *id) {
    const DriverFns &f = driver_fns();
    if (f.get_current == nullptr || f.get_id == nullptr) return false;
    CUcontext c = nullptr;
    if (f.get_current(&c) != CUDA_SUCCESS) return false;
    if (c == nullptr) {
        if (cudaSetDevice(dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        if (f.get_current(&c) != CUDA_SUCCESS || c == nullptr) return false;
    }
    return f.get_id(c, id) == CUDA_SUCCESS;
}

}  // namespace sg_ctx
