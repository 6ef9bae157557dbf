// Host-side helpers shared by the entry points of libdn.so: argument checks and
// launch-error mapping. Nothing here touches the GPU except launch_status.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "dn.h"

namespace dn {

inline bool aligned(const void *p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline bool head_dim_ok(int d) { return d == 64 || d == 128; }

inline size_t dtype_bytes(dn_dtype t) { return t == DN_F16 ? 2 : 4; }

inline bool dtype_ok(dn_dtype t) { return t == DN_F16 || t == DN_F32; }

// After a launch: map a launch failure to DN_ERR_CUDA (and clear it).
inline dn_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? DN_OK : DN_ERR_CUDA;
}

// Launch with programmatic stream serialisation allowed: the kernel may be scheduled
// before the previous kernel on `st` has finished. Only kernels that call grid_dep_wait()
// (dn_device.cuh) before touching global memory are launched this way.
template <typename... Params, typename... Args>
inline void launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// Streaming multiprocessors of the current device (0 if the query fails).
inline int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sms;
}

// Chunkwise fp16 prefill on tcgen05 tensor cores for dk = dv = 128 (dn_prefill_tc.cu).
dn_status launch_prefill_tc(int N, int H, int P, const void *q, const void *k, const void *v, const float *beta,
                            const float *g, const void *s_in, void *out, void *ckpt, void *s_out, cudaStream_t st);
unsigned int prefill_tc_wait_timeouts();

}  // namespace dn
