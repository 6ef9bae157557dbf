// Device helpers shared by the libdn kernels: 8-element vector loads/stores in
// fp16 or fp32 with fp32 registers, and a PTX cache-hint store.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

namespace dn {

// ---- programmatic dependent launch ----------------------------------------------------
// The step kernels are launched with programmatic stream serialisation allowed (see
// launch_pdl in dn_internal.h): a kernel may be scheduled while the kernel before it on
// the stream is still running. Each calls grid_dep_wait() before its first global
// memory access, which returns once every earlier kernel on the stream has completed and
// its writes are visible, so results are as with plain stream order. Right after that
// wait it calls grid_dep_trigger(), which lets the next kernel be scheduled onto free
// SM slots meanwhile: its launch latency then overlaps this kernel's run. Both are
// no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- 8 consecutive elements <-> 8 floats ---------------------------------------------

__device__ __forceinline__ void load8(const __half *p, float (&x)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __half22float2(h[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ void load8(const float *p, float (&x)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    const float4 b = *reinterpret_cast<const float4 *>(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Streaming (evict-first) 16-byte store: checkpoint pages are written once per
// step and read back at most once, so they should not displace reused lines in L2.
__device__ __forceinline__ void st_cs_v4(void *p, uint4 u) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(u.x), "r"(u.y), "r"(u.z), "r"(u.w) : "memory");
}

__device__ __forceinline__ uint4 pack8_half(const float (&x)[8]) {
    uint4 u;
    __half2 *h = reinterpret_cast<__half2 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
    return u;
}

template <bool STREAM>
__device__ __forceinline__ void store8(__half *p, const float (&x)[8]) {
    const uint4 u = pack8_half(x);
    if (STREAM) st_cs_v4(p, u);
    else *reinterpret_cast<uint4 *>(p) = u;
}

template <bool STREAM>
__device__ __forceinline__ void store8(float *p, const float (&x)[8]) {
    uint4 a = make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]),
                         __float_as_uint(x[2]), __float_as_uint(x[3]));
    uint4 b = make_uint4(__float_as_uint(x[4]), __float_as_uint(x[5]),
                         __float_as_uint(x[6]), __float_as_uint(x[7]));
    if (STREAM) {
        st_cs_v4(p, a);
        st_cs_v4(p + 4, b);
    } else {
        *reinterpret_cast<uint4 *>(p) = a;
        *reinterpret_cast<uint4 *>(p + 4) = b;
    }
}

// Round a float to the storage type and back (the value a store would keep).
__device__ __forceinline__ float round_as(float x, const __half *) {
    return __half2float(__float2half_rn(x));
}
__device__ __forceinline__ float round_as(float x, const float *) { return x; }

__device__ __forceinline__ float to_f(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f(float x) { return x; }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }

}  // namespace dn
