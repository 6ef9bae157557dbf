// The per-token gated delta-rule update on a register-resident slice of the state,
// shared by the verify-block and the sequential prefill kernels.
//
// Math (gated delta rule, Yang et al. 2024), per row i of the dv x dk state S:
//   u_i   = S_{t-1}[i,:] . k_t                (read before the update)
//   w_i   = beta_t (v_t[i] - g_t u_i)
//   S_t[i,:] = g_t S_{t-1}[i,:] + w_i k_t^T   (== g S (I - beta k k^T) + beta v k^T)
//   o_t[i] = S_t[i,:] . q_t = g_t (S_{t-1}[i,:] . q_t) + w_i (k_t . q_t)
// so one pass over the row gives both dot products, and a second pass updates it.
//
// Thread mapping. A row of dk elements is split over TPR consecutive lanes. Lane
// `ln` of the row holds the 8-element chunks c*TPR + ln (c = 0 .. EPT/8 - 1), so a
// warp-wide 16-byte store of chunk c writes TPR*16 contiguous bytes of every row.
// k_t and q_t sit in shared memory as fp32 with an XOR swizzle of 16-byte words
// (word f lives at f ^ ((f >> 3) & 1)), which makes the lanes' 16-byte reads of
// their chunks bank-conflict free.
#pragma once

#include "dn_device.cuh"

namespace dn {

__device__ __forceinline__ int swz4(int f) { return f ^ ((f >> 3) & 1); }

// Store 8 consecutive floats x (logical elements 8*j8 .. 8*j8+7) into a swizzled row.
__device__ __forceinline__ void smem_put8(float *row, int j8, const float (&x)[8]) {
    float4 *r4 = reinterpret_cast<float4 *>(row);
    r4[swz4(2 * j8)] = make_float4(x[0], x[1], x[2], x[3]);
    r4[swz4(2 * j8 + 1)] = make_float4(x[4], x[5], x[6], x[7]);
}

__device__ __forceinline__ void smem_get8(const float *row, int j8, float (&x)[8]) {
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    const float4 a = r4[swz4(2 * j8)];
    const float4 b = r4[swz4(2 * j8 + 1)];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// Dot product of two swizzled shared rows of DK floats, by one warp.
template <int DK>
__device__ __forceinline__ float warp_dot_swz(const float *a, const float *b, int lane) {
    float acc = 0.f;
    for (int j8 = lane; j8 < DK / 8; j8 += 32) {
        float x[8], y[8];
        smem_get8(a, j8, x);
        smem_get8(b, j8, y);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(x[e], y[e], acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    return acc;
}

// One token on this lane's EPT elements of one row. k_s/q_s: swizzled fp32 rows.
// Returns o_t for the row (identical in all TPR lanes of the row).
template <int DK, int TPR>
__device__ __forceinline__ float token_step(float (&s)[DK / TPR], const float *k_s,
                                            const float *q_s, int ln, float beta,
                                            float g, float v, float kq) {
    constexpr int EPT = DK / TPR;
    constexpr int NCH = EPT / 8;
    float kk[EPT];
    float pk0 = 0.f, pk1 = 0.f, pq0 = 0.f, pq1 = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int j8 = c * TPR + ln;
        float kv[8], qv[8];
        smem_get8(k_s, j8, kv);
        smem_get8(q_s, j8, qv);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            kk[c * 8 + e] = kv[e];
            kk[c * 8 + e + 1] = kv[e + 1];
            pk0 = fmaf(s[c * 8 + e], kv[e], pk0);
            pk1 = fmaf(s[c * 8 + e + 1], kv[e + 1], pk1);
            pq0 = fmaf(s[c * 8 + e], qv[e], pq0);
            pq1 = fmaf(s[c * 8 + e + 1], qv[e + 1], pq1);
        }
    }
    float pk = pk0 + pk1, pq = pq0 + pq1;
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) {
        pk += __shfl_xor_sync(0xffffffffu, pk, off);
        pq += __shfl_xor_sync(0xffffffffu, pq, off);
    }
    const float w = beta * (v - g * pk);
#pragma unroll
    for (int e = 0; e < EPT; ++e) s[e] = fmaf(w, kk[e], g * s[e]);
    return fmaf(g, pq, w * kq);
}

}  // namespace dn
