// dn_commit: make the checkpoint at each request's accepted position its state.
//
// After greedy verification the accepted prefix is kept and the rejected drafts
// are discarded ("Qwen3.8-27B on a Single RTX 3090: ...", Technical Insight); for
// the DeltaNet state this is a copy of one checkpoint page (all heads of one
// state set) over the state, or nothing when no draft was accepted.
//
// Pure copy, HBM bound: one CTA per (set, piece of kPiece bytes), numbered set-major on
// grid.x (so the set count is not bounded by grid.y); each thread
// moves kUnroll 16-byte words with all loads issued before the stores. The
// accepted length is read on the device, so no host round trip sits between
// accept and commit.
#include <cuda_runtime.h>

#include "dn.h"
#include "dn_device.cuh"
#include "dn_internal.h"
#include "dn_mma.cuh"
#include "dn_recurrence.cuh"

namespace dn {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;
constexpr size_t kPiece = (size_t)kThreads * kUnroll * 16;  // 32 KiB per CTA

__global__ void __launch_bounds__(kThreads)
commit_kernel(int B, int T, unsigned pieces, size_t set_bytes, const uint4 *__restrict__ ckpt,
              const int *__restrict__ accepted, uint4 *__restrict__ state) {
    const size_t n = blockIdx.x / pieces;
    const unsigned piece = blockIdx.x % pieces;
    grid_dep_wait();
    grid_dep_trigger();
    const int a = __ldg(&accepted[n % B]);
    if (a < 1 || a > T) return;  // a == 0: keep the state; out of range: ignored
    const size_t words = set_bytes / 16;
    const uint4 *src = ckpt + (n * T + (a - 1)) * words;
    uint4 *dst = state + n * words;
    const size_t base = (size_t)piece * (kPiece / 16) + threadIdx.x;
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const size_t i = base + (size_t)u * kThreads;
        if (i < words) r[u] = __ldcs(src + i);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const size_t i = base + (size_t)u * kThreads;
        if (i < words) dst[i] = r[u];
    }
}

// ---------------------------------------------------------------------------------------
// Recompute on commit. dn_verify_block_deltas keeps no per-position states; it writes
// delta_t = beta_t (v_t - g_t S_{t-1} k_t) for every position, and the accepted state is
// S_a = g_{a-1} ( ... (g_0 S_0 + delta_0 k_0^T) ... ) + delta_{a-1} k_{a-1}^T
//     = Gam S_0 + D^T K,   Gam = g_0 ... g_{a-1},  D[s][i] = (g_{s+1} ... g_{a-1}) delta_s[i]
// with K the a accepted keys. D^T K is one rank-a product per 64-row block of the state, on
// the tensor cores: tf32 MMAs (m16n8k8) with D split into a tf32 high part and the tf32 of
// the remainder, so the product keeps about 22 bits of D (k is fp16, exact in tf32) and the
// fp32 range. The sum is as accurate as the token-by-token replay but in another order, so the
// committed state can differ from dn_verify_block + dn_commit in the last fp16 bit.
// A CTA owns 64 rows of one (state set, head): the rows go through shared memory (16-byte
// loads and stores, 16-byte chunks swizzled by row so the fragment reads are conflict free);
// warp w computes rows 16 (w / 2) .. +15 and half of the dk columns.
constexpr int kDeltaRows = 64;

__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <int DK>
__global__ void __launch_bounds__(256, 5)
commit_deltas_kernel(int B, int H, int T, int DV, const __half *__restrict__ k,
                     const float *__restrict__ g, const float *__restrict__ delta,
                     const int *__restrict__ accepted, __half *__restrict__ state) {
    constexpr int ROWS = kDeltaRows, CPR = DK / 8, NTW = DK / 16;  // 16-byte chunks per row; n-tiles per warp
    __shared__ __align__(16) uint4 sS[ROWS * CPR];                  // the state rows, fp16
    __shared__ __align__(16) __half sK[DN_MAX_BLOCK][DK + 8];       // the accepted keys (zeros past a)
    __shared__ __align__(16) float sD[DN_MAX_BLOCK][ROWS + 8];     // delta_s[row] (zeros past a)
    __shared__ float sgate[DN_MAX_BLOCK + 1];  // decay of each position, then Gam
    const int rblocks = DV / ROWS;
    const int rb = blockIdx.x % rblocks;
    const int h = (blockIdx.x / rblocks) % H;
    const size_t n = blockIdx.x / (rblocks * H);
    grid_dep_wait();
    grid_dep_trigger();
    const int a = __ldg(&accepted[n % B]);
    if (a < 1 || a > T) return;  // a == 0: keep the state; out of range: ignored
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int gid = lane >> 2, t4 = lane & 3;
    uint4 *sp = reinterpret_cast<uint4 *>(state + ((n * H + h) * (size_t)DV + rb * ROWS) * DK);

    // The state rows (chunk c of row r at c ^ (r & 7)), the keys and the deltas (zeros past a)
    // go in by cp.async first, all in flight together; their latency overlaps the gates below.
    for (int i = tid; i < ROWS * CPR; i += 256) {
        const int r = i / CPR, c = i % CPR;
        cp_async16(&sS[r * CPR + (c ^ (r & 7))], sp + i, 16);
    }
    for (int i = tid; i < DN_MAX_BLOCK * (DK / 8); i += 256) {
        const int s2 = i / (DK / 8), j8 = i % (DK / 8);
        const bool live = s2 < a;
        cp_async16(&sK[s2][8 * j8], live ? (const void *)(k + ((n * T + s2) * H + h) * DK + (size_t)j8 * 8) : (const void *)k,
                   live ? 16 : 0);
    }
    for (int i = tid; i < DN_MAX_BLOCK * (ROWS / 4); i += 256) {
        const int s2 = i / (ROWS / 4), j4 = i % (ROWS / 4);
        const bool live = s2 < a;
        cp_async16(&sD[s2][4 * j4],
                   live ? (const void *)(delta + ((n * T + s2) * H + h) * DV + rb * ROWS + 4 * j4) : (const void *)delta,
                   live ? 16 : 0);
    }
    cp_async_commit();
    // decay of position s: g_{s+1} ... g_{a-1} (suffix products, one warp), and Gam = g_0 ... g_{a-1}
    if (warp == 0) {
        float gt = lane < a ? __ldg(&g[(n * T + lane) * H + h]) : 1.f;
        float suf = gt;  // inclusive suffix product over lanes >= this one, then shifted by one
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_down_sync(0xffffffffu, suf, off);
            if (lane + off < 32) suf *= o;
        }
        const float excl = __shfl_down_sync(0xffffffffu, suf, 1);
        if (lane < DN_MAX_BLOCK) sgate[lane] = lane + 1 < 32 ? excl : 1.f;
        if (lane == 0) sgate[DN_MAX_BLOCK] = suf;  // the product of every gate: Gam
    }
    cp_async_wait<0>();
    __syncthreads();
    const float gam = sgate[DN_MAX_BLOCK];

    // this warp's rows, and its n-tiles in groups of four (four accumulators of four floats)
    const int m0 = 16 * (warp >> 1), nt0 = (warp & 1) * NTW;
    __half *sh = reinterpret_cast<__half *>(sS);
#pragma unroll 1
    for (int j0 = 0; j0 < NTW; j0 += 4) {
        float acc[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
            if (8 * ks >= a) break;
            // D[s][row] = decay_s delta_s[row]
            const float d0 = sgate[8 * ks + t4], d1 = sgate[8 * ks + t4 + 4];
            const float x[4] = {d0 * sD[8 * ks + t4][m0 + gid], d0 * sD[8 * ks + t4][m0 + gid + 8],
                                d1 * sD[8 * ks + t4 + 4][m0 + gid], d1 * sD[8 * ks + t4 + 4][m0 + gid + 8]};
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                hi[e] = to_tf32(x[e]);
                lo[e] = to_tf32(x[e] - __uint_as_float(hi[e]));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int col = 8 * (nt0 + j0 + j) + gid;
                const uint32_t b[2] = {__float_as_uint(__half2float(sK[8 * ks + t4][col])),
                                       __float_as_uint(__half2float(sK[8 * ks + t4 + 4][col]))};
                mma_tf32(acc[j], hi, b);
                mma_tf32(acc[j], lo, b);
            }
        }
        // S_a = Gam S_0 + D^T K, rounded to fp16, back into the rows in shared memory
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int col = 8 * (nt0 + j0 + j) + 2 * t4;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int r = m0 + gid + 8 * hh;
                __half2 *p = reinterpret_cast<__half2 *>(sh + r * DK + (((col >> 3) ^ (r & 7)) << 3) + (col & 7));
                const float2 s0 = __half22float2(*p);
                *p = __floats2half2_rn(fmaf(gam, s0.x, acc[j][2 * hh]), fmaf(gam, s0.y, acc[j][2 * hh + 1]));
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < ROWS * CPR; i += 256) {
        const int r = i / CPR, c = i % CPR;
        __stcs(sp + i, sS[r * CPR + (c ^ (r & 7))]);
    }
}

}  // namespace
}  // namespace dn

extern "C" dn_status dn_commit_deltas(int N, int B, int H, int T, int dk, int dv, dn_dtype state_dt,
                                      const void *k, const float *g, const float *delta,
                                      const int32_t *accepted_len, void *state, dn_stream_t stream) {
    using namespace dn;
    if (N < 0 || B < 1 || H < 1 || T < 1 || T > DN_MAX_BLOCK || !dtype_ok(state_dt))
        return DN_ERR_INVALID_ARG;
    if (N % B != 0) return DN_ERR_INVALID_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return DN_ERR_UNSUPPORTED;
    if (state_dt != DN_F16) return DN_ERR_UNSUPPORTED;
    if (N == 0) return DN_OK;
    if (!k || !g || !delta || !accepted_len || !state) return DN_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(state, 16) || !aligned(delta, 16) || !aligned(g, 4) ||
        !aligned(accepted_len, 4))
        return DN_ERR_INVALID_ARG;
    if ((long long)N * H * (dv / kDeltaRows) > 0x7fffffffLL) return DN_ERR_INVALID_ARG;
    const unsigned blocks = (unsigned)((long long)N * H * (dv / kDeltaRows));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const __half *kh = static_cast<const __half *>(k);
    __half *sh = static_cast<__half *>(state);
    if (dk == 128)
        launch_pdl(commit_deltas_kernel<128>, dim3(blocks), dim3(256), 0, st, B, H, T, dv, kh, g, delta, accepted_len, sh);
    else
        launch_pdl(commit_deltas_kernel<64>, dim3(blocks), dim3(256), 0, st, B, H, T, dv, kh, g, delta, accepted_len, sh);
    return launch_status();
}

extern "C" dn_status dn_commit(int N, int B, int H, int T, int dk, int dv, dn_dtype state_dt,
                               const void *ckpt, const int32_t *accepted_len, void *state,
                               dn_stream_t stream) {
    using namespace dn;
    if (N < 0 || B < 1 || H < 1 || T < 1 || T > DN_MAX_BLOCK || !dtype_ok(state_dt))
        return DN_ERR_INVALID_ARG;
    if (N % B != 0) return DN_ERR_INVALID_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return DN_ERR_UNSUPPORTED;
    if (N == 0) return DN_OK;
    if (!ckpt || !accepted_len || !state) return DN_ERR_INVALID_ARG;
    if (!aligned(ckpt, 16) || !aligned(state, 16) || !aligned(accepted_len, 4))
        return DN_ERR_INVALID_ARG;
    const size_t set_bytes = (size_t)H * dv * dk * dtype_bytes(state_dt);
    const size_t pieces = (set_bytes + kPiece - 1) / kPiece;
    if ((unsigned long long)pieces * (unsigned long long)N > 0x7fffffffULL) return DN_ERR_INVALID_ARG;
    const unsigned grid = (unsigned)(pieces * (size_t)N);
    launch_pdl(commit_kernel, dim3(grid), dim3(kThreads), 0, reinterpret_cast<cudaStream_t>(stream), B, T,
               (unsigned)pieces, set_bytes, static_cast<const uint4 *>(ckpt), accepted_len,
               static_cast<uint4 *>(state));
    return launch_status();
}
