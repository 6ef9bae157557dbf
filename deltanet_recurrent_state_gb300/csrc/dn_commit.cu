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
// S_a = g_{a-1} ( ... (g_0 S_0 + delta_0 k_0^T) ... ) + delta_{a-1} k_{a-1}^T, applied here
// to the old state in place with exactly the arithmetic (packed fp32x2 FMAs in the same
// order) the checkpoint path uses, so both paths commit bit-identical states.
// A CTA owns 64 rows of one (state set, head): warp w the rows 8w .. 8w+7, lane l the DK/32
// columns from l DK/32 in all of them. Per step a lane reads its columns of k_t once from
// shared memory (distinct addresses across the warp: no quarter-warp pass repeats another)
// and reuses them for its eight rows; delta and the gate are broadcasts. (With eight lanes
// per row, each 16-byte read of k served four rows of a warp in four separate quarter-warp
// passes, and the shared-memory pipe, not HBM, bounded the kernel; with four rows per warp
// the shared reads and loop overhead, not the packed FMAs, still made up most of the
// instructions.)
constexpr int kDeltaRows = 64;

template <int DK>
__global__ void __launch_bounds__(256, 4)
commit_deltas_kernel(int B, int H, int T, int DV, const __half *__restrict__ k,
                     const float *__restrict__ g, const float *__restrict__ delta,
                     const int *__restrict__ accepted, __half *__restrict__ state) {
    constexpr int ROWS = kDeltaRows, RPW = ROWS / 8, CPL = DK / 32, NP = CPL / 2;
    static_assert(CPL == 2 || CPL == 4, "two or four columns per lane");
    __shared__ __align__(16) float sk[DN_MAX_BLOCK][DK];
    __shared__ float sd[DN_MAX_BLOCK][ROWS], sg[DN_MAX_BLOCK];
    const int rblocks = DV / ROWS;
    const int rb = blockIdx.x % rblocks;
    const int h = (blockIdx.x / rblocks) % H;
    const size_t n = blockIdx.x / (rblocks * H);
    grid_dep_wait();
    grid_dep_trigger();
    const int a = __ldg(&accepted[n % B]);
    if (a < 1 || a > T) return;  // a == 0: keep the state; out of range: ignored
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    __half *sp = state + ((n * H + h) * (size_t)DV + rb * ROWS + warp * RPW) * DK + lane * CPL;

    float2 s[RPW][NP];  // rows 4w + r, columns lane CPL + 2p, + 1
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        __half2 hv[NP];
        if constexpr (NP == 2) {
            const uint2 u = *reinterpret_cast<const uint2 *>(sp + (size_t)r * DK);
            hv[0] = *reinterpret_cast<const __half2 *>(&u.x);
            hv[1] = *reinterpret_cast<const __half2 *>(&u.y);
        } else {
            hv[0] = *reinterpret_cast<const __half2 *>(sp + (size_t)r * DK);
        }
#pragma unroll
        for (int p = 0; p < NP; ++p) s[r][p] = __half22float2(hv[p]);
    }
    for (int i = tid; i < a * (DK / 8); i += 256) {
        const int t = i / (DK / 8), j8 = i % (DK / 8);
        float x[8];
        load8(k + ((n * T + t) * H + h) * DK + (size_t)j8 * 8, x);
        *reinterpret_cast<float4 *>(&sk[t][8 * j8]) = make_float4(x[0], x[1], x[2], x[3]);
        *reinterpret_cast<float4 *>(&sk[t][8 * j8 + 4]) = make_float4(x[4], x[5], x[6], x[7]);
    }
    for (int i = tid; i < a * ROWS; i += 256) {
        const int t = i / ROWS, r = i % ROWS;
        sd[t][r] = delta[((n * T + t) * H + h) * DV + rb * ROWS + r];
    }
    if (tid < a) sg[tid] = g[(n * T + tid) * H + h];
    __syncthreads();
    for (int t = 0; t < a; ++t) {
        const float gt = sg[t];
        const float2 g2 = make_float2(gt, gt);
        float2 kf[NP];
        if constexpr (NP == 2) {
            const float4 k4 = *reinterpret_cast<const float4 *>(&sk[t][lane * CPL]);
            kf[0] = make_float2(k4.x, k4.y);
            kf[1] = make_float2(k4.z, k4.w);
        } else {
            kf[0] = *reinterpret_cast<const float2 *>(&sk[t][lane * CPL]);
        }
#pragma unroll
        for (int r = 0; r < RPW; ++r) {
            const float dt = sd[t][warp * RPW + r];
            const float2 d2 = make_float2(dt, dt);
#pragma unroll
            for (int p = 0; p < NP; ++p) s[r][p] = __ffma2_rn(d2, kf[p], __fmul2_rn(g2, s[r][p]));
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        __half2 hv[NP];
#pragma unroll
        for (int p = 0; p < NP; ++p) hv[p] = __float22half2_rn(s[r][p]);
        if constexpr (NP == 2) {
            uint2 u;
            u.x = *reinterpret_cast<const unsigned *>(&hv[0]);
            u.y = *reinterpret_cast<const unsigned *>(&hv[1]);
            *reinterpret_cast<uint2 *>(sp + (size_t)r * DK) = u;
        } else {
            *reinterpret_cast<__half2 *>(sp + (size_t)r * DK) = hv[0];
        }
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
    if (!aligned(k, 16) || !aligned(state, 16) || !aligned(delta, 4) || !aligned(g, 4) ||
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
