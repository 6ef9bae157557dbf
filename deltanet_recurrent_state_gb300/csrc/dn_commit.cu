// dn_commit: make the checkpoint at each request's accepted position its state.
//
// After greedy verification the accepted prefix is kept and the rejected drafts
// are discarded ("Qwen3.8-27B on a Single RTX 3090: ...", Technical Insight); for
// the DeltaNet state this is a copy of one checkpoint page (all heads of one
// state set) over the state, or nothing when no draft was accepted.
//
// Pure copy, HBM bound: grid = (pieces of kPiece bytes per set) x N; each thread
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
commit_kernel(int B, int T, size_t set_bytes, const uint4 *__restrict__ ckpt,
              const int *__restrict__ accepted, uint4 *__restrict__ state) {
    const size_t n = blockIdx.y;
    const int a = __ldg(&accepted[n % B]);
    if (a < 1 || a > T) return;  // a == 0: keep the state; out of range: ignored
    const size_t words = set_bytes / 16;
    const uint4 *src = ckpt + (n * T + (a - 1)) * words;
    uint4 *dst = state + n * words;
    const size_t base = blockIdx.x * (kPiece / 16) + threadIdx.x;
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
// order) the checkpoint path uses, so both paths commit bit-identical states. A CTA owns
// 32 rows of one (state set, head), 8 lanes per row, 16 fp32 elements per lane; six CTAs
// share an SM so that one's loads overlap the others' replays.
template <int DK>
__global__ void __launch_bounds__(256, 6)
commit_deltas_kernel(int B, int H, int T, int DV, const __half *__restrict__ k,
                     const float *__restrict__ g, const float *__restrict__ delta,
                     const int *__restrict__ accepted, __half *__restrict__ state) {
    constexpr int ROWS = 32, TPR = 8, NT = 256;
    constexpr int NCH = DK / 8 / TPR;
    __shared__ __align__(16) float sk[DN_MAX_BLOCK][DK];
    __shared__ float sd[DN_MAX_BLOCK][ROWS], sg[DN_MAX_BLOCK];
    const int rblocks = DV / ROWS;
    const int rb = blockIdx.x % rblocks;
    const int h = (blockIdx.x / rblocks) % H;
    const size_t n = blockIdx.x / (rblocks * H);
    const int a = __ldg(&accepted[n % B]);
    if (a < 1 || a > T) return;  // a == 0: keep the state; out of range: ignored
    const int tid = threadIdx.x, lr = tid / TPR, ln = tid % TPR, row = rb * ROWS + lr;
    __half *sp = state + ((n * H + h) * (size_t)DV + row) * DK;
    float2 s[NCH * 4];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(sp + (c * TPR + ln) * 8);
        const __half2 *h2 = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) s[c * 4 + i] = __half22float2(h2[i]);
    }
    for (int i = tid; i < a * (DK / 8); i += NT) {
        const int t = i / (DK / 8), j8 = i % (DK / 8);
        float x[8];
        load8(k + ((n * T + t) * H + h) * DK + (size_t)j8 * 8, x);
        smem_put8(sk[t], j8, x);
    }
    for (int i = tid; i < a * ROWS; i += NT) {
        const int t = i / ROWS, r = i % ROWS;
        sd[t][r] = delta[((n * T + t) * H + h) * DV + rb * ROWS + r];
    }
    if (tid < a) sg[tid] = g[(n * T + tid) * H + h];
    __syncthreads();
    for (int t = 0; t < a; ++t) {
        const float dt = sd[t][lr], gt = sg[t];
        const float2 d2 = make_float2(dt, dt), g2 = make_float2(gt, gt);
        const float4 *k4 = reinterpret_cast<const float4 *>(sk[t]);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int j8 = c * TPR + ln;
            const float4 ka = k4[swz4(2 * j8)], kb = k4[swz4(2 * j8 + 1)];
            s[c * 4 + 0] = __ffma2_rn(d2, make_float2(ka.x, ka.y), __fmul2_rn(g2, s[c * 4 + 0]));
            s[c * 4 + 1] = __ffma2_rn(d2, make_float2(ka.z, ka.w), __fmul2_rn(g2, s[c * 4 + 1]));
            s[c * 4 + 2] = __ffma2_rn(d2, make_float2(kb.x, kb.y), __fmul2_rn(g2, s[c * 4 + 2]));
            s[c * 4 + 3] = __ffma2_rn(d2, make_float2(kb.z, kb.w), __fmul2_rn(g2, s[c * 4 + 3]));
        }
    }
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        uint4 u;
        __half2 *hh = reinterpret_cast<__half2 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) hh[i] = __float22half2_rn(s[c * 4 + i]);
        *reinterpret_cast<uint4 *>(sp + (c * TPR + ln) * 8) = u;
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
    if ((long long)N * H * (dv / 32) > 0x7fffffffLL) return DN_ERR_INVALID_ARG;
    const unsigned blocks = (unsigned)((long long)N * H * (dv / 32));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const __half *kh = static_cast<const __half *>(k);
    __half *sh = static_cast<__half *>(state);
    if (dk == 128)
        commit_deltas_kernel<128><<<blocks, 256, 0, st>>>(B, H, T, dv, kh, g, delta, accepted_len, sh);
    else
        commit_deltas_kernel<64><<<blocks, 256, 0, st>>>(B, H, T, dv, kh, g, delta, accepted_len, sh);
    return launch_status();
}

extern "C" dn_status dn_commit(int N, int B, int H, int T, int dk, int dv, dn_dtype state_dt,
                               const void *ckpt, const int32_t *accepted_len, void *state,
                               dn_stream_t stream) {
    using namespace dn;
    if (N < 0 || B < 1 || H < 1 || T < 1 || T > DN_MAX_BLOCK || !dtype_ok(state_dt))
        return DN_ERR_INVALID_ARG;
    if (N % B != 0 || N > 65535) return DN_ERR_INVALID_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return DN_ERR_UNSUPPORTED;
    if (N == 0) return DN_OK;
    if (!ckpt || !accepted_len || !state) return DN_ERR_INVALID_ARG;
    if (!aligned(ckpt, 16) || !aligned(state, 16) || !aligned(accepted_len, 4))
        return DN_ERR_INVALID_ARG;
    const size_t set_bytes = (size_t)H * dv * dk * dtype_bytes(state_dt);
    const size_t pieces = (set_bytes + kPiece - 1) / kPiece;
    if (pieces > 0x7fffffffULL) return DN_ERR_INVALID_ARG;
    const dim3 grid((unsigned)pieces, (unsigned)N);
    commit_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        B, T, set_bytes, static_cast<const uint4 *>(ckpt), accepted_len,
        static_cast<uint4 *>(state));
    return launch_status();
}
