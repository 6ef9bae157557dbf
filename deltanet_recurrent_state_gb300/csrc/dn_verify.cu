// dn_verify_block: one verify block of T <= 16 draft tokens through the gated
// delta rule, writing the output and a state checkpoint at every position.
//
// Per-position state copies are what the "recurrent-state pages" of a
// speculating request hold ("HyperQwen: 1,000 tok/s on a Single RTX 3090 ...",
// Technical Insight; "HyperQwen" README, The numbers behind that).
//
// Work decomposition. The dv rows of S evolve independently (row i only needs
// v_t[i] and the shared k_t, q_t), so a CTA owns ROWS rows of one (state set,
// head) and keeps that slice in registers, in fp32, for all T tokens. Grid =
// N * H * (dv / ROWS) CTAs. The kernel is bound by the checkpoint stores (T
// copies of the state slice), issued as 16-byte streaming stores.
#include <cuda_runtime.h>

#include "dn.h"
#include "dn_device.cuh"
#include "dn_internal.h"
#include "dn_recurrence.cuh"

namespace dn {
namespace {

constexpr int kMaxT = DN_MAX_BLOCK;

template <int DK, int ROWS, int TPR, typename IO, typename ST>
__global__ void __launch_bounds__(ROWS * TPR)
verify_block_kernel(int H, int T, int DV, const IO *__restrict__ q, const IO *__restrict__ k,
                    const IO *__restrict__ v, const float *__restrict__ beta,
                    const float *__restrict__ g, const ST *__restrict__ s_in,
                    IO *__restrict__ out, ST *__restrict__ ckpt) {
    constexpr int NT = ROWS * TPR;
    constexpr int EPT = DK / TPR;
    constexpr int NCH = EPT / 8;
    __shared__ __align__(16) float sk[kMaxT][DK];
    __shared__ __align__(16) float sq[kMaxT][DK];
    __shared__ float sv[kMaxT][ROWS];
    __shared__ float so[kMaxT][ROWS];
    __shared__ float sbeta[kMaxT], sg[kMaxT], skq[kMaxT];

    const int rblocks = DV / ROWS;
    const int rb = blockIdx.x % rblocks;
    const int h = (blockIdx.x / rblocks) % H;
    const size_t n = blockIdx.x / (rblocks * H);
    const int tid = threadIdx.x;
    const int lr = tid / TPR;
    const int ln = tid % TPR;
    const int row = rb * ROWS + lr;

    // State slice -> registers (issued first so it overlaps the staging loads).
    float s[EPT];
    const size_t set_elems = (size_t)DV * DK;
    {
        const ST *sp = s_in + (n * H + h) * set_elems + (size_t)row * DK;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float x[8];
            load8(sp + (c * TPR + ln) * 8, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) s[c * 8 + e] = x[e];
        }
    }

    // Stage q_t, k_t (fp32, swizzled), v_t[rows], beta_t, g_t for the block.
    for (int i = tid; i < T * (DK / 8); i += NT) {
        const int t = i / (DK / 8), j8 = i % (DK / 8);
        const size_t off = ((n * T + t) * H + h) * DK + (size_t)j8 * 8;
        float x[8];
        load8(q + off, x);
        smem_put8(sq[t], j8, x);
        load8(k + off, x);
        smem_put8(sk[t], j8, x);
    }
    for (int i = tid; i < T * ROWS; i += NT) {
        const int t = i / ROWS, r = i % ROWS;
        sv[t][r] = to_f(v[((n * T + t) * H + h) * DV + rb * ROWS + r]);
    }
    if (tid < T) {
        sbeta[tid] = beta[(n * T + tid) * H + h];
        sg[tid] = g[(n * T + tid) * H + h];
    }
    __syncthreads();
    {
        const int warp = tid / 32, lane = tid % 32;
        for (int t = warp; t < T; t += NT / 32) {
            const float d = warp_dot_swz<DK>(sk[t], sq[t], lane);
            if (lane == 0) skq[t] = d;
        }
    }
    __syncthreads();

    ST *cp = ckpt + (size_t)row * DK;
    for (int t = 0; t < T; ++t) {
        const float o = token_step<DK, TPR>(s, sk[t], sq[t], ln, sbeta[t], sg[t], sv[t][lr], skq[t]);
        if (ln == 0) so[t][lr] = o;
        ST *dst = cp + ((n * T + t) * H + h) * set_elems;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = s[c * 8 + e];
            store8<true>(dst + (c * TPR + ln) * 8, x);
        }
    }
    __syncthreads();
    for (int i = tid; i < T * ROWS; i += NT) {
        const int t = i / ROWS, r = i % ROWS;
        out[((n * T + t) * H + h) * DV + rb * ROWS + r] = from_f<IO>(so[t][r]);
    }
}

constexpr int kRows = 32;
constexpr int kTpr = 8;

template <int DK, typename IO, typename ST>
void launch_verify(int N, int H, int T, int dv, const void *q, const void *k, const void *v,
                   const float *beta, const float *g, const void *s_in, void *out, void *ckpt,
                   cudaStream_t st) {
    const long long blocks = (long long)N * H * (dv / kRows);
    verify_block_kernel<DK, kRows, kTpr, IO, ST><<<(unsigned)blocks, kRows * kTpr, 0, st>>>(
        H, T, dv, static_cast<const IO *>(q), static_cast<const IO *>(k),
        static_cast<const IO *>(v), beta, g, static_cast<const ST *>(s_in),
        static_cast<IO *>(out), static_cast<ST *>(ckpt));
}

}  // namespace
}  // namespace dn

extern "C" dn_status dn_verify_block(int N, int H, int T, int dk, int dv, dn_dtype io_dt,
                                     dn_dtype state_dt, const void *q, const void *k,
                                     const void *v, const float *beta, const float *g,
                                     const void *state_in, void *out, void *ckpt,
                                     dn_stream_t stream) {
    using namespace dn;
    if (N < 0 || H < 1 || T < 1 || T > DN_MAX_BLOCK) return DN_ERR_INVALID_ARG;
    if (!dtype_ok(io_dt) || !dtype_ok(state_dt)) return DN_ERR_INVALID_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return DN_ERR_UNSUPPORTED;
    if (io_dt != state_dt) return DN_ERR_UNSUPPORTED;
    if (N == 0) return DN_OK;
    if (!q || !k || !v || !beta || !g || !state_in || !out || !ckpt) return DN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(state_in, 16) ||
        !aligned(out, 16) || !aligned(ckpt, 16) || !aligned(beta, 4) || !aligned(g, 4))
        return DN_ERR_INVALID_ARG;
    if ((long long)N * H * (dv / kRows) > 0x7fffffffLL) return DN_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (io_dt == DN_F16) {
        if (dk == 128) launch_verify<128, __half, __half>(N, H, T, dv, q, k, v, beta, g, state_in, out, ckpt, st);
        else launch_verify<64, __half, __half>(N, H, T, dv, q, k, v, beta, g, state_in, out, ckpt, st);
    } else {
        if (dk == 128) launch_verify<128, float, float>(N, H, T, dv, q, k, v, beta, g, state_in, out, ckpt, st);
        else launch_verify<64, float, float>(N, H, T, dv, q, k, v, beta, g, state_in, out, ckpt, st);
    }
    return launch_status();
}
