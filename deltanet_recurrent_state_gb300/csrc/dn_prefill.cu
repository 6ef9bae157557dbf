// dn_prefill_checkpoint: a prompt through the gated delta rule with a state
// checkpoint every 64 tokens, for prefix caching of the DeltaNet state
// ("HyperQwen: 1,000 tok/s on a Single RTX 3090 ...", Technical Insight: the
// recurrent state is checkpointed next to the attention context so that a later
// turn restores it instead of recomputing the prompt).
//
// This file holds the sequential form: a CTA owns ROWS rows of one (sequence,
// head) state in registers and walks the prompt token by token, staging 16
// tokens of q/k/v/beta/g at a time in shared memory. At every chunk end the
// carry is rounded to the state dtype and stored, so the carry equals the
// checkpoint and a restored run continues bit-identically.
#include <cuda_runtime.h>

#include "dn.h"
#include "dn_device.cuh"
#include "dn_internal.h"
#include "dn_recurrence.cuh"

namespace dn {
namespace {

constexpr int kSub = 16;  // tokens staged per round

template <int DK, int ROWS, int TPR, typename IO, typename ST>
__global__ void __launch_bounds__(ROWS * TPR)
prefill_seq_kernel(int H, int P, int DV, int chunk, const IO *__restrict__ q,
                   const IO *__restrict__ k, const IO *__restrict__ v,
                   const float *__restrict__ beta, const float *__restrict__ g,
                   const ST *s_in, IO *__restrict__ out, ST *__restrict__ ckpt, ST *s_out) {
    constexpr int NT = ROWS * TPR;
    constexpr int EPT = DK / TPR;
    constexpr int NCH = EPT / 8;
    __shared__ __align__(16) float sk[kSub][DK];
    __shared__ __align__(16) float sq[kSub][DK];
    __shared__ float sv[kSub][ROWS];
    __shared__ float so[kSub][ROWS];
    __shared__ float sbeta[kSub], sg[kSub], skq[kSub];

    const int rblocks = DV / ROWS;
    const int rb = blockIdx.x % rblocks;
    const int h = (blockIdx.x / rblocks) % H;
    const size_t n = blockIdx.x / (rblocks * H);
    const int tid = threadIdx.x;
    const int lr = tid / TPR;
    const int ln = tid % TPR;
    const int row = rb * ROWS + lr;
    const size_t set_elems = (size_t)DV * DK;
    const size_t row_off = (n * H + h) * set_elems + (size_t)row * DK;

    float s[EPT];
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        float x[8];
        if (s_in) {
            load8(s_in + row_off + (c * TPR + ln) * 8, x);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) s[c * 8 + e] = x[e];
    }

    const size_t nchunks = (size_t)P / chunk;
    for (int p0 = 0; p0 < P; p0 += kSub) {
        const int ns = min(kSub, P - p0);
        __syncthreads();
        for (int i = tid; i < ns * (DK / 8); i += NT) {
            const int t = i / (DK / 8), j8 = i % (DK / 8);
            const size_t off = ((n * P + p0 + t) * H + h) * DK + (size_t)j8 * 8;
            float x[8];
            load8(q + off, x);
            smem_put8(sq[t], j8, x);
            load8(k + off, x);
            smem_put8(sk[t], j8, x);
        }
        for (int i = tid; i < ns * ROWS; i += NT) {
            const int t = i / ROWS, r = i % ROWS;
            sv[t][r] = to_f(v[((n * P + p0 + t) * H + h) * DV + rb * ROWS + r]);
        }
        if (tid < ns) {
            sbeta[tid] = beta[(n * P + p0 + tid) * H + h];
            sg[tid] = g[(n * P + p0 + tid) * H + h];
        }
        __syncthreads();
        {
            const int warp = tid / 32, lane = tid % 32;
            for (int t = warp; t < ns; t += NT / 32) {
                const float d = warp_dot_swz<DK>(sk[t], sq[t], lane);
                if (lane == 0) skq[t] = d;
            }
        }
        __syncthreads();
        for (int t = 0; t < ns; ++t) {
            const float o = token_step<DK, TPR>(s, sk[t], sq[t], ln, sbeta[t], sg[t], sv[t][lr], skq[t]);
            if (ln == 0) so[t][lr] = o;
            const int p = p0 + t + 1;
            if (p % chunk == 0) {
#pragma unroll
                for (int e = 0; e < EPT; ++e) s[e] = round_as(s[e], (const ST *)nullptr);
                ST *dst = ckpt + ((n * nchunks + (size_t)(p / chunk - 1)) * H + h) * set_elems +
                          (size_t)row * DK;
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = s[c * 8 + e];
                    store8<true>(dst + (c * TPR + ln) * 8, x);
                }
            }
        }
        __syncthreads();
        for (int i = tid; i < ns * ROWS; i += NT) {
            const int t = i / ROWS, r = i % ROWS;
            out[((n * P + p0 + t) * H + h) * DV + rb * ROWS + r] = from_f<IO>(so[t][r]);
        }
    }
    // Final state (rounded to the state dtype by the store).
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = s[c * 8 + e];
        store8<false>(s_out + row_off + (c * TPR + ln) * 8, x);
    }
}

constexpr int kRows = 16;
constexpr int kTpr = 8;

template <int DK, typename IO, typename ST>
void launch_prefill_seq(int N, int H, int P, int chunk, int dv, const void *q, const void *k,
                        const void *v, const float *beta, const float *g, const void *s_in,
                        void *out, void *ckpt, void *s_out, cudaStream_t st) {
    const long long blocks = (long long)N * H * (dv / kRows);
    prefill_seq_kernel<DK, kRows, kTpr, IO, ST><<<(unsigned)blocks, kRows * kTpr, 0, st>>>(
        H, P, dv, chunk, static_cast<const IO *>(q), static_cast<const IO *>(k),
        static_cast<const IO *>(v), beta, g, static_cast<const ST *>(s_in),
        static_cast<IO *>(out), static_cast<ST *>(ckpt), static_cast<ST *>(s_out));
}

}  // namespace
}  // namespace dn

extern "C" dn_status dn_prefill_checkpoint(int N, int H, int P, int chunk, int dk, int dv,
                                           dn_dtype io_dt, dn_dtype state_dt, const void *q,
                                           const void *k, const void *v, const float *beta,
                                           const float *g, const void *state_in, void *out,
                                           void *ckpt, void *state_out, dn_stream_t stream) {
    using namespace dn;
    if (N < 0 || H < 1 || P < 0) return DN_ERR_INVALID_ARG;
    if (!dtype_ok(io_dt) || !dtype_ok(state_dt)) return DN_ERR_INVALID_ARG;
    if (chunk != DN_PREFILL_CHUNK) return DN_ERR_UNSUPPORTED;
    if (!head_dim_ok(dk) || !head_dim_ok(dv) || io_dt != state_dt) return DN_ERR_UNSUPPORTED;
    if (N == 0) return DN_OK;
    if (!state_out) return DN_ERR_INVALID_ARG;
    if (P > 0 && (!q || !k || !v || !beta || !g || !out)) return DN_ERR_INVALID_ARG;
    if (P >= chunk && !ckpt) return DN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        !aligned(ckpt, 16) || !aligned(state_in, 16) || !aligned(state_out, 16) ||
        !aligned(beta, 4) || !aligned(g, 4))
        return DN_ERR_INVALID_ARG;
    if ((long long)N * H * (dv / kRows) > 0x7fffffffLL) return DN_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (io_dt == DN_F16) {
        if (dk == 128) launch_prefill_seq<128, __half, __half>(N, H, P, chunk, dv, q, k, v, beta, g, state_in, out, ckpt, state_out, st);
        else launch_prefill_seq<64, __half, __half>(N, H, P, chunk, dv, q, k, v, beta, g, state_in, out, ckpt, state_out, st);
    } else {
        if (dk == 128) launch_prefill_seq<128, float, float>(N, H, P, chunk, dv, q, k, v, beta, g, state_in, out, ckpt, state_out, st);
        else launch_prefill_seq<64, float, float>(N, H, P, chunk, dv, q, k, v, beta, g, state_in, out, ckpt, state_out, st);
    }
    return launch_status();
}
