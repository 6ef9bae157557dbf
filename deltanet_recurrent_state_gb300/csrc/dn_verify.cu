// dn_verify_block: one verify block of T <= 16 draft tokens through the gated
// delta rule, writing the output and a state checkpoint at every position.
//
// Per-position state copies are what the "recurrent-state pages" of a
// speculating request hold ("HyperQwen: 1,000 tok/s on a Single RTX 3090 ...",
// Technical Insight; "HyperQwen" README, The numbers behind that).
//
// Work decomposition. The dv rows of S evolve independently (row i only needs
// v_t[i] and the shared k_t, q_t), so a CTA owns 32 rows of one (state set,
// head) and keeps that slice in registers, in fp32, for all T tokens. Grid =
// N * H * (dv / 32) CTAs. The kernel is bound by the checkpoint stores (T copies
// of the state slice), issued as 16-byte streaming stores.
//
// Two kernels:
//  * verify_wy_kernel (fp16 state): the chunkwise (WY) form of the block. One
//    tensor-core contraction per CTA gives S0 k_t and S0 q_t for every t, a 16 x 16
//    forward substitution per row gives delta_t and o_t, and the per-token loop
//    only applies the rank-1 checkpoint update. See the derivation below.
//  * verify_block_kernel (any supported dtype, the fp32 path): the token-by-token
//    form, two dot products and the update per token on CUDA cores.
#include <cuda_runtime.h>

#include "dn.h"
#include "dn_device.cuh"
#include "dn_internal.h"
#include "dn_mma.cuh"
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
    grid_dep_wait();
    grid_dep_trigger();

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


// ---------------------------------------------------------------------------------------
// WY (chunkwise) form of one verify block, fp16 state.
//
// With Gamma_t = g_0 ... g_t and delta_t = beta_t (v_t - g_t S_{t-1} k_t), the rule
// S_t = g_t S_{t-1} + delta_t k_t^T unrolls to (gated delta rule, chunkwise form)
//
//   S_t     = Gamma_t S0 + sum_{s<=t} (Gamma_t / Gamma_s) delta_s k_s^T
//   delta_t = beta_t ( v_t - Gamma_t (S0 k_t) - sum_{s<t} L[t][s] delta_s ),
//             L[t][s] = (Gamma_t / Gamma_s) (k_t . k_s)
//   o_t     = Gamma_t (S0 q_t) + sum_{s<=t} M[t][s] delta_s,
//             M[t][s] = (Gamma_t / Gamma_s) (q_t . k_s)
//
// Gamma ratios are formed as exp(G_t - G_s) with G the running sum of log g, so
// they never exceed 1. Per CTA (32 rows of one head):
//   1. S0 rows, k_t and q_t go to shared memory as fp16 (the contraction operands);
//   2. mma.sync m16n8k16 (fp16 in, fp32 accumulate): proj[32 x 32] = S0 [K;Q]^T and
//      gram[32 x 16] = [K;Q] K^T;
//   3. L, M and Gamma (16 x 16 per head) from gram and the gates;
//   4. one lane per row solves delta_t by forward substitution;
//   5. every lane applies S_t = g_t S_{t-1} + delta_t k_t^T to its 16 fp32 state
//      elements with packed fp32x2 FMAs, reading k_t from the fp16 tile of step 1 (one
//      16-byte read per 8 elements; fp16 -> fp32 is exact), and streams the fp16 checkpoint;
//   6. o_t from proj, M and delta.
// The contraction is a few dozen m16n8k16 MMAs per CTA; its job is to remove the
// two per-token dot products (two FMAs per state element per token) from the
// store-bound loop, not throughput, so warp-level MMAs fit it (no TMEM round trip).

__device__ __forceinline__ uint4 pack8_half2(const float2 *s) {
    uint4 u;
    __half2 *h = reinterpret_cast<__half2 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __float22half2_rn(s[i]);
    return u;
}

// CKPT: write the T checkpoints (dn_verify_block); otherwise write delta_t instead
// (dn_verify_block_deltas), from which dn_commit_deltas rebuilds the accepted state.
// TM: the block capacity the shared tiles are sized for (16, or 8 for blocks of up to 8
// tokens, whose smaller tiles let more CTAs share an SM).
// ROWS: the state rows of a CTA (32, or 64 so that the head's state-independent work -- the
// k/q tiles, the grams, L and M, the gate scan -- is shared by twice the rows).
static_assert(DN_MAX_BLOCK == 16, "tile capacities 8 and 16");
template <int DK, bool CKPT, int TM, int ROWS>
__global__ void __launch_bounds__(256, ROWS == 64 ? (CKPT ? 4 : 5) : (ROWS == 16 ? 6 : (TM == 8 ? 6 : 5)))
verify_wy_kernel(int H, int T, int DV, const __half *__restrict__ q, const __half *__restrict__ k,
                 const __half *__restrict__ v, const float *__restrict__ beta,
                 const float *__restrict__ g, const __half *__restrict__ s_in,
                 __half *__restrict__ out, __half *__restrict__ ckpt, float *__restrict__ delta) {
    constexpr int NT = 256, TPR = NT / ROWS;  // threads per state row
    constexpr int CPR = DK / 8;        // 16-byte chunks per row
    constexpr int NCH = CPR / TPR;     // chunks per lane
    constexpr int KS = DK / 16;        // MMA k-steps
    __shared__ __align__(128) uint4 sS0[ROWS * CPR];
    __shared__ __align__(128) uint4 sKQ[2 * TM * CPR];  // rows 0..TM-1 k_t, TM..2TM-1 q_t
    __shared__ float proj[ROWS][2 * TM + 1];              // [row][t] S0 k_t, [row][TM+t] S0 q_t
    __shared__ float sL[TM][TM], sM[TM][TM];
    __shared__ float sgam[TM], sG[TM], sbeta[TM], sg[TM];
    __shared__ __align__(16) __half sv[TM][ROWS];
    __shared__ float sd[TM][ROWS];

    const int rblocks = DV / ROWS;
    const int rb = blockIdx.x % rblocks;
    const int h = (blockIdx.x / rblocks) % H;
    const size_t n = blockIdx.x / (rblocks * H);
    const int tid = threadIdx.x, lr = tid / TPR, ln = tid % TPR, row = rb * ROWS + lr;
    const int warp = tid / 32, lane = tid % 32;
    const size_t set_elems = (size_t)DV * DK;
    static_assert(NCH >= 1, "a lane holds at least one 16-byte chunk of its row");
    grid_dep_wait();
    grid_dep_trigger();

    // 1. The state rows, k_t and q_t (zeros past T) and the rows' v_t go to shared memory by
    //    cp.async, all in flight at once (one memory latency for the prologue); the gates load
    //    meanwhile. After the barrier each lane takes its state chunks to fp32 registers.
    {
        const __half *sp = s_in + (n * H + h) * set_elems + (size_t)row * DK;
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int j = c * TPR + ln;
            cp_async16(&sS0[hsw<CPR>(lr, j)], sp + j * 8, 16);
        }
    }
    for (int i = tid; i < TM * CPR; i += NT) {
        const int t = i / CPR, j = i % CPR;
        const bool live = t < T;
        const size_t off = live ? ((n * T + t) * H + h) * DK + (size_t)j * 8 : 0;
        cp_async16(&sKQ[hsw<CPR>(t, j)], k + off, live ? 16 : 0);
        cp_async16(&sKQ[hsw<CPR>(TM + t, j)], q + off, live ? 16 : 0);
    }
    for (int i = tid; i < T * (ROWS / 8); i += NT) {
        const int t = i / (ROWS / 8), j = i % (ROWS / 8);
        cp_async16(&sv[t][8 * j], v + ((n * T + t) * H + h) * DV + rb * ROWS + 8 * j, 16);
    }
    cp_async_commit();
    if (warp == 0) {
        // G_t = sum_{r<=t} log g_r: inclusive scan over lanes 0..15
        float lg = 0.f, gg = 1.f, bb = 0.f;
        if (lane < T) {
            gg = g[(n * T + lane) * H + h];
            bb = beta[(n * T + lane) * H + h];
            lg = logf(fmaxf(gg, 1e-30f));
        }
#pragma unroll
        for (int off = 1; off < TM; off <<= 1) {
            const float o = __shfl_up_sync(0xffffffffu, lg, off);
            if (lane >= off) lg += o;
        }
        if (lane < TM) {
            sG[lane] = lg;
            sgam[lane] = expf(lg);
            sg[lane] = gg;
            sbeta[lane] = bb;
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    float2 s[NCH * 4];  // this lane's state chunks c*TPR + ln, fp32
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const uint4 u = sS0[hsw<CPR>(lr, c * TPR + ln)];
        const __half2 *h2 = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) s[c * 4 + i] = __half22float2(h2[i]);
    }

    // 2. proj = S0 [K;Q]^T in 16x8 tiles; [K;Q] K^T, turned in registers into L (strictly
    //    lower) and M (lower including the diagonal):
    //    L[t][s] = e^{G_t - G_s} k_t.k_s (s < t), M[t][s] = e^{G_t - G_s} q_t.k_s (s <= t)
    constexpr int NG = TM / 8, MG = 2 * TM / 16;  // gram tiles: n (tokens of K), m (rows of [K;Q])
    auto proj_epi = [&](int m, int nn, const float (&d)[4]) {
        const int r0 = m * 16 + (lane >> 2), c0 = nn * 8 + 2 * (lane & 3);
        proj[r0][c0] = d[0];
        proj[r0][c0 + 1] = d[1];
        proj[r0 + 8][c0] = d[2];
        proj[r0 + 8][c0 + 1] = d[3];
    };
    auto gram_epi = [&](int m, int nn, const float (&e)[4]) {
        const int g0 = m * 16 + (lane >> 2), h0 = nn * 8 + 2 * (lane & 3);
        auto put = [&](int gr, int s2, float val) {  // gram row gr: k_t (gr < TM) or q_t (gr = TM + t)
            const int t = gr < TM ? gr : gr - TM;
            const bool keep = gr < TM ? (s2 < t) : (s2 <= t);
            const float r = keep ? expf(sG[t] - sG[s2]) * val : 0.f;
            if (gr < TM) sL[t][s2] = r;
            else sM[t][s2] = r;
        };
        put(g0, h0, e[0]);
        put(g0, h0 + 1, e[1]);
        put(g0 + 8, h0, e[2]);
        put(g0 + 8, h0 + 1, e[3]);
    };
    auto proj_tile = [&](int mt, int nt) {
        float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            unsigned a[4], b[2];
            ldsm_x4(a, &sS0[hsw<CPR>(mt * 16 + (lane & 15), 2 * ks + (lane >> 4))]);
            ldsm_x2(b, &sKQ[hsw<CPR>(nt * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1))]);
            mma_16816(d, a, b);
        }
        proj_epi(mt, nt, d);
    };
    auto gram_tile = [&](int gm, int gn) {
        float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            unsigned a[4], b[2];
            ldsm_x4(a, &sKQ[hsw<CPR>(gm * 16 + (lane & 15), 2 * ks + (lane >> 4))]);
            ldsm_x2(b, &sKQ[hsw<CPR>(gn * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1))]);
            mma_16816(e, a, b);
        }
        gram_epi(gm, gn, e);
    };
    if constexpr (ROWS == 64) {
        constexpr int PN = 2 * TM / 8, PTILES = (ROWS / 16) * PN, GTILES = MG * NG, NWARP = NT / 32;
        // 64-row CTAs: every warp holds PPW projection tiles (warp, warp + 8) and warps 7, 6, ..
        // a gram tile too; the tiles' k-loops run side by side, each with its own accumulator,
        // in the same order as one tile alone.
        constexpr int PPW = PTILES / NWARP;
        static_assert(PTILES % NWARP == 0 && PPW <= 2 && GTILES <= NWARP, "tiles per warp");
        const bool hasg = NWARP - 1 - warp < GTILES;
        const int q2 = NWARP - 1 - warp;
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
        const int m0 = warp / PN, n0 = warp % PN, m1 = (warp + NWARP) / PN, n1 = (warp + NWARP) % PN;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            unsigned a[4], b[2];
            ldsm_x4(a, &sS0[hsw<CPR>(m0 * 16 + (lane & 15), 2 * ks + (lane >> 4))]);
            ldsm_x2(b, &sKQ[hsw<CPR>(n0 * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1))]);
            mma_16816(d0, a, b);
            if constexpr (PPW == 2) {
                ldsm_x4(a, &sS0[hsw<CPR>(m1 * 16 + (lane & 15), 2 * ks + (lane >> 4))]);
                ldsm_x2(b, &sKQ[hsw<CPR>(n1 * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1))]);
                mma_16816(d1, a, b);
            }
            if (hasg) {
                ldsm_x4(a, &sKQ[hsw<CPR>((q2 / NG) * 16 + (lane & 15), 2 * ks + (lane >> 4))]);
                ldsm_x2(b, &sKQ[hsw<CPR>((q2 % NG) * 8 + (lane & 7), 2 * ks + ((lane >> 3) & 1))]);
                mma_16816(e, a, b);
            }
        }
        proj_epi(m0, n0, d0);
        if constexpr (PPW == 2) proj_epi(m1, n1, d1);
        if (hasg) gram_epi(q2 / NG, q2 % NG, e);
    } else {
        if constexpr (ROWS == 32) {  // warp = (m tile) * 4 + (n tile)
            if ((warp & 3) * 8 < 2 * TM) {
                proj_tile(warp >> 2, warp & 3);
                if (warp < MG * NG) gram_tile(warp / NG, warp % NG);
            }
        } else {
            constexpr int PN = 2 * TM / 8, PTILES = (ROWS / 16) * PN;
            for (int tile = warp; tile < PTILES; tile += NT / 32) proj_tile(tile / PN, tile % PN);
            if (warp < MG * NG) gram_tile(warp / NG, warp % NG);
        }
    }
    __syncthreads();

    // 4. delta_t by forward substitution, one lane per row
    if (warp * 32 + lane < ROWS) {
        const int rl = warp * 32 + lane;  // the row of this lane
        float dl[TM];
#pragma unroll
        for (int t = 0; t < TM; ++t) {
            dl[t] = 0.f;
            if (t < T) {
                float acc = 0.f;
#pragma unroll
                for (int s2 = 0; s2 < t; ++s2) acc = fmaf(sL[t][s2], dl[s2], acc);
                dl[t] = sbeta[t] * (__half2float(sv[t][rl]) - sgam[t] * proj[rl][t] - acc);
                sd[t][rl] = dl[t];
            }
        }
    }
    __syncthreads();

    if (!CKPT) {  // 5'. delta_t for the rows of this CTA: [N][T][H][DV] fp32
        for (int i = tid; i < T * ROWS; i += NT) {
            const int t = i / ROWS, r = i % ROWS;
            delta[((n * T + t) * H + h) * DV + rb * ROWS + r] = sd[t][r];
        }
    }
    // 5. checkpoints S_t = g_t S_{t-1} + delta_t k_t^T
    __half *dst = CKPT ? ckpt + ((n * T) * H + h) * set_elems + (size_t)row * DK + ln * 8 : nullptr;
    const size_t tstride = (size_t)H * set_elems;
    for (int t = 0; CKPT && t < T; ++t) {
        const float dt = sd[t][lr], gt = sg[t];
        const float2 d2 = make_float2(dt, dt), g2 = make_float2(gt, gt);
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const uint4 ku = sKQ[hsw<CPR>(t, c * TPR + ln)];  // k_t, 8 fp16 values (exact in fp32)
            const __half2 *kh = reinterpret_cast<const __half2 *>(&ku);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                s[c * 4 + i] = __ffma2_rn(d2, __half22float2(kh[i]), __fmul2_rn(g2, s[c * 4 + i]));
            __stcs(reinterpret_cast<uint4 *>(dst + c * TPR * 8), pack8_half2(&s[c * 4]));
        }
        dst += tstride;
    }

    // 6. outputs, stored straight from registers (consecutive threads, consecutive rows). In
    //    64-row CTAs a thread's four outputs are unrolled so that their sums run side by side.
    if constexpr (ROWS == 64) {
        constexpr int KO = (TM * ROWS + NT - 1) / NT;
#pragma unroll
        for (int k2 = 0; k2 < KO; ++k2) {
            const int i = tid + k2 * NT;
            if (i < T * ROWS) {
                const int t = i / ROWS, r = i % ROWS;
                float o = sgam[t] * proj[r][TM + t];
                for (int s2 = 0; s2 <= t; ++s2) o = fmaf(sM[t][s2], sd[s2][r], o);
                out[((n * T + t) * H + h) * DV + rb * ROWS + r] = __float2half_rn(o);
            }
        }
    } else {
        for (int i = tid; i < T * ROWS; i += NT) {
            const int t = i / ROWS, r = i % ROWS;
            float o = sgam[t] * proj[r][TM + t];
            for (int s2 = 0; s2 <= t; ++s2) o = fmaf(sM[t][s2], sd[s2][r], o);
            out[((n * T + t) * H + h) * DV + rb * ROWS + r] = __float2half_rn(o);
        }
    }
}

constexpr int kRows = 32;
constexpr int kTpr = 8;

// State rows per CTA of verify_wy_kernel. With checkpoints, 32: the rows' state lives in
// registers for the update, and 64-row CTAs measured slower (fewer CTAs per SM, spills at
// T = 16). A launch of a few state sets (one layer of one request: 48 heads, 192 CTAs of 32
// rows on 152 SMs) leaves some SMs with two CTAs' stores and others with one, so such
// launches take 16-row CTAs (dk = 128, 16 lanes per row): twice the CTAs, an even spread,
// each repeating its head's small state-independent work. Writing deltas, 64: no state in
// registers, and the head's state-independent work is shared by twice the rows (a whole head
// per CTA measured slower again).
constexpr int kWyRowsCkpt = 32, kWyRowsCkptSmall = 16, kWyRowsDelta = 64;
// Blocks of up to kWyShortBlock tokens in large launches: 64-row CTAs, so the head's prologue
// (k/q tiles, grams, gates, L and M) is shared by twice the rows against only a few
// checkpoint stores per row.
constexpr int kWyRowsCkptShort = 64, kWyShortBlock = 4;

template <int DK, bool CKPT, int TM, int R>
void launch_verify_wy_rows(int N, int H, int T, int dv, const __half *q, const __half *k, const __half *v,
                           const float *beta, const float *g, const __half *s_in, __half *out, __half *ckpt,
                           float *delta, cudaStream_t st) {
    const unsigned blocks = (unsigned)((long long)N * H * (dv / R));
    launch_pdl(verify_wy_kernel<DK, CKPT, TM, R>, dim3(blocks), dim3(256), 0, st, H, T, dv, q, k, v, beta, g,
               s_in, out, ckpt, delta);
}

template <int DK, bool CKPT, int TM>
void launch_verify_wy(int N, int H, int T, int dv, const __half *q, const __half *k, const __half *v,
                      const float *beta, const float *g, const __half *s_in, __half *out, __half *ckpt,
                      float *delta, cudaStream_t st) {
    if constexpr (!CKPT) {
        launch_verify_wy_rows<DK, CKPT, TM, kWyRowsDelta>(N, H, T, dv, q, k, v, beta, g, s_in, out, ckpt, delta, st);
        return;
    } else {
        const long long ctas32 = (long long)N * H * (dv / kWyRowsCkpt);
        const bool few = ctas32 < 2LL * device_sm_count();
        if constexpr (DK == 128) {
            // fewer 32-row CTAs than two per SM: the 16-row CTAs spread the stores evenly
            if (few) {
                launch_verify_wy_rows<DK, CKPT, TM, kWyRowsCkptSmall>(N, H, T, dv, q, k, v, beta, g, s_in, out, ckpt,
                                                                      delta, st);
                return;
            }
        }
        if constexpr (TM == 8) {
            if (!few && T <= kWyShortBlock) {
                launch_verify_wy_rows<DK, CKPT, TM, kWyRowsCkptShort>(N, H, T, dv, q, k, v, beta, g, s_in, out, ckpt,
                                                                      delta, st);
                return;
            }
        }
        launch_verify_wy_rows<DK, CKPT, TM, kWyRowsCkpt>(N, H, T, dv, q, k, v, beta, g, s_in, out, ckpt, delta, st);
    }
}

template <int DK, typename IO, typename ST>
void launch_verify(int N, int H, int T, int dv, const void *q, const void *k, const void *v,
                   const float *beta, const float *g, const void *s_in, void *out, void *ckpt,
                   cudaStream_t st) {
    const long long blocks = (long long)N * H * (dv / kRows);
    launch_pdl(verify_block_kernel<DK, kRows, kTpr, IO, ST>, dim3((unsigned)blocks), dim3(kRows * kTpr), 0, st, H,
               T, dv, static_cast<const IO *>(q), static_cast<const IO *>(k), static_cast<const IO *>(v), beta, g,
               static_cast<const ST *>(s_in), static_cast<IO *>(out), static_cast<ST *>(ckpt));
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
        const __half *qh = static_cast<const __half *>(q), *kh = static_cast<const __half *>(k);
        const __half *vh = static_cast<const __half *>(v), *sh = static_cast<const __half *>(state_in);
        __half *oh = static_cast<__half *>(out), *ch = static_cast<__half *>(ckpt);
        if (dk == 128 && T <= 8)
            launch_verify_wy<128, true, 8>(N, H, T, dv, qh, kh, vh, beta, g, sh, oh, ch, nullptr, st);
        else if (dk == 128)
            launch_verify_wy<128, true, kMaxT>(N, H, T, dv, qh, kh, vh, beta, g, sh, oh, ch, nullptr, st);
        else if (T <= 8)
            launch_verify_wy<64, true, 8>(N, H, T, dv, qh, kh, vh, beta, g, sh, oh, ch, nullptr, st);
        else
            launch_verify_wy<64, true, kMaxT>(N, H, T, dv, qh, kh, vh, beta, g, sh, oh, ch, nullptr, st);
    } else {
        if (dk == 128) launch_verify<128, float, float>(N, H, T, dv, q, k, v, beta, g, state_in, out, ckpt, st);
        else launch_verify<64, float, float>(N, H, T, dv, q, k, v, beta, g, state_in, out, ckpt, st);
    }
    return launch_status();
}

extern "C" dn_status dn_verify_block_deltas(int N, int H, int T, int dk, int dv, dn_dtype io_dt,
                                            dn_dtype state_dt, const void *q, const void *k,
                                            const void *v, const float *beta, const float *g,
                                            const void *state_in, void *out, float *delta,
                                            dn_stream_t stream) {
    using namespace dn;
    if (N < 0 || H < 1 || T < 1 || T > DN_MAX_BLOCK) return DN_ERR_INVALID_ARG;
    if (!dtype_ok(io_dt) || !dtype_ok(state_dt)) return DN_ERR_INVALID_ARG;
    if (!head_dim_ok(dk) || !head_dim_ok(dv)) return DN_ERR_UNSUPPORTED;
    if (io_dt != DN_F16 || state_dt != DN_F16) return DN_ERR_UNSUPPORTED;
    if (N == 0) return DN_OK;
    if (!q || !k || !v || !beta || !g || !state_in || !out || !delta) return DN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(state_in, 16) ||
        !aligned(out, 16) || !aligned(delta, 16) || !aligned(beta, 4) || !aligned(g, 4))
        return DN_ERR_INVALID_ARG;
    if ((long long)N * H * (dv / kRows) > 0x7fffffffLL) return DN_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const __half *qh = static_cast<const __half *>(q), *kh = static_cast<const __half *>(k);
    const __half *vh = static_cast<const __half *>(v), *sh = static_cast<const __half *>(state_in);
    __half *oh = static_cast<__half *>(out);
    if (dk == 128 && T <= 8)
        launch_verify_wy<128, false, 8>(N, H, T, dv, qh, kh, vh, beta, g, sh, oh, nullptr, delta, st);
    else if (dk == 128)
        launch_verify_wy<128, false, kMaxT>(N, H, T, dv, qh, kh, vh, beta, g, sh, oh, nullptr, delta, st);
    else if (T <= 8)
        launch_verify_wy<64, false, 8>(N, H, T, dv, qh, kh, vh, beta, g, sh, oh, nullptr, delta, st);
    else
        launch_verify_wy<64, false, kMaxT>(N, H, T, dv, qh, kh, vh, beta, g, sh, oh, nullptr, delta, st);
    return launch_status();
}
