// Chunkwise prefill on the fifth-generation tensor cores (tcgen05, accumulators in tensor
// memory), fp16 state and io, dk = dv = 128: a prompt through the gated delta rule with a
// state checkpoint every 64 tokens, for prefix caching of the DeltaNet state ("HyperQwen:
// 1,000 tok/s on a Single RTX 3090 ...", Technical Insight).
//
// Per 64-token chunk, from the chunk-start state S0 (dv x dk, exactly the fp16 carry), with
// G_t the cumulative log gate from the chunk start, gam_t = e^{G_t}, dec_s = e^{G_63 - G_s}:
//   A[t][s]  = beta_t e^{G_t - G_s} (k_t . k_s)   (s < t)     T = (I + A)^{-1} diag(beta)
//   Mq[t][s] = e^{G_t - G_s} (q_t . k_s)          (s <= t)
//   U = T V,  W = T diag(gam) K                   (state independent)
//   delta    = U - W S0^T                          (= beta_t (v_t - g_t S_{t-1} k_t) for every t)
//   o_t      = gam_t S0 q_t + sum_s Mq[t][s] delta_s
//   S64      = gam_63 S0 + delta^T diag(dec) K
// which is the token-by-token rule summed over the chunk. The carry is rounded to fp16 at
// every chunk end and stored as the checkpoint, so a restored run continues bit-identically.
//
// One CTA per (sequence, head), two warp roles joined by named barriers:
//  * prep (8 warps), a chunk ahead: q/k/v by tensor-map (TMA) loads; the grams [K;Q] K^T
//    by one MMA into tensor memory; A and Mq with their decays; T by blocks: the 16 x 16
//    diagonal blocks of (I + A)^{-1} by forward substitution in fp32, the blocks below
//    them by warp-level MMAs (four warps, one per 16 columns); U^T = V^T T^T (left in tensor
//    memory) and W^T = K^T (T diag gam)^T by MMA; W and K scaled by dec written back to
//    shared memory as MMA operands.
//  * chain (8 warps, state row i = tensor-memory lane i, two threads per row splitting the
//    columns): one MMA for S0 [W;Q]^T,
//    delta in registers, one MMA pair for delta Mq^T and delta^T (dec K), then the output
//    tile and, at a full chunk, the new carry as the checkpoint (both by TMA store; the
//    carry tile stays in shared memory as the next chunk's MMA operand).
// Every operand tile is in the 128-byte-swizzled layout that the TMA engine writes, so
// the same shared memory feeds TMA and the tensor cores.
#include <cstring>

#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "dn.h"
#include "dn_internal.h"
#include "dn_mma.cuh"
#include "dn_tc05.cuh"
#include "dn_tmap.h"

namespace dn {
namespace {

constexpr int kC = 64;            // tokens per chunk = checkpoint interval
constexpr int kRoleThreads = 256; // 8 chain warps, then 8 prep warps
constexpr int kTcThreads = 2 * kRoleThreads;
constexpr int kTcTries = 1 << 22; // polls before a wait is reported as run out

// tensor-memory columns (128 lanes each)
constexpr uint32_t kColDW = 0;    // S0 W^T, then delta Mq^T      (64)
constexpr uint32_t kColDQ = 64;   // S0 Q^T                        (64)
constexpr uint32_t kColDS = 128;  // delta^T (dec K)               (128)
constexpr uint32_t kColU = 256;   // U^T, two chunk parities       (2 x 64)
constexpr uint32_t kColScr = 384; // prep: grams, then W^T         (64)
constexpr int kTmemCols = 512;

// named barriers (0 is __syncthreads)
constexpr int kBFull = 1, kBEmpty = 3, kBWFree = 5, kBPrep = 6, kBChain = 7;

// Shared memory (bytes). 128-byte-swizzled tiles start on 1024-byte boundaries.
struct TcSmem {
    static constexpr uint32_t kKQ = 0;          // [3 stages][2 dk boxes][128 rows][128 B]: k rows 0-63, q rows 64-127
    static constexpr uint32_t kStage = 32768, kKQBox = 16384;
    static constexpr uint32_t kV = 98304;       // [2 dv boxes][64 tokens][128 B]
    static constexpr uint32_t kW = 114688;      // [2 dk boxes][64 tokens][128 B]
    static constexpr uint32_t kMq = 131072;     // [2 parities][64 t][128 B (64 s)]
    static constexpr uint32_t kT = 147456;      // T = X diag(beta) at +0, T diag(gam) at +8192: fp16 [64 t][128 B (64 s)]
    static constexpr uint32_t kAt = 163840;     // fp16 [64 t][72]: e^{G_t - G_s} (k_t . k_s), s < t
    static constexpr uint32_t kLinv = kAt + 64 * 72 * 2;       // fp16 [4][16][16]: inverses of the diagonal blocks of I + A
    static constexpr uint32_t kAjj = kLinv + 4 * 16 * 16 * 2;  // fp32 [4][16][16]: diagonal blocks of A
    static constexpr uint32_t kG = kAjj + 4 * 16 * 16 * 4;     // fp32 [2 parities][64]: cumulative log gate
    static constexpr uint32_t kDec = kG + 2 * kC * 4;          // fp32 [2 parities][64]: e^{G_63 - G_s}
    static constexpr uint32_t kCk = 180224;     // carry: [2 dk boxes][128 dv rows][128 B]
    static constexpr uint32_t kD = 212992;      // delta [128 dv rows][128 B (64 t)]; output boxes [2][64 t][128 B] alias it
    static constexpr uint32_t kGates = 229376;  // fp32 [2 parities][beta | g][64]
    static constexpr uint32_t kGam = kGates + 2 * 2 * kC * 4;  // fp32 [3][64]: e^{G_t} (chunk c in slot c % 3)
    static constexpr uint32_t kE = kGam + 3 * kC * 4;          // fp32 [2 parities][64]: e^{G_end(block of s) - G_s}
    static constexpr uint32_t kMbar = kE + 2 * kC * 4;         // q/k stages x3, v, prep MMA, chain MMA
    static constexpr uint32_t kTslot = kMbar + 6 * 8;
    static constexpr uint32_t kBytes = kTslot + 16;
};
static_assert(TcSmem::kDec + 2 * kC * 4 <= TcSmem::kCk, "prep scratch overlaps the carry tile");
static_assert(TcSmem::kBytes <= 232448, "shared memory above the per-block limit");

// Count of waits that ran out (read by dn_prefill_wait_timeouts).
__device__ unsigned int g_prefill_tc_timeouts;

struct TcMaps {
    CUtensorMap q, k, v, o, ck;
};

__device__ __forceinline__ void tc_wait(unsigned long long *mb, unsigned parity, int lane) {
    if (!mbar_wait(mb, parity, kTcTries) && lane == 0) atomicAdd(&g_prefill_tc_timeouts, 1u);
}

// 16-byte chunk `ch` of row `r` in a 64-row tile of 128-byte rows (128-byte swizzle), in uint4 units.
__device__ __forceinline__ int sw_chunk(int r, int ch) { return r * 8 + (ch ^ (r & 7)); }

__global__ void __launch_bounds__(kTcThreads, 1)
prefill_tc_kernel(int H, int P, const __grid_constant__ TcMaps maps, const float *__restrict__ beta,
                  const float *__restrict__ g, const __half *s_in, __half *s_out, __half *ckpt) {
    using L = TcSmem;
    extern __shared__ __align__(1024) unsigned char smem[];
    float(*sGates)[2][kC] = reinterpret_cast<float(*)[2][kC]>(smem + L::kGates);
    float(*sGam)[kC] = reinterpret_cast<float(*)[kC]>(smem + L::kGam);
    float(*sG)[kC] = reinterpret_cast<float(*)[kC]>(smem + L::kG);
    float(*sDec)[kC] = reinterpret_cast<float(*)[kC]>(smem + L::kDec);
    float(*sE)[kC] = reinterpret_cast<float(*)[kC]>(smem + L::kE);
    __half *sAt = reinterpret_cast<__half *>(smem + L::kAt);
    __half(*sLinv)[16][16] = reinterpret_cast<__half(*)[16][16]>(smem + L::kLinv);
    float(*sAjj)[16][16] = reinterpret_cast<float(*)[16][16]>(smem + L::kAjj);
    unsigned long long *mb = reinterpret_cast<unsigned long long *>(smem + L::kMbar);  // 0-2 qk, 3 v, 4 prep, 5 chain
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::kTslot);

    const int h = blockIdx.x % H, n = blockIdx.x / H;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int nchunks = (P + kC - 1) / kC, nfull = P / kC;
    const size_t set_off = ((size_t)n * H + h) * 128 * 128;
    // Two warps share each tensor-memory lane quarter (warp & 3) and split the columns:
    // row = 32 (warp & 3) + lane, column half = (warp >> 2) & 1, in both roles.
    const int row = 32 * (warp & 3) + lane, half = (warp >> 2) & 1;

    if (tid == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(&mb[i], 1);
        fence_proxy_async();
    }
    if (warp == 0) tmem_alloc<kTmemCols>(tslot);
    if (tid < kRoleThreads) {  // chain: the initial state becomes the carry tile (half a row each)
#pragma unroll 1
        for (int q = 0; q < 8; ++q) {
            const int ch = 8 * half + q;
            uint4 u = make_uint4(0u, 0u, 0u, 0u);
            if (s_in) u = *reinterpret_cast<const uint4 *>(s_in + set_off + (size_t)row * 128 + ch * 8);
            *reinterpret_cast<uint4 *>(smem + L::kCk + half * 16384 + row * 128 + ((q ^ (row & 7)) * 16)) = u;
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's lane quarter

    if (tid >= kRoleThreads) {
        // ================================ prep ================================
        const int pt = tid - kRoleThreads;
        auto issue_qk = [&](int c) {  // k, q boxes of chunk c; beta, g by 4-byte cp.async
            const int p0 = c * kC, s = c % 3;
            unsigned char *st = smem + L::kKQ + s * L::kStage;
            if (pt == 0) {
                mbar_arrive_expect_tx(&mb[s], 4 * 8192);
                for (int x = 0; x < 2; ++x) {
                    tma_load_4d(st + x * L::kKQBox, &maps.k, 64 * x, h, p0, n, &mb[s]);
                    tma_load_4d(st + x * L::kKQBox + 8192, &maps.q, 64 * x, h, p0, n, &mb[s]);
                }
            }
            if (pt < 2 * kC) {
                const int which = pt / kC, t = pt % kC;
                const bool ok = p0 + t < P;
                const float *src = which ? g : beta;
                const size_t row0 = ((size_t)n * P + p0) * H + h;
                cp_async4(&sGates[c & 1][which][t], ok ? (const void *)(src + row0 + (size_t)t * H) : (const void *)src,
                          ok ? 4 : 0);
            }
        };
        auto issue_v = [&](int c) {
            if (pt == 0) {
                mbar_arrive_expect_tx(&mb[3], 2 * 8192);
                for (int x = 0; x < 2; ++x) tma_load_4d(smem + L::kV + x * 8192, &maps.v, 64 * x, h, c * kC, n, &mb[3]);
            }
        };
        // gates of chunk c from its beta / g (one warp, two tokens a lane): G_t = sum_{r<=t} log g_r
        // (0 past the prompt), gam_t = e^{G_t}, dec_t = e^{G_63 - G_t}, E_t = e^{G_end(block of t) - G_t}
        auto gates = [&](int c) {
            const int nc = min(kC, P - c * kC), gb = c & 1, t0 = 2 * lane;
            const float l0 = (t0 < nc) ? __logf(fmaxf(sGates[gb][1][t0], 1e-30f)) : 0.f;
            const float l1 = (t0 + 1 < nc) ? __logf(fmaxf(sGates[gb][1][t0 + 1], 1e-30f)) : 0.f;
            float G1 = l0 + l1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, G1, off);
                if (lane >= off) G1 += o;
            }
            const float G0 = G1 - l1;
            const float Gend = __shfl_sync(0xffffffffu, G1, 31), Gblk = __shfl_sync(0xffffffffu, G1, lane | 7);
            sG[gb][t0] = G0;
            sG[gb][t0 + 1] = G1;
            sGam[c % 3][t0] = __expf(G0);
            sGam[c % 3][t0 + 1] = __expf(G1);
            sDec[gb][t0] = __expf(Gend - G0);
            sDec[gb][t0 + 1] = __expf(Gend - G1);
            sE[gb][t0] = __expf(Gblk - G0);
            sE[gb][t0 + 1] = __expf(Gblk - G1);
        };
        if (nchunks > 0) {
            issue_qk(0);
            issue_v(0);
        }
        cp_async_commit();
        cp_async_wait<0>();
        bar_sync(kBPrep, kRoleThreads);
        if (nchunks > 0 && pt < 32) gates(0);
        for (int c = 0; c < nchunks; ++c) {
            const int p0 = c * kC, nc = min(kC, P - p0), s = c % 3, pb = c & 1;
            unsigned char *sK = smem + L::kKQ + s * L::kStage;
            if (c >= 2) bar_sync(kBEmpty + pb, kTcThreads);  // chain done with chunk c-2
            if (c + 1 < nchunks) issue_qk(c + 1);
            cp_async_commit();
            tc_wait(&mb[s], (unsigned)((c / 3) & 1), lane);
            tc_fence_before();
            bar_sync(kBPrep, kRoleThreads);  // k, q and the gates of chunk c ready; last chunk's scratch reads done
            tc_fence_after();
            if (pt == 0) {  // grams: [K;Q] (128 rows) x K^T -> scratch columns
                const uint32_t id = umma_idesc(128, 64, 0, 0);
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t a = smem_addr(sK + (ks >> 2) * L::kKQBox) + (ks & 3) * 32;
                    umma_f16(tmem + kColScr, desc_kmajor(a), desc_kmajor(a), id, ks > 0);
                }
                umma_commit(&mb[4]);
            }
            tc_wait(&mb[4], 0u, lane);
            tc_fence_after();
            {   // row `row` of [K;Q] K^T, columns 32 half .. +31 (two 16-token blocks). Decay
                // e^{G_t - G_s}: direct inside t's block; across blocks e^{G_t - G_end(b)} e^{G_end(b) - G_s},
                // both <= 1.
                const bool krow = row < kC;
                const int t = krow ? row : row - kC, bt = t >> 4;
                const int gb = c & 1;
                const float Gt = sG[gb][t], beta_t = sGates[gb][0][t];
                const int lim = krow ? t : t + 1;  // columns s < lim are kept
                uint32_t gr[32];
                tmem_ld32u(tq + kColScr + 32 * half, gr);
                float dd[16];  // e^{G_t - G_s} for s in t's own block (only used when that block is in this half)
#pragma unroll
                for (int e = 0; e < 16; ++e) dd[e] = __expf(Gt - sG[gb][16 * bt + e]);
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    const int b = 2 * half + bb;
                    const float fb = (b < bt) ? __expf(Gt - sG[gb][16 * b + 15]) : 0.f;
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float dcy = (b == bt) ? dd[e] : fb * sE[gb][16 * b + e];
                        v[e] = (16 * b + e < lim) ? dcy * __uint_as_float(gr[16 * bb + e]) : 0.f;
                    }
                    if (krow) {
                        uint4 *dst = reinterpret_cast<uint4 *>(sAt + t * 72 + 16 * b);
                        dst[0] = make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
                        dst[1] = make_uint4(pack_h2(v[8], v[9]), pack_h2(v[10], v[11]), pack_h2(v[12], v[13]),
                                            pack_h2(v[14], v[15]));
                        if (b == bt) {  // diagonal block, fp32, float4 groups swizzled by row
                            const int rl = t & 15;
                            float4 *aj = reinterpret_cast<float4 *>(&sAjj[bt][rl][0]);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4)
                                aj[q4 ^ ((rl >> 1) & 3)] = make_float4(beta_t * v[4 * q4], beta_t * v[4 * q4 + 1],
                                                                       beta_t * v[4 * q4 + 2], beta_t * v[4 * q4 + 3]);
                        }
                    } else {
                        uint4 *mq = reinterpret_cast<uint4 *>(smem + L::kMq + pb * 8192);
                        mq[sw_chunk(t, 2 * b)] =
                            make_uint4(pack_h2(v[0], v[1]), pack_h2(v[2], v[3]), pack_h2(v[4], v[5]), pack_h2(v[6], v[7]));
                        mq[sw_chunk(t, 2 * b + 1)] = make_uint4(pack_h2(v[8], v[9]), pack_h2(v[10], v[11]),
                                                                pack_h2(v[12], v[13]), pack_h2(v[14], v[15]));
                    }
                }
            }
            bar_sync(kBPrep, kRoleThreads);
            // Inverses of the diagonal 16 x 16 blocks of L = I + A (unit lower triangular), one
            // thread per (block, column): right-looking forward substitution in fp32.
            if (pt < kC) {
                const int jb = pt >> 4, col = pt & 15;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) x[i] = (i == col) ? 1.f : 0.f;
#pragma unroll
                for (int k = 0; k < 15; ++k) {
#pragma unroll
                    for (int i = k + 1; i < 16; ++i)
                        x[i] = fmaf(-sAjj[jb][i][(((k >> 2) ^ ((i >> 1) & 3)) << 2) | (k & 3)], x[k], x[i]);
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) sLinv[jb][i][col] = __float2half_rn(x[i]);
            }
            bar_sync(kBPrep, kRoleThreads);
            if (pt < 4 * 32) {  // Block solve: prep warp w owns columns 16w .. 16w+15 of X = L^{-1}, as
                // X^T (rows s, columns t): X^T_w = Linv_w^T, and for blocks j > w
                //   X^T_j = -(sum_{i=w}^{j-1} X^T_i At_ji^T) diag(beta_j) Linv_j^T
                // by warp-level MMAs. Then T = X diag(beta), T diag(gam) -> fp16 operand tiles [t][s].
                const int w = pt >> 5, fr = lane >> 2, fc = 2 * (lane & 3);
                const float *bs = sGates[c & 1][0];
                const float *gs = sGam[c % 3];
                const float br0 = bs[16 * w + fr], br1 = bs[16 * w + fr + 8];
                const float gr0 = br0 * gs[16 * w + fr], gr1 = br1 * gs[16 * w + fr + 8];
                uint4 *tt = reinterpret_cast<uint4 *>(smem + L::kT), *tg = reinterpret_cast<uint4 *>(smem + L::kT + 8192);
                const int m = lane >> 3;
                unsigned xa[4][4];
                float xc[2][4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j < w) {  // above the diagonal: zero tiles
                        const int trow = 16 * j + 8 * (m >> 1) + (lane & 7);
                        stsm_x4_t(tt + sw_chunk(trow, 2 * w + (m & 1)), 0u, 0u, 0u, 0u);
                        stsm_x4_t(tg + sw_chunk(trow, 2 * w + (m & 1)), 0u, 0u, 0u, 0u);
                        continue;
                    }
                    if (j == w) {
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            const int tl = 8 * nt + fc;
                            xc[nt][0] = __half2float(sLinv[w][tl][fr]);
                            xc[nt][1] = __half2float(sLinv[w][tl + 1][fr]);
                            xc[nt][2] = __half2float(sLinv[w][tl][fr + 8]);
                            xc[nt][3] = __half2float(sLinv[w][tl + 1][fr + 8]);
                        }
                    } else {
                        float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            if (i < w || i >= j) continue;
                            unsigned bb[4];
                            ldsm_x4(bb, sAt + (16 * j + (lane & 7) + ((lane >> 4) << 3)) * 72 + 16 * i + 8 * ((lane >> 3) & 1));
                            const unsigned b0[2] = {bb[0], bb[1]}, b1[2] = {bb[2], bb[3]};
                            mma_16816(y[0], xa[i], b0);
                            mma_16816(y[1], xa[i], b1);
                        }
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            const int tc = 16 * j + 8 * nt + fc;
                            const float nb0 = -bs[tc], nb1 = -bs[tc + 1];
                            y[nt][0] *= nb0; y[nt][1] *= nb1; y[nt][2] *= nb0; y[nt][3] *= nb1;
                        }
                        unsigned ya[4], bl[4];
                        acc_to_a(ya, y[0], y[1]);
                        ldsm_x4(bl, &sLinv[j][(lane & 7) + ((lane >> 4) << 3)][8 * ((lane >> 3) & 1)]);
                        const unsigned l0[2] = {bl[0], bl[1]}, l1[2] = {bl[2], bl[3]};
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) xc[nt][0] = xc[nt][1] = xc[nt][2] = xc[nt][3] = 0.f;
                        mma_16816(xc[0], ya, l0);
                        mma_16816(xc[1], ya, l1);
                    }
                    acc_to_a(xa[j], xc[0], xc[1]);
                    const int trow = 16 * j + 8 * (m >> 1) + (lane & 7);
                    stsm_x4_t(tt + sw_chunk(trow, 2 * w + (m & 1)), pack_h2(br0 * xc[0][0], br0 * xc[0][1]),
                              pack_h2(br1 * xc[0][2], br1 * xc[0][3]), pack_h2(br0 * xc[1][0], br0 * xc[1][1]),
                              pack_h2(br1 * xc[1][2], br1 * xc[1][3]));
                    stsm_x4_t(tg + sw_chunk(trow, 2 * w + (m & 1)), pack_h2(gr0 * xc[0][0], gr0 * xc[0][1]),
                              pack_h2(gr1 * xc[0][2], gr1 * xc[0][3]), pack_h2(gr0 * xc[1][0], gr0 * xc[1][1]),
                              pack_h2(gr1 * xc[1][2], gr1 * xc[1][3]));
                }
            }
            fence_proxy_async();
            tc_fence_before();
            bar_sync(kBPrep, kRoleThreads);
            tc_fence_after();
            if (pt == 0) {  // U^T = V^T T^T (kept for the chain), W^T = K^T (T diag gam)^T (scratch)
                tc_wait(&mb[3], (unsigned)(c & 1), 0);
                tc_fence_after();
                const uint32_t id = umma_idesc(128, 64, 1, 0);
                for (int ks = 0; ks < 4; ++ks) {
                    umma_f16(tmem + kColU + 64 * pb, desc_mnmajor(smem_addr(smem + L::kV) + ks * 2048, 8192),
                             desc_kmajor(smem_addr(smem + L::kT) + ks * 32), id, ks > 0);
                    umma_f16(tmem + kColScr, desc_mnmajor(smem_addr(sK) + ks * 2048, L::kKQBox),
                             desc_kmajor(smem_addr(smem + L::kT + 8192) + ks * 32), id, ks > 0);
                }
                umma_commit(&mb[4]);
            }
            cp_async_wait<0>();  // beta / g of chunk c+1 (issued above) landed; gates while U, W run
            bar_sync(kBPrep, kRoleThreads);
            if (c + 1 < nchunks && pt < 32) gates(c + 1);
            tc_wait(&mb[4], 1u, lane);
            tc_fence_after();
            if (c + 1 < nchunks) issue_v(c + 1);  // v of this chunk consumed
            if (c >= 1) bar_sync(kBWFree, kTcThreads);  // the chain's first MMA of chunk c-1 read W
            {   // W^T row `row` (dk index), tokens 32 half .. +31 -> W tile [t][dk]
                uint32_t r[32];
                tmem_ld32u(tq + kColScr + 32 * half, r);
                unsigned char *wb = smem + L::kW + (row >> 6) * 8192 + (row & 7) * 2;
                const int dch = (row & 63) >> 3;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int t = 32 * half + e;
                    *reinterpret_cast<__half *>(wb + t * 128 + ((dch ^ (t & 7)) * 16)) = __float2half_rn(__uint_as_float(r[e]));
                }
            }
            {   // K rows scaled by dec (in place: the chain's state update reads dec K); 4 chunks each
                const int bx = pt >> 7, sr = (pt >> 1) & 63, c4 = 4 * (pt & 1);
                const float2 f2 = make_float2(sDec[c & 1][sr], sDec[c & 1][sr]);
                unsigned char *rp = sK + bx * L::kKQBox + sr * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int ch = (c4 + q) ^ (sr & 7);
                    uint4 u = *reinterpret_cast<uint4 *>(rp + ch * 16);
                    __half2 *h2 = reinterpret_cast<__half2 *>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) h2[e] = __float22half2_rn(__fmul2_rn(f2, __half22float2(h2[e])));
                    *reinterpret_cast<uint4 *>(rp + ch * 16) = u;
                }
            }
            fence_proxy_async();
            tc_fence_before();
            bar_arrive(kBFull + pb, kTcThreads);  // chunk c ready for the chain
        }
    } else {
        // ================================ chain ================================
        for (int c = 0; c < nchunks; ++c) {
            const int p0 = c * kC, nc = min(kC, P - p0), s = c % 3, pb = c & 1;
            unsigned char *sK = smem + L::kKQ + s * L::kStage;
            bar_sync(kBFull + pb, kTcThreads);
            tc_fence_after();
            if (tid == 0) {
                bulk_wait_read();  // the previous stores have read the delta / output tile and the carry tile
                const uint32_t id = umma_idesc(128, 64, 0, 0);
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t a = desc_kmajor(smem_addr(smem + L::kCk + (ks >> 2) * 16384) + (ks & 3) * 32);
                    umma_f16(tmem + kColDW, a, desc_kmajor(smem_addr(smem + L::kW + (ks >> 2) * 8192) + (ks & 3) * 32),
                             id, ks > 0);
                    umma_f16(tmem + kColDQ, a,
                             desc_kmajor(smem_addr(sK + (ks >> 2) * L::kKQBox + 8192) + (ks & 3) * 32), id, ks > 0);
                }
                umma_commit(&mb[5]);
            }
            tc_wait(&mb[5], 0u, lane);
            tc_fence_after();
            if (c + 1 < nchunks) bar_arrive(kBWFree, kTcThreads);  // W read
            {   // delta = U - S0 W^T, row `row`, tokens 32 half .. +31 -> fp16 operand tile
                uint32_t a[32], u[32];
                tmem_ld32x2(tq + kColDW + 32 * half, a, tq + kColU + 64 * pb + 32 * half, u);
                uint4 *dr = reinterpret_cast<uint4 *>(smem + L::kD + row * 128);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_h2(__uint_as_float(u[8 * q + 2 * e]) - __uint_as_float(a[8 * q + 2 * e]),
                                       __uint_as_float(u[8 * q + 2 * e + 1]) - __uint_as_float(a[8 * q + 2 * e + 1]));
                    dr[(4 * half + q) ^ (row & 7)] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async();
            tc_fence_before();
            bar_sync(kBChain, kRoleThreads);
            tc_fence_after();
            if (tid == 0) {  // delta Mq^T -> DW columns; delta^T (dec K) -> DS columns
                const uint32_t idm = umma_idesc(128, 64, 0, 0), ids = umma_idesc(128, 128, 0, 1);
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t a = desc_kmajor(smem_addr(smem + L::kD) + ks * 32);
                    umma_f16(tmem + kColDW, a, desc_kmajor(smem_addr(smem + L::kMq + pb * 8192) + ks * 32), idm, ks > 0);
                    umma_f16(tmem + kColDS, a, desc_mnmajor(smem_addr(sK) + ks * 2048, L::kKQBox), ids, ks > 0);
                }
                umma_commit(&mb[5]);
            }
            tc_wait(&mb[5], 1u, lane);
            tc_fence_after();
            {   // o_t = gam_t (S0 q_t) + (delta Mq^T)_t, tokens 32 half .. +31 -> output boxes [t][dv]
                const float *gam = sGam[c % 3];
                unsigned char *ob = smem + L::kD + (row >> 6) * 8192 + (row & 7) * 2;
                const int rch = (row & 63) >> 3;
                uint32_t a[32], b[32];
                tmem_ld32x2(tq + kColDQ + 32 * half, a, tq + kColDW + 32 * half, b);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int t = 32 * half + e;
                    *reinterpret_cast<__half *>(ob + t * 128 + ((rch ^ (t & 7)) * 16)) =
                        __float2half_rn(fmaf(gam[t], __uint_as_float(a[e]), __uint_as_float(b[e])));
                }
            }
            {   // S64 = gam_63 S0 + delta^T (dec K) for dk 64 half .. +63: new carry (fp16),
                // checkpoint, final state
                const float gl = sGam[c % 3][kC - 1];
                __half *so = (c + 1 == nchunks) ? s_out + set_off + (size_t)row * 128 : nullptr;
#pragma unroll 1
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t ds[32];
                    tmem_ld32u(tq + kColDS + 64 * half + 32 * hq, ds);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int lq = 4 * hq + q, ch = 8 * half + lq;
                        unsigned char *cp = smem + L::kCk + half * 16384 + row * 128 + ((lq ^ (row & 7)) * 16);
                        uint4 u = *reinterpret_cast<uint4 *>(cp);
                        __half2 *h2 = reinterpret_cast<__half2 *>(&u);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(h2[e]);
                            h2[e] = __floats2half2_rn(fmaf(gl, f.x, __uint_as_float(ds[8 * q + 2 * e])),
                                                      fmaf(gl, f.y, __uint_as_float(ds[8 * q + 2 * e + 1])));
                        }
                        *reinterpret_cast<uint4 *>(cp) = u;
                        if (so) *reinterpret_cast<uint4 *>(so + ch * 8) = u;
                    }
                }
            }
            fence_proxy_async();
            tc_fence_before();
            if (c + 2 < nchunks) bar_arrive(kBEmpty + pb, kTcThreads);  // q/k stage, Mq, U, gam of chunk c consumed
            bar_sync(kBChain, kRoleThreads);
            if (tid == 0) {  // output boxes; at a full chunk the carry tile is the checkpoint
                for (int x = 0; x < 2; ++x) tma_store_4d(&maps.o, 64 * x, h, p0, n, smem + L::kD + x * 8192);
                if (nc == kC)
                    for (int x = 0; x < 2; ++x)
                        tma_store_3d(&maps.ck, 64 * x, 0, (n * nfull + c) * H + h, smem + L::kCk + x * 16384);
                bulk_commit();
            }
        }
        if (nchunks == 0) {  // empty prompt: the state passes through
#pragma unroll 1
            for (int q = 0; q < 8; ++q) {
                const int ch = 8 * half + q;
                uint4 u = make_uint4(0u, 0u, 0u, 0u);
                if (s_in) u = *reinterpret_cast<const uint4 *>(s_in + set_off + (size_t)row * 128 + ch * 8);
                *reinterpret_cast<uint4 *>(s_out + set_off + (size_t)row * 128 + ch * 8) = u;
            }
        }
        if (tid == 0) bulk_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_free<kTmemCols>(tmem);
}

// The kernel uses more than the default 48 KB of shared memory; the opt-in is a per-device
// function attribute, set once per device.
bool allow_tc_smem() {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const unsigned long long bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return true;
    if (cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)TcSmem::kBytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done.fetch_or(bit, std::memory_order_acq_rel);
    return true;
}

}  // namespace

dn_status launch_prefill_tc(int N, int H, int P, const void *q, const void *k, const void *v, const float *beta,
                            const float *g, const void *s_in, void *out, void *ckpt, void *s_out, cudaStream_t st) {
    if (!allow_tc_smem()) return DN_ERR_CUDA;
    TcMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (P > 0) {
        // q, k, v, out [N][P][H][128] as 4-d (d, head, token, sequence), 64 x 64 boxes
        const cuuint64_t dims[4] = {128, (cuuint64_t)H, (cuuint64_t)P, (cuuint64_t)N};
        const cuuint64_t str[3] = {256, (cuuint64_t)H * 256, (cuuint64_t)P * H * 256};
        const cuuint32_t box[4] = {64, 1, 64, 1};
        if (!encode_map(&maps.q, q, 4, dims, str, box) || !encode_map(&maps.k, k, 4, dims, str, box) ||
            !encode_map(&maps.v, v, 4, dims, str, box) || !encode_map(&maps.o, out, 4, dims, str, box))
            return DN_ERR_CUDA;
    }
    if (P >= kC) {
        // ckpt [N][P/64][H][128][128] as 3-d (dk, dv, checkpoint tile); a box is 64 dk x 128 dv
        const cuuint64_t dims[3] = {128, 128, (cuuint64_t)N * (P / kC) * H};
        const cuuint64_t str[2] = {256, 128 * 256};
        const cuuint32_t box[3] = {64, 128, 1};
        if (!encode_map(&maps.ck, ckpt, 3, dims, str, box)) return DN_ERR_CUDA;
    }
    prefill_tc_kernel<<<(unsigned)((long long)N * H), kTcThreads, TcSmem::kBytes, st>>>(
        H, P, maps, beta, g, static_cast<const __half *>(s_in), static_cast<__half *>(s_out),
        static_cast<__half *>(ckpt));
    return DN_OK;
}

unsigned int prefill_tc_wait_timeouts() {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_prefill_tc_timeouts, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return 0xffffffffu;
    }
    return v;
}

}  // namespace dn
