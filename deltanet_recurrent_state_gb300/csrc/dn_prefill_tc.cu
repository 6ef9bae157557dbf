// Chunkwise prefill on the fifth-generation tensor cores (tcgen05, accumulators in tensor
// memory), fp16 state and io, dk = dv = 128: a prompt through the gated delta rule with a
// state checkpoint every 64 tokens, for prefix caching of the DeltaNet state ("HyperQwen:
// 1,000 tok/s on a Single RTX 3090 ...", Technical Insight).
//
// Per 64-token chunk, from the chunk-start state S0 (dv x dk, exactly the fp16 carry), with
// G_t the cumulative log gate from the chunk start, gam_t = e^{G_t}, dec_s = e^{G_63 - G_s}:
//   A[t][s]  = beta_t e^{G_t - G_s} (k_t . k_s)   (s < t)     T = (I + A)^{-1} diag(beta)
//   Mq[t][s] = e^{G_t - G_s} (q_t . k_s)          (s <= t)    (state independent)
//   R        = V - diag(gam) K S0^T
//   delta    = T R                                 (= beta_t (v_t - g_t S_{t-1} k_t) for every t)
//   O        = diag(gam) Q S0^T + Mq delta
//   S64      = gam_63 S0 + (diag(dec) delta)^T K
// which is the token-by-token rule summed over the chunk. The carry is rounded to fp16 at
// every chunk end and stored as the checkpoint, so a restored run continues bit-identically.
//
// Token-major products. Every matrix indexed by token (K S0^T, Q S0^T, delta, O) is an MMA
// accumulator with the token on the tensor-memory lane and dv along the columns, so each
// epilogue thread owns one token row and writes it as contiguous 16-byte pieces. A 64-token
// operand fills half of an M = 128 MMA: [K; Q] S0^T uses both halves (K rows 0-63, Q rows
// 64-127); T R and Mq delta read a 128-row window of which only the T (rows 0-63) or the Mq
// half (rows 64-127) is kept, the other half of the accumulator being left unused.
//
// One CTA per (sequence, head), two warp roles joined by named barriers:
//  * prep (8 warps), a chunk ahead: the grams [K;Q] K^T by one MMA; A and Mq with their
//    decays; T by blocks (the 16 x 16 diagonal blocks of (I + A)^{-1} by forward
//    substitution in fp32, the blocks below them by warp-level MMAs), written as an fp16
//    operand tile; Q scaled by gam in place. beta and g come in by plain loads one chunk
//    ahead, into registers; the next chunk's grams start as soon as this chunk's are read.
//  * chain (8 warps): [K; gam Q] S0^T; R (warps on lanes 0-63); delta = T R, written twice:
//    as the operand tile and scaled by dec into the chunk's v buffer (v is consumed by then);
//    (dec delta)^T K and Mq delta accumulated onto the gam Q S0^T half; the new carry; the
//    output rows (into the v buffer again). Thread 64 issues the q/k/v tensor-map (TMA)
//    loads ahead of use and the TMA stores of the output rows and of the checkpoint (the
//    carry tile, which is also the next chunk's MMA operand); nothing on the chain waits
//    for a store except the reuse of a v buffer a chunk later.
// Every operand tile is in the 128-byte-swizzled layout that the TMA engine writes, so the
// same shared memory feeds TMA and the tensor cores.
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

// tensor-memory columns (128 lanes each)
constexpr uint32_t kColD1 = 0;    // [K; gam Q] S0^T, then + Mq delta; two chunk parities (2 x 128)
constexpr uint32_t kColD3 = 256;  // delta = T R, then delta^T (dec K)                      (128)
constexpr uint32_t kColGr = 384;  // prep: the grams [K;Q] K^T                               (64)
constexpr int kTmemCols = 512;

// named barriers (0 is __syncthreads)
constexpr int kBFull = 1, kBEmpty = 3, kBTFree = 5, kBPrep = 6, kBChain = 7, kBOut = 8, kBPrepK = 9;
constexpr int kSolveThreads = 128;  // prep warps 8-11: the block solve

// mbarriers
constexpr int kMbLoad = 0;  // q/k of a stage (3)
constexpr int kMbV = 3;     // v of a buffer (2)
constexpr int kMbGram = 5, kMbC1 = 6, kMbC2 = 7, kMbC3 = 8, kMbC4 = 9;
constexpr int kMbDrainChain = 10, kMbDrainPrep = 11;  // final drains of the two MMA issuers
constexpr int kNumMbar = 12;

// Shared memory (bytes). 128-byte-swizzled tiles start on 1024-byte boundaries.
struct TcSmem {
    static constexpr uint32_t kKQ = 0;          // [3 stages][2 dk boxes][128 rows][128 B]: k rows 0-63, q rows 64-127
    static constexpr uint32_t kStage = 32768, kKQBox = 16384;
    static constexpr uint32_t kV = 98304;       // [2 buffers][2 dv boxes][64 t][128 B]
    static constexpr uint32_t kVBuf = 16384;
    static constexpr uint32_t kCk = 131072;     // carry [2 dk boxes][128 dv rows][128 B]
    static constexpr uint32_t kR = 163840;      // R, then delta, then the output: [2 dv boxes][64 t][128 B]
    static constexpr uint32_t kT = 180224;      // T, fp16 [64 t][128 B (64 s)]; the junk half of delta's window
    static constexpr uint32_t kMq = 188416;     // [2 parities][64 t][128 B (64 s)]; the window of parity p starts 8 KB before
    static constexpr uint32_t kAt = 204800;     // fp16 [64 t][72]: e^{G_t - G_s} (k_t . k_s), s < t
    static constexpr uint32_t kLinv = kAt + 64 * 72 * 2;       // fp16 [4][16][16]: inverses of the diagonal blocks of I + A
    static constexpr uint32_t kAjj = kLinv + 4 * 16 * 16 * 2;  // fp32 [4][16][16]: diagonal blocks of A
    // gates, computed a chunk ahead: prep-only ones in slot c % 3, the chain's in slot c % 4
    static constexpr uint32_t kBeta = kAjj + 4 * 16 * 16 * 4;  // fp32 [3][64]
    static constexpr uint32_t kG = kBeta + 3 * kC * 4;         // fp32 [3][64]: cumulative log gate
    static constexpr uint32_t kE = kG + 3 * kC * 4;            // fp32 [3][64]: e^{G_end(block of s) - G_s}
    static constexpr uint32_t kGam = kE + 3 * kC * 4;          // fp32 [4][64]: e^{G_t}
    static constexpr uint32_t kDec = kGam + 4 * kC * 4;        // fp32 [4][64]: e^{G_63 - G_s}
    static constexpr uint32_t kMbar = kDec + 4 * kC * 4;
    static constexpr uint32_t kTslot = kMbar + kNumMbar * 8;
    static constexpr uint32_t kAbort = kTslot + 8;  // int: a wait ran out
    static constexpr uint32_t kBytes = kTslot + 16;
};
static_assert(TcSmem::kV == 3 * TcSmem::kStage && TcSmem::kCk == TcSmem::kV + 2 * TcSmem::kVBuf, "layout");
static_assert(TcSmem::kR == TcSmem::kCk + 32768 && TcSmem::kT == TcSmem::kR + 16384, "layout");
static_assert(TcSmem::kMq == TcSmem::kT + 8192 && TcSmem::kAt == TcSmem::kMq + 16384, "layout");
static_assert(TcSmem::kBytes <= 232448, "shared memory above the per-block limit");

// Count of waits that ran out (read by dn_prefill_wait_timeouts).
__device__ unsigned int g_prefill_tc_timeouts;

struct TcMaps {
    CUtensorMap q, k, v, o, ck;
};

// Bounded wait (kWaitBudgetNs). When one runs out, the CTA's abort flag goes up: from then on
// no copies or global stores are issued, every role still passes its named barriers to the
// end of its loop, the copies and MMAs issued are drained (bounded) and the CTA exits.
__device__ __forceinline__ void tc_wait(unsigned long long *mb, unsigned parity, volatile int *abort) {
    mbar_wait_guarded(mb, parity, abort, &g_prefill_tc_timeouts);
}

// 16-byte chunk `ch` of row `r` in a 64-row tile of 128-byte rows (128-byte swizzle), in uint4 units.
__device__ __forceinline__ int sw_chunk(int r, int ch) { return r * 8 + (ch ^ (r & 7)); }

// 32 accumulator columns (raw fp32 bits) -> four 16-byte fp16 chunks j0 .. j0+3 of swizzled row r.
__device__ __forceinline__ void put_row32(uint4 *row, int r, int j0, const uint32_t (&d)[32]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_h2(__uint_as_float(d[8 * q + 2 * e]), __uint_as_float(d[8 * q + 2 * e + 1]));
        row[(j0 + q) ^ (r & 7)] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__global__ void __launch_bounds__(kTcThreads, 1)
prefill_tc_kernel(int H, int P, const __grid_constant__ TcMaps maps, const float *__restrict__ beta,
                  const float *__restrict__ g, const __half *s_in, __half *s_out) {
    using L = TcSmem;
    extern __shared__ __align__(1024) unsigned char smem[];
    float(*sBeta)[kC] = reinterpret_cast<float(*)[kC]>(smem + L::kBeta);
    float(*sG)[kC] = reinterpret_cast<float(*)[kC]>(smem + L::kG);
    float(*sGam)[kC] = reinterpret_cast<float(*)[kC]>(smem + L::kGam);
    float(*sDec)[kC] = reinterpret_cast<float(*)[kC]>(smem + L::kDec);
    float(*sE)[kC] = reinterpret_cast<float(*)[kC]>(smem + L::kE);
    __half *sAt = reinterpret_cast<__half *>(smem + L::kAt);
    __half(*sLinv)[16][16] = reinterpret_cast<__half(*)[16][16]>(smem + L::kLinv);
    float(*sAjj)[16][16] = reinterpret_cast<float(*)[16][16]>(smem + L::kAjj);
    unsigned long long *mb = reinterpret_cast<unsigned long long *>(smem + L::kMbar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::kTslot);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L::kAbort);

    const int h = blockIdx.x % H, n = blockIdx.x / H;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int nchunks = (P + kC - 1) / kC, nfull = P / kC;
    const size_t set_off = ((size_t)n * H + h) * 128 * 128;
    // Two warps share each tensor-memory lane quarter (warp & 3) and split the columns:
    // lane row = 32 (warp & 3) + lane, column half = (warp >> 2) & 1, in both roles.
    const int row = 32 * (warp & 3) + lane, half = (warp >> 2) & 1;

    if (tid == 0) {
        for (int i = 0; i < kNumMbar; ++i) mbar_init(&mb[i], 1);
        *abort = 0;
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
        const int pt = tid - kRoleThreads, pw = pt >> 5;
        // beta and g of tokens 2 lane, 2 lane + 1 of the next chunk (warp 15), loaded a chunk ahead
        float gb0 = 0.f, gb1 = 0.f, gg0 = 1.f, gg1 = 1.f;
        auto fetch = [&](int c) {
            const int t0 = c * kC + 2 * lane;
            const size_t r0 = ((size_t)n * P + t0) * H + h;
            gb0 = (t0 < P) ? __ldg(beta + r0) : 0.f;
            gg0 = (t0 < P) ? __ldg(g + r0) : 1.f;
            gb1 = (t0 + 1 < P) ? __ldg(beta + r0 + H) : 0.f;
            gg1 = (t0 + 1 < P) ? __ldg(g + r0 + H) : 1.f;
        };
        // gates of chunk c (warp 15, two tokens a lane): G_t = sum_{r<=t} log g_r (0 past the
        // prompt), gam_t = e^{G_t}, dec_t = e^{G_63 - G_t}, E_t = e^{G_end(block of t) - G_t}
        auto gates = [&](int c) {
            const int nc = min(kC, P - c * kC), t0 = 2 * lane, g3 = c % 3, g4 = c % 4;
            const float l0 = (t0 < nc) ? __logf(fmaxf(gg0, 1e-30f)) : 0.f;
            const float l1 = (t0 + 1 < nc) ? __logf(fmaxf(gg1, 1e-30f)) : 0.f;
            float G1 = l0 + l1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float o = __shfl_up_sync(0xffffffffu, G1, off);
                if (lane >= off) G1 += o;
            }
            const float G0 = G1 - l1;
            const float Gend = __shfl_sync(0xffffffffu, G1, 31), Gblk = __shfl_sync(0xffffffffu, G1, lane | 7);
            sBeta[g3][t0] = (t0 < nc) ? gb0 : 0.f;
            sBeta[g3][t0 + 1] = (t0 + 1 < nc) ? gb1 : 0.f;
            sG[g3][t0] = G0;
            sG[g3][t0 + 1] = G1;
            sE[g3][t0] = __expf(Gblk - G0);
            sE[g3][t0 + 1] = __expf(Gblk - G1);
            sGam[g4][t0] = __expf(G0);
            sGam[g4][t0 + 1] = __expf(G1);
            sDec[g4][t0] = __expf(Gend - G0);
            sDec[g4][t0 + 1] = __expf(Gend - G1);
        };
        // Prep warps on lane quarters 0-1 (8, 9, 12, 13: the K warps) read the K rows of the grams
        // (A), those on quarters 2-3 (10, 11, 14, 15: the Q warps) the Q rows (Mq).
        auto grams = [&](int c) {  // warp 14: the grams MMA of chunk c once its k, q have landed
            tc_wait(&mb[kMbLoad + c % 3], (unsigned)((c / 3) & 1), abort);
            tc_fence_after();
            if (lane == 0) {  // [K;Q] (128 rows) x K^T
                unsigned char *sKc = smem + L::kKQ + (c % 3) * L::kStage;
                const uint32_t id = umma_idesc(128, 64, 0, 0);
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t a = smem_addr(sKc + (ks >> 2) * L::kKQBox) + (ks & 3) * 32;
                    umma_f16(tmem + kColGr, desc_kmajor(a), desc_kmajor(a), id, ks > 0);
                }
                umma_commit(&mb[kMbGram]);
            }
            __syncwarp();
        };
        if (nchunks > 0) {
            if (pw == 6) grams(0);
            if (pw == 7) {
                fetch(0);
                gates(0);
                if (nchunks > 1) fetch(1);
            }
        }
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % 3, p = c & 1;
            unsigned char *sK = smem + L::kKQ + s * L::kStage;
            if (c >= 2) bar_sync(kBEmpty + p, kTcThreads);  // the chain is done with chunk c-2 (Mq of parity p)
            bar_sync(kBPrep, kRoleThreads);                 // gates of chunk c written
            tc_wait(&mb[kMbGram], (unsigned)p, abort);
            tc_fence_after();
            {   // row `row` of [K;Q] K^T, columns 32 half .. +31 (blocks b = 2 half, 2 half + 1 of 16 tokens).
                // Decay e^{G_t - G_s}: direct inside t's block; across blocks e^{G_t - G_end(b)} e^{G_end(b) - G_s},
                // both <= 1. Shared-memory reads first, then the arithmetic, then the stores.
                const bool krow = row < kC;
                const int t = krow ? row : row - kC, bt = t >> 4;
                const int lim = krow ? t : t + 1;    // columns s < lim are kept
                const bool own = (bt >> 1) == half;  // t's own block is in this half (warp-uniform)
                const float Gt = sG[s][t], beta_t = sBeta[s][t];
                const float gend0 = sG[s][32 * half + 15], gend1 = sG[s][32 * half + 31];
                float gs[16], ge[32];  // G over t's own block; E over this half's two blocks
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 x = reinterpret_cast<const float4 *>(&sG[s][16 * bt])[q];
                    gs[4 * q] = x.x; gs[4 * q + 1] = x.y; gs[4 * q + 2] = x.z; gs[4 * q + 3] = x.w;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 x = reinterpret_cast<const float4 *>(&sE[s][32 * half])[q];
                    ge[4 * q] = x.x; ge[4 * q + 1] = x.y; ge[4 * q + 2] = x.z; ge[4 * q + 3] = x.w;
                }
                uint32_t gr[32];
                tmem_ld32u(tq + kColGr + 32 * half, gr);
                float dd[16];  // e^{G_t - G_s} for s in t's own block
#pragma unroll
                for (int e = 0; e < 16; ++e) dd[e] = own ? __expf(Gt - gs[e]) : 0.f;
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    const int b = 2 * half + bb;
                    const float fb = (b < bt) ? __expf(Gt - (bb ? gend1 : gend0)) : 0.f;
                    float w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float dcy = (b == bt) ? dd[e] : fb * ge[16 * bb + e];
                        w[e] = (16 * b + e < lim) ? dcy * __uint_as_float(gr[16 * bb + e]) : 0.f;
                    }
                    const uint4 lo4 = make_uint4(pack_h2(w[0], w[1]), pack_h2(w[2], w[3]), pack_h2(w[4], w[5]), pack_h2(w[6], w[7]));
                    const uint4 hi4 = make_uint4(pack_h2(w[8], w[9]), pack_h2(w[10], w[11]), pack_h2(w[12], w[13]),
                                                 pack_h2(w[14], w[15]));
                    if (krow) {
                        uint4 *dst = reinterpret_cast<uint4 *>(sAt + t * 72 + 16 * b);
                        dst[0] = lo4;
                        dst[1] = hi4;
                        if (b == bt) {  // diagonal block, fp32, float4 groups swizzled by row
                            const int rl = t & 15;
                            float4 *aj = reinterpret_cast<float4 *>(&sAjj[bt][rl][0]);
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4)
                                aj[q4 ^ ((rl >> 1) & 3)] = make_float4(beta_t * w[4 * q4], beta_t * w[4 * q4 + 1],
                                                                       beta_t * w[4 * q4 + 2], beta_t * w[4 * q4 + 3]);
                        }
                    } else {
                        uint4 *mq = reinterpret_cast<uint4 *>(smem + L::kMq + p * 8192);
                        mq[sw_chunk(t, 2 * b)] = lo4;
                        mq[sw_chunk(t, 2 * b + 1)] = hi4;
                    }
                }
            }
            fence_proxy_async();
            tc_fence_before();
            bar_sync(kBPrep, kRoleThreads);  // A, Ajj and Mq written; the grams read
            // Rows of the grams read. Warps 8-11 (one per scheduler) invert the diagonal blocks and solve
            // for T; warps 12-15 scale Q by gam, then warp 14 issues the next chunk's grams and warp 15
            // computes its gates.
            if (pw < 4) {
                // Inverses of the diagonal 16 x 16 blocks of L = I + A (unit lower triangular), one
                // thread per (block, column) of warps 8-9: right-looking forward substitution in fp32.
                if (pw < 2) {
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
                bar_sync(kBPrepK, kSolveThreads);
                {   // Block solve: warp 8 + w owns columns 16w .. 16w+15 of X = L^{-1}, as
                    // X^T (rows s, columns t): X^T_w = Linv_w^T, and for blocks j > w
                    //   X^T_j = -(sum_{i=w}^{j-1} X^T_i At_ji^T) diag(beta_j) Linv_j^T
                    // by warp-level MMAs. Then T = X diag(beta) -> fp16 operand tile [t][s].
                    if (c >= 1) bar_sync(kBTFree, kRoleThreads + kSolveThreads);  // the chain's T R of chunk c-1 is done
                    const int w = pw, fr = lane >> 2, fc = 2 * (lane & 3);
                    const float *bs = sBeta[s];
                    const float br0 = bs[16 * w + fr], br1 = bs[16 * w + fr + 8];
                    uint4 *tt = reinterpret_cast<uint4 *>(smem + L::kT);
                    const int m = lane >> 3;
                    unsigned xa[4][4];
                    float xc[2][4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int trow = 16 * j + 8 * (m >> 1) + (lane & 7);
                        if (j < w) {  // above the diagonal: zero tiles
                            stsm_x4_t(tt + sw_chunk(trow, 2 * w + (m & 1)), 0u, 0u, 0u, 0u);
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
                        stsm_x4_t(tt + sw_chunk(trow, 2 * w + (m & 1)), pack_h2(br0 * xc[0][0], br0 * xc[0][1]),
                                  pack_h2(br1 * xc[0][2], br1 * xc[0][3]), pack_h2(br0 * xc[1][0], br0 * xc[1][1]),
                                  pack_h2(br1 * xc[1][2], br1 * xc[1][3]));
                    }
                }
                fence_proxy_async();
                bar_arrive(kBFull + p, kTcThreads);  // T of chunk c ready for the chain
            } else {
                // q scaled by gam_t in place (fp16 products), for [K; gam Q] S0^T: one row of one dk box a thread
                const int r = pt & 63, bx = (pt >> 6) & 1;
                uint4 *rp = reinterpret_cast<uint4 *>(sK + bx * L::kKQBox + 8192 + r * 128);
                const __half2 g2 = __float2half2_rn(sGam[c % 4][r]);
                uint4 u[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) u[q] = rp[q ^ (r & 7)];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    __half2 *h2 = reinterpret_cast<__half2 *>(&u[q]);
#pragma unroll
                    for (int e = 0; e < 4; ++e) h2[e] = __hmul2(h2[e], g2);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) rp[q ^ (r & 7)] = u[q];
                fence_proxy_async();
                bar_arrive(kBFull + p, kTcThreads);  // gam Q of chunk c ready for the chain
                if (pw == 6 && c + 1 < nchunks) grams(c + 1);  // both halves of the grams are read
                if (pw == 7 && c + 1 < nchunks) {
                    gates(c + 1);
                    if (c + 2 < nchunks) fetch(c + 2);
                }
            }
        }
        if (pt == 6 * 32) {  // warp 14 issued the grams: they have completed before tensor memory is released
            umma_commit(&mb[kMbDrainPrep]);
            mbar_drain(&mb[kMbDrainPrep], 0u);
        }
    } else {
        // ================================ chain ================================
        // Token-major halves: warps on lane quarters 0-1 ("lo") hold the K rows (R, delta), warps on
        // quarters 2-3 the Q rows (output); token t = 32 (warp & 1) + lane, dv columns 64 half ..
        const bool lo = (warp & 3) < 2;
        const int t = 32 * (warp & 1) + lane;
        uint4 *rrow = reinterpret_cast<uint4 *>(smem + L::kR + half * 8192 + t * 128);
        int last_qk = -1, last_v = -1;  // the last chunks whose copies were issued (thread 64), in order
        auto load_qk = [&](int c) {  // k, q boxes of chunk c into stage c % 3
            const int s = c % 3;
            last_qk = c;
            unsigned char *st = smem + L::kKQ + s * L::kStage;
            mbar_arrive_expect_tx(&mb[kMbLoad + s], 4 * 8192);
            for (int x = 0; x < 2; ++x) {
                tma_load_4d(st + x * L::kKQBox, &maps.k, 64 * x, h, c * kC, n, &mb[kMbLoad + s]);
                tma_load_4d(st + x * L::kKQBox + 8192, &maps.q, 64 * x, h, c * kC, n, &mb[kMbLoad + s]);
            }
        };
        auto load_v = [&](int c) {  // v boxes of chunk c into buffer c & 1
            const int b = c & 1;
            last_v = c;
            mbar_arrive_expect_tx(&mb[kMbV + b], 2 * 8192);
            for (int x = 0; x < 2; ++x)
                tma_load_4d(smem + L::kV + b * L::kVBuf + x * 8192, &maps.v, 64 * x, h, c * kC, n, &mb[kMbV + b]);
        };
        // Thread 0 issues the MMAs; thread 64 (a Q-row warp) the TMA loads and stores and their waits.
        if (tid == 64) {
            for (int c = 0; c < 2 && c < nchunks; ++c) {
                load_qk(c);
                load_v(c);
            }
        }
        for (int c = 0; c < nchunks; ++c) {
            const int p0 = c * kC, nc = min(kC, P - p0), s = c % 3, p = c & 1;
            unsigned char *sK = smem + L::kKQ + s * L::kStage;
            unsigned char *vb = smem + L::kV + p * L::kVBuf;  // v, then dec_t delta_t, then the output rows of chunk c
            bar_sync(kBFull + p, kTcThreads);
            tc_fence_after();
            if (tid == 0) {  // [K; gam Q] S0^T -> D1[p]: K rows on lanes 0-63, Q rows on lanes 64-127
                const uint32_t id = umma_idesc(128, 128, 0, 0);
                for (int ks = 0; ks < 8; ++ks)
                    umma_f16(tmem + kColD1 + 128 * p, desc_kmajor(smem_addr(sK + (ks >> 2) * L::kKQBox) + (ks & 3) * 32),
                             desc_kmajor(smem_addr(smem + L::kCk + (ks >> 2) * 16384) + (ks & 3) * 32), id, ks > 0);
                umma_commit(&mb[kMbC1]);
            }
            if (tid == 64 && c + 2 < nchunks && !*abort) load_qk(c + 2);  // into the stage of chunk c-1, done with in both roles
            // Completion of this commit covers every earlier MMA too: delta of chunk c-1 has been read.
            tc_wait(&mb[kMbC1], (unsigned)p, abort);
            tc_fence_after();
            if (lo) {  // R = V - gam_t (K S0^T)_t -> fp16 operand tile [t][dv]
                const float gt = sGam[c % 4][t];
                tc_wait(&mb[kMbV + p], (unsigned)((c >> 1) & 1), abort);
                const uint4 *vrow = reinterpret_cast<const uint4 *>(vb + half * 8192 + t * 128);
                uint4 vv[8];  // this row's v, chunk j = dv 64 half + 8 j ..
#pragma unroll
                for (int j = 0; j < 8; ++j) vv[j] = vrow[j ^ (t & 7)];
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t d[32];
                    tmem_ld32u(tq + kColD1 + 128 * p + 64 * half + 32 * hq, d);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int ch = (4 * hq + q) ^ (t & 7);
                        const __half2 *v2 = reinterpret_cast<const __half2 *>(&vv[4 * hq + q]);
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(v2[e]);
                            w[e] = pack_h2(fmaf(-gt, __uint_as_float(d[8 * q + 2 * e]), f.x),
                                           fmaf(-gt, __uint_as_float(d[8 * q + 2 * e + 1]), f.y));
                        }
                        rrow[ch] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            fence_proxy_async();
            tc_fence_before();
            bar_sync(kBChain, kRoleThreads);
            tc_fence_after();
            if (tid == 0) {  // delta = T R -> D3 (lanes 0-63; the window's other half is unused)
                const uint32_t id = umma_idesc(128, 128, 0, 1);
                for (int ks = 0; ks < 4; ++ks)
                    umma_f16(tmem + kColD3, desc_kmajor(smem_addr(smem + L::kT) + ks * 32),
                             desc_mnmajor(smem_addr(smem + L::kR) + ks * 2048, 8192), id, ks > 0);
                umma_commit(&mb[kMbC2]);
            }
            if (tid == 64 && c >= 1) {
                bulk_wait_read();                      // the stores of chunk c-1 have read its output rows and the carry
                if (c + 1 < nchunks && !*abort) load_v(c + 1);  // into the buffer of chunk c-1
            }
            tc_wait(&mb[kMbC2], (unsigned)p, abort);
            tc_fence_after();
            if (c + 1 < nchunks) bar_arrive(kBTFree, kRoleThreads + kSolveThreads);  // T read
            if (lo) {  // delta rows -> fp16 operand tile (over R); dec_t delta_t -> the v buffer
                const float dt = sDec[c % 4][t];
                uint4 *drow = reinterpret_cast<uint4 *>(vb + half * 8192 + t * 128);
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t d[32];
                    tmem_ld32u(tq + kColD3 + 64 * half + 32 * hq, d);
                    put_row32(rrow, t, 4 * hq, d);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_h2(dt * __uint_as_float(d[8 * q + 2 * e]), dt * __uint_as_float(d[8 * q + 2 * e + 1]));
                        drow[(4 * hq + q) ^ (t & 7)] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            fence_proxy_async();
            tc_fence_before();
            bar_sync(kBChain, kRoleThreads);
            tc_fence_after();
            if (tid == 0) {
                const uint32_t ids = umma_idesc(128, 128, 1, 1), ido = umma_idesc(128, 128, 0, 1);
                for (int ks = 0; ks < 4; ++ks)  // (diag(dec) delta)^T K -> D3
                    umma_f16(tmem + kColD3, desc_mnmajor(smem_addr(vb) + ks * 2048, 8192),
                             desc_mnmajor(smem_addr(sK) + ks * 2048, L::kKQBox), ids, ks > 0);
                umma_commit(&mb[kMbC3]);
                for (int ks = 0; ks < 4; ++ks)  // + Mq delta onto the gam Q S0^T half of D1[p]
                    umma_f16(tmem + kColD1 + 128 * p, desc_kmajor(smem_addr(smem + L::kT + 8192 * p) + ks * 32),
                             desc_mnmajor(smem_addr(smem + L::kR) + ks * 2048, 8192), ido, true);
                umma_commit(&mb[kMbC4]);
            }
            tc_wait(&mb[kMbC3], (unsigned)p, abort);
            tc_fence_after();
            {   // S64 = gam_63 S0 + (dec delta)^T K, row dv = `row`, dk 64 half .. +63: new carry (fp16),
                // checkpoint, final state
                const float gl = sGam[c % 4][kC - 1];
                __half *so = (c + 1 == nchunks && !*abort) ? s_out + set_off + (size_t)row * 128 : nullptr;
                uint4 *crow = reinterpret_cast<uint4 *>(smem + L::kCk + half * 16384 + row * 128);
                uint4 cv[8];  // this row's carry, chunk lq = dk 64 half + 8 lq ..
#pragma unroll
                for (int lq = 0; lq < 8; ++lq) cv[lq] = crow[lq ^ (row & 7)];
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t ds[32];
                    tmem_ld32u(tq + kColD3 + 64 * half + 32 * hq, ds);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int lq = 4 * hq + q;
                        __half2 *h2 = reinterpret_cast<__half2 *>(&cv[lq]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(h2[e]);
                            h2[e] = __floats2half2_rn(fmaf(gl, f.x, __uint_as_float(ds[8 * q + 2 * e])),
                                                      fmaf(gl, f.y, __uint_as_float(ds[8 * q + 2 * e + 1])));
                        }
                    }
                }
#pragma unroll
                for (int lq = 0; lq < 8; ++lq) crow[lq ^ (row & 7)] = cv[lq];
                if (so)
#pragma unroll
                    for (int lq = 0; lq < 8; ++lq) *reinterpret_cast<uint4 *>(so + (8 * half + lq) * 8) = cv[lq];
            }
            fence_proxy_async();
            tc_fence_before();
            bar_sync(kBChain, kRoleThreads);
            if (!lo) {  // output rows O_t = (gam Q S0^T + Mq delta)_t -> v buffer [t][dv] -> TMA store
                tc_wait(&mb[kMbC4], (unsigned)p, abort);
                tc_fence_after();
                uint4 *orow = reinterpret_cast<uint4 *>(vb + half * 8192 + t * 128);
#pragma unroll
                for (int hq = 0; hq < 2; ++hq) {
                    uint32_t d[32];
                    tmem_ld32u(tq + kColD1 + 128 * p + 64 * half + 32 * hq, d);
                    put_row32(orow, t, 4 * hq, d);
                }
                fence_proxy_async();
                tc_fence_before();
                bar_sync(kBOut, kRoleThreads / 2);
                if (tid == 64 && !*abort) {  // at a full chunk the carry tile is the checkpoint
                    if (nc == kC)
                        for (int x = 0; x < 2; ++x)
                            tma_store_3d(&maps.ck, 64 * x, 0, (n * nfull + c) * H + h, smem + L::kCk + x * 16384);
                    for (int x = 0; x < 2; ++x) tma_store_4d(&maps.o, 64 * x, h, p0, n, vb + x * 8192);
                    bulk_commit();
                }
            }
            if (c + 2 < nchunks) bar_arrive(kBEmpty + p, kTcThreads);  // Mq and gates of chunk c consumed
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
        if (tid == 64) {
            bulk_wait();
            // every copy issued has landed before the CTA's shared memory is released (bounded)
            for (int b = 0; b < 3 && b <= last_qk; ++b)  // stage b took chunks b, b + 3, ...
                mbar_drain(&mb[kMbLoad + b], (unsigned)(((last_qk - b) / 3) & 1));
            for (int b = 0; b < 2 && b <= last_v; ++b)   // buffer b took chunks b, b + 2, ...
                mbar_drain(&mb[kMbV + b], (unsigned)(((last_v - b) / 2) & 1));
        }
        if (tid == 0) {  // every MMA this thread issued has completed before tensor memory is released
            umma_commit(&mb[kMbDrainChain]);
            mbar_drain(&mb[kMbDrainChain], 0u);
        }
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
        H, P, maps, beta, g, static_cast<const __half *>(s_in), static_cast<__half *>(s_out));
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
