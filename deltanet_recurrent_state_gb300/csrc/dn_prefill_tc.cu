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
//  * prep (4 warps), a chunk ahead: q/k/v by tensor-map (TMA) loads; the grams [K;Q] K^T
//    by one MMA into tensor memory; A and Mq with their decays; the 64 x 64 inverse T in
//    fp32 (16 x 16 diagonal blocks by forward substitution, then the off-diagonal blocks
//    level by level); U^T = V^T T^T (left in tensor memory) and W^T = K^T (T diag gam)^T
//    by MMA; W and K scaled by dec written back to shared memory as MMA operands.
//  * chain (4 warps, thread i = state row i = tensor-memory lane i): one MMA for S0 [W;Q]^T,
//    delta in registers, one MMA pair for delta Mq^T and delta^T (dec K), then the output
//    tile (TMA store) and the new carry (shared memory for the next chunk's MMA, global
//    memory as the checkpoint).
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
constexpr int kTcThreads = 256;   // 4 chain warps, then 4 prep warps
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
    static constexpr uint32_t kA = 147456;      // fp32 [64][64] (swizzled); then T at +0, T diag(gam) at +8192
    static constexpr uint32_t kX = 163840;      // fp32 [64][64] (swizzled): (I + A)^{-1}
    static constexpr uint32_t kCk = 180224;     // carry: [2 dk boxes][128 dv rows][128 B]
    static constexpr uint32_t kD = 212992;      // delta [128 dv rows][128 B (64 t)]; output boxes [2][64 t][128 B] alias it
    static constexpr uint32_t kGates = 229376;  // fp32 [3 stages][beta | g][64]
    static constexpr uint32_t kGam = kGates + 3 * 2 * kC * 4;  // fp32 [2 parities][64]
    static constexpr uint32_t kG = kGam + 2 * kC * 4;          // fp32 [64]
    static constexpr uint32_t kDec = kG + kC * 4;              // fp32 [64]
    static constexpr uint32_t kMbar = kDec + kC * 4;           // q/k stages x3, v, prep MMA, chain MMA
    static constexpr uint32_t kTslot = kMbar + 6 * 8;
    static constexpr uint32_t kBytes = kTslot + 16;
};
static_assert(TcSmem::kBytes <= 232448, "shared memory above the per-block limit");

// fp32 64 x 64 tile, float4 groups XOR-swizzled by row so that row-wise float4 and
// column-wise scalar accesses of a warp spread over the banks.
__device__ __forceinline__ int fidx(int r, int c) { return r * 64 + (c ^ ((r & 7) << 2)); }

// Count of waits that ran out (read by dn_prefill_wait_timeouts).
__device__ unsigned int g_prefill_tc_timeouts;

struct TcMaps {
    CUtensorMap q, k, v, o;
};

__device__ __forceinline__ void tc_wait(unsigned long long *mb, unsigned parity, int lane) {
    if (!mbar_wait(mb, parity, kTcTries) && lane == 0) atomicAdd(&g_prefill_tc_timeouts, 1u);
}

// Off-diagonal blocks (i, j), i - j = LEV, of X = (I + A)^{-1} given the diagonal blocks and
// all blocks of lower levels: X_ij = -X_ii sum_{k=j}^{i-1} A_ik X_kj. A task is one column
// c of one block and R of its 16 rows; Y = sum_k A_ik X_kj goes through the X_ij slot.
template <int LEV, int R>
__device__ __forceinline__ void inverse_level(const float *sA, float *sX, int pt) {
    constexpr int PER = 16 / R, NB = 4 - LEV, TASKS = NB * 16 * PER;
    const bool act = pt < TASKS;
    const int blk = pt / (16 * PER), rem = pt % (16 * PER), c = rem / PER, r0 = (rem % PER) * R;
    const int j = blk, i = blk + LEV;
    if (act) {
        float y[R];
#pragma unroll
        for (int r = 0; r < R; ++r) y[r] = 0.f;
#pragma unroll
        for (int k = 0; k < LEV; ++k) {
            const int kb = j + k;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float xv = sX[fidx(16 * kb + m, 16 * j + c)];
#pragma unroll
                for (int r = 0; r < R; ++r) y[r] = fmaf(sA[fidx(16 * i + r0 + r, 16 * kb + m)], xv, y[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) sX[fidx(16 * i + r0 + r, 16 * j + c)] = y[r];
    }
    bar_sync(kBPrep, 128);
    float ycol[16];
    if (act) {
#pragma unroll
        for (int m = 0; m < 16; ++m) ycol[m] = sX[fidx(16 * i + m, 16 * j + c)];
    }
    bar_sync(kBPrep, 128);
    if (act) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) acc = fmaf(sX[fidx(16 * i + r0 + r, 16 * i + m)], ycol[m], acc);
            sX[fidx(16 * i + r0 + r, 16 * j + c)] = -acc;
        }
    }
    bar_sync(kBPrep, 128);
}

__global__ void __launch_bounds__(kTcThreads, 1)
prefill_tc_kernel(int H, int P, const __grid_constant__ TcMaps maps, const float *__restrict__ beta,
                  const float *__restrict__ g, const __half *s_in, __half *s_out, __half *ckpt) {
    using L = TcSmem;
    extern __shared__ __align__(1024) unsigned char smem[];
    float(*sGates)[2][kC] = reinterpret_cast<float(*)[2][kC]>(smem + L::kGates);
    float(*sGam)[kC] = reinterpret_cast<float(*)[kC]>(smem + L::kGam);
    float *sG = reinterpret_cast<float *>(smem + L::kG);
    float *sDec = reinterpret_cast<float *>(smem + L::kDec);
    float *sA = reinterpret_cast<float *>(smem + L::kA);
    float *sX = reinterpret_cast<float *>(smem + L::kX);
    unsigned long long *mb = reinterpret_cast<unsigned long long *>(smem + L::kMbar);  // 0-2 qk, 3 v, 4 prep, 5 chain
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + L::kTslot);

    const int h = blockIdx.x % H, n = blockIdx.x / H;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int nchunks = (P + kC - 1) / kC, nfull = P / kC;
    const size_t set_off = ((size_t)n * H + h) * 128 * 128;

    if (tid == 0) {
        for (int i = 0; i < 6; ++i) mbar_init(&mb[i], 1);
        fence_proxy_async();
    }
    if (warp == 0) tmem_alloc<kTmemCols>(tslot);
    if (tid < 128) {  // chain: the initial state becomes the carry tile
        for (int ch = 0; ch < 16; ++ch) {
            uint4 u = make_uint4(0u, 0u, 0u, 0u);
            if (s_in) u = *reinterpret_cast<const uint4 *>(s_in + set_off + (size_t)tid * 128 + ch * 8);
            *reinterpret_cast<uint4 *>(smem + L::kCk + (ch >> 3) * 16384 + tid * 128 + (((ch & 7) ^ (tid & 7)) * 16)) = u;
        }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's lane quarter

    if (warp >= 4) {
        // ================================ prep ================================
        const int pt = tid - 128;
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
            const size_t row0 = ((size_t)n * P + p0) * H + h;
            for (int i = pt; i < 2 * kC; i += 128) {
                const int which = i / kC, t = i % kC;
                const bool ok = p0 + t < P;
                const float *src = which ? g : beta;
                cp_async4(&sGates[s][which][t], ok ? (const void *)(src + row0 + (size_t)t * H) : (const void *)src,
                          ok ? 4 : 0);
            }
        };
        auto issue_v = [&](int c) {
            if (pt == 0) {
                mbar_arrive_expect_tx(&mb[3], 2 * 8192);
                for (int x = 0; x < 2; ++x) tma_load_4d(smem + L::kV + x * 8192, &maps.v, 64 * x, h, c * kC, n, &mb[3]);
            }
        };
        if (nchunks > 0) {
            issue_qk(0);
            issue_v(0);
        }
        cp_async_commit();
        for (int c = 0; c < nchunks; ++c) {
            const int p0 = c * kC, nc = min(kC, P - p0), s = c % 3, pb = c & 1;
            unsigned char *sK = smem + L::kKQ + s * L::kStage;
            if (c >= 2) bar_sync(kBEmpty + pb, kTcThreads);  // chain done with chunk c-2
            if (c + 1 < nchunks) issue_qk(c + 1);
            cp_async_commit();
            cp_async_wait<1>();
            tc_wait(&mb[s], (unsigned)((c / 3) & 1), lane);
            tc_fence_before();
            bar_sync(kBPrep, 128);  // gates landed for every prep thread; last chunk's scratch reads done
            tc_fence_after();
            if (pt == 0) {  // grams: [K;Q] (128 rows) x K^T -> scratch columns
                const uint32_t id = umma_idesc(128, 64, 0, 0);
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t a = smem_addr(sK + (ks >> 2) * L::kKQBox) + (ks & 3) * 32;
                    umma_f16(tmem + kColScr, desc_kmajor(a), desc_kmajor(a), id, ks > 0);
                }
                umma_commit(&mb[4]);
            }
            // gates: G_t = sum_{r<=t} log g_r (0 past the prompt), gam, dec
            if (pt < kC) {
                float G = (pt < nc) ? __logf(fmaxf(sGates[s][1][pt], 1e-30f)) : 0.f;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, G, off);
                    if (lane >= off) G += o;
                }
                sG[pt] = G;
            }
            bar_sync(kBPrep, 128);
            if (pt >= 32 && pt < kC) sG[pt] += sG[31];
            bar_sync(kBPrep, 128);
            if (pt < kC) {
                const float G = sG[pt];
                sGam[pb][pt] = __expf(G);
                sDec[pt] = __expf(sG[kC - 1] - G);
            }
            tc_wait(&mb[4], 0u, lane);
            tc_fence_after();
            {   // row pt of [K;Q] K^T: A (k rows, fp32) or Mq (q rows, fp16 operand tile)
                float d[64];
                tmem_ld32(tq + kColScr, *reinterpret_cast<float(*)[32]>(d));
                tmem_ld32(tq + kColScr + 32, *reinterpret_cast<float(*)[32]>(d + 32));
                if (pt < kC) {
                    const int t = pt;
                    const float Gt = sG[t], bt = sGates[s][0][t];
#pragma unroll
                    for (int q4 = 0; q4 < 16; ++q4) {
                        float4 v;
                        float *vv = reinterpret_cast<float *>(&v);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int sc = 4 * q4 + e;
                            vv[e] = (sc < t) ? bt * __expf(Gt - sG[sc]) * d[sc] : 0.f;
                        }
                        *reinterpret_cast<float4 *>(&sA[fidx(t, 4 * q4)]) = v;
                    }
                } else {
                    const int t = pt - kC;
                    const float Gt = sG[t];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        unsigned w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int s0 = 8 * ch + 2 * e;
                            const float a0 = (s0 <= t) ? __expf(Gt - sG[s0]) * d[s0] : 0.f;
                            const float a1 = (s0 + 1 <= t) ? __expf(Gt - sG[s0 + 1]) * d[s0 + 1] : 0.f;
                            w[e] = pack_h2(a0, a1);
                        }
                        *reinterpret_cast<uint4 *>(smem + L::kMq + pb * 8192 + t * 128 + ((ch ^ (t & 7)) * 16)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            fence_proxy_async();
            tc_fence_before();
            bar_sync(kBPrep, 128);
            // diagonal 16 x 16 blocks of (I + A)^{-1}: one thread per (block, column)
            if (pt < kC) {
                const int b0 = 16 * (pt >> 4), col = pt & 15;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int k = 0; k < i; ++k) acc[k & 3] = fmaf(sA[fidx(b0 + i, b0 + k)], x[k], acc[k & 3]);
                    x[i] = (i < col) ? 0.f : (i == col ? 1.f : -((acc[0] + acc[1]) + (acc[2] + acc[3])));
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) sX[fidx(b0 + i, b0 + col)] = x[i];
            }
            bar_sync(kBPrep, 128);
            inverse_level<1, 8>(sA, sX, pt);
            inverse_level<2, 4>(sA, sX, pt);
            inverse_level<3, 2>(sA, sX, pt);
            {   // T = X diag(beta) and T diag(gam) as fp16 operand tiles [t][s] (over A's space)
                const int t = pt >> 1, hh = pt & 1;
                const float *bs = sGates[s][0];
                const float *gs = sGam[pb];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int c0 = 32 * hh + 8 * u;
                    const float4 x0 = *reinterpret_cast<const float4 *>(&sX[fidx(t, c0)]);
                    const float4 x1 = *reinterpret_cast<const float4 *>(&sX[fidx(t, c0 + 4)]);
                    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    unsigned wt[4], wg[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {  // X is lower triangular; its upper blocks are never written
                        const int sa = c0 + 2 * e;
                        const float t0 = (sa <= t) ? xv[2 * e] * bs[sa] : 0.f;
                        const float t1 = (sa + 1 <= t) ? xv[2 * e + 1] * bs[sa + 1] : 0.f;
                        wt[e] = pack_h2(t0, t1);
                        wg[e] = pack_h2(t0 * gs[c0 + 2 * e], t1 * gs[c0 + 2 * e + 1]);
                    }
                    const int off = t * 128 + (((4 * hh + u) ^ (t & 7)) * 16);
                    *reinterpret_cast<uint4 *>(smem + L::kA + off) = make_uint4(wt[0], wt[1], wt[2], wt[3]);
                    *reinterpret_cast<uint4 *>(smem + L::kA + 8192 + off) = make_uint4(wg[0], wg[1], wg[2], wg[3]);
                }
            }
            fence_proxy_async();
            tc_fence_before();
            bar_sync(kBPrep, 128);
            tc_fence_after();
            if (pt == 0) {  // U^T = V^T T^T (kept for the chain), W^T = K^T (T diag gam)^T (scratch)
                tc_wait(&mb[3], (unsigned)(c & 1), 0);
                tc_fence_after();
                const uint32_t id = umma_idesc(128, 64, 1, 0);
                for (int ks = 0; ks < 4; ++ks) {
                    umma_f16(tmem + kColU + 64 * pb, desc_mnmajor(smem_addr(smem + L::kV) + ks * 2048, 8192),
                             desc_kmajor(smem_addr(smem + L::kA) + ks * 32), id, ks > 0);
                    umma_f16(tmem + kColScr, desc_mnmajor(smem_addr(sK) + ks * 2048, L::kKQBox),
                             desc_kmajor(smem_addr(smem + L::kA + 8192) + ks * 32), id, ks > 0);
                }
                umma_commit(&mb[4]);
            }
            tc_wait(&mb[4], 1u, lane);
            tc_fence_after();
            if (c + 1 < nchunks) issue_v(c + 1);  // v of this chunk consumed
            if (c >= 1) bar_sync(kBWFree, kTcThreads);  // the chain's first MMA of chunk c-1 read W
            {   // W^T row pt (dk index) -> W tile [t][dk]
                float w[64];
                tmem_ld32(tq + kColScr, *reinterpret_cast<float(*)[32]>(w));
                tmem_ld32(tq + kColScr + 32, *reinterpret_cast<float(*)[32]>(w + 32));
                unsigned char *wb = smem + L::kW + (pt >> 6) * 8192 + (pt & 7) * 2;
                const int dch = (pt & 63) >> 3;
#pragma unroll
                for (int t = 0; t < kC; ++t)
                    *reinterpret_cast<__half *>(wb + t * 128 + ((dch ^ (t & 7)) * 16)) = __float2half_rn(w[t]);
            }
            {   // K rows scaled by dec (in place: the chain's state update reads dec K)
                const int bx = pt >> 6, sr = pt & 63;
                const float2 f2 = make_float2(sDec[sr], sDec[sr]);
                unsigned char *rp = sK + bx * L::kKQBox + sr * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
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
        cp_async_wait<0>();
    } else {
        // ================================ chain ================================
        const int row = tid;  // state row = tensor-memory lane
        for (int c = 0; c < nchunks; ++c) {
            const int p0 = c * kC, nc = min(kC, P - p0), s = c % 3, pb = c & 1;
            unsigned char *sK = smem + L::kKQ + s * L::kStage;
            bar_sync(kBFull + pb, kTcThreads);
            tc_fence_after();
            if (tid == 0) {
                bulk_wait_read();  // the previous output store has read the delta / output tile
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
            {   // delta = U - S0 W^T, row `row`, 64 tokens -> fp16 operand tile
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float a[32], u[32];
                    tmem_ld32(tq + kColDW + 32 * hf, a);
                    tmem_ld32(tq + kColU + 64 * pb + 32 * hf, u);
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        unsigned w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_h2(u[8 * ch + 2 * e] - a[8 * ch + 2 * e], u[8 * ch + 2 * e + 1] - a[8 * ch + 2 * e + 1]);
                        const int lch = 4 * hf + ch;
                        *reinterpret_cast<uint4 *>(smem + L::kD + row * 128 + ((lch ^ (row & 7)) * 16)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            fence_proxy_async();
            tc_fence_before();
            bar_sync(kBChain, 128);
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
            {   // o_t = gam_t (S0 q_t) + (delta Mq^T)_t -> output boxes [t][dv] (over the delta tile)
                const float *gam = sGam[pb];
                unsigned char *ob = smem + L::kD + (row >> 6) * 8192 + (row & 7) * 2;
                const int rch = (row & 63) >> 3;
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float a[32], b[32];
                    tmem_ld32(tq + kColDQ + 32 * hf, a);
                    tmem_ld32(tq + kColDW + 32 * hf, b);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int t = 32 * hf + j;
                        *reinterpret_cast<__half *>(ob + t * 128 + ((rch ^ (t & 7)) * 16)) =
                            __float2half_rn(fmaf(gam[t], a[j], b[j]));
                    }
                }
            }
            {   // S64 = gam_63 S0 + delta^T (dec K): new carry (fp16), checkpoint, final state
                const float gl = sGam[pb][kC - 1];
                __half *ck = (nc == kC) ? ckpt + ((size_t)(n * nfull + c) * H + h) * 16384 + (size_t)row * 128 : nullptr;
                __half *so = (c + 1 == nchunks) ? s_out + set_off + (size_t)row * 128 : nullptr;
#pragma unroll
                for (int piece = 0; piece < 4; ++piece) {
                    float ds[32];
                    tmem_ld32(tq + kColDS + 32 * piece, ds);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int ch = 4 * piece + q;
                        unsigned char *cp = smem + L::kCk + (ch >> 3) * 16384 + row * 128 + (((ch & 7) ^ (row & 7)) * 16);
                        uint4 u = *reinterpret_cast<uint4 *>(cp);
                        __half2 *h2 = reinterpret_cast<__half2 *>(&u);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(h2[e]);
                            h2[e] = __floats2half2_rn(fmaf(gl, f.x, ds[8 * q + 2 * e]), fmaf(gl, f.y, ds[8 * q + 2 * e + 1]));
                        }
                        *reinterpret_cast<uint4 *>(cp) = u;
                        if (ck) *reinterpret_cast<uint4 *>(ck + ch * 8) = u;
                        if (so) *reinterpret_cast<uint4 *>(so + ch * 8) = u;
                    }
                }
            }
            fence_proxy_async();
            tc_fence_before();
            if (c + 2 < nchunks) bar_arrive(kBEmpty + pb, kTcThreads);  // q/k stage, Mq, U, gam of chunk c consumed
            bar_sync(kBChain, 128);
            if (tid == 0) {
                for (int x = 0; x < 2; ++x) tma_store_4d(&maps.o, 64 * x, h, p0, n, smem + L::kD + x * 8192);
                bulk_commit();
            }
        }
        if (nchunks == 0) {  // empty prompt: the state passes through
            for (int ch = 0; ch < 16; ++ch) {
                uint4 u = make_uint4(0u, 0u, 0u, 0u);
                if (s_in) u = *reinterpret_cast<const uint4 *>(s_in + set_off + (size_t)tid * 128 + ch * 8);
                *reinterpret_cast<uint4 *>(s_out + set_off + (size_t)tid * 128 + ch * 8) = u;
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
