// dn_prefill_checkpoint: a prompt through the gated delta rule with a state
// checkpoint every 64 tokens, for prefix caching of the DeltaNet state
// ("HyperQwen: 1,000 tok/s on a Single RTX 3090 ...", Technical Insight: the
// recurrent state is checkpointed next to the attention context so that a later
// turn restores it instead of recomputing the prompt).
//
// Two kernels:
//  * prefill_wy_kernel (fp16 state and io): the chunkwise (WY) form on tensor
//    cores. A CTA owns one (sequence, head); each warp owns 16 dv-rows of the
//    state, kept in fp32 MMA accumulator fragments for the whole prompt. Every
//    16-token sub-chunk costs a handful of m16n8k16 MMAs per warp (derivation at
//    the kernel); the next 64-token chunk of q/k/v streams in with cp.async while
//    the current one is processed.
//  * prefill_seq_kernel (fp32 path): the token-by-token form. A CTA owns ROWS rows
//    of one (sequence, head) state in registers and walks the prompt, staging 16
//    tokens of q/k/v/beta/g at a time in shared memory.
// In both, at every chunk end the carry is rounded to the state dtype and stored,
// so the carry equals the checkpoint and a restored run continues bit-identically.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "dn.h"
#include "dn_device.cuh"
#include "dn_internal.h"
#include "dn_mma.cuh"
#include "dn_recurrence.cuh"
#include "dn_tmap.h"

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


// ---------------------------------------------------------------------------------------
// Chunkwise (WY) prefill, fp16 state and io.
//
// Inside a sub-chunk of 16 tokens starting from state S (dv x dk), with gates
// accumulated from the sub-chunk start, G_t = sum_{r<=t} log g_r, gam_t = e^{G_t}:
//   A[t][s]  = beta_t e^{G_t - G_s} (k_t . k_s)          (s < t, else 0)
//   Tb       = (I + A)^{-1} diag(beta)                    (16 x 16, per head)
//   Delta    = Tb (V - diag(gam) K S^T)                   (16 x dv)
//   O        = diag(gam) Q S^T + Mq Delta,  Mq[t][s] = e^{G_t - G_s} (q_t . k_s) (s <= t)
//   S_next   = gam_15 S + Delta^T diag(e^{G_15 - G}) K
// which is the token-by-token rule summed over the sub-chunk (the same algebra as
// the verify block). Four sub-chunks make a 64-token checkpoint chunk.
//
// Per chunk (one CTA = one (sequence, head), DV/16 warps):
//   prep (state independent, all warps): grams K_j K_j^T and Q_j K_j^T by MMA, the
//     gate scans, A and Mq, and the four 16 x 16 inverses (one thread per column,
//     forward substitution in fp32);
//   chain (each warp on its 16 dv-rows, no block barrier inside): per sub-chunk
//     X = S [K_j;Q_j]^T (MMA, S packed to fp16 from the accumulators), R = V^T -
//     gam X_K, Delta^T = R Tb^T, O^T = gam X_Q + Delta^T Mq^T, and S += (scaled
//     Delta)^T K_j on the accumulators;
//   chunk end: S rounded to fp16 (the carry) and stored as the checkpoint; the O tile
//     goes out with 16-byte stores.
// Operands are fp16 with fp32 accumulation; the carry is fp32 inside a chunk.

// Shared-memory tiles. q/k/v, O and the checkpoint move with the tensor-map (TMA) engine
// in 64-column boxes of 128-byte rows, swizzled by the engine: 16-byte chunk c of row r
// of a box sits at chunk c ^ (r & 7). Every box starts on a 1024-byte boundary.
// A = beta_t e^{G_t - G_s} k_t.k_s of sub-chunk j, 16 x 16 fp32: element (i, s) at
// j kAStride + 16 i + 4 ((s >> 2) ^ ((i >> 1) & 3)) + (s & 3). Each row is four 16-byte groups,
// so the inverse reads a row four elements at a time; the groups are swizzled by row so that
// the grams' pair stores spread over the banks, and sub-chunks sit 260 floats apart so that
// one warp's reads of two sub-chunks hit different banks.
constexpr int kAStride = 260;
__device__ __forceinline__ int a_index(int j, int i, int s) {
    return j * kAStride + 16 * i + 4 * ((s >> 2) ^ ((i >> 1) & 3)) + (s & 3);
}

template <int DK, int DVC>
struct PrefillSmem {
    static constexpr int C = 64, NSUB = 4, NKQV = 3, NPREP = 2;
    static constexpr int KH = DK / 64, VH = DVC / 64;   // 64-column boxes per row
    static constexpr size_t kBox = (size_t)C * 128;      // one 64 x 64 fp16 box
    // byte offsets
    static constexpr size_t kK = 0;                                       // [3][KH] boxes
    static constexpr size_t kQ = kK + (size_t)NKQV * KH * kBox;
    static constexpr size_t kV = kQ + (size_t)NKQV * KH * kBox;          // [3][VH] boxes
    static constexpr size_t kO = kV + (size_t)NKQV * VH * kBox;          // [2][VH] boxes
    static constexpr size_t kCk = kO + (size_t)2 * VH * kBox;            // [KH] boxes of DVC rows
    static constexpr size_t kTb = kCk + (size_t)KH * DVC * 128;          // [2][NSUB][16][24] half
    static constexpr size_t kMq = kTb + NPREP * NSUB * 16 * 24 * 2;      // [2][NSUB][16][24] half
    static constexpr size_t kGam = kMq + NPREP * NSUB * 16 * 24 * 2;     // [2][C] float
    static constexpr size_t kDec = kGam + NPREP * C * 4;                 // [2][C] float
    static constexpr size_t kA = kDec + NPREP * C * 4;                   // [NSUB][kAStride] float
    static constexpr size_t kGates = kA + NSUB * kAStride * 4;           // [3][2][C] float: beta, g
    static constexpr size_t kMbar = kGates + (size_t)NKQV * 2 * C * 4;   // [3] mbarrier
    static constexpr size_t kAbort = kMbar + NKQV * 8;                   // int: a wait ran out
    static constexpr size_t kBytes = kAbort + 8;
};

// 16-byte chunk `ch` (of D/8) of row `r` in a run of 64-column swizzled boxes with
// `rows` rows each.
__device__ __forceinline__ int box_chunk(int rows, int r, int ch) {
    return (ch >> 3) * rows * 8 + r * 8 + ((ch & 7) ^ (r & 7));
}

// A CTA owns DVC of the DV rows of one (sequence, head) state: all of them, or half when
// there are fewer (sequence, head) pairs than SMs (each half then repeats the
// state-independent work, which idle SMs absorb).
// Warp roles. Chain warps (DVC/16 of them, 16 dv-rows each) hold the state and run
// the state-dependent steps of chunk c; four prep warps meanwhile fetch chunk c+1's gates
// and compute its state-independent products. Hand-off per chunk parity p with named
// barriers over all threads: FULL[p] (prep arrives, chain waits) when chunk c's
// inputs and products are ready, EMPTY[p] (chain arrives, prep waits) when the
// chain is done with them. Inputs are triple buffered (chunk c, chunk c+1 and the
// load of the next one), the prep products double buffered.
// Issuing a TMA copy holds its thread for a hundred or more cycles (a chunk's six input
// boxes about 1,300 cycles, its four output and checkpoint boxes about 450), and issuing
// them from several warps at once is no faster. A producer warp issues every copy, off
// both roles' critical paths: it loads chunk c+3 once the chain is done with chunk c
// (EMPTY), stores chunk c's output and checkpoint boxes once the chain has staged them
// (STORE), and when those stores have read shared memory tells the chain (STORE_FREE),
// which waits for that before staging the next checkpoint.
constexpr int kBarFull = 1, kBarEmpty = 3, kBarPrep = 5, kBarStore = 6, kBarStoreFree = 7;
constexpr int kPrepThreads = 128, kProducerThreads = 32;

// A thirteenth warp caps every thread of the CTA at 128 registers: the register file is
// split between the SM's four schedulers, and one of them then holds four warps. The chain
// warps of a dk = 128 state want about 157 and measure slower squeezed, so those CTAs are
// launched as four whole warpgroups (512 threads at 128 registers each) and the registers
// are redistributed by warpgroup: the producer's warpgroup drops to kProducerRegs and three
// of its warps leave, the chain warpgroups rise to kChainRegs, the prep warpgroups keep 128.
// Over 128 rows that is two chain warpgroups and one prep warpgroup (2 x 168 + 128 + 24 =
// 488 of a scheduler's 512 registers per thread slot); over 64 rows, one chain warpgroup
// and two prep warpgroups, a gram tile per prep warp (168 + 2 x 128 + 24 = 448). Either way
// the rise never waits on registers that are not there.
constexpr int kChainRegs = 168, kProducerRegs = 24;
template <int DK, int DVC>
constexpr bool prefill_regsplit() { return DK == 128; }
// prep threads: two warpgroups for 64-row CTAs (one gram tile per warp), one for 128 rows
template <int DK, int DVC>
constexpr int prefill_prep_threads() { return DVC == 64 ? 2 * kPrepThreads : kPrepThreads; }
template <int DK, int DVC, int RT>
constexpr int prefill_threads() {
    return DVC * 2 / RT + prefill_prep_threads<DK, DVC>() +
           (prefill_regsplit<DK, DVC>() ? 4 * kProducerThreads : kProducerThreads);
}
static_assert(2 * kChainRegs + 65536 / 512 + kProducerRegs <= 512, "register split exceeds a scheduler's file");
static_assert(kChainRegs + 2 * (65536 / 512) + kProducerRegs <= 512, "register split exceeds a scheduler's file");

template <int N>
__device__ __forceinline__ void regs_raise() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_lower() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
// 16-row state tiles per chain warp. Two tiles per warp halve the operand fragments each
// warp loads from shared memory (which runs at about 80 % of its throughput here), but they
// leave one chain warp per scheduler instead of two and need 128 fp32 state registers a
// thread; even with the chain warpgroup raised to 232 registers they measure slower, so one
// it is.
constexpr int kRowTiles = 1;

// Count of prefill input waits that ran out (read by dn_prefill_wait_timeouts).
__device__ unsigned int g_prefill_wait_timeouts;

struct PrefillMaps {
    CUtensorMap q, k, v, o, ck;
};

template <int DK, int DV, int DVC, int RT>
__global__ void __launch_bounds__(prefill_threads<DK, DVC, RT>(), 1)
prefill_wy_kernel(int H, int P, const __grid_constant__ PrefillMaps maps,
                  const float *__restrict__ beta, const float *__restrict__ g,
                  const __half *s_in, __half *s_out) {
    using L = PrefillSmem<DK, DVC>;
    constexpr int C = L::C, NSUB = L::NSUB, KH = L::KH, VH = L::VH;
    constexpr int NW = DVC / (16 * RT), NTC = NW * 32, NTP = prefill_prep_threads<DK, DVC>(), NTALL = NTC + NTP;
    constexpr bool SPLIT = prefill_regsplit<DK, DVC>();
    static_assert(!SPLIT || ((NW == 8 && NTP == 128) || (NW == 4 && NTP == 256)),
                  "the register split assumes 4 whole warpgroups of 128 registers");
    constexpr int NTX = kProducerThreads;  // the producer warp follows the prep warps
    constexpr int NTK = DK / 8;   // accumulator tiles of the state over dk
    constexpr int KS = DK / 16;   // k-steps of the projection
    constexpr int BOXU = C * 8;   // uint4 per 64 x 64 box
    extern __shared__ __align__(1024) unsigned char smem[];
    uint4 *sK = reinterpret_cast<uint4 *>(smem + L::kK);
    uint4 *sQ = reinterpret_cast<uint4 *>(smem + L::kQ);
    uint4 *sV = reinterpret_cast<uint4 *>(smem + L::kV);
    uint4 *sO = reinterpret_cast<uint4 *>(smem + L::kO);
    uint4 *sCk = reinterpret_cast<uint4 *>(smem + L::kCk);
    __half(*sTb)[NSUB][16][24] = reinterpret_cast<__half(*)[NSUB][16][24]>(smem + L::kTb);
    __half(*sMq)[NSUB][16][24] = reinterpret_cast<__half(*)[NSUB][16][24]>(smem + L::kMq);
    float(*sgam)[C] = reinterpret_cast<float(*)[C]>(smem + L::kGam);
    float(*sdec)[C] = reinterpret_cast<float(*)[C]>(smem + L::kDec);
    float *sA = reinterpret_cast<float *>(smem + L::kA);
    float(*sGates)[2][C] = reinterpret_cast<float(*)[2][C]>(smem + L::kGates);  // [buf][beta|g][t]
    unsigned long long *mbar = reinterpret_cast<unsigned long long *>(smem + L::kMbar);
    // Raised when a wait runs out (kWaitBudgetNs): from then on no role issues copies or global
    // stores, every role still passes its named barriers to the end of the loop, and the
    // producer waits (bounded) for the copies it issued before the CTA exits.
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L::kAbort);

    constexpr int RB = DV / DVC;  // CTAs per (sequence, head)
    const int rb = blockIdx.x % RB;
    const int h = (blockIdx.x / RB) % H;
    const int n = blockIdx.x / (RB * H);
    const int r0 = rb * DVC;      // first state row of this CTA
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int fr = lane >> 2, fc = 2 * (lane & 3);  // fragment row / column pair
    const size_t set_elems = (size_t)DV * DK;
    const size_t state_off = ((size_t)n * H + h) * set_elems;
    const int nchunks = (P + C - 1) / C;
    const int nfull = P / C;

    if (tid == NTC) {
        for (int b = 0; b < 3; ++b) mbar_init(&mbar[b], 1);
        *abort = 0;
        fence_proxy_async();
    }
    __syncthreads();

    // chunk c's q/k/v boxes on mbar[c % 3] (rows past the prompt arrive as zeros)
    auto load_chunk = [&](int c) {
        const int p0 = c * C, kb = c % 3;
        mbar_arrive_expect_tx(&mbar[kb], (unsigned)((2 * KH + VH) * L::kBox));
        for (int x = 0; x < KH; ++x) {
            tma_load_4d(sK + (kb * KH + x) * BOXU, &maps.k, 64 * x, h, p0, n, &mbar[kb]);
            tma_load_4d(sQ + (kb * KH + x) * BOXU, &maps.q, 64 * x, h, p0, n, &mbar[kb]);
        }
        for (int x = 0; x < VH; ++x)
            tma_load_4d(sV + (kb * VH + x) * BOXU, &maps.v, r0 + 64 * x, h, p0, n, &mbar[kb]);
    };
    // chunk c's output boxes O[c & 1], and its checkpoint box when the chunk is full
    auto store_chunk = [&](int c) {
        const int p0 = c * C;
        const uint4 *cO = sO + (c & 1) * VH * BOXU;
        for (int x = 0; x < VH; ++x) tma_store_4d(&maps.o, r0 + 64 * x, h, p0, n, cO + x * BOXU);
        if (P - p0 >= C)
            for (int x = 0; x < KH; ++x)
                tma_store_3d(&maps.ck, 64 * x, r0, (n * nfull + c) * H + h, sCk + x * DVC * 8);
        bulk_commit();
    };

    if (warp >= NW + NTP / 32) {
        // ============================= producer warp =============================
        if constexpr (SPLIT) {
            regs_lower<kProducerRegs>();  // the whole warpgroup, then its spare warps leave
            if (warp != NW + NTP / 32) return;
        }
        int last = -1;  // the last chunk whose copies were issued (lane 0); chunks load in order
        if (lane == 0)
            for (int c = 0; c < min(3, nchunks); ++c) {
                load_chunk(c);
                last = c;
            }
        for (int c = 0; c < nchunks; ++c) {
            if (c + 2 < nchunks) {
                bar_sync(kBarEmpty + (c & 1), NTALL + NTX);  // inputs[c % 3] consumed
                if (c + 3 < nchunks && lane == 0 && !*abort) {
                    load_chunk(c + 3);
                    last = c + 3;
                }
            }
            bar_sync(kBarStore, NTC + NTX);  // chunk c's output (and checkpoint) boxes staged
            if (lane == 0 && !*abort) store_chunk(c);
            if (c + 1 < nchunks) {
                if (lane == 0) bulk_wait_read();
                __syncwarp();
                bar_arrive(kBarStoreFree, NTC + NTX);  // the checkpoint box and O[c & 1] free again
            }
        }
        if (lane == 0) {
            bulk_wait();
            // every copy issued has landed before the CTA's shared memory is released (bounded)
            for (int b = 0; b < 3 && b <= last; ++b)  // barrier b took chunks b, b + 3, ..., its last one
                mbar_drain(&mbar[b], (unsigned)(((last - b) / 3) & 1));
        }
        return;
    }

    if (warp >= NW) {
        // ============================== prep warps ==============================
        const int pt = tid - NTC, pw = pt / 32;
        // chunk c: beta and g by 4-byte cp.async (zeros past the prompt); the producer
        // warp loads q, k and v
        auto issue = [&](int c) {
            const int p0 = c * C, kb = c % 3;
            const size_t row0 = ((size_t)n * P + p0) * H + h;
            for (int i = pt; i < 2 * C; i += NTP) {
                const int which = i / C, t = i % C;
                const bool ok = p0 + t < P;
                const float *src = which ? g : beta;
                cp_async4(&sGates[kb][which][t], ok ? (const void *)(src + row0 + (size_t)t * H) : (const void *)src,
                          ok ? 4 : 0);
            }
        };
        if (nchunks > 0) issue(0);
        cp_async_commit();
        for (int c = 0; c < nchunks; ++c) {
            const int p0 = c * C, nc = min(C, P - p0), pb = c & 1, kb = c % 3;
            if (c >= 2) bar_sync(kBarEmpty + pb, NTALL + NTX);  // chunk c-2 done: products[pb], gates[(c+1)%3] free
            if (c + 1 < nchunks) issue(c + 1);
            cp_async_commit();
            cp_async_wait<1>();
            mbar_wait_guarded(&mbar[kb], (unsigned)((c / 3) & 1), abort, &g_prefill_wait_timeouts);
            bar_sync(kBarPrep, NTP);
            const uint4 *cK = sK + kb * KH * BOXU, *cQ = sQ + kb * KH * BOXU;
            const float *sbeta = sGates[kb][0], *sgr = sGates[kb][1];
            (void)p0;
            // grams by MMA, tile = (sub-chunk j, K or Q rows) x K_j^T, with the gate scan of
            // the sub-chunk in the same warp; the epilogue applies the decays in registers:
            // A = beta_t e^{G_t-G_s} k_t.k_s (s < t), Mq = e^{G_t-G_s} q_t.k_s (s <= t).
            // A warp's tiles run their k-loops side by side (independent accumulators). With
            // two tiles a warp, warp pw takes sub-chunk pw's K and Q tiles, which share the
            // K_j fragments (three fragment loads a k-step instead of four).
            constexpr int TPW = 2 * NSUB / (NTP / 32);  // gram tiles per prep warp
            auto tile_of = [&](int u) { return TPW == 2 ? 2 * pw + u : pw + u * (NTP / 32); };
            float e[TPW][2][4];
#pragma unroll
            for (int u = 0; u < TPW; ++u)
#pragma unroll
                for (int w = 0; w < 4; ++w) e[u][0][w] = e[u][1][w] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                unsigned bb[4];
                if constexpr (TPW == 2)
                    ldsm_x4(bb, cK + box_chunk(C, 16 * pw + (lane & 7) + ((lane >> 4) << 3),
                                               2 * ks + ((lane >> 3) & 1)));
#pragma unroll
                for (int u = 0; u < TPW; ++u) {
                    const int tile = tile_of(u), j = tile >> 1;
                    const uint4 *rows = (tile & 1) ? cQ : cK;
                    unsigned a[4];
                    ldsm_x4(a, rows + box_chunk(C, 16 * j + (lane & 15), 2 * ks + (lane >> 4)));
                    if constexpr (TPW != 2) {
                        // K_j^T of a K tile is made of its own A fragments (tokens 0-7: a[0],
                        // a[2]; tokens 8-15: a[1], a[3]); a Q tile loads it
                        if (tile & 1) {
                            ldsm_x4(bb, cK + box_chunk(C, 16 * j + (lane & 7) + ((lane >> 4) << 3),
                                                       2 * ks + ((lane >> 3) & 1)));
                        } else {
                            bb[0] = a[0];
                            bb[1] = a[2];
                            bb[2] = a[1];
                            bb[3] = a[3];
                        }
                    }
                    const unsigned b0[2] = {bb[0], bb[1]}, b1[2] = {bb[2], bb[3]};
                    mma_16816(e[u][0], a, b0);
                    mma_16816(e[u][1], a, b1);
                }
            }
#pragma unroll
            for (int u = 0; u < TPW; ++u) {
                const int tile = tile_of(u);
                const int j = tile >> 1, isq = tile & 1;
                const float *e0 = e[u][0], *e1 = e[u][1];
                const int tl = 16 * j + (lane & 15);
                float G = (tl < nc) ? __logf(fmaxf(sgr[tl], 1e-30f)) : 0.f;  // log g, 0 past the prompt
#pragma unroll
                for (int off = 1; off < 16; off <<= 1) {
                    const float o = __shfl_up_sync(0xffffffffu, G, off, 16);
                    if ((lane & 15) >= off) G += o;
                }
                const float last = __shfl_sync(0xffffffffu, G, 15);
                if (!isq && lane < 16) {
                    sgam[pb][16 * j + lane] = __expf(G);
                    sdec[pb][16 * j + lane] = __expf(last - G);
                }
                const float Gr0 = __shfl_sync(0xffffffffu, G, fr), Gr1 = __shfl_sync(0xffffffffu, G, fr + 8);
                const float Gc[4] = {__shfl_sync(0xffffffffu, G, fc), __shfl_sync(0xffffffffu, G, fc + 1),
                                     __shfl_sync(0xffffffffu, G, fc + 8), __shfl_sync(0xffffffffu, G, fc + 9)};
                const int cs[4] = {fc, fc + 1, fc + 8, fc + 9};
                const float v0[4] = {e0[0], e0[1], e1[0], e1[1]};  // row fr
                const float v1[4] = {e0[2], e0[3], e1[2], e1[3]};  // row fr + 8
                if (!isq) {
                    const float b0r = sbeta[16 * j + fr], b1r = sbeta[16 * j + fr + 8];
                    float a0[4], a1[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        a0[w] = (cs[w] < fr) ? b0r * __expf(Gr0 - Gc[w]) * v0[w] : 0.f;
                        a1[w] = (cs[w] < fr + 8) ? b1r * __expf(Gr1 - Gc[w]) * v1[w] : 0.f;
                    }
                    // columns (fc, fc + 1) and (fc + 8, fc + 9) are pairs within a 16-byte group
                    *reinterpret_cast<float2 *>(sA + a_index(j, fr, fc)) = make_float2(a0[0], a0[1]);
                    *reinterpret_cast<float2 *>(sA + a_index(j, fr, fc + 8)) = make_float2(a0[2], a0[3]);
                    *reinterpret_cast<float2 *>(sA + a_index(j, fr + 8, fc)) = make_float2(a1[0], a1[1]);
                    *reinterpret_cast<float2 *>(sA + a_index(j, fr + 8, fc + 8)) = make_float2(a1[2], a1[3]);
                } else {
                    float m0[4], m1[4];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        m0[w] = (cs[w] <= fr) ? __expf(Gr0 - Gc[w]) * v0[w] : 0.f;
                        m1[w] = (cs[w] <= fr + 8) ? __expf(Gr1 - Gc[w]) * v1[w] : 0.f;
                    }
                    // columns (fc, fc + 1) and (fc + 8, fc + 9) as fp16 pairs
                    *reinterpret_cast<unsigned *>(&sMq[pb][j][fr][fc]) = pack_h2(m0[0], m0[1]);
                    *reinterpret_cast<unsigned *>(&sMq[pb][j][fr][fc + 8]) = pack_h2(m0[2], m0[3]);
                    *reinterpret_cast<unsigned *>(&sMq[pb][j][fr + 8][fc]) = pack_h2(m1[0], m1[1]);
                    *reinterpret_cast<unsigned *>(&sMq[pb][j][fr + 8][fc + 8]) = pack_h2(m1[2], m1[3]);
                }
            }
            bar_sync(kBarPrep, NTP);
            // Tb = (I + A)^{-1} diag(beta): one thread per (sub-chunk, column), forward
            // substitution in fp32; row i of A is read four elements at a time
            if (pt < NSUB * 16) {
                const int j = pt >> 4, col = pt & 15;
                float x[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int g4 = 0; g4 < (i + 3) / 4; ++g4) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(sA + a_index(j, i, 4 * g4));
                        const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            if (4 * g4 + u < i) acc[u] = fmaf(av[u], x[4 * g4 + u], acc[u]);
                    }
                    x[i] = (i < col) ? 0.f : (i == col ? 1.f : -((acc[0] + acc[1]) + (acc[2] + acc[3])));
                }
                const float bc = sbeta[16 * j + col];
#pragma unroll
                for (int i = 0; i < 16; ++i) sTb[pb][j][i][col] = __float2half_rn(x[i] * bc);
            }
            bar_arrive(kBarFull + pb, NTALL);  // chunk c: inputs and products ready
            bar_sync(kBarPrep, NTP);           // prep scratch (A) free again
        }
        cp_async_wait<0>();
        return;
    }

    // ============================== chain warps ==============================
    if constexpr (SPLIT) regs_raise<kChainRegs>();
    // A chain warp owns RT 16-row tiles of the state (rows i0 .. i0 + 16 RT - 1); every
    // operand fragment it loads from shared memory for the projections and the state
    // update serves all RT tiles.
    const int i0 = warp * 16 * RT;  // this warp's rows within the CTA (state rows r0 + i0 ..)
    float DS[RT][NTK][4];           // tile mt, nt: rows i0 + 16 mt .., dk columns 8nt .. 8nt+7
#pragma unroll
    for (int mt = 0; mt < RT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NTK; ++nt) {
            float2 lo = make_float2(0.f, 0.f), hi = lo;
            if (s_in) {
                lo = __half22float2(*reinterpret_cast<const __half2 *>(
                    s_in + state_off + (size_t)(r0 + i0 + 16 * mt + fr) * DK + 8 * nt + fc));
                hi = __half22float2(*reinterpret_cast<const __half2 *>(
                    s_in + state_off + (size_t)(r0 + i0 + 16 * mt + fr + 8) * DK + 8 * nt + fc));
            }
            DS[mt][nt][0] = lo.x; DS[mt][nt][1] = lo.y; DS[mt][nt][2] = hi.x; DS[mt][nt][3] = hi.y;
        }

    for (int c = 0; c < nchunks; ++c) {
        const int p0 = c * C, nc = min(C, P - p0), pb = c & 1, kb = c % 3, ob = c & 1;
        bar_sync(kBarFull + pb, NTALL);
        // the inputs landed (already observed by the prep warps; re-checked, bounded)
        mbar_wait_guarded(&mbar[kb], (unsigned)((c / 3) & 1), abort, &g_prefill_wait_timeouts);
        const uint4 *cK = sK + kb * KH * BOXU, *cQ = sQ + kb * KH * BOXU, *cV = sV + kb * VH * BOXU;
        uint4 *cO = sO + ob * VH * BOXU;
        const float *gam = sgam[pb], *dec = sdec[pb];
#pragma unroll 1
        for (int j = 0; j < NSUB; ++j) {
            if (16 * j >= nc) break;
            float X[RT][4][4];
#pragma unroll
            for (int mt = 0; mt < RT; ++mt)
#pragma unroll
                for (int u = 0; u < 4; ++u) X[mt][u][0] = X[mt][u][1] = X[mt][u][2] = X[mt][u][3] = 0.f;
            // X = S [K_j;Q_j]^T. With two chain warps per scheduler the K and Q fragments of
            // k-step ks + 1 are loaded before the MMAs of step ks (folded 128-row launch 21.18 ->
            // 20.88 ms); with one the loads stay beside their MMAs (the 64-row launch measured
            // 1.4 % slower with the early loads).
            constexpr bool kEarlyKQ = NW == 8;
            const int fr0 = 16 * j + (lane & 7) + ((lane >> 4) << 3), fc0 = (lane >> 3) & 1;
            unsigned fk[2][4], fq[2][4];
            auto load_kq = [&](int ks) {
                ldsm_x4(fk[ks & 1], cK + box_chunk(C, fr0, 2 * ks + fc0));
                ldsm_x4(fq[ks & 1], cQ + box_chunk(C, fr0, 2 * ks + fc0));
            };
            if constexpr (kEarlyKQ) load_kq(0);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if constexpr (kEarlyKQ) {
                    if (ks + 1 < KS) load_kq(ks + 1);
                } else {
                    load_kq(ks);
                }
                const unsigned *bk = fk[ks & 1], *bq = fq[ks & 1];
                const unsigned k0[2] = {bk[0], bk[1]}, k1[2] = {bk[2], bk[3]};
                const unsigned q0[2] = {bq[0], bq[1]}, q1[2] = {bq[2], bq[3]};
#pragma unroll
                for (int mt = 0; mt < RT; ++mt) {
                    unsigned aS[4];
                    acc_to_a(aS, DS[mt][2 * ks], DS[mt][2 * ks + 1]);
                    mma_16816(X[mt][0], aS, k0);
                    mma_16816(X[mt][1], aS, k1);
                    mma_16816(X[mt][2], aS, q0);
                    mma_16816(X[mt][3], aS, q1);
                }
            }
            unsigned bt[4], bm[4];
            ldsm_x4(bt, &sTb[pb][j][(lane & 7) + ((lane >> 4) << 3)][8 * ((lane >> 3) & 1)]);
            ldsm_x4(bm, &sMq[pb][j][(lane & 7) + ((lane >> 4) << 3)][8 * ((lane >> 3) & 1)]);
            const unsigned t0[2] = {bt[0], bt[1]}, t1[2] = {bt[2], bt[3]};
            const unsigned m0[2] = {bm[0], bm[1]}, m1[2] = {bm[2], bm[3]};
            unsigned aT[RT][4];
#pragma unroll
            for (int mt = 0; mt < RT; ++mt) {
                const int im = i0 + 16 * mt;
                unsigned vt[4];
                ldsm_x4_t(vt, cV + box_chunk(C, 16 * j + ((lane >> 4) << 3) + (lane & 7), (im >> 3) + ((lane >> 3) & 1)));
                float R[2][4], Dl[2][4], O[2][4];
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {  // R = V^T - gam X_K ; O starts at gam X_Q
                    const int t = 16 * j + 8 * nt + fc;
                    const float2 gg = *reinterpret_cast<const float2 *>(gam + t);  // t even
                    const float ga = gg.x, gb = gg.y;
                    const float2 lo = unpack_h2(vt[2 * nt]), hi = unpack_h2(vt[2 * nt + 1]);
                    R[nt][0] = lo.x - ga * X[mt][nt][0];
                    R[nt][1] = lo.y - gb * X[mt][nt][1];
                    R[nt][2] = hi.x - ga * X[mt][nt][2];
                    R[nt][3] = hi.y - gb * X[mt][nt][3];
                    O[nt][0] = ga * X[mt][2 + nt][0];
                    O[nt][1] = gb * X[mt][2 + nt][1];
                    O[nt][2] = ga * X[mt][2 + nt][2];
                    O[nt][3] = gb * X[mt][2 + nt][3];
                    Dl[nt][0] = Dl[nt][1] = Dl[nt][2] = Dl[nt][3] = 0.f;
                }
                {   // Delta^T = R Tb^T
                    unsigned aR[4];
                    acc_to_a(aR, R[0], R[1]);
                    mma_16816(Dl[0], aR, t0);
                    mma_16816(Dl[1], aR, t1);
                }
                {   // O^T += Delta^T Mq^T
                    unsigned aD[4];
                    acc_to_a(aD, Dl[0], Dl[1]);
                    mma_16816(O[0], aD, m0);
                    mma_16816(O[1], aD, m1);
                }
                {   // O^T tile -> O box rows t (token), columns i (dv)
                    const int m = lane >> 3, t = 16 * j + 8 * (m >> 1) + (lane & 7);
                    stsm_x4_t(cO + box_chunk(C, t, (im >> 3) + (m & 1)),
                              pack_h2(O[0][0], O[0][1]), pack_h2(O[0][2], O[0][3]),
                              pack_h2(O[1][0], O[1][1]), pack_h2(O[1][2], O[1][3]));
                }
                float Dt[2][4];  // Delta^T diag(e^{G_15 - G}) as the A operand of the state update
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int t = 16 * j + 8 * nt + fc;
                    const float2 dd = *reinterpret_cast<const float2 *>(dec + t);  // t even
                    const float da = dd.x, db = dd.y;
                    Dt[nt][0] = Dl[nt][0] * da;
                    Dt[nt][1] = Dl[nt][1] * db;
                    Dt[nt][2] = Dl[nt][2] * da;
                    Dt[nt][3] = Dl[nt][3] * db;
                }
                acc_to_a(aT[mt], Dt[0], Dt[1]);
            }
            {   // S = gam_15 S + (Delta^T diag(e^{G_15 - G})) K_j
                const float gend = gam[16 * j + 15];
                const float2 g2 = make_float2(gend, gend);
#pragma unroll
                for (int mt = 0; mt < RT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt) {
                        const float2 lo = __fmul2_rn(g2, make_float2(DS[mt][nt][0], DS[mt][nt][1]));
                        const float2 hi = __fmul2_rn(g2, make_float2(DS[mt][nt][2], DS[mt][nt][3]));
                        DS[mt][nt][0] = lo.x; DS[mt][nt][1] = lo.y; DS[mt][nt][2] = hi.x; DS[mt][nt][3] = hi.y;
                    }
#pragma unroll
                for (int c2 = 0; c2 < NTK / 2; ++c2) {
                    unsigned bk[4];
                    ldsm_x4_t(bk, cK + box_chunk(C, 16 * j + (lane & 7) + (((lane >> 3) & 1) << 3),
                                                 2 * c2 + (lane >> 4)));
                    const unsigned b0[2] = {bk[0], bk[1]}, b1[2] = {bk[2], bk[3]};
#pragma unroll
                    for (int mt = 0; mt < RT; ++mt) {
                        mma_16816(DS[mt][2 * c2], aT[mt], b0);
                        mma_16816(DS[mt][2 * c2 + 1], aT[mt], b1);
                    }
                }
            }
        }
        if (c + 2 < nchunks) bar_arrive(kBarEmpty + pb, NTALL + NTX);  // inputs / products of chunk c consumed
        // The previous chunk's TMA stores have read the checkpoint box (and O[ob ^ 1]).
        if (c >= 1) bar_sync(kBarStoreFree, NTC + NTX);
        if (nc == C) {   // chunk end: the carry becomes the fp16 checkpoint, staged for the TMA store
#pragma unroll
            for (int mt = 0; mt < RT; ++mt)
#pragma unroll
                for (int c2 = 0; c2 < NTK / 2; ++c2) {
                    unsigned r[4];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const __half2 lo = __floats2half2_rn(DS[mt][2 * c2 + u][0], DS[mt][2 * c2 + u][1]);
                        const __half2 hi = __floats2half2_rn(DS[mt][2 * c2 + u][2], DS[mt][2 * c2 + u][3]);
                        r[2 * u] = *reinterpret_cast<const unsigned *>(&lo);
                        r[2 * u + 1] = *reinterpret_cast<const unsigned *>(&hi);
                        const float2 l2 = __half22float2(lo), h2 = __half22float2(hi);
                        DS[mt][2 * c2 + u][0] = l2.x; DS[mt][2 * c2 + u][1] = l2.y;
                        DS[mt][2 * c2 + u][2] = h2.x; DS[mt][2 * c2 + u][3] = h2.y;
                    }
                    // matrices: rows 0-7 / 8-15 of dk columns 16c2.., then of 16c2+8..
                    const int m = lane >> 3, row = i0 + 16 * mt + (m & 1) * 8 + (lane & 7);
                    stsm_x4(sCk + box_chunk(DVC, row, 2 * c2 + (m >> 1)), r[0], r[1], r[2], r[3]);
                }
        }
        fence_proxy_async();
        bar_arrive(kBarStore, NTC + NTX);  // O boxes and checkpoint boxes staged for the producer
    }
    if (*abort) return;  // a wait ran out: no results are stored
#pragma unroll
    for (int mt = 0; mt < RT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NTK; ++nt) {
            *reinterpret_cast<__half2 *>(s_out + state_off + (size_t)(r0 + i0 + 16 * mt + fr) * DK + 8 * nt + fc) =
                __floats2half2_rn(DS[mt][nt][0], DS[mt][nt][1]);
            *reinterpret_cast<__half2 *>(s_out + state_off + (size_t)(r0 + i0 + 16 * mt + fr + 8) * DK + 8 * nt + fc) =
                __floats2half2_rn(DS[mt][nt][2], DS[mt][nt][3]);
        }
}

int sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sms;
}

template <int DK, int DV, int DVC, int RT>
dn_status launch_prefill_wy_split(int N, int H, int P, const void *q, const void *k, const void *v,
                                  const float *beta, const float *g, const void *s_in, void *out,
                                  void *ckpt, void *s_out, cudaStream_t st) {
    constexpr size_t bytes = PrefillSmem<DK, DVC>::kBytes;
    // Set on every launch (a host call of about a microsecond): the attribute belongs to the
    // current device's context, and a flag cached across calls would race between host
    // threads and miss a second device.
    if (cudaFuncSetAttribute(prefill_wy_kernel<DK, DV, DVC, RT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)bytes) != cudaSuccess) {
        cudaGetLastError();
        return DN_ERR_CUDA;
    }
    PrefillMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (P > 0) {
        // q, k [N][P][H][DK], v, out [N][P][H][DV] as 4-d (d, head, token, sequence)
        const cuuint64_t dk_dims[4] = {(cuuint64_t)DK, (cuuint64_t)H, (cuuint64_t)P, (cuuint64_t)N};
        const cuuint64_t dk_str[3] = {(cuuint64_t)DK * 2, (cuuint64_t)H * DK * 2, (cuuint64_t)P * H * DK * 2};
        const cuuint64_t dv_dims[4] = {(cuuint64_t)DV, (cuuint64_t)H, (cuuint64_t)P, (cuuint64_t)N};
        const cuuint64_t dv_str[3] = {(cuuint64_t)DV * 2, (cuuint64_t)H * DV * 2, (cuuint64_t)P * H * DV * 2};
        const cuuint32_t box4[4] = {64, 1, 64, 1};
        if (!encode_map(&maps.q, q, 4, dk_dims, dk_str, box4) ||
            !encode_map(&maps.k, k, 4, dk_dims, dk_str, box4) ||
            !encode_map(&maps.v, v, 4, dv_dims, dv_str, box4) ||
            !encode_map(&maps.o, out, 4, dv_dims, dv_str, box4))
            return DN_ERR_CUDA;
    }
    if (P >= 64) {
        // ckpt [N][P/64][H][DV][DK] as 3-d (dk, dv, checkpoint tile); a box is DVC rows
        const cuuint64_t dims[3] = {(cuuint64_t)DK, (cuuint64_t)DV, (cuuint64_t)N * (P / 64) * H};
        const cuuint64_t str[2] = {(cuuint64_t)DK * 2, (cuuint64_t)DV * DK * 2};
        const cuuint32_t box3[3] = {64, (cuuint32_t)DVC, 1};
        if (!encode_map(&maps.ck, ckpt, 3, dims, str, box3)) return DN_ERR_CUDA;
    }
    prefill_wy_kernel<DK, DV, DVC, RT><<<(unsigned)((long long)N * H * (DV / DVC)),
                                      prefill_threads<DK, DVC, RT>(), bytes,
                                      st>>>(
        H, P, maps, beta, g, static_cast<const __half *>(s_in), static_cast<__half *>(s_out));
    return DN_OK;
}

template <int DK, int DV>
dn_status launch_prefill_wy(int N, int H, int P, const void *q, const void *k, const void *v,
                            const float *beta, const float *g, const void *s_in, void *out,
                            void *ckpt, void *s_out, cudaStream_t st) {
    if (DV == 128 && (long long)N * H < sm_count())
        return launch_prefill_wy_split<DK, DV, 64, kRowTiles>(N, H, P, q, k, v, beta, g, s_in, out, ckpt, s_out, st);
    return launch_prefill_wy_split<DK, DV, DV, kRowTiles>(N, H, P, q, k, v, beta, g, s_in, out, ckpt, s_out, st);
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

extern "C" unsigned int dn_prefill_wait_timeouts(void) {
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, dn::g_prefill_wait_timeouts, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return 0xffffffffu;
    }
    const unsigned int w = dn::prefill_tc_wait_timeouts();
    return w == 0xffffffffu ? w : v + w;
}

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
        dn_status r;
        if (dk == 128 && dv == 128) r = launch_prefill_wy<128, 128>(N, H, P, q, k, v, beta, g, state_in, out, ckpt, state_out, st);
        else if (dk == 128) r = launch_prefill_wy<128, 64>(N, H, P, q, k, v, beta, g, state_in, out, ckpt, state_out, st);
        else if (dv == 128) r = launch_prefill_wy<64, 128>(N, H, P, q, k, v, beta, g, state_in, out, ckpt, state_out, st);
        else r = launch_prefill_wy<64, 64>(N, H, P, q, k, v, beta, g, state_in, out, ckpt, state_out, st);
        if (r != DN_OK) return r;
    } else {
        if (dk == 128) launch_prefill_seq<128, float, float>(N, H, P, chunk, dv, q, k, v, beta, g, state_in, out, ckpt, state_out, st);
        else launch_prefill_seq<64, float, float>(N, H, P, chunk, dv, q, k, v, beta, g, state_in, out, ckpt, state_out, st);
    }
    return launch_status();
}

extern "C" dn_status dn_prefill_checkpoint_tc(int N, int H, int P, int chunk, int dk, int dv, dn_dtype io_dt,
                                              dn_dtype state_dt, const void *q, const void *k, const void *v,
                                              const float *beta, const float *g, const void *state_in, void *out,
                                              void *ckpt, void *state_out, dn_stream_t stream) {
    using namespace dn;
    if (N < 0 || H < 1 || P < 0) return DN_ERR_INVALID_ARG;
    if (!dtype_ok(io_dt) || !dtype_ok(state_dt)) return DN_ERR_INVALID_ARG;
    if (chunk != DN_PREFILL_CHUNK) return DN_ERR_UNSUPPORTED;
    if (dk != 128 || dv != 128 || io_dt != DN_F16 || state_dt != DN_F16) return DN_ERR_UNSUPPORTED;
    if (N == 0) return DN_OK;
    if (!state_out) return DN_ERR_INVALID_ARG;
    if (P > 0 && (!q || !k || !v || !beta || !g || !out)) return DN_ERR_INVALID_ARG;
    if (P >= chunk && !ckpt) return DN_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(ckpt, 16) ||
        !aligned(state_in, 16) || !aligned(state_out, 16) || !aligned(beta, 4) || !aligned(g, 4))
        return DN_ERR_INVALID_ARG;
    if ((long long)N * H > 0x7fffffffLL) return DN_ERR_INVALID_ARG;
    const dn_status r = launch_prefill_tc(N, H, P, q, k, v, beta, g, state_in, out, ckpt, state_out,
                                          reinterpret_cast<cudaStream_t>(stream));
    if (r != DN_OK) return r;
    return launch_status();
}
