// dn_context_drafts: draft tokens copied from the request's own context.
//
// In single-user mode the later positions of a verify block are filled from the request's
// context instead of by the drafter, because models often quote their input verbatim
// ("HyperQwen: 1,000 tok/s on a Single RTX 3090 ...", Technical Insight; "HyperQwen on one
// RTX 3090: a first-time developer's guide ...", What actually became faster?). The match
// rule: the pattern is the last n tokens of the context; take its latest earlier occurrence
// that has at least one token after it, for the largest n in n_min..n_max that has one, and
// propose the (up to K) tokens that follow.
//
// One pass computes it for every n at once. For each end position e in 1..L-1 let len(e)
// be the length of the common suffix of context[0, e) and context[0, L), capped at n_max.
// The chosen n is max_e len(e) and the chosen occurrence the largest e with that length, so
// the answer is the maximum of the key (len(e), e) over all e with len(e) >= n_min. A
// position costs one coalesced 4-byte load (context[e-1] against the last token); the
// comparison extends backwards only on a hit.
//
// One thread-block cluster per request: its CTAs claim the request's 4096-token tiles
// (two fixed ones each, then dynamically from a counter in the leader CTA's shared memory)
// and stream them through a three-stage shared-memory ring filled by cp.async: two tiles
// in flight while one is scanned. Each stage also holds the 16 tokens before its tile, so
// the backward compares after a hit never go to global memory. Each thread turns its 16
// tokens into a hit mask and walks only the hits. Keys are reduced in shared memory and
// then into the leader CTA's shared memory with distributed-shared-memory atomics; the
// leader writes the drafts. HBM bound: L * 4 bytes read per request.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "dn.h"
#include "dn_internal.h"
#include "dn_mma.cuh"

namespace cg = cooperative_groups;

namespace dn {
namespace {

constexpr int kCtxThreads = 256;
constexpr int kTile = 4096;            // tokens per CTA iteration (16 KB)
constexpr int kHalo = DN_MAX_NGRAM;    // tokens kept before a tile for backward compares
constexpr int kStages = 3;             // tile ring: two tiles in flight while one is scanned
constexpr int kStageInts = kHalo + kTile;
constexpr size_t kCtxSmemBytes = (size_t)kStages * kStageInts * sizeof(int32_t);
constexpr int kPerThread = kTile / kCtxThreads;  // 16 tokens: 4 runs of 4
constexpr int kPosBits = 27;  // e < 2^27 so that (len, e) packs into 32 bits
constexpr unsigned kPosMask = (1u << kPosBits) - 1u;
constexpr int kMaxCluster = 8;
constexpr int kPositionsPerCta = 4096;

// Tile tokens t0 - 16 .. t0 + 4095 into a stage by cp.async (the 16 before the tile first,
// then the tile itself as runs of 4 at t0 + 4 (tid + 256 u)): 16-byte copies when the row
// allows them (VEC), else 4-byte copies. Tokens before the context or past its end are
// written as zeros (they are never compared).
template <bool VEC>
__device__ __forceinline__ void issue_tile(int32_t *stage, const int32_t *__restrict__ c, int t0, int L) {
    const int tid = threadIdx.x;
    if (VEC) {
        if (tid < kHalo / 4) {
            const int j = t0 - kHalo + 4 * tid;  // t0 >= 16 or the whole run is before 0
            cp_async16(&stage[4 * tid], j >= 0 ? c + j : c, j >= 0 ? 16 : 0);
        }
    } else if (tid < kHalo) {
        const int j = t0 - kHalo + tid;
        cp_async4(&stage[tid], j >= 0 ? c + j : c, j >= 0 ? 4 : 0);
    }
#pragma unroll
    for (int u = 0; u < kPerThread / 4; ++u) {
        const int q = tid + kCtxThreads * u, j = t0 + 4 * q;
        if (VEC) {
            // the row pitch is a multiple of 4 tokens, so the run at j < L is inside the row
            cp_async16(&stage[kHalo + 4 * q], j < L ? c + j : c, j < L ? 16 : 0);
        } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
                cp_async4(&stage[kHalo + 4 * q + v], j + v < L ? c + j + v : c, j + v < L ? 4 : 0);
        }
    }
}

template <bool VEC>
__global__ void __launch_bounds__(kCtxThreads)
context_drafts_kernel(int stride, int n_max, int n_min, int K, const int32_t *__restrict__ context,
                      const int32_t *__restrict__ lengths, int32_t *__restrict__ drafts,
                      int32_t *__restrict__ count, int32_t *__restrict__ match_len) {
    cg::cluster_group cluster = cg::this_cluster();
    const unsigned C = cluster.num_blocks();
    const unsigned rank = cluster.block_rank();
    const size_t n = blockIdx.x / C;
    extern __shared__ __align__(16) int32_t ring[];  // kStages x (halo + tile)
    __shared__ int32_t pat[DN_MAX_NGRAM];
    __shared__ unsigned warp_best[kCtxThreads / 32];
    __shared__ unsigned cluster_best, next_tile;
    __shared__ int tile_of[4];  // tile index of iteration it, slot it % 4

    const int32_t *c = context + n * (size_t)stride;
    int L = __ldg(&lengths[n]);
    L = L < 0 ? 0 : (L > stride ? stride : L);
    const int tid = threadIdx.x;

    // Token j = e - 1 for the end positions e = 1 .. L-1: j in [0, J), J = L - 1, in tiles
    // of 4096 (each starts on a 16-byte boundary). CTA r of the cluster takes tiles r and
    // r + C first; after that each CTA takes the next unclaimed tile from a counter in the
    // leader's shared memory, so CTAs on busier SMs take fewer tiles.
    const int J = L > 1 ? L - 1 : 0;
    const int ntiles = (J + kTile - 1) / kTile;
    const int first = (int)rank, second = (int)(rank + C);
    if (first < ntiles) issue_tile<VEC>(ring, c, first * kTile, L);
    cp_async_commit();
    if (second < ntiles) issue_tile<VEC>(ring + kStageInts, c, second * kTile, L);
    cp_async_commit();
    if (tid < DN_MAX_NGRAM) pat[tid] = (tid < n_max && tid < L) ? __ldg(&c[L - 1 - tid]) : 0;
    if (tid == 0) {
        cluster_best = 0u;
        next_tile = 0u;
        tile_of[0] = first;
        tile_of[1] = second;
    }
    cluster.sync();  // pattern loaded; the leader's cells are set before any remote atomic
    unsigned *leader_next = cluster.map_shared_rank(&next_tile, 0);
    if (tid == 0) tile_of[2] = (int)(2 * C + atomicAdd(leader_next, 1u));
    // (visible to the other threads at the first barrier of the loop)

    const int32_t last = pat[0], p1 = pat[1], p2 = pat[2], p3 = pat[3];
    unsigned best = 0u;
    for (int it = 0;; ++it) {
        int32_t *b = ring + (it % kStages) * kStageInts;
        cp_async_wait<1>();  // this thread's copies for iteration `it` landed
        __syncthreads();     // ... and everyone's; every reader of the stage refilled below is done
        const int tile = tile_of[it & 3];
        if (tile >= ntiles) break;  // claims only grow: nothing left for this CTA
        const int t2 = tile_of[(it + 2) & 3];
        if (t2 < ntiles) issue_tile<VEC>(ring + ((it + 2) % kStages) * kStageInts, c, t2 * kTile, L);
        cp_async_commit();
        if (tid == 0) tile_of[(it + 3) & 3] = t2 < ntiles ? (int)(2 * C + atomicAdd(leader_next, 1u)) : ntiles;
        const int t0 = tile * kTile;
        // this thread's 16 tokens -> a mask of the ones equal to the last token
        unsigned m = 0u;
#pragma unroll
        for (int u = 0; u < kPerThread / 4; ++u) {
            const int4 x = *reinterpret_cast<const int4 *>(&b[kHalo + 4 * (tid + kCtxThreads * u)]);
            m |= (x.x == last ? 1u : 0u) << (4 * u);
            m |= (x.y == last ? 2u : 0u) << (4 * u);
            m |= (x.z == last ? 4u : 0u) << (4 * u);
            m |= (x.w == last ? 8u : 0u) << (4 * u);
        }
        // only the hits walk backwards (a lane handles one of its hits per round)
        while (m) {
            const int bit = __ffs(m) - 1;
            m &= m - 1u;
            const int o = 4 * (tid + kCtxThreads * (bit >> 2)) + (bit & 3);  // offset in the tile
            const int j = t0 + o;
            if (j >= J) continue;
            const int e = j + 1;
            const int lim = n_max < e ? n_max : e;
            // the three tokens before the hit in one go (the stage's halo makes them
            // readable; they only count while l < lim <= e, i.e. inside the context)
            const int32_t a1 = b[kHalo + o - 1], a2 = b[kHalo + o - 2], a3 = b[kHalo + o - 3];
            int l = 1;
            if (lim > 1 && a1 == p1) {
                l = 2;
                if (lim > 2 && a2 == p2) {
                    l = 3;
                    if (lim > 3 && a3 == p3) {
                        l = 4;
                        while (l < lim && b[kHalo + o - l] == pat[l]) ++l;
                    }
                }
            }
            if (l >= n_min) {
                const unsigned key = ((unsigned)l << kPosBits) | (unsigned)e;
                best = key > best ? key : best;
            }
        }
    }
    cp_async_wait<0>();
    best = __reduce_max_sync(0xffffffffu, best);
    if ((tid & 31) == 0) warp_best[tid >> 5] = best;
    __syncthreads();
    if (tid < 32) {
        unsigned bw = tid < kCtxThreads / 32 ? warp_best[tid] : 0u;
        bw = __reduce_max_sync(0xffffffffu, bw);
        if (tid == 0 && bw) atomicMax(cluster.map_shared_rank(&cluster_best, 0), bw);
    }
    cluster.sync();  // every CTA's key is in the leader's cell
    if (rank != 0) return;

    const unsigned key = cluster_best;
    const int l = (int)(key >> kPosBits), e = (int)(key & kPosMask);
    const int m = key ? (K < L - e ? K : L - e) : 0;
    if (tid < K) drafts[n * K + tid] = tid < m ? __ldg(&c[e + tid]) : -1;
    if (tid == 0) {
        count[n] = m;
        if (match_len) match_len[n] = l;
    }
}

// The tile ring is above the 48 KB a kernel gets without opting in; the opt-in is a
// per-device function attribute, set once per device and variant.
bool allow_ring_smem(bool vec) {
    static std::atomic<unsigned long long> done[2];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const unsigned long long bit = 1ull << dev;
    if (done[vec].load(std::memory_order_acquire) & bit) return true;
    const cudaError_t err =
        vec ? cudaFuncSetAttribute(context_drafts_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kCtxSmemBytes)
            : cudaFuncSetAttribute(context_drafts_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kCtxSmemBytes);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    done[vec].fetch_or(bit, std::memory_order_acq_rel);
    return true;
}

}  // namespace
}  // namespace dn

extern "C" dn_status dn_context_drafts(int N, int stride, int n_max, int n_min, int K,
                                       const int32_t *context, const int32_t *lengths,
                                       int32_t *drafts, int32_t *count, int32_t *match_len,
                                       dn_stream_t stream) {
    using namespace dn;
    if (N < 0 || stride < 0 || stride > (int)kPosMask || n_min < 1 || n_max < n_min ||
        n_max > DN_MAX_NGRAM || K < 1 || K > DN_MAX_BLOCK)
        return DN_ERR_INVALID_ARG;
    if (N == 0) return DN_OK;
    if (!context || !lengths || !drafts || !count) return DN_ERR_INVALID_ARG;
    if (!aligned(context, 4) || !aligned(lengths, 4) || !aligned(drafts, 4) || !aligned(count, 4) ||
        (match_len && !aligned(match_len, 4)))
        return DN_ERR_INVALID_ARG;
    int C = (stride + kPositionsPerCta - 1) / kPositionsPerCta;
    C = C < 1 ? 1 : (C > kMaxCluster ? kMaxCluster : C);
    if ((long long)N * C > 0x7fffffffLL) return DN_ERR_INVALID_ARG;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(N * C));
    cfg.blockDim = dim3(kCtxThreads);
    cfg.dynamicSmemBytes = kCtxSmemBytes;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool vec = aligned(context, 16) && stride % 4 == 0;
    if (!allow_ring_smem(vec)) return DN_ERR_CUDA;
    const cudaError_t err =
        vec ? cudaLaunchKernelEx(&cfg, context_drafts_kernel<true>, stride, n_max, n_min, K, context,
                                 lengths, drafts, count, match_len)
            : cudaLaunchKernelEx(&cfg, context_drafts_kernel<false>, stride, n_max, n_min, K, context,
                                 lengths, drafts, count, match_len);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return DN_ERR_CUDA;
    }
    return launch_status();
}
