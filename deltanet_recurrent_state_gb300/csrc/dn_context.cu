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
// One thread-block cluster per request: its CTAs split 1..L-1, reduce their keys in shared
// memory and then into the leader CTA's shared memory with distributed-shared-memory
// atomics. The leader writes the drafts. HBM bound: L * 4 bytes read per request.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dn.h"
#include "dn_internal.h"

namespace cg = cooperative_groups;

namespace dn {
namespace {

constexpr int kCtxThreads = 256;
constexpr int kCtxUnroll = 8;
constexpr int kPosBits = 27;  // e < 2^27 so that (len, e) packs into 32 bits
constexpr unsigned kPosMask = (1u << kPosBits) - 1u;
constexpr int kMaxCluster = 8;
constexpr int kPositionsPerCta = 4096;

__global__ void __launch_bounds__(kCtxThreads)
context_drafts_kernel(int stride, int n_max, int n_min, int K, const int32_t *__restrict__ context,
                      const int32_t *__restrict__ lengths, int32_t *__restrict__ drafts,
                      int32_t *__restrict__ count, int32_t *__restrict__ match_len) {
    cg::cluster_group cluster = cg::this_cluster();
    const unsigned C = cluster.num_blocks();
    const unsigned rank = cluster.block_rank();
    const size_t n = blockIdx.x / C;
    __shared__ int32_t pat[DN_MAX_NGRAM];
    __shared__ unsigned warp_best[kCtxThreads / 32];
    __shared__ unsigned cluster_best;

    const int32_t *c = context + n * (size_t)stride;
    int L = __ldg(&lengths[n]);
    L = L < 0 ? 0 : (L > stride ? stride : L);
    const int tid = threadIdx.x;
    if (tid < n_max && tid < L) pat[tid] = __ldg(&c[L - 1 - tid]);
    if (tid == 0) cluster_best = 0u;
    cluster.sync();  // pattern loaded; the leader's cell is cleared before any remote atomic

    // this CTA's share of the end positions 1 .. L-1
    const long long E = L > 1 ? L - 1 : 0;
    const int lo = 1 + (int)(E * rank / C), hi = 1 + (int)(E * (rank + 1) / C);
    const int32_t last = L > 0 ? pat[0] : 0;
    unsigned best = 0u;
    for (int base = lo; base < hi; base += kCtxThreads * kCtxUnroll) {
        int32_t x[kCtxUnroll];
#pragma unroll
        for (int u = 0; u < kCtxUnroll; ++u) {
            const int e = base + u * kCtxThreads + tid;
            x[u] = e < hi ? __ldg(&c[e - 1]) : ~last;
        }
#pragma unroll
        for (int u = 0; u < kCtxUnroll; ++u) {
            if (x[u] != last) continue;
            const int e = base + u * kCtxThreads + tid;
            const int lim = n_max < e ? n_max : e;
            int l = 1;
            while (l < lim && __ldg(&c[e - 1 - l]) == pat[l]) ++l;
            if (l >= n_min) {
                const unsigned key = ((unsigned)l << kPosBits) | (unsigned)e;
                best = key > best ? key : best;
            }
        }
    }
    best = __reduce_max_sync(0xffffffffu, best);
    if ((tid & 31) == 0) warp_best[tid >> 5] = best;
    __syncthreads();
    if (tid < 32) {
        unsigned b = tid < kCtxThreads / 32 ? warp_best[tid] : 0u;
        b = __reduce_max_sync(0xffffffffu, b);
        if (tid == 0 && b) atomicMax(cluster.map_shared_rank(&cluster_best, 0), b);
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
    cfg.dynamicSmemBytes = 0;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, context_drafts_kernel, stride, n_max, n_min, K, context, lengths,
                           drafts, count, match_len) != cudaSuccess) {
        cudaGetLastError();
        return DN_ERR_CUDA;
    }
    return launch_status();
}
