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
#include "dn_internal.h"

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

}  // namespace
}  // namespace dn

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
