// dn_accept_greedy: greedy verification of B draft blocks in one launch.
//
// Greedy verify ("Qwen3.8-27B on a Single RTX 3090: ...", Technical Insight,
// split-KV verify): the target token at each position is the argmax of its
// logits row, and the accepted length is the longest prefix on which the drafts
// equal the targets.
//
// One pass over the logits. One CTA per (row, chunk of kChunk vocab entries), B*T rows,
// numbered row-major on grid.x (so the row count is not bounded by grid.y).
// Each CTA reduces its chunk to one 64-bit key, (order-preserving value bits << 32)
// | (0xffffffff - index), so an unsigned max picks the largest value and, among
// equal values, the lowest index; the order of the reduction cannot change the
// answer. The last CTA of a row (found with a counter in the workspace) reduces
// the row's chunk keys and writes the target id; the last row of a request then
// computes the accepted length. With few rows (a single request's verify block, or a
// few), one level does it all: the last CTA of the whole grid reduces every row and
// computes every accepted length, which saves the second level's fence and atomic
// round trips on the launch's serial tail. Counters are reset by the CTA that
// finishes them, so the workspace is ready for the next call. Nothing spins or waits.
#include <mutex>

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "dn.h"
#include "dn_device.cuh"
#include "dn_internal.h"

namespace dn {
namespace {

constexpr int kChunk = 8192;   // vocab entries per CTA
constexpr int kThreads = 256;
constexpr int kFlatRows = 16;  // up to this many rows (B x T), the one-level reduction

__host__ __device__ inline int accept_chunks(int V) { return (V + kChunk - 1) / kChunk; }

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// One CTA per (row, chunk) on grid.x: at most 2^31 - 1 of them; the last row's index must
// also fit the int32 target/draft arrays.
inline bool accept_grid_ok(int B, int T, int V) {
    const long long rows = (long long)B * T;
    return rows <= 0x7fffffffLL && rows * accept_chunks(V) <= 0x7fffffffLL;
}

struct AcceptWorkspace {
    unsigned long long *keys;   // [rows][chunks]
    unsigned int *row_count;    // [rows]
    unsigned int *req_count;    // [B]
};

__host__ __device__ inline size_t accept_ws_bytes(int B, int T, int V) {
    const size_t rows = (size_t)B * T;
    return align16(rows * accept_chunks(V) * sizeof(unsigned long long)) +
           align16(rows * sizeof(unsigned int)) + align16((size_t)B * sizeof(unsigned int));
}

__host__ __device__ inline AcceptWorkspace accept_ws(void *base, int B, int T, int V) {
    const size_t rows = (size_t)B * T;
    char *p = static_cast<char *>(base);
    AcceptWorkspace w;
    w.keys = reinterpret_cast<unsigned long long *>(p);
    p += align16(rows * accept_chunks(V) * sizeof(unsigned long long));
    w.row_count = reinterpret_cast<unsigned int *>(p);
    p += align16(rows * sizeof(unsigned int));
    w.req_count = reinterpret_cast<unsigned int *>(p);
    return w;
}

// Order-preserving maps of the value bits to unsigned integers (any value but NaN).
// -0.0 is folded onto +0.0 first, so the two compare equal as numbers do.
__device__ __forceinline__ unsigned int order_key(unsigned short h) {
    if ((h & 0x7fffu) == 0) h = 0;
    return (h & 0x8000u) ? (unsigned int)(~h & 0xffffu) : (unsigned int)(h | 0x8000u);
}
__device__ __forceinline__ unsigned int order_key(unsigned int f) {
    if ((f & 0x7fffffffu) == 0) f = 0;
    return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}

__device__ __forceinline__ unsigned long long pack_key(unsigned int key, int idx) {
    return ((unsigned long long)key << 32) | (unsigned long long)(0xffffffffu - (unsigned int)idx);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

__device__ __forceinline__ unsigned long long block_max(unsigned long long x, unsigned long long *red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = umax64(x, __shfl_xor_sync(0xffffffffu, x, off));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (lane == 0) red[warp] = x;
    __syncthreads();
    if (warp == 0) {
        x = lane < kThreads / 32 ? red[lane] : 0ull;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x = umax64(x, __shfl_xor_sync(0xffffffffu, x, off));
    }
    return x;  // valid in warp 0
}

// Element bits type -> elements per 16-byte vector
template <typename E> struct Bits;
template <> struct Bits<unsigned short> { static constexpr int kVec = 8; };
template <> struct Bits<unsigned int> { static constexpr int kVec = 4; };

// FLAT: the one-level reduction (rows <= kFlatRows), chosen at launch.
template <typename E, bool FLAT>
__global__ void __launch_bounds__(kThreads)
accept_greedy_kernel(int B, int T, int V, int chunks, const E *__restrict__ logits,
                     const int *__restrict__ draft, int *__restrict__ target,
                     int *__restrict__ accepted, AcceptWorkspace ws) {
    constexpr int VEC = Bits<E>::kVec;
    __shared__ unsigned long long red[kThreads / 32];
    __shared__ int is_last;
    const int c = (int)(blockIdx.x % (unsigned)chunks);
    const int row = (int)(blockIdx.x / (unsigned)chunks);
    grid_dep_wait();
    grid_dep_trigger();
    const E *rp = logits + (size_t)row * V;
    const int c0 = c * kChunk;
    const int c1 = min(V, c0 + kChunk);

    unsigned long long best = 0ull;
    // 16-byte vector loads where the row stays 16-byte aligned, scalar otherwise.
    const bool vec_ok = ((size_t)V * sizeof(E)) % 16 == 0;
    int done = c0;
    if (vec_ok) {
        // all of this thread's 16-byte loads are issued before any is used
        constexpr int kPer = kChunk / (VEC * kThreads);
        const int nvec = (c1 - c0) / VEC;
        const uint4 *vp = reinterpret_cast<const uint4 *>(rp + c0);
        uint4 u[kPer];
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            const int i = threadIdx.x + r * kThreads;
            if (i < nvec) u[r] = __ldcs(vp + i);
        }
        if constexpr (VEC == 8) {
            // fp16: the thread's maximum by packed max, then the lowest index holding it (its
            // elements are in increasing index order); -0 and +0 compare equal, as numbers do.
            // The running maximum starts at -inf, so a row masked to -inf still finds index 0.
            const __half2 lowest = __halves2half2(__ushort_as_half(0xfc00u), __ushort_as_half(0xfc00u));
            __half2 m2 = lowest;
#pragma unroll
            for (int r = 0; r < kPer; ++r) {
                const int i = threadIdx.x + r * kThreads;
                if (i < nvec) {
                    const __half2 *h2 = reinterpret_cast<const __half2 *>(&u[r]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) m2 = __hmax2(m2, h2[j]);
                }
            }
            const __half m = __hmax(__low2half(m2), __high2half(m2));
            int idx = -1;
#pragma unroll
            for (int r = kPer - 1; r >= 0; --r) {
                const int i = threadIdx.x + r * kThreads;
                if (i < nvec) {
                    const __half *e = reinterpret_cast<const __half *>(&u[r]);
#pragma unroll
                    for (int j = VEC - 1; j >= 0; --j)
                        if (__heq(e[j], m)) idx = c0 + i * VEC + j;
                }
            }
            if (idx >= 0) best = pack_key(order_key(__half_as_ushort(m)), idx);
        } else {
#pragma unroll
            for (int r = 0; r < kPer; ++r) {
                const int i = threadIdx.x + r * kThreads;
                if (i < nvec) {
                    const E *e = reinterpret_cast<const E *>(&u[r]);
                    const int base = c0 + i * VEC;
#pragma unroll
                    for (int j = 0; j < VEC; ++j) best = umax64(best, pack_key(order_key(e[j]), base + j));
                }
            }
        }
        done = c0 + nvec * VEC;
    }
    for (int i = done + threadIdx.x; i < c1; i += kThreads)
        best = umax64(best, pack_key(order_key(rp[i]), i));
    best = block_max(best, red);

    if constexpr (FLAT) {
        const int rows = B * T;
        // One level: the last CTA of the grid reduces every row, then every request.
        __shared__ int s_tgt[kFlatRows];
        if (threadIdx.x == 0) {
            ws.keys[(size_t)row * chunks + c] = best;
            __threadfence();
            const unsigned int prev = atomicAdd(&ws.row_count[0], 1u);
            is_last = (prev == (unsigned int)(chunks * rows) - 1);
        }
        __syncthreads();
        if (!is_last) return;
        __threadfence();
        const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
        for (int r = warp; r < rows; r += kThreads / 32) {
            unsigned long long kr = 0ull;
            for (int i = lane; i < chunks; i += 32) kr = umax64(kr, __ldcg(&ws.keys[(size_t)r * chunks + i]));
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) kr = umax64(kr, __shfl_xor_sync(0xffffffffu, kr, off));
            if (lane == 0) {
                const int t = (int)(0xffffffffu - (unsigned int)(kr & 0xffffffffull));
                target[r] = t;
                s_tgt[r] = t;
            }
        }
        __syncthreads();
        for (int b = warp; b < B; b += kThreads / 32) {  // accepted length = first mismatch
            int a = T;
            for (int t0 = 0; t0 < T && a == T; t0 += 32) {
                const int t = t0 + lane;
                const bool miss = t < T && __ldg(&draft[b * T + t]) != s_tgt[b * T + t];
                const unsigned m = __ballot_sync(0xffffffffu, miss);
                if (m) a = t0 + __ffs(m) - 1;
            }
            if (lane == 0) accepted[b] = a;
        }
        if (threadIdx.x == 0) ws.row_count[0] = 0u;
        return;
    }

    if (threadIdx.x == 0) {
        ws.keys[(size_t)row * chunks + c] = best;
        __threadfence();
        const unsigned int prev = atomicAdd(&ws.row_count[row], 1u);
        is_last = (prev == (unsigned int)chunks - 1);
    }
    __syncthreads();
    if (!is_last) return;

    // Last CTA of this row: reduce the row's chunk keys.
    __threadfence();
    unsigned long long k = 0ull;
    for (int i = threadIdx.x; i < chunks; i += kThreads)
        k = umax64(k, __ldcg(&ws.keys[(size_t)row * chunks + i]));
    k = block_max(k, red);
    if (threadIdx.x < 32) {  // warp 0 finishes the row, and the request when it is the last row
        const int b = row / T;
        unsigned int prev = 0;
        if (threadIdx.x == 0) {
            target[row] = (int)(0xffffffffu - (unsigned int)(k & 0xffffffffull));
            ws.row_count[row] = 0u;
            __threadfence();
            prev = atomicAdd(&ws.req_count[b], 1u);
        }
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == (unsigned int)T - 1) {
            // Last row of request b: every target of b is written and visible. The
            // accepted length is the first mismatch, found 32 positions per step.
            __threadfence();
            int a = T;
            for (int t0 = 0; t0 < T && a == T; t0 += 32) {
                const int t = t0 + (int)threadIdx.x;
                const bool miss = t < T && __ldcg(&draft[b * T + t]) != __ldcg(&target[b * T + t]);
                const unsigned m = __ballot_sync(0xffffffffu, miss);
                if (m) a = t0 + __ffs(m) - 1;
            }
            if (threadIdx.x == 0) {
                accepted[b] = a;
                ws.req_count[b] = 0u;
            }
        }
    }
}

template <typename E, bool FLAT>
void launch_accept_as(int B, int T, int V, const void *logits, const int32_t *draft, int32_t *target,
                      int32_t *accepted, const AcceptWorkspace &ws, cudaStream_t st) {
    const int chunks = accept_chunks(V);
    const unsigned grid = (unsigned)((long long)B * T * chunks);
    launch_pdl(accept_greedy_kernel<E, FLAT>, dim3(grid), dim3(kThreads), 0, st, B, T, V, chunks,
               static_cast<const E *>(logits), draft, target, accepted, ws);
}

void launch_accept(int B, int T, int V, dn_dtype logit_dt, const void *logits, const int32_t *draft,
                   int32_t *target, int32_t *accepted, const AcceptWorkspace &ws, cudaStream_t st) {
    const bool flat = B * T <= kFlatRows;
    if (logit_dt == DN_F16) {
        if (flat) launch_accept_as<unsigned short, true>(B, T, V, logits, draft, target, accepted, ws, st);
        else launch_accept_as<unsigned short, false>(B, T, V, logits, draft, target, accepted, ws, st);
    } else {
        if (flat) launch_accept_as<unsigned int, true>(B, T, V, logits, draft, target, accepted, ws, st);
        else launch_accept_as<unsigned int, false>(B, T, V, logits, draft, target, accepted, ws, st);
    }
}

}  // namespace
}  // namespace dn

extern "C" size_t dn_accept_workspace_bytes(int B, int T, int V) {
    if (B < 1 || T < 1 || V < 1) return 0;
    return dn::accept_ws_bytes(B, T, V);
}

extern "C" dn_status dn_accept_greedy(int B, int T, int V, dn_dtype logit_dt, const void *logits,
                                      const int32_t *draft_ids, int32_t *target_ids,
                                      int32_t *accepted_len, void *workspace,
                                      size_t workspace_bytes, dn_stream_t stream) {
    using namespace dn;
    if (B < 0 || T < 1 || V < 1 || !dtype_ok(logit_dt)) return DN_ERR_INVALID_ARG;
    if (!accept_grid_ok(B, T, V)) return DN_ERR_INVALID_ARG;
    if (B == 0) return DN_OK;
    if (!logits || !draft_ids || !target_ids || !accepted_len || !workspace) return DN_ERR_INVALID_ARG;
    if (!aligned(logits, 16) || !aligned(draft_ids, 4) || !aligned(target_ids, 4) ||
        !aligned(accepted_len, 4) || !aligned(workspace, 16))
        return DN_ERR_INVALID_ARG;
    if (workspace_bytes < accept_ws_bytes(B, T, V)) return DN_ERR_INVALID_ARG;
    const AcceptWorkspace ws = accept_ws(workspace, B, T, V);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    launch_accept(B, T, V, logit_dt, logits, draft_ids, target_ids, accepted_len, ws, st);
    return launch_status();
}

// ---------------------------------------------------------------------------------------
// dn_accept_greedy_noalloc: the same kernel with its scratch in a fixed device array, for
// callers that cannot allocate device memory where they verify (see include/dn.h).
namespace dn {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DN_ACCEPT_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch. In host code the array's name is only a host-side
// stand-in; the kernel must be given the address the runtime reports, and that address
// belongs to one CUDA context: a device reset, or a second context on the same device,
// loads the module again and may place the array elsewhere. So the address is looked up
// once per context and cached under the context's unique id (cuCtxGetId, never reused
// within a process), not under the device ordinal.
typedef CUresult (*PFN_ctx_get_current)(CUcontext *);
typedef CUresult (*PFN_ctx_get_id)(CUcontext, unsigned long long *);

struct NoallocSlot {
    unsigned long long ctx_id;
    void *addr;
};
constexpr int kNoallocSlots = 64;
std::mutex g_noalloc_mu;
NoallocSlot g_noalloc_slots[kNoallocSlots] = {};
int g_noalloc_next = 0;

template <typename F>
F driver_fn(const char *name) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return reinterpret_cast<F>(p);
}

// Unique id of the calling thread's current context, or 0 when it has none yet.
dn_status current_ctx_id(unsigned long long *id) {
    static const PFN_ctx_get_current get_current = driver_fn<PFN_ctx_get_current>("cuCtxGetCurrent");
    static const PFN_ctx_get_id get_id = driver_fn<PFN_ctx_get_id>("cuCtxGetId");
    if (!get_current || !get_id) return DN_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return DN_ERR_CUDA;
    *id = 0;
    if (ctx != nullptr && get_id(ctx, id) != CUDA_SUCCESS) return DN_ERR_CUDA;
    return DN_OK;
}

dn_status noalloc_scratch_address(void **out) {
    unsigned long long id = 0;
    if (current_ctx_id(&id) != DN_OK) return DN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (id != 0)
        for (const NoallocSlot &sl : g_noalloc_slots)
            if (sl.addr != nullptr && sl.ctx_id == id) {
                *out = sl.addr;
                return DN_OK;
            }
    // First call in this context (the lookup also creates the current device's primary
    // context if the thread had none, so the id is read again after it).
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return DN_ERR_CUDA;
    }
    if (id == 0 && (current_ctx_id(&id) != DN_OK || id == 0)) return DN_ERR_CUDA;
    g_noalloc_slots[g_noalloc_next] = NoallocSlot{id, p};
    g_noalloc_next = (g_noalloc_next + 1) % kNoallocSlots;
    *out = p;
    return DN_OK;
}

}  // namespace
}  // namespace dn

extern "C" dn_status dn_accept_greedy_noalloc(int B, int T, int V, dn_dtype logit_dt,
                                              const void *logits, const int32_t *draft_ids,
                                              int32_t *target_ids, int32_t *accepted_len,
                                              dn_stream_t stream) {
    using namespace dn;
    if (B < 0 || T < 1 || V < 1 || !dtype_ok(logit_dt)) return DN_ERR_INVALID_ARG;
    if (!accept_grid_ok(B, T, V)) return DN_ERR_INVALID_ARG;
    if (B == 0) return DN_OK;
    if (!logits || !draft_ids || !target_ids || !accepted_len) return DN_ERR_INVALID_ARG;
    if (!aligned(logits, 16) || !aligned(draft_ids, 4) || !aligned(target_ids, 4) ||
        !aligned(accepted_len, 4))
        return DN_ERR_INVALID_ARG;
    const size_t need = accept_ws_bytes(B, T, V);
    if (need > DN_ACCEPT_NOALLOC_SCRATCH_BYTES) return DN_ERR_INVALID_ARG;
    void *scratch = nullptr;
    const dn_status st_addr = noalloc_scratch_address(&scratch);
    if (st_addr != DN_OK) return st_addr;
    const AcceptWorkspace ws = accept_ws(scratch, B, T, V);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // The counters must start at zero; the chunk keys are always written before read.
    const size_t counters = static_cast<size_t>(
        static_cast<char *>(scratch) + need - reinterpret_cast<char *>(ws.row_count));
    if (cudaMemsetAsync(ws.row_count, 0, counters, st) != cudaSuccess) {
        cudaGetLastError();
        return DN_ERR_CUDA;
    }
    launch_accept(B, T, V, logit_dt, logits, draft_ids, target_ids, accepted_len, ws, st);
    return launch_status();
}
