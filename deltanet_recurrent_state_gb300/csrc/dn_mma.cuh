// Warp-level tensor-core helpers shared by the chunkwise (WY) kernels:
// ldmatrix loads of fp16 tiles from shared memory, the m16n8k16 fp16 MMA with fp32
// accumulation, the XOR swizzle of 16-byte chunks that keeps ldmatrix conflict
// free, and packing of fp32 accumulator fragments into fp16 operand fragments.
//
// Fragment layout (per warp, lane L): an m16n8 fp32 accumulator tile holds
// d0, d1 at row L/4, columns 2(L%4), 2(L%4)+1 and d2, d3 at row L/4 + 8. The fp16
// A operand of a 16x16 tile holds a0 = rows 0-7 / cols 0-7, a1 = rows 8-15 / cols
// 0-7, a2 = rows 0-7 / cols 8-15, a3 = rows 8-15 / cols 8-15, each as two fp16
// at the same (row, column-pair) positions as the accumulator, so two adjacent
// accumulator tiles repack into one A operand without leaving registers.
#pragma once

#include <cstdint>

#include <cuda_fp16.h>

namespace dn {

__device__ __forceinline__ void ldsm_x4(unsigned (&r)[4], const void *p) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

__device__ __forceinline__ void ldsm_x2(unsigned (&r)[2], const void *p) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(a));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const unsigned (&a)[4],
                                          const unsigned (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// fp16 tile with CPR 16-byte chunks per row; chunk c of row r lives at c ^ (r & 7),
// so the 8 row addresses of an ldmatrix hit 8 different bank groups.
template <int CPR>
__device__ __forceinline__ int hsw(int r, int c) { return r * CPR + (c ^ (r & 7)); }

__device__ __forceinline__ void ldsm_x4_t(unsigned (&r)[4], const void *p) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(a));
}

// Four 8x8 fp16 matrices from fragment registers to shared memory, transposed: lane L
// gives the address of stored row L % 8 of matrix L / 8, which receives column L % 8
// of that matrix.
__device__ __forceinline__ void stsm_x4_t(void *p, unsigned r0, unsigned r1, unsigned r2, unsigned r3) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(p);
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};"
                 :: "r"(a), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
}

// Four 8x8 fp16 matrices from fragment registers to shared memory, not transposed.
__device__ __forceinline__ void stsm_x4(void *p, unsigned r0, unsigned r1, unsigned r2, unsigned r3) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(p);
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1,%2,%3,%4};"
                 :: "r"(a), "r"(r0), "r"(r1), "r"(r2), "r"(r3) : "memory");
}

// ---- mbarrier and tensor-map (TMA) copies -------------------------------------------

__device__ __forceinline__ void mbar_init(unsigned long long *mb, unsigned count) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(mb);
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(a), "r"(count) : "memory");
}
// One arrival that also announces `bytes` of copies still to land in this phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long *mb, unsigned bytes) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(mb);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(a), "r"(bytes) : "memory");
}
__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// A wait of the prefill kernels gives up after this long (the global timer, in ns): 1 s,
// against waits of a few microseconds when the copies and MMAs they wait for progress.
constexpr unsigned long long kWaitBudgetNs = 1000000000ull;

// Bounded wait for the phase with the given parity by time: false if it did not complete
// within `budget_ns`, or once `*abort` is set by another thread of the CTA (checked every
// 64 polls). On its own timeout the wait raises `*abort` and counts the CTA's failure in
// `*timeouts` once, so every role of the CTA stops issuing work at its next check.
__device__ __forceinline__ bool mbar_wait_guarded(unsigned long long *mb, unsigned parity, volatile int *abort,
                                                  unsigned int *timeouts,
                                                  unsigned long long budget_ns = kWaitBudgetNs) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(mb);
    const unsigned long long t0 = global_timer_ns();
    for (int it = 0;; ++it) {
        unsigned ok;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                     " selp.u32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(a), "r"(parity) : "memory");
        if (ok) return true;
        if ((it & 63) == 63) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > budget_ns) {
                if (atomicExch(const_cast<int *>(abort), 1) == 0 && timeouts) atomicAdd(timeouts, 1u);
                return false;
            }
        }
    }
}

// Drain of a copy this thread issued: waits at most `budget_ns` for the phase, ignoring any
// abort (the copy was issued and lands unless something is broken); true if it landed.
__device__ __forceinline__ bool mbar_drain(unsigned long long *mb, unsigned parity,
                                           unsigned long long budget_ns = kWaitBudgetNs) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(mb);
    const unsigned long long t0 = global_timer_ns();
    for (;;) {
        unsigned ok;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                     " selp.u32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(a), "r"(parity) : "memory");
        if (ok) return true;
        if (global_timer_ns() - t0 > budget_ns) return false;
    }
}

// Contiguous global -> shared copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned), completing on the mbarrier.
__device__ __forceinline__ void bulk_load(void *smem, const void *gmem, unsigned bytes, unsigned long long *mb) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem);
    const unsigned m = (unsigned)__cvta_generic_to_shared(mb);
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(d), "l"(gmem), "r"(bytes), "r"(m) : "memory");
}

// Box of a 4-d tensor map -> shared memory, completing `bytes` on the mbarrier.
__device__ __forceinline__ void tma_load_4d(void *smem, const void *tmap, int c0, int c1, int c2, int c3,
                                            unsigned long long *mb) {
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem);
    const unsigned m = (unsigned)__cvta_generic_to_shared(mb);
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5}], [%6];"
                 :: "r"(d), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(m) : "memory");
}
// Shared memory -> box of a 4-d / 3-d tensor map (elements outside the tensor are skipped).
__device__ __forceinline__ void tma_store_4d(const void *tmap, int c0, int c1, int c2, int c3, const void *smem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];"
                 :: "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(s) : "memory");
}
__device__ __forceinline__ void tma_store_3d(const void *tmap, int c0, int c1, int c2, const void *smem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
                 :: "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(s) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the shared-memory sources of all of this thread's bulk groups have been read.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's generic-proxy shared-memory accesses before later async-proxy ones.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Named barriers (0 is __syncthreads): sync waits for `count` threads, arrive does not wait.
__device__ __forceinline__ void bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" :: "r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ unsigned pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const unsigned *>(&h);
}

__device__ __forceinline__ float2 unpack_h2(unsigned u) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&u));
}

// Two accumulator tiles (columns 0-7 and 8-15 of a 16x16 block) -> one fp16 A operand.
__device__ __forceinline__ void acc_to_a(unsigned (&a)[4], const float (&d0)[4], const float (&d1)[4]) {
    a[0] = pack_h2(d0[0], d0[1]);
    a[1] = pack_h2(d0[2], d0[3]);
    a[2] = pack_h2(d1[0], d1[1]);
    a[3] = pack_h2(d1[2], d1[3]);
}

// cp.async of 16 bytes global -> shared; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem, int src_bytes) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(a), "l"(gmem), "r"(src_bytes)
                 : "memory");
}
// cp.async of 4 bytes global -> shared; src_bytes = 0 writes zero.
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem, int src_bytes) {
    const unsigned a = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" :: "r"(a), "l"(gmem), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

}  // namespace dn
