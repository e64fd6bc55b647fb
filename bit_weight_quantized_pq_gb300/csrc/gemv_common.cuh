// Device helpers shared by the decode GEMVs: cp.async streaming of weight
// chunks into per-warp rings, and the activation rows brought into shared
// memory by one bulk copy that completes on an mbarrier (so that waiting for
// the rows never waits for weight copies issued earlier).
#pragma once

#include "pq_internal.cuh"

namespace pqg {

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool valid) {
    const uint32_t n = valid ? 16u : 0u;   // 0 source bytes: the 16 bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool bar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// One thread: make the rows' mbarrier (arrival count 1) before any use, and
// visible to the bulk-copy (async) proxy.  The CTA synchronises before
// another thread waits on it.
__device__ __forceinline__ void rows_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(bar) : "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One thread: copy `bytes` (a multiple of 16; both addresses 16-byte
// aligned) from global to shared memory in bulk copies of at most 16 KB,
// all completing on `bar`.
__device__ __forceinline__ void rows_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
    const char* s = static_cast<const char*>(src);
    for (uint32_t off = 0; off < bytes; off += 16384u) {
        const uint32_t n = bytes - off < 16384u ? bytes - off : 16384u;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
            :: "r"(dst + off), "l"(s + off), "r"(n), "r"(bar) : "memory");
    }
}

// Every thread of the CTA: wait (at most ~1 s) for the rows.  The result is
// the same in every thread; on a timeout PQ_ERR_DEVICE_TIMEOUT goes to the
// status word, and the caller drains its copies and returns.
__device__ __forceinline__ bool rows_wait(uint32_t bar, uint32_t* status) {
    const uint64_t t0 = gtimer();
    bool ok = false;
    for (uint32_t i = 0;; ++i) {
        if (bar_try(bar, 0)) {
            ok = true;
            break;
        }
        if ((i & 63) == 63 && gtimer() - t0 > 1000000000ull) break;
    }
    if (!ok) atomicCAS(status, 0u, (uint32_t)(int32_t)PQ_ERR_DEVICE_TIMEOUT);
    return __syncthreads_and(ok ? 1 : 0) != 0;
}

// After a failed rows_wait: let the copies in flight land (bounded) before
// the CTA exits.
__device__ __forceinline__ void rows_drain(uint32_t bar) {
    cp_wait<0>();
    const uint64_t t0 = gtimer();
    while (!bar_try(bar, 0) && gtimer() - t0 < 200000000ull) {
    }
}

// Thread-block clusters: this CTA's rank, the barrier in two halves (every
// thread of every CTA of the cluster arrives, then waits), and stores into
// another CTA's shared memory at the address of a local variable.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void dsmem_st_u32(uint32_t a, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st_f2(uint32_t a, float x, float y) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" :: "r"(a), "f"(x), "f"(y) : "memory");
}
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}

}  // namespace pqg
