// ptx.cuh -- small inline-PTX memory helpers shared by the libmoe kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

constexpr unsigned kFull = 0xffffffffu;

// 16-byte load of data read once by this launch: non-coherent path, do not
// allocate in L1 (the rows are streamed, never re-read by the same SM).
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte store.
__device__ __forceinline__ void st16(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// bf16 halves of a 32-bit word -> fp32 (exact widening).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> packed bf16x2, round to nearest even (lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ void set_error(int32_t* err, int bits) { atomicOr(err, bits); }


// Programmatic dependent launch.  Every kernel of the library calls
// grid_dependency_sync() before its first access to memory that the preceding
// kernel may write: it returns once that kernel has completed and its writes
// are visible (immediately if there is none).  Dispatch reads x, which its
// preceding kernel (the plan) never writes, before the call.  allow_dependents() then lets the next
// kernel's CTAs be scheduled while this grid drains; they park in their own
// grid_dependency_sync(), so ordering is unchanged -- only launch latency is
// hidden.
__device__ __forceinline__ void grid_dependency_sync() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Asynchronous 4- and 8-byte copies global -> shared (no register staging);
// complete after cp_async_wait_all() in the issuing thread.
__device__ __forceinline__ void cp_async4(void* smem_dst, const void* gmem_src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem_dst, const void* gmem_src) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Thread-block clusters.  The CTAs of a cluster are scheduled together, so
// the cluster barrier is a hardware barrier like __syncthreads (every thread
// of every CTA of the cluster arrives), not a wait on a flag.  arrive has
// release semantics and wait acquire semantics at cluster scope: shared-memory
// writes before the arrive are visible to every CTA after its wait.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// Arrive without memory ordering: for a thread whose remote shared-memory
// loads have all been consumed (so they have completed) and that publishes
// nothing to the cluster, e.g. to say "done reading your shared memory".
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// 32-bit load from the shared memory of CTA `rank` of this cluster, at the
// address that `local` has in this CTA's shared memory (same layout in every
// CTA of the cluster).
__device__ __forceinline__ uint32_t ld_cluster_shared_u32(const void* local, uint32_t rank) {
    const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t ra, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
    return v;
}

}  // namespace moe
