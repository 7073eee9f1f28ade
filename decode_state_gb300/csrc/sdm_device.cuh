// Device helpers shared by the SDM kernels: bf16 conversion, element access, and inline PTX for
// bulk stores (cp.async.bulk shared->global), the async-proxy fence they need, and programmatic
// dependent launch.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sdm {

// ---------------------------------------------------------------- element types
// bf16 travels as uint16_t bits; float32 as float.

__device__ __forceinline__ float to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }
__device__ __forceinline__ float to_f32(float x) { return x; }

template <typename E>
__device__ __forceinline__ E from_f32(float x);
template <>
__device__ __forceinline__ uint16_t from_f32<uint16_t>(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));  // round to nearest even
}
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }

// x rounded to the bank dtype E and widened back to float32
template <typename E>
__device__ __forceinline__ float round_to(float x) { return to_f32(from_f32<E>(x)); }

template <typename I>
__device__ __forceinline__ int64_t load_index(const void* p, int64_t i) {
    return (int64_t)__ldg(static_cast<const I*>(p) + i);
}

// ---------------------------------------------------------------- shared-memory addresses

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// ---------------------------------------------------------------- L2 eviction policy

// A cache policy that marks every line it touches evict-first in L2: for output that this launch
// never reads again (readings, stash rows, written-back rows that a later token rarely names).
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// A 4-byte global store under an L2 cache policy.
__device__ __forceinline__ void st_hint(float* p, float v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;" ::"l"(p), "r"(__float_as_uint(v)), "l"(pol) : "memory");
}

// A 16-byte global store of four floats under an L2 cache policy.
__device__ __forceinline__ void st_hint4(void* p, float a, float b, float c, float d, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d), "l"(pol)
                 : "memory");
}

// ---------------------------------------------------------------- bulk stores (async proxy)

// shared -> global, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}

// the same, with the destination lines marked by an L2 cache policy
__device__ __forceinline__ void bulk_s2g_hint(void* dst, const void* src, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// wait until every committed bulk store of this thread has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Order this thread's earlier generic-proxy shared writes before later async-proxy accesses.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels are launched with programmatic stream serialization: a launch may start while the
// previous kernel on the stream finishes. Every kernel calls grid_dependency_wait() before its
// first global-memory access, which returns once the previous grid has completed and its writes
// are visible (at once when there is no such grid), so results never depend on the overlap.

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the next kernel on the stream be scheduled now (its blocks then wait in grid_dependency_wait).
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace sdm
