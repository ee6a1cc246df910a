// pkv_device.cuh -- device-side building blocks shared by the sm_103a kernels:
// mbarrier pipeline primitives with bounded waits, TMA tile loads, 1-D bulk
// copies, 16-byte cp.async, 16-bit float unpacking and the device error word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// A bounded wait gives up after this many nanoseconds of %globaltimer, sets
// PKV_DEVERR_TIMEOUT and lets the kernel finish instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

// atomicAdd at gpu scope with acquire-release semantics: the writes that
// precede it (this thread's, and those ordered before it by a CTA barrier) are
// visible to whoever observes the new count, and the writes released by earlier
// adders are visible to this thread afterwards.  One operation instead of a
// sequentially consistent fence on each side of a relaxed add (measured ~0.7 us
// less per publication under a full DRAM stream).
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* addr, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test, letting the hardware suspend the thread for up to ns
// nanoseconds until the phase completes (one instruction per wait instead of a
// spin of tests that takes issue slots from the warps that have work).
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, "
        "p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}

// Longest single suspension of a bounded wait (the timer is checked between them).
constexpr uint32_t kWaitSuspendNs = 1u << 20;

// Wait for the phase with the given parity to complete.  Returns false (and
// the caller flags PKV_DEVERR_TIMEOUT) if it has not after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    const uint32_t a = smem_addr(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait_suspend(a, parity, kWaitSuspendNs)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// ---------------------------------------------------------------- programmatic dependent launch

// Wait until every grid this launch programmatically depends on has completed
// and its writes are visible.  Returns at once for a launch without such a
// dependency.  Every kernel here calls it before its first global write and
// before reading anything a kernel of this library writes.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the next kernel of the stream be scheduled now; it still runs its own
// grid_dep_wait() before touching memory this grid writes.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- TMA / bulk copies

// L2 policy for data read once: its lines are the first evicted, so a stream
// of them leaves the small inputs (block tables, lengths, queries) and the
// partials cached in L2 from one launch to the next.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`, with
// an L2 cache policy (see l2_evict_first_policy).  x (innermost coordinate)
// must be a multiple of 16 bytes / element size.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

// 3-D tiled TMA load (coordinates innermost first), the same way.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, int32_t x, int32_t y, int32_t z,
                                                 uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, "
        "{%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar)), "l"(pol)
        : "memory");
}

// 16-byte global -> shared copy through the load/store path (not the TMA engine).
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}

// The same copy with an L2 cache policy (see l2_evict_first_policy).
__device__ __forceinline__ void cp_async_16_hint(void* dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
                 "l"(pol)
                 : "memory");
}

// 16-byte shared-memory copy by explicit shared addresses.
__device__ __forceinline__ void lds_sts_16(uint32_t dst, uint32_t src) {
    asm volatile(
        "{\n\t.reg .b32 a, b, c, d;\n\tld.shared.v4.b32 {a, b, c, d}, [%1];\n\tst.shared.v4.b32 [%0], {a, b, c, d};\n\t}" ::"r"(
            dst),
        "r"(src)
        : "memory");
}

__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void sts_u8(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// 8- and 4-byte global -> shared copies through the load/store path.
__device__ __forceinline__ void cp_async_8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Makes the current phase of `bar` also wait for every cp.async this thread has
// issued so far: the pending arrival count goes up by one now and comes back
// down when those copies have landed.  Call it before this thread's own arrive
// on the phase, so the phase cannot complete in between.
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Named barrier over a subset of the CTA's warps (id 1.., `threads` a multiple of 32).
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------- 16-bit floats

template <typename T>
struct Half16;

template <>
struct Half16<__nv_bfloat16> {
    // two packed bf16 -> two fp32 (exact: bf16 is the top half of fp32)
    static __device__ __forceinline__ float2 unpack2(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    static __device__ __forceinline__ float to_float(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }
};

template <>
struct Half16<__half> {
    static __device__ __forceinline__ float2 unpack2(uint32_t w) {
        __half2 h;
        memcpy(&h, &w, 4);
        return __half22float2(h);
    }
    static __device__ __forceinline__ float to_float(uint16_t b) {
        __half h;
        memcpy(&h, &b, 2);
        return __half2float(h);
    }
};

__device__ __forceinline__ void store_out(void* out, int dtype, size_t i, float v) {
    if (dtype == PKV_BF16)
        reinterpret_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
    else if (dtype == PKV_F16)
        reinterpret_cast<__half*>(out)[i] = __float2half_rn(v);
    else
        reinterpret_cast<float*>(out)[i] = v;
}

// Four consecutive outputs from element i (a multiple of 4): one 16-byte or 8-byte store.
__device__ __forceinline__ void store_out4(void* out, int dtype, size_t i, float4 v) {
    if (dtype == PKV_F32) {
        reinterpret_cast<float4*>(out)[i >> 2] = v;
    } else if (dtype == PKV_BF16) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
        uint2 w;
        memcpy(&w.x, &a, 4);
        memcpy(&w.y, &b, 4);
        reinterpret_cast<uint2*>(out)[i >> 2] = w;
    } else {
        const __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
        uint2 w;
        memcpy(&w.x, &a, 4);
        memcpy(&w.y, &b, 4);
        reinterpret_cast<uint2*>(out)[i >> 2] = w;
    }
}

__device__ __forceinline__ float load_q(const void* q, int dtype, size_t i) {
    const uint16_t b = reinterpret_cast<const uint16_t*>(q)[i];
    return dtype == PKV_BF16 ? Half16<__nv_bfloat16>::to_float(b) : Half16<__half>::to_float(b);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace pkv
