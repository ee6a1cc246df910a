// pkv_umma.cuh -- hand-written PTX for the 5th-generation tensor cores
// (tcgen05): tensor-memory allocation, the f16 MMA with shared-memory operands,
// its completion on an mbarrier, and tensor-memory loads.
//
// Operands live in shared memory in the 128-byte swizzled layout that a TMA
// copy with CU_TENSOR_MAP_SWIZZLE_128B produces for 16-bit elements: rows of
// 128 bytes (64 elements), the 16-byte chunk c of row r stored at chunk
// position c ^ (r % 8), eight rows (1024 bytes, 1024-byte aligned) forming one
// swizzle atom.  A tile wider than 64 elements is stored as column blocks of
// 64 elements, one after the other (`rows` x 128 bytes each).
//
// A K-major operand (the contraction dimension K contiguous in a row) of R rows
// advances by 32 bytes per 16-element k-step inside a column block and by one
// column block every 4 k-steps; consecutive 8-row atoms are 1024 bytes apart.
// An MN-major operand (rows indexed by K, the M or N index contiguous) takes
// the same storage: 16 K-rows per k-step are two atoms (2048 bytes), and the
// next 64 elements of M / N are the next column block.
#pragma once

#include <cstdint>

namespace pkv {

// Shared-memory matrix descriptor: start address, leading- and stride-byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= uint64_t((saddr >> 4) & 0x3FFFu);
    d |= uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= uint64_t((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= uint64_t(1) << 46;   // version
    d |= uint64_t(2) << 61;   // 128-byte swizzle
    return d;
}

// Instruction descriptor of kind::f16 with f16 A and B, f32 accumulator.
// a_mn / b_mn: the operand is MN-major (else K-major).
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                        // D: f32
           | (0u << 7) | (0u << 10)         // A, B: f16
           | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16)
           | (uint32_t(N >> 3) << 17)
           | (uint32_t(M >> 4) << 24);
}

// Tensor memory: `ncols` columns (a power of two >= 32) for this CTA; the base
// address lands in shared memory at `dst`.  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_saddr, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_saddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void umma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
        : "memory");
}

// Arrive (once) on the mbarrier when every tcgen05 operation this thread issued
// before has completed.
__device__ __forceinline__ void umma_commit(uint32_t mbar_saddr) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar_saddr)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Generic-proxy shared-memory writes made visible to the tensor core's reads.
__device__ __forceinline__ void fence_proxy_async_cta() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 consecutive 32-bit columns of this thread's tensor-memory lane (a warp
// reads the 32 lanes of its quarter: lanes 32 * (warp % 4) + 0..31).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of 16-bit element (r, c) of a swizzled tile of `rows` rows.
__host__ __device__ constexpr uint32_t sw128_off(int r, int c, int rows) {
    return uint32_t((c >> 6) * rows * 128 + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + ((c & 7) << 1));
}

}  // namespace pkv
