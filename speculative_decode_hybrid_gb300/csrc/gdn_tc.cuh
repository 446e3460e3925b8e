// tcgen05 (5th-generation tensor core) helpers for sm_100-family GPUs:
// tensor memory allocation, shared-memory operand descriptors, kind::tf32
// MMA with the accumulator in tensor memory, completion through an mbarrier,
// and tensor-memory loads/stores. Inline PTX only.
//
// Operand layout: K-major tiles in shared memory with the 128-byte swizzle.
// A tile of `rows` rows keeps each row's K elements in 128-byte chunks: chunk
// c of all rows is one block of rows * 128 bytes, row r at r * 128 in it,
// and 16-byte unit u of the chunk at ((u ^ (r % 8)) * 16). The block base
// must be 1024-byte aligned, so that the hardware's swizzle (address bits
// [4,7) XOR bits [7,10)) is this one. One MMA step consumes K = 8 tf32
// (32 bytes) of a chunk: its descriptor starts at block + 32 * (step % 4).
#pragma once

#include <cstdint>

namespace gdntc {

// Shared-memory matrix descriptor: start address, leading byte offset
// (unused by swizzled K-major layouts), stride byte offset between 8-row
// groups (8 rows x 128 bytes), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_sw128(unsigned saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::tf32: f32 accumulator, tf32 A and B, both
// K-major, M x N.
__host__ __device__ constexpr unsigned idesc_tf32(unsigned M, unsigned N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// x rounded to tf32 (nearest, ties away from zero), as an f32 whose low 13
// mantissa bits are zero.
__device__ __forceinline__ float tf32_rna(float x) {
    unsigned r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Executed by one full warp: allocate `cols` tensor-memory columns (a power
// of two >= 32); the base address is written to *dst_smem.
template <int kCols>
__device__ __forceinline__ void tmem_alloc(unsigned *dst_smem) {
    static_assert(kCols >= 32 && (kCols & (kCols - 1)) == 0, "tensor memory columns: a power of two >= 32");
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     (unsigned)__cvta_generic_to_shared(dst_smem)),
                 "n"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int kCols>
__device__ __forceinline__ void tmem_dealloc(unsigned taddr) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(kCols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// generic-proxy shared-memory writes -> visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// D (tmem) (+)= A (smem descriptor) x B (smem descriptor)
__device__ __forceinline__ void mma_tf32_ss(unsigned d_tmem, uint64_t a_desc, uint64_t b_desc, unsigned idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// D (tmem) (+)= A (tmem: row i in lane i, K along columns) x B (smem descriptor)
__device__ __forceinline__ void mma_tf32_ts(unsigned d_tmem, unsigned a_tmem, uint64_t b_desc, unsigned idesc,
                                            bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

// The mbarrier at `bar` gets one arrival when every MMA this thread issued
// has completed.
__device__ __forceinline__ void mma_commit(unsigned bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Wait (bounded) for phase `parity` of the mbarrier at `bar`; false if the
// wait gave up.
__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity, unsigned polls) {
    unsigned done = 0;
    for (unsigned i = 0; i < polls && !done; ++i)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.b32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
    return done != 0;
}

// Warp-collective: this thread's lane of the warp's 32 tensor-memory lanes,
// 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_st8(unsigned taddr, const unsigned (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Warp-collective: 8 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_ld8(unsigned taddr, unsigned (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}

// Warp-collective: 32 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(unsigned taddr, unsigned (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace gdntc
