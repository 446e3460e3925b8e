// Small device helpers of the gdnspec kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "gdnspec.h"

namespace gdndev {

// A global buffer: its base and its size in bytes.
struct Buf {
    const void *base;
    size_t bytes;
};

// Debug builds (compiled with GDN_DEBUG_BOUNDS) check every global access of
// the kernels against the extent of its buffer first: an access of n bytes
// at ptr that would not lie inside the buffer is skipped and GDN_DEV_BOUNDS
// is OR-ed into the status word (when the caller passed one). There is no
// trap. Release builds compile the checks away: GDN_IN is `true` there and
// its arguments are never evaluated.
#ifdef GDN_DEBUG_BOUNDS
__device__ __forceinline__ bool in_buf(const void *ptr, size_t n, Buf b, int32_t *status) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(ptr), lo = reinterpret_cast<uintptr_t>(b.base);
    const bool ok = b.base != nullptr && a >= lo && n <= b.bytes && a - lo <= b.bytes - n;
    if (!ok && status) atomicOr(status, GDN_DEV_BOUNDS);
    return ok;
}
#define GDN_IN(ptr, nbytes, buf, status) (::gdndev::in_buf((ptr), (nbytes), (buf), (status)))
#else
#define GDN_IN(ptr, nbytes, buf, status) true
#endif

// Programmatic dependent launch. pdl_wait(): wait until the kernels this
// grid depends on (the previous work on the stream) have completed and their
// writes are visible; returns at once for a grid launched without the
// attribute. Every kernel of this library calls it before its first global
// memory access. pdl_launch_dependents(): let the grid launched after this
// one be scheduled now (it still waits for this grid's completion).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kern` with programmatic stream serialization, so that its launch
// and scheduling overlap the tail of the previous kernel on the stream
// (which pdl_wait() in `kern` then waits for).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Fill L2 with the 128-byte lines of [base, base + bytes), the lines spread
// over the group's threads. A prefetch only fills L2, the point of
// coherence, and has no effect on what any load later returns.
__device__ __forceinline__ void prefetch_l2_range(const void *base, size_t bytes, int tid, int nthreads) {
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(base) + bytes;
    for (uintptr_t a = (reinterpret_cast<uintptr_t>(base) & ~uintptr_t(127)) + (uintptr_t)tid * 128u; a < a1;
         a += (uintptr_t)nthreads * 128u)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// The same with the L2 evict-last priority, for data that must survive a
// stream of writes until it is read; the reader hands the lines back with
// l2_normal_range() so that nothing stays ahead of other data.
__device__ __forceinline__ void prefetch_l2_keep_range(const void *base, size_t bytes, int tid, int nthreads) {
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(base) + bytes;
    for (uintptr_t a = (reinterpret_cast<uintptr_t>(base) & ~uintptr_t(127)) + (uintptr_t)tid * 128u; a < a1;
         a += (uintptr_t)nthreads * 128u)
        asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(a));
}

__device__ __forceinline__ void l2_normal_range(const void *base, size_t bytes, int tid, int nthreads) {
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(base) + bytes;
    for (uintptr_t a = (reinterpret_cast<uintptr_t>(base) & ~uintptr_t(127)) + (uintptr_t)tid * 128u; a < a1;
         a += (uintptr_t)nthreads * 128u)
        asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(a));
}

// Load element i of an input array stored as bf16 or f32, widened to f32
// (bf16 -> f32 is exact).
template <bool BF16>
__device__ __forceinline__ float ld_in(const void *p, size_t i) {
    if constexpr (BF16) {
        return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
    } else {
        return reinterpret_cast<const float *>(p)[i];
    }
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

__device__ __forceinline__ void st4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

// Checked accesses: GDN_IN first in debug builds (an access outside the
// buffer is skipped; a load then returns zero), plain accesses in release
// builds (the buffer arguments are pure arithmetic the compiler drops).
__device__ __forceinline__ float4 ld4c(const float *p, Buf b, int32_t *st) {
    return GDN_IN(p, 16, b, st) ? ld4(p) : make_float4(0.f, 0.f, 0.f, 0.f);
}
__device__ __forceinline__ void st4c(float *p, float4 v, Buf b, int32_t *st) {
    if (GDN_IN(p, 16, b, st)) st4(p, v);
}
__device__ __forceinline__ float ldfc(const float *p, Buf b, int32_t *st) { return GDN_IN(p, 4, b, st) ? *p : 0.f; }
__device__ __forceinline__ void stfc(float *p, float v, Buf b, int32_t *st) {
    if (GDN_IN(p, 4, b, st)) *p = v;
}
__device__ __forceinline__ int ldic(const int32_t *p, Buf b, int32_t *st) { return GDN_IN(p, 4, b, st) ? *p : 0; }
template <bool BF16>
__device__ __forceinline__ float ld_inc(const void *base, size_t i, Buf b, int32_t *st) {
    return GDN_IN(static_cast<const char *>(base) + i * (BF16 ? 2 : 4), BF16 ? 2 : 4, b, st) ? ld_in<BF16>(base, i)
                                                                                             : 0.f;
}

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
    acc = fmaf(a.z, b.z, acc);
    acc = fmaf(a.w, b.w, acc);
    return acc;
}

// SiLU(y) = y / (1 + e^-y) with the fast exponential and division
// intrinsics (a few ulp each, far inside the 2e-3 tolerance of the states
// and outputs). Large -y gives e^-y = inf and a zero quotient, the limit.
__device__ __forceinline__ float silu(float y) { return __fdividef(y, 1.0f + __expf(-y)); }

// Greedy-order key of logit f at index idx: the order-preserving bits of the
// value in the high word (every NaN maps to the top, -0.0 is folded into
// +0.0) and ~idx in the low word, so a larger key is a larger value or, among
// equal values, a lower index. Every real key is > 0.
__device__ __forceinline__ unsigned long long make_key(float f, unsigned idx) {
    unsigned u = __float_as_uint(f);
    unsigned ord;
    if (f != f) {
        ord = 0xFFFFFFFFu;
    } else {
        if (u == 0x80000000u) u = 0u;  // -0.0 == +0.0
        ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    }
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - idx);
}

__device__ __forceinline__ unsigned key_index(unsigned long long key) {
    return 0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull);
}

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
    return a > b ? a : b;
}

}  // namespace gdndev
