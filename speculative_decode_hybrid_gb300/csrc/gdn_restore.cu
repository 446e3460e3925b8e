// gdn_rollback_restore: on-device restore of the live SSM and conv state to
// the checkpoint of the accepted node (lucebox PR #533, Changes: restore
// split SSM and convolution state on-device; lucebox PR #506, Summary: fast
// rollback from F32 checkpoints, no replay).
//
// grid (chunks, B*Y), at most one wave of 8 resident CTAs per SM: every CTA
// reads the accepted node of its request from device memory (no host round
// trip), returns at once for node 0 (verify never touched the live state)
// and otherwise copies its share of the 16-byte vectors of slot node-1, 4
// independent loads in flight per thread, then 4 stores. The copy is
// bit-exact.
#include <cuda_runtime.h>

#include "gdn_device.cuh"
#include "gdn_host.h"
#include "gdnspec.h"

namespace {

using gdndev::launch_pdl;
using gdndev::pdl_wait;

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int kCtasPerSm = 8;

// Copy n4 16-byte vectors, this thread taking begin, begin + step, ...
// (32-bit offsets: the host routes slots of 2^31 vectors or more elsewhere).
// bs / bd: the source and destination buffers (bounds checks of debug builds).
__device__ __forceinline__ void copy_range4(const float4 *__restrict__ src, float4 *__restrict__ dst,
                                            unsigned n4, unsigned begin, unsigned step, gdndev::Buf bs,
                                            gdndev::Buf bd, int32_t *st) {
    unsigned i = begin;
    for (; i + (kUnroll - 1) * step < n4; i += kUnroll * step) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            v[u] = GDN_IN(src + i + u * step, 16, bs, st) ? __ldcs(src + i + u * step) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (GDN_IN(dst + i + u * step, 16, bd, st)) dst[i + u * step] = v[u];
    }
    for (; i < n4; i += step)
        if (GDN_IN(src + i, 16, bs, st) && GDN_IN(dst + i, 16, bd, st)) dst[i] = __ldcs(src + i);
}

__global__ void __launch_bounds__(kThreads, kCtasPerSm)
gdn_restore_kernel(int Y, int T, size_t ssm_slot, size_t conv_slot, const int32_t *__restrict__ accept_node,
                   const float *__restrict__ ssm_ckpt, const float *__restrict__ conv_ckpt,
                   float *__restrict__ ssm_state, float *__restrict__ conv_state, int32_t *dev_status) {
    const int by = blockIdx.y;
    const int b = by / Y;
    // buffer extents, for the bounds checks of debug builds (GDN_IN)
    const size_t rows = gridDim.y;
    const gdndev::Buf bsc{ssm_ckpt, rows * T * ssm_slot * 4}, bss{ssm_state, rows * ssm_slot * 4},
        bcc{conv_ckpt, rows * T * conv_slot * 4}, bcs{conv_state, rows * conv_slot * 4},
        bn{accept_node, rows / Y * 4};
    pdl_wait();  // accept_node and the checkpoints come from the kernels before
    const int node = gdndev::ldic(accept_node + b, bn, dev_status);
    if (node == 0) return;
    if (node < 0 || node > T) {
        if (dev_status && blockIdx.x == 0 && by % Y == 0 && threadIdx.x == 0)
            atomicOr(dev_status, GDN_DEV_NODE_RANGE);
        return;
    }
    const unsigned begin = blockIdx.x * kThreads + threadIdx.x;
    const unsigned step = gridDim.x * kThreads;
    {
        const float4 *src = reinterpret_cast<const float4 *>(ssm_ckpt + ((size_t)by * T + (node - 1)) * ssm_slot);
        float4 *dst = reinterpret_cast<float4 *>(ssm_state + (size_t)by * ssm_slot);
        copy_range4(src, dst, (unsigned)(ssm_slot / 4), begin, step, bsc, bss, dev_status);
    }
    if (conv_slot > 0) {
        const float *src = conv_ckpt + ((size_t)by * T + (node - 1)) * conv_slot;
        float *dst = conv_state + (size_t)by * conv_slot;
        if ((conv_slot & 3) == 0) {
            copy_range4(reinterpret_cast<const float4 *>(src), reinterpret_cast<float4 *>(dst),
                        (unsigned)(conv_slot / 4), begin, step, bcc, bcs, dev_status);
        } else {
            for (unsigned i = begin; i < conv_slot; i += step)
                if (GDN_IN(src + i, 4, bcc, dev_status) && GDN_IN(dst + i, 4, bcs, dev_status)) dst[i] = src[i];
        }
    }
}

}  // namespace

extern "C" int gdn_rollback_restore(const gdn_dims *d, int32_t n_tok, const int32_t *accept_node_dev,
                                    const float *ssm_ckpt, const float *conv_ckpt, float *ssm_state,
                                    float *conv_state, int32_t *dev_status, gdn_stream_t stream) {
    int rc = gdnhost::check_dims(d, n_tok);
    if (rc != GDN_OK) return rc;
    if (!accept_node_dev || !ssm_ckpt || !ssm_state) return GDN_ERR_NULL;
    if (d->conv_k > 1 && (!conv_ckpt || !conv_state)) return GDN_ERR_NULL;
    using gdnhost::aligned16;
    using gdnhost::aligned_to;
    if (!aligned16(ssm_ckpt) || !aligned16(ssm_state) || !aligned_to(accept_node_dev, 4) ||
        (dev_status && !aligned_to(dev_status, 4)))
        return GDN_ERR_ALIGN;
    if (d->conv_k > 1 && (!aligned16(conv_ckpt) || !aligned16(conv_state))) return GDN_ERR_ALIGN;

    const size_t ssm_slot = gdnhost::ssm_slot_elems(d);
    const size_t conv_slot = gdnhost::conv_slot_elems(d);
    if (ssm_slot >= (1ull << 31) || conv_slot >= (1ull << 31)) return GDN_ERR_DIMS;
    const int rows = d->batch * d->layers;
    const int sms = gdnhost::sm_count();
    const int target = kCtasPerSm * (sms > 0 ? sms : 152);
    int chunks = target / rows;  // one wave: a second, partial wave would run after the first
    const size_t per_cta_min = (size_t)kThreads * kUnroll;  // float4 per CTA, at least one full round
    const size_t max_chunks = (ssm_slot / 4 + per_cta_min - 1) / per_cta_min;
    if ((size_t)chunks > max_chunks) chunks = (int)max_chunks;
    if (chunks < 1) chunks = 1;
    dim3 grid(chunks, rows);
    return launch_pdl(gdn_restore_kernel, grid, dim3(kThreads), 0, static_cast<cudaStream_t>(stream), d->layers,
                      n_tok, ssm_slot, conv_slot, accept_node_dev, ssm_ckpt, conv_ckpt, ssm_state, conv_state,
                      dev_status) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}
