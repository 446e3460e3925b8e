// spec_topk: top-k logits of each row in the greedy order (larger value
// first, lower index among equals, NaN above every number), for draft-side
// tree construction (lucebox PR #533, Changes: draft top-K runs on the GPU's
// logits; DDTree expands the draft's top candidates).
//
// One launch, grid (splits, rows):
//  * Each warp scans a contiguous slice of its CTA's chunk with float4 loads
//    and keeps its top-k as one 64-bit greedy key per lane (lane i = i-th
//    largest). A ballot against the current k-th key rejects almost every
//    element; each survivor is inserted with one shuffle-shift.
//  * The 8 warp lists merge in shared memory into the CTA's top-k, stored
//    in the caller's workspace; a per-row ticket (threadfence + atomic, no
//    waiting) lets the last CTA of the row merge the chunks and write the
//    indices and values, then reset the keys it read and the ticket to zero.
#include <cuda_runtime.h>

#include "gdn_device.cuh"
#include "gdn_host.h"
#include "gdnspec.h"

namespace {

using gdndev::key_index;
using gdndev::make_key;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSplits = 64;
constexpr size_t counter_bytes(int32_t rows) { return (((size_t)rows * 4 + 255) / 256) * 256; }

// Insert candidate c into the warp's sorted list (lane i holds the i-th
// largest of k; lanes >= k hold 0). Keys are distinct.
__device__ __forceinline__ void list_insert(unsigned long long &list, unsigned long long c, int k, int lane) {
    const unsigned pos = __popc(__ballot_sync(0xffffffffu, lane < k && list > c));
    if (pos >= (unsigned)k) return;
    const unsigned long long up = __shfl_up_sync(0xffffffffu, list, 1);
    if (lane == (int)pos) list = c;
    else if (lane > (int)pos && lane < k) list = up;
}

// Offer one candidate per lane (0 = none) to the warp's list.
__device__ __forceinline__ void offer(unsigned long long &list, unsigned long long cand, int k, int lane) {
    const unsigned long long kth = __shfl_sync(0xffffffffu, list, k - 1);
    unsigned m = __ballot_sync(0xffffffffu, cand > kth);
    while (m) {
        const int src = __ffs(m) - 1;
        m &= m - 1;
        list_insert(list, __shfl_sync(0xffffffffu, cand, src), k, lane);
    }
}

__global__ void __launch_bounds__(kThreads)
spec_topk_kernel(int V, int k, int splits, int chunk, const float *__restrict__ logits, int32_t *idx_out,
                 float *val_out, unsigned *counters, unsigned long long *keys, int32_t *dev_status) {
    __shared__ unsigned long long lists[kWarps][GDN_MAX_TOPK];
    __shared__ bool is_last;
    const int split = blockIdx.x, row = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *r = logits + (size_t)row * V;
    const int lo = split * chunk, hi = min(V, lo + chunk);
    // buffer extents, for the bounds checks of debug builds (GDN_IN)
    const size_t rows = gridDim.y;
    const gdndev::Buf bl{logits, rows * V * 4}, bi{idx_out, rows * k * 4}, bv{val_out, rows * k * 4},
        bc{counters, rows * 4}, bk{keys, rows * splits * k * 8};
    gdndev::pdl_wait();

    unsigned long long list = 0ull;
    if ((V & 3) == 0) {
        // warp w scans float4 indices [a, b) of the chunk
        const int lo4 = lo >> 2, hi4 = hi >> 2, per = (hi4 - lo4 + kWarps - 1) / kWarps;
        const int a = lo4 + warp * per, b = min(hi4, a + per);
        const float4 *r4 = reinterpret_cast<const float4 *>(r);
        for (int base = a; base < b; base += 32) {
            const int i = base + lane;
            float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < b && GDN_IN(r4 + i, 16, bl, dev_status)) f = __ldcs(r4 + i);
            const unsigned e = (unsigned)i * 4u;
            offer(list, i < b ? make_key(f.x, e) : 0ull, k, lane);
            offer(list, i < b ? make_key(f.y, e + 1) : 0ull, k, lane);
            offer(list, i < b ? make_key(f.z, e + 2) : 0ull, k, lane);
            offer(list, i < b ? make_key(f.w, e + 3) : 0ull, k, lane);
        }
    } else {
        const int per = (hi - lo + kWarps - 1) / kWarps;
        const int a = lo + warp * per, b = min(hi, a + per);
        for (int base = a; base < b; base += 32) {
            const int i = base + lane;
            offer(list, i < b ? make_key(GDN_IN(r + i, 4, bl, dev_status) ? __ldcs(r + i) : 0.f, (unsigned)i) : 0ull,
                  k, lane);
        }
    }
    if (lane < k) lists[warp][lane] = list;
    __syncthreads();
    if (warp == 0) {
        list = lane < k ? lists[0][lane] : 0ull;
        for (int w = 1; w < kWarps; ++w) offer(list, lane < k ? lists[w][lane] : 0ull, k, lane);
        if (lane < k && GDN_IN(keys + ((size_t)row * splits + split) * k + lane, 8, bk, dev_status))
            keys[((size_t)row * splits + split) * k + lane] = list;
        __threadfence();
        unsigned prev = 0;
        const bool cin = GDN_IN(counters + row, 4, bc, dev_status);
        if (lane == 0 && cin) prev = atomicAdd(&counters[row], 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (lane == 0) is_last = cin && prev == (unsigned)(splits - 1);
    }
    __syncthreads();
    if (!is_last || warp != 0) return;
    __threadfence();
    // last CTA of the row: merge the chunks' lists
    list = 0ull;
    unsigned long long *kr = keys + (size_t)row * splits * k;
    for (int base = 0; base < splits * k; base += 32) {
        const int i = base + lane;
        unsigned long long c = 0ull;
        if (i < splits * k && GDN_IN(kr + i, 8, bk, dev_status)) {
            c = __ldcg(kr + i);
            kr[i] = 0ull;  // leave the workspace zero-filled
        }
        offer(list, c, k, lane);
    }
    if (lane < k) {
        const unsigned ix = key_index(list);
        if (GDN_IN(idx_out + (size_t)row * k + lane, 4, bi, dev_status)) idx_out[(size_t)row * k + lane] = (int32_t)ix;
        if (GDN_IN(val_out + (size_t)row * k + lane, 4, bv, dev_status))
            val_out[(size_t)row * k + lane] = GDN_IN(r + ix, 4, bl, dev_status) ? r[ix] : 0.f;
        if ((unsigned)(list >> 32) == 0xFFFFFFFFu && dev_status) atomicOr(dev_status, GDN_DEV_NAN_LOGIT);
    }
    if (lane == 0 && GDN_IN(counters + row, 4, bc, dev_status)) counters[row] = 0u;  // leave the workspace zero-filled
}

int topk_splits(int rows, int V) {
    const int sms = gdnhost::sm_count();
    const int target = 4 * (sms > 0 ? sms : 152);
    int s = (target + rows - 1) / rows;
    const int by_size = (V + 2047) / 2048;
    if (s > by_size) s = by_size;
    if (s > kMaxSplits) s = kMaxSplits;
    if (s < 1) s = 1;
    return s;
}

}  // namespace

extern "C" size_t spec_topk_workspace_bytes(int32_t rows, int32_t k) {
    if (rows < 1 || rows > 65535 || k < 1 || k > GDN_MAX_TOPK) return 0;
    return counter_bytes(rows) + (size_t)rows * kMaxSplits * k * sizeof(unsigned long long);
}

extern "C" int spec_topk(int32_t rows, int32_t vocab, int32_t k, const float *logits, int32_t *idx_out,
                         float *val_out, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                         gdn_stream_t stream) {
    if (rows < 1 || rows > 65535 || k < 1 || k > GDN_MAX_TOPK || vocab < k) return GDN_ERR_DIMS;
    if (!logits || !idx_out || !val_out) return GDN_ERR_NULL;
    using gdnhost::aligned_to;
    if (!aligned_to(logits, 16) || !aligned_to(idx_out, 4) || !aligned_to(val_out, 4) ||
        (dev_status && !aligned_to(dev_status, 4)))
        return GDN_ERR_ALIGN;
    const size_t need = spec_topk_workspace_bytes(rows, k);
    if (!workspace || workspace_bytes < need || !aligned_to(workspace, 256)) return GDN_ERR_WORKSPACE;
    const int splits = topk_splits(rows, vocab);
    int chunk = (vocab + splits - 1) / splits;
    chunk = (chunk + 3) & ~3;
    unsigned *counters = static_cast<unsigned *>(workspace);
    unsigned long long *keys =
        reinterpret_cast<unsigned long long *>(static_cast<char *>(workspace) + counter_bytes(rows));
    dim3 grid(splits, rows);
    spec_topk_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        vocab, k, splits, chunk, logits, idx_out, val_out, counters, keys, dev_status);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
