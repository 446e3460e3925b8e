// spec_accept_greedy: greedy acceptance of drafted chains / trees against
// the target's argmax, on sm_103a (openinfer PR #626, Summary: the
// speculative output must match plain greedy decoding; lucebox PR #533,
// Changes: top-K/argmax run on the GPU's logits).
//
// One launch:
//  * grid (splits, N, B): each CTA scans a contiguous, 16-byte aligned chunk
//    of one logit row with streaming float4 loads and reduces it to one
//    64-bit key  (order-preserving bits of the value << 32) | (~index),
//    so a plain max picks the largest value and, among equal values, the
//    lowest index; every NaN maps to the top value and the first NaN wins.
//    -0.0 is folded into +0.0 so that equal values tie by index. Before it
//    waits for the previous grid on the stream, the CTA prefetches its chunk
//    into L2 with the evict-last priority (a prefetch only fills L2; the
//    CTAs of this launch are resident well before that grid ends, which
//    streams its writes until then) and sets it back to normal once read.
//  * The CTA folds its key into its row's key in the caller's workspace
//    (a 64-bit atomic max in L2) and bumps a per-request arrival counter.
//    The last CTA of a request (an acquire-release atomic counter, no spinning)
//    reads the N row keys (one thread each), writes argmax_out, and decides
//    the acceptance in parallel: a chain's accepted length is the number of
//    leading matches (a warp ballot of the mismatches); a tree's nodes find
//    their depth and whether their whole root path matches by walking to
//    the root, one thread per node, and one thread picks the deepest
//    matching node. It then puts the row keys and the counter back to zero
//    (so a later call of any shape finds a zero-filled workspace).
#include <cuda_runtime.h>

#include <mutex>

#include "gdn_device.cuh"
#include "gdn_host.h"
#include "gdnspec.h"

namespace {

constexpr int kThreads = 256;
constexpr int kMaxSplits = 64;
constexpr int kLoads = 4;                        // float4 loads in flight per thread
constexpr int kRoundLogits = kThreads * kLoads * 4;  // logits one CTA covers in one round
constexpr int kMaxNodes = GDN_MAX_TOKENS + 1;
static_assert(kMaxNodes <= kThreads, "one thread per node");
constexpr int kBallotWarps = (kMaxNodes + 31) / 32;  // warps that cover the nodes of a chain
constexpr size_t kCounterBytes(int32_t batch) { return (((size_t)batch * 4 + 255) / 256) * 256; }

using gdndev::make_key;
using gdndev::umax64;

// Among two distinct matching nodes of equal depth: is i's root path lower
// than j's at the first divergence?
__device__ bool path_less(const int *par, int i, int j) {
    for (int guard = 0; guard < kMaxNodes && par[i] != par[j]; ++guard) {
        i = par[i];
        j = par[j];
    }
    return i < j;
}

__global__ void __launch_bounds__(kThreads)
spec_accept_kernel(int N, int V, int splits, int chunk, const float *__restrict__ logits,
                   const int32_t *__restrict__ tokens, const int32_t *__restrict__ parent,
                   int32_t *argmax_out, int32_t *accept_len, int32_t *accept_node,
                   unsigned *counters, unsigned long long *rowkeys, int32_t *dev_status) {
    __shared__ unsigned long long red[kThreads / 32];
    __shared__ bool is_last;
    __shared__ int am_s[kMaxNodes], par_s[kMaxNodes], dep_s[kMaxNodes], tok_s[kMaxNodes];
    __shared__ unsigned char ok_s[kMaxNodes], bad_s[kMaxNodes];
    __shared__ unsigned miss_s[kBallotWarps];

    const int split = blockIdx.x, n = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x;
    const float *row = logits + ((size_t)b * N + n) * (size_t)V;
    // buffer extents, for the bounds checks of debug builds (GDN_IN)
    const size_t B = gridDim.z;
    const gdndev::Buf bl{logits, B * N * (size_t)V * 4}, bt{tokens, B * N * 4}, bp{parent, B * N * 4},
        ba{argmax_out, B * N * 4}, bk{accept_len, B * 4}, bn{accept_node, B * 4}, bc{counters, B * 4},
        br{rowkeys, B * N * 8};
    const int lo = split * chunk;
    const int hi = min(V, lo + chunk);
    // evict-last: the chunk must outlast the previous grid's writes (the
    // verify streams its checkpoints at full bandwidth until it ends)
    if (lo < hi && GDN_IN(row + lo, (size_t)(hi - lo) * 4, bl, dev_status))
        gdndev::prefetch_l2_keep_range(row + lo, (size_t)(hi - lo) * 4, tid, kThreads);
    gdndev::pdl_wait();
    gdndev::pdl_launch_dependents();  // the restore may be scheduled; it waits for this grid
    // the request's draft tokens / parents, loaded now so that the last CTA
    // does not wait for them after the ticket
    const int my_tok = tid < N ? gdndev::ldic(tokens + (size_t)b * N + tid, bt, dev_status) : 0;
    const int my_par = tid < N ? (parent ? gdndev::ldic(parent + (size_t)b * N + tid, bp, dev_status) : tid - 1) : 0;

    unsigned long long best = 0ull;  // below every real element
    if ((V & 3) == 0) {
        // rounds of kLoads independent 16-byte loads per thread, all issued
        // before the first is used (one chunk is normally a single round)
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        const int lo4 = lo >> 2, hi4 = hi >> 2;  // lo is a multiple of 4
        for (int i0 = lo4 + tid; i0 < hi4; i0 += kLoads * kThreads) {
            float4 f[kLoads];
#pragma unroll
            for (int u = 0; u < kLoads; ++u)
                if (i0 + u * kThreads < hi4)
                    f[u] = GDN_IN(r4 + i0 + u * kThreads, 16, bl, dev_status) ? __ldcs(r4 + i0 + u * kThreads)
                                                                                : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int u = 0; u < kLoads; ++u) {
                const int i = i0 + u * kThreads;
                if (i < hi4) {
                    const unsigned base = (unsigned)i * 4u;
                    best = umax64(best, make_key(f[u].x, base));
                    best = umax64(best, make_key(f[u].y, base + 1));
                    best = umax64(best, make_key(f[u].z, base + 2));
                    best = umax64(best, make_key(f[u].w, base + 3));
                }
            }
        }
    } else {
        for (int i = lo + tid; i < hi; i += kThreads)
            best = umax64(best, make_key(GDN_IN(row + i, 4, bl, dev_status) ? __ldcs(row + i) : 0.f, (unsigned)i));
    }
    if (lo < hi && GDN_IN(row + lo, (size_t)(hi - lo) * 4, bl, dev_status))
        gdndev::l2_normal_range(row + lo, (size_t)(hi - lo) * 4, tid, kThreads);  // read: priority back
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) best = umax64(best, __shfl_xor_sync(0xffffffffu, best, off));
    if ((tid & 31) == 0) red[tid >> 5] = best;
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kThreads / 32; ++w) best = umax64(best, red[w]);
        if ((unsigned)(best >> 32) == 0xFFFFFFFFu && dev_status) atomicOr(dev_status, GDN_DEV_NAN_LOGIT);
        if (GDN_IN(rowkeys + (size_t)b * N + n, 8, br, dev_status))
            atomicMax(&rowkeys[(size_t)b * N + n], best);  // the row's key: the max over its chunks
        // the ticket: release orders this CTA's key fold before it, acquire
        // orders the last CTA's reads of every row key after it
        const bool cin = GDN_IN(counters + b, 4, bc, dev_status);
        unsigned prev = 0u;
        if (cin)
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(counters + b) : "memory");
        is_last = cin && prev == (unsigned)(N * splits - 1);
    }
    __syncthreads();
    if (!is_last) return;

    // ---- last CTA of request b: every chunk's max has landed in the row keys
    if (tid < N) {  // N <= kMaxNodes <= kThreads
        unsigned long long *kp = rowkeys + (size_t)b * N + tid;
        const bool kin = GDN_IN(kp, 8, br, dev_status);
        const int am = (int)gdndev::key_index(kin ? __ldcg(kp) : 0ull);
        if (kin) *kp = 0ull;  // leave the workspace zero-filled
        am_s[tid] = am;
        if (GDN_IN(argmax_out + (size_t)b * N + tid, 4, ba, dev_status)) argmax_out[(size_t)b * N + tid] = am;
        tok_s[tid] = my_tok;
        // a tree node whose parent is outside [0, i) hangs under the root and
        // never matches, nor does anything below it (flagged below)
        const bool bad = tid > 0 && (my_par < 0 || my_par >= tid);
        par_s[tid] = tid == 0 ? -1 : (bad ? 0 : my_par);
        bad_s[tid] = bad ? 1 : 0;
    }
    __syncthreads();
    if (parent == nullptr) {
        // node i of a chain matches when its token is the argmax of row i - 1;
        // k = the number of leading matches (a token outside [0, V) never matches)
        if (tid < kBallotWarps * 32) {
            const int i = tid;
            const bool node = i >= 1 && i < N;
            const int tk = node ? tok_s[i] : 0;
            const bool range = node && (tk < 0 || tk >= V);
            const unsigned miss = __ballot_sync(0xffffffffu, node && tk != am_s[node ? i - 1 : 0]);
            const unsigned bad = __ballot_sync(0xffffffffu, range);
            if ((tid & 31) == 0) {
                miss_s[tid >> 5] = miss;
                if (bad && dev_status) atomicOr(dev_status, GDN_DEV_TOKEN_RANGE);
            }
        }
        __syncthreads();
        if (tid == 0) {
            int k = N - 1;
            for (int w = 0; w < kBallotWarps; ++w)
                if (miss_s[w]) {
                    k = 32 * w + __ffs((int)miss_s[w]) - 2;  // the first mismatching node, minus one
                    break;
                }
            if (GDN_IN(accept_len + b, 4, bk, dev_status)) accept_len[b] = k;
            if (GDN_IN(accept_node + b, 4, bn, dev_status)) accept_node[b] = k;
            if (GDN_IN(counters + b, 4, bc, dev_status)) counters[b] = 0u;  // leave the workspace zero-filled
        }
    } else {
        // every node: its depth and whether its whole root path matches
        // (tokens[j] == argmax of row parent(j) for every j on it)
        if (tid < N) {
            int flags = bad_s[tid] ? GDN_DEV_TREE : 0;
            if (tid > 0 && (my_tok < 0 || my_tok >= V)) flags |= GDN_DEV_TOKEN_RANGE;
            int dep = 0;
            bool ok = true;
            for (int j = tid; j > 0; j = par_s[j]) {
                ++dep;
                ok = ok && !bad_s[j] && tok_s[j] == am_s[par_s[j]];
            }
            dep_s[tid] = dep;
            ok_s[tid] = ok ? 1 : 0;
            if (flags && dev_status) atomicOr(dev_status, flags);
        }
        __syncthreads();
        if (tid == 0) {
            // the deepest matching node; among equally deep ones the lower
            // node index at the first divergence of their root paths
            int best_node = 0;
            for (int i = 1; i < N; ++i)
                if (ok_s[i] && (dep_s[i] > dep_s[best_node] ||
                                (dep_s[i] == dep_s[best_node] && path_less(par_s, i, best_node))))
                    best_node = i;
            if (GDN_IN(accept_len + b, 4, bk, dev_status)) accept_len[b] = dep_s[best_node];
            if (GDN_IN(accept_node + b, 4, bn, dev_status)) accept_node[b] = best_node;
            if (GDN_IN(counters + b, 4, bc, dev_status)) counters[b] = 0u;
        }
    }
}

// Chunks per logit row: enough that a chunk is one round of loads (the scan
// is then a single memory round trip), and, for few rows, enough CTAs to
// cover the SMs, down to ~2K logits per chunk.
int choose_splits(int rows, int V) {
    const int sms = gdnhost::sm_count();
    const int target = 4 * (sms > 0 ? sms : 152);
    int s = (V + kRoundLogits - 1) / kRoundLogits;
    const int by_sms = (target + rows - 1) / rows;
    const int by_size = (V + 2047) / 2048;
    if (s < by_sms) s = by_sms < by_size ? by_sms : by_size;
    if (s > kMaxSplits) s = kMaxSplits;
    if (s < 1) s = 1;
    return s;
}

}  // namespace

extern "C" size_t spec_accept_workspace_bytes(int32_t batch, int32_t n_nodes) {
    if (batch < 1 || n_nodes < 1 || n_nodes > kMaxNodes || (int64_t)batch * n_nodes > (1 << 20)) return 0;
    return kCounterBytes(batch) + (size_t)batch * n_nodes * sizeof(unsigned long long);  // counters, row keys
}

extern "C" int spec_accept_greedy(int32_t batch, int32_t n_nodes, int32_t vocab, const float *logits,
                                  const int32_t *tokens, const int32_t *parent_dev, int32_t *argmax_out,
                                  int32_t *accept_len, int32_t *accept_node, void *workspace,
                                  size_t workspace_bytes, int32_t *dev_status, gdn_stream_t stream) {
    if (batch < 1 || batch > 65535 || n_nodes < 1 || n_nodes > kMaxNodes || vocab < 1 ||
        (int64_t)batch * n_nodes > (1 << 20))
        return GDN_ERR_DIMS;
    if (!logits || !tokens || !argmax_out || !accept_len || !accept_node) return GDN_ERR_NULL;
    using gdnhost::aligned_to;
    if (!aligned_to(logits, 16) || !aligned_to(tokens, 4) || !aligned_to(argmax_out, 4) ||
        !aligned_to(accept_len, 4) || !aligned_to(accept_node, 4) ||
        (parent_dev && !aligned_to(parent_dev, 4)) || (dev_status && !aligned_to(dev_status, 4)))
        return GDN_ERR_ALIGN;
    const size_t need = spec_accept_workspace_bytes(batch, n_nodes);
    if (!workspace || workspace_bytes < need || !aligned_to(workspace, 256)) return GDN_ERR_WORKSPACE;

    const int splits = choose_splits(batch * n_nodes, vocab);
    int chunk = (vocab + splits - 1) / splits;
    chunk = (chunk + 3) & ~3;
    unsigned *counters = static_cast<unsigned *>(workspace);
    unsigned long long *rowkeys =
        reinterpret_cast<unsigned long long *>(static_cast<char *>(workspace) + kCounterBytes(batch));
    dim3 grid(splits, n_nodes, batch);
    return gdndev::launch_pdl(spec_accept_kernel, grid, dim3(kThreads), 0, static_cast<cudaStream_t>(stream), n_nodes,
                              vocab, splits, chunk, logits, tokens, parent_dev, argmax_out, accept_len, accept_node,
                              counters, rowkeys, dev_status) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// spec_accept_greedy_static: the same acceptance for callers that cannot
// allocate device memory. Its scratch (arrival counters + per-chunk keys)
// lives in the fixed array below, which every GPU that loads this library
// holds until the process exits.
// ---------------------------------------------------------------------------
namespace {

static __device__ __align__(256) unsigned char g_accept_scratch[GDN_STATIC_SCRATCH_BYTES];

// Device address of g_accept_scratch, looked up per device. In host code the
// symbol itself is only a host-side stand-in, never a device address, so
// kernels must be given the looked-up pointer. Only a successful lookup is
// kept: a failed one (for example a first call made during a stream capture
// that forbids it) fails that call alone, and the next call tries again.
// The kept address belongs to the device's current context; after a
// cudaDeviceReset the array lives elsewhere, which this cache does not
// follow (the entry point does not support cudaDeviceReset).
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices];

int static_scratch(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();  // leave no sticky launch error behind for the next call
            return GDN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" int spec_accept_greedy_static(int32_t batch, int32_t n_nodes, int32_t vocab, const float *logits,
                                         const int32_t *tokens, const int32_t *parent_dev,
                                         int32_t *argmax_out, int32_t *accept_len, int32_t *accept_node,
                                         int32_t *dev_status, gdn_stream_t stream) {
    if (batch < 1 || batch > 65535 || n_nodes < 1 || n_nodes > kMaxNodes || vocab < 1 ||
        (int64_t)batch * n_nodes > (1 << 20))
        return GDN_ERR_DIMS;
    if (!logits || !tokens || !argmax_out || !accept_len || !accept_node) return GDN_ERR_NULL;
    using gdnhost::aligned_to;
    if (!aligned_to(logits, 16) || !aligned_to(tokens, 4) || !aligned_to(argmax_out, 4) ||
        !aligned_to(accept_len, 4) || !aligned_to(accept_node, 4) ||
        (parent_dev && !aligned_to(parent_dev, 4)) || (dev_status && !aligned_to(dev_status, 4)))
        return GDN_ERR_ALIGN;
    const size_t need = spec_accept_workspace_bytes(batch, n_nodes);
    if (need == 0 || need > (size_t)GDN_STATIC_SCRATCH_BYTES) return GDN_ERR_WORKSPACE;
    void *scratch = nullptr;
    int rc = static_scratch(&scratch);
    if (rc != GDN_OK) return rc;

    // The array keeps whatever the previous call left (a completed call
    // leaves the bytes it used at zero): zero the arrival counters and row
    // keys of this call on the same stream all the same.
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, need, st) != cudaSuccess) return GDN_ERR_CUDA;
    const int splits = choose_splits(batch * n_nodes, vocab);
    int chunk = (vocab + splits - 1) / splits;
    chunk = (chunk + 3) & ~3;
    unsigned *counters = static_cast<unsigned *>(scratch);
    unsigned long long *rowkeys =
        reinterpret_cast<unsigned long long *>(static_cast<char *>(scratch) + kCounterBytes(batch));
    dim3 grid(splits, n_nodes, batch);
    spec_accept_kernel<<<grid, kThreads, 0, st>>>(n_nodes, vocab, splits, chunk, logits, tokens, parent_dev,
                                                  argmax_out, accept_len, accept_node, counters, rowkeys,
                                                  dev_status);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
