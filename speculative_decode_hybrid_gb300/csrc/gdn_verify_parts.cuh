// Device parts shared by the GDN span kernels (gdn_verify.cu, gdn_wy.cu):
// the argument block, work items, shared-memory layouts, cp.async staging of
// an item's inputs, conv1d + SiLU, the q/k L2 norms, and work stealing by
// cluster launch control. Each including translation unit gets its own copy
// (anonymous namespace).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "gdn_device.cuh"
#include "gdnspec.h"

namespace {

using namespace gdndev;

constexpr int kLanesPerRow = 8;
constexpr int kRowsPerSlot = 32 / kLanesPerRow;        // 4 rows per warp instruction
constexpr int kSlots = 4;
constexpr int kRowsPerWarp = kRowsPerSlot * kSlots;    // 16
constexpr int kMaxWarps = 8;
constexpr int kRowsPerCta = kRowsPerWarp * kMaxWarps;  // 128
constexpr int kColStride = 4 * kLanesPerRow;           // lane j owns columns 4j + kColStride*m + 0..3
constexpr int kThreads = kMaxWarps * 32;
constexpr size_t kMaxSmem = 227 * 1024;
constexpr size_t kStaticSmem = 64;  // the work-stealing kernel's static shared memory
static_assert(kRowsPerWarp <= 16 && 16 % kRowsPerWarp == 0, "d_v is validated as a multiple of 16");

struct VerifyArgs {
    int Y, H_k, H_v, d_v, C, K, T;
    float q_scale;
    const void *x, *a, *b, *w;
    const float *ssm_in, *conv_in;
    float *ssm_ckpt, *conv_ckpt, *out;  // ssm_ckpt / conv_ckpt NULL: no checkpoints
    const int32_t *parent;  // [B][T+1] for trees, nullptr for chains
    int32_t *dev_status;
    float *ssm_out;         // replay commit: the live state, updated in place
    const int32_t *accept_len;  // replay commit: tokens to replay per request
    int rpi;                // value rows per work item: a multiple of 16, <= kRowsPerCta
};

// One work item: (request*layer by, value head h, row block rb).
struct Item {
    int by, h, rb, y, bidx, g, row0, R;
};

// Row blocks per value head.
__host__ __device__ __forceinline__ int row_blocks(const VerifyArgs &p) { return (p.d_v + p.rpi - 1) / p.rpi; }

__device__ __forceinline__ Item decode_item(const VerifyArgs &p, int it, int nrb) {
    Item I;
    I.rb = it % nrb;
    const int r = it / nrb;
    I.h = r % p.H_v;
    I.by = r / p.H_v;
    I.y = I.by % p.Y;
    I.bidx = I.by / p.Y;
    I.g = I.h / (p.H_v / p.H_k);  // key head floor(h * H_k / H_v)
    I.row0 = I.rb * p.rpi;
    I.R = min(p.rpi, p.d_v - I.row0);  // a multiple of kRowsPerWarp
    return I;
}

// Global channel of local channel lc of an item: [q (DK) | k (DK) | v (R)].
template <int DK>
__device__ __forceinline__ int item_channel(const VerifyArgs &p, const Item &I, int lc) {
    if (lc < DK) return I.g * DK + lc;
    if (lc < 2 * DK) return p.H_k * DK + I.g * DK + (lc - DK);
    return 2 * p.H_k * DK + I.h * p.d_v + I.row0 + (lc - 2 * DK);
}

__host__ __device__ constexpr size_t al16(size_t v) { return (v + 15) & ~size_t(15); }

// Shared-memory carve-up of the one-item-per-CTA kernel (byte offsets),
// identical on host and device.
struct Layout {
    size_t q, k, v, o, a, b, kq, par, src, total;
};

__host__ __device__ inline Layout make_layout(int T, int DK, int K) {
    Layout L;
    size_t off = 0;
    L.q = off; off = al16(off + (size_t)T * DK * 4);
    L.k = off; off = al16(off + (size_t)T * DK * 4);
    L.v = off; off = al16(off + (size_t)T * kRowsPerCta * 4);
    L.o = off; off = al16(off + (size_t)T * kRowsPerCta * 4);
    L.a = off; off = al16(off + (size_t)T * 4);
    L.b = off; off = al16(off + (size_t)T * 4);
    L.kq = off; off = al16(off + (size_t)T * 4);
    L.par = off; off = al16(off + (size_t)(2 * T + 1) * 4);  // parents, then the DFS order
    L.src = off; off = al16(off + (size_t)T * K * 4);
    L.total = off;
    return L;
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Cluster launch control (sm_100 family): a running CTA asks the hardware to
// cancel the launch of a CTA of the same grid that has not started; on
// success it gets that CTA's index and does its work. The 16-byte response
// lands in shared memory and completes a transaction on an mbarrier. A
// request is never issued again after one has failed. One thread (the
// leader) drives all of it.
// ---------------------------------------------------------------------------
constexpr unsigned kStealPolls = 1u << 22;  // bound on the response wait

__device__ __forceinline__ void steal_init(unsigned bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}

// Ask for the next pending CTA. The response buffer was last read through
// the generic proxy; the proxy fence orders that read before the
// asynchronous write of the new response.
__device__ __forceinline__ void steal_issue(unsigned resp, unsigned bar) {
    asm volatile(
        "fence.proxy.async.shared::cta;\n\t"
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], 16;" ::"r"(resp),
        "r"(bar)
        : "memory");
}

// Wait for the response of phase `phase` (bounded); then the x index of the
// cancelled CTA, or -1 when the request failed (nothing left to take), or -2
// when the wait gave up.
__device__ __forceinline__ int steal_result(unsigned resp, unsigned bar, unsigned phase) {
    unsigned done = 0;
    for (unsigned i = 0; i < kStealPolls && !done; ++i)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.b32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(phase)
            : "memory");
    if (!done) return -2;
    unsigned long long lo, hi;
    asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(lo), "=l"(hi) : "r"(resp) : "memory");
    int ok = 0, x = -1;
    asm volatile(
        "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
        "mov.b128 r, {%2, %3};\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
        : "=r"(ok), "+r"(x)
        : "l"(lo), "l"(hi)
        : "memory");
    return ok ? x : -1;
}

// Tree: validated parents -> par_s, and the conv-window table src_s:
// position j of node i's window holds the input of the node at path depth
// depth(i) - (K-1-j) when that is >= 1, else conv-state slot K-2 + that
// depth (encoded -1 - slot). pg is the request's parent array in global
// memory; `pr` is pg[tid] already loaded by this thread (when tid <= T).
__device__ __forceinline__ void bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// tid / nthreads: this thread's rank in the calling group; the group syncs
// on hardware barrier `bar` (0 with the whole block = __syncthreads).
__device__ __forceinline__ void tree_tables(const VerifyArgs &p, const int32_t *pg, int pr, int *par_s,
                                            int *src_s, int tid, int nthreads, int bar) {
    const int T = p.T, K = p.K;
    for (int i = tid; i <= T; i += nthreads) {
        int v = i == 0 ? -1 : (i == tid ? pr : pg[i]);
        if (i > 0 && (v < 0 || v >= i)) {
            v = i - 1;
            if (p.dev_status) atomicOr(p.dev_status, GDN_DEV_TREE);
        }
        par_s[i] = v;
    }
    bar_sync(bar, nthreads);
    if (tid == 0) {
        // Depth-first preorder of nodes 1..T: a node's state is still in
        // registers when its first child runs, and a parent's state is
        // reloaded (from its checkpoint) only on a branch switch. Children
        // go in ascending order of subtree size (ties: lower index first),
        // which keeps each reload close in time to the write of the state
        // it reads, so that the checkpoint is still in L2 (48 layers, 23
        // nodes: DRAM reads 245 -> 132 MB per launch).
        int *ord_s = par_s + (T + 1);
        int first[GDN_MAX_TOKENS + 1], next[GDN_MAX_TOKENS + 1], size[GDN_MAX_TOKENS + 1];
        for (int i = 0; i <= T; ++i) {
            first[i] = next[i] = -1;
            size[i] = 1;
        }
        for (int i = T; i >= 1; --i) size[par_s[i]] += size[i];
        for (int i = T; i >= 1; --i) {  // insert i among its siblings, ordered by (size, index)
            int *link = &first[par_s[i]];
            while (*link > 0 && (size[*link] < size[i] || (size[*link] == size[i] && *link < i))) link = &next[*link];
            next[i] = *link;
            *link = i;
        }
        int n = first[0], q = 0;
        while (n > 0 && q < T) {
            ord_s[q++] = n;
            if (first[n] > 0) {
                n = first[n];
            } else {
                while (n > 0 && next[n] < 0) n = par_s[n];
                n = n > 0 ? next[n] : -1;
            }
        }
    }
    for (int i = tid + 1; i <= T; i += nthreads) {
        int depth = 0;
        for (int n = i; n > 0; n = par_s[n]) ++depth;
        int node = i;
        for (int j = K - 1; j >= 0; --j) {
            const int pos = depth - (K - 1 - j);
            if (pos >= 1) {
                src_s[(i - 1) * K + j] = node;
                node = par_s[node];
            } else {
                src_s[(i - 1) * K + j] = -1 - (K - 2 + pos);
            }
        }
    }
}

// Per-head L2 norm of q and k, q scale, k.q; one warp per node.
template <int DK>
__device__ __forceinline__ void norm_qk(const VerifyArgs &p, float *q_s, float *k_s, float *kq_s, int count,
                                       int warp, int nwarps) {
    constexpr int PER = DK / 32;
    const int lane = threadIdx.x & 31;
    for (int t = warp; t < count; t += nwarps) {
        float qv[PER], kv[PER];
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            qv[e] = q_s[(size_t)t * DK + lane + 32 * e];
            kv[e] = k_s[(size_t)t * DK + lane + 32 * e];
            sq = fmaf(qv[e], qv[e], sq);
            sk = fmaf(kv[e], kv[e], sk);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, off);
            sk += __shfl_xor_sync(0xffffffffu, sk, off);
        }
        const float iq = 1.0f / sqrtf(sq + 1e-6f);
        const float ik = 1.0f / sqrtf(sk + 1e-6f);
        float kq = 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            qv[e] = qv[e] * iq * p.q_scale;
            kv[e] = kv[e] * ik;
            q_s[(size_t)t * DK + lane + 32 * e] = qv[e];
            k_s[(size_t)t * DK + lane + 32 * e] = kv[e];
            kq = fmaf(qv[e], kv[e], kq);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
        if (lane == 0) kq_s[t] = kq;
    }
}

// One conv output: sum_j w[j] * win[j] over the K-window, then SiLU.
__device__ __forceinline__ float conv_out(const float (&wr)[GDN_MAX_CONV_K], const float (&win)[GDN_MAX_CONV_K],
                                          int K) {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < GDN_MAX_CONV_K; ++j)
        if (j < K) acc = fmaf(wr[j], win[j], acc);
    return silu(acc);
}

// ---------------------------------------------------------------------------
// Staged prologue: the next item's inputs are copied into shared memory while
// the current item runs, then convolved there.
// ---------------------------------------------------------------------------

// Queue the asynchronous copies of item I's x tile, conv taps and conv state
// into the staging buffers (16-byte cp.async; every source and destination
// offset is a multiple of 16 bytes, see the host-side eligibility check).
// with_qk false: the v range only (the q/k of the item are already on chip).
// ntok: the tokens to copy (the first ntok of the span, ntok <= p.T).
template <int DK, bool BF16>
__device__ __forceinline__ void prefetch_item(const VerifyArgs &p, const Item &I, unsigned char *xst,
                                              unsigned char *wst, unsigned char *cst, bool with_qk, int tid,
                                              int nthreads, int ntok) {
    constexpr int ES = BF16 ? 2 : 4;
    constexpr int XS = 2 * DK + kRowsPerCta;
    const int T = p.T, K = p.K;
    const unsigned char *xg = static_cast<const unsigned char *>(p.x);
    const unsigned char *wg = static_cast<const unsigned char *>(p.w);
    const unsigned char *cg = reinterpret_cast<const unsigned char *>(p.conv_in);
    const size_t c_q = (size_t)I.g * DK, c_k = (size_t)p.H_k * DK + (size_t)I.g * DK;
    const size_t c_v = 2 * (size_t)p.H_k * DK + (size_t)I.h * p.d_v + I.row0;
    // x: per node, the three channel ranges [q | k | v]
    {
        const int cq = DK * ES / 16, cv = I.R * ES / 16;
        const int r0 = with_qk ? 0 : 2 * cq, per_node = 2 * cq + cv - r0;
        for (int i = tid; i < ntok * per_node; i += nthreads) {
            const int t = i / per_node, r = r0 + (i - t * per_node);
            size_t c0;
            int dch, off;
            if (r < cq) { c0 = c_q; dch = 0; off = r; }
            else if (r < 2 * cq) { c0 = c_k; dch = DK; off = r - cq; }
            else { c0 = c_v; dch = 2 * DK; off = r - 2 * cq; }
            cp_async16(xst + ((size_t)t * XS + dch) * ES + (size_t)off * 16,
                       xg + (((size_t)I.by * T + t) * p.C + c0) * ES + (size_t)off * 16);
        }
    }
    // conv taps [c][K] and conv state [c][K-1] of the three ranges
    {
        const int wq = DK * K * ES / 16, wv = I.R * K * ES / 16, wn = 2 * wq + wv;
        for (int i = (with_qk ? 0 : 2 * wq) + tid; i < wn; i += nthreads) {
            size_t c0;
            int dch, off;
            if (i < wq) { c0 = c_q; dch = 0; off = i; }
            else if (i < 2 * wq) { c0 = c_k; dch = DK; off = i - wq; }
            else { c0 = c_v; dch = 2 * DK; off = i - 2 * wq; }
            cp_async16(wst + (size_t)dch * K * ES + (size_t)off * 16,
                       wg + ((size_t)I.y * p.C + c0) * K * ES + (size_t)off * 16);
        }
        const int sq = DK * (K - 1) * 4 / 16, sv = I.R * (K - 1) * 4 / 16, sn = 2 * sq + sv;
        for (int i = (with_qk ? 0 : 2 * sq) + tid; i < sn; i += nthreads) {
            size_t c0;
            int dch, off;
            if (i < sq) { c0 = c_q; dch = 0; off = i; }
            else if (i < 2 * sq) { c0 = c_k; dch = DK; off = i - sq; }
            else { c0 = c_v; dch = 2 * DK; off = i - 2 * sq; }
            cp_async16(cst + (size_t)dch * (K - 1) * 4 + (size_t)off * 16,
                       cg + ((size_t)I.by * p.C + c0) * (K - 1) * 4 + (size_t)off * 16);
        }
    }
    cp_async_commit();
}

// The small per-item values that are not contiguous: gates (thread t < T)
// and, for trees, the parent array (thread i <= T); loaded into registers.
template <bool BF16, bool TREE>
__device__ __forceinline__ void prefetch_scalars(const VerifyArgs &p, const Item &I, float &ga, float &gb,
                                                 int &pr, int tid) {
    const int T = p.T;
    if (tid < T) {
        const size_t gi = ((size_t)I.by * T + tid) * p.H_v + I.h;
        ga = ld_in<BF16>(p.a, gi);
        gb = ld_in<BF16>(p.b, gi);
    }
    if constexpr (TREE) pr = tid <= T ? (tid == 0 ? -1 : p.parent[(size_t)I.bidx * (T + 1) + tid]) : 0;
}

// Shared-memory carve-up of the work-stealing kernel: the item's buffers plus
// the staging of the next item's inputs.
struct PipeLayout {
    size_t q, k, v, o, a, b, kq, par, src, xst, wst, cst, total;
};

__host__ __device__ inline PipeLayout make_pipe_layout(int T, int DK, int K, int esize) {
    PipeLayout L;
    size_t off = 0;
    const size_t XS = 2 * (size_t)DK + kRowsPerCta;  // staged channels per item
    L.q = off; off = al16(off + (size_t)T * DK * 4);
    L.k = off; off = al16(off + (size_t)T * DK * 4);
    L.v = off; off = al16(off + (size_t)T * kRowsPerCta * 4);
    L.o = off; off = al16(off + (size_t)T * kRowsPerCta * 4);
    L.a = off; off = al16(off + (size_t)T * 4);
    L.b = off; off = al16(off + (size_t)T * 4);
    L.kq = off; off = al16(off + (size_t)T * 4);
    L.par = off; off = al16(off + (size_t)(2 * T + 1) * 4);  // parents, then the DFS order
    L.src = off; off = al16(off + (size_t)T * K * 4);
    L.xst = off; off = al16(off + (size_t)T * XS * esize);
    L.wst = off; off = al16(off + XS * K * esize);
    L.cst = off; off = al16(off + XS * (K - 1) * 4);
    L.total = off;
    return L;
}

// conv1d + SiLU of item I from its staged inputs, by threads tid of nthreads.
// Work unit = (channel, half of the nodes), consecutive threads on
// consecutive channels (coalesced conv-checkpoint stores, conflict-free
// staging reads). A chain keeps its K-window in registers (one staged load
// per output); a tree gathers each node's window along its root path.
// skip_qk: only the v channels (q and k are the previous item's, still in
// shared memory; that item also wrote their conv checkpoints).
template <int DK, bool BF16, bool TREE, int KT>
__device__ __forceinline__ void conv_staged(const VerifyArgs &p, const Item &I, const unsigned char *xst,
                                            const unsigned char *wst, const unsigned char *cst,
                                            const int *src_s, float *q_s, float *k_s, float *v_s,
                                            bool skip_qk, int tid, int nthreads) {
    constexpr int XS = 2 * DK + kRowsPerCta;
    constexpr int KM = KT > 0 ? KT : GDN_MAX_CONV_K;
    const int T = p.T, K = KT > 0 ? KT : p.K;
    const float *cstf = reinterpret_cast<const float *>(cst);
    const size_t cc_tok = (size_t)p.C * (K - 1);
    {
        const int lc0 = skip_qk ? 2 * DK : 0, nch = 2 * DK + I.R - lc0;
        const bool own_qk = (I.h % (p.H_v / p.H_k) == 0) && I.rb == 0;
        const int nchunk = T >= 8 ? 2 : 1;
        const int tc = (T + nchunk - 1) / nchunk;
        for (int u = tid; u < nch * nchunk; u += nthreads) {
            const int lc = lc0 + u % nch, tb = (u / nch) * tc, te = min(T, tb + tc);
            float *dst = lc < DK ? q_s + lc : lc < 2 * DK ? k_s + (lc - DK) : v_s + (lc - 2 * DK);
            const int stride = lc < 2 * DK ? DK : kRowsPerCta;
            const bool own = (lc >= 2 * DK || own_qk) && p.conv_ckpt != nullptr;
            float *cck = p.conv_ckpt + (size_t)I.by * T * cc_tok + (size_t)item_channel<DK>(p, I, lc) * (K - 1);
            float wr[KM];
#pragma unroll
            for (int j = 0; j < KM; ++j) wr[j] = j < K ? ld_in<BF16>(wst, (size_t)lc * K + j) : 0.f;
            if constexpr (!TREE) {
                // win[j], j < K-1: sequence position tb-(K-1)+j (x row when >= 0,
                // else conv-state slot K-1+position)
                float win[KM];
#pragma unroll
                for (int j = 0; j < KM; ++j) {
                    win[j] = 0.f;
                    if (j < K - 1) {
                        const int sp = tb - (K - 1) + j;
                        win[j] = sp >= 0 ? ld_in<BF16>(xst, (size_t)sp * XS + lc)
                                         : cstf[(size_t)lc * (K - 1) + (K - 1 + sp)];
                    }
                }
                for (int t = tb; t < te; ++t) {
                    const float xv = ld_in<BF16>(xst, (size_t)t * XS + lc);
                    float acc = 0.f;
#pragma unroll
                    for (int j = 0; j < KM; ++j)
                        if (j < K) acc = fmaf(wr[j], j < K - 1 ? win[j] : xv, acc);
                    dst[(size_t)t * stride] = silu(acc);
#pragma unroll
                    for (int j = 0; j < KM - 1; ++j) {
                        if (j < K - 2) win[j] = win[j + 1];
                        else if (j == K - 2) win[j] = xv;
                    }
                    if (own) {
#pragma unroll
                        for (int j = 0; j < KM - 1; ++j)
                            if (j < K - 1) cck[(size_t)t * cc_tok + j] = win[j];
                    }
                }
            } else {
                for (int t = tb; t < te; ++t) {
                    float win[KM];
                    float acc = 0.f;
#pragma unroll
                    for (int j = 0; j < KM; ++j) {
                        win[j] = 0.f;
                        if (j < K) {
                            const int sn = src_s[t * K + j];  // >= 1: node; else -1 - conv-state slot
                            win[j] = sn >= 1 ? ld_in<BF16>(xst, (size_t)(sn - 1) * XS + lc)
                                             : cstf[(size_t)lc * (K - 1) + (-1 - sn)];
                            acc = fmaf(wr[j], win[j], acc);
                        }
                    }
                    dst[(size_t)t * stride] = silu(acc);
                    if (own) {
#pragma unroll
                        for (int j = 0; j < KM - 1; ++j)
                            if (j < K - 1) cck[(size_t)t * cc_tok + j] = win[j + 1];
                    }
                }
            }
        }
    }
}

// Raise a kernel's dynamic shared-memory limit once per size (per process;
// raising it again is harmless).
template <typename K>
bool ensure_smem(K kern, size_t smem, std::atomic<size_t> &set) {
    if (smem <= set.load(std::memory_order_relaxed)) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return false;
    set.store(smem, std::memory_order_relaxed);
    return true;
}

VerifyArgs make_args(const gdn_dims *d, int32_t T, const void *x, const void *a, const void *b,
                     const void *w, const float *ssm_in, const float *conv_in, float *ssm_ckpt,
                     float *conv_ckpt, float *out, const int32_t *parent, int32_t *dev_status) {
    VerifyArgs v;
    v.Y = d->layers;
    v.H_k = d->h_k;
    v.H_v = d->h_v;
    v.d_v = d->d_v;
    v.C = d->conv_ch;
    v.K = d->conv_k;
    v.T = T;
    v.q_scale = d->q_scale;
    v.x = x;
    v.a = a;
    v.b = b;
    v.w = w;
    v.ssm_in = ssm_in;
    v.conv_in = conv_in;
    v.ssm_ckpt = ssm_ckpt;
    v.conv_ckpt = conv_ckpt;
    v.out = out;
    v.parent = parent;
    v.dev_status = dev_status;
    v.ssm_out = nullptr;
    v.accept_len = nullptr;
    v.rpi = kRowsPerCta;
    return v;
}

// The live conv state after the replayed tokens: the last K-1 inputs of
// [conv_state, x_0 .. x_{k-1}], one thread per channel (reads before writes).
template <bool BF16>
__global__ void __launch_bounds__(256) gdn_conv_state_kernel(const VerifyArgs p, const int32_t *accept_len,
                                                            float *conv_state) {
    pdl_wait();
    const int by = blockIdx.y, bidx = by / p.Y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const int K = p.K, T = p.T;
    const int k = accept_len[bidx];
    if (c >= p.C || k <= 0 || k > T) return;
    float *cs = conv_state + ((size_t)by * p.C + c) * (K - 1);
    float nw[GDN_MAX_CONV_K];
#pragma unroll
    for (int j = 0; j < GDN_MAX_CONV_K - 1; ++j) {
        nw[j] = 0.f;
        if (j < K - 1) {
            const int sp = k - (K - 1) + j;  // sequence position: x row when >= 0
            nw[j] = sp >= 0 ? ld_in<BF16>(p.x, ((size_t)by * T + sp) * p.C + c) : cs[K - 1 + sp];
        }
    }
#pragma unroll
    for (int j = 0; j < GDN_MAX_CONV_K - 1; ++j)
        if (j < K - 1) cs[j] = nw[j];
}

}  // namespace
