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
    int B, Tb;              // requests; tokens of the call's buffers (T itself may be fewer: a replay's k)
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
    int steal;              // work-stealing kernel: ask for pending items (0: every CTA runs its own item)
    int early;              // GDN_VERIFY_STATE_READY: the state, conv taps / state and parents may be
                            // read before the wait for the previous grid on the stream
    const int32_t *x_ready; // inputs landing during the launch: the x, a, b rows of (request, layer)
                            // by may be read once x_ready[by] != 0 (null: all there at launch)
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

// Extents of the argument buffers, for the bounds checks of debug builds
// (GDN_IN; never evaluated in release builds). ES: bytes per input element;
// DK: the key head size.
__device__ __forceinline__ size_t n_by(const VerifyArgs &p) { return (size_t)p.B * p.Y; }
template <int ES>
__device__ __forceinline__ Buf buf_x(const VerifyArgs &p) { return {p.x, n_by(p) * p.Tb * p.C * ES}; }
template <int ES>
__device__ __forceinline__ Buf buf_a(const VerifyArgs &p) { return {p.a, n_by(p) * p.Tb * p.H_v * ES}; }
template <int ES>
__device__ __forceinline__ Buf buf_b(const VerifyArgs &p) { return {p.b, n_by(p) * p.Tb * p.H_v * ES}; }
template <int ES>
__device__ __forceinline__ Buf buf_w(const VerifyArgs &p) { return {p.w, (size_t)p.Y * p.C * p.K * ES}; }
template <int DK>
__device__ __forceinline__ Buf buf_state(const VerifyArgs &p) { return {p.ssm_in, n_by(p) * p.H_v * p.d_v * DK * 4}; }
__device__ __forceinline__ Buf buf_conv(const VerifyArgs &p) { return {p.conv_in, n_by(p) * p.C * (p.K - 1) * 4}; }
template <int DK>
__device__ __forceinline__ Buf buf_ckpt(const VerifyArgs &p) {
    return {p.ssm_ckpt, n_by(p) * p.Tb * p.H_v * p.d_v * DK * 4};
}
__device__ __forceinline__ Buf buf_cckpt(const VerifyArgs &p) { return {p.conv_ckpt, n_by(p) * p.Tb * p.C * (p.K - 1) * 4}; }
__device__ __forceinline__ Buf buf_out(const VerifyArgs &p) { return {p.out, n_by(p) * p.Tb * p.H_v * p.d_v * 4}; }
__device__ __forceinline__ Buf buf_parent(const VerifyArgs &p) { return {p.parent, (size_t)p.B * (p.Tb + 1) * 4}; }
__device__ __forceinline__ Buf buf_accept(const VerifyArgs &p) { return {p.accept_len, (size_t)p.B * 4}; }
__device__ __forceinline__ Buf buf_ready(const VerifyArgs &p) { return {p.x_ready, (size_t)p.B * p.Y * 4}; }

__host__ __device__ constexpr size_t al16(size_t v) { return (v + 15) & ~size_t(15); }

// Ints of the tree-table region of shared memory for T processed nodes:
// parents (T+1), the depth-first order (T), the reload plan (T+1) and six
// scratch arrays of T+1.
__host__ __device__ constexpr size_t tree_table_ints(int T) { return 9 * (size_t)T + 8; }

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
    L.par = off; off = al16(off + tree_table_ints(T) * 4);  // the tree tables
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

// ---------------------------------------------------------------------------
// Inputs landing during the launch (x_ready non-null): the x, a and b rows of
// (request, layer) by may be read once x_ready[by] != 0. A copy engine sets
// the flag after it has copied the rows (the caller's contract: no kernel
// sets it, since a kernel could wait for an SM that this launch holds). The
// flag is read with acquire semantics at system scope, so the rows' bytes
// are visible to the reading thread after it; a warp or block barrier then
// orders the other threads' reads after that one.
// ---------------------------------------------------------------------------
constexpr unsigned kReadyPolls = 1u << 20;  // with the back-off below, about a quarter second

__device__ __forceinline__ bool ready_flag(const VerifyArgs &p, int by) {
    const int32_t *f = p.x_ready + by;
    if (!GDN_IN(f, 4, buf_ready(p), p.dev_status)) return true;
    int v;
    asm volatile("ld.acquire.sys.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v != 0;
}

// Wait (bounded) until the rows of by have landed: lane 0 of each calling
// warp polls, then the warp's barrier. A wait that gives up sets
// GDN_DEV_SCHED (the item then reads whatever is there).
__device__ __forceinline__ void wait_ready(const VerifyArgs &p, int by) {
    if (!p.x_ready) return;
    if ((threadIdx.x & 31) == 0) {
        bool ok = false;
        for (unsigned i = 0; i < kReadyPolls && !ok; ++i) {
            ok = ready_flag(p, by);
            if (!ok) __nanosleep(200);
        }
        if (!ok && p.dev_status) atomicOr(p.dev_status, GDN_DEV_SCHED);
    }
    __syncwarp();
}

__device__ __forceinline__ void bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Tree tables of one request, built by the calling group of threads
// (tid / nthreads: this thread's rank; the group syncs on hardware barrier
// `bar`, 0 with the whole block = __syncthreads), one thread per node:
//  * par_s: the parents, validated (a parent outside [0, i) becomes i-1 and
//    sets GDN_DEV_TREE). pg is the request's parent array in global memory;
//    `pr` is pg[tid] already loaded by this thread (when tid <= T).
//  * ord_s (= par_s + T+1): the depth-first preorder of nodes 1..T. A
//    node's state is still in registers when its first child runs, and a
//    parent's state is fetched again only on a branch switch. Children run
//    in ascending order of subtree size (ties: lower index first), which
//    keeps each fetch close in time to the write of the state it reads (48
//    layers, 23 nodes: DRAM reads 245 -> 132 MB per launch with the root
//    alone parked). A node's position is the sum, along its root path, of
//    1 + the sizes of the siblings that run before each node on it.
//  * plan_s (= ord_s + T): the reload plan of the recurrence. Entry q < T,
//    for the q-th node n of the order, is (park << 16) | (src & 0xffff):
//    src says where the state of parent(n) comes from when it is not the
//    state just computed (-1: it is; k >= 0: tensor-memory slot k; -2: its
//    checkpoint, or the initial state for the root), park >= 0 is the slot
//    that keeps n's own state after its step, for its later children. Entry
//    T is the slot of the initial (root) state, or -1. The slots form a
//    stack of the branch points whose later children are still to run (a
//    depth-first order returns to them innermost first); a branch point is
//    parked when fewer than `cap` slots are taken at its step, i.e. when it
//    has fewer than `cap` such branch points above it (an ancestor is one
//    while the child on the way down is not its last), and then that count
//    is its slot. cap = 0: every fetch reads memory.
//  * src_s: the conv-window table: position j of node i's window holds the
//    input of the node at path depth depth(i) - (K-1-j) when that is >= 1,
//    else conv-state slot K-2 + that depth (encoded -1 - slot).
// The caller syncs the group before anyone reads the tables.
__device__ __forceinline__ void tree_tables(const VerifyArgs &p, const int32_t *pg, int pr, int *par_s,
                                            int *src_s, int tid, int nthreads, int bar, int cap = 0) {
    const int T = p.T, K = p.K;
    int *ord_s = par_s + (T + 1), *plan_s = ord_s + T;
    int *size_s = plan_s + (T + 1), *nch_s = size_s + (T + 1), *off_s = nch_s + (T + 1);
    int *pos_s = off_s + (T + 1), *last_s = pos_s + (T + 1), *slot_s = last_s + (T + 1);
    for (int i = tid; i <= T; i += nthreads) {
        int v = i == 0 ? -1 : (i == tid ? pr : ldic(pg + i, buf_parent(p), p.dev_status));
        if (i > 0 && (v < 0 || v >= i)) {
            v = i - 1;
            if (p.dev_status) atomicOr(p.dev_status, GDN_DEV_TREE);
        }
        par_s[i] = v;
        size_s[i] = 1;
        nch_s[i] = 0;
        last_s[i] = 0;
    }
    bar_sync(bar, nthreads);
    // subtree sizes and child counts: every node adds itself to its ancestors
    for (int i = tid + 1; i <= T; i += nthreads) {
        atomicAdd(&nch_s[par_s[i]], 1);
        for (int a = par_s[i]; a >= 0; a = par_s[a]) atomicAdd(&size_s[a], 1);
    }
    bar_sync(bar, nthreads);
    // offset after the parent in the preorder; the sibling that runs last
    for (int i = tid + 1; i <= T; i += nthreads) {
        const int pp = par_s[i], si = size_s[i];
        int off = 1;
        bool last = true;
        for (int j = 1; j <= T; ++j) {
            if (j == i || par_s[j] != pp) continue;
            const int sj = size_s[j];
            if (sj < si || (sj == si && j < i)) off += sj;
            else last = false;
        }
        off_s[i] = off;
        if (last) last_s[pp] = i;
    }
    bar_sync(bar, nthreads);
    // preorder positions; parking slots
    for (int i = tid; i <= T; i += nthreads) {
        if (i > 0) {
            int pos = -1;
            for (int a = i; a > 0; a = par_s[a]) pos += off_s[a];
            pos_s[i] = pos;
            ord_s[pos] = i;
        }
        int slot = -1;
        if (cap > 0 && nch_s[i] >= 2) {
            int open = 0;
            for (int c = i, a = par_s[i]; a >= 0; c = a, a = par_s[a]) open += last_s[a] != c;
            if (open < cap) slot = open;
        }
        slot_s[i] = slot;
    }
    bar_sync(bar, nthreads);
    for (int i = tid + 1; i <= T; i += nthreads) {
        const int pos = pos_s[i], pp = par_s[i];
        const int prev = pos > 0 ? ord_s[pos - 1] : 0;
        const int src = pp == prev ? -1 : (slot_s[pp] >= 0 ? slot_s[pp] : -2);
        plan_s[pos] = (slot_s[i] << 16) | (src & 0xffff);
    }
    if (tid == 0) plan_s[T] = slot_s[0];
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

// L2 norms of one node's q and k, held by one warp: lane l holds elements
// l, l + 32, ..., l + 32 (CPL - 1) of each. u / sqrt(sum u^2 + 1e-6) in place, q
// also scaled by q_scale; returns k.q of the normalised vectors, computed as
// (sum q k) iq q_scale ik from the raw q.k, reduced in the same butterfly as
// the two sums of squares (one chain of shuffles per node, not two). Every
// value is the same in every lane: each xor-butterfly stage adds the same
// two operands in both partner lanes. Every kernel normalises through this
// function, so the bytes of q, k and k.q do not depend on which kernel
// computed them.
template <int CPL>
__device__ __forceinline__ float norm_node(float (&qv)[CPL], float (&kv)[CPL], float q_scale) {
    float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
        sq = fmaf(qv[e], qv[e], sq);
        sk = fmaf(kv[e], kv[e], sk);
        sqk = fmaf(qv[e], kv[e], sqk);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, off);
        sk += __shfl_xor_sync(0xffffffffu, sk, off);
        sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
    }
    // the hardware reciprocal square root (a few ulp), far inside the 2e-3
    // tolerance of the states and outputs
    const float iq = rsqrtf(sq + 1e-6f);
    const float ik = rsqrtf(sk + 1e-6f);
#pragma unroll
    for (int e = 0; e < CPL; ++e) {
        qv[e] = qv[e] * iq * q_scale;
        kv[e] = kv[e] * ik;
    }
    return sqk * iq * q_scale * ik;
}

// Per-head L2 norm of q and k (already convolved, in shared memory), q scale,
// k.q; one warp per node.
template <int DK>
__device__ __forceinline__ void norm_qk(const VerifyArgs &p, float *q_s, float *k_s, float *kq_s, int count,
                                       int warp, int nwarps) {
    constexpr int CPL = DK / 32;
    const int lane = threadIdx.x & 31;
    for (int t = warp; t < count; t += nwarps) {
        float qv[CPL], kv[CPL];
#pragma unroll
        for (int e = 0; e < CPL; ++e) {
            qv[e] = q_s[(size_t)t * DK + lane + 32 * e];
            kv[e] = k_s[(size_t)t * DK + lane + 32 * e];
        }
        const float kq = norm_node<CPL>(qv, kv, p.q_scale);
#pragma unroll
        for (int e = 0; e < CPL; ++e) {
            q_s[(size_t)t * DK + lane + 32 * e] = qv[e];
            k_s[(size_t)t * DK + lane + 32 * e] = kv[e];
        }
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
// parts: kStageX (the x tile), kStageTaps (conv taps and conv state) or both.
constexpr int kStageX = 1, kStageTaps = 2, kStageAll = 3;
template <int DK, bool BF16>
__device__ __forceinline__ void prefetch_item(const VerifyArgs &p, const Item &I, unsigned char *xst,
                                              unsigned char *wst, unsigned char *cst, bool with_qk, int tid,
                                              int nthreads, int ntok, int parts = kStageAll) {
    constexpr int ES = BF16 ? 2 : 4;
    constexpr int XS = 2 * DK + kRowsPerCta;
    const int T = p.T, K = p.K;
    const unsigned char *xg = static_cast<const unsigned char *>(p.x);
    const unsigned char *wg = static_cast<const unsigned char *>(p.w);
    const unsigned char *cg = reinterpret_cast<const unsigned char *>(p.conv_in);
    const size_t c_q = (size_t)I.g * DK, c_k = (size_t)p.H_k * DK + (size_t)I.g * DK;
    const size_t c_v = 2 * (size_t)p.H_k * DK + (size_t)I.h * p.d_v + I.row0;
    // x: per node, the three channel ranges [q | k | v]
    if (parts & kStageX) {
        const int cq = DK * ES / 16, cv = I.R * ES / 16;
        const int r0 = with_qk ? 0 : 2 * cq, per_node = 2 * cq + cv - r0;
        for (int i = tid; i < ntok * per_node; i += nthreads) {
            const int t = i / per_node, r = r0 + (i - t * per_node);
            size_t c0;
            int dch, off;
            if (r < cq) { c0 = c_q; dch = 0; off = r; }
            else if (r < 2 * cq) { c0 = c_k; dch = DK; off = r - cq; }
            else { c0 = c_v; dch = 2 * DK; off = r - 2 * cq; }
            const unsigned char *src = xg + (((size_t)I.by * T + t) * p.C + c0) * ES + (size_t)off * 16;
            if (GDN_IN(src, 16, buf_x<ES>(p), p.dev_status)) cp_async16(xst + ((size_t)t * XS + dch) * ES + (size_t)off * 16, src);
        }
    }
    // conv taps [c][K] and conv state [c][K-1] of the three ranges
    if (parts & kStageTaps) {
        const int wq = DK * K * ES / 16, wv = I.R * K * ES / 16, wn = 2 * wq + wv;
        for (int i = (with_qk ? 0 : 2 * wq) + tid; i < wn; i += nthreads) {
            size_t c0;
            int dch, off;
            if (i < wq) { c0 = c_q; dch = 0; off = i; }
            else if (i < 2 * wq) { c0 = c_k; dch = DK; off = i - wq; }
            else { c0 = c_v; dch = 2 * DK; off = i - 2 * wq; }
            const unsigned char *src = wg + ((size_t)I.y * p.C + c0) * K * ES + (size_t)off * 16;
            if (GDN_IN(src, 16, buf_w<ES>(p), p.dev_status)) cp_async16(wst + (size_t)dch * K * ES + (size_t)off * 16, src);
        }
        const int sq = DK * (K - 1) * 4 / 16, sv = I.R * (K - 1) * 4 / 16, sn = 2 * sq + sv;
        for (int i = (with_qk ? 0 : 2 * sq) + tid; i < sn; i += nthreads) {
            size_t c0;
            int dch, off;
            if (i < sq) { c0 = c_q; dch = 0; off = i; }
            else if (i < 2 * sq) { c0 = c_k; dch = DK; off = i - sq; }
            else { c0 = c_v; dch = 2 * DK; off = i - 2 * sq; }
            const unsigned char *src = cg + ((size_t)I.by * p.C + c0) * (K - 1) * 4 + (size_t)off * 16;
            if (GDN_IN(src, 16, buf_conv(p), p.dev_status)) cp_async16(cst + (size_t)dch * (K - 1) * 4 + (size_t)off * 16, src);
        }
    }
    cp_async_commit();
}

// The small per-item values that are not contiguous: gates (thread t < T)
// and, for trees, the parent array (thread i <= T); loaded into registers.
// The gates stay raw (bf16 bits zero-extended, or f32 bits) until
// gate_value() widens them, so that nothing waits for these loads before
// the staging wait (a widening right after the load would expose its
// latency).
template <bool BF16, bool TREE>
__device__ __forceinline__ void prefetch_scalars(const VerifyArgs &p, const Item &I, unsigned &ga, unsigned &gb,
                                                 int &pr, int tid) {
    const int T = p.T;
    if (tid < T) {
        const size_t gi = ((size_t)I.by * T + tid) * p.H_v + I.h;
        constexpr int ES = BF16 ? 2 : 4;
        const bool ina = GDN_IN(static_cast<const char *>(p.a) + gi * ES, ES, buf_a<ES>(p), p.dev_status);
        const bool inb = GDN_IN(static_cast<const char *>(p.b) + gi * ES, ES, buf_b<ES>(p), p.dev_status);
        if constexpr (BF16) {
            ga = ina ? reinterpret_cast<const unsigned short *>(p.a)[gi] : 0u;
            gb = inb ? reinterpret_cast<const unsigned short *>(p.b)[gi] : 0u;
        } else {
            ga = ina ? reinterpret_cast<const unsigned *>(p.a)[gi] : 0u;
            gb = inb ? reinterpret_cast<const unsigned *>(p.b)[gi] : 0u;
        }
    }
    if constexpr (TREE)
        pr = tid <= T ? (tid == 0 ? -1 : ldic(p.parent + (size_t)I.bidx * (T + 1) + tid, buf_parent(p), p.dev_status))
                      : 0;
}

// A raw gate from prefetch_scalars as f32 (bf16 -> f32 is exact).
template <bool BF16>
__device__ __forceinline__ float gate_value(unsigned raw) {
    return BF16 ? __uint_as_float(raw << 16) : __uint_as_float(raw);
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
    L.par = off; off = al16(off + tree_table_ints(T) * 4);  // the tree tables
    L.src = off; off = al16(off + (size_t)T * K * 4);
    L.xst = off; off = al16(off + (size_t)T * XS * esize);
    L.wst = off; off = al16(off + XS * K * esize);
    L.cst = off; off = al16(off + XS * (K - 1) * 4);
    L.total = off;
    return L;
}

// The K taps of local channel c from the staging buffer ([channel][K], bf16
// or f32), widened to f32 (bf16 -> f32 is exact: the bits move to the high
// half). With K = 4 one 8- or 16-byte load; consecutive channels in
// consecutive lanes read consecutive words (no bank conflict).
template <bool BF16, int KT, int KM>
__device__ __forceinline__ void load_taps(const unsigned char *wst, int c, int K, float (&w)[KM]) {
    if constexpr (KT == 4) {
        if constexpr (BF16) {
            const uint2 u = *reinterpret_cast<const uint2 *>(wst + (size_t)c * 8);
            w[0] = __uint_as_float(u.x << 16);
            w[1] = __uint_as_float(u.x & 0xffff0000u);
            w[2] = __uint_as_float(u.y << 16);
            w[3] = __uint_as_float(u.y & 0xffff0000u);
        } else {
            const float4 f = *reinterpret_cast<const float4 *>(wst + (size_t)c * 16);
            w[0] = f.x; w[1] = f.y; w[2] = f.z; w[3] = f.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < KM; ++j) w[j] = j < K ? ld_in<BF16>(wst, (size_t)c * K + j) : 0.f;
    }
}

// What every node of an item's conv prologue shares.
struct ConvCtx {
    const unsigned char *xst, *wst;  // staged x tile and conv taps
    const float *cstf;               // staged conv state
    float *q_s, *k_s, *v_s, *kq_s;   // outputs in shared memory
    float *cck;                      // this request's conv checkpoints (or null)
    size_t cc_tok, gq, gk, gv;       // checkpoint floats per node; global q, k channel of element 0, v row 0
    unsigned qk_own;                 // q/k channel groups whose conv checkpoints this item writes
    int K, lane;
    bool skip_qk;
};

// Window position j of a node: x row s >= 0 or conv-state slot -1 - s of
// local channel c. AX: the caller knows s >= 0 (no branch).
template <bool BF16, bool AX, int XS>
__device__ __forceinline__ float win_at(const ConvCtx &x, int s, int c) {
    if constexpr (AX) return ld_in<BF16>(x.xst, (unsigned)(s * XS + c));
    else
        return s >= 0 ? ld_in<BF16>(x.xst, (unsigned)(s * XS + c)) : x.cstf[(unsigned)(c * (x.K - 1) + (-1 - s))];
}

// conv1d + SiLU of one node t (window sources src), the q/k norms and k.q.
// AX: every window position is an x row (every chain node from K - 1 on):
// the loads of all the node's channels can then issue before the first use.
// QK / V: the q/k half (with the norms) and the v half of the node.
template <int DK, bool BF16, int KT, int KM, bool AX, bool QK, bool V>
__device__ __forceinline__ void conv_node(const VerifyArgs &p, const Item &I, const ConvCtx &x, int t,
                                          const int (&src)[KM]) {
    constexpr int XS = 2 * DK + kRowsPerCta;
    constexpr int CPL = DK / 32;
    const int K = KT > 0 ? KT : x.K, lane = x.lane;
    if (QK && !x.skip_qk) {
        // q (half 0) and k (half 1): element e is channel lane + 32 e
        float acc[2][CPL];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
            for (int e = 0; e < CPL; ++e) {
                const int c = hf * DK + lane + 32 * e;  // local channel
                float w[KM];
                load_taps<BF16, KT, KM>(x.wst, c, K, w);
                float *cc = (x.qk_own >> (hf * CPL + e)) & 1u
                                ? x.cck + (size_t)t * x.cc_tok + ((hf ? x.gk : x.gq) + 32 * e) * (K - 1)
                                : nullptr;
                float a = 0.f;
#pragma unroll
                for (int j = 0; j < KM; ++j) {
                    if (j < K) {
                        const float xv = win_at<BF16, AX, XS>(x, src[j], c);
                        a = fmaf(w[j], xv, a);
                        if (cc && j >= 1) stfc(cc + (j - 1), xv, buf_cckpt(p), p.dev_status);
                    }
                }
                acc[hf][e] = silu(a);
            }
        }
        const float kq = norm_node<CPL>(acc[0], acc[1], p.q_scale);
#pragma unroll
        for (int e = 0; e < CPL; ++e) {
            x.q_s[t * DK + lane + 32 * e] = acc[0][e];
            x.k_s[t * DK + lane + 32 * e] = acc[1][e];
        }
        if (lane == 0) x.kq_s[t] = kq;
    }
    if constexpr (!V) return;
    for (int lc = lane; lc < I.R; lc += 32) {
        const int c = 2 * DK + lc;
        float w[KM];
        load_taps<BF16, KT, KM>(x.wst, c, K, w);
        float *cv = x.cck ? x.cck + (size_t)t * x.cc_tok + (x.gv + lc) * (K - 1) : nullptr;
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < KM; ++j) {
            if (j < K) {
                const float xv = win_at<BF16, AX, XS>(x, src[j], c);
                acc = fmaf(w[j], xv, acc);
                if (cv && j >= 1) stfc(cv + (j - 1), xv, buf_cckpt(p), p.dev_status);
            }
        }
        x.v_s[t * kRowsPerCta + lc] = silu(acc);
    }
}

// Node t: its window sources (x row >= 0, or -1 - conv-state slot), then
// conv_node, branch-free when the whole window is in x (chains).
template <int DK, bool BF16, bool TREE, int KT, int KM, bool QK, bool V>
__device__ __forceinline__ void conv_at(const VerifyArgs &p, const Item &I, const ConvCtx &x, int t,
                                        const int *src_s) {
    const int K = KT > 0 ? KT : x.K;
    int src[KM];
    bool all_x = true;
#pragma unroll
    for (int j = 0; j < KM; ++j) {
        int s = 0;
        if (j < K) {
            if constexpr (TREE) {
                const int sn = src_s[t * K + j];  // >= 1: node; else -1 - slot
                s = sn >= 1 ? sn - 1 : sn;
            } else {
                const int sp = t - (K - 1) + j;
                s = sp >= 0 ? sp : -1 - (K - 1 + sp);
            }
            all_x = all_x && s >= 0;
        }
        src[j] = s;
    }
    if (!TREE && all_x)  // the same for the whole warp (chains: measured slower for trees)
        conv_node<DK, BF16, KT, KM, true, QK, V>(p, I, x, t, src);
    else
        conv_node<DK, BF16, KT, KM, false, QK, V>(p, I, x, t, src);
}

// conv1d + SiLU of item I from its staged inputs, fused with the q/k L2
// norms: one warp per node. Lane l owns q and k channels l, l + 32, ... of
// the key head (d_k / 32 each) and v channels l, l + 32, ... of the item, so
// a node's sums of squares reduce inside its warp and q, k go to shared
// memory once, normalised; consecutive lanes touch consecutive channels
// (conflict-free staging reads, coalesced conv-checkpoint stores). Window position j of node t
// comes from x row t - (K-1) + j of a chain (the conv state for negative
// rows) or from the root-path table src_s of a tree. Each output is the
// same fmaf chain over j = 0..K-1 as in the other kernels, so the bytes do
// not depend on the kernel. The conv checkpoint after a node (window
// positions 1..K-1, the last K-1 inputs) is written by the items that own
// the channels: v, every item its own rows; q/k, when every CTA runs just
// its own item (no work stealing, so no item skips the q/k conv), the
// M = (value heads per key head) x (row blocks) items of the key head
// share the 2 d_k / 32 channel groups (group hf * d_k/32 + e: channels
// lane + 32 e of q (hf = 0) or k (hf = 1)) round robin, else the key head's
// first item (never one that reuses q/k) writes them all.
// skip_qk: only the v channels (q, k and k.q are the previous item's, still
// in shared memory; that item also wrote their conv checkpoints).
template <int DK, bool BF16, bool TREE, int KT>
__device__ __forceinline__ void conv_norm_staged(const VerifyArgs &p, const Item &I, const unsigned char *xst,
                                                 const unsigned char *wst, const unsigned char *cst,
                                                 const int *src_s, float *q_s, float *k_s, float *v_s,
                                                 float *kq_s, bool skip_qk, int warp, int nwarps) {
    constexpr int CPL = DK / 32;
    constexpr int KM = KT > 0 ? KT : GDN_MAX_CONV_K;
    const int T = p.T, K = KT > 0 ? KT : p.K;
    const int lane = threadIdx.x & 31;
    ConvCtx x;
    x.xst = xst;
    x.wst = wst;
    x.cstf = reinterpret_cast<const float *>(cst);
    x.q_s = q_s;
    x.k_s = k_s;
    x.v_s = v_s;
    x.kq_s = kq_s;
    x.cc_tok = (size_t)p.C * (K - 1);
    const bool ckpt = p.conv_ckpt != nullptr;
    // q/k channel groups whose conv checkpoints this item writes (bit hf * CPL + e)
    unsigned qk_own = 0;
    if (ckpt && !skip_qk) {
        const int G = p.H_v / p.H_k, nrb = row_blocks(p);
        if (p.steal == 0) {
            const int M = G * nrb, m = (I.h % G) * nrb + I.rb;
            for (int gr = m; gr < 2 * CPL; gr += M) qk_own |= 1u << gr;
        } else if (I.h % G == 0 && I.rb == 0) {
            qk_own = (1u << (2 * CPL)) - 1u;
        }
    }
    x.qk_own = qk_own;
    x.cck = ckpt ? p.conv_ckpt + (size_t)I.by * T * x.cc_tok : nullptr;
    x.gq = (size_t)I.g * DK + lane;                                   // global q channel of this lane's element 0
    x.gk = (size_t)p.H_k * DK + x.gq;                                 // and k channel
    x.gv = 2 * (size_t)p.H_k * DK + (size_t)I.h * p.d_v + I.row0;     // global channel of v row 0
    x.K = K;
    x.lane = lane;
    x.skip_qk = skip_qk;
    for (int t = warp; t < T; t += nwarps) conv_at<DK, BF16, TREE, KT, KM, true, true>(p, I, x, t, src_s);
}

// Warm L2 with item I's inputs: its state rows, x tile (all p.T nodes), conv
// taps and conv state, gates and (tree) parents. Called before the kernel
// waits for the previous grid on the stream: that grid may still be writing
// some of these bytes, which is harmless for a prefetch, and the real loads
// after the wait then hit L2 instead of DRAM.
// with_state false: only the x tile, gates and parents (the rest is being
// loaded already).
template <int DK, bool BF16, bool TREE>
__device__ __forceinline__ void prefetch_l2_item(const VerifyArgs &p, const Item &I, int tid, int nthreads,
                                                 bool with_state = true) {
    constexpr int ES = BF16 ? 2 : 4;
    const int T = p.T, K = p.K;
    const size_t head_off = ((size_t)I.by * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
    if (with_state && GDN_IN(p.ssm_in + head_off, (size_t)I.R * DK * 4, buf_state<DK>(p), p.dev_status))
        prefetch_l2_range(p.ssm_in + head_off, (size_t)I.R * DK * 4, tid, nthreads);
    const size_t c_q = (size_t)I.g * DK, c_k = (size_t)p.H_k * DK + c_q;
    const size_t c_v = 2 * (size_t)p.H_k * DK + (size_t)I.h * p.d_v + I.row0;
    const unsigned char *xg = static_cast<const unsigned char *>(p.x);
    for (int i = tid; i < 3 * T; i += nthreads) {  // (node, channel range) pairs
        const int t = i / 3, r = i - 3 * t;
        const size_t c0 = r == 0 ? c_q : r == 1 ? c_k : c_v;
        const unsigned char *xa = xg + (((size_t)I.by * T + t) * p.C + c0) * ES;
        const size_t xn = (r < 2 ? DK : I.R) * (size_t)ES;
        if (GDN_IN(xa, xn, buf_x<ES>(p), p.dev_status)) prefetch_l2_range(xa, xn, 0, 1);
    }
    const unsigned char *wg = static_cast<const unsigned char *>(p.w);
    const int sub = tid & 31, lanes = 32;  // small ranges: one warp each
    const int w = tid >> 5;
    const int nw = nthreads >> 5;
    for (int r = w; with_state && r < 6; r += nw) {
        const size_t c0 = (r % 3) == 0 ? c_q : (r % 3) == 1 ? c_k : c_v;
        const size_t n = (r % 3) == 2 ? (size_t)I.R : (size_t)DK;
        if (r < 3) {
            if (GDN_IN(wg + ((size_t)I.y * p.C + c0) * K * ES, n * K * ES, buf_w<ES>(p), p.dev_status))
                prefetch_l2_range(wg + ((size_t)I.y * p.C + c0) * K * ES, n * K * ES, sub, lanes);
        } else if (p.conv_in && K > 1) {
            if (GDN_IN(p.conv_in + ((size_t)I.by * p.C + c0) * (K - 1), n * (K - 1) * 4, buf_conv(p), p.dev_status))
                prefetch_l2_range(p.conv_in + ((size_t)I.by * p.C + c0) * (K - 1), n * (K - 1) * 4, sub, lanes);
        }
    }
    if (tid < T) {
        const size_t gi = ((size_t)I.by * T + tid) * p.H_v + I.h;
        if (GDN_IN(static_cast<const unsigned char *>(p.a) + gi * ES, ES, buf_a<ES>(p), p.dev_status))
            prefetch_l2_range(static_cast<const unsigned char *>(p.a) + gi * ES, ES, 0, 1);
        if (GDN_IN(static_cast<const unsigned char *>(p.b) + gi * ES, ES, buf_b<ES>(p), p.dev_status))
            prefetch_l2_range(static_cast<const unsigned char *>(p.b) + gi * ES, ES, 0, 1);
    }
    if constexpr (TREE) {
        if (tid == 0 && GDN_IN(p.parent + (size_t)I.bidx * (T + 1), (size_t)(T + 1) * 4, buf_parent(p), p.dev_status))
            prefetch_l2_range(p.parent + (size_t)I.bidx * (T + 1), (size_t)(T + 1) * 4, 0, 1);
    }
}

// The dynamic shared-memory limit one kernel has been raised to, per device:
// cudaFuncSetAttribute applies to the current device only, so a process that
// drives several GPUs must raise it on each of them.
constexpr int kSmemDevices = 64;
struct SmemSet {
    std::atomic<size_t> v[kSmemDevices];
    SmemSet() {
        for (auto &x : v) x.store(48 * 1024, std::memory_order_relaxed);
    }
};

// Raise a kernel's dynamic shared-memory limit on the current device once per
// size (raising it again is harmless; devices beyond the cache raise it on
// every call).
template <typename K>
bool ensure_smem(K kern, size_t smem, SmemSet &set) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
    const bool cached = dev < kSmemDevices;
    if (cached && smem <= set.v[dev].load(std::memory_order_relaxed)) return true;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return false;
    if (cached) set.v[dev].store(smem, std::memory_order_relaxed);
    return true;
}

VerifyArgs make_args(const gdn_dims *d, int32_t T, const void *x, const void *a, const void *b,
                     const void *w, const float *ssm_in, const float *conv_in, float *ssm_ckpt,
                     float *conv_ckpt, float *out, const int32_t *parent, int32_t *dev_status) {
    VerifyArgs v;
    v.B = d->batch;
    v.Tb = T;
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
    v.steal = 1;
    v.early = 0;
    v.x_ready = nullptr;
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
    const int k = ldic(accept_len + bidx, buf_accept(p), p.dev_status);
    if (c >= p.C || k <= 0 || k > T) return;
    float *cs = conv_state + ((size_t)by * p.C + c) * (K - 1);
    float nw[GDN_MAX_CONV_K];
#pragma unroll
    for (int j = 0; j < GDN_MAX_CONV_K - 1; ++j) {
        nw[j] = 0.f;
        if (j < K - 1) {
            const int sp = k - (K - 1) + j;  // sequence position: x row when >= 0
            nw[j] = sp >= 0 ? ld_inc<BF16>(p.x, ((size_t)by * T + sp) * p.C + c, buf_x<BF16 ? 2 : 4>(p), p.dev_status)
                            : ldfc(cs + (K - 1 + sp), buf_conv(p), p.dev_status);
        }
    }
#pragma unroll
    for (int j = 0; j < GDN_MAX_CONV_K - 1; ++j)
        if (j < K - 1) stfc(cs + j, nw[j], buf_conv(p), p.dev_status);
}

}  // namespace
