// gdn_verify_span / gdn_tree_verify: GDN span verify with per-token F32
// checkpoints, on sm_103a.
//
// What is computed (per request b, layer y, value head h, processed node t):
// causal depthwise conv1d + SiLU over the [q | k | v] channels, per-head L2
// normalisation of q and k, then the gated delta rule
//     S_t = a_t S_p (I - b_t k_t k_t^T) + b_t v_t k_t^T,   o_t = S_t q_t,
// written after every node into an F32 checkpoint slot (lucebox PR #506,
// "perf(dflash): split-chain fast rollback with F32 SSM checkpoints",
// Summary; the pages name the SSM and conv state, lucebox PR #533, Changes).
//
// Design (HBM-write bound: the checkpoints are ~83% of the bytes):
//  * A work item is (request*layer, value head, block of up to 128 value
//    rows). Row i of S only needs k_t, q_t, a_t, b_t and v_t[i], so value
//    rows are independent and S never leaves registers between tokens.
//  * 8 lanes own one 128-float row (16 floats each, as 4 float4 at columns
//    4*j + 32*m), a warp holds 4 rows per "slot" and 4 slots (16 rows).
//    Every checkpoint store is a coalesced st.global.v4: one warp
//    instruction writes four full 128-byte lines.
//  * Both dot products S.k and S.q of the old state reduce together over the
//    8 lanes (3 xor-shuffles each). o_t = a (S_p.q) + c (k.q) with
//    c = b (v - a S_p.k), which equals S_t q_t and needs no second
//    dependent reduction; k.q is computed once per node in the prologue.
//  * Prologue per item: conv + SiLU of the head's 2*d_k q/k channels and its
//    v channels for all nodes into shared memory, L2 norms, gates. The conv
//    checkpoint (the last K-1 inputs) is a shifted copy of the inputs and is
//    written by the item that owns the channels.
//  * Work-stealing kernel (the default): one CTA per item, 2 resident per
//    SM; a running CTA takes the item of a CTA that has not started yet by
//    cancelling that CTA's launch (cluster launch control), so the items run
//    in index order and a CTA on a slow SM simply runs fewer of them. While
//    an item streams its checkpoints, cp.async copies the next item's inputs
//    (x tile, conv taps, conv state) into shared memory and its gates /
//    parent array into registers, so the next prologue is pure on-chip
//    compute; its state loads are issued first and overlap it.
//    Items whose staging does not fit in shared memory (long f32 spans) use
//    the one-item-per-CTA kernel, which loads its inputs directly.
//  * Tree: nodes run in depth-first preorder (children in index order);
//    when a node's parent is not the node just processed, each thread
//    reloads its rows of the parent's checkpoint, which it wrote itself
//    (same thread, same addresses: program order makes it visible; the
//    slot is still in L2). Outputs stay indexed by node.
#include <cuda_runtime.h>

#include <atomic>

#include "gdn_device.cuh"
#include "gdn_host.h"
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
};

// One work item: (request*layer by, value head h, row block rb).
struct Item {
    int by, h, rb, y, bidx, g, row0, R;
};

__device__ __forceinline__ Item decode_item(const VerifyArgs &p, int it, int nrb) {
    Item I;
    I.rb = it % nrb;
    const int r = it / nrb;
    I.h = r % p.H_v;
    I.by = r / p.H_v;
    I.y = I.by % p.Y;
    I.bidx = I.by / p.Y;
    I.g = I.h / (p.H_v / p.H_k);  // key head floor(h * H_k / H_v)
    I.row0 = I.rb * kRowsPerCta;
    I.R = min(kRowsPerCta, p.d_v - I.row0);  // a multiple of kRowsPerWarp
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
        // depth-first preorder of nodes 1..T, children in index order: a
        // node's state is then mostly still in registers when its first
        // child runs, and a parent state is reloaded only on a branch switch
        int *ord_s = par_s + (T + 1);
        int first[GDN_MAX_TOKENS + 1], next[GDN_MAX_TOKENS + 1];
        for (int i = 0; i <= T; ++i) first[i] = next[i] = -1;
        for (int i = T; i >= 1; --i) {
            next[i] = first[par_s[i]];
            first[par_s[i]] = i;
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

// The register-resident state of this thread's rows (4 slots x NV4 float4).
template <int DK>
struct RowState {
    static constexpr int NV4 = DK / (4 * kLanesPerRow);
    float4 S[kSlots][NV4];
    int lrow[kSlots];
};

template <int DK>
__device__ __forceinline__ void load_rows(RowState<DK> &rs, const float *src, bool has_rows) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j8 = lane & (kLanesPerRow - 1), rsub = lane / kLanesPerRow;
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        rs.lrow[s] = warp * kRowsPerWarp + s * kRowsPerSlot + rsub;
#pragma unroll
        for (int m = 0; m < RowState<DK>::NV4; ++m)
            rs.S[s][m] = has_rows ? ld4(src + (size_t)rs.lrow[s] * DK + 4 * j8 + kColStride * m)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// One node t of the recurrence for this thread's rows: one checkpoint slot.
// s_in: the item's initial rows; ck0: slot 0 of the item's rows.
// `prev` is the node whose state the registers hold (0: the initial state).
template <int DK, bool TREE>
__device__ __forceinline__ void recurrence_step(const VerifyArgs &p, RowState<DK> &rs, int t, int prev,
                                               const float *s_in, float *ck0, const float *q_s,
                                               const float *k_s, const float *v_s, float *o_s,
                                               const float *a_s, const float *b_s, const float *kq_s,
                                               const int *par_s) {
    constexpr int NV4 = RowState<DK>::NV4;
    const int lane = threadIdx.x & 31;
    const int j8 = lane & (kLanesPerRow - 1);
    const size_t slot = (size_t)p.H_v * p.d_v * DK;
    if constexpr (TREE) {
        const int pp = par_s[t + 1];
        if (pp != prev) {
            const float *src = pp == 0 ? s_in : ck0 + (size_t)(pp - 1) * slot;
#pragma unroll
            for (int s = 0; s < kSlots; ++s)
#pragma unroll
                for (int m = 0; m < NV4; ++m)
                    rs.S[s][m] = ld4(src + (size_t)rs.lrow[s] * DK + 4 * j8 + kColStride * m);
        }
    }
    float4 kk[NV4], qq[NV4];
#pragma unroll
    for (int m = 0; m < NV4; ++m) {
        kk[m] = ld4(k_s + (size_t)t * DK + 4 * j8 + kColStride * m);
        qq[m] = ld4(q_s + (size_t)t * DK + 4 * j8 + kColStride * m);
    }
    const float at = a_s[t], bt = b_s[t], kqt = kq_s[t];
    float u[kSlots], w[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        u[s] = 0.f;
        w[s] = 0.f;
#pragma unroll
        for (int m = 0; m < NV4; ++m) {
            u[s] = dot4(rs.S[s][m], kk[m], u[s]);
            w[s] = dot4(rs.S[s][m], qq[m], w[s]);
        }
    }
#pragma unroll
    for (int off = 1; off < kLanesPerRow; off <<= 1) {
#pragma unroll
        for (int s = 0; s < kSlots; ++s) {
            u[s] += __shfl_xor_sync(0xffffffffu, u[s], off);
            w[s] += __shfl_xor_sync(0xffffffffu, w[s], off);
        }
    }
    float *ck = ck0 + (size_t)t * slot;
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        const float vv = v_s[(size_t)t * kRowsPerCta + rs.lrow[s]];
        const float c = bt * (vv - at * u[s]);
#pragma unroll
        for (int m = 0; m < NV4; ++m) {
            float4 n;
            n.x = fmaf(c, kk[m].x, at * rs.S[s][m].x);
            n.y = fmaf(c, kk[m].y, at * rs.S[s][m].y);
            n.z = fmaf(c, kk[m].z, at * rs.S[s][m].z);
            n.w = fmaf(c, kk[m].w, at * rs.S[s][m].w);
            rs.S[s][m] = n;
            if (p.ssm_ckpt) st4(ck + (size_t)rs.lrow[s] * DK + 4 * j8 + kColStride * m, n);
        }
        if (j8 == 0) o_s[(size_t)t * kRowsPerCta + rs.lrow[s]] = fmaf(c, kqt, at * w[s]);
    }
}

// The recurrence over all nodes of one item.
template <int DK, bool TREE>
__device__ __forceinline__ void recurrence(const VerifyArgs &p, RowState<DK> &rs, const float *s_in,
                                          float *ck0, const float *q_s, const float *k_s,
                                          const float *v_s, float *o_s, const float *a_s,
                                          const float *b_s, const float *kq_s, const int *par_s) {
    if constexpr (TREE) {
        const int *ord_s = par_s + (p.T + 1);  // depth-first order of the nodes
        int prev = 0;
        for (int q = 0; q < p.T; ++q) {
            const int node = ord_s[q];
            recurrence_step<DK, TREE>(p, rs, node - 1, prev, s_in, ck0, q_s, k_s, v_s, o_s, a_s, b_s, kq_s, par_s);
            prev = node;
        }
    } else {
        for (int t = 0; t < p.T; ++t)
            recurrence_step<DK, TREE>(p, rs, t, t, s_in, ck0, q_s, k_s, v_s, o_s, a_s, b_s, kq_s, par_s);
    }
}

// o of one item, from shared memory [T][kRowsPerCta] to out[b][y][t][h][row]
// with 16-byte stores (d_v, row0 and R are multiples of 16).
__device__ __forceinline__ void write_out(const VerifyArgs &p, const Item &I, const float *o_s, int tid,
                                          int nthreads) {
    const int r4 = I.R / 4;
    for (int i = tid; i < p.T * r4; i += nthreads) {
        const int t = i / r4, r = (i - t * r4) * 4;
        st4(p.out + (((size_t)I.by * p.T + t) * p.H_v + I.h) * p.d_v + I.row0 + r,
            ld4(o_s + (size_t)t * kRowsPerCta + r));
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
// One item per CTA, inputs loaded directly from global memory.
// ---------------------------------------------------------------------------
template <int DK, bool BF16, bool TREE>
__global__ void __launch_bounds__(kThreads, 2) gdn_verify_kernel(const VerifyArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const Layout L = make_layout(p.T, DK, p.K);
    float *q_s = reinterpret_cast<float *>(smem + L.q), *k_s = reinterpret_cast<float *>(smem + L.k);
    float *v_s = reinterpret_cast<float *>(smem + L.v), *o_s = reinterpret_cast<float *>(smem + L.o);
    float *a_s = reinterpret_cast<float *>(smem + L.a), *b_s = reinterpret_cast<float *>(smem + L.b);
    float *kq_s = reinterpret_cast<float *>(smem + L.kq);
    int *par_s = reinterpret_cast<int *>(smem + L.par), *src_s = reinterpret_cast<int *>(smem + L.src);
    const int T = p.T, K = p.K;
    const int nrb = (p.d_v + kRowsPerCta - 1) / kRowsPerCta;
    const Item I = decode_item(p, (blockIdx.z * p.H_v + blockIdx.y) * nrb + blockIdx.x, nrb);
    const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5;
    const void *__restrict__ xin = p.x;

    // the initial state of this thread's rows, loaded first so that its
    // latency overlaps the prologue below
    const bool has_rows = warp * kRowsPerWarp < I.R;
    const size_t head_off = ((size_t)I.by * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
    RowState<DK> rs;
    load_rows<DK>(rs, p.ssm_in + head_off, has_rows);

    if constexpr (TREE) {
        const int32_t *pg = p.parent + (size_t)I.bidx * (T + 1);
        const int pr = tid <= T ? (tid == 0 ? -1 : pg[tid]) : 0;
        tree_tables(p, pg, pr, par_s, src_s, tid, nthreads, 0);
    }
    for (int t = tid; t < T; t += nthreads) {
        const size_t gi = ((size_t)I.by * T + t) * p.H_v + I.h;
        a_s[t] = ld_in<BF16>(p.a, gi);
        b_s[t] = ld_in<BF16>(p.b, gi);
    }
    if constexpr (TREE) __syncthreads();  // src_s ready

    // conv1d + SiLU, one thread per channel; the inputs of a chunk of nodes
    // are loaded together (one memory round trip per chunk)
    {
        const int nch = 2 * DK + I.R;
        const bool own_qk = (I.h % (p.H_v / p.H_k) == 0) && I.rb == 0;
        const size_t x_base = (size_t)I.by * T * p.C;
        const size_t cc_tok = (size_t)p.C * (K - 1);
        for (int lc = tid; lc < nch; lc += nthreads) {
            const int c = item_channel<DK>(p, I, lc);
            float *dst = lc < DK ? q_s + lc : lc < 2 * DK ? k_s + (lc - DK) : v_s + (lc - 2 * DK);
            const int stride = lc < 2 * DK ? DK : kRowsPerCta;
            const bool own = (lc >= 2 * DK || own_qk) && p.conv_ckpt != nullptr;
            float wr[GDN_MAX_CONV_K], st[GDN_MAX_CONV_K];
#pragma unroll
            for (int j = 0; j < GDN_MAX_CONV_K; ++j) {
                wr[j] = j < K ? ld_in<BF16>(p.w, ((size_t)I.y * p.C + c) * K + j) : 0.f;
                st[j] = j < K - 1 ? p.conv_in[((size_t)I.by * p.C + c) * (K - 1) + j] : 0.f;
            }
            float *cck = p.conv_ckpt + (size_t)I.by * T * cc_tok + (size_t)c * (K - 1);
            if constexpr (!TREE) {
                constexpr int CH = 8;
                for (int t0 = 0; t0 < T; t0 += CH) {
                    float xr[CH];
#pragma unroll
                    for (int u = 0; u < CH; ++u)
                        xr[u] = t0 + u < T ? ld_in<BF16>(xin, x_base + (size_t)(t0 + u) * p.C + c) : 0.f;
#pragma unroll
                    for (int u = 0; u < CH; ++u) {
                        const int t = t0 + u;
                        if (t < T) {
                            float win[GDN_MAX_CONV_K];
#pragma unroll
                            for (int j = 0; j < GDN_MAX_CONV_K; ++j) win[j] = j < K - 1 ? st[j] : xr[u];
                            dst[(size_t)t * stride] = conv_out(wr, win, K);
#pragma unroll
                            for (int j = 0; j < GDN_MAX_CONV_K - 1; ++j) {
                                if (j < K - 2) st[j] = st[j + 1];
                                else if (j == K - 2) st[j] = xr[u];
                            }
                            if (own) {
#pragma unroll
                                for (int j = 0; j < GDN_MAX_CONV_K - 1; ++j)
                                    if (j < K - 1) cck[(size_t)t * cc_tok + j] = st[j];
                            }
                        }
                    }
                }
            } else {
                constexpr int CH = 4;
                for (int t0 = 0; t0 < T; t0 += CH) {
                    float wv[CH][GDN_MAX_CONV_K];
#pragma unroll
                    for (int u = 0; u < CH; ++u) {
#pragma unroll
                        for (int j = 0; j < GDN_MAX_CONV_K; ++j) {
                            float v = 0.f;
                            if (t0 + u < T && j < K) {
                                const int s = src_s[(t0 + u) * K + j];
                                if (s >= 1) {
                                    v = ld_in<BF16>(xin, x_base + (size_t)(s - 1) * p.C + c);
                                } else {
                                    const int slot = -1 - s;
#pragma unroll
                                    for (int q = 0; q < GDN_MAX_CONV_K - 1; ++q)
                                        if (q == slot) v = st[q];
                                }
                            }
                            wv[u][j] = v;
                        }
                    }
#pragma unroll
                    for (int u = 0; u < CH; ++u) {
                        const int t = t0 + u;
                        if (t < T) {
                            dst[(size_t)t * stride] = conv_out(wr, wv[u], K);
                            if (own) {
#pragma unroll
                                for (int j = 0; j < GDN_MAX_CONV_K - 1; ++j)
                                    if (j < K - 1) cck[(size_t)t * cc_tok + j] = wv[u][j + 1];
                            }
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    norm_qk<DK>(p, q_s, k_s, kq_s, p.T, threadIdx.x >> 5, blockDim.x >> 5);
    __syncthreads();
    if (has_rows) {
        float *ck0 = p.ssm_ckpt + ((size_t)I.by * T * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
        recurrence<DK, TREE>(p, rs, p.ssm_in + head_off, ck0, q_s, k_s, v_s, o_s, a_s, b_s, kq_s, par_s);
    }
    __syncthreads();
    write_out(p, I, o_s, threadIdx.x, blockDim.x);
}

// ---------------------------------------------------------------------------
// Persistent kernel: CTAs walk the items round-robin and prefetch the next
// item's inputs while the current one streams its checkpoints.
// ---------------------------------------------------------------------------

// Queue the asynchronous copies of item I's x tile, conv taps and conv state
// into the staging buffers (16-byte cp.async; every source and destination
// offset is a multiple of 16 bytes, see the host-side eligibility check).
// with_qk false: the v range only (the q/k of the item are already on chip).
template <int DK, bool BF16>
__device__ __forceinline__ void prefetch_item(const VerifyArgs &p, const Item &I, unsigned char *xst,
                                              unsigned char *wst, unsigned char *cst, bool with_qk, int tid,
                                              int nthreads) {
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
        for (int i = tid; i < T * per_node; i += nthreads) {
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

// Shared-memory carve-up of the persistent kernel: the item's buffers plus
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

// Work-stealing kernel: one CTA per item (grid = n_items); a running CTA
// cancels the launch of the next pending CTA and runs its item, so the items
// run in index order (the CTAs in flight write neighbouring checkpoint rows)
// and the load balances itself across SMs whose store bandwidth differs.
// While an item streams its checkpoints, the next item's inputs are copied
// into the staging buffers, so its prologue is on-chip compute only. When a
// CTA's next item shares the key head of the current one (another value head
// of the GQA group, or another row block), the q/k conv and norms already in
// shared memory are reused: only the v channels are staged and convolved.
//
// KT: the conv width as a compile-time constant (4 for Qwen3.5/3.6), or 0 to
// read it from the arguments.
template <int DK, bool BF16, bool TREE, int KT>
__global__ void __launch_bounds__(kThreads, 2) gdn_verify_persistent(const VerifyArgs p, int n_items) {
    constexpr int ES = BF16 ? 2 : 4;
    extern __shared__ __align__(16) unsigned char smem[];
    const int T = p.T, K = KT > 0 ? KT : p.K;
    const PipeLayout L = make_pipe_layout(T, DK, K, ES);
    float *q_s = reinterpret_cast<float *>(smem + L.q), *k_s = reinterpret_cast<float *>(smem + L.k);
    float *v_s = reinterpret_cast<float *>(smem + L.v), *o_s = reinterpret_cast<float *>(smem + L.o);
    float *a_s = reinterpret_cast<float *>(smem + L.a), *b_s = reinterpret_cast<float *>(smem + L.b);
    float *kq_s = reinterpret_cast<float *>(smem + L.kq);
    int *par_s = reinterpret_cast<int *>(smem + L.par), *src_s = reinterpret_cast<int *>(smem + L.src);
    unsigned char *xst = smem + L.xst, *wst = smem + L.wst, *cst = smem + L.cst;
    const int nrb = (p.d_v + kRowsPerCta - 1) / kRowsPerCta;
    const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5;

    // work stealing: this CTA's own item first, then items of cancelled CTAs
    __shared__ __align__(16) unsigned long long steal_s[3];  // response (16 B), mbarrier
    __shared__ int next_s;
    const unsigned resp = (unsigned)__cvta_generic_to_shared(steal_s);
    const unsigned bar = resp + 16;
    unsigned phase = 0;
    bool stealing = true;  // the last request succeeded
    if (tid == 0) steal_init(bar);
    int it = blockIdx.x;
    if (it >= n_items) return;
    float ga = 0.f, gb = 0.f;
    int pr = 0;
    int tables_of = -1;  // request whose tree tables are in shared memory
    bool reuse_qk = false;  // q_s / k_s / kq_s hold this item's normalised q, k
    {
        const Item I0 = decode_item(p, it, nrb);
        prefetch_item<DK, BF16>(p, I0, xst, wst, cst, true, tid, nthreads);
        prefetch_scalars<BF16, TREE>(p, I0, ga, gb, pr, tid);
    }
    while (true) {
        if (tid == 0 && stealing) steal_issue(resp, bar);  // the next item, answered during this prologue
        const Item I = decode_item(p, it, nrb);
        const bool has_rows = warp * kRowsPerWarp < I.R;
        const size_t head_off = ((size_t)I.by * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
        RowState<DK> rs;
        load_rows<DK>(rs, p.ssm_in + head_off, has_rows);  // overlaps the prologue

        cp_async_wait_all();
        if (tid < T) {
            a_s[tid] = ga;
            b_s[tid] = gb;
        }
        __syncthreads();  // staged inputs and gates visible to every thread
        if constexpr (TREE) {
            if (I.bidx != tables_of) {  // the tables depend on the request only
                tree_tables(p, p.parent + (size_t)I.bidx * (T + 1), pr, par_s, src_s, tid, nthreads, 0);
                __syncthreads();
                tables_of = I.bidx;
            }
        }

        conv_staged<DK, BF16, TREE, KT>(p, I, xst, wst, cst, src_s, q_s, k_s, v_s, reuse_qk, tid, nthreads);
        if (tid == 0) {
            int nx = -1;
            if (stealing) {
                nx = steal_result(resp, bar, phase);
                phase ^= 1u;
                if (nx == -2 && p.dev_status) atomicOr(p.dev_status, GDN_DEV_SCHED);
                if (nx < 0 || nx >= n_items) stealing = false;
            }
            next_s = nx;
        }
        __syncthreads();  // staging consumed; q, k, v ready; next_s set

        const int next = next_s >= 0 && next_s < n_items ? next_s : n_items;
        bool next_reuse = false;
        if (next < n_items) {
            const Item In = decode_item(p, next, nrb);
            next_reuse = In.by == I.by && In.g == I.g;
            prefetch_item<DK, BF16>(p, In, xst, wst, cst, !next_reuse, tid, nthreads);
            prefetch_scalars<BF16, TREE>(p, In, ga, gb, pr, tid);
        }
        if (!reuse_qk) norm_qk<DK>(p, q_s, k_s, kq_s, p.T, threadIdx.x >> 5, blockDim.x >> 5);
        __syncthreads();
        if (has_rows) {
            float *ck0 =
                p.ssm_ckpt + ((size_t)I.by * T * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
            recurrence<DK, TREE>(p, rs, p.ssm_in + head_off, ck0, q_s, k_s, v_s, o_s, a_s, b_s, kq_s, par_s);
        }
        __syncthreads();
        write_out(p, I, o_s, threadIdx.x, blockDim.x);
        if (next >= n_items) break;
        it = next;
        reuse_qk = next_reuse;
    }
}

// ---------------------------------------------------------------------------
// Replay commit: re-run the accepted tokens of a chain from the live state.
// ---------------------------------------------------------------------------

// One item per CTA, like gdn_verify_kernel, over the first Te = accept_len[b]
// tokens only; writes the final rows of S back into the live state. The
// conv window comes from the (not yet updated) live conv state.
template <int DK, bool BF16>
__global__ void __launch_bounds__(kThreads, 2) gdn_replay_kernel(const VerifyArgs p, const int32_t *accept_len) {
    extern __shared__ __align__(16) unsigned char smem[];
    const Layout L = make_layout(p.T, DK, p.K);
    float *q_s = reinterpret_cast<float *>(smem + L.q), *k_s = reinterpret_cast<float *>(smem + L.k);
    float *v_s = reinterpret_cast<float *>(smem + L.v), *o_s = reinterpret_cast<float *>(smem + L.o);
    float *a_s = reinterpret_cast<float *>(smem + L.a), *b_s = reinterpret_cast<float *>(smem + L.b);
    float *kq_s = reinterpret_cast<float *>(smem + L.kq);
    const int T = p.T, K = p.K;
    const int nrb = (p.d_v + kRowsPerCta - 1) / kRowsPerCta;
    const Item I = decode_item(p, (blockIdx.z * p.H_v + blockIdx.y) * nrb + blockIdx.x, nrb);
    const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5;
    const int Te = accept_len[I.bidx];
    if (Te <= 0 || Te > T) {
        if (Te != 0 && p.dev_status && tid == 0 && I.y == 0 && I.h == 0 && I.rb == 0)
            atomicOr(p.dev_status, GDN_DEV_NODE_RANGE);
        return;
    }
    const bool has_rows = warp * kRowsPerWarp < I.R;
    const size_t head_off = ((size_t)I.by * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
    RowState<DK> rs;
    load_rows<DK>(rs, p.ssm_out + head_off, has_rows);
    for (int t = tid; t < Te; t += nthreads) {
        const size_t gi = ((size_t)I.by * T + t) * p.H_v + I.h;
        a_s[t] = ld_in<BF16>(p.a, gi);
        b_s[t] = ld_in<BF16>(p.b, gi);
    }
    {
        const int nch = 2 * DK + I.R;
        const size_t x_base = (size_t)I.by * T * p.C;
        for (int lc = tid; lc < nch; lc += nthreads) {
            const int c = item_channel<DK>(p, I, lc);
            float *dst = lc < DK ? q_s + lc : lc < 2 * DK ? k_s + (lc - DK) : v_s + (lc - 2 * DK);
            const int stride = lc < 2 * DK ? DK : kRowsPerCta;
            float wr[GDN_MAX_CONV_K], st[GDN_MAX_CONV_K];
#pragma unroll
            for (int j = 0; j < GDN_MAX_CONV_K; ++j) {
                wr[j] = j < K ? ld_in<BF16>(p.w, ((size_t)I.y * p.C + c) * K + j) : 0.f;
                st[j] = j < K - 1 ? p.conv_in[((size_t)I.by * p.C + c) * (K - 1) + j] : 0.f;
            }
            constexpr int CH = 8;
            for (int t0 = 0; t0 < Te; t0 += CH) {
                float xr[CH];
#pragma unroll
                for (int u = 0; u < CH; ++u)
                    xr[u] = t0 + u < Te ? ld_in<BF16>(p.x, x_base + (size_t)(t0 + u) * p.C + c) : 0.f;
#pragma unroll
                for (int u = 0; u < CH; ++u) {
                    const int t = t0 + u;
                    if (t < Te) {
                        float win[GDN_MAX_CONV_K];
#pragma unroll
                        for (int j = 0; j < GDN_MAX_CONV_K; ++j) win[j] = j < K - 1 ? st[j] : xr[u];
                        dst[(size_t)t * stride] = conv_out(wr, win, K);
#pragma unroll
                        for (int j = 0; j < GDN_MAX_CONV_K - 1; ++j) {
                            if (j < K - 2) st[j] = st[j + 1];
                            else if (j == K - 2) st[j] = xr[u];
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    norm_qk<DK>(p, q_s, k_s, kq_s, Te, threadIdx.x >> 5, blockDim.x >> 5);
    __syncthreads();
    if (has_rows) {
        const float *s_in = p.ssm_out + head_off;
        for (int t = 0; t < Te; ++t)
            recurrence_step<DK, false>(p, rs, t, t, s_in, nullptr, q_s, k_s, v_s, o_s, a_s, b_s, kq_s, nullptr);
        const int lane = tid & 31, j8 = lane & (kLanesPerRow - 1);
#pragma unroll
        for (int s2 = 0; s2 < kSlots; ++s2)
#pragma unroll
            for (int m = 0; m < RowState<DK>::NV4; ++m)
                st4(p.ssm_out + head_off + (size_t)rs.lrow[s2] * DK + 4 * j8 + kColStride * m, rs.S[s2][m]);
    }
}

// The live conv state after the replayed tokens: the last K-1 inputs of
// [conv_state, x_0 .. x_{k-1}], one thread per channel (reads before writes).
template <bool BF16>
__global__ void __launch_bounds__(256) gdn_conv_state_kernel(const VerifyArgs p, const int32_t *accept_len,
                                                            float *conv_state) {
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

template <int DK, bool BF16, bool TREE>
int launch_verify(const VerifyArgs &a, int batch, bool aligned_inputs, cudaStream_t stream) {
    const int nrb = (a.d_v + kRowsPerCta - 1) / kRowsPerCta;
    const int n_items = batch * a.Y * a.H_v * nrb;
    const int rows = a.d_v < kRowsPerCta ? a.d_v : kRowsPerCta;  // d_v % kRowsPerWarp == 0
    const int threads = rows / kRowsPerWarp * 32;
    const PipeLayout Lp = make_pipe_layout(a.T, DK, a.K, BF16 ? 2 : 4);
    // the persistent kernel keeps one gate / parent value per thread in registers
    if (aligned_inputs && Lp.total + kStaticSmem <= kMaxSmem && threads > a.T) {
        auto kern = a.K == 4 ? gdn_verify_persistent<DK, BF16, TREE, 4> : gdn_verify_persistent<DK, BF16, TREE, 0>;
        static std::atomic<size_t> set4{48 * 1024}, set0{48 * 1024};
        std::atomic<size_t> &set = a.K == 4 ? set4 : set0;
        if (!ensure_smem(kern, Lp.total, set)) return GDN_ERR_CUDA;
        // one CTA per item: the running CTAs take the pending ones' items
        const int grid = n_items;
        kern<<<grid, threads, Lp.total, stream>>>(a, n_items);
    } else {
        auto kern = gdn_verify_kernel<DK, BF16, TREE>;
        static std::atomic<size_t> set{48 * 1024};
        const Layout L = make_layout(a.T, DK, a.K);
        if (!ensure_smem(kern, L.total, set)) return GDN_ERR_CUDA;
        dim3 grid(nrb, a.H_v, batch * a.Y);
        kern<<<grid, threads, L.total, stream>>>(a);
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <bool TREE>
int dispatch_verify(const gdn_dims *d, const VerifyArgs &a, cudaStream_t stream) {
    const bool bf = d->in_dtype == GDN_BF16;
    // cp.async staging needs 16-byte aligned x and conv taps (the offsets it
    // copies from are then multiples of 16 bytes: C, d_k and every row block
    // are multiples of 16 channels)
    const bool al = gdnhost::aligned16(a.x) && gdnhost::aligned16(a.w);
    if (d->d_k == 128)
        return bf ? launch_verify<128, true, TREE>(a, d->batch, al, stream)
                  : launch_verify<128, false, TREE>(a, d->batch, al, stream);
    return bf ? launch_verify<64, true, TREE>(a, d->batch, al, stream)
              : launch_verify<64, false, TREE>(a, d->batch, al, stream);
}

int check_common(const gdn_dims *d, int32_t n_tok, const void *x, const void *a, const void *b,
                 const void *w, const float *ssm_in, const float *conv_in, float *ssm_ckpt,
                 float *conv_ckpt, float *out) {
    int rc = gdnhost::check_dims(d, n_tok);
    if (rc != GDN_OK) return rc;
    if (!x || !a || !b || !w || !ssm_in || !ssm_ckpt || !out) return GDN_ERR_NULL;
    if (d->conv_k > 1 && (!conv_in || !conv_ckpt)) return GDN_ERR_NULL;
    const size_t es = d->in_dtype == GDN_BF16 ? 2 : 4;
    using gdnhost::aligned16;
    using gdnhost::aligned_to;
    if (!aligned_to(x, es) || !aligned_to(a, es) || !aligned_to(b, es) || !aligned_to(w, es))
        return GDN_ERR_ALIGN;
    if (!aligned16(ssm_in) || !aligned16(ssm_ckpt) || !aligned16(out)) return GDN_ERR_ALIGN;
    if (d->conv_k > 1 && (!aligned16(conv_in) || !aligned16(conv_ckpt))) return GDN_ERR_ALIGN;
    return GDN_OK;
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
    return v;
}

}  // namespace

extern "C" int gdn_verify_span(const gdn_dims *d, int32_t n_tok, const void *x, const void *a,
                               const void *b, const void *conv_w, const float *ssm_in,
                               const float *conv_in, float *ssm_ckpt, float *conv_ckpt, float *out,
                               int32_t *dev_status, gdn_stream_t stream) {
    int rc = check_common(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt, out);
    if (rc != GDN_OK) return rc;
    if (dev_status && !gdnhost::aligned_to(dev_status, 4)) return GDN_ERR_ALIGN;
    const VerifyArgs v = make_args(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt,
                                   out, nullptr, dev_status);
    return dispatch_verify<false>(d, v, static_cast<cudaStream_t>(stream));
}

extern "C" int gdn_tree_verify(const gdn_dims *d, int32_t n_nodes, const int32_t *parent_host,
                               const int32_t *parent_dev, const void *x, const void *a,
                               const void *b, const void *conv_w, const float *ssm_in,
                               const float *conv_in, float *ssm_ckpt, float *conv_ckpt,
                               float *out, int32_t *dev_status, gdn_stream_t stream) {
    if (!d) return GDN_ERR_NULL;
    if (n_nodes < 2) return GDN_ERR_TREE_TRUNCATED;
    int rc = check_common(d, n_nodes - 1, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt, out);
    if (rc != GDN_OK) return rc;
    if (!parent_host || !parent_dev) return GDN_ERR_NULL;
    if (!gdnhost::aligned_to(parent_dev, 4) || (dev_status && !gdnhost::aligned_to(dev_status, 4)))
        return GDN_ERR_ALIGN;
    rc = gdnhost::check_tree(parent_host, d->batch, n_nodes, false, 0);
    if (rc != GDN_OK) return rc;
    const VerifyArgs v = make_args(d, n_nodes - 1, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt,
                                   conv_ckpt, out, parent_dev, dev_status);
    return dispatch_verify<true>(d, v, static_cast<cudaStream_t>(stream));
}

extern "C" int gdn_verify_span_nockpt(const gdn_dims *d, int32_t n_tok, const void *x, const void *a,
                                      const void *b, const void *conv_w, const float *ssm_in,
                                      const float *conv_in, float *out, int32_t *dev_status,
                                      gdn_stream_t stream) {
    int rc = gdnhost::check_dims(d, n_tok);
    if (rc != GDN_OK) return rc;
    if (!x || !a || !b || !conv_w || !ssm_in || !out) return GDN_ERR_NULL;
    if (d->conv_k > 1 && !conv_in) return GDN_ERR_NULL;
    const size_t es = d->in_dtype == GDN_BF16 ? 2 : 4;
    using gdnhost::aligned16;
    using gdnhost::aligned_to;
    if (!aligned_to(x, es) || !aligned_to(a, es) || !aligned_to(b, es) || !aligned_to(conv_w, es))
        return GDN_ERR_ALIGN;
    if (!aligned16(ssm_in) || !aligned16(out) || (d->conv_k > 1 && !aligned16(conv_in))) return GDN_ERR_ALIGN;
    if (dev_status && !aligned_to(dev_status, 4)) return GDN_ERR_ALIGN;
    const VerifyArgs v = make_args(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, nullptr, nullptr, out,
                                   nullptr, dev_status);
    return dispatch_verify<false>(d, v, static_cast<cudaStream_t>(stream));
}

extern "C" int gdn_commit_replay(const gdn_dims *d, int32_t n_tok, const int32_t *accept_len_dev,
                                 const void *x, const void *a, const void *b, const void *conv_w,
                                 float *ssm_state, float *conv_state, int32_t *dev_status,
                                 gdn_stream_t stream) {
    int rc = gdnhost::check_dims(d, n_tok);
    if (rc != GDN_OK) return rc;
    if (!accept_len_dev || !x || !a || !b || !conv_w || !ssm_state) return GDN_ERR_NULL;
    if (d->conv_k > 1 && !conv_state) return GDN_ERR_NULL;
    const size_t es = d->in_dtype == GDN_BF16 ? 2 : 4;
    using gdnhost::aligned16;
    using gdnhost::aligned_to;
    if (!aligned_to(x, es) || !aligned_to(a, es) || !aligned_to(b, es) || !aligned_to(conv_w, es) ||
        !aligned_to(accept_len_dev, 4) || (dev_status && !aligned_to(dev_status, 4)))
        return GDN_ERR_ALIGN;
    if (!aligned16(ssm_state) || (d->conv_k > 1 && !aligned16(conv_state))) return GDN_ERR_ALIGN;
    VerifyArgs v = make_args(d, n_tok, x, a, b, conv_w, ssm_state, conv_state, nullptr, nullptr, nullptr,
                             nullptr, dev_status);
    v.ssm_out = ssm_state;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int nrb = (d->d_v + kRowsPerCta - 1) / kRowsPerCta;
    const int rows = d->d_v < kRowsPerCta ? d->d_v : kRowsPerCta;
    const int threads = rows / kRowsPerWarp * 32;
    const Layout L = make_layout(n_tok, d->d_k, d->conv_k);
    const dim3 grid(nrb, d->h_v, d->batch * d->layers);
    const bool bf = d->in_dtype == GDN_BF16;
    if (d->d_k == 128) {
        auto kern = bf ? gdn_replay_kernel<128, true> : gdn_replay_kernel<128, false>;
        static std::atomic<size_t> set_b{48 * 1024}, set_f{48 * 1024};
        if (!ensure_smem(kern, L.total, bf ? set_b : set_f)) return GDN_ERR_CUDA;
        kern<<<grid, threads, L.total, st>>>(v, accept_len_dev);
    } else {
        auto kern = bf ? gdn_replay_kernel<64, true> : gdn_replay_kernel<64, false>;
        static std::atomic<size_t> set_b{48 * 1024}, set_f{48 * 1024};
        if (!ensure_smem(kern, L.total, bf ? set_b : set_f)) return GDN_ERR_CUDA;
        kern<<<grid, threads, L.total, st>>>(v, accept_len_dev);
    }
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    if (d->conv_k > 1) {
        const dim3 g2((d->conv_ch + 255) / 256, d->batch * d->layers);
        if (bf) gdn_conv_state_kernel<true><<<g2, 256, 0, st>>>(v, accept_len_dev, conv_state);
        else gdn_conv_state_kernel<false><<<g2, 256, 0, st>>>(v, accept_len_dev, conv_state);
        if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    }
    return GDN_OK;
}
