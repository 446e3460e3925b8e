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
//  * Small launches (one layer at a time) split heads into blocks of down to
//    32 rows and hold 4 rows per warp instead of 16, so that the GPU's SMs
//    and each CTA's warps all get rows.
//  * Kernels are launched with programmatic dependent launch: each waits
//    (griddepcontrol.wait) for the previous kernel on the stream before its
//    first global access, so its launch overlaps that kernel's tail.
//  * Tree: nodes run in depth-first preorder, children in ascending order of
//    subtree size. When a node's parent is not the node just processed, each
//    thread reloads its rows of the parent's checkpoint, which it wrote
//    itself (same thread, same addresses: program order makes it visible;
//    the order keeps the slot in L2). The root's rows, needed again by its
//    later children, are parked in tensor memory (each thread's own lane)
//    instead of being re-read from DRAM. Outputs stay indexed by node.
#include <cuda_runtime.h>

#include <atomic>

#include "gdn_device.cuh"
#include "gdn_host.h"
#include "gdn_tc.cuh"
#include "gdn_verify_parts.cuh"
#include "gdnspec.h"

namespace {


// The register-resident state of this thread's rows (SL slots x NV4 float4;
// a warp holds 4 * SL rows). SL = 4 (16 rows per warp) is the default; small
// launches use SL = 1 so that a head's few rows spread over more warps.
template <int DK, int SL = kSlots>
struct RowState {
    static constexpr int NV4 = DK / (4 * kLanesPerRow);
    static constexpr int kRows = kRowsPerSlot * SL;  // rows per warp
    static constexpr int kWords = SL * NV4 * 4;       // floats of state per thread
    float4 S[SL][NV4];
    int lrow[SL];
};

template <int DK, int SL>
__device__ __forceinline__ void load_rows(const VerifyArgs &p, RowState<DK, SL> &rs, const float *src, bool has_rows) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int j8 = lane & (kLanesPerRow - 1), rsub = lane / kLanesPerRow;
#pragma unroll
    for (int s = 0; s < SL; ++s) {
        rs.lrow[s] = warp * RowState<DK, SL>::kRows + s * kRowsPerSlot + rsub;
#pragma unroll
        for (int m = 0; m < RowState<DK, SL>::NV4; ++m)
            rs.S[s][m] = has_rows ? ld4c(src + (size_t)rs.lrow[s] * DK + 4 * j8 + kColStride * m, buf_state<DK>(p),
                                         p.dev_status)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// Trees park the state of a branch point (the initial rows, or a node with
// children still to run) in tensor memory, so that its later children
// restart from there instead of from its checkpoint. Slot k of a thread's
// rows: its own lane, columns from 2 k kWords (warps 4..7 after those of
// warps 0..3). Warp-collective.
template <int DK, int SL>
__device__ __forceinline__ unsigned park_addr(unsigned tmem, int slot) {
    const int warp = threadIdx.x >> 5;
    constexpr int W = RowState<DK, SL>::kWords;
    return tmem + ((unsigned)(32 * (warp & 3)) << 16) + (unsigned)((2 * slot + (warp >> 2)) * W);
}

template <int DK, int SL>
__device__ __forceinline__ void park_rows(const RowState<DK, SL> &rs, unsigned tmem, int slot) {
    constexpr int NV4 = RowState<DK, SL>::NV4;
    static_assert((SL * NV4) % 2 == 0, "8 words per tensor-memory store");
    const unsigned base = park_addr<DK, SL>(tmem, slot);
#pragma unroll
    for (int k = 0; k < SL * NV4; k += 2) {
        const float4 x = rs.S[k / NV4][k % NV4], y = rs.S[(k + 1) / NV4][(k + 1) % NV4];
        const unsigned v[8] = {__float_as_uint(x.x), __float_as_uint(x.y), __float_as_uint(x.z), __float_as_uint(x.w),
                               __float_as_uint(y.x), __float_as_uint(y.y), __float_as_uint(y.z), __float_as_uint(y.w)};
        gdntc::tmem_st8(base + (unsigned)(4 * k), v);
    }
    gdntc::tmem_wait_st();
}

template <int DK, int SL>
__device__ __forceinline__ void fetch_rows(RowState<DK, SL> &rs, unsigned tmem, int slot) {
    constexpr int NV4 = RowState<DK, SL>::NV4;
    const unsigned base = park_addr<DK, SL>(tmem, slot);
#pragma unroll
    for (int k = 0; k < SL * NV4; k += 2) {
        unsigned v[8];
        gdntc::tmem_ld8(base + (unsigned)(4 * k), v);
        gdntc::tmem_wait_ld();
        rs.S[k / NV4][k % NV4] = make_float4(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]),
                                             __uint_as_float(v[3]));
        rs.S[(k + 1) / NV4][(k + 1) % NV4] = make_float4(__uint_as_float(v[4]), __uint_as_float(v[5]),
                                                         __uint_as_float(v[6]), __uint_as_float(v[7]));
    }
}

// One node t of the recurrence for this thread's rows (whose registers hold
// the state of the node's parent): one checkpoint slot.
// ck0: slot 0 of the item's rows.
template <int DK, int SL>
__device__ __forceinline__ void recurrence_step(const VerifyArgs &p, RowState<DK, SL> &rs, int t, float *ck0,
                                               const float *q_s, const float *k_s, const float *v_s,
                                               float *o_s, const float *a_s, const float *b_s,
                                               const float *kq_s) {
    constexpr int NV4 = RowState<DK, SL>::NV4;
    const int lane = threadIdx.x & 31;
    const int j8 = lane & (kLanesPerRow - 1);
    const size_t slot = (size_t)p.H_v * p.d_v * DK;
    float4 kk[NV4], qq[NV4];
#pragma unroll
    for (int m = 0; m < NV4; ++m) {
        kk[m] = ld4(k_s + (size_t)t * DK + 4 * j8 + kColStride * m);
        qq[m] = ld4(q_s + (size_t)t * DK + 4 * j8 + kColStride * m);
    }
    const float at = a_s[t], bt = b_s[t], kqt = kq_s[t];
    float u[SL], w[SL];
#pragma unroll
    for (int s = 0; s < SL; ++s) {
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
        for (int s = 0; s < SL; ++s) {
            u[s] += __shfl_xor_sync(0xffffffffu, u[s], off);
            w[s] += __shfl_xor_sync(0xffffffffu, w[s], off);
        }
    }
    float *ck = ck0 + (size_t)t * slot;
#pragma unroll
    for (int s = 0; s < SL; ++s) {
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
            if (p.ssm_ckpt) st4c(ck + (size_t)rs.lrow[s] * DK + 4 * j8 + kColStride * m, n, buf_ckpt<DK>(p), p.dev_status);
        }
        if (j8 == 0) o_s[(size_t)t * kRowsPerCta + rs.lrow[s]] = fmaf(c, kqt, at * w[s]);
    }
}

// The operands of one node's step for this thread's rows: k and q (this
// lane's columns), the gates, k.q and v of the rows.
template <int DK, int SL>
struct StepIn {
    float4 kk[RowState<DK, SL>::NV4], qq[RowState<DK, SL>::NV4];
    float at, bt, kqt, vv[SL];
};

template <int DK, int SL>
__device__ __forceinline__ void load_step(StepIn<DK, SL> &in, const RowState<DK, SL> &rs, int t, const float *q_s,
                                          const float *k_s, const float *v_s, const float *a_s, const float *b_s,
                                          const float *kq_s) {
    const int j8 = (threadIdx.x & 31) & (kLanesPerRow - 1);
#pragma unroll
    for (int m = 0; m < RowState<DK, SL>::NV4; ++m) {
        in.kk[m] = ld4(k_s + (size_t)t * DK + 4 * j8 + kColStride * m);
        in.qq[m] = ld4(q_s + (size_t)t * DK + 4 * j8 + kColStride * m);
    }
    in.at = a_s[t];
    in.bt = b_s[t];
    in.kqt = kq_s[t];
#pragma unroll
    for (int s = 0; s < SL; ++s) in.vv[s] = v_s[(size_t)t * kRowsPerCta + rs.lrow[s]];
}

// recurrence_step with the operands of node t already in `in`; the next
// node's (tn >= 0) are loaded into `in` as soon as node t's dot products are
// reduced, ahead of t's checkpoint stores, so that they do not queue behind
// those stores. The arithmetic is recurrence_step's, operation for operation.
template <int DK, int SL>
__device__ __forceinline__ void recurrence_step_ahead(const VerifyArgs &p, RowState<DK, SL> &rs, StepIn<DK, SL> &in,
                                                      int t, int tn, float *ck0, const float *q_s, const float *k_s,
                                                      const float *v_s, float *o_s, const float *a_s,
                                                      const float *b_s, const float *kq_s) {
    constexpr int NV4 = RowState<DK, SL>::NV4;
    const int j8 = (threadIdx.x & 31) & (kLanesPerRow - 1);
    const size_t slot = (size_t)p.H_v * p.d_v * DK;
    float u[SL], w[SL];
#pragma unroll
    for (int s = 0; s < SL; ++s) {
        u[s] = 0.f;
        w[s] = 0.f;
#pragma unroll
        for (int m = 0; m < NV4; ++m) {
            u[s] = dot4(rs.S[s][m], in.kk[m], u[s]);
            w[s] = dot4(rs.S[s][m], in.qq[m], w[s]);
        }
    }
#pragma unroll
    for (int off = 1; off < kLanesPerRow; off <<= 1) {
#pragma unroll
        for (int s = 0; s < SL; ++s) {
            u[s] += __shfl_xor_sync(0xffffffffu, u[s], off);
            w[s] += __shfl_xor_sync(0xffffffffu, w[s], off);
        }
    }
    const float at = in.at, bt = in.bt, kqt = in.kqt;
    float c[SL];
#pragma unroll
    for (int s = 0; s < SL; ++s) c[s] = bt * (in.vv[s] - at * u[s]);
    float4 kk[NV4];
#pragma unroll
    for (int m = 0; m < NV4; ++m) kk[m] = in.kk[m];
    if (tn >= 0) load_step(in, rs, tn, q_s, k_s, v_s, a_s, b_s, kq_s);
    float *ck = ck0 + (size_t)t * slot;
#pragma unroll
    for (int s = 0; s < SL; ++s) {
#pragma unroll
        for (int m = 0; m < NV4; ++m) {
            float4 n;
            n.x = fmaf(c[s], kk[m].x, at * rs.S[s][m].x);
            n.y = fmaf(c[s], kk[m].y, at * rs.S[s][m].y);
            n.z = fmaf(c[s], kk[m].z, at * rs.S[s][m].z);
            n.w = fmaf(c[s], kk[m].w, at * rs.S[s][m].w);
            rs.S[s][m] = n;
            if (p.ssm_ckpt) st4c(ck + (size_t)rs.lrow[s] * DK + 4 * j8 + kColStride * m, n, buf_ckpt<DK>(p), p.dev_status);
        }
        if (j8 == 0) o_s[(size_t)t * kRowsPerCta + rs.lrow[s]] = fmaf(c[s], kqt, at * w[s]);
    }
}

// The recurrence over all nodes of one item. Trees run the nodes in the
// depth-first order of the tree tables and follow their reload plan: a
// node whose parent is not the node just computed takes the parent's state
// from its tensor-memory slot (PARK, the plan's slots were sized for
// `tmem`), or from its checkpoint (the same thread wrote those addresses:
// program order makes them visible), or from the initial rows; a branch
// point is parked after its step.
template <int DK, bool TREE, int SL, bool PARK = false>
__device__ __forceinline__ void recurrence(const VerifyArgs &p, RowState<DK, SL> &rs, const float *s_in,
                                          float *ck0, const float *q_s, const float *k_s,
                                          const float *v_s, float *o_s, const float *a_s,
                                          const float *b_s, const float *kq_s, const int *par_s,
                                          unsigned tmem = 0) {
    if constexpr (TREE) {
        constexpr int NV4 = RowState<DK, SL>::NV4;
        const int j8 = (threadIdx.x & 31) & (kLanesPerRow - 1);
        const size_t slot = (size_t)p.H_v * p.d_v * DK;
        const int *ord_s = par_s + (p.T + 1);  // depth-first order of the nodes
        const int *plan_s = ord_s + p.T;
        if constexpr (PARK) {
            const int root_slot = plan_s[p.T];
            if (root_slot >= 0) park_rows(rs, tmem, root_slot);  // the item's initial loads have landed by now
        }
        // each node's order and plan entries are read one node ahead, before
        // the stores of the node in hand
        int node_n = p.T > 0 ? ord_s[0] : 0, pl_n = p.T > 0 ? plan_s[0] : 0;
        for (int q = 0; q < p.T; ++q) {
            const int node = node_n, pl = pl_n;
            if (q + 1 < p.T) {
                node_n = ord_s[q + 1];
                pl_n = plan_s[q + 1];
            }
            const int src = (int)(short)(pl & 0xffff), park = pl >> 16;
            if (src >= 0) {
                if constexpr (PARK) fetch_rows(rs, tmem, src);
            } else if (src == -2) {
                const int pp = par_s[node];
                const float *from = pp == 0 ? s_in : ck0 + (size_t)(pp - 1) * slot;
                const Buf fb = pp == 0 ? buf_state<DK>(p) : buf_ckpt<DK>(p);
#pragma unroll
                for (int s = 0; s < SL; ++s)
#pragma unroll
                    for (int m = 0; m < NV4; ++m)
                        rs.S[s][m] = ld4c(from + (size_t)rs.lrow[s] * DK + 4 * j8 + kColStride * m, fb, p.dev_status);
            }
            recurrence_step<DK, SL>(p, rs, node - 1, ck0, q_s, k_s, v_s, o_s, a_s, b_s, kq_s);
            if constexpr (PARK) {
                if (park >= 0) park_rows(rs, tmem, park);
            }
        }
    } else if constexpr (SL <= 2) {
        // few rows per thread leave registers for the next node's operands
        // (not in the tree loop: measured slower there, where parks and
        // reloads sit between the steps)
        StepIn<DK, SL> in;
        if (p.T > 0) load_step(in, rs, 0, q_s, k_s, v_s, a_s, b_s, kq_s);
        for (int t = 0; t < p.T; ++t)
            recurrence_step_ahead<DK, SL>(p, rs, in, t, t + 1 < p.T ? t + 1 : -1, ck0, q_s, k_s, v_s, o_s, a_s, b_s,
                                          kq_s);
    } else {
        for (int t = 0; t < p.T; ++t) recurrence_step<DK, SL>(p, rs, t, ck0, q_s, k_s, v_s, o_s, a_s, b_s, kq_s);
    }
}

// o of one item, from shared memory [T][kRowsPerCta] to out[b][y][t][h][row]
// with 16-byte stores (d_v, row0 and R are multiples of 16).
__device__ __forceinline__ void write_out(const VerifyArgs &p, const Item &I, const float *o_s, int tid,
                                          int nthreads) {
    const int r4 = I.R / 4;
    for (int i = tid; i < p.T * r4; i += nthreads) {
        const int t = i / r4, r = (i - t * r4) * 4;
        st4c(p.out + (((size_t)I.by * p.T + t) * p.H_v + I.h) * p.d_v + I.row0 + r,
             ld4(o_s + (size_t)t * kRowsPerCta + r), buf_out(p), p.dev_status);
    }
}


// ---------------------------------------------------------------------------
// One item per CTA, inputs loaded directly from global memory.
// ---------------------------------------------------------------------------
template <int DK, bool BF16, bool TREE>
__global__ void __launch_bounds__(kThreads, 2) gdn_verify_kernel(const VerifyArgs p) {
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smem[];
    const Layout L = make_layout(p.T, DK, p.K);
    float *q_s = reinterpret_cast<float *>(smem + L.q), *k_s = reinterpret_cast<float *>(smem + L.k);
    float *v_s = reinterpret_cast<float *>(smem + L.v), *o_s = reinterpret_cast<float *>(smem + L.o);
    float *a_s = reinterpret_cast<float *>(smem + L.a), *b_s = reinterpret_cast<float *>(smem + L.b);
    float *kq_s = reinterpret_cast<float *>(smem + L.kq);
    int *par_s = reinterpret_cast<int *>(smem + L.par), *src_s = reinterpret_cast<int *>(smem + L.src);
    const int T = p.T, K = p.K;
    const int nrb = row_blocks(p);
    const Item I = decode_item(p, (blockIdx.z * p.H_v + blockIdx.y) * nrb + blockIdx.x, nrb);
    const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5;
    const void *__restrict__ xin = p.x;
    wait_ready(p, I.by);  // inputs landing during the launch: this item's x, a, b rows

    // the initial state of this thread's rows, loaded first so that its
    // latency overlaps the prologue below
    const bool has_rows = warp * kRowsPerWarp < I.R;
    const size_t head_off = ((size_t)I.by * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
    RowState<DK> rs;
    load_rows<DK>(p, rs, p.ssm_in + head_off, has_rows);

    if constexpr (TREE) {
        const int32_t *pg = p.parent + (size_t)I.bidx * (T + 1);
        const int pr = tid <= T ? (tid == 0 ? -1 : ldic(pg + tid, buf_parent(p), p.dev_status)) : 0;
        tree_tables(p, pg, pr, par_s, src_s, tid, nthreads, 0);
    }
    for (int t = tid; t < T; t += nthreads) {
        const size_t gi = ((size_t)I.by * T + t) * p.H_v + I.h;
        a_s[t] = ld_inc<BF16>(p.a, gi, buf_a<BF16 ? 2 : 4>(p), p.dev_status);
        b_s[t] = ld_inc<BF16>(p.b, gi, buf_b<BF16 ? 2 : 4>(p), p.dev_status);
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
                wr[j] = j < K ? ld_inc<BF16>(p.w, ((size_t)I.y * p.C + c) * K + j, buf_w<BF16 ? 2 : 4>(p), p.dev_status)
                              : 0.f;
                st[j] = j < K - 1 ? ldfc(p.conv_in + ((size_t)I.by * p.C + c) * (K - 1) + j, buf_conv(p), p.dev_status)
                                  : 0.f;
            }
            float *cck = p.conv_ckpt + (size_t)I.by * T * cc_tok + (size_t)c * (K - 1);
            if constexpr (!TREE) {
                constexpr int CH = 8;
                for (int t0 = 0; t0 < T; t0 += CH) {
                    float xr[CH];
#pragma unroll
                    for (int u = 0; u < CH; ++u)
                        xr[u] = t0 + u < T ? ld_inc<BF16>(xin, x_base + (size_t)(t0 + u) * p.C + c,
                                                          buf_x<BF16 ? 2 : 4>(p), p.dev_status)
                                           : 0.f;
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
                                    if (j < K - 1) stfc(cck + (size_t)t * cc_tok + j, st[j], buf_cckpt(p), p.dev_status);
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
                                    v = ld_inc<BF16>(xin, x_base + (size_t)(s - 1) * p.C + c, buf_x<BF16 ? 2 : 4>(p),
                                                     p.dev_status);
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
                                    if (j < K - 1)
                                        stfc(cck + (size_t)t * cc_tok + j, wv[u][j + 1], buf_cckpt(p), p.dev_status);
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
//
// SL: slots of 4 rows per warp in the recurrence (4 by default, 1 for small
// launches, whose items have few rows).
//
// RP (chains): the replay commit. An item runs only the first
// k = accept_len[request] tokens, from the live state, without checkpoints
// or outputs, and writes its rows' final state back over the live state
// (k = 0: untouched). The staged prologue then covers those k tokens only.
template <int DK, bool BF16, bool TREE, int KT, int SL, bool RP = false>
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
    const int nrb = row_blocks(p);
    const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5;

    // work stealing: this CTA's own item first, then items of cancelled CTAs
    __shared__ __align__(16) unsigned long long steal_s[3];  // response (16 B), mbarrier
    __shared__ int next_s;
    __shared__ int next_ready_s;  // the next item's inputs have landed (x_ready), or need no wait
    __shared__ unsigned park_s;  // tensor-memory columns of the parked branch points (trees)
    // Tree branch points are parked in tensor memory: 2 states of 16 rows
    // per warp (2 x 128 columns at d_k = 128, half of the SM's 512 for each
    // of its 2 CTAs), 4 of 4 rows per warp (small launches). Two slots take
    // all but ~0.4 % of the reloads of the random 23-node trees of the
    // DDTree workload; the rest read the checkpoint.
    constexpr bool kPark = TREE;
    constexpr int kParkSlots = SL == kSlots ? 2 : 4;
    constexpr int kParkWant = kParkSlots * 2 * RowState<DK, SL>::kWords;
    constexpr int kParkCols = kParkWant <= 32 ? 32 : kParkWant <= 64 ? 64 : kParkWant <= 128 ? 128 : 256;
    static_assert(kParkWant <= 256, "two CTAs per SM share its 512 tensor-memory columns");
    const unsigned resp = (unsigned)__cvta_generic_to_shared(steal_s);
    const unsigned bar = resp + 16;
    unsigned phase = 0;
    bool stealing = p.steal != 0;  // the last request succeeded (or: the host found every CTA resident)
    if (tid == 0) steal_init(bar);
    int it = blockIdx.x;
    if (it >= n_items) return;
    const Item I0 = decode_item(p, it, nrb);
    RowState<DK, SL> rs;
    unsigned ga = 0u, gb = 0u;  // raw gates of the staged item
    int pr = 0;
    int tables_of = -1;  // request whose tree tables are in shared memory
    // Before the wait for the previous grid on the stream: with the caller's
    // promise that this grid does not write them (p.early, never for the
    // replay commit), the first item's state rows, conv taps, conv state and
    // (trees) parents are loaded and its tree tables built; everything else
    // of the item only goes to L2 (a prefetch is safe even for bytes the
    // previous grid still writes).
    const bool early = !RP && p.early;
    prefetch_l2_item<DK, BF16, TREE>(p, I0, tid, nthreads, !early);
    if (early) {
        load_rows(p, rs, p.ssm_in + ((size_t)I0.by * p.H_v + I0.h) * (size_t)p.d_v * DK + (size_t)I0.row0 * DK,
                  warp * RowState<DK, SL>::kRows < I0.R);
        prefetch_item<DK, BF16>(p, I0, xst, wst, cst, true, tid, nthreads, T, kStageTaps);
        if constexpr (TREE) {
            pr = tid <= T ? (tid == 0 ? -1 : ldic(p.parent + (size_t)I0.bidx * (T + 1) + tid, buf_parent(p), p.dev_status))
                          : 0;
            tree_tables(p, p.parent + (size_t)I0.bidx * (T + 1), pr, par_s, src_s, tid, nthreads, 0, kParkSlots);
            tables_of = I0.bidx;  // the barrier after the staging wait publishes them
        }
    }
    if constexpr (kPark) {
        if (warp == 0) gdntc::tmem_alloc<kParkCols>(&park_s);
        gdntc::fence_before_sync();
        __syncthreads();
        gdntc::fence_after_sync();
    }
    pdl_wait();
    bool rows_ready = early;  // rs holds the current item's rows already
    bool reuse_qk = false;  // q_s / k_s / kq_s hold this item's normalised q, k
    // the tokens an item runs: all of them, or (replay) the accepted ones
    auto tokens_of = [&](const Item &J) -> int {
        if constexpr (!RP) return T;
        const int k = ldic(p.accept_len + J.bidx, buf_accept(p), p.dev_status);
        return k >= 0 && k <= T ? k : 0;  // out of range: flagged below, nothing changes
    };
    VerifyArgs pn = p;  // p with T = the staged item's tokens
    pn.T = tokens_of(I0);
    // Inputs landing during the launch (x_ready): compiled into the full-size
    // instantiations only; the host never picks the 4-rows-per-warp one for a
    // call with x_ready (its code stays as it is without the wait).
    constexpr bool kReady = SL == kSlots;
    if constexpr (kReady) wait_ready(p, I0.by);  // the first item's x, a, b rows
    prefetch_item<DK, BF16>(p, I0, xst, wst, cst, true, tid, nthreads, pn.T, early ? kStageX : kStageAll);
    prefetch_scalars<BF16, TREE>(p, I0, ga, gb, pr, tid);
    while (true) {
        if (tid == 0 && stealing) steal_issue(resp, bar);  // the next item, answered during this prologue
        const Item I = decode_item(p, it, nrb);
        const VerifyArgs pi = pn;  // this item's token count (pn moves on to the next item)
        if constexpr (RP) {
            const int k = ldic(p.accept_len + I.bidx, buf_accept(p), p.dev_status);
            if ((k < 0 || k > T) && p.dev_status && tid == 0 && I.y == 0 && I.h == 0 && I.rb == 0)
                atomicOr(p.dev_status, GDN_DEV_NODE_RANGE);
        }
        const bool has_rows = warp * RowState<DK, SL>::kRows < I.R && pi.T > 0;
        const size_t head_off = ((size_t)I.by * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
        if (!rows_ready) load_rows(p, rs, p.ssm_in + head_off, has_rows);  // overlaps the prologue
        rows_ready = false;

        cp_async_wait_all();
        if (tid < T) {
            a_s[tid] = gate_value<BF16>(ga);
            b_s[tid] = gate_value<BF16>(gb);
        }
        __syncthreads();  // staged inputs and gates visible to every thread
        if constexpr (TREE) {
            if (I.bidx != tables_of) {  // the tables depend on the request only
                tree_tables(p, p.parent + (size_t)I.bidx * (T + 1), pr, par_s, src_s, tid, nthreads, 0,
                            kParkSlots);
                __syncthreads();
                tables_of = I.bidx;
            }
        }

        conv_norm_staged<DK, BF16, TREE, KT>(pi, I, xst, wst, cst, src_s, q_s, k_s, v_s, kq_s, reuse_qk, warp,
                                             nthreads >> 5);
        if (tid == 0) {
            int nx = -1;
            if (stealing) {
                nx = steal_result(resp, bar, phase);
                // After a give-up the answer may still land (asynchronously,
                // in this CTA's shared memory): wait once more on the same
                // phase, so that a late cancellation is still run here and
                // the CTA does not exit with the write pending. Only when
                // both waits give up is the item taken as lost.
                if (nx == -2) nx = steal_result(resp, bar, phase);
                phase ^= 1u;
                if (nx == -2 && p.dev_status) atomicOr(p.dev_status, GDN_DEV_SCHED);
                if (nx < 0 || nx >= n_items) stealing = false;
            }
            next_s = nx;
            // inputs landing during the launch: whether the next item's rows
            // are there already (the acquire here and the barrier below order
            // every thread's staging reads after the flag)
            if constexpr (kReady) {
                next_ready_s = 1;
                if (p.x_ready && nx >= 0 && nx < n_items) next_ready_s = ready_flag(p, decode_item(p, nx, nrb).by);
            }
        }
        __syncthreads();  // staging consumed; q, k (normalised), k.q, v ready; next_s set

        const int next = next_s >= 0 && next_s < n_items ? next_s : n_items;
        if (next >= n_items) pdl_launch_dependents();  // nothing left to take: this CTA's last item
        bool next_reuse = false;
        // the next item's inputs are staged during this item's recurrence,
        // unless they have not landed yet (x_ready): then after it
        const bool stage_now = !kReady || next_ready_s != 0;
        Item In{};
        if (next < n_items) {
            In = decode_item(p, next, nrb);
            next_reuse = In.by == I.by && In.g == I.g;
            pn.T = tokens_of(In);
            if (stage_now) {
                prefetch_item<DK, BF16>(p, In, xst, wst, cst, !next_reuse, tid, nthreads, pn.T);
                prefetch_scalars<BF16, TREE>(p, In, ga, gb, pr, tid);
            }
        }
        if (has_rows) {
            float *ck0 =
                p.ssm_ckpt + ((size_t)I.by * T * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
            recurrence<DK, TREE, SL, kPark>(pi, rs, p.ssm_in + head_off, ck0, q_s, k_s, v_s, o_s, a_s, b_s, kq_s,
                                            par_s, kPark ? park_s : 0u);
            if constexpr (RP) {  // the rows after token k-1 replace the live rows (each thread its own)
                const int j8 = (tid & 31) & (kLanesPerRow - 1);
#pragma unroll
                for (int s2 = 0; s2 < SL; ++s2)
#pragma unroll
                    for (int m = 0; m < RowState<DK, SL>::NV4; ++m)
                        st4c(p.ssm_out + head_off + (size_t)rs.lrow[s2] * DK + 4 * j8 + kColStride * m, rs.S[s2][m],
                             buf_state<DK>(p), p.dev_status);
            }
        }
        __syncthreads();
        if constexpr (!RP) write_out(p, I, o_s, threadIdx.x, blockDim.x);
        if (next >= n_items) break;
        if (kReady && !stage_now) {
            wait_ready(p, In.by);
            prefetch_item<DK, BF16>(p, In, xst, wst, cst, !next_reuse, tid, nthreads, pn.T);
            prefetch_scalars<BF16, TREE>(p, In, ga, gb, pr, tid);
        }
        it = next;
        reuse_qk = next_reuse;
    }
    if constexpr (kPark) {
        gdntc::fence_before_sync();
        __syncthreads();  // no warp reads its parked rows any more
        if (warp == 0) gdntc::tmem_dealloc<kParkCols>(park_s);
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
    pdl_wait();
    extern __shared__ __align__(16) unsigned char smem[];
    const Layout L = make_layout(p.T, DK, p.K);
    float *q_s = reinterpret_cast<float *>(smem + L.q), *k_s = reinterpret_cast<float *>(smem + L.k);
    float *v_s = reinterpret_cast<float *>(smem + L.v), *o_s = reinterpret_cast<float *>(smem + L.o);
    float *a_s = reinterpret_cast<float *>(smem + L.a), *b_s = reinterpret_cast<float *>(smem + L.b);
    float *kq_s = reinterpret_cast<float *>(smem + L.kq);
    const int T = p.T, K = p.K;
    const int nrb = row_blocks(p);
    const Item I = decode_item(p, (blockIdx.z * p.H_v + blockIdx.y) * nrb + blockIdx.x, nrb);
    const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5;
    const int Te = ldic(accept_len + I.bidx, buf_accept(p), p.dev_status);
    if (Te <= 0 || Te > T) {
        if (Te != 0 && p.dev_status && tid == 0 && I.y == 0 && I.h == 0 && I.rb == 0)
            atomicOr(p.dev_status, GDN_DEV_NODE_RANGE);
        return;
    }
    const bool has_rows = warp * kRowsPerWarp < I.R;
    const size_t head_off = ((size_t)I.by * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
    RowState<DK> rs;
    load_rows<DK>(p, rs, p.ssm_out + head_off, has_rows);
    for (int t = tid; t < Te; t += nthreads) {
        const size_t gi = ((size_t)I.by * T + t) * p.H_v + I.h;
        a_s[t] = ld_inc<BF16>(p.a, gi, buf_a<BF16 ? 2 : 4>(p), p.dev_status);
        b_s[t] = ld_inc<BF16>(p.b, gi, buf_b<BF16 ? 2 : 4>(p), p.dev_status);
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
                wr[j] = j < K ? ld_inc<BF16>(p.w, ((size_t)I.y * p.C + c) * K + j, buf_w<BF16 ? 2 : 4>(p), p.dev_status)
                              : 0.f;
                st[j] = j < K - 1 ? ldfc(p.conv_in + ((size_t)I.by * p.C + c) * (K - 1) + j, buf_conv(p), p.dev_status)
                                  : 0.f;
            }
            constexpr int CH = 8;
            for (int t0 = 0; t0 < Te; t0 += CH) {
                float xr[CH];
#pragma unroll
                for (int u = 0; u < CH; ++u)
                    xr[u] = t0 + u < Te ? ld_inc<BF16>(p.x, x_base + (size_t)(t0 + u) * p.C + c, buf_x<BF16 ? 2 : 4>(p),
                                                       p.dev_status)
                                        : 0.f;
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
        for (int t = 0; t < Te; ++t)
            recurrence_step<DK, kSlots>(p, rs, t, nullptr, q_s, k_s, v_s, o_s, a_s, b_s, kq_s);
        const int lane = tid & 31, j8 = lane & (kLanesPerRow - 1);
#pragma unroll
        for (int s2 = 0; s2 < kSlots; ++s2)
#pragma unroll
            for (int m = 0; m < RowState<DK>::NV4; ++m)
                st4c(p.ssm_out + head_off + (size_t)rs.lrow[s2] * DK + 4 * j8 + kColStride * m, rs.S[s2][m],
                     buf_state<DK>(p), p.dev_status);
    }
}



template <int DK, bool BF16, bool TREE>
int launch_verify(const VerifyArgs &a, int batch, bool aligned_inputs, cudaStream_t stream) {
    const int nrb = row_blocks(a);
    const int rows = a.d_v < kRowsPerCta ? a.d_v : kRowsPerCta;  // d_v % kRowsPerWarp == 0
    const int threads = rows / kRowsPerWarp * 32;
    const PipeLayout Lp = make_pipe_layout(a.T, DK, a.K, BF16 ? 2 : 4);
    // the work-stealing kernel (gdn_verify_persistent: its CTAs stay resident and take
    // item after item) keeps one gate / parent value per thread in registers
    if (aligned_inputs && Lp.total + kStaticSmem <= kMaxSmem && threads > a.T) {
        // Small launches (one layer, a few heads) split each head's rows into
        // smaller blocks, down to 32 rows, until there are items for about
        // two resident CTAs per SM; every CTA still runs its item's whole
        // conv prologue. Items of <= 32 rows run the recurrence with 4 rows
        // per warp (SL = 1), so that all the CTA's warps share them. (A
        // layer as 128 CTAs of 32 rows ran 48 back-to-back launches in 675
        // us, as 256 CTAs of 16 rows in 880 us, as 32 CTAs of 128 rows in
        // 773 us.) Each row's arithmetic is the same whatever the block size
        // or the warp that holds it. Without the K = 4 instantiation, blocks
        // go down to 16 rows with 16 rows per warp.
        VerifyArgs pa = a;
        const int sms = gdnhost::sm_count();
        const long long want = 2LL * (sms > 0 ? sms : 152);
        const int min_rpi = a.K == 4 ? 32 : kRowsPerWarp;
        while (pa.rpi > min_rpi && (long long)batch * a.Y * a.H_v * row_blocks(pa) < want) pa.rpi /= 2;
        const bool small = pa.rpi <= 32 && a.K == 4 && !a.x_ready;  // (x_ready: full-size instantiations)
        // with 4 rows per warp an item of rpi rows needs rpi / 4 warps
        const int thr = small && threads < pa.rpi / kRowsPerSlot * 32 ? pa.rpi / kRowsPerSlot * 32 : threads;
        auto kern = small ? gdn_verify_persistent<DK, BF16, TREE, 4, 1>
                          : (a.K == 4 ? gdn_verify_persistent<DK, BF16, TREE, 4, kSlots>
                                      : gdn_verify_persistent<DK, BF16, TREE, 0, kSlots>);
        static SmemSet set4, set0, set1;
        SmemSet &set = small ? set1 : (a.K == 4 ? set4 : set0);
        if (!ensure_smem(kern, Lp.total, set)) return GDN_ERR_CUDA;
        // one CTA per item: the running CTAs take the pending ones' items.
        // When every CTA fits at once (2 per SM) there is nothing to take,
        // and the CTAs skip the requests (a hint only: a CTA that starts
        // late still runs its own item).
        const int grid = batch * a.Y * a.H_v * row_blocks(pa);
        pa.steal = grid > 2 * (sms > 0 ? sms : 152) ? 1 : 0;
        if (launch_pdl(kern, dim3(grid), dim3(thr), Lp.total, stream, pa, grid) != cudaSuccess)
            return GDN_ERR_CUDA;
    } else {
        auto kern = gdn_verify_kernel<DK, BF16, TREE>;
        static SmemSet set;
        const Layout L = make_layout(a.T, DK, a.K);
        if (!ensure_smem(kern, L.total, set)) return GDN_ERR_CUDA;
        dim3 grid(nrb, a.H_v, batch * a.Y);
        if (launch_pdl(kern, grid, dim3(threads), L.total, stream, a) != cudaSuccess) return GDN_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// The replay commit on the work-stealing kernel (chains): returns GDN_OK when
// launched, 1 when the shape or the inputs' alignment calls for the
// one-item-per-CTA replay kernel instead.
template <int DK, bool BF16>
int launch_replay(const VerifyArgs &a, int batch, bool aligned_inputs, cudaStream_t stream) {
    const int rows = a.d_v < kRowsPerCta ? a.d_v : kRowsPerCta;
    const int threads = rows / kRowsPerWarp * 32;
    const PipeLayout Lp = make_pipe_layout(a.T, DK, a.K, BF16 ? 2 : 4);
    if (!(aligned_inputs && Lp.total + kStaticSmem <= kMaxSmem && threads > a.T)) return 1;
    VerifyArgs pa = a;
    const int sms = gdnhost::sm_count();
    const long long want = 2LL * (sms > 0 ? sms : 152);
    while (pa.rpi > kRowsPerWarp && (long long)batch * a.Y * a.H_v * row_blocks(pa) < want) pa.rpi /= 2;
    auto kern = a.K == 4 ? gdn_verify_persistent<DK, BF16, false, 4, kSlots, true>
                         : gdn_verify_persistent<DK, BF16, false, 0, kSlots, true>;
    static SmemSet set4, set0;
    if (!ensure_smem(kern, Lp.total, a.K == 4 ? set4 : set0)) return GDN_ERR_CUDA;
    const int grid = batch * a.Y * a.H_v * row_blocks(pa);
    return launch_pdl(kern, dim3(grid), dim3(threads), Lp.total, stream, pa, grid) == cudaSuccess ? GDN_OK
                                                                                                   : GDN_ERR_CUDA;
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


}  // namespace

extern "C" int gdn_verify_span_pipelined(const gdn_dims *d, int32_t n_tok, const void *x, const void *a,
                                         const void *b, const void *conv_w, const float *ssm_in,
                                         const float *conv_in, float *ssm_ckpt, float *conv_ckpt, float *out,
                                         int32_t *dev_status, uint32_t flags, const int32_t *x_ready,
                                         gdn_stream_t stream) {
    int rc = check_common(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt, out);
    if (rc != GDN_OK) return rc;
    if (flags & ~(uint32_t)GDN_VERIFY_STATE_READY) return GDN_ERR_FLAGS;
    if (dev_status && !gdnhost::aligned_to(dev_status, 4)) return GDN_ERR_ALIGN;
    if (x_ready && !gdnhost::aligned_to(x_ready, 4)) return GDN_ERR_ALIGN;
    VerifyArgs v = make_args(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt, out, nullptr,
                             dev_status);
    v.early = (flags & GDN_VERIFY_STATE_READY) ? 1 : 0;
    v.x_ready = x_ready;
    return dispatch_verify<false>(d, v, static_cast<cudaStream_t>(stream));
}

extern "C" int gdn_verify_span_ex(const gdn_dims *d, int32_t n_tok, const void *x, const void *a,
                                  const void *b, const void *conv_w, const float *ssm_in,
                                  const float *conv_in, float *ssm_ckpt, float *conv_ckpt, float *out,
                                  int32_t *dev_status, uint32_t flags, gdn_stream_t stream) {
    return gdn_verify_span_pipelined(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt, out,
                                     dev_status, flags, nullptr, stream);
}

extern "C" int gdn_verify_span(const gdn_dims *d, int32_t n_tok, const void *x, const void *a,
                               const void *b, const void *conv_w, const float *ssm_in,
                               const float *conv_in, float *ssm_ckpt, float *conv_ckpt, float *out,
                               int32_t *dev_status, gdn_stream_t stream) {
    return gdn_verify_span_ex(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt, out, dev_status,
                              0u, stream);
}

extern "C" int gdn_tree_verify(const gdn_dims *d, int32_t n_nodes, const int32_t *parent_host,
                               const int32_t *parent_dev, const void *x, const void *a,
                               const void *b, const void *conv_w, const float *ssm_in,
                               const float *conv_in, float *ssm_ckpt, float *conv_ckpt,
                               float *out, int32_t *dev_status, gdn_stream_t stream) {
    return gdn_tree_verify_ex(d, n_nodes, parent_host, parent_dev, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt,
                              conv_ckpt, out, dev_status, 0u, stream);
}

extern "C" int gdn_tree_verify_ex(const gdn_dims *d, int32_t n_nodes, const int32_t *parent_host,
                                  const int32_t *parent_dev, const void *x, const void *a,
                                  const void *b, const void *conv_w, const float *ssm_in,
                                  const float *conv_in, float *ssm_ckpt, float *conv_ckpt,
                                  float *out, int32_t *dev_status, uint32_t flags, gdn_stream_t stream) {
    return gdn_tree_verify_pipelined(d, n_nodes, parent_host, parent_dev, x, a, b, conv_w, ssm_in, conv_in,
                                     ssm_ckpt, conv_ckpt, out, dev_status, flags, nullptr, stream);
}

extern "C" int gdn_tree_verify_pipelined(const gdn_dims *d, int32_t n_nodes, const int32_t *parent_host,
                                         const int32_t *parent_dev, const void *x, const void *a,
                                         const void *b, const void *conv_w, const float *ssm_in,
                                         const float *conv_in, float *ssm_ckpt, float *conv_ckpt,
                                         float *out, int32_t *dev_status, uint32_t flags,
                                         const int32_t *x_ready, gdn_stream_t stream) {
    if (!d) return GDN_ERR_NULL;
    if (n_nodes < 2) return GDN_ERR_TREE_TRUNCATED;
    int rc = check_common(d, n_nodes - 1, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt, out);
    if (rc != GDN_OK) return rc;
    if (!parent_host || !parent_dev) return GDN_ERR_NULL;
    if (!gdnhost::aligned_to(parent_dev, 4) || (dev_status && !gdnhost::aligned_to(dev_status, 4)))
        return GDN_ERR_ALIGN;
    rc = gdnhost::check_tree(parent_host, d->batch, n_nodes, false, 0);
    if (rc != GDN_OK) return rc;
    if (flags & ~(uint32_t)GDN_VERIFY_STATE_READY) return GDN_ERR_FLAGS;
    if (x_ready && !gdnhost::aligned_to(x_ready, 4)) return GDN_ERR_ALIGN;
    VerifyArgs v = make_args(d, n_nodes - 1, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt, out,
                             parent_dev, dev_status);
    v.early = (flags & GDN_VERIFY_STATE_READY) ? 1 : 0;
    v.x_ready = x_ready;
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
    v.accept_len = accept_len_dev;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int nrb = row_blocks(v);
    const int rows = d->d_v < kRowsPerCta ? d->d_v : kRowsPerCta;
    const int threads = rows / kRowsPerWarp * 32;
    const Layout L = make_layout(n_tok, d->d_k, d->conv_k);
    const dim3 grid(nrb, d->h_v, d->batch * d->layers);
    const bool bf = d->in_dtype == GDN_BF16;
    // the staged work-stealing kernel when the inputs allow cp.async staging
    const bool al = aligned16(x) && aligned16(conv_w);
    if (d->d_k == 128)
        rc = bf ? launch_replay<128, true>(v, d->batch, al, st) : launch_replay<128, false>(v, d->batch, al, st);
    else
        rc = bf ? launch_replay<64, true>(v, d->batch, al, st) : launch_replay<64, false>(v, d->batch, al, st);
    if (rc != GDN_OK && rc != 1) return rc;
    if (rc == 1) {  // the one-item-per-CTA replay kernel: inputs loaded directly
        if (d->d_k == 128) {
            auto kern = bf ? gdn_replay_kernel<128, true> : gdn_replay_kernel<128, false>;
            static SmemSet set_b, set_f;
            if (!ensure_smem(kern, L.total, bf ? set_b : set_f)) return GDN_ERR_CUDA;
            if (launch_pdl(kern, grid, dim3(threads), L.total, st, v, accept_len_dev) != cudaSuccess)
                return GDN_ERR_CUDA;
        } else {
            auto kern = bf ? gdn_replay_kernel<64, true> : gdn_replay_kernel<64, false>;
            static SmemSet set_b, set_f;
            if (!ensure_smem(kern, L.total, bf ? set_b : set_f)) return GDN_ERR_CUDA;
            if (launch_pdl(kern, grid, dim3(threads), L.total, st, v, accept_len_dev) != cudaSuccess)
                return GDN_ERR_CUDA;
        }
    }
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    if (d->conv_k > 1) {
        const dim3 g2((d->conv_ch + 255) / 256, d->batch * d->layers);
        if (launch_pdl(bf ? gdn_conv_state_kernel<true> : gdn_conv_state_kernel<false>, g2, dim3(256), 0, st, v,
                       accept_len_dev, conv_state) != cudaSuccess)
            return GDN_ERR_CUDA;
        if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    }
    return GDN_OK;
}
