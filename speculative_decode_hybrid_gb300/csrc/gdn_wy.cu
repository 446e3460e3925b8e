// gdn_verify_span_wy / gdn_commit_wy: the checkpoint-free chain verify and
// the commit of the accepted prefix, with the span's gated delta rule in
// chunked (WY) form, on sm_103a.
//
// The recurrence is the one of the span verify (lucebox PR #506, Summary:
// split-chain verify with F32 SSM checkpoints; the recurrence is the gated delta
// rule S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t).
// The commit is the conservative "replay the accepted span" of openinfer
// PR #626 (Summary), computed in closed form instead of token by token.
//
// Chunked form. With A_t = a_0 a_1 .. a_t and D[t][j] = a_{j+1} .. a_t
// (D[t][t] = 1), one row s of the initial state gives, for all t at once,
//     g_t = s.k_t,  h_t = s.q_t                            (one S_0 [K | Q] product)
//     u_t = v_t - A_t g_t - sum_{j<t} D[t][j] b_j (k_j.k_t) u_j
//     o_t = A_t h_t + sum_{j<=t} D[t][j] b_j (k_j.q_t) u_j
// and the row after token k-1
//     s_k = A_{k-1} s + sum_{j<k} D[k-1][j] b_j u_j k_j.
// u_t is the rank-1 form's v_t - a_t (S_{t-1}.k_t), so both forms perform
// the same arithmetic, reordered: the T x T unit lower triangular system
// (forward substitution) is shared by every row of a head, and the only
// product over d_k is S_0 [K | Q], with no dependence between tokens.
//
// Kernel: one CTA (256 threads) per (request*layer, value head, block of
// <= 128 value rows). cp.async brings the item's x tile, conv taps and conv
// state (the staged prologue of the verify kernel) and the head's 128 x d_k
// state rows into shared memory. The state tile and the [K | Q] tile are
// kept in the 128-byte-swizzled K-major layout of the tensor-core operand
// descriptors.
//  * Verify: S_0 [K | Q] (M = 128 rows, N = 2T <= 32, K = d_k) runs on the
//    5th-generation tensor cores (tcgen05.mma kind::tf32, accumulator in
//    tensor memory) as 3 x TF32, which keeps f32 accuracy; thread r < 128
//    reads row r of the accumulator (tcgen05.ld), runs the forward
//    substitution in registers and writes o_t for every t.
//  * Commit: S_0 K over the k accepted tokens and the update A S_0 + C K
//    are register-blocked over all 256 threads on the FMA pipe.
#include <cuda_runtime.h>

#include <atomic>

#include "gdn_device.cuh"
#include "gdn_host.h"
#include "gdn_tc.cuh"
#include "gdn_verify_parts.cuh"
#include "gdnspec.h"

namespace {

constexpr int kWyMaxT = GDN_WY_MAX_TOKENS;  // tokens per span in this form
constexpr int kWyRows = kRowsPerCta;  // value rows per item (128)
constexpr int kWyB = 2 * kWyMaxT;     // rows of the [K | Q] tile
// tensor memory of the verify's product: the small part of S_0 (d_k <= 128
// columns) and the accumulator (kWyB columns from column 128)
constexpr int kWyTmemCols = 256;
constexpr unsigned kWyTmemD = 128;
constexpr unsigned kWyPolls = 1u << 22;  // bound on the wait for the product

// Byte offset of the 16-byte unit ug of row r in a K-major tile of `rows`
// rows whose row is split in 128-byte chunks: chunk-major, then row, the
// unit index XOR-ed with r mod 8 (the 128-byte swizzle). Eight consecutive
// rows read at one unit index touch eight different bank groups.
__host__ __device__ __forceinline__ unsigned swz(int rows, int r, int ug) {
    return (unsigned)(ug >> 3) * (unsigned)(rows * 128) + (unsigned)r * 128u +
           ((unsigned)((ug & 7) ^ (r & 7)) << 4);
}

// Shared-memory carve-up (byte offsets): the state tile first (1024-byte
// aligned offset), then the staging buffers, which the [K | Q] tile reuses
// once the prologue has consumed them, then the small arrays.
struct WyLayout {
    size_t s0, xst, wst, cst, bkq, q, k, v, a, b, kq, ac, lm, mm, dm, bar, tmem, total;
};

__host__ __device__ inline WyLayout make_wy_layout(int T, int DK, int K, int esize) {
    WyLayout L;
    const size_t XS = 2 * (size_t)DK + kRowsPerCta;  // staged channels per item
    size_t off = 0;
    L.s0 = off;
    off += (size_t)kWyRows * DK * 4;
    L.xst = off;
    size_t o2 = al16(off + (size_t)T * XS * esize);
    L.wst = o2;
    o2 = al16(o2 + XS * K * esize);
    L.cst = o2;
    o2 = al16(o2 + XS * (K - 1) * 4);
    L.bkq = off;
    const size_t bkq_end = off + (size_t)kWyB * DK * 4;
    off = o2 > bkq_end ? o2 : bkq_end;
    // q and k. Once the small matrices are formed the region is reused: by
    // the verify's tensor-core product for the small part of [K | Q] (a
    // kWyB-row swizzled tile, 1024-byte aligned), by the commit for its G /
    // coefficient rows (kWyRows x (kWyMaxT + 1) floats at most).
    off = (off + 1023) & ~size_t(1023);
    L.q = off;
    L.k = al16(off + (size_t)T * DK * 4);
    {
        size_t end = L.k + (size_t)T * DK * 4;
        const size_t g_end = L.q + (size_t)kWyRows * (kWyMaxT + 1) * 4, b_end = L.q + (size_t)kWyB * DK * 4;
        end = end > g_end ? end : g_end;
        off = al16(end > b_end ? end : b_end);
    }
    L.v = off; off = al16(off + (size_t)T * kWyRows * 4);
    L.a = off; off = al16(off + (size_t)T * 4);
    L.b = off; off = al16(off + (size_t)T * 4);
    L.kq = off; off = al16(off + (size_t)T * 4);
    L.ac = off; off = al16(off + (size_t)T * 4);
    L.lm = off; off = al16(off + (size_t)T * T * 4);
    L.mm = off; off = al16(off + (size_t)T * T * 4);
    L.dm = off; off = al16(off + (size_t)T * T * 4);
    L.bar = off; off += 8;   // mbarrier of the tensor-core product
    L.tmem = off; off += 8;  // tensor-memory base address
    // the offsets above are relative to the first 1024-byte boundary of the
    // dynamic shared memory (the tensor-core swizzle's period): up to 1 KB
    // of slack in front
    L.total = off + 1024;
    return L;
}

// COMMIT false: o of every token (verify, no checkpoints, live state read
// only). COMMIT true: the live state rows after token k-1, k = accept_len of
// the request, written over the live state (k = 0: untouched).
template <int DK, bool BF16, int KT, bool COMMIT>
__global__ void __launch_bounds__(kThreads, 2) gdn_wy_kernel(const VerifyArgs p, const int32_t *accept_len) {
    constexpr int ES = BF16 ? 2 : 4;
    constexpr int U = DK / 4;  // 16-byte units per state row
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const int T = p.T, K = KT > 0 ? KT : p.K;
    const WyLayout L = make_wy_layout(T, DK, K, ES);
    // The tiles start on a 1024-byte boundary, the period of the hardware's
    // 128-byte swizzle, wherever the dynamic shared memory begins.
    const unsigned raw_base = (unsigned)__cvta_generic_to_shared(smem_raw);
    unsigned char *smem = smem_raw + ((1024u - (raw_base & 1023u)) & 1023u);
    const unsigned smem_base = (unsigned)__cvta_generic_to_shared(smem);
    // The verify's S_0 [K | Q] product runs on the tensor cores; the
    // commit's products on the FMA pipe.
    constexpr bool tc = !COMMIT;
    unsigned *tmem_s = reinterpret_cast<unsigned *>(smem + L.tmem);
    const unsigned bar = smem_base + (unsigned)L.bar;
    if constexpr (tc) {
        if (threadIdx.x < 32) gdntc::tmem_alloc<kWyTmemCols>(tmem_s);
        if (threadIdx.x == 0) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
            gdntc::fence_smem_to_async();
        }
    }
    unsigned char *s0 = smem + L.s0, *bkq = smem + L.bkq;
    unsigned char *xst = smem + L.xst, *wst = smem + L.wst, *cst = smem + L.cst;
    float *q_s = reinterpret_cast<float *>(smem + L.q), *k_s = reinterpret_cast<float *>(smem + L.k);
    float *v_s = reinterpret_cast<float *>(smem + L.v);
    float *a_s = reinterpret_cast<float *>(smem + L.a), *b_s = reinterpret_cast<float *>(smem + L.b);
    float *kq_s = reinterpret_cast<float *>(smem + L.kq), *ac_s = reinterpret_cast<float *>(smem + L.ac);
    float *lm_s = reinterpret_cast<float *>(smem + L.lm), *mm_s = reinterpret_cast<float *>(smem + L.mm);
    float *dm_s = reinterpret_cast<float *>(smem + L.dm);
    const int nrb = row_blocks(p);
    const Item I = decode_item(p, blockIdx.x, nrb);
    const int tid = threadIdx.x, nthreads = blockDim.x;
    pdl_wait();

    int Te = T;  // tokens that count: all for the verify, the accepted k for the commit
    if constexpr (COMMIT) {
        const int k = ldic(accept_len + I.bidx, buf_accept(p), p.dev_status);
        if (k <= 0 || k > T) {
            if (k != 0 && p.dev_status && tid == 0 && I.y == 0 && I.h == 0 && I.rb == 0)
                atomicOr(p.dev_status, GDN_DEV_NODE_RANGE);
            return;
        }
        Te = k;
    }
    const size_t head_off = ((size_t)I.by * p.H_v + I.h) * (size_t)p.d_v * DK + (size_t)I.row0 * DK;
    const float *s_in = (COMMIT ? p.ssm_out : p.ssm_in) + head_off;

    // staged inputs (first cp.async group), then the state tile (second group)
    prefetch_item<DK, BF16>(p, I, xst, wst, cst, true, tid, nthreads, p.T);
    unsigned ga = 0u, gb = 0u;  // raw gates of the staged item
    int pr = 0;
    prefetch_scalars<BF16, false>(p, I, ga, gb, pr, tid);
    for (int i = tid; i < I.R * U; i += nthreads) {
        const int r = i / U, ug = i - r * U;
        if (GDN_IN(s_in + (size_t)r * DK + ug * 4, 16, buf_state<DK>(p), p.dev_status))
            cp_async16(s0 + swz(kWyRows, r, ug), s_in + (size_t)r * DK + ug * 4);
    }
    cp_async_commit();

    asm volatile("cp.async.wait_group 1;" ::: "memory");  // the staged inputs have landed
    if (tid < T) {
        a_s[tid] = gate_value<BF16>(ga);
        b_s[tid] = gate_value<BF16>(gb);
    }
    __syncthreads();
    {
        VerifyArgs pc = p;  // the commit only needs its first Te tokens
        pc.T = Te;
        conv_norm_staged<DK, BF16, false, KT>(pc, I, xst, wst, cst, nullptr, q_s, k_s, v_s, kq_s, false, tid >> 5,
                                              nthreads >> 5);
    }
    __syncthreads();  // q, k normalised; the staging buffers are free

    // [K | Q] tile: row n < T is k_n, row T + n is q_n
    for (int i = tid; i < 2 * T * U; i += nthreads) {
        const int n = i / U, ug = i - n * U;
        const float *src = n < T ? k_s + (size_t)n * DK : q_s + (size_t)(n - T) * DK;
        *reinterpret_cast<float4 *>(bkq + swz(kWyB, n, ug)) = ld4(src + ug * 4);
    }
    // decays and the T x T matrices: entry (t, j), j <= t < Te, per thread
    for (int e = tid; e < T * T; e += nthreads) {
        const int t = e / T, j = e - t * T;
        float lv = 0.f, mv = 0.f, dv = 0.f;
        if (j <= t && t < Te) {
            float d = 1.f;
            for (int m = j + 1; m <= t; ++m) d *= a_s[m];
            dv = d;
            const float *kt = k_s + (size_t)t * DK, *kj = k_s + (size_t)j * DK, *qt = q_s + (size_t)t * DK;
            float skk = 0.f, sqk = 0.f;
            for (int s = 0; s < U; ++s) {
                const int ug = (s + e) & (U - 1);  // staggered start: neighbours read different banks
                const float4 kj4 = ld4(kj + ug * 4);
                skk = dot4(ld4(kt + ug * 4), kj4, skk);
                sqk = dot4(ld4(qt + ug * 4), kj4, sqk);
            }
            const float w = d * b_s[j];
            if (j < t) lv = w * skk;
            mv = w * sqk;
        }
        lm_s[e] = lv;
        mm_s[e] = mv;
        dm_s[e] = dv;
    }
    if (tid < T) {
        float A = 1.f;
        for (int m = 0; m <= tid; ++m) A *= a_s[m];
        ac_s[tid] = A;
    }
    cp_async_wait_all();
    __syncthreads();  // state tile, [K | Q] tile and the small matrices are visible

    // First product: G = S_0 [K | Q] (verify: 2T vectors, tensor cores) or
    // G = S_0 K over the Te accepted tokens (commit, FMA pipe). G goes
    // through shared memory (rows padded to an odd stride) to the thread
    // that owns the row: in the dead state tile for the verify, over the
    // dead q / k for the commit (whose update still reads the state tile).
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = (warp & 3) * 8 + (lane & 7), cg = (warp >> 2) * 4 + (lane >> 3);
    const int NV = COMMIT ? Te : 2 * T;
    const int gs = NV | 1;
    float *gh = COMMIT ? q_s : reinterpret_cast<float *>(s0);
    static_assert(kWyRows * (kWyB + 1) * 4 <= kWyRows * 64 * 4, "the verify's G fits in the state tile");
    if constexpr (tc) {
        // Tensor cores, kind::tf32 at f32 accuracy (3 x TF32): with
        // x = big + small, big = tf32(x), the product is
        // big(S_0) big(B) + big(S_0) small(B) + small(S_0) big(B) (the
        // small x small term is below f32 rounding). big(S_0) replaces the
        // state tile in place and small(S_0) goes to tensor memory (thread
        // r < 128 owns row r, its warp's 32 lanes); big(B) replaces the
        // [K | Q] tile, small(B) goes over the dead q / k. Rows of the
        // tiles beyond R / 2T hold stale bytes and only feed dropped
        // accumulator rows / columns.
        gdntc::fence_before_sync();
        __syncthreads();  // the tensor-memory address is visible
        gdntc::fence_after_sync();
        const unsigned tmem = *tmem_s;
        unsigned char *bsm = reinterpret_cast<unsigned char *>(q_s);
        if (tid < kWyRows) {
            const unsigned lanes = tmem + ((unsigned)(tid & ~31) << 16);
#pragma unroll 1
            for (int c0 = 0; c0 < DK; c0 += 8) {
                unsigned v[8];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    float4 *pp = reinterpret_cast<float4 *>(s0 + swz(kWyRows, tid, (c0 >> 2) + h2));
                    const float4 x = *pp;
                    const float4 hi = make_float4(gdntc::tf32_rna(x.x), gdntc::tf32_rna(x.y), gdntc::tf32_rna(x.z),
                                                  gdntc::tf32_rna(x.w));
                    *pp = hi;
                    v[4 * h2 + 0] = __float_as_uint(x.x - hi.x);
                    v[4 * h2 + 1] = __float_as_uint(x.y - hi.y);
                    v[4 * h2 + 2] = __float_as_uint(x.z - hi.z);
                    v[4 * h2 + 3] = __float_as_uint(x.w - hi.w);
                }
                gdntc::tmem_st8(lanes + (unsigned)c0, v);
            }
            gdntc::tmem_wait_st();
        } else {
            for (int i = tid - kWyRows; i < kWyB * U; i += nthreads - kWyRows) {
                const int n = i / U, ug = i - n * U;
                float4 *pp = reinterpret_cast<float4 *>(bkq + swz(kWyB, n, ug));
                const float4 x = *pp;
                const float4 hi = make_float4(gdntc::tf32_rna(x.x), gdntc::tf32_rna(x.y), gdntc::tf32_rna(x.z),
                                              gdntc::tf32_rna(x.w));
                *pp = hi;
                *reinterpret_cast<float4 *>(bsm + swz(kWyB, n, ug)) =
                    make_float4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w);
            }
        }
        gdntc::fence_smem_to_async();
        gdntc::fence_before_sync();
        __syncthreads();
        gdntc::fence_after_sync();
        const unsigned tD = tmem + kWyTmemD;
        if (tid == 0) {
            constexpr unsigned idesc = gdntc::idesc_tf32(kWyRows, kWyB);
            const unsigned a0 = smem_base + (unsigned)L.s0, b0 = smem_base + (unsigned)L.bkq,
                           bs0 = smem_base + (unsigned)L.q;
#pragma unroll 1
            for (int ks = 0; ks < DK / 8; ++ks) {
                const unsigned in_chunk = (unsigned)(ks & 3) * 32u;
                const uint64_t da = gdntc::smem_desc_sw128(a0 + (unsigned)(ks >> 2) * (kWyRows * 128u) + in_chunk);
                const uint64_t db = gdntc::smem_desc_sw128(b0 + (unsigned)(ks >> 2) * (kWyB * 128u) + in_chunk);
                const uint64_t dbs = gdntc::smem_desc_sw128(bs0 + (unsigned)(ks >> 2) * (kWyB * 128u) + in_chunk);
                gdntc::mma_tf32_ss(tD, da, db, idesc, ks > 0);
                gdntc::mma_tf32_ss(tD, da, dbs, idesc, true);
                gdntc::mma_tf32_ts(tD, tmem + (unsigned)ks * 8u, db, idesc, true);
            }
            gdntc::mma_commit(bar);
        }
        if (!gdntc::mbar_wait(bar, 0, kWyPolls)) {
            if (tid == 0 && p.dev_status) atomicOr(p.dev_status, GDN_DEV_SCHED);
            gdntc::mbar_wait(bar, 0, kWyPolls);  // the product may still be running: wait once more
        }
        gdntc::fence_after_sync();
        if (tid < kWyRows) {
            unsigned v[32];
            gdntc::tmem_ld32(tD + ((unsigned)(tid & ~31) << 16), v);
            gdntc::tmem_wait_ld();
            if (tid < I.R) {
#pragma unroll
                for (int n = 0; n < kWyB; ++n)
                    if (n < NV) gh[tid * gs + n] = __uint_as_float(v[n]);
            }
        }
        gdntc::fence_before_sync();
        __syncthreads();  // G is in shared memory; the tensor memory is no longer read
        gdntc::fence_after_sync();
        if (tid < 32) gdntc::tmem_dealloc<kWyTmemCols>(tmem);
    } else {
        // Register-blocked on the FMA pipe: thread (row group rg, column
        // group cg) accumulates rows rg + 32 j against vectors cg + 8 i
        // (j, i < 4), per 16-byte unit 8 shared loads for 64 FMAs. For one
        // (j, i) the 8 row groups of a warp read 8 rows of distinct r mod 8
        // (distinct bank groups under the swizzle) and its 4 column groups 4
        // vectors of distinct n mod 8. Rows >= R read unused tile rows and
        // are dropped.
        float acc[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[j][i] = 0.f;
        if (cg < NV) {
#pragma unroll 2
            for (int ug = 0; ug < U; ++ug) {
                float4 s4[4], b4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    s4[j] = *reinterpret_cast<const float4 *>(s0 + swz(kWyRows, rg + 32 * j, ug));
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (cg + 8 * i < NV) b4[i] = *reinterpret_cast<const float4 *>(bkq + swz(kWyB, cg + 8 * i, ug));
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (cg + 8 * i < NV) acc[j][i] = dot4(s4[j], b4[i], acc[j][i]);
            }
        }
        if constexpr (!COMMIT) __syncthreads();  // every read of the state tile is done: G reuses it
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int row = rg + 32 * j, n = cg + 8 * i;
                if (row < I.R && n < NV) gh[row * gs + n] = acc[j][i];
            }
        __syncthreads();
    }

    const int r = tid;
    if (r < I.R) {
        float g[kWyMaxT], h[kWyMaxT];
#pragma unroll
        for (int t = 0; t < kWyMaxT; ++t) {
            g[t] = t < Te ? gh[r * gs + t] : 0.f;
            h[t] = 0.f;
            if constexpr (!COMMIT) h[t] = t < T ? gh[r * gs + T + t] : 0.f;
        }
        // forward substitution: (I + L) u = v - A g
        float u[kWyMaxT];
#pragma unroll
        for (int t = 0; t < kWyMaxT; ++t) {
            u[t] = 0.f;
            if (t < Te) {
                float acc = fmaf(-ac_s[t], g[t], v_s[(size_t)t * kWyRows + r]);
#pragma unroll
                for (int j = 0; j < t; ++j) acc = fmaf(-lm_s[t * T + j], u[j], acc);
                u[t] = acc;
            }
        }
        if constexpr (!COMMIT) {
            float *o_row = p.out + ((size_t)I.by * T * p.H_v + I.h) * p.d_v + I.row0 + r;
#pragma unroll
            for (int t = 0; t < kWyMaxT; ++t) {
                if (t < T) {
                    float o = ac_s[t] * h[t];
#pragma unroll
                    for (int j = 0; j <= t; ++j) o = fmaf(mm_s[t * T + j], u[j], o);
                    stfc(o_row + (size_t)t * p.H_v * p.d_v, o, buf_out(p), p.dev_status);
                }
            }
        } else {
            // the row's coefficients D[k-1][j] b_j u_j over its own G row
#pragma unroll
            for (int j = 0; j < kWyMaxT; ++j)
                if (j < Te) gh[r * gs + j] = dm_s[(Te - 1) * T + j] * b_s[j] * u[j];
        }
    }
    if constexpr (COMMIT) {
        __syncthreads();  // every row's coefficients are visible
        // S_k = A_{k-1} S_0 + C K, register-blocked like the first product:
        // thread (rg, cg) forms rows rg + 32 j, 16-byte units cg + 8 m, and
        // stores them straight to the live state (64 contiguous bytes per
        // row per warp store).
        constexpr int MU = U / 8;
        const float Ak = ac_s[Te - 1];
        float4 acc[4][MU];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int m = 0; m < MU; ++m) {
                const float4 s4 = *reinterpret_cast<const float4 *>(s0 + swz(kWyRows, rg + 32 * j, cg + 8 * m));
                acc[j][m] = make_float4(Ak * s4.x, Ak * s4.y, Ak * s4.z, Ak * s4.w);
            }
        for (int jj = 0; jj < Te; ++jj) {
            float c[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) c[j] = rg + 32 * j < I.R ? gh[(rg + 32 * j) * gs + jj] : 0.f;
#pragma unroll
            for (int m = 0; m < MU; ++m) {
                const float4 k4 = *reinterpret_cast<const float4 *>(bkq + swz(kWyB, jj, cg + 8 * m));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[j][m].x = fmaf(c[j], k4.x, acc[j][m].x);
                    acc[j][m].y = fmaf(c[j], k4.y, acc[j][m].y);
                    acc[j][m].z = fmaf(c[j], k4.z, acc[j][m].z);
                    acc[j][m].w = fmaf(c[j], k4.w, acc[j][m].w);
                }
            }
        }
        float *s_out = p.ssm_out + head_off;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int row = rg + 32 * j;
            if (row < I.R) {
#pragma unroll
                for (int m = 0; m < MU; ++m)
                    st4c(s_out + (size_t)row * DK + (cg + 8 * m) * 4, acc[j][m], buf_state<DK>(p), p.dev_status);
            }
        }
    }
}

template <int DK, bool BF16, bool COMMIT>
int launch_wy(const VerifyArgs &a, int batch, const int32_t *accept_len, cudaStream_t st) {
    const int nrb = row_blocks(a);
    const long long n_items = (long long)batch * a.Y * a.H_v * nrb;
    if (n_items < 1 || n_items > 0x7fffffffLL) return GDN_ERR_DIMS;
    const WyLayout L = make_wy_layout(a.T, DK, a.K, BF16 ? 2 : 4);
    if (L.total > kMaxSmem) return GDN_ERR_DIMS;
    auto kern = a.K == 4 ? gdn_wy_kernel<DK, BF16, 4, COMMIT> : gdn_wy_kernel<DK, BF16, 0, COMMIT>;
    static SmemSet set4, set0;
    if (!ensure_smem(kern, L.total, a.K == 4 ? set4 : set0)) return GDN_ERR_CUDA;
    return launch_pdl(kern, dim3((unsigned)n_items), dim3(kThreads), L.total, st, a, accept_len) == cudaSuccess
               ? GDN_OK
               : GDN_ERR_CUDA;
}

template <bool COMMIT>
int dispatch_wy(const gdn_dims *d, const VerifyArgs &a, const int32_t *accept_len, cudaStream_t st) {
    const bool bf = d->in_dtype == GDN_BF16;
    if (d->d_k == 128)
        return bf ? launch_wy<128, true, COMMIT>(a, d->batch, accept_len, st)
                  : launch_wy<128, false, COMMIT>(a, d->batch, accept_len, st);
    return bf ? launch_wy<64, true, COMMIT>(a, d->batch, accept_len, st)
              : launch_wy<64, false, COMMIT>(a, d->batch, accept_len, st);
}

// Argument checks shared by both entry points; `state` is the state read
// (and, for the commit, written), `conv` the conv state.
int check_wy(const gdn_dims *d, int32_t n_tok, const void *x, const void *a, const void *b, const void *w,
             const float *state, const float *conv, int32_t *dev_status) {
    int rc = gdnhost::check_dims(d, n_tok);
    if (rc != GDN_OK) return rc;
    if (n_tok > kWyMaxT) return GDN_ERR_DIMS;
    if (!x || !a || !b || !w || !state) return GDN_ERR_NULL;
    if (d->conv_k > 1 && !conv) return GDN_ERR_NULL;
    const size_t es = d->in_dtype == GDN_BF16 ? 2 : 4;
    using gdnhost::aligned16;
    using gdnhost::aligned_to;
    // the staged prologue copies x and the conv taps with 16-byte cp.async
    if (!aligned16(x) || !aligned16(w) || !aligned_to(a, es) || !aligned_to(b, es)) return GDN_ERR_ALIGN;
    if (!aligned16(state) || (d->conv_k > 1 && !aligned16(conv))) return GDN_ERR_ALIGN;
    if (dev_status && !aligned_to(dev_status, 4)) return GDN_ERR_ALIGN;
    return GDN_OK;
}

}  // namespace

extern "C" int gdn_verify_span_wy(const gdn_dims *d, int32_t n_tok, const void *x, const void *a,
                                  const void *b, const void *conv_w, const float *ssm_in,
                                  const float *conv_in, float *out, int32_t *dev_status, gdn_stream_t stream) {
    int rc = check_wy(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, dev_status);
    if (rc != GDN_OK) return rc;
    if (!out) return GDN_ERR_NULL;
    if (!gdnhost::aligned16(out)) return GDN_ERR_ALIGN;
    const VerifyArgs v = make_args(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, nullptr, nullptr, out,
                                   nullptr, dev_status);
    return dispatch_wy<false>(d, v, nullptr, static_cast<cudaStream_t>(stream));
}

extern "C" int gdn_commit_wy(const gdn_dims *d, int32_t n_tok, const int32_t *accept_len_dev, const void *x,
                             const void *a, const void *b, const void *conv_w, float *ssm_state,
                             float *conv_state, int32_t *dev_status, gdn_stream_t stream) {
    int rc = check_wy(d, n_tok, x, a, b, conv_w, ssm_state, conv_state, dev_status);
    if (rc != GDN_OK) return rc;
    if (!accept_len_dev) return GDN_ERR_NULL;
    if (!gdnhost::aligned_to(accept_len_dev, 4)) return GDN_ERR_ALIGN;
    VerifyArgs v = make_args(d, n_tok, x, a, b, conv_w, ssm_state, conv_state, nullptr, nullptr, nullptr,
                             nullptr, dev_status);
    v.ssm_out = ssm_state;
    v.accept_len = accept_len_dev;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    rc = dispatch_wy<true>(d, v, accept_len_dev, st);
    if (rc != GDN_OK) return rc;
    if (d->conv_k > 1) {  // after the state kernel, which reads the old conv state
        const dim3 g2((d->conv_ch + 255) / 256, d->batch * d->layers);
        if (launch_pdl(d->in_dtype == GDN_BF16 ? gdn_conv_state_kernel<true> : gdn_conv_state_kernel<false>, g2,
                       dim3(256), 0, st, v, accept_len_dev, conv_state) != cudaSuccess)
            return GDN_ERR_CUDA;
    }
    return GDN_OK;
}
