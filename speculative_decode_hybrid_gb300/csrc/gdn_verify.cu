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
//  * One CTA per (request*layer, value head, block of up to 128 value rows).
//    Row i of S only needs k_t, q_t, a_t, b_t and v_t[i], so value rows are
//    independent and S never leaves registers between tokens.
//  * 8 lanes own one 128-float row (16 floats each, as 4 float4 at columns
//    4*j + 32*m), a warp holds 4 rows per "slot" and 4 slots (16 rows).
//    Every checkpoint store is a coalesced st.global.v4: one warp
//    instruction writes four full 128-byte lines.
//  * Both dot products S.k and S.q of the old state reduce together over the
//    8 lanes (3 xor-shuffles each). o_t = a (S_p.q) + c (k.q) with
//    c = b (v - a S_p.k), which equals S_t q_t and needs no second
//    dependent reduction; k.q is computed once per node in the prologue.
//  * Prologue per CTA: conv + SiLU of its 256 q/k channels and its v
//    channels for all nodes into shared memory, L2 norms, gates. The
//    conv checkpoint (the last K-1 inputs) is a shifted copy of the inputs
//    and is written here by the CTA that owns the channels.
//  * Tree: nodes run in index order; when parent(i) != i-1 each thread
//    reloads its rows of the parent's checkpoint, which it wrote itself
//    (same thread, same addresses: program order makes it visible; the
//    slot is still in L2).
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
static_assert(kRowsPerWarp <= 16 && 16 % kRowsPerWarp == 0, "d_v is validated as a multiple of 16");

struct VerifyArgs {
    int Y, H_k, H_v, d_v, C, K, T;
    float q_scale;
    const void *x, *a, *b, *w;
    const float *ssm_in, *conv_in;
    float *ssm_ckpt, *conv_ckpt, *out;
    const int32_t *parent;  // [B][T+1] for trees, nullptr for chains
    int32_t *dev_status;
};

__host__ __device__ constexpr size_t verify_smem_floats(int T, int DK) {
    return (size_t)2 * T * DK + (size_t)2 * T * kRowsPerCta + 3 * (size_t)T;
}

size_t verify_smem_bytes(int T, int DK, int K) {
    return verify_smem_floats(T, DK) * sizeof(float) + ((size_t)T + 1 + (size_t)T * K) * sizeof(int);
}

template <int DK, bool BF16, bool TREE>
__global__ void __launch_bounds__(256, 2) gdn_verify_kernel(const VerifyArgs p) {
    constexpr int NV4 = DK / (4 * kLanesPerRow);  // float4 per lane per row
    extern __shared__ __align__(16) float smem[];
    const int T = p.T, K = p.K;
    const int rb = blockIdx.x, h = blockIdx.y, by = blockIdx.z;
    const int y = by % p.Y, bidx = by / p.Y;
    const int ratio = p.H_v / p.H_k;
    const int g = h / ratio;  // key head floor(h * H_k / H_v)
    const int row0 = rb * kRowsPerCta;
    const int R = min(kRowsPerCta, p.d_v - row0);  // rows of this CTA, a multiple of kRowsPerWarp
    const int tid = threadIdx.x, nthreads = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthreads >> 5;
    const void *__restrict__ xin = p.x;

    float *q_s = smem;                   // [T][DK]
    float *k_s = q_s + (size_t)T * DK;   // [T][DK]
    float *v_s = k_s + (size_t)T * DK;   // [T][kRowsPerCta]
    float *o_s = v_s + (size_t)T * kRowsPerCta;
    float *a_s = o_s + (size_t)T * kRowsPerCta;
    float *b_s = a_s + T;
    float *kq_s = b_s + T;
    int *par_s = reinterpret_cast<int *>(kq_s + T);  // [T+1]
    int *src_s = par_s + (T + 1);                    // [T][K]

    // ---- the initial state of this thread's rows, loaded first so that its
    //      latency overlaps the prologue below
    const bool has_rows = warp * kRowsPerWarp < R;
    const int j8 = lane & (kLanesPerRow - 1), rsub = lane / kLanesPerRow;
    const size_t head_off = ((size_t)by * p.H_v + h) * (size_t)p.d_v * DK + (size_t)row0 * DK;
    const float *s_in = p.ssm_in + head_off;
    int lrow[kSlots];
    float4 S[kSlots][NV4];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
        lrow[s] = warp * kRowsPerWarp + s * kRowsPerSlot + rsub;
#pragma unroll
        for (int m = 0; m < NV4; ++m)
            S[s][m] = has_rows ? ld4(s_in + (size_t)lrow[s] * DK + 4 * j8 + kColStride * m)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // ---- tree geometry (re-checked on the device; never read out of bounds)
    if constexpr (TREE) {
        const int32_t *pg = p.parent + (size_t)bidx * (T + 1);
        for (int i = tid; i <= T; i += nthreads) {
            int v = i == 0 ? -1 : pg[i];
            if (i > 0 && (v < 0 || v >= i)) {
                v = i - 1;
                if (p.dev_status) atomicOr(p.dev_status, GDN_DEV_TREE);
            }
            par_s[i] = v;
        }
        __syncthreads();
        // Window table: position j of node i's conv window holds the input of
        // the node at path depth depth(i) - (K-1-j) when that is >= 1, else
        // conv-state slot K-2 + that depth (encoded -1 - slot).
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

    // ---- gates
    for (int t = tid; t < T; t += nthreads) {
        const size_t gi = ((size_t)by * T + t) * p.H_v + h;
        a_s[t] = ld_in<BF16>(p.a, gi);
        b_s[t] = ld_in<BF16>(p.b, gi);
    }
    if constexpr (TREE) __syncthreads();  // src_s ready

    // ---- conv1d + SiLU, one thread per channel, all nodes. The inputs of a
    //      chunk of nodes are loaded together (one memory round trip per
    //      chunk), then the chunk is computed.
    {
        const int nch = 2 * DK + R;
        const bool own_qk = (h % ratio == 0) && rb == 0;
        const size_t x_base = (size_t)by * T * p.C;
        const size_t cc_tok = (size_t)p.C * (K - 1);
        for (int lc = tid; lc < nch; lc += nthreads) {
            int c, stride;
            float *dst;
            if (lc < DK) {
                c = g * DK + lc;
                dst = q_s + lc;
                stride = DK;
            } else if (lc < 2 * DK) {
                c = p.H_k * DK + g * DK + (lc - DK);
                dst = k_s + (lc - DK);
                stride = DK;
            } else {
                c = 2 * p.H_k * DK + h * p.d_v + row0 + (lc - 2 * DK);
                dst = v_s + (lc - 2 * DK);
                stride = kRowsPerCta;
            }
            const bool own = lc >= 2 * DK || own_qk;
            float wr[GDN_MAX_CONV_K], st[GDN_MAX_CONV_K];
#pragma unroll
            for (int j = 0; j < GDN_MAX_CONV_K; ++j) {
                wr[j] = j < K ? ld_in<BF16>(p.w, ((size_t)y * p.C + c) * K + j) : 0.f;
                st[j] = j < K - 1 ? p.conv_in[((size_t)by * p.C + c) * (K - 1) + j] : 0.f;
            }
            float *cck = p.conv_ckpt + (size_t)by * T * cc_tok + (size_t)c * (K - 1);
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
                            const float xv = xr[u];
                            float acc = 0.f;
#pragma unroll
                            for (int j = 0; j < GDN_MAX_CONV_K; ++j)
                                if (j < K) acc = fmaf(wr[j], j < K - 1 ? st[j] : xv, acc);
                            dst[(size_t)t * stride] = silu(acc);
#pragma unroll
                            for (int j = 0; j < GDN_MAX_CONV_K - 1; ++j) {
                                if (j < K - 2) st[j] = st[j + 1];
                                else if (j == K - 2) st[j] = xv;
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
                            float acc = 0.f;
#pragma unroll
                            for (int j = 0; j < GDN_MAX_CONV_K; ++j)
                                if (j < K) acc = fmaf(wr[j], wv[u][j], acc);
                            dst[(size_t)t * stride] = silu(acc);
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

    // ---- per-head L2 norm of q and k, q scale, k.q; one warp per node
    {
        constexpr int PER = DK / 32;
        for (int t = warp; t < T; t += nwarps) {
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
    __syncthreads();

    // ---- the recurrence: S in registers, one checkpoint slot per node
    if (has_rows) {
        const size_t slot = (size_t)p.H_v * p.d_v * DK;
        float *ck0 = p.ssm_ckpt + ((size_t)by * T * p.H_v + h) * (size_t)p.d_v * DK + (size_t)row0 * DK;
        for (int t = 0; t < T; ++t) {
            if constexpr (TREE) {
                const int pp = par_s[t + 1];
                if (pp != t) {
                    const float *src = pp == 0 ? s_in : ck0 + (size_t)(pp - 1) * slot;
#pragma unroll
                    for (int s = 0; s < kSlots; ++s)
#pragma unroll
                        for (int m = 0; m < NV4; ++m)
                            S[s][m] = ld4(src + (size_t)lrow[s] * DK + 4 * j8 + kColStride * m);
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
                    u[s] = dot4(S[s][m], kk[m], u[s]);
                    w[s] = dot4(S[s][m], qq[m], w[s]);
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
                const float vv = v_s[(size_t)t * kRowsPerCta + lrow[s]];
                const float c = bt * (vv - at * u[s]);
#pragma unroll
                for (int m = 0; m < NV4; ++m) {
                    float4 n;
                    n.x = fmaf(c, kk[m].x, at * S[s][m].x);
                    n.y = fmaf(c, kk[m].y, at * S[s][m].y);
                    n.z = fmaf(c, kk[m].z, at * S[s][m].z);
                    n.w = fmaf(c, kk[m].w, at * S[s][m].w);
                    S[s][m] = n;
                    st4(ck + (size_t)lrow[s] * DK + 4 * j8 + kColStride * m, n);
                }
                if (j8 == 0) o_s[(size_t)t * kRowsPerCta + lrow[s]] = fmaf(c, kqt, at * w[s]);
            }
        }
    }
    __syncthreads();

    // ---- o, coalesced: out[b][y][t][h][row]
    for (int i = tid; i < T * R; i += nthreads) {
        const int t = i / R, r = i - t * R;
        p.out[(((size_t)by * T + t) * p.H_v + h) * p.d_v + row0 + r] = o_s[(size_t)t * kRowsPerCta + r];
    }
}

template <int DK, bool BF16, bool TREE>
int launch_verify(const VerifyArgs &a, int batch, cudaStream_t stream) {
    auto kern = gdn_verify_kernel<DK, BF16, TREE>;
    const size_t smem = verify_smem_bytes(a.T, DK, a.K);
    // Largest dynamic shared memory opted into so far, per instantiation (and
    // per process: the attribute is set on every device the first time a
    // larger size is needed there; raising it again is harmless).
    static std::atomic<size_t> smem_set{48 * 1024};
    if (smem > smem_set.load(std::memory_order_relaxed)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return GDN_ERR_CUDA;
        smem_set.store(smem, std::memory_order_relaxed);
    }
    const int nrb = (a.d_v + kRowsPerCta - 1) / kRowsPerCta;
    const int rows = a.d_v < kRowsPerCta ? a.d_v : kRowsPerCta;  // d_v % kRowsPerWarp == 0
    const int threads = rows / kRowsPerWarp * 32;
    dim3 grid(nrb, a.H_v, batch * a.Y);
    kern<<<grid, threads, smem, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <bool TREE>
int dispatch_verify(const gdn_dims *d, const VerifyArgs &a, cudaStream_t stream) {
    const bool bf = d->in_dtype == GDN_BF16;
    if (d->d_k == 128)
        return bf ? launch_verify<128, true, TREE>(a, d->batch, stream)
                  : launch_verify<128, false, TREE>(a, d->batch, stream);
    return bf ? launch_verify<64, true, TREE>(a, d->batch, stream)
              : launch_verify<64, false, TREE>(a, d->batch, stream);
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
    return v;
}

}  // namespace

extern "C" int gdn_verify_span(const gdn_dims *d, int32_t n_tok, const void *x, const void *a,
                               const void *b, const void *conv_w, const float *ssm_in,
                               const float *conv_in, float *ssm_ckpt, float *conv_ckpt, float *out,
                               gdn_stream_t stream) {
    int rc = check_common(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt, out);
    if (rc != GDN_OK) return rc;
    const VerifyArgs v = make_args(d, n_tok, x, a, b, conv_w, ssm_in, conv_in, ssm_ckpt, conv_ckpt,
                                   out, nullptr, nullptr);
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
