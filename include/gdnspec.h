/*
 * gdnspec — target-side verify and rollback of a speculative span over the
 * Gated DeltaNet (GDN) linear-attention layers of a hybrid model, on one
 * GB300 (sm_103a).
 *
 * A step of DFlash / DDTree speculative decoding on a Qwen3.5/3.6 hybrid
 * target feeds the drafted tokens through the target, keeps an F32 SSM and
 * conv checkpoint after every drafted token, accepts the longest prefix (or
 * root path) whose tokens equal the target's greedy argmax, and restores the
 * recurrent state at the accepted token on the device, with no replay:
 *   - lucebox PR #506 "perf(dflash): split-chain fast rollback with F32 SSM
 *     checkpoints", Summary and Memory trade-off (per-token F32 checkpoints,
 *     fast rollback);
 *   - lucebox PR #533 "feat: DFlash support for tensor-parallel Qwen3.6
 *     targets", Changes (restore SSM and convolution state on-device; DDTree);
 *   - openinfer PR #626 "feat(qwen35): add opt-in DFlash speculative
 *     decoding", Summary and What Changed (greedy verify; recurrent state,
 *     conv state).
 *
 * Per GDN layer the pages name the recurrent (SSM) state and the conv state
 * but do not print the equations; this library computes, per request, layer
 * and processed node t (in node-index order):
 *   conv:  y[c] = SiLU( sum_{j<K} w[c][j] * win_t[c][j] ),  win_t[c][K-1] = x_t[c]
 *          and win_t[c][0..K-2] the K-1 previous inputs on the node's root
 *          path (the initial conv state above the root), oldest first;
 *   split: y = [ q (H_k*d_k) | k (H_k*d_k) | v (H_v*d_v) ];
 *          q, k L2-normalised per key head: u / sqrt(sum u^2 + 1e-6); q *= q_scale;
 *   rule:  value head h uses key head g = floor(h * H_k / H_v) and
 *          S_t = a_t S_p (I - b_t k_t k_t^T) + b_t v_t k_t^T,   o_t = S_t q_t
 *          with S_p the state after the parent node (the initial state for
 *          children of the root); S is [d_v][d_k] (row = value index).
 *
 * Conventions for every call:
 *   - Node 0 is the committed root. Its effect is already in the initial
 *     state; a span processes nodes 1..N-1 (n_tok = N-1 tokens). Row t-1 of
 *     every per-token array belongs to node t.
 *   - All arrays are row-major, contiguous, in the layouts given below, and
 *     owned by the caller. Device arrays live on the current CUDA device.
 *     The library allocates nothing.
 *   - Every call validates its arguments on the host first and returns a
 *     non-zero status with NOTHING queued when a check fails (fail-closed).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream); the library never synchronises the host with the
 *     device. Launch failures return GDN_ERR_CUDA.
 *   - Problems that only the device can see (a draft token outside the
 *     vocabulary, an accepted node out of range, a NaN logit) never trap:
 *     they are OR-ed into *dev_status (nullable) as GDN_DEV_* bits.
 *   - Calls are stateless; concurrent calls on distinct buffers are safe.
 */
#ifndef GDNSPEC_H
#define GDNSPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, passed as an opaque pointer (NULL = legacy default stream). */
typedef void *gdn_stream_t;

/* Element type of the inputs x, a, b and conv_w. States, checkpoints, outputs
 * and logits are always float32. */
#define GDN_F32 0
#define GDN_BF16 1

/* Status codes returned by every call. */
#define GDN_OK 0
#define GDN_ERR_NULL 1            /* a required pointer is NULL */
#define GDN_ERR_DIMS 2            /* a size is out of the supported range, see gdn_dims */
#define GDN_ERR_ALIGN 3           /* a float state/checkpoint/output pointer is not 16-byte aligned */
#define GDN_ERR_DTYPE 4           /* in_dtype is neither GDN_F32 nor GDN_BF16 */
#define GDN_ERR_TREE_ROOT 5       /* parent[0] != -1 (malformed root) */
#define GDN_ERR_TREE_PARENT 6     /* parent[i] outside [0, i) for i >= 1: forward, cyclic,
                                     self, out-of-range or second-root parent */
#define GDN_ERR_TREE_DEPTH 7      /* a node deeper than the allowed maximum */
#define GDN_ERR_TREE_TRUNCATED 8  /* fewer than 2 nodes: nothing to verify */
#define GDN_ERR_TREE_NOT_CHAIN 9  /* a sibling / skipped parent where a pure chain is required */
#define GDN_ERR_WORKSPACE 10      /* workspace NULL, misaligned or smaller than required */
#define GDN_ERR_CUDA 11           /* a CUDA launch or query failed */
#define GDN_ERR_FLAGS 12          /* a flags argument has a bit this library does not define */

/* Device-side status bits, OR-ed into *dev_status (int32, device memory). */
#define GDN_DEV_TOKEN_RANGE 0x1   /* a draft token id outside [0, vocab): counted as a mismatch */
#define GDN_DEV_NAN_LOGIT 0x2     /* a NaN logit was seen: it ranks above every number */
#define GDN_DEV_NODE_RANGE 0x4    /* accepted node outside [0, n_tok]: nothing restored for it */
#define GDN_DEV_TREE 0x8          /* a device parent array broke parent[i] in [0, i): the kernel
                                     used parent i-1 for that node (verify) or left it unmatched
                                     (acceptance) instead of reading out of bounds */
#define GDN_DEV_SCHED 0x10        /* verify: a CTA gave up waiting for an asynchronous hardware
                                     operation (the answer to a work-stealing request, a
                                     tensor-core product, or (the _pipelined calls) an input
                                     flag); its outputs are incomplete */
#define GDN_DEV_BOUNDS 0x20       /* debug builds of the library only (GDN_DEBUG_BOUNDS): a kernel
                                     skipped a global access that fell outside its buffer */

/* Limits of this library. */
#define GDN_MAX_TOKENS 64         /* n_tok (= N - 1) per span */
#define GDN_MAX_CONV_K 8
#define GDN_MAX_TOPK 32           /* k of spec_topk */
#define GDN_WY_MAX_TOKENS 16      /* n_tok of the chunked-form calls */

/*
 * Model and batch dimensions shared by the verify and restore calls.
 *   batch    B  >= 1 requests
 *   layers   Y  >= 1 GDN layers (B * Y <= 65535)
 *   h_k, h_v    key and value heads, h_v % h_k == 0
 *   d_k         key head size: 64 or 128
 *   d_v         value head size: a multiple of 16, 16..1024
 *   conv_ch  C  = 2 * h_k * d_k + h_v * d_v (channels of the [q | k | v] conv)
 *   conv_k   K  conv kernel width, 1..GDN_MAX_CONV_K (4 for Qwen3.5/3.6)
 *   in_dtype    GDN_F32 or GDN_BF16 for x, a, b, conv_w
 *   q_scale     multiplies the normalised q (1.0 keeps o_t = S_t q_t as written)
 */
typedef struct gdn_dims {
    int32_t batch, layers, h_k, h_v, d_k, d_v, conv_ch, conv_k;
    int32_t in_dtype;
    float q_scale;
} gdn_dims;

/*
 * gdn_verify_span — verify a drafted CHAIN of n_tok tokens over every layer
 * and request, writing an F32 checkpoint after every token.
 * (lucebox PR #506, Summary: F32 SSM checkpoint capture; pure-chain path.)
 *
 * Inputs (device):
 *   x        [B][Y][n_tok][C]        pre-conv channels [q | k | v], in_dtype
 *   a, b     [B][Y][n_tok][h_v]      decay a_t and write strength b_t, in_dtype
 *   conv_w   [Y][C][K]               conv taps; tap K-1 multiplies the current token, in_dtype
 *   ssm_in   [B][Y][h_v][d_v][d_k]   f32 state before the span (read only)
 *   conv_in  [B][Y][C][K-1]          f32 last K-1 conv inputs before the span, oldest first
 *                                    (may be NULL only when K == 1)
 * Outputs (device, fully overwritten):
 *   ssm_ckpt  [B][Y][n_tok][h_v][d_v][d_k]  f32 state after each token
 *   conv_ckpt [B][Y][n_tok][C][K-1]         f32 conv window after each token
 *                                           (may be NULL only when K == 1)
 *   out       [B][Y][n_tok][h_v][d_v]       f32 o_t
 * The live state (ssm_in, conv_in) is never written: rejecting every token
 * needs no work. Outputs must not overlap inputs.
 *   dev_status  nullable, device int32 for device-side findings, as in
 *               gdn_tree_verify (a chain defines none today; it is accepted so
 *               both verify calls take the same arguments).
 * Returns GDN_OK or GDN_ERR_{NULL,DIMS,ALIGN,DTYPE,CUDA}.
 */
int gdn_verify_span(const gdn_dims *dims, int32_t n_tok,
                    const void *x, const void *a, const void *b, const void *conv_w,
                    const float *ssm_in, const float *conv_in,
                    float *ssm_ckpt, float *conv_ckpt, float *out,
                    int32_t *dev_status, gdn_stream_t stream);

/*
 * Flags of gdn_verify_span_ex and gdn_tree_verify_ex.
 *
 * GDN_VERIFY_STATE_READY — the caller promises that ssm_in, conv_in, conv_w
 * and (trees) parent_dev are not written by any work on `stream` that may
 * still be running when this call's kernel starts: with programmatic
 * dependent launch that is the kernel queued just before the call, whose
 * tail the verify overlaps (earlier work has completed). The verify then
 * loads those inputs, and builds its tree tables, before it waits for that
 * kernel, and only x, a and b (which the previous kernel may produce) after
 * it. Typical use: the verify of layer y + 1 queued right after the verify
 * of layer y, as a model whose layers run in sequence calls it; the
 * previous call writes only layer y's checkpoints and outputs. Not for the
 * first verify after a restore or commit, which writes the live state. The
 * results are the same with or without the flag; if the promise is broken,
 * the verify may read stale state.
 */
#define GDN_VERIFY_STATE_READY 0x1u

/*
 * gdn_verify_span_ex — gdn_verify_span with a flags word (GDN_VERIFY_*;
 * 0 = gdn_verify_span). Returns, in addition, GDN_ERR_FLAGS for an unknown
 * bit.
 */
int gdn_verify_span_ex(const gdn_dims *dims, int32_t n_tok,
                       const void *x, const void *a, const void *b, const void *conv_w,
                       const float *ssm_in, const float *conv_in,
                       float *ssm_ckpt, float *conv_ckpt, float *out,
                       int32_t *dev_status, uint32_t flags, gdn_stream_t stream);

/*
 * gdn_tree_verify — verify a DDTree of n_nodes nodes (node 0 = committed
 * root, T = n_nodes - 1 processed nodes) per request. Node i starts from the
 * state of parent(i) and its conv window follows its root path.
 * (lucebox PR #533, Changes and Verification: DDTree verify; lucebox PR #506,
 * Safety boundary: malformed geometry is rejected before execution.)
 *
 *   parent_host [B][n_nodes] int32, host memory: validated before anything is
 *               queued (GDN_ERR_TREE_* as for gdn_tree_check, depth <= T).
 *   parent_dev  [B][n_nodes] int32, device memory, the same contents; read by
 *               the kernel, which re-checks parent[i] in [0, i) and flags
 *               GDN_DEV_TREE in *dev_status (nullable) instead of reading out
 *               of bounds if the two copies differ.
 * Other arguments and layouts are those of gdn_verify_span with n_tok = T.
 */
int gdn_tree_verify(const gdn_dims *dims, int32_t n_nodes,
                    const int32_t *parent_host, const int32_t *parent_dev,
                    const void *x, const void *a, const void *b, const void *conv_w,
                    const float *ssm_in, const float *conv_in,
                    float *ssm_ckpt, float *conv_ckpt, float *out,
                    int32_t *dev_status, gdn_stream_t stream);

/* gdn_tree_verify_ex — gdn_tree_verify with a flags word, as gdn_verify_span_ex. */
int gdn_tree_verify_ex(const gdn_dims *dims, int32_t n_nodes,
                       const int32_t *parent_host, const int32_t *parent_dev,
                       const void *x, const void *a, const void *b, const void *conv_w,
                       const float *ssm_in, const float *conv_in,
                       float *ssm_ckpt, float *conv_ckpt, float *out,
                       int32_t *dev_status, uint32_t flags, gdn_stream_t stream);

/*
 * gdn_verify_span_pipelined / gdn_tree_verify_pipelined — the _ex calls (the
 * same operation, the same bytes) for inputs that are still landing when the
 * kernel starts: a step whose x, a and b arrive over the host link while
 * the verify already runs the layers that are there. This is an interface
 * of this library, not of the pages.
 *
 *   x_ready [B][layers] int32, device memory, nullable (null: the _ex call).
 *           The kernel reads the x, a and b rows of (request b, layer y) only
 *           after x_ready[b * layers + y] != 0. It waits for that (bounded,
 *           about a quarter second; a wait that gives up sets GDN_DEV_SCHED in
 *           *dev_status and the item reads whatever is there). Everything
 *           else (ssm_in, conv_in, conv_w, parent_dev) must be in place when
 *           the call's kernel starts, as for the _ex calls.
 *           The caller sets a flag only after that (request, layer)'s rows
 *           have landed, with a copy-engine write queued behind them (a
 *           host-to-device cudaMemcpyAsync on the stream that copied the
 *           rows), never from a kernel: a kernel could be waiting for an SM
 *           that this launch holds. The kernel reads the flags and never
 *           clears them: the caller zeroes them before the next call's
 *           copies set them again.
 * Returns as the _ex calls, and GDN_ERR_ALIGN for an x_ready not 4-byte
 * aligned.
 */
int gdn_verify_span_pipelined(const gdn_dims *dims, int32_t n_tok,
                              const void *x, const void *a, const void *b, const void *conv_w,
                              const float *ssm_in, const float *conv_in,
                              float *ssm_ckpt, float *conv_ckpt, float *out,
                              int32_t *dev_status, uint32_t flags, const int32_t *x_ready,
                              gdn_stream_t stream);
int gdn_tree_verify_pipelined(const gdn_dims *dims, int32_t n_nodes,
                              const int32_t *parent_host, const int32_t *parent_dev,
                              const void *x, const void *a, const void *b, const void *conv_w,
                              const float *ssm_in, const float *conv_in,
                              float *ssm_ckpt, float *conv_ckpt, float *out,
                              int32_t *dev_status, uint32_t flags, const int32_t *x_ready,
                              gdn_stream_t stream);

/*
 * spec_accept_greedy — greedy acceptance for a batch of requests.
 * (openinfer PR #626, Summary: single greedy request whose speculative output
 * matches plain greedy decoding; lucebox PR #533, Changes: top-K / argmax on
 * the GPU's logits.)
 *
 *   logits     [B][N][V] f32 (device): row n is the target's prediction after node n
 *   tokens     [B][N] int32 (device): tokens[b][n] = drafted token of node n (n >= 1;
 *              entry 0 is ignored)
 *   parent_dev [B][N] int32 (device) for trees, NULL for chains (parent[i] = i-1)
 * Outputs (device):
 *   argmax_out [B][N] int32: argmax of each row, lowest index on ties, the first
 *              NaN ranking above every number (flagged GDN_DEV_NAN_LOGIT)
 *   accept_len [B] int32: depth of the accepted node (chain: k in [0, N-1])
 *   accept_node[B] int32: the accepted node = the deepest node whose root path
 *              matches (tokens[i] == argmax[parent(i)] all along); among equally
 *              deep ones the lower node index at the first divergence wins.
 *              The bonus token is argmax_out[b][accept_node[b]].
 *   workspace  device scratch of at least spec_accept_workspace_bytes(B, N)
 *              bytes, 256-byte aligned, ZERO-FILLED before its first use; every
 *              call leaves every byte it used zero again, so one workspace serves
 *              calls of any shape. Calls that overlap in time must not share it.
 *   dev_status nullable, device int32: GDN_DEV_TOKEN_RANGE / NAN_LOGIT / TREE bits.
 * Limits: 1 <= N <= GDN_MAX_TOKENS + 1, 1 <= V < 2^31, B * N <= 2^20.
 * Returns GDN_OK or GDN_ERR_{NULL,DIMS,WORKSPACE,CUDA}.
 */
int spec_accept_greedy(int32_t batch, int32_t n_nodes, int32_t vocab,
                       const float *logits, const int32_t *tokens,
                       const int32_t *parent_dev,
                       int32_t *argmax_out, int32_t *accept_len, int32_t *accept_node,
                       void *workspace, size_t workspace_bytes,
                       int32_t *dev_status, gdn_stream_t stream);

/* Bytes of workspace spec_accept_greedy needs for (batch, n_nodes); 0 if the
 * sizes are out of range. */
size_t spec_accept_workspace_bytes(int32_t batch, int32_t n_nodes);

/* Size of the fixed device scratch behind spec_accept_greedy_static (1 MiB). */
#define GDN_STATIC_SCRATCH_BYTES (1 << 20)

/*
 * spec_accept_greedy_static — spec_accept_greedy without a caller-supplied
 * workspace, for callers that cannot allocate device memory: code that runs
 * where cudaMalloc is unavailable or forbidden (for example inside an
 * allocator-less runtime, a plugin host that owns all device memory, or a
 * hot loop that must never reach the allocator). The pages have no
 * counterpart of this call; it is a convenience of this library.
 *
 * Arguments, outputs and results are those of spec_accept_greedy, minus the
 * workspace. The scratch is a fixed GDN_STATIC_SCRATCH_BYTES array in the
 * library's device memory, present on every GPU that loads the library until
 * the process exits. The first call on a device (with that device current)
 * looks up the array's device address; make that first call before any
 * stream capture. If the lookup fails, that call returns GDN_ERR_CUDA and
 * the next call looks again; once found, the address is kept for the life
 * of the process, so cudaDeviceReset is not supported with this call. Every
 * call zeroes the part of the array that must start at zero (a small
 * cudaMemsetAsync on `stream`) and allocates nothing.
 * All calls share the one array: calls that may overlap on the GPU (other
 * streams, other host threads) race and must be serialised by the caller.
 * Returns GDN_ERR_WORKSPACE when spec_accept_workspace_bytes(batch, n_nodes)
 * exceeds GDN_STATIC_SCRATCH_BYTES (8 bytes per logit row plus 4 per
 * request: about 130,000 rows, e.g. batch 2,000 with n_nodes 65 fits), and
 * the other codes of spec_accept_greedy.
 */
int spec_accept_greedy_static(int32_t batch, int32_t n_nodes, int32_t vocab,
                              const float *logits, const int32_t *tokens,
                              const int32_t *parent_dev,
                              int32_t *argmax_out, int32_t *accept_len, int32_t *accept_node,
                              int32_t *dev_status, gdn_stream_t stream);

/*
 * gdn_rollback_restore — restore, on the device, the live SSM and conv state
 * of every request and layer to the checkpoint of its accepted node.
 * (lucebox PR #533, Changes: restore split SSM and convolution state
 * on-device; lucebox PR #506, Summary: fast rollback from F32 checkpoints.)
 *
 *   accept_node_dev [B] int32 (device), e.g. spec_accept_greedy's accept_node:
 *       node 0 leaves the state untouched; node in [1, n_tok] copies slot
 *       node-1; anything else copies nothing and sets GDN_DEV_NODE_RANGE.
 *   ssm_ckpt, conv_ckpt  as written by gdn_verify_span / gdn_tree_verify
 *   ssm_state [B][Y][h_v][d_v][d_k], conv_state [B][Y][C][K-1]: the live state
 *       (normally the verify call's ssm_in / conv_in buffers), overwritten
 *       bit-exactly with the chosen slot.
 * Returns GDN_OK or GDN_ERR_{NULL,DIMS,ALIGN,CUDA}.
 */
int gdn_rollback_restore(const gdn_dims *dims, int32_t n_tok,
                         const int32_t *accept_node_dev,
                         const float *ssm_ckpt, const float *conv_ckpt,
                         float *ssm_state, float *conv_state,
                         int32_t *dev_status, gdn_stream_t stream);

/*
 * Replay commit (the conservative alternative to checkpoints): verify without
 * writing any checkpoint, then, once the accepted length is known, re-run
 * only the accepted tokens from the live state and update it in place.
 * (openinfer PR #626, What Changed: commit restores the canonical state and
 * replays the accepted target span; Future Work: a lower-overhead commit.)
 * Restoring checkpoint k and replaying the first k tokens give the same
 * bytes. Chains only: a tree's branches need the per-node states.
 *
 * gdn_verify_span_nockpt — gdn_verify_span writing only `out` (no ssm or
 * conv checkpoints); the live state is read, never written.
 */
int gdn_verify_span_nockpt(const gdn_dims *dims, int32_t n_tok,
                           const void *x, const void *a, const void *b, const void *conv_w,
                           const float *ssm_in, const float *conv_in, float *out,
                           int32_t *dev_status, gdn_stream_t stream);

/*
 * gdn_commit_replay — for every request b with k = accept_len_dev[b] in
 * [1, n_tok], re-run conv + recurrence over tokens 0..k-1 of the span (the
 * same x, a, b, conv_w as the verify call, layouts of gdn_verify_span) from
 * ssm_state / conv_state and overwrite both with the state after token k-1.
 * k = 0 leaves the request untouched; k outside [0, n_tok] changes nothing
 * and sets GDN_DEV_NODE_RANGE in *dev_status (nullable). Two kernels on
 * `stream` (the state replay, then the conv-state update).
 * Returns GDN_OK or GDN_ERR_{NULL,DIMS,ALIGN,DTYPE,CUDA}.
 */
int gdn_commit_replay(const gdn_dims *dims, int32_t n_tok, const int32_t *accept_len_dev,
                      const void *x, const void *a, const void *b, const void *conv_w,
                      float *ssm_state, float *conv_state, int32_t *dev_status,
                      gdn_stream_t stream);

/*
 * gdn_verify_span_wy — gdn_verify_span_nockpt computed in chunked (WY) form:
 * per (request, layer, value head) the span's tokens are solved together
 * (one S_0 [K | Q] product, a shared T x T unit lower triangular forward
 * substitution) instead of one rank-1 update per token. Same arguments,
 * layouts and results (up to rounding order) as gdn_verify_span_nockpt.
 * (lucebox PR #506, Summary: the span's gated delta rule; openinfer PR #626,
 * Summary: the conservative commit this verify pairs with.)
 * Limits: n_tok <= GDN_WY_MAX_TOKENS; x and conv_w 16-byte aligned.
 * Returns GDN_OK or GDN_ERR_{NULL,DIMS,ALIGN,DTYPE,CUDA}.
 */
int gdn_verify_span_wy(const gdn_dims *dims, int32_t n_tok,
                       const void *x, const void *a, const void *b, const void *conv_w,
                       const float *ssm_in, const float *conv_in, float *out,
                       int32_t *dev_status, gdn_stream_t stream);

/*
 * gdn_commit_wy — gdn_commit_replay in chunked form: for every request b with
 * k = accept_len_dev[b] in [1, n_tok], the live state becomes
 * A_{k-1} S + sum_{j<k} D[k-1][j] b_j u_j k_j^T (the state after token k-1,
 * u from the same forward substitution as gdn_verify_span_wy) and the live
 * conv state the last K-1 inputs; k = 0 leaves the request untouched; k
 * outside [0, n_tok] changes nothing and sets GDN_DEV_NODE_RANGE. Same
 * arguments and layouts as gdn_commit_replay; two kernels on `stream`.
 * Limits: n_tok <= GDN_WY_MAX_TOKENS; x and conv_w 16-byte aligned.
 * Returns GDN_OK or GDN_ERR_{NULL,DIMS,ALIGN,DTYPE,CUDA}.
 */
int gdn_commit_wy(const gdn_dims *dims, int32_t n_tok, const int32_t *accept_len_dev,
                  const void *x, const void *a, const void *b, const void *conv_w,
                  float *ssm_state, float *conv_state, int32_t *dev_status,
                  gdn_stream_t stream);

/*
 * spec_topk — the k best logits of each row in the greedy order: larger value
 * first, lower index among equal values, every NaN above every number (the
 * first NaN first; flagged GDN_DEV_NAN_LOGIT), -0.0 equal to +0.0. For
 * draft-side tree construction (lucebox PR #533, Changes: draft top-K on the
 * GPU's logits).
 *   logits  [rows][V] f32 (device, 16-byte aligned)
 *   idx_out [rows][k] int32, val_out [rows][k] f32 (device): the k indices and
 *           their logits, best first
 *   workspace: at least spec_topk_workspace_bytes(rows, k) bytes of device
 *           memory, 256-byte aligned, zero-filled before first use; every call
 *           leaves it zero-filled. Overlapping calls must not share it.
 * Limits: 1 <= k <= GDN_MAX_TOPK, k <= V, 1 <= rows <= 65535.
 * Returns GDN_OK or GDN_ERR_{NULL,DIMS,ALIGN,WORKSPACE,CUDA}.
 */
int spec_topk(int32_t rows, int32_t vocab, int32_t k, const float *logits,
              int32_t *idx_out, float *val_out, void *workspace, size_t workspace_bytes,
              int32_t *dev_status, gdn_stream_t stream);

/* Bytes of workspace spec_topk needs; 0 if the sizes are out of range. */
size_t spec_topk_workspace_bytes(int32_t rows, int32_t k);

/*
 * gdn_tree_check — host-only geometry check of B parent arrays of n_nodes
 * nodes each (the pure-chain guard of lucebox PR #506, Safety boundary).
 *   require_chain != 0: additionally require parent[i] == i-1 (no sibling or
 *   skipped parent). max_depth > 0 bounds every node's depth.
 * Returns GDN_OK, GDN_ERR_NULL, GDN_ERR_DIMS (batch < 1),
 * GDN_ERR_TREE_{TRUNCATED,ROOT,PARENT,DEPTH,NOT_CHAIN}. Touches no GPU.
 */
int gdn_tree_check(const int32_t *parent_host, int32_t batch, int32_t n_nodes,
                   int32_t require_chain, int32_t max_depth);

/* A static, human-readable name for a status code. */
const char *gdn_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* GDNSPEC_H */
