/*
 * CPU oracle for target-side GDN span verify, greedy acceptance and rollback.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this code. The product path (the CUDA library)
 * shares nothing with it: no header, helper, table or constant.
 *
 * Plain, slow, obviously correct: every floating-point value is widened to
 * double on entry and every step is a literal loop in the order the method
 * states. Sources of each step:
 *
 *   - Gated DeltaNet layer of a Qwen3.5/3.6 hybrid target: causal depthwise
 *     conv1d over the concatenated [q | k | v] channels, SiLU, per-head L2
 *     normalisation of q and k, then the gated delta rule
 *         S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t q_t
 *     per value head, with the key head shared by H_v/H_k value heads.
 *     The pages name the state objects but never print these equations:
 *     "recurrent state, conv state" (openinfer PR #626, "What Changed"),
 *     "SSM and convolution state" (lucebox PR #533, "Changes").
 *   - One F32 SSM + conv checkpoint after every drafted token / tree node
 *     (lucebox PR #506, "Summary" and "Memory trade-off").
 *   - Greedy acceptance against the target argmax, longest matching prefix
 *     or root path (openinfer PR #626, "Summary": single active greedy
 *     request whose output matches plain greedy decoding).
 *   - Restore of the checkpoint at the accepted index, on the device in the
 *     product (lucebox PR #533, "Changes": restore split SSM and convolution
 *     state on-device).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   node 0 is the committed root, already absorbed in the initial state; the
 *   span processes nodes 1..N-1; conv weight tap K-1 multiplies the current
 *   token and the conv state keeps the oldest input first; no conv bias;
 *   L2 norm x / sqrt(sum x^2 + 1e-6); value head h reads key head
 *   floor(h * H_k / H_v); argmax takes the lowest index on ties and the first
 *   NaN ranks above every number.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -shared -fPIC (same results on
 * x86-64 and aarch64: no fused multiply-add contraction, no intrinsics).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_ERR_ARG 1
#define ORA_ERR_TREE 2
#define ORA_ERR_NOMEM 3

static double silu(double y) { return y / (1.0 + exp(-y)); }

/* One output of the causal depthwise conv of one channel: sum_j w[j] * win[j]
 * over the K-window win (win[K-1] is the current input), then SiLU. */
static double conv_tap_silu(int K, const double *w, const double *win)
{
    double acc = 0.0;
    for (int j = 0; j < K; ++j)
        acc += w[j] * win[j];
    return silu(acc);
}

/* Causal conv1d + SiLU of one channel over a chain of T inputs.
 * state: the K-1 previous inputs, oldest first. Writes y[T] and, after
 * every input t, the new conv state (the last K-1 inputs) to state_out[T][K-1]. */
int ora_conv1d_silu(int K, int T, const double *w, const double *state,
                    const double *x, double *y, double *state_out)
{
    if (K < 1 || T < 0 || !w || !x || !y || (K > 1 && !state))
        return ORA_ERR_ARG;
    double *seq = (double *)malloc(sizeof(double) * (size_t)(K - 1 + T));
    double *win = (double *)malloc(sizeof(double) * (size_t)K);
    if (!seq || !win) { free(seq); free(win); return ORA_ERR_NOMEM; }
    for (int j = 0; j < K - 1; ++j) seq[j] = state[j];
    for (int t = 0; t < T; ++t) seq[K - 1 + t] = x[t];
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < K; ++j) win[j] = seq[t + j];
        y[t] = conv_tap_silu(K, w, win);
        if (state_out)
            for (int j = 0; j < K - 1; ++j) state_out[(size_t)t * (K - 1) + j] = win[j + 1];
    }
    free(seq); free(win);
    return ORA_OK;
}

/* In-place L2 normalisation: v / sqrt(sum v^2 + 1e-6). */
void ora_l2norm(int n, double *v)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += v[i] * v[i];
    double inv = 1.0 / sqrt(ss + 1e-6);
    for (int i = 0; i < n; ++i) v[i] *= inv;
}

/* One gated delta-rule step of one head, rank-1 form.
 * Row r of S (a d_k vector s_r):
 *   s_r <- a s_r (I - b k k^T) + b v_r k^T = a s_r + b (v_r - a (s_r . k)) k
 * then o_r = s_r . q with the updated row. Sp and Sn may not alias. */
static void delta_step(int d_k, int d_v, const double *Sp, const double *q,
                       const double *k, const double *v, double a, double b,
                       double *Sn, double *o)
{
    for (int r = 0; r < d_v; ++r) {
        const double *sp = Sp + (size_t)r * d_k;
        double *sn = Sn + (size_t)r * d_k;
        double u = 0.0;
        for (int c = 0; c < d_k; ++c) u += sp[c] * k[c];
        double coef = b * (v[r] - a * u);
        for (int c = 0; c < d_k; ++c) sn[c] = a * sp[c] + coef * k[c];
        double acc = 0.0;
        for (int c = 0; c < d_k; ++c) acc += sn[c] * q[c];
        o[r] = acc;
    }
}

/* Gated delta rule of one head over a chain of T tokens, inputs fed straight
 * to the recurrence (no conv, no normalisation).
 * q,k [T][d_k]; v [T][d_v]; a,b [T]; S0 [d_v][d_k];
 * S_out [T][d_v][d_k] (state after each token); o [T][d_v]. */
int ora_gdn_delta_rule(int d_k, int d_v, int T, const double *q, const double *k,
                       const double *v, const double *a, const double *b,
                       const double *S0, double *S_out, double *o)
{
    if (d_k < 1 || d_v < 1 || T < 0 || !S0 || !S_out || !o) return ORA_ERR_ARG;
    const size_t hs = (size_t)d_v * d_k;
    for (int t = 0; t < T; ++t) {
        const double *Sp = t == 0 ? S0 : S_out + (size_t)(t - 1) * hs;
        delta_step(d_k, d_v, Sp, q + (size_t)t * d_k, k + (size_t)t * d_k,
                   v + (size_t)t * d_v, a[t], b[t], S_out + (size_t)t * hs,
                   o + (size_t)t * d_v);
    }
    return ORA_OK;
}

/* The same recurrence with explicit d_k x d_k matrices, exactly as written:
 * M = I - b k k^T;  S_t = a (S_{t-1} M) + b v k^T;  o_t = S_t q.
 * Brute force for small d (O(d_v d_k^2) per token). */
int ora_gdn_delta_rule_explicit(int d_k, int d_v, int T, const double *q,
                                const double *k, const double *v, const double *a,
                                const double *b, const double *S0, double *S_out,
                                double *o)
{
    if (d_k < 1 || d_v < 1 || T < 0 || !S0 || !S_out || !o) return ORA_ERR_ARG;
    const size_t hs = (size_t)d_v * d_k;
    double *M = (double *)malloc(sizeof(double) * (size_t)d_k * d_k);
    if (!M) return ORA_ERR_NOMEM;
    for (int t = 0; t < T; ++t) {
        const double *Sp = t == 0 ? S0 : S_out + (size_t)(t - 1) * hs;
        double *Sn = S_out + (size_t)t * hs;
        const double *kt = k + (size_t)t * d_k, *qt = q + (size_t)t * d_k;
        const double *vt = v + (size_t)t * d_v;
        for (int i = 0; i < d_k; ++i)
            for (int j = 0; j < d_k; ++j)
                M[(size_t)i * d_k + j] = (i == j ? 1.0 : 0.0) - b[t] * kt[i] * kt[j];
        for (int r = 0; r < d_v; ++r)
            for (int j = 0; j < d_k; ++j) {
                double sm = 0.0;
                for (int i = 0; i < d_k; ++i) sm += Sp[(size_t)r * d_k + i] * M[(size_t)i * d_k + j];
                Sn[(size_t)r * d_k + j] = a[t] * sm + b[t] * vt[r] * kt[j];
            }
        for (int r = 0; r < d_v; ++r) {
            double acc = 0.0;
            for (int j = 0; j < d_k; ++j) acc += Sn[(size_t)r * d_k + j] * qt[j];
            o[(size_t)t * d_v + r] = acc;
        }
    }
    free(M);
    return ORA_OK;
}

/* Tree geometry check: parent[0] == -1 and 0 <= parent[i] < i for i >= 1.
 * Writes depth[N] (root depth 0) when depth != NULL. */
int ora_tree_depths(int N, const int32_t *parent, int32_t *depth)
{
    if (N < 1 || !parent) return ORA_ERR_ARG;
    if (parent[0] != -1) return ORA_ERR_TREE;
    for (int i = 1; i < N; ++i)
        if (parent[i] < 0 || parent[i] >= i) return ORA_ERR_TREE;
    if (depth) {
        depth[0] = 0;
        for (int i = 1; i < N; ++i) depth[i] = depth[parent[i]] + 1;
    }
    return ORA_OK;
}

/*
 * Verify one (request, layer) over the N-1 processed nodes of a chain
 * (parent == NULL: parent[i] = i-1) or a tree (parent array, node 0 = root).
 *
 * x [T][C] pre-conv channels [q (H_k d_k) | k (H_k d_k) | v (H_v d_v)]
 * a, b [T][H_v]; w [C][K]; ssm_in [H_v][d_v][d_k]; conv_in [C][K-1]
 * Outputs: ssm_ckpt [T][H_v][d_v][d_k], conv_ckpt [T][C][K-1], out [T][H_v][d_v].
 * Row t-1 of every per-token array belongs to node t. Nodes run in index
 * order; node i starts from the state of parent(i) (the initial state when
 * the parent is the root), and its conv window follows its root path, with
 * positions above the root taken from the initial conv state.
 */
int ora_gdn_verify_layer(int h_k, int h_v, int d_k, int d_v, int K, int N,
                         const int32_t *parent, const double *x, const double *a,
                         const double *b, const double *w, const double *ssm_in,
                         const double *conv_in, double q_scale, double *ssm_ckpt,
                         double *conv_ckpt, double *out)
{
    if (h_k < 1 || h_v < 1 || d_k < 1 || d_v < 1 || K < 1 || N < 2) return ORA_ERR_ARG;
    if (h_v % h_k != 0) return ORA_ERR_ARG;
    if (!x || !a || !b || !w || !ssm_in || !ssm_ckpt || !out) return ORA_ERR_ARG;
    if (K > 1 && (!conv_in || !conv_ckpt)) return ORA_ERR_ARG;
    const int T = N - 1;
    const int C = 2 * h_k * d_k + h_v * d_v;
    const size_t hs = (size_t)d_v * d_k;

    int32_t *par = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    int32_t *depth = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    int *src = (int *)malloc(sizeof(int) * (size_t)K);
    double *win = (double *)malloc(sizeof(double) * (size_t)K);
    double *y = (double *)malloc(sizeof(double) * (size_t)C);
    if (!par || !depth || !src || !win || !y) {
        free(par); free(depth); free(src); free(win); free(y);
        return ORA_ERR_NOMEM;
    }
    par[0] = -1;
    for (int i = 1; i < N; ++i) par[i] = parent ? parent[i] : i - 1;
    if (parent && parent[0] != -1) { free(par); free(depth); free(src); free(win); free(y); return ORA_ERR_TREE; }
    if (ora_tree_depths(N, par, depth) != ORA_OK) {
        free(par); free(depth); free(src); free(win); free(y);
        return ORA_ERR_TREE;
    }

    for (int i = 1; i <= T; ++i) {
        /* Window position j (0..K-1) holds the input at path depth
         * p = depth[i] - (K-1-j): node on the root path when p >= 1
         * (encoded as its index), else conv state slot K-2+p (encoded -1-slot). */
        int node = i;
        for (int j = K - 1; j >= 0; --j) {
            int p = depth[i] - (K - 1 - j);
            if (p >= 1) { src[j] = node; node = par[node]; }
            else src[j] = -1 - (K - 2 + p);
        }
        for (int c = 0; c < C; ++c) {
            for (int j = 0; j < K; ++j)
                win[j] = src[j] >= 0 ? x[(size_t)(src[j] - 1) * C + c]
                                     : conv_in[(size_t)c * (K - 1) + (size_t)(-1 - src[j])];
            y[c] = conv_tap_silu(K, w + (size_t)c * K, win);
            for (int j = 0; j < K - 1; ++j)
                conv_ckpt[((size_t)(i - 1) * C + c) * (K - 1) + j] = win[j + 1];
        }
        double *qs = y, *ks = y + (size_t)h_k * d_k, *vs = y + (size_t)2 * h_k * d_k;
        for (int g = 0; g < h_k; ++g) {
            ora_l2norm(d_k, qs + (size_t)g * d_k);
            ora_l2norm(d_k, ks + (size_t)g * d_k);
            for (int c = 0; c < d_k; ++c) qs[(size_t)g * d_k + c] *= q_scale;
        }
        for (int h = 0; h < h_v; ++h) {
            const int g = (int)(((long long)h * h_k) / h_v);
            const double *Sp = par[i] == 0 ? ssm_in + (size_t)h * hs
                                           : ssm_ckpt + ((size_t)(par[i] - 1) * h_v + h) * hs;
            double *Sn = ssm_ckpt + ((size_t)(i - 1) * h_v + h) * hs;
            delta_step(d_k, d_v, Sp, qs + (size_t)g * d_k, ks + (size_t)g * d_k,
                       vs + (size_t)h * d_v, a[(size_t)(i - 1) * h_v + h],
                       b[(size_t)(i - 1) * h_v + h], Sn,
                       out + ((size_t)(i - 1) * h_v + h) * d_v);
        }
    }
    free(par); free(depth); free(src); free(win); free(y);
    return ORA_OK;
}

/* Index of the largest value; lowest index on ties; the first NaN ranks above
 * every number. Values are compared exactly (no rounding). */
int ora_argmax_f32(int V, const float *row)
{
    int best = 0;
    for (int v = 0; v < V; ++v) {
        if (isnan(row[v])) return v;
        if (v > 0 && row[v] > row[best]) best = v;
    }
    return best;
}

/* Among two distinct nodes of equal depth, is the root path of i smaller than
 * that of j at their first divergence (lower node index wins)? */
static int path_less(const int32_t *par, int i, int j)
{
    while (par[i] != par[j]) { i = par[i]; j = par[j]; }
    return i < j;
}

/*
 * Greedy acceptance of one request.
 * logits [N][V] fp32: row n is the target's prediction after node n.
 * tokens [N]: tokens[n] is node n's drafted token (tokens[0] unused).
 * parent: NULL for a chain, else the tree's parent array.
 * Node n (n >= 1) matches when its parent matches (the root always does) and
 * tokens[n] == argmax(row parent(n)). The accepted node is the deepest
 * matching node; among equally deep ones, the one whose root path has the
 * lower node index at the first divergence. accept_len = its depth.
 */
int ora_accept_greedy(int N, int V, const float *logits, const int32_t *tokens,
                      const int32_t *parent, int32_t *argmax_out,
                      int32_t *accept_len, int32_t *accept_node)
{
    if (N < 1 || V < 1 || !logits || !tokens || !argmax_out || !accept_len || !accept_node)
        return ORA_ERR_ARG;
    int32_t *par = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    int32_t *depth = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
    unsigned char *ok = (unsigned char *)malloc((size_t)N);
    if (!par || !depth || !ok) { free(par); free(depth); free(ok); return ORA_ERR_NOMEM; }
    par[0] = -1;
    for (int i = 1; i < N; ++i) par[i] = parent ? parent[i] : i - 1;
    if ((parent && parent[0] != -1) || ora_tree_depths(N, par, depth) != ORA_OK) {
        free(par); free(depth); free(ok);
        return ORA_ERR_TREE;
    }
    for (int n = 0; n < N; ++n)
        argmax_out[n] = ora_argmax_f32(V, logits + (size_t)n * V);
    ok[0] = 1;
    int best = 0;
    for (int i = 1; i < N; ++i) {
        ok[i] = ok[par[i]] && tokens[i] == argmax_out[par[i]];
        if (!ok[i]) continue;
        if (depth[i] > depth[best] || (depth[i] == depth[best] && path_less(par, i, best)))
            best = i;
    }
    *accept_len = depth[best];
    *accept_node = best;
    free(par); free(depth); free(ok);
    return ORA_OK;
}

/* Restore: state <- checkpoint slot node-1 when node > 0; node 0 leaves the
 * state as it is (verify never wrote it). n = elements per slot. */
int ora_restore(long long n, int node, const double *ckpt, double *state)
{
    if (n < 0 || node < 0 || !state || (node > 0 && !ckpt)) return ORA_ERR_ARG;
    if (node > 0)
        memcpy(state, ckpt + (size_t)(node - 1) * (size_t)n, sizeof(double) * (size_t)n);
    return ORA_OK;
}

/* a ranks above b in the greedy order: NaN above every number (the first NaN
 * first), otherwise the larger value, and the lower index among equals. */
static int ranks_above(float a, int ia, float b, int ib)
{
    const int na = isnan(a), nb = isnan(b);
    if (na || nb) {
        if (na && nb) return ia < ib;
        return na;
    }
    if (a > b) return 1;
    if (a < b) return 0;
    return ia < ib;
}

/* Top-k of one row in that order, by k rounds of selection (a draft-side
 * top-K over the vocabulary; lucebox PR #533, Changes). idx[k], val[k]. */
int ora_topk_f32(int V, const float *row, int k, int32_t *idx, float *val)
{
    if (V < 1 || k < 1 || k > V || !row || !idx || !val) return ORA_ERR_ARG;
    unsigned char *taken = (unsigned char *)calloc((size_t)V, 1);
    if (!taken) return ORA_ERR_NOMEM;
    for (int r = 0; r < k; ++r) {
        int best = -1;
        for (int v = 0; v < V; ++v) {
            if (taken[v]) continue;
            if (best < 0 || ranks_above(row[v], v, row[best], best)) best = v;
        }
        taken[best] = 1;
        idx[r] = best;
        val[r] = row[best];
    }
    free(taken);
    return ORA_OK;
}
