// Host-side argument checks, the tree/chain geometry guard and status names.
//
// Every entry point runs these checks before queuing anything, so a bad call
// leaves the device untouched (lucebox PR #506, Safety boundary: malformed
// geometry is rejected before execution).
#include "gdn_host.h"

#include <cmath>
#include <vector>

#include <cuda_runtime.h>

namespace gdnhost {

int check_dims(const gdn_dims *d, int32_t n_tok) {
    if (!d) return GDN_ERR_NULL;
    if (d->in_dtype != GDN_F32 && d->in_dtype != GDN_BF16) return GDN_ERR_DTYPE;
    if (d->batch < 1 || d->layers < 1 || (int64_t)d->batch * d->layers > 65535) return GDN_ERR_DIMS;
    if (d->h_k < 1 || d->h_v < 1 || d->h_v % d->h_k != 0 || d->h_v > 65535) return GDN_ERR_DIMS;
    if (d->d_k != 64 && d->d_k != 128) return GDN_ERR_DIMS;
    if (d->d_v < 16 || d->d_v > 1024 || d->d_v % 16 != 0) return GDN_ERR_DIMS;
    if (d->conv_k < 1 || d->conv_k > GDN_MAX_CONV_K) return GDN_ERR_DIMS;
    const int64_t C = 2LL * d->h_k * d->d_k + (int64_t)d->h_v * d->d_v;
    if (C != d->conv_ch || C > (1LL << 30)) return GDN_ERR_DIMS;
    if (n_tok < 1 || n_tok > GDN_MAX_TOKENS) return GDN_ERR_DIMS;
    if (!std::isfinite(d->q_scale)) return GDN_ERR_DIMS;
    return GDN_OK;
}

int check_tree(const int32_t *parent, int32_t batch, int32_t n_nodes, bool require_chain,
               int32_t max_depth) {
    if (batch < 1) return GDN_ERR_DIMS;
    if (n_nodes < 2) return GDN_ERR_TREE_TRUNCATED;
    if (!parent) return GDN_ERR_NULL;
    std::vector<int32_t> depth((size_t)n_nodes);
    for (int32_t r = 0; r < batch; ++r) {
        const int32_t *p = parent + (size_t)r * n_nodes;
        if (p[0] != -1) return GDN_ERR_TREE_ROOT;
        depth[0] = 0;
        for (int32_t i = 1; i < n_nodes; ++i) {
            if (p[i] < 0 || p[i] >= i) return GDN_ERR_TREE_PARENT;
            if (require_chain && p[i] != i - 1) return GDN_ERR_TREE_NOT_CHAIN;
            depth[i] = depth[p[i]] + 1;
            if (max_depth > 0 && depth[i] > max_depth) return GDN_ERR_TREE_DEPTH;
        }
    }
    return GDN_OK;
}

int sm_count() {
    static int cached[256] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace gdnhost

extern "C" int gdn_tree_check(const int32_t *parent_host, int32_t batch, int32_t n_nodes,
                              int32_t require_chain, int32_t max_depth) {
    return gdnhost::check_tree(parent_host, batch, n_nodes, require_chain != 0, max_depth);
}

extern "C" const char *gdn_status_str(int status) {
    switch (status) {
        case GDN_OK: return "ok";
        case GDN_ERR_NULL: return "a required pointer is NULL";
        case GDN_ERR_DIMS: return "a size is outside the supported range";
        case GDN_ERR_ALIGN: return "a float buffer is not 16-byte aligned";
        case GDN_ERR_DTYPE: return "unsupported input dtype";
        case GDN_ERR_TREE_ROOT: return "tree: parent[0] must be -1 (malformed root)";
        case GDN_ERR_TREE_PARENT: return "tree: parent[i] must lie in [0, i) (forward, cyclic or out-of-range parent)";
        case GDN_ERR_TREE_DEPTH: return "tree: a node is deeper than allowed";
        case GDN_ERR_TREE_TRUNCATED: return "tree: fewer than two nodes";
        case GDN_ERR_TREE_NOT_CHAIN: return "tree: sibling or skipped parent where a pure chain is required";
        case GDN_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case GDN_ERR_CUDA: return "CUDA launch failed";
        case GDN_ERR_FLAGS: return "a flags argument has an undefined bit";
        default: return "unknown status";
    }
}
