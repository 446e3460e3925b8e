// Host-side validation shared by the gdnspec entry points (no CUDA calls).
#pragma once

#include <cstddef>
#include <cstdint>

#include "gdnspec.h"

namespace gdnhost {

// Checks gdn_dims and the span length (1..GDN_MAX_TOKENS).
int check_dims(const gdn_dims *d, int32_t n_tok);

// Pointer alignment helper.
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Geometry of B parent arrays (see gdn_tree_check).
int check_tree(const int32_t *parent, int32_t batch, int32_t n_nodes, bool require_chain,
               int32_t max_depth);

// Elements per checkpoint slot.
inline size_t ssm_slot_elems(const gdn_dims *d) {
    return (size_t)d->h_v * (size_t)d->d_v * (size_t)d->d_k;
}
inline size_t conv_slot_elems(const gdn_dims *d) {
    return (size_t)d->conv_ch * (size_t)(d->conv_k - 1);
}

// SM count of the current device (cached per device); 0 on failure.
int sm_count();

}  // namespace gdnhost
