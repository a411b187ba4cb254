// Host-side argument checks shared by the C entry points (lora_abi.cu and
// noalloc.cu), so that every entry point applies the same rules.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace lora {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline lora_status_t check_shape(const lora_shape_t *shape, Shape *out) {
    if (shape == nullptr) return LORA_ERR_INVALID_ARG;
    const lora_shape_t &s = *shape;
    if (s.S < 1 || s.S > LORA_MAX_SLOTS) return LORA_ERR_INVALID_ARG;
    if (s.n_slices < 1 || s.n_slices > LORA_MAX_SLICES) return LORA_ERR_INVALID_ARG;
    if (s.k < 8) return LORA_ERR_INVALID_ARG;
    if (s.k % 8 != 0) return LORA_ERR_ALIGNMENT;
    if (s.r_max < 8 || s.r_max > LORA_MAX_RANK || s.r_max % 8 != 0) return LORA_ERR_RANK;
    if (s.slice_offsets[0] != 0) return LORA_ERR_INVALID_ARG;
    for (int i = 0; i < s.n_slices; ++i) {
        const int32_t w = s.slice_offsets[i + 1] - s.slice_offsets[i];
        if (w <= 0) return LORA_ERR_INVALID_ARG;
        if (w % 8 != 0) return LORA_ERR_ALIGNMENT;
    }
    out->S = s.S;
    out->r_max = s.r_max;
    out->k = s.k;
    out->n = s.n_slices;
    for (int i = 0; i <= LORA_MAX_SLICES; ++i)
        out->off[i] = i <= s.n_slices ? s.slice_offsets[i] : s.slice_offsets[s.n_slices];
    return LORA_OK;
}

inline lora_status_t check_index_ptrs(const void *table, const int32_t *sorted_ids, const int32_t *seg,
                               const int32_t *active, int32_t T) {
    if (table == nullptr || seg == nullptr || active == nullptr) return LORA_ERR_INVALID_ARG;
    if (T > 0 && sorted_ids == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(table)) return LORA_ERR_ALIGNMENT;
    return LORA_OK;
}

inline lora_status_t check_rows(const void *p, int64_t ld, int32_t T, int32_t width) {
    if (T > 0 && p == nullptr) return LORA_ERR_INVALID_ARG;
    if (ld < width) return LORA_ERR_INVALID_ARG;
    if (!aligned16(p) || ld % 8 != 0) return LORA_ERR_ALIGNMENT;
    return LORA_OK;
}

}  // namespace lora
