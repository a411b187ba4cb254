// extern "C" entry points of the LoRA branch library: argument checks, slot
// table packing, workspace sizing and kernel dispatch.  Declarations and the
// contract of every call are in include/lora_gemm.h.
#include <algorithm>
#include <cmath>
#include <cstring>

#include "checks.cuh"
#include "common.cuh"

namespace lora {
cudaError_t launch_build_index(const int32_t *slot_ids, const int32_t *expert_ids, int32_t T, int32_t tps, int32_t K,
                               int32_t E, int32_t S, const void *table,
                               int32_t *sorted_ids, int32_t *seg_offsets, int32_t *active, int32_t *err,
                               cudaStream_t stream, const int32_t *seq_ids = nullptr,
                               const int32_t *positions = nullptr, const int32_t *seq_slot = nullptr,
                               const int32_t *invocation_start = nullptr, int32_t n_seq = 0);
cudaError_t launch_shrink(const uint16_t *x, int64_t ldx, const Shape &sh, const void *table,
                          const int32_t *sorted_ids, const int32_t *seg, float *xa, int32_t T, int32_t *err,
                          bool trigger_dependents, cudaStream_t stream);
cudaError_t launch_expand(const float *xa, uint16_t *y, int64_t ldy, const Shape &sh, const void *table,
                          const int32_t *sorted_ids, const int32_t *seg, int32_t T, int32_t *err,
                          bool programmatic, cudaStream_t stream);
cudaError_t launch_fused_decode(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                const void *table, const int32_t *sorted_ids, const int32_t *seg,
                                float *ws, int32_t T, int32_t *err, cudaStream_t stream);
cudaError_t launch_premultiply(uint16_t *w, int64_t n, float scale, cudaStream_t stream);
cudaError_t launch_premultiply_e4m3(uint8_t *w, int64_t n, double scale, cudaStream_t stream);
bool prefill_supported(int32_t r_max);
bool fused_decode_supported(int32_t T, int32_t r_max, int32_t k);
bool decode_direct_supported(int32_t T, const Shape &sh, bool fp8);
cudaError_t launch_direct_shrink(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                 const void *table, const int32_t *sorted_ids, const int32_t *seg,
                                 const int32_t *active, float *ws, int32_t T, int32_t *err, bool fp8,
                                 cudaStream_t stream, int32_t x_div = 1, const unsigned char *plan = nullptr);
cudaError_t launch_direct_expand(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                 const void *table, const int32_t *sorted_ids, const int32_t *seg,
                                 const int32_t *active, float *ws, int32_t T, int32_t *err, bool fp8,
                                 bool programmatic, cudaStream_t stream, const unsigned char *plan = nullptr);
cudaError_t launch_decode_direct(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                 const void *table, const int32_t *sorted_ids, const int32_t *seg,
                                 const int32_t *active, float *ws, int32_t T, int32_t *err, bool fp8,
                                 cudaStream_t stream, int32_t x_div = 1, const unsigned char *plan = nullptr);
size_t direct_plan_bytes(int32_t T, const Shape &sh);
cudaError_t launch_direct_plans(const Shape &sh, const void *const *tables, unsigned char *const *plans,
                                int32_t count, const int32_t *sorted_ids, const int32_t *seg, const int32_t *active,
                                int32_t T, bool fp8, int32_t *err, cudaStream_t stream);
cudaError_t launch_prefill(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                           const void *table, const int32_t *sorted_ids, const int32_t *seg, float *ws,
                           int32_t T, int32_t *err, cudaStream_t stream);
size_t tma_table_bytes(int32_t S, int32_t n);
bool encode_tma_table(void *host_buf, const Shape &sh, const int32_t *ranks, const uint64_t *A_ptrs,
                      const uint64_t *B_ptrs);
bool decode_tma_supported(int32_t T, const Shape &sh);
size_t tma_plan_bytes(int32_t T, const Shape &sh);
cudaError_t launch_tma_plans(const Shape &sh, const void *const *tables, unsigned char *const *plans, int32_t count,
                             const int32_t *sorted_ids, const int32_t *seg, const int32_t *active, int32_t T,
                             int32_t *err, cudaStream_t stream);
cudaError_t launch_tma_decode(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                              const unsigned char *plan, float *acc0, float *acc1, int32_t *ctrl, int32_t T,
                              int32_t *err, cudaStream_t stream, int32_t xdiv = 1);
bool cluster_decode_supported(int32_t T, const Shape &sh);
cudaError_t launch_cluster_decode(const uint16_t *x, int64_t ldx, uint16_t *y, int64_t ldy, const Shape &sh,
                                  const void *table, const int32_t *sorted_ids, const int32_t *seg, int32_t T,
                                  int32_t *err, cudaStream_t stream, int32_t xdiv = 1);
}  // namespace lora

using lora::Shape;
using lora::aligned16;
using lora::check_index_ptrs;
using lora::check_rows;
using lora::check_shape;

namespace {

lora_status_t check_ws(const float *ws, size_t ws_bytes, int32_t T, const Shape &sh) {
    const lora::WorkspaceLayout L(T, sh.n, sh.r_max, sh.S);
    if (ws == nullptr || ws_bytes < L.bytes) return LORA_ERR_WORKSPACE;
    if (!aligned16(ws)) return LORA_ERR_ALIGNMENT;
    return LORA_OK;
}

lora_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? LORA_OK : LORA_ERR_CUDA; }

constexpr int32_t kSmallDecodeT = 64;

bool fused_ok(int32_t T, const Shape &sh) { return lora::fused_decode_supported(T, sh.r_max, sh.k); }

lora_path_t resolve(lora_path_t path, int32_t T, int32_t max_seg_hint, const Shape &sh, int32_t *launches) {
    if (max_seg_hint <= 0 || max_seg_hint > T) max_seg_hint = T;
    if (path == LORA_PATH_AUTO) {
        // measured on GB300: the warp-streaming kernels lead from a few hundred
        // tokens up; at 64 tokens and fewer the one-cluster-per-slot kernel (a
        // 64-token q_proj call: 8.8 us against 11.0 for the split kernels)
        if (max_seg_hint > LORA_DECODE_MAX_SEG && lora::prefill_supported(sh.r_max)) path = LORA_PATH_PREFILL;
        else if (T > kSmallDecodeT && lora::decode_direct_supported(T, sh, false)) path = LORA_PATH_DECODE_DIRECT;
        else if (T > kSmallDecodeT && fused_ok(T, sh)) path = LORA_PATH_DECODE_FUSED;
        else if (T <= kSmallDecodeT && lora::cluster_decode_supported(T, sh)) path = LORA_PATH_DECODE_CLUSTER;
        else path = LORA_PATH_DECODE_SPLIT;
    }
    if (launches != nullptr)
        *launches = ((path == LORA_PATH_DECODE_FUSED && lora::fused_decode_supported(T, sh.r_max, sh.k)) ||
                     path == LORA_PATH_DECODE_CLUSTER)
                        ? 1
                        : 2;
    return path;
}

// The one-kernel TMA decode call on a plan (its own or the workspace's).
lora_status_t tma_call(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T, const Shape &sh,
                       const unsigned char *plan, float *ws, int32_t *err, cudaStream_t s, int32_t xdiv = 1) {
    const lora::WorkspaceLayout L(T, sh.n, sh.r_max, sh.S);
    char *base = reinterpret_cast<char *>(ws);
    return from_cuda(lora::launch_tma_decode(static_cast<const uint16_t *>(x), ldx, static_cast<uint16_t *>(y), ldy,
                                             sh, plan, reinterpret_cast<float *>(base + L.tacc0_off),
                                             reinterpret_cast<float *>(base + L.tacc1_off),
                                             reinterpret_cast<int32_t *>(base + L.tctrl_off), T, err, s, xdiv));
}

float *xa_of(float *ws, int32_t T, const Shape &sh) {
    const lora::WorkspaceLayout L(T, sh.n, sh.r_max, sh.S);
    return reinterpret_cast<float *>(reinterpret_cast<char *>(ws) + L.xa_off);
}

}  // namespace

extern "C" {

int32_t lora_abi_version(void) { return LORA_ABI_VERSION; }

const char *lora_status_string(lora_status_t status) {
    switch (status) {
    case LORA_OK: return "LORA_OK";
    case LORA_ERR_INVALID_ARG: return "LORA_ERR_INVALID_ARG: invalid argument (null pointer, size or shape)";
    case LORA_ERR_ALIGNMENT: return "LORA_ERR_ALIGNMENT: pointer, leading dimension or width not 16-byte aligned";
    case LORA_ERR_RANK: return "LORA_ERR_RANK: rank not 0 or a multiple of 8, or above r_max / LORA_MAX_RANK";
    case LORA_ERR_SLOT_RANGE: return "LORA_ERR_SLOT_RANGE: a slot id outside [-1, S)";
    case LORA_ERR_NULL_WEIGHT: return "LORA_ERR_NULL_WEIGHT: a slot with rank > 0 has a null A or B pointer";
    case LORA_ERR_WORKSPACE: return "LORA_ERR_WORKSPACE: workspace missing or too small";
    case LORA_ERR_TIMEOUT: return "LORA_ERR_TIMEOUT: a bounded wait between thread blocks gave up";
    case LORA_ERR_CUDA: return "LORA_ERR_CUDA: a CUDA runtime call failed";
    case LORA_ERR_UNSUPPORTED: return "LORA_ERR_UNSUPPORTED: no kernel for this device or configuration";
    }
    return "LORA_ERR_UNKNOWN";
}

double lora_scale(double alpha, int32_t rank, int32_t rslora, double adapter_scale) {
    if (rank <= 0 || alpha == 0.0) return adapter_scale;
    const double denom = rslora ? std::sqrt(static_cast<double>(rank)) : static_cast<double>(rank);
    return adapter_scale * alpha / denom;
}

lora_status_t lora_premultiply(void *w, int64_t n, float scale, lora_stream_t stream) {
    if (n < 0 || (n > 0 && w == nullptr)) return LORA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(w) & 1u) != 0) return LORA_ERR_ALIGNMENT;
    return from_cuda(lora::launch_premultiply(static_cast<uint16_t *>(w), n, scale,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_premultiply_e4m3(void *w, int64_t n, float scale, lora_stream_t stream) {
    if (n < 0 || (n > 0 && w == nullptr)) return LORA_ERR_INVALID_ARG;
    return from_cuda(lora::launch_premultiply_e4m3(static_cast<uint8_t *>(w), n, static_cast<double>(scale),
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

size_t lora_slot_table_bytes(int32_t S, int32_t n_slices) {
    if (S < 1 || n_slices < 1) return 0;
    return lora::TableLayout(S, n_slices).bytes;
}

lora_status_t lora_pack_slot_table(void *host_buf, int32_t S, int32_t n_slices, int32_t r_max,
                                   const int32_t *ranks, const float *scales, const uint64_t *A_ptrs,
                                   const uint64_t *B_ptrs) {
    if (host_buf == nullptr || ranks == nullptr || scales == nullptr || A_ptrs == nullptr || B_ptrs == nullptr)
        return LORA_ERR_INVALID_ARG;
    if (S < 1 || S > LORA_MAX_SLOTS || n_slices < 1 || n_slices > LORA_MAX_SLICES) return LORA_ERR_INVALID_ARG;
    if (r_max < 8 || r_max > LORA_MAX_RANK || r_max % 8 != 0) return LORA_ERR_RANK;
    for (int32_t s = 0; s < S; ++s) {
        const int32_t r = ranks[s];
        if (r < 0 || r % 8 != 0 || r > r_max) return LORA_ERR_RANK;
        if (!std::isfinite(scales[s])) return LORA_ERR_INVALID_ARG;
        if (r == 0) continue;
        for (int32_t i = 0; i < n_slices; ++i) {
            const uint64_t a = A_ptrs[s * n_slices + i], b = B_ptrs[s * n_slices + i];
            if (a == 0 || b == 0) return LORA_ERR_NULL_WEIGHT;
            if ((a & 15u) != 0 || (b & 15u) != 0) return LORA_ERR_ALIGNMENT;
        }
    }
    const lora::TableLayout L(S, n_slices);
    char *p = static_cast<char *>(host_buf);
    std::memset(p, 0, L.bytes);
    const int32_t hdr[4] = {lora::kTableMagic, S, n_slices, r_max};
    std::memcpy(p, hdr, sizeof hdr);
    std::memcpy(p + L.rank_off, ranks, sizeof(int32_t) * size_t(S));
    std::memcpy(p + L.scale_off, scales, sizeof(float) * size_t(S));
    uint64_t *a = reinterpret_cast<uint64_t *>(p + L.a_off);
    uint64_t *b = reinterpret_cast<uint64_t *>(p + L.b_off);
    for (int32_t e = 0; e < S * n_slices; ++e) {
        const bool used = ranks[e / n_slices] > 0;  // empty slots carry null pointers
        a[e] = used ? A_ptrs[e] : 0;
        b[e] = used ? B_ptrs[e] : 0;
    }
    return LORA_OK;
}

lora_status_t lora_set_slot_table(void *dev_table, void *host_staging, int32_t S, int32_t n_slices,
                                  int32_t r_max, const int32_t *ranks, const float *scales,
                                  const uint64_t *A_ptrs, const uint64_t *B_ptrs, lora_stream_t stream) {
    if (dev_table == nullptr || host_staging == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(dev_table)) return LORA_ERR_ALIGNMENT;
    const lora_status_t st = lora_pack_slot_table(host_staging, S, n_slices, r_max, ranks, scales, A_ptrs, B_ptrs);
    if (st != LORA_OK) return st;
    return from_cuda(cudaMemcpyAsync(dev_table, host_staging, lora::TableLayout(S, n_slices).bytes,
                                     cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream)));
}

size_t lora_slot_table_tma_bytes(int32_t S, const lora_shape_t *shape) {
    Shape sh;
    if (S < 1 || S > LORA_MAX_SLOTS || check_shape(shape, &sh) != LORA_OK || sh.S != S) return 0;
    return lora::tma_table_bytes(S, sh.n);
}

lora_status_t lora_set_slot_table_tma(void *dev_table, void *host_staging, const lora_shape_t *shape,
                                      const int32_t *ranks, const float *scales, const uint64_t *A_ptrs,
                                      const uint64_t *B_ptrs, lora_stream_t stream) {
    Shape sh;
    lora_status_t st;
    if (dev_table == nullptr || host_staging == nullptr) return LORA_ERR_INVALID_ARG;
    if ((st = check_shape(shape, &sh)) != LORA_OK) return st;
    if ((reinterpret_cast<uintptr_t>(dev_table) & 127u) != 0) return LORA_ERR_ALIGNMENT;
    if ((st = lora_pack_slot_table(host_staging, sh.S, sh.n, sh.r_max, ranks, scales, A_ptrs, B_ptrs)) != LORA_OK)
        return st;
    if (!lora::encode_tma_table(host_staging, sh, ranks, A_ptrs, B_ptrs)) return LORA_ERR_UNSUPPORTED;
    return from_cuda(cudaMemcpyAsync(dev_table, host_staging, lora::tma_table_bytes(sh.S, sh.n),
                                     cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_build_index(const int32_t *slot_ids, int32_t T, int32_t S, const void *dev_table,
                               int32_t *sorted_ids, int32_t *seg_offsets, int32_t *active, int32_t *err,
                               lora_stream_t stream) {
    if (T < 0 || S < 1 || S > LORA_MAX_SLOTS) return LORA_ERR_INVALID_ARG;
    if (T > 0 && (slot_ids == nullptr || sorted_ids == nullptr)) return LORA_ERR_INVALID_ARG;
    if (dev_table == nullptr || seg_offsets == nullptr || active == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(dev_table)) return LORA_ERR_ALIGNMENT;
    return from_cuda(lora::launch_build_index(slot_ids, nullptr, T, 1, 1, 1, S, dev_table, sorted_ids, seg_offsets,
                                              active, err, reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_build_index_seq(const int32_t *seq_slot_ids, int32_t n_seq, int32_t tokens_per_seq, int32_t S,
                                   const void *dev_table, int32_t *sorted_ids, int32_t *seg_offsets,
                                   int32_t *active, int32_t *err, lora_stream_t stream) {
    if (n_seq < 0 || tokens_per_seq < 1 || S < 1 || S > LORA_MAX_SLOTS) return LORA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(n_seq) * tokens_per_seq > INT32_MAX) return LORA_ERR_INVALID_ARG;
    if (n_seq > 0 && (seq_slot_ids == nullptr || sorted_ids == nullptr)) return LORA_ERR_INVALID_ARG;
    if (dev_table == nullptr || seg_offsets == nullptr || active == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(dev_table)) return LORA_ERR_ALIGNMENT;
    return from_cuda(lora::launch_build_index(seq_slot_ids, nullptr, n_seq, tokens_per_seq, 1, 1, S, dev_table,
                                              sorted_ids, seg_offsets, active, err,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_build_index_activated(const int32_t *seq_ids, const int32_t *positions, int32_t T,
                                         const int32_t *seq_slot, const int32_t *invocation_start, int32_t n_seq,
                                         int32_t S, const void *dev_table, int32_t *sorted_ids, int32_t *seg_offsets,
                                         int32_t *active, int32_t *err, lora_stream_t stream) {
    if (T < 0 || n_seq < 0 || S < 1 || S > LORA_MAX_SLOTS) return LORA_ERR_INVALID_ARG;
    if (T > 0 && (seq_ids == nullptr || positions == nullptr || sorted_ids == nullptr)) return LORA_ERR_INVALID_ARG;
    if (n_seq > 0 && (seq_slot == nullptr || invocation_start == nullptr)) return LORA_ERR_INVALID_ARG;
    if (dev_table == nullptr || seg_offsets == nullptr || active == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(dev_table)) return LORA_ERR_ALIGNMENT;
    return from_cuda(lora::launch_build_index(seq_ids, nullptr, T, 1, 1, 1, S, dev_table, sorted_ids, seg_offsets,
                                              active, err, reinterpret_cast<cudaStream_t>(stream), seq_ids,
                                              positions, seq_slot, invocation_start, n_seq));
}

lora_status_t lora_build_index_moe(const int32_t *slot_ids, const int32_t *expert_ids, int32_t T, int32_t K,
                                   int32_t E, int32_t S, const void *dev_table, int32_t *sorted_ids,
                                   int32_t *seg_offsets, int32_t *active, int32_t *err, lora_stream_t stream) {
    if (T < 0 || K < 1 || E < 1 || S < 1 || S > LORA_MAX_SLOTS || S % E != 0) return LORA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * K > INT32_MAX) return LORA_ERR_INVALID_ARG;
    if (T > 0 && (slot_ids == nullptr || expert_ids == nullptr || sorted_ids == nullptr)) return LORA_ERR_INVALID_ARG;
    if (dev_table == nullptr || seg_offsets == nullptr || active == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(dev_table)) return LORA_ERR_ALIGNMENT;
    return from_cuda(lora::launch_build_index(slot_ids, expert_ids, T * K, 1, K, E, S, dev_table, sorted_ids,
                                              seg_offsets, active, err, reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_moe_slot_pointers(int32_t n_adapters, int32_t E, const lora_shape_t *shape, int32_t elem_bytes,
                                     const int32_t *ranks, const float *scales, const uint64_t *A_base,
                                     const uint64_t *B_base, int32_t *v_ranks, float *v_scales, uint64_t *A_ptrs,
                                     uint64_t *B_ptrs) {
    Shape sh;
    if (n_adapters < 1 || E < 1 || (elem_bytes != 1 && elem_bytes != 2)) return LORA_ERR_INVALID_ARG;
    if (ranks == nullptr || scales == nullptr || A_base == nullptr || B_base == nullptr || v_ranks == nullptr ||
        v_scales == nullptr || A_ptrs == nullptr || B_ptrs == nullptr)
        return LORA_ERR_INVALID_ARG;
    const lora_status_t st = check_shape(shape, &sh);
    if (st != LORA_OK) return st;
    if (static_cast<int64_t>(n_adapters) * E != sh.S) return LORA_ERR_INVALID_ARG;
    for (int32_t a = 0; a < n_adapters; ++a) {
        const int32_t r = ranks[a];
        for (int32_t e = 0; e < E; ++e) {
            const int32_t v = a * E + e;
            v_ranks[v] = r;
            v_scales[v] = scales[a];
            for (int32_t i = 0; i < sh.n; ++i) {
                const uint64_t ab = A_base[a * sh.n + i], bb = B_base[a * sh.n + i];
                const uint64_t di = static_cast<uint64_t>(sh.off[i + 1] - sh.off[i]);
                // expert e's slice starts expert * dim * rank elements in
                A_ptrs[v * sh.n + i] = ab == 0 ? 0 : ab + static_cast<uint64_t>(e) * r * sh.k * elem_bytes;
                B_ptrs[v * sh.n + i] = bb == 0 ? 0 : bb + static_cast<uint64_t>(e) * di * r * elem_bytes;
            }
        }
    }
    return LORA_OK;
}

lora_status_t lora_workspace_bytes(int32_t T, const lora_shape_t *shape, size_t *bytes) {
    Shape sh;
    if (bytes == nullptr || T < 0) return LORA_ERR_INVALID_ARG;
    const lora_status_t st = check_shape(shape, &sh);
    if (st != LORA_OK) return st;
    *bytes = lora::WorkspaceLayout(T, sh.n, sh.r_max, sh.S).bytes;
    return LORA_OK;
}

size_t lora_workspace_xa_offset(const lora_shape_t *shape) {
    Shape sh;
    if (check_shape(shape, &sh) != LORA_OK) return 0;
    return lora::WorkspaceLayout(0, sh.n, sh.r_max, sh.S).xa_off;
}

lora_status_t lora_shrink(const void *x, int64_t ldx, int32_t T, const lora_shape_t *shape, const void *dev_table,
                          const int32_t *sorted_ids, const int32_t *seg_offsets, const int32_t *active,
                          float *ws, size_t ws_bytes, int32_t *err, lora_stream_t stream) {
    Shape sh;
    lora_status_t st;
    if (T < 0) return LORA_ERR_INVALID_ARG;
    if ((st = check_shape(shape, &sh)) != LORA_OK) return st;
    if ((st = check_index_ptrs(dev_table, sorted_ids, seg_offsets, active, T)) != LORA_OK) return st;
    if ((st = check_rows(x, ldx, T, sh.k)) != LORA_OK) return st;
    if ((st = check_ws(ws, ws_bytes, T, sh)) != LORA_OK) return st;
    if (T == 0) return LORA_OK;
    return from_cuda(lora::launch_shrink(static_cast<const uint16_t *>(x), ldx, sh, dev_table, sorted_ids,
                                         seg_offsets, xa_of(ws, T, sh), T, err, false,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_expand(const float *ws, size_t ws_bytes, void *y, int64_t ldy, int32_t T,
                          const lora_shape_t *shape, const void *dev_table, const int32_t *sorted_ids,
                          const int32_t *seg_offsets, const int32_t *active, int32_t *err, lora_stream_t stream) {
    Shape sh;
    lora_status_t st;
    if (T < 0) return LORA_ERR_INVALID_ARG;
    if ((st = check_shape(shape, &sh)) != LORA_OK) return st;
    if ((st = check_index_ptrs(dev_table, sorted_ids, seg_offsets, active, T)) != LORA_OK) return st;
    if ((st = check_rows(y, ldy, T, sh.off[sh.n])) != LORA_OK) return st;
    if ((st = check_ws(ws, ws_bytes, T, sh)) != LORA_OK) return st;
    if (T == 0) return LORA_OK;
    return from_cuda(lora::launch_expand(xa_of(const_cast<float *>(ws), T, sh), static_cast<uint16_t *>(y), ldy,
                                         sh, dev_table, sorted_ids, seg_offsets, T, err, false,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

lora_path_t lora_resolve_path(lora_path_t requested, int32_t T, int32_t max_seg_hint, int32_t *launches) {
    // without a shape the rank bound is unknown here: report the choice for one
    // 4096 -> 4096 slice with r_max 64; lora_apply_ex re-resolves with the shape
    Shape sh{};
    sh.S = 1;
    sh.r_max = 64;
    sh.k = 4096;
    sh.n = 1;
    for (int i = 1; i <= LORA_MAX_SLICES; ++i) sh.off[i] = 4096;
    return resolve(requested, T, max_seg_hint, sh, launches);
}

lora_status_t lora_apply_ex(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T, const lora_shape_t *shape,
                            const void *dev_table, const int32_t *sorted_ids, const int32_t *seg_offsets,
                            const int32_t *active, int32_t max_seg_hint, lora_path_t path, float *ws,
                            size_t ws_bytes, int32_t *err, lora_stream_t stream) {
    Shape sh;
    lora_status_t st;
    if (T < 0) return LORA_ERR_INVALID_ARG;
    if ((st = check_shape(shape, &sh)) != LORA_OK) return st;
    if ((st = check_index_ptrs(dev_table, sorted_ids, seg_offsets, active, T)) != LORA_OK) return st;
    if ((st = check_rows(x, ldx, T, sh.k)) != LORA_OK) return st;
    if ((st = check_rows(y, ldy, T, sh.off[sh.n])) != LORA_OK) return st;
    if ((st = check_ws(ws, ws_bytes, T, sh)) != LORA_OK) return st;
    if (T == 0) return LORA_OK;
    if (max_seg_hint <= 0 || max_seg_hint > T) max_seg_hint = T;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const uint16_t *xb = static_cast<const uint16_t *>(x);
    uint16_t *yb = static_cast<uint16_t *>(y);
    path = resolve(path, T, max_seg_hint, sh, nullptr);
    switch (path) {
    case LORA_PATH_DECODE_FUSED:
        if (!lora::fused_decode_supported(T, sh.r_max, sh.k)) return LORA_ERR_UNSUPPORTED;
        return from_cuda(lora::launch_fused_decode(xb, ldx, yb, ldy, sh, dev_table, sorted_ids, seg_offsets, ws, T,
                                                   err, s));
    case LORA_PATH_DECODE_TC:
    case LORA_PATH_DECODE_STREAM:
        return LORA_ERR_UNSUPPORTED;  // retired: slower than LORA_PATH_DECODE_DIRECT on every measured shape
    case LORA_PATH_DECODE_DIRECT:
    case LORA_PATH_DECODE_DIRECT_FP8: {
        const bool fp8 = path == LORA_PATH_DECODE_DIRECT_FP8;
        if (!lora::decode_direct_supported(T, sh, fp8)) return LORA_ERR_UNSUPPORTED;
        return from_cuda(lora::launch_decode_direct(xb, ldx, yb, ldy, sh, dev_table, sorted_ids, seg_offsets, active,
                                                    ws, T, err, fp8, s));
    }
    case LORA_PATH_DECODE_SPLIT: {
        float *xa = xa_of(ws, T, sh);
        cudaError_t e = lora::launch_shrink(xb, ldx, sh, dev_table, sorted_ids, seg_offsets, xa, T, err, true, s);
        if (e != cudaSuccess) return LORA_ERR_CUDA;
        return from_cuda(lora::launch_expand(xa, yb, ldy, sh, dev_table, sorted_ids, seg_offsets, T, err, true, s));
    }
    case LORA_PATH_PREFILL:
        if (!lora::prefill_supported(sh.r_max)) return LORA_ERR_UNSUPPORTED;
        return from_cuda(lora::launch_prefill(xb, ldx, yb, ldy, sh, dev_table, sorted_ids, seg_offsets, ws, T, err, s));
    case LORA_PATH_DECODE_TMA: {
        // a plan for this call in the workspace, then the call on it
        if (!lora::decode_tma_supported(T, sh)) return LORA_ERR_UNSUPPORTED;
        const lora::WorkspaceLayout L(T, sh.n, sh.r_max, sh.S);
        unsigned char *plan = reinterpret_cast<unsigned char *>(ws) + L.tplan_off;
        if (lora::launch_tma_plans(sh, &dev_table, &plan, 1, sorted_ids, seg_offsets, active, T, err, s) !=
            cudaSuccess)
            return LORA_ERR_CUDA;
        return tma_call(x, ldx, y, ldy, T, sh, plan, ws, err, s);
    }
    case LORA_PATH_DECODE_CLUSTER:
        if (!lora::cluster_decode_supported(T, sh)) return LORA_ERR_UNSUPPORTED;
        return from_cuda(lora::launch_cluster_decode(xb, ldx, yb, ldy, sh, dev_table, sorted_ids, seg_offsets, T, err,
                                                     s));
    default:
        return LORA_ERR_INVALID_ARG;
    }
}

lora_status_t lora_apply_overlap(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T,
                                 const lora_shape_t *shape, const void *dev_table, const int32_t *sorted_ids,
                                 const int32_t *seg_offsets, const int32_t *active, int32_t max_seg_hint,
                                 lora_path_t path, float *ws, size_t ws_bytes, int32_t *err, lora_stream_t stream,
                                 lora_event_t y_ready) {
    Shape sh;
    lora_status_t st;
    if (T < 0) return LORA_ERR_INVALID_ARG;
    if ((st = check_shape(shape, &sh)) != LORA_OK) return st;
    if ((st = check_index_ptrs(dev_table, sorted_ids, seg_offsets, active, T)) != LORA_OK) return st;
    if ((st = check_rows(x, ldx, T, sh.k)) != LORA_OK) return st;
    if ((st = check_rows(y, ldy, T, sh.off[sh.n])) != LORA_OK) return st;
    if ((st = check_ws(ws, ws_bytes, T, sh)) != LORA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaEvent_t ev = reinterpret_cast<cudaEvent_t>(y_ready);
    if (max_seg_hint <= 0 || max_seg_hint > T) max_seg_hint = T;
    const lora_path_t p = T == 0 ? LORA_PATH_DECODE_SPLIT : resolve(path, T, max_seg_hint, sh, nullptr);
    const uint16_t *xb = static_cast<const uint16_t *>(x);
    uint16_t *yb = static_cast<uint16_t *>(y);
    const bool fp8 = p == LORA_PATH_DECODE_DIRECT_FP8;
    if (T > 0 && (p == LORA_PATH_DECODE_DIRECT || fp8)) {
        if (!lora::decode_direct_supported(T, sh, fp8)) return LORA_ERR_UNSUPPORTED;
        if (lora::launch_direct_shrink(xb, ldx, yb, ldy, sh, dev_table, sorted_ids, seg_offsets, active, ws, T, err,
                                       fp8, s) != cudaSuccess)
            return LORA_ERR_CUDA;
        if (ev != nullptr && cudaStreamWaitEvent(s, ev, 0) != cudaSuccess) return LORA_ERR_CUDA;
        return from_cuda(lora::launch_direct_expand(xb, ldx, yb, ldy, sh, dev_table, sorted_ids, seg_offsets, active,
                                                    ws, T, err, fp8, false, s));
    }
    if (T > 0 && p == LORA_PATH_DECODE_SPLIT) {
        float *xa = xa_of(ws, T, sh);
        if (lora::launch_shrink(xb, ldx, sh, dev_table, sorted_ids, seg_offsets, xa, T, err, false, s) != cudaSuccess)
            return LORA_ERR_CUDA;
        if (ev != nullptr && cudaStreamWaitEvent(s, ev, 0) != cudaSuccess) return LORA_ERR_CUDA;
        return from_cuda(lora::launch_expand(xa, yb, ldy, sh, dev_table, sorted_ids, seg_offsets, T, err, false, s));
    }
    // one-launch and tensor-core paths: y is ready before any of their work
    if (ev != nullptr && cudaStreamWaitEvent(s, ev, 0) != cudaSuccess) return LORA_ERR_CUDA;
    return lora_apply_ex(x, ldx, y, ldy, T, shape, dev_table, sorted_ids, seg_offsets, active, max_seg_hint, p, ws,
                         ws_bytes, err, stream);
}

lora_status_t lora_apply_moe_ex(const void *x, int64_t ldx, int32_t x_per_token, void *y, int64_t ldy, int32_t T,
                                int32_t K, const lora_shape_t *shape, const void *dev_table, const int32_t *sorted_ids,
                                const int32_t *seg_offsets, const int32_t *active, lora_path_t path, float *ws,
                                size_t ws_bytes, int32_t *err, lora_stream_t stream) {
    Shape sh;
    lora_status_t st;
    if (T < 0 || K < 1 || static_cast<int64_t>(T) * K > INT32_MAX) return LORA_ERR_INVALID_ARG;
    const int32_t P = T * K;  // (token, choice) pairs: the rows of y
    if ((st = check_shape(shape, &sh)) != LORA_OK) return st;
    if ((st = check_index_ptrs(dev_table, sorted_ids, seg_offsets, active, P)) != LORA_OK) return st;
    if ((st = check_rows(x, ldx, x_per_token ? T : P, sh.k)) != LORA_OK) return st;
    if ((st = check_rows(y, ldy, P, sh.off[sh.n])) != LORA_OK) return st;
    if ((st = check_ws(ws, ws_bytes, P, sh)) != LORA_OK) return st;
    if (path != LORA_PATH_DECODE_DIRECT && path != LORA_PATH_DECODE_TMA && path != LORA_PATH_DECODE_CLUSTER)
        return LORA_ERR_UNSUPPORTED;
    if (P == 0) return LORA_OK;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (path == LORA_PATH_DECODE_CLUSTER) {
        if (!lora::cluster_decode_supported(P, sh)) return LORA_ERR_UNSUPPORTED;
        return from_cuda(lora::launch_cluster_decode(static_cast<const uint16_t *>(x), ldx, static_cast<uint16_t *>(y),
                                                     ldy, sh, dev_table, sorted_ids, seg_offsets, P, err, s,
                                                     x_per_token ? K : 1));
    }
    if (path == LORA_PATH_DECODE_TMA) {
        if (!lora::decode_tma_supported(P, sh)) return LORA_ERR_UNSUPPORTED;
        const lora::WorkspaceLayout L(P, sh.n, sh.r_max, sh.S);
        unsigned char *plan = reinterpret_cast<unsigned char *>(ws) + L.tplan_off;
        if (lora::launch_tma_plans(sh, &dev_table, &plan, 1, sorted_ids, seg_offsets, active, P, err, s) !=
            cudaSuccess)
            return LORA_ERR_CUDA;
        return tma_call(x, ldx, y, ldy, P, sh, plan, ws, err, s, x_per_token ? K : 1);
    }
    if (!lora::decode_direct_supported(P, sh, false)) return LORA_ERR_UNSUPPORTED;
    return from_cuda(lora::launch_decode_direct(static_cast<const uint16_t *>(x), ldx, static_cast<uint16_t *>(y), ldy,
                                                sh, dev_table, sorted_ids, seg_offsets, active, ws, P, err, false, s,
                                                x_per_token ? K : 1));
}

lora_status_t lora_apply_moe(const void *x, int64_t ldx, int32_t x_per_token, void *y, int64_t ldy, int32_t T,
                             int32_t K, const lora_shape_t *shape, const void *dev_table, const int32_t *sorted_ids,
                             const int32_t *seg_offsets, const int32_t *active, float *ws, size_t ws_bytes,
                             int32_t *err, lora_stream_t stream) {
    return lora_apply_moe_ex(x, ldx, x_per_token, y, ldy, T, K, shape, dev_table, sorted_ids, seg_offsets, active,
                             LORA_PATH_DECODE_DIRECT, ws, ws_bytes, err, stream);
}

size_t lora_plan_bytes(int32_t T, const lora_shape_t *shape) {
    Shape sh;
    if (T < 1 || check_shape(shape, &sh) != LORA_OK) return 0;
    return std::max(lora::direct_plan_bytes(T, sh), lora::tma_plan_bytes(T, sh));
}

lora_status_t lora_build_plans(int32_t T, const lora_shape_t *shape, int32_t count, const void *const *dev_tables,
                               void *const *plans, size_t plan_bytes, const int32_t *sorted_ids,
                               const int32_t *seg_offsets, const int32_t *active, lora_path_t path, int32_t *err,
                               lora_stream_t stream) {
    Shape sh;
    lora_status_t st;
    if (T < 1 || count < 0 || (count > 0 && (dev_tables == nullptr || plans == nullptr))) return LORA_ERR_INVALID_ARG;
    if ((st = check_shape(shape, &sh)) != LORA_OK) return st;
    if (path == LORA_PATH_DECODE_TMA) {
        if (!lora::decode_tma_supported(T, sh)) return LORA_ERR_UNSUPPORTED;
        if (plan_bytes < lora::tma_plan_bytes(T, sh)) return LORA_ERR_WORKSPACE;
        for (int32_t j = 0; j < count; ++j) {
            if ((st = check_index_ptrs(dev_tables[j], sorted_ids, seg_offsets, active, T)) != LORA_OK) return st;
            if (plans[j] == nullptr) return LORA_ERR_WORKSPACE;
            if (!aligned16(plans[j])) return LORA_ERR_ALIGNMENT;
        }
        if (count == 0) return LORA_OK;
        return from_cuda(lora::launch_tma_plans(sh, dev_tables, reinterpret_cast<unsigned char *const *>(plans), count,
                                                sorted_ids, seg_offsets, active, T, err,
                                                reinterpret_cast<cudaStream_t>(stream)));
    }
    if (path != LORA_PATH_DECODE_DIRECT && path != LORA_PATH_DECODE_DIRECT_FP8) return LORA_ERR_UNSUPPORTED;
    const bool fp8 = path == LORA_PATH_DECODE_DIRECT_FP8;
    if (!lora::decode_direct_supported(T, sh, fp8)) return LORA_ERR_UNSUPPORTED;
    if (plan_bytes < lora::direct_plan_bytes(T, sh)) return LORA_ERR_WORKSPACE;
    for (int32_t j = 0; j < count; ++j) {
        if ((st = check_index_ptrs(dev_tables[j], sorted_ids, seg_offsets, active, T)) != LORA_OK) return st;
        if (plans[j] == nullptr) return LORA_ERR_WORKSPACE;
        if (!aligned16(plans[j])) return LORA_ERR_ALIGNMENT;
    }
    if (count == 0) return LORA_OK;
    return from_cuda(lora::launch_direct_plans(sh, dev_tables, reinterpret_cast<unsigned char *const *>(plans), count,
                                               sorted_ids, seg_offsets, active, T, fp8, err,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

lora_status_t lora_build_plan(int32_t T, const lora_shape_t *shape, const void *dev_table, const int32_t *sorted_ids,
                              const int32_t *seg_offsets, const int32_t *active, lora_path_t path, void *plan,
                              size_t plan_bytes, int32_t *err, lora_stream_t stream) {
    if (plan == nullptr) return LORA_ERR_WORKSPACE;
    return lora_build_plans(T, shape, 1, &dev_table, &plan, plan_bytes, sorted_ids, seg_offsets, active, path, err,
                            stream);
}

lora_status_t lora_apply_plan(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T, const lora_shape_t *shape,
                              const void *plan, size_t plan_bytes, lora_path_t path, float *ws, size_t ws_bytes,
                              int32_t *err, lora_stream_t stream) {
    Shape sh;
    lora_status_t st;
    if (T < 0) return LORA_ERR_INVALID_ARG;
    if ((st = check_shape(shape, &sh)) != LORA_OK) return st;
    if ((st = check_rows(x, ldx, T, sh.k)) != LORA_OK) return st;
    if ((st = check_rows(y, ldy, T, sh.off[sh.n])) != LORA_OK) return st;
    if ((st = check_ws(ws, ws_bytes, T, sh)) != LORA_OK) return st;
    if (T == 0) return LORA_OK;
    if (path == LORA_PATH_DECODE_TMA) {
        if (!lora::decode_tma_supported(T, sh)) return LORA_ERR_UNSUPPORTED;
        if (plan == nullptr || plan_bytes < lora::tma_plan_bytes(T, sh)) return LORA_ERR_WORKSPACE;
        if (!aligned16(plan)) return LORA_ERR_ALIGNMENT;
        return tma_call(x, ldx, y, ldy, T, sh, static_cast<const unsigned char *>(plan), ws, err,
                        reinterpret_cast<cudaStream_t>(stream));
    }
    if (path != LORA_PATH_DECODE_DIRECT && path != LORA_PATH_DECODE_DIRECT_FP8) return LORA_ERR_UNSUPPORTED;
    const bool fp8 = path == LORA_PATH_DECODE_DIRECT_FP8;
    if (!lora::decode_direct_supported(T, sh, fp8)) return LORA_ERR_UNSUPPORTED;
    if (plan == nullptr || plan_bytes < lora::direct_plan_bytes(T, sh)) return LORA_ERR_WORKSPACE;
    if (!aligned16(plan)) return LORA_ERR_ALIGNMENT;
    return from_cuda(lora::launch_decode_direct(static_cast<const uint16_t *>(x), ldx, static_cast<uint16_t *>(y), ldy,
                                                sh, nullptr, nullptr, nullptr, nullptr, ws, T, err, fp8,
                                                reinterpret_cast<cudaStream_t>(stream), 1,
                                                static_cast<const unsigned char *>(plan)));
}

lora_status_t lora_apply_moe_plan_ex(const void *x, int64_t ldx, int32_t x_per_token, void *y, int64_t ldy,
                                     int32_t T, int32_t K, const lora_shape_t *shape, const void *plan,
                                     size_t plan_bytes, lora_path_t path, float *ws, size_t ws_bytes, int32_t *err,
                                     lora_stream_t stream) {
    Shape sh;
    lora_status_t st;
    if (T < 0 || K < 1 || static_cast<int64_t>(T) * K > INT32_MAX) return LORA_ERR_INVALID_ARG;
    const int32_t P = T * K;
    if ((st = check_shape(shape, &sh)) != LORA_OK) return st;
    if ((st = check_rows(x, ldx, x_per_token ? T : P, sh.k)) != LORA_OK) return st;
    if ((st = check_rows(y, ldy, P, sh.off[sh.n])) != LORA_OK) return st;
    if ((st = check_ws(ws, ws_bytes, P, sh)) != LORA_OK) return st;
    if (path != LORA_PATH_DECODE_DIRECT && path != LORA_PATH_DECODE_TMA) return LORA_ERR_UNSUPPORTED;
    if (P == 0) return LORA_OK;
    if (path == LORA_PATH_DECODE_TMA) {
        if (!lora::decode_tma_supported(P, sh)) return LORA_ERR_UNSUPPORTED;
        if (plan == nullptr || plan_bytes < lora::tma_plan_bytes(P, sh)) return LORA_ERR_WORKSPACE;
        if (!aligned16(plan)) return LORA_ERR_ALIGNMENT;
        return tma_call(x, ldx, y, ldy, P, sh, static_cast<const unsigned char *>(plan), ws, err,
                        reinterpret_cast<cudaStream_t>(stream), x_per_token ? K : 1);
    }
    if (!lora::decode_direct_supported(P, sh, false)) return LORA_ERR_UNSUPPORTED;
    if (plan == nullptr || plan_bytes < lora::direct_plan_bytes(P, sh)) return LORA_ERR_WORKSPACE;
    if (!aligned16(plan)) return LORA_ERR_ALIGNMENT;
    return from_cuda(lora::launch_decode_direct(static_cast<const uint16_t *>(x), ldx, static_cast<uint16_t *>(y), ldy,
                                                sh, nullptr, nullptr, nullptr, nullptr, ws, P, err, false,
                                                reinterpret_cast<cudaStream_t>(stream), x_per_token ? K : 1,
                                                static_cast<const unsigned char *>(plan)));
}

lora_status_t lora_apply_moe_plan(const void *x, int64_t ldx, int32_t x_per_token, void *y, int64_t ldy, int32_t T,
                                  int32_t K, const lora_shape_t *shape, const void *plan, size_t plan_bytes, float *ws,
                                  size_t ws_bytes, int32_t *err, lora_stream_t stream) {
    return lora_apply_moe_plan_ex(x, ldx, x_per_token, y, ldy, T, K, shape, plan, plan_bytes, LORA_PATH_DECODE_DIRECT,
                                  ws, ws_bytes, err, stream);
}

lora_status_t lora_apply(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T, const lora_shape_t *shape,
                         const void *dev_table, const int32_t *sorted_ids, const int32_t *seg_offsets,
                         const int32_t *active, int32_t max_seg_hint, float *ws, size_t ws_bytes, int32_t *err,
                         lora_stream_t stream) {
    return lora_apply_ex(x, ldx, y, ldy, T, shape, dev_table, sorted_ids, seg_offsets, active, max_seg_hint,
                         LORA_PATH_AUTO, ws, ws_bytes, err, stream);
}

}  // extern "C"
