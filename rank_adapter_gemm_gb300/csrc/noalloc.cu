// lora_apply for callers that cannot hand the library a workspace.
//
// Some callers have no way to allocate device memory at the point where they
// run the branch: a plug-in inside a host engine that owns every byte of device
// memory through its own pool and exposes no allocator to plug-ins, or code
// that must not call cudaMalloc because it would synchronise the device in a
// latency-critical path.  For them this entry point keeps its scratch (the
// fp32 shrink output xa) in a fixed-size array that is part of the library's
// device image, so it allocates nothing at all.
#include <mutex>

#include "common.cuh"

namespace lora {
cudaError_t launch_shrink(const uint16_t *x, int64_t ldx, const Shape &sh, const void *table,
                          const int32_t *sorted_ids, const int32_t *seg, float *xa, int32_t T, int32_t *err,
                          bool trigger_dependents, cudaStream_t stream);
cudaError_t launch_expand(const float *xa, uint16_t *y, int64_t ldy, const Shape &sh, const void *table,
                          const int32_t *sorted_ids, const int32_t *seg, int32_t T, int32_t *err,
                          bool programmatic, cudaStream_t stream);
}  // namespace lora

// The scratch array: LORA_NOALLOC_WS_BYTES on every device that loads the
// library, until the process exits.
static __device__ __align__(256) float g_noalloc_xa[LORA_NOALLOC_WS_BYTES / sizeof(float)];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
float *g_xa_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device with that device current.  In host code the array's name is only a
// host-side stand-in; a kernel must be given this address instead.
cudaError_t scratch_address(float **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_xa_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_xa);
        if (e != cudaSuccess) return e;
        g_xa_addr[dev] = static_cast<float *>(p);
    }
    *out = g_xa_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" lora_status_t lora_apply_noalloc(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T,
                                            const lora_shape_t *shape, const void *dev_table,
                                            const int32_t *sorted_ids, const int32_t *seg_offsets,
                                            const int32_t *active, int32_t *err, lora_stream_t stream) {
    // argument checks: the same rules as lora_apply
    if (shape == nullptr || T < 0) return LORA_ERR_INVALID_ARG;
    const lora_shape_t &s = *shape;
    if (s.S < 1 || s.S > LORA_MAX_SLOTS || s.n_slices < 1 || s.n_slices > LORA_MAX_SLICES || s.k < 8)
        return LORA_ERR_INVALID_ARG;
    if (s.k % 8 != 0) return LORA_ERR_ALIGNMENT;
    if (s.r_max < 8 || s.r_max > LORA_MAX_RANK || s.r_max % 8 != 0) return LORA_ERR_RANK;
    if (s.slice_offsets[0] != 0) return LORA_ERR_INVALID_ARG;
    for (int i = 0; i < s.n_slices; ++i) {
        const int32_t w = s.slice_offsets[i + 1] - s.slice_offsets[i];
        if (w <= 0) return LORA_ERR_INVALID_ARG;
        if (w % 8 != 0) return LORA_ERR_ALIGNMENT;
    }
    if (dev_table == nullptr || seg_offsets == nullptr || active == nullptr) return LORA_ERR_INVALID_ARG;
    if (T > 0 && (sorted_ids == nullptr || x == nullptr || y == nullptr)) return LORA_ERR_INVALID_ARG;
    if (ldx < s.k || ldy < s.slice_offsets[s.n_slices]) return LORA_ERR_INVALID_ARG;
    if (!aligned16(dev_table) || !aligned16(x) || !aligned16(y) || ldx % 8 != 0 || ldy % 8 != 0)
        return LORA_ERR_ALIGNMENT;
    // the fixed scratch bounds the problem size
    const size_t need = sizeof(float) * size_t(s.n_slices) * size_t(T) * size_t(s.r_max);
    if (need > LORA_NOALLOC_WS_BYTES) return LORA_ERR_WORKSPACE;
    if (T == 0) return LORA_OK;

    lora::Shape sh;
    sh.S = s.S;
    sh.r_max = s.r_max;
    sh.k = s.k;
    sh.n = s.n_slices;
    for (int i = 0; i <= LORA_MAX_SLICES; ++i)
        sh.off[i] = i <= s.n_slices ? s.slice_offsets[i] : s.slice_offsets[s.n_slices];

    float *xa = nullptr;
    if (scratch_address(&xa) != cudaSuccess) return LORA_ERR_CUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // nothing in the scratch has to start at zero: the shrink writes every
    // entry the expand then reads
    if (lora::launch_shrink(static_cast<const uint16_t *>(x), ldx, sh, dev_table, sorted_ids, seg_offsets, xa, T,
                            err, true, st) != cudaSuccess)
        return LORA_ERR_CUDA;
    if (lora::launch_expand(xa, static_cast<uint16_t *>(y), ldy, sh, dev_table, sorted_ids, seg_offsets, T, err,
                            true, st) != cudaSuccess)
        return LORA_ERR_CUDA;
    return LORA_OK;
}
