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

#include "checks.cuh"
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

}  // namespace

extern "C" lora_status_t lora_apply_noalloc(const void *x, int64_t ldx, void *y, int64_t ldy, int32_t T,
                                            const lora_shape_t *shape, const void *dev_table,
                                            const int32_t *sorted_ids, const int32_t *seg_offsets,
                                            const int32_t *active, int32_t *err, lora_stream_t stream) {
    // argument checks: the same rules (and the same code) as lora_apply
    lora::Shape sh;
    lora_status_t st;
    if (T < 0) return LORA_ERR_INVALID_ARG;
    if ((st = lora::check_shape(shape, &sh)) != LORA_OK) return st;
    if ((st = lora::check_index_ptrs(dev_table, sorted_ids, seg_offsets, active, T)) != LORA_OK) return st;
    if ((st = lora::check_rows(x, ldx, T, sh.k)) != LORA_OK) return st;
    if ((st = lora::check_rows(y, ldy, T, sh.off[sh.n])) != LORA_OK) return st;
    const lora_shape_t &s = *shape;
    // the fixed scratch bounds the problem size
    const size_t need = sizeof(float) * size_t(s.n_slices) * size_t(T) * size_t(s.r_max);
    if (need > LORA_NOALLOC_WS_BYTES) return LORA_ERR_WORKSPACE;
    if (T == 0) return LORA_OK;

    float *xa = nullptr;
    if (scratch_address(&xa) != cudaSuccess) return LORA_ERR_CUDA;
    cudaStream_t strm = reinterpret_cast<cudaStream_t>(stream);
    // nothing in the scratch has to start at zero: the shrink writes every
    // entry the expand then reads
    if (lora::launch_shrink(static_cast<const uint16_t *>(x), ldx, sh, dev_table, sorted_ids, seg_offsets, xa, T,
                            err, true, strm) != cudaSuccess)
        return LORA_ERR_CUDA;
    if (lora::launch_expand(xa, static_cast<uint16_t *>(y), ldy, sh, dev_table, sorted_ids, seg_offsets, T, err,
                            true, strm) != cudaSuccess)
        return LORA_ERR_CUDA;
    return LORA_OK;
}
