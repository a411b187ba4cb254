// Tensor-core (tcgen05 / TMEM) prefill path.
#include "common.cuh"

namespace lora {

bool prefill_available() { return false; }

cudaError_t launch_prefill(const uint16_t *, int64_t, uint16_t *, int64_t, const Shape &, const void *,
                           const int32_t *, const int32_t *, float *, int32_t, int32_t *, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace lora
