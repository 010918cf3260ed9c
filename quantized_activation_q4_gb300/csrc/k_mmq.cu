// Prefill dense contraction on a Q8_0 image (minfer doc 52 "r49 A-quantize
// prepass shared-A dedup", sections 1 and 5).

#include "qk_internal.cuh"

namespace qk {

qk_status launch_mmq(const int8_t *, const uint16_t *, int64_t, int, int, const qk_proj *, cudaStream_t) {
    return fail(QK_ERR_UNSUPPORTED, "qk_mmq: not built yet");
}

}  // namespace qk
