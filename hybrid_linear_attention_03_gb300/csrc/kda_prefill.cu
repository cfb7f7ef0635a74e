// kda_prefill.cu -- chunked prefill (placeholder until the chunked kernels land).
#include "kda_internal.h"

namespace kda {

size_t prefill_workspace_bytes(const kda_pool *, const int32_t *, int, int) { return 0; }

kda_status launch_prefill(const kda_pool *, const kda_weights *, const kda_io *, const int32_t *,
                          const int32_t *, const uint8_t *, int, int, const kda_ckpt_req *, int, void *,
                          size_t, cudaStream_t) {
    return KDA_ERR_UNSUPPORTED;
}

}  // namespace kda
