// kda_copy.cu -- bit-exact slot-to-slot copy of KDA state + conv tail.
//
// Interval-based retention ("vLLM Kimi K3 지원", section "에이전틱 캐시 유지
// 정책") keeps copies of a request's recurrent state; restoring one is the
// same copy in the other direction.  A plain HBM copy: one CTA row per slot
// pair, 16-byte vector loads and stores, grid sized to a multiple of the SM
// count.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kPairsPerLaunch = 256;

struct CopyBatch {
    int32_t n;
    int32_t src[kPairsPerLaunch];
    int32_t dst[kPairsPerLaunch];
};

__global__ void __launch_bounds__(256) slot_copy_kernel(float4 *states, size_t state_f4_per_slot,
                                                        int4 *tails, size_t tail_i4_per_slot,
                                                        const CopyBatch batch) {
    const int pair = blockIdx.y;
    if (pair >= batch.n) return;
    const size_t s = size_t(batch.src[pair]), d = size_t(batch.dst[pair]);
    const size_t stride = size_t(gridDim.x) * blockDim.x;
    const size_t i0 = size_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const float4 *ssrc = states + s * state_f4_per_slot;
    float4 *sdst = states + d * state_f4_per_slot;
    for (size_t i = i0; i < state_f4_per_slot; i += stride) sdst[i] = ssrc[i];
    const int4 *tsrc = tails + s * tail_i4_per_slot;
    int4 *tdst = tails + d * tail_i4_per_slot;
    for (size_t i = i0; i < tail_i4_per_slot; i += stride) tdst[i] = tsrc[i];
}

}  // namespace

kda_status launch_slot_copy(const kda_pool *pool, const int32_t *src, const int32_t *dst, int n,
                            cudaStream_t stream) {
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t state_f4 = pool->slot_state_elems / 4;
    const size_t tail_i4 = pool->slot_tail_elems * pool->act_bytes / 16;
    for (int base = 0; base < n; base += kPairsPerLaunch) {
        CopyBatch batch;
        batch.n = (n - base < kPairsPerLaunch) ? (n - base) : kPairsPerLaunch;
        for (int i = 0; i < batch.n; ++i) {
            batch.src[i] = src[base + i];
            batch.dst[i] = dst[base + i];
        }
        // enough CTAs per pair that all SMs stream, at least one per 64 KiB
        unsigned per_pair = unsigned((state_f4 + 4095) / 4096);
        const unsigned want = unsigned((2 * sms + batch.n - 1) / batch.n);
        if (per_pair > want) per_pair = want;
        if (per_pair < 1) per_pair = 1;
        const ProfScope prof(KDA_KERNEL_SLOT_COPY, stream);
        slot_copy_kernel<<<dim3(per_pair, unsigned(batch.n)), 256, 0, stream>>>(
            reinterpret_cast<float4 *>(pool->states), state_f4, reinterpret_cast<int4 *>(pool->tails),
            tail_i4, batch);
        if (cudaGetLastError() != cudaSuccess) return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // namespace kda
