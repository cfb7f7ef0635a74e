// kda_prefetch.cu -- L2 prefetch of the slots a coming decode or verify step
// reads (kda_state_prefetch in include/kda.h).
//
// "vLLM Kimi K3 지원", section "Fused Kernels 및 메타데이터 최적화", KDA Decode
// bullet: the decode step is bound by its repeated state traffic.  At small
// batch a step's state (4 MiB per slot at H = 64, d = 128) fits in L2, but
// when other layers run between two tokens it has left L2, and the step's
// chain of dependent round trips to HBM (slot index, then state and conv
// tail, then the write-back) sets its time.  This kernel asks L2 to fetch
// the states and tails ahead, e.g. one layer early, and with them the
// layer's conv taps and norm weight, which another layer's work has also
// pushed out: each thread hands one head's state rows, one tail row or one
// piece of the weights to the TMA engine as a bulk L2 prefetch, which
// completes on its own and changes no data.
#include "kda_internal.h"
#include "kda_sm100.cuh"

namespace kda {
namespace {

// One CTA per slot of the table: threads 0 .. H-1 prefetch one head's state
// each (d_v rows of d_k fp32, contiguous), threads H .. H+2 one row of the
// conv tail each.  Slots outside the pool are skipped (a hint has no error).
// CTA 0 also prefetches the layer weights when given: the conv taps in
// pieces of w_piece bytes (threads 128 .. 255), the norm weight (thread 127).
__global__ void __launch_bounds__(256) state_prefetch_kernel(const float *states, size_t head_bytes, int H,
                                                             const unsigned char *tails, size_t tail_row_bytes,
                                                             const int32_t *slots, int num_slots,
                                                             const unsigned char *conv_w, size_t conv_bytes,
                                                             size_t w_piece, const unsigned char *norm_w,
                                                             size_t norm_bytes) {
    if (blockIdx.x == 0 && conv_w) {
        if (threadIdx.x >= 128) {
            const size_t off = size_t(threadIdx.x - 128) * w_piece;
            if (off < conv_bytes) {
                const size_t n = conv_bytes - off < w_piece ? conv_bytes - off : w_piece;
                sm100::bulk_prefetch_l2(conv_w + off, uint32_t(n));
            }
        } else if (threadIdx.x == 127 && norm_bytes >= 16) {
            // the norm weight need not be 16-byte aligned: cover its aligned interior
            const uintptr_t a = (reinterpret_cast<uintptr_t>(norm_w) + 15) & ~uintptr_t(15);
            const uintptr_t e = (reinterpret_cast<uintptr_t>(norm_w) + norm_bytes) & ~uintptr_t(15);
            if (e > a) sm100::bulk_prefetch_l2(reinterpret_cast<const void *>(a), uint32_t(e - a));
        }
    }
    const int slot = slots[blockIdx.x];
    if (slot < 0 || slot >= num_slots) return;
    const unsigned char *st = reinterpret_cast<const unsigned char *>(states) + size_t(slot) * size_t(H) * head_bytes;
    for (int h = threadIdx.x; h < H; h += blockDim.x) sm100::bulk_prefetch_l2(st + size_t(h) * head_bytes, uint32_t(head_bytes));
    if (threadIdx.x >= blockDim.x - 3) {
        const int row = int(threadIdx.x) - int(blockDim.x - 3);
        sm100::bulk_prefetch_l2(tails + (size_t(slot) * 3 + size_t(row)) * tail_row_bytes, uint32_t(tail_row_bytes));
    }
}

}  // namespace

kda_status launch_state_prefetch(const kda_pool *pool, const kda_weights *w, const int32_t *slots, int B,
                                 cudaStream_t stream) {
    const size_t head_bytes = size_t(pool->desc.d_k) * size_t(pool->desc.d_v) * sizeof(float);
    const size_t tail_row_bytes = size_t(pool->n_ch) * size_t(pool->act_bytes);
    // conv taps: n_ch x 4 values, a multiple of 16 bytes (n_ch is even); 128 pieces at most
    const size_t conv_bytes = w ? size_t(pool->n_ch) * 4 * size_t(pool->act_bytes) : 0;
    const size_t w_piece = ((conv_bytes + 127) / 128 + 15) / 16 * 16;
    const size_t norm_bytes = w ? size_t(pool->desc.d_v) * size_t(pool->act_bytes) : 0;
    const ProfScope prof(KDA_KERNEL_STATE_PREFETCH, stream);
    state_prefetch_kernel<<<unsigned(B), 256, 0, stream>>>(
        pool->states, head_bytes, pool->desc.num_heads, static_cast<const unsigned char *>(pool->tails),
        tail_row_bytes, slots, pool->desc.num_slots, w ? static_cast<const unsigned char *>(w->conv_w) : nullptr,
        conv_bytes, w_piece, w ? static_cast<const unsigned char *>(w->norm_w) : nullptr, norm_bytes);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda
