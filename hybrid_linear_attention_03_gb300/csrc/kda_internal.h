// kda_internal.h -- pool handle and launcher declarations shared by the
// library's translation units (not part of the C ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "kda.h"

struct kda_pool {
    kda_pool_desc desc;
    char *base;               // caller's device buffer
    size_t bytes;
    uint32_t *err;            // device error word (pool header)
    float *states;            // [num_slots][H][d_v][d_k]
    void *tails;              // [num_slots][3][n_ch] act
    size_t slot_state_elems;  // H * d_v * d_k
    size_t slot_tail_elems;   // 3 * n_ch
    int n_ch;
    int act_bytes;
    int device;
    uint32_t flags;           // KDA_POOL_* launch options (kda_state_pool_set_flags)
};

namespace kda {

constexpr int kConvWidth = 4;
constexpr int kMaxVerifyT = 16;

// ---- activation load/store --------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename Act> __device__ __forceinline__ Act from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Parameters of one decode / verify launch.
struct StepParams {
    float *states;
    void *tails;
    uint32_t *err;
    const void *q, *k, *v, *alpha, *beta, *gate;
    void *out;
    const void *conv_w, *norm_w;
    const int32_t *in_slots;    // [B]
    const int32_t *snap_slots;  // [B*T]
    int32_t B, T, H, num_slots, n_ch;
    int32_t early_inputs;  // read inputs before the grid-dependency wait (KDA_POOL_OVERLAP_INPUTS)
    float eps_l2, eps_rms;
};

kda_status launch_step(const kda_pool *pool, const StepParams &p, cudaStream_t stream);

// Brackets one kernel launch (made inside the scope) with CUDA events on its
// stream while a profile runs (kda_profile_start); a no-op otherwise.
class ProfScope {
  public:
    ProfScope(int kind, cudaStream_t s);
    ~ProfScope();
    ProfScope(const ProfScope &) = delete;
    ProfScope &operator=(const ProfScope &) = delete;

  private:
    cudaStream_t s_;
    int slot_ = -1;
};

// L2 prefetch of the slots' state and conv tail (device slot table [B]).
kda_status launch_state_prefetch(const kda_pool *pool, const kda_weights *w, const int32_t *slots, int B,
                                 cudaStream_t stream);

// Slot-to-slot copy of state + tail.
kda_status launch_slot_copy(const kda_pool *pool, const int32_t *src, const int32_t *dst, int n,
                            cudaStream_t stream);

struct PrefillArgs;
size_t prefill_workspace_bytes(const kda_pool *pool, const int32_t *cu_seqlens, int N, int chunk);
kda_status launch_prefill(const kda_pool *pool, const kda_weights *w, const kda_io *io,
                          const int32_t *cu_seqlens, const int32_t *slots,
                          const uint8_t *has_initial_state, int N, int chunk,
                          const kda_ckpt_req *reqs, int n_reqs, void *workspace,
                          size_t workspace_bytes, cudaStream_t stream);
kda_status launch_prefill_noalloc(const kda_pool *pool, const kda_weights *w, const kda_io *io,
                                  const int32_t *cu_seqlens, const int32_t *slots,
                                  const uint8_t *has_initial_state, int N, int chunk, const kda_ckpt_req *reqs,
                                  int n_reqs, cudaStream_t stream);
size_t prefill_workspace_bytes_bound(const kda_pool *pool, int N, int max_tokens, int n_reqs, int chunk);
kda_status launch_prefill_dev(const kda_pool *pool, const kda_weights *w, const kda_io *io, const int32_t *cu_seqlens,
                              const int32_t *slots, const uint8_t *has_initial_state, int N, int max_tokens,
                              int chunk, const kda_ckpt_req *reqs, int n_reqs, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);

}  // namespace kda
