// kda_step.cu -- the fused KDA decode / speculative-verify kernel (sm_103a).
//
// One launch advances B sequences by T tokens (decode: T = 1, written in
// place; verify: T draft tokens with a state snapshot after each).  Per
// (sequence, head) the whole step is fused, as in "vLLM Kimi K3 지원", section
// "Fused Kernels 및 메타데이터 최적화", KDA Decode bullet: causal conv + SiLU,
// L2 norm of q and k, the delta-rule update with per-channel decay, the
// readout and the sigmoid-gated RMSNorm.
//
// The op is bound by HBM: every token reads and writes the D x D fp32 head
// state (64 KiB at D = 128) and does ~6 flops per state element.  So the
// design keeps the state in registers for all T tokens and touches HBM once
// per state element per read or snapshot:
//   * One CTA per (sequence, head); D/16 warps, 16 state rows per warp.  The
//     state is stored transposed (S^T: row j = value channel, d_k key channels
//     contiguous); lane l holds one float4 of each of its warp's rows
//     (D/4 lanes share a row), so every warp-wide load or store is one
//     contiguous 512-byte segment (128-bit per lane).
//   * u_j = sum_i k_i alpha_i S_ij and o_j = sum_i q_i S'_ij are per-row dot
//     products over d_k: 4 FMAs per lane, then a transpose-reduce across the
//     row's lanes that halves the number of live partial sums at each shuffle
//     stage (16 shuffles for 16 rows instead of 80).
//   * The per-token inputs of all T tokens (q, k, v, alpha, gate, beta, the
//     snapshot slots) are copied into shared memory asynchronously as the
//     very first thing, the old conv tail right after the state loads are
//     issued; conv + SiLU + L2 for all T tokens then run from shared memory
//     while the state loads are in flight.  The prologue costs one memory
//     latency whatever T is.
//   * Inside the token loop warps synchronise only with themselves, so each
//     warp streams its snapshot rows as soon as they are ready.  The gated
//     RMSNorm needs sum_j o_j^2 over the whole head: every warp keeps its
//     per-token partial, and all T outputs are normalised after one CTA
//     barrier at the end.
// Splitting a head over a thread-block cluster (DSMEM reduction of the norm)
// was measured slower at every batch size tried (batch 1..16, T = 1 and 8):
// the cluster barriers cost more than the shorter per-CTA state stream saved.
#include "kda_internal.h"
#include "kda_sm100.cuh"

#include <mutex>

namespace kda {
namespace {

// sigma(x) = 1 / (1 + e^-x) with e^-x = 2^(-x log2 e), from PTX's approximate
// 2^x and 1/x (flush-to-zero; relative errors of a few 1e-7 and about 1 ulp).
// 0 for x below about -88, where 2^(-x log2 e) is +inf.
__device__ __forceinline__ float sigmoid_f(float x) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-x * 1.4426950408889634f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return r;
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
    return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}

__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
    const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}

template <int D>
struct StepCfg {
    static constexpr int WPC = D / 16;      // warps per CTA (16 state rows each)
    static constexpr int NT = 32 * WPC;     // threads per CTA
    static constexpr int LPR = D / 4;       // lanes per state row (one float4 each)
    static constexpr int RPL = 32 / LPR;    // rows per warp-wide float4 access
    static constexpr int NV = 16 / RPL;     // float4 registers per lane
    static constexpr int OWN = LPR / NV;    // lanes that end up holding the same row sum
    static_assert(NV <= LPR, "transpose reduce needs NV <= lanes per row");
};

// Transpose-reduce: NV partial sums per lane, summed over the LPR lanes of a
// row group.  At the stage with xor-offset O the upper lane of each pair
// keeps the upper half of its values, so the number of live values halves;
// once one value is left the remaining stages are plain butterflies.  After
// the call v[0] of lane l is the full sum for register index
// (l % LPR) / OWN.
template <int CNT, int O>
struct RowReduce {
    static __device__ __forceinline__ void run(float *v, int lane) {
        if constexpr (O == 0) {
            return;
        } else if constexpr (CNT > 1) {
            constexpr int HALF = CNT / 2;
            const bool upper = (lane & O) != 0;
#pragma unroll
            for (int m = 0; m < HALF; ++m) {
                const float send = upper ? v[m] : v[m + HALF];
                const float keep = upper ? v[m + HALF] : v[m];
                v[m] = keep + __shfl_xor_sync(0xffffffffu, send, O);
            }
            RowReduce<HALF, O / 2>::run(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
            RowReduce<1, O / 2>::run(v, lane);
        }
    }
};

// Snapshot staging (multi-token launches only): 16 rows x D floats per warp,
// placed first in dynamic shared memory so every warp's block starts on a
// 16-byte boundary (bulk copies need it); D*D*4 bytes is a multiple of 16.
template <int D>
__host__ __device__ constexpr size_t stage_floats(int T) { return T > 1 ? size_t(D) * D : 0; }

__host__ __device__ constexpr size_t pad4(size_t n) { return (n + 3) / 4 * 4; }

// Dynamic shared memory, in order (every part starts on a 16-byte boundary):
// staging, conv outputs [T][3][D], u rows [WPC][16], o [T][D], per-warp sums
// of squares [T][WPC], beta [T], snapshot slots [T], then in the activation
// type the raw conv window [T+3][3][D] (old tail + tokens), alpha [T][D],
// the gate logits [T][D] and the head's conv taps [3][D][4].
template <int D, typename Act>
__host__ __device__ constexpr size_t step_smem_bytes(int T) {
    constexpr int WPC = D / 16;
    return sizeof(float) * (stage_floats<D>(T) + size_t(T) * 3 * D + WPC * 16 + size_t(T) * D +
                            pad4(size_t(T) * WPC) + 2 * pad4(size_t(T))) +
           sizeof(Act) * (size_t(T + 3) * 3 * D + 2 * size_t(T) * D + 3 * D * 4);
}

template <int D, typename Act>
__global__ void __launch_bounds__(StepCfg<D>::NT)
kda_step_kernel(const StepParams p) {
    using C = StepCfg<D>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int T = p.T;
    float *stage_all = reinterpret_cast<float *>(smem_raw);  // [D][D] if T > 1 (16 rows per warp)
    float *conv = stage_all + stage_floats<D>(T);            // [T][3][D]
    float *ubuf = conv + size_t(T) * 3 * D;                  // [WPC][16]
    float *obuf = ubuf + C::WPC * 16;                        // [T][D]
    float *sq = obuf + size_t(T) * D;                        // [T][WPC]
    float *bsm = sq + pad4(size_t(T) * C::WPC);              // [T] beta
    int *snap_sm = reinterpret_cast<int *>(bsm + pad4(T));   // [T] snapshot slots
    Act *raw = reinterpret_cast<Act *>(snap_sm + pad4(T));   // [T+3][3][D]
    Act *araw = raw + size_t(T + 3) * 3 * D;                 // [T][D] alpha
    Act *graw = araw + size_t(T) * D;                        // [T][D] gate logits
    Act *wtap = graw + size_t(T) * D;                        // [3][D][4] conv taps

    const int b = blockIdx.x / p.H, h = blockIdx.x - b * p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t head_elems = size_t(D) * D;
    const size_t slot_elems = size_t(p.H) * head_elems;
    const Act *beta = static_cast<const Act *>(p.beta);

    // Programmatic dependent launch: this grid may start before the
    // preceding kernel on the stream has completed, and only
    // griddepcontrol.wait makes that kernel's writes visible.  By default
    // every input is read after the wait, so any kernel may produce them
    // right before this launch (the q/k/v projection of a serving step).
    // With KDA_POOL_OVERLAP_INPUTS the caller guarantees the preceding kernel
    // writes none of the inputs (a chain of steps over staged inputs), and
    // the slot tables, beta, weights and token rows are fetched ahead of the
    // wait, so their latency overlaps it; only the pool (state and conv
    // tail, which the preceding step writes) is read after it.
    if (!p.early_inputs) asm volatile("griddepcontrol.wait;" ::: "memory");
    // The slot indices and beta go into registers first; nothing consumes
    // them before the copies below are issued, so their latency overlaps the
    // copies (consuming them here cost two dependent memory round trips
    // ahead of the wait: 2.4K of 8.7K cycles per batch-1 step).
    const int sub = lane / C::LPR, c4 = lane % C::LPR;
    const int n_own = c4 / C::OWN;
    const bool owner = (c4 % C::OWN) == 0;
    const int own_row = n_own * C::RPL + sub;  // 0..15 within the warp
    const int own_j = warp * 16 + own_row;     // value channel this lane reports
    const int in_slot = p.in_slots[b];
    int snap_r = 0;
    const Act wn_r = static_cast<const Act *>(p.norm_w)[own_j];  // a weight: safe before the wait
    Act beta_r = from_f32<Act>(0.f);
    if (threadIdx.x < T) {
        snap_r = p.snap_slots[b * T + threadIdx.x];
        beta_r = beta[(size_t(b) * T + threadIdx.x) * p.H + h];
    }

    // Per-token inputs of all T tokens: 16-byte asynchronous copies into
    // shared memory, issued first so the whole prologue costs one memory
    // latency.  Every (token, head)
    // row of D activations starts on a 16-byte boundary (16-byte aligned
    // bases, D * sizeof(Act) a multiple of 16).
    constexpr int CPR = int(D * sizeof(Act) / 16);  // 16-byte chunks per row
    constexpr int EPC = int(16 / sizeof(Act));      // elements per chunk
    for (int i = threadIdx.x; i < T * 5 * CPR; i += C::NT) {
        const int row = i / CPR, cc = i - row * CPR;
        const int t = row / 5, r = row - t * 5;
        const size_t src_off = ((size_t(b) * T + t) * p.H + h) * D + size_t(cc) * EPC;
        const Act *src = static_cast<const Act *>(r == 0 ? p.q : r == 1 ? p.k : r == 2 ? p.v : r == 3 ? p.alpha : p.gate);
        Act *dst = r < 3 ? raw + size_t((t + 3) * 3 + r) * D : (r == 3 ? araw : graw) + size_t(t) * D;
        sm100::cp_async16(dst + cc * EPC, src + src_off);
    }
    // the head's conv taps: per stream, D channels x 4 taps contiguous
    for (int i = threadIdx.x; i < 3 * 4 * CPR; i += C::NT) {
        const int st = i / (4 * CPR), cc = i - st * 4 * CPR;
        sm100::cp_async16(wtap + size_t(st) * D * 4 + cc * EPC,
                          static_cast<const Act *>(p.conv_w) + (size_t(st) * p.H + h) * D * 4 + cc * EPC);
    }
    sm100::cp_async_commit();


    // The pool's state and tail may have been written by the preceding step
    // launch: wait for it to complete before reading them.
    if (p.early_inputs) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x < T) {
        bsm[threadIdx.x] = to_f32(beta_r);
        snap_sm[threadIdx.x] = snap_r;
    }
    // A bad input slot (uniform over the CTA) stops before any state access;
    // bad snapshot slots are found at the barrier below, before any write.
    if (in_slot < 0 || in_slot >= p.num_slots) {
        if (threadIdx.x == 0) atomicOr(p.err, KDA_DEVERR_SLOT_RANGE);
        sm100::cp_async_wait_all();  // no copy may land after the CTA is gone
        return;
    }
    const float *Sin = p.states + size_t(in_slot) * slot_elems + size_t(h) * head_elems;
    float4 S[C::NV];
#pragma unroll
    for (int n = 0; n < C::NV; ++n) {
        const int row = warp * 16 + n * C::RPL + sub;
        S[n] = load4(Sin + size_t(row) * D + 4 * c4);
    }
    // old tail rows (3 taps x 3 streams, D channels of this head each)
    const Act *tail_in = static_cast<const Act *>(p.tails) + size_t(in_slot) * 3 * p.n_ch;
    for (int i = threadIdx.x; i < 9 * CPR; i += C::NT) {
        const int row = i / CPR, cc = i - row * CPR;
        const int j = row / 3, st = row - j * 3;
        sm100::cp_async16(raw + size_t(j * 3 + st) * D + cc * EPC,
                          tail_in + size_t(j) * p.n_ch + size_t(st) * p.H * D + size_t(h) * D + cc * EPC);
    }
    sm100::cp_async_commit();
    sm100::cp_async_wait_all();
    if (__syncthreads_or(threadIdx.x < T && (snap_r < 0 || snap_r >= p.num_slots))) {
        if (threadIdx.x == 0) atomicOr(p.err, KDA_DEVERR_SLOT_RANGE);
        return;
    }

    // ---- conv + SiLU (+ L2 for q and k): a warp per (token, stream) row --------
    for (int row = warp; row < 3 * T; row += C::WPC) {
        const int t = row / 3, s = row - t * 3;
        float y[(D + 31) / 32];
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < (D + 31) / 32; ++m) {
            const int c = lane + 32 * m;
            y[m] = 0.f;
            if (c < D) {
                const float4 w = load4(wtap + (size_t(s) * D + c) * 4);
                float acc = w.x * to_f32(raw[((t + 0) * 3 + s) * D + c]);
                acc = fmaf(w.y, to_f32(raw[((t + 1) * 3 + s) * D + c]), acc);
                acc = fmaf(w.z, to_f32(raw[((t + 2) * 3 + s) * D + c]), acc);
                acc = fmaf(w.w, to_f32(raw[((t + 3) * 3 + s) * D + c]), acc);
                y[m] = acc * sigmoid_f(acc);
                ss = fmaf(y[m], y[m], ss);
            }
        }
        float r = 1.f;
        if (s < 2) {  // q and k: L2 norm over the head's D channels
#pragma unroll
            for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            r = rsqrtf(ss + p.eps_l2);
        }
#pragma unroll
        for (int m = 0; m < (D + 31) / 32; ++m) {
            const int c = lane + 32 * m;
            if (c < D) conv[(t * 3 + s) * D + c] = y[m] * r;
        }
    }
    // New conv tails: the raw rows t+1 .. t+3 of the window, already in
    // shared memory (the old tail was read into it above, so the global
    // tail may be overwritten).  When the conv leaves warps idle (3T < warps)
    // they store every token's tail now, off the critical path; otherwise
    // each warp stores its channels' tails in the token loop.
    const bool early_tails = 3 * T < C::WPC;
    Act *tails = static_cast<Act *>(p.tails);
    if (early_tails && warp >= 3 * T) {
        for (int i = threadIdx.x - 3 * T * 32; i < T * 9 * CPR; i += (C::WPC - 3 * T) * 32) {
            const int row = i / CPR, cc = i - row * CPR;  // row = t * 9 + tap * 3 + stream
            const int t = row / 9, js = row - t * 9, j = js / 3, st = js - j * 3;
            Act *dst = tails + size_t(snap_sm[t]) * 3 * p.n_ch + size_t(j) * p.n_ch + size_t(st) * p.H * D +
                       size_t(h) * D + cc * EPC;
            *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(raw + size_t((t + 1 + j) * 3 + st) * D + cc * EPC);
        }
    }
    __syncthreads();

    // Programmatic dependent launch: the next step-kernel launch on this
    // stream may start now and run its own prologue up to its
    // griddepcontrol.wait, which waits for this whole grid to complete (so
    // the trigger's position only moves the overlap).  Measured at batch 1
    // (graph of 1000 steps, same GPU): 3.86 us per step with the trigger
    // here, 4.09 us after the token loop, 3.88 us right after the wait;
    // batch 64: 87.8, 88.0 and 88.1 us.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    Act *out = static_cast<Act *>(p.out);

    for (int t = 0; t < T; ++t) {
        const float4 qv = load4(conv + (t * 3 + 0) * D + 4 * c4);
        const float4 kv = load4(conv + (t * 3 + 1) * D + 4 * c4);
        const float4 av = load4(araw + size_t(t) * D + 4 * c4);
        const float bt = bsm[t];
        const float4 ka = make_float4(kv.x * av.x, kv.y * av.y, kv.z * av.z, kv.w * av.w);
        const float4 bk = make_float4(bt * kv.x, bt * kv.y, bt * kv.z, bt * kv.w);

        const float *vrow = conv + (t * 3 + 2) * D + warp * 16;
        float vv[C::NV];
#pragma unroll
        for (int n = 0; n < C::NV; ++n) vv[n] = vrow[n * C::RPL + sub];

        // u_j = sum_i k_i alpha_i S_ij  (prediction of v_j by the decayed state)
        float red[C::NV];
#pragma unroll
        for (int n = 0; n < C::NV; ++n) red[n] = dot4(ka, S[n]);
        RowReduce<C::NV, C::LPR / 2>::run(red, lane);
        if (owner) ubuf[warp * 16 + own_row] = red[0];
        __syncwarp();
        // S'_ij = alpha_i S_ij + beta k_i (v_j - u_j)
#pragma unroll
        for (int n = 0; n < C::NV; ++n) {
            const float d = vv[n] - ubuf[warp * 16 + n * C::RPL + sub];
            S[n].x = fmaf(av.x, S[n].x, bk.x * d);
            S[n].y = fmaf(av.y, S[n].y, bk.y * d);
            S[n].z = fmaf(av.z, S[n].z, bk.z * d);
            S[n].w = fmaf(av.w, S[n].w, bk.w * d);
        }

        // Snapshot, issued before the readout so the stores drain while it
        // runs.  A single-token launch stores its rows directly (in
        // place).  With several drafts the snapshot stream dominates: this
        // warp's 16 state rows are one contiguous 16*D*4-byte block in HBM,
        // staged in shared memory and handed to the TMA engine as one bulk
        // store, which keeps the warp's load/store pipe free (batch 64 x 8
        // drafts: 613 -> 527 us per launch on GB300; a single token got
        // slower, so it keeps direct stores).  The staging buffer is reused
        // once the previous bulk store has finished reading it.
        const int snap = snap_sm[t];
        float *Sout = p.states + size_t(snap) * slot_elems + size_t(h) * head_elems;
        if (T == 1) {
#pragma unroll
            for (int n = 0; n < C::NV; ++n)
                *reinterpret_cast<float4 *>(Sout + size_t(warp * 16 + n * C::RPL + sub) * D + 4 * c4) = S[n];
        } else {
            float *stage = stage_all + size_t(warp) * 16 * D;
            if (t > 0) {
                if (lane == 0) sm100::bulk_wait_read();
                __syncwarp();
            }
#pragma unroll
            for (int n = 0; n < C::NV; ++n)
                *reinterpret_cast<float4 *>(stage + (n * C::RPL + sub) * D + 4 * c4) = S[n];
            sm100::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                sm100::bulk_store(Sout + size_t(warp) * 16 * D, stage, 16 * D * sizeof(float));
                sm100::bulk_commit();
            }
        }

        // o_j = sum_i q_i S'_ij; this warp's sum of o_j^2 for the norm
#pragma unroll
        for (int n = 0; n < C::NV; ++n) red[n] = dot4(qv, S[n]);
        RowReduce<C::NV, C::LPR / 2>::run(red, lane);
        if (owner) obuf[t * D + own_j] = red[0];
        float o2 = owner ? red[0] * red[0] : 0.f;  // each of the warp's 16 rows has exactly one owner lane
#pragma unroll
        for (int o = 16; o; o >>= 1) o2 += __shfl_xor_sync(0xffffffffu, o2, o);
        if (lane == 0) sq[t * C::WPC + warp] = o2;

        if (!early_tails) {
            Act *tail_out = tails + size_t(snap) * 3 * p.n_ch;
            for (int idx = lane; idx < 9 * 16; idx += 32) {  // 3 taps x 3 streams x this warp's 16 channels
                const int j = idx / 48, rem = idx - j * 48;
                const int s = rem >> 4, c = warp * 16 + (rem & 15);
                tail_out[j * p.n_ch + s * p.H * D + h * D + c] = raw[((t + 1 + j) * 3 + s) * D + c];
            }
        }
        __syncwarp();  // ubuf is rewritten by the next token
    }

    // The staging buffers must stay valid until the bulk stores have read
    // them (their writes land before the grid completes).
    if (T > 1 && lane == 0) sm100::bulk_wait_read();
    // Gated RMSNorm of every token over the head's D value channels.
    __syncthreads();
    const float wn = to_f32(wn_r);
    for (int t = 0; t < T; ++t) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < C::WPC; ++w) tot += sq[t * C::WPC + w];
        const float r = rsqrtf(tot * (1.0f / D) + p.eps_rms);
        if (owner) {
            const float o = obuf[t * D + own_j];
            out[((size_t(b) * T + t) * p.H + h) * D + own_j] =
                from_f32<Act>(wn * (o * r) * sigmoid_f(to_f32(graw[t * D + own_j])));
        }
    }
}

template <int D, typename Act>
kda_status launch_d(const StepParams &p, cudaStream_t stream) {
    using C = StepCfg<D>;
    auto kern = kda_step_kernel<D, Act>;
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KDA_ERR_CUDA;
    cudaError_t attr_err = cudaSuccess;
    std::call_once(once[dev], [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        int(step_smem_bytes<D, Act>(kMaxVerifyT)));
    });
    if (attr_err != cudaSuccess) return KDA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.B) * unsigned(p.H), 1, 1);
    cfg.blockDim = dim3(C::NT, 1, 1);
    cfg.dynamicSmemBytes = step_smem_bytes<D, Act>(p.T);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const ProfScope prof(KDA_KERNEL_STEP, stream);
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

template <typename Act>
kda_status launch_act(int D, const StepParams &p, cudaStream_t stream) {
    switch (D) {
        case 16: return launch_d<16, Act>(p, stream);
        case 32: return launch_d<32, Act>(p, stream);
        case 64: return launch_d<64, Act>(p, stream);
        case 128: return launch_d<128, Act>(p, stream);
    }
    return KDA_ERR_UNSUPPORTED;
}

}  // namespace

kda_status launch_step(const kda_pool *pool, const StepParams &p, cudaStream_t stream) {
    const int D = pool->desc.d_k;
    if (pool->desc.act == KDA_BF16) return launch_act<__nv_bfloat16>(D, p, stream);
    return launch_act<float>(D, p, stream);
}

}  // namespace kda
