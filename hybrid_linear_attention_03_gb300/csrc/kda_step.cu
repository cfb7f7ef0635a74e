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
//   * The state is stored transposed (S^T: row j = value channel, d_k key
//     channels contiguous).  A warp owns 16 rows; lane l holds one float4 of
//     each row (lanes_per_row = D/4 lanes share a row).  Every warp-wide load
//     or store is one contiguous 512-byte segment (128-bit per lane).
//   * u_j = sum_i k_i alpha_i S_ij and o_j = sum_i q_i S'_ij are per-row dot
//     products over d_k: 4 FMAs per lane, then a transpose-reduce across the
//     row's lanes that halves the number of live partial sums at each shuffle
//     stage (16 shuffles for 16 rows instead of 80).
//   * The gated RMSNorm needs sum_j o_j^2 over the head: each warp sums its
//     16 rows in a fixed order and the 8 warp partials are added in warp
//     order.  When a head is split over a thread-block cluster (small batches,
//     so that all 152 SMs get work) the partials of the other CTAs are read
//     through distributed shared memory, in the same order, so the result is
//     bit-identical for every split.
//   * Conv + SiLU + L2 for all T tokens are computed once up front into
//     shared memory while the state loads are in flight.
#include "kda_internal.h"

#include <mutex>

namespace kda {
namespace {

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Read a float at the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ float ld_peer_f32(const float *local, uint32_t rank) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local));
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(a), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

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

template <int D, int CL>
struct StepCfg {
    static constexpr int WPH = D / 16;      // warps per head (16 state rows each)
    static constexpr int WPC = WPH / CL;    // warps per CTA
    static constexpr int NT = 32 * WPC;     // threads per CTA
    static constexpr int LPR = D / 4;       // lanes per state row (one float4 each)
    static constexpr int RPL = 32 / LPR;    // rows per warp-wide float4 access
    static constexpr int NV = 16 / RPL;     // float4 registers per lane
    static constexpr int OWN = LPR / NV;    // lanes that end up holding the same row sum
    static_assert(WPC >= 1 && WPH % CL == 0, "cluster split must divide the head");
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

template <int D, typename Act>
__host__ __device__ constexpr size_t step_smem_bytes(int T, int wpc) {
    return sizeof(float) * (size_t(T) * 3 * D      // conv outputs
                            + 2 * wpc * 16         // u and o row buffers
                            + kMaxVerifyT * wpc)   // per-token sum of squares
           + sizeof(Act) * size_t(T + 3) * 3 * D;  // raw window (tail + tokens)
}

template <int D, typename Act, int CL>
__global__ void __launch_bounds__(StepCfg<D, CL>::NT)
kda_step_kernel(const StepParams p) {
    using C = StepCfg<D, CL>;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int T = p.T;
    float *conv = reinterpret_cast<float *>(smem_raw);  // [T][3][D]
    float *ubuf = conv + size_t(T) * 3 * D;              // [WPC][16]
    float *obuf = ubuf + C::WPC * 16;                    // [WPC][16]
    float *sq = obuf + C::WPC * 16;                      // [kMaxVerifyT][WPC]
    Act *raw = reinterpret_cast<Act *>(sq + kMaxVerifyT * C::WPC);  // [T+3][3][D]

    const int rank = (CL == 1) ? 0 : static_cast<int>(cluster_ctarank());
    const int item = blockIdx.x / CL;  // b * H + h
    const int b = item / p.H, h = item - b * p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gwarp = rank * C::WPC + warp;
    const size_t head_elems = size_t(D) * D;
    const size_t slot_elems = size_t(p.H) * head_elems;

    // Slot checks are uniform over the cluster (all its CTAs serve one head).
    const int in_slot = p.in_slots[b];
    bool bad = in_slot < 0 || in_slot >= p.num_slots;
    for (int t = 0; t < T; ++t) {
        const int s = p.snap_slots[b * T + t];
        bad |= (s < 0 || s >= p.num_slots);
    }
    if (bad) {
        if (threadIdx.x == 0 && rank == 0) atomicOr(p.err, KDA_DEVERR_SLOT_RANGE);
        return;
    }

    // Issue the state loads first; the conv prologue runs while they fly.
    const int sub = lane / C::LPR, c4 = lane % C::LPR;
    const float *Sin = p.states + size_t(in_slot) * slot_elems + size_t(h) * head_elems;
    float4 S[C::NV];
#pragma unroll
    for (int n = 0; n < C::NV; ++n) {
        const int row = gwarp * 16 + n * C::RPL + sub;
        S[n] = load4(Sin + size_t(row) * D + 4 * c4);
    }

    // Per-token gate inputs of the first token, fetched before the prologue.
    const int n_own = c4 / C::OWN;
    const bool owner = (c4 % C::OWN) == 0;
    const int own_row = n_own * C::RPL + sub;  // 0..15 within the warp
    const int own_j = gwarp * 16 + own_row;    // value channel this lane reports
    const Act *alpha = static_cast<const Act *>(p.alpha);
    const Act *beta = static_cast<const Act *>(p.beta);
    const Act *gate = static_cast<const Act *>(p.gate);
    float4 av_next = load4(alpha + (size_t(b) * T * p.H + h) * D + 4 * c4);
    float bt_next = to_f32(beta[size_t(b) * T * p.H + h]);
    float gj_next = to_f32(gate[(size_t(b) * T * p.H + h) * D + own_j]);

    // ---- conv + SiLU for the head's 3*D channels over the T tokens --------
    // All loads of a thread's channels (taps, old tail, first token) are
    // issued before any use, so the prologue costs one memory latency.
    const Act *tail_in = static_cast<const Act *>(p.tails) + size_t(in_slot) * 3 * p.n_ch;
    const Act *cw = static_cast<const Act *>(p.conv_w);
    constexpr int PER = (3 * D + C::NT - 1) / C::NT;
    float4 wv[PER];
    Act xv[PER][4];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int idx = threadIdx.x + u * C::NT;
        if (idx < 3 * D) {
            const int s = idx / D, c = idx - s * D;
            const int ch = s * p.H * D + h * D + c;
            const Act *src = static_cast<const Act *>(s == 0 ? p.q : (s == 1 ? p.k : p.v));
            wv[u] = load4(cw + size_t(ch) * 4);
            xv[u][0] = tail_in[ch];
            xv[u][1] = tail_in[p.n_ch + ch];
            xv[u][2] = tail_in[2 * p.n_ch + ch];
            xv[u][3] = src[size_t(b) * T * p.H * D + size_t(h) * D + c];
        }
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int idx = threadIdx.x + u * C::NT;
        if (idx < 3 * D) {
            const int s = idx / D, c = idx - s * D;
            const Act *src = static_cast<const Act *>(s == 0 ? p.q : (s == 1 ? p.k : p.v));
            Act x0 = xv[u][0], x1 = xv[u][1], x2 = xv[u][2];
            raw[(0 * 3 + s) * D + c] = x0;
            raw[(1 * 3 + s) * D + c] = x1;
            raw[(2 * 3 + s) * D + c] = x2;
            for (int t = 0; t < T; ++t) {
                const Act xt = t == 0 ? xv[u][3] : src[(size_t(b) * T + t) * p.H * D + size_t(h) * D + c];
                raw[((t + 3) * 3 + s) * D + c] = xt;
                float acc = wv[u].x * to_f32(x0);
                acc = fmaf(wv[u].y, to_f32(x1), acc);
                acc = fmaf(wv[u].z, to_f32(x2), acc);
                acc = fmaf(wv[u].w, to_f32(xt), acc);
                conv[(t * 3 + s) * D + c] = acc * sigmoid_f(acc);
                x0 = x1;
                x1 = x2;
                x2 = xt;
            }
        }
    }
    __syncthreads();
    // ---- L2 norm of q and k per token ---------------------------------------
    for (int pr = warp; pr < 2 * T; pr += C::WPC) {
        float *x = conv + ((pr >> 1) * 3 + (pr & 1)) * D;
        float ss = 0.f;
        for (int c = lane; c < D; c += 32) ss = fmaf(x[c], x[c], ss);
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = rsqrtf(ss + p.eps_l2);
        for (int c = lane; c < D; c += 32) x[c] *= r;
    }
    // All CTAs of the cluster have read the old tail before anyone writes one.
    if constexpr (CL == 1) __syncthreads(); else cluster_sync_all();

    Act *out = static_cast<Act *>(p.out);
    Act *tails = static_cast<Act *>(p.tails);
    const float wn = to_f32(static_cast<const Act *>(p.norm_w)[own_j]);
    constexpr int TC = D / CL;  // tail channels per stream written by this CTA

    for (int t = 0; t < T; ++t) {
        const size_t tok = size_t(b) * T + t;
        const float4 qv = load4(conv + (t * 3 + 0) * D + 4 * c4);
        const float4 kv = load4(conv + (t * 3 + 1) * D + 4 * c4);
        const float4 av = av_next;
        const float bt = bt_next, gj = gj_next;
        if (t + 1 < T) {
            av_next = load4(alpha + ((tok + 1) * p.H + h) * D + 4 * c4);
            bt_next = to_f32(beta[(tok + 1) * p.H + h]);
            gj_next = to_f32(gate[((tok + 1) * p.H + h) * D + own_j]);
        }
        const float4 ka = make_float4(kv.x * av.x, kv.y * av.y, kv.z * av.z, kv.w * av.w);
        const float4 bk = make_float4(bt * kv.x, bt * kv.y, bt * kv.z, bt * kv.w);

        // u_j = sum_i k_i alpha_i S_ij  (prediction of v_j by the decayed state)
        float red[C::NV];
#pragma unroll
        for (int n = 0; n < C::NV; ++n) red[n] = dot4(ka, S[n]);
        RowReduce<C::NV, C::LPR / 2>::run(red, lane);
        if (owner) ubuf[warp * 16 + own_row] = red[0];
        __syncwarp();
        // S'_ij = alpha_i S_ij + beta k_i (v_j - u_j)
        const float *vrow = conv + (t * 3 + 2) * D + gwarp * 16;
#pragma unroll
        for (int n = 0; n < C::NV; ++n) {
            const int r = n * C::RPL + sub;
            const float d = vrow[r] - ubuf[warp * 16 + r];
            S[n].x = fmaf(av.x, S[n].x, bk.x * d);
            S[n].y = fmaf(av.y, S[n].y, bk.y * d);
            S[n].z = fmaf(av.z, S[n].z, bk.z * d);
            S[n].w = fmaf(av.w, S[n].w, bk.w * d);
        }
        // o_j = sum_i q_i S'_ij
#pragma unroll
        for (int n = 0; n < C::NV; ++n) red[n] = dot4(qv, S[n]);
        RowReduce<C::NV, C::LPR / 2>::run(red, lane);
        if (owner) obuf[warp * 16 + own_row] = red[0];
        __syncwarp();
        if (lane == 0) {
            float a = 0.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) a = fmaf(obuf[warp * 16 + r], obuf[warp * 16 + r], a);
            sq[t * C::WPC + warp] = a;
        }

        // Snapshot: this warp's state rows and this CTA's share of the tail.
        const int snap = p.snap_slots[b * T + t];
        float *Sout = p.states + size_t(snap) * slot_elems + size_t(h) * head_elems;
#pragma unroll
        for (int n = 0; n < C::NV; ++n) {
            float4 *dst = reinterpret_cast<float4 *>(Sout + size_t(gwarp * 16 + n * C::RPL + sub) * D + 4 * c4);
            if (T > 1) __stcs(dst, S[n]); else *dst = S[n];
        }
        Act *tail_out = tails + size_t(snap) * 3 * p.n_ch;
        for (int idx = threadIdx.x; idx < 9 * TC; idx += C::NT) {
            const int j = idx / (3 * TC), rem = idx - j * 3 * TC;
            const int s = rem / TC, c = rank * TC + (rem - s * TC);
            tail_out[j * p.n_ch + s * p.H * D + h * D + c] = raw[((t + 1 + j) * 3 + s) * D + c];
        }

        // Gated RMSNorm over the head's D value channels.
        if constexpr (CL == 1) __syncthreads(); else cluster_sync_all();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < C::WPH; ++w) {
            const int cta = w / C::WPC, lw = w - cta * C::WPC;
            float part;
            if constexpr (CL == 1) part = sq[t * C::WPC + lw];
            else part = (cta == rank) ? sq[t * C::WPC + lw] : ld_peer_f32(&sq[t * C::WPC + lw], cta);
            tot += part;
        }
        const float r = rsqrtf(tot * (1.0f / D) + p.eps_rms);
        if (owner) {
            const float o = obuf[warp * 16 + own_row];
            out[(tok * p.H + h) * D + own_j] = from_f32<Act>(wn * (o * r) * sigmoid_f(gj));
        }
    }
    // Peers may still read this CTA's partial sums.
    if constexpr (CL > 1) cluster_sync_all();
}

template <int D, typename Act, int CL>
kda_status launch_cfg(const StepParams &p, cudaStream_t stream) {
    using C = StepCfg<D, CL>;
    auto kern = kda_step_kernel<D, Act, CL>;
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KDA_ERR_CUDA;
    cudaError_t attr_err = cudaSuccess;
    std::call_once(once[dev], [&] {
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        int(step_smem_bytes<D, Act>(kMaxVerifyT, C::WPC)));
    });
    if (attr_err != cudaSuccess) return KDA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.B) * unsigned(p.H) * CL, 1, 1);
    cfg.blockDim = dim3(C::NT, 1, 1);
    cfg.dynamicSmemBytes = step_smem_bytes<D, Act>(p.T, C::WPC);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (CL > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (cached[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 152;
    }
    return cached[dev];
}

// Split each head over a cluster only for multi-token launches with too few
// heads to give every SM two CTAs.  A single-token launch is latency-bound:
// measured at batch 1 (64 heads), one CTA per head takes 5.3 us per step and
// splits of 2/4/8 CTAs take 6.6/7.7/9.5 us, the cluster barriers costing more
// than the shorter per-CTA state stream saves.
int pick_cluster(int items, int wph, int T) {
    if (T == 1) return 1;
    const int target = 2 * sm_count();
    int cl = 1;
    while (cl < wph && cl < 8 && items * cl < target) cl *= 2;
    return cl;
}

template <int D, typename Act>
kda_status launch_d(const StepParams &p, cudaStream_t stream) {
    constexpr int WPH = D / 16;
    const int cl = pick_cluster(p.B * p.H, WPH, p.T);
    switch (cl) {
        case 1: return launch_cfg<D, Act, 1>(p, stream);
        case 2: if constexpr (WPH >= 2) return launch_cfg<D, Act, 2>(p, stream); break;
        case 4: if constexpr (WPH >= 4) return launch_cfg<D, Act, 4>(p, stream); break;
        case 8: if constexpr (WPH >= 8) return launch_cfg<D, Act, 8>(p, stream); break;
    }
    return KDA_ERR_UNSUPPORTED;
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
