// kda_prefill_intra_generic.cu -- the generic intra-chunk prefill kernel:
// every activation type, and the chunks whose decay span is too wide for the
// fast kernel's split exponent (the fast kernel lists those and this kernel,
// launched in list mode, takes them over).
//
// "vLLM Kimi K3 지원", section "Fused Kernels 및 메타데이터 최적화", KDA Prefill
// bullet: prefill runs chunked (FlashKDA).  Per (chunk, head) with cumulative
// log decay G_r = sum_{s<=r} log alpha_s (per key channel):
//   A_rs = beta_r sum_i k_ri k_si exp(G_ri - G_si)  (s < r),  T = (I + A)^-1
//   W = T diag(beta) (exp(G) . K),    Ut = T diag(beta) V
//   P_rs = sum_i q_ri k_si exp(G_ri - G_si)  (s <= r)
// exp(G_r - G_s) is split around a per-channel reference c_i (the middle of
// the chunk's log-decay range) while the span is at most 160; a chunk beyond
// that computes A and P with exact per-element exponentials instead.  The
// record this kernel writes (kda_prefill.cuh) stores K^ as k^ exp(G_last - G)
// with ELC = 1.
#include "kda_prefill.cuh"

#include <mutex>

namespace kda {
namespace pf {
namespace {

namespace is {  // intra shared-memory map (bytes from a 1 KiB-aligned base)
constexpr uint32_t X_HI = 0, X_LO = 32768, KB_HI = 65536, KB_LO = 81920;           // phase 1 images
constexpr uint32_t A_F32 = 0, T_F32 = 81920;                                        // inverse (fp32)
constexpr uint32_t T_HI = 0, T_LO = 8192, AK_HI = 16384, AK_LO = 32768, AV_HI = 49152, AV_LO = 65536;  // phase 3
constexpr uint32_t RQ = 0;        // raw q, k (67 rows each) and, 2-byte, alpha tiles; then the phase-1 images
constexpr uint32_t IN0 = 98304;   // q^, then v, then the W image staging (32 KiB)
constexpr uint32_t SSQ = IN0 - 4096;  // [2 qk][2 halves][4 warps][32] sums of squares, then [16 warps][32] norms (conv phase)
constexpr uint32_t KH = 131072;   // fp32 [64][128] k^
constexpr uint32_t GG = 163840;   // fp32 [64][128] G, then E = exp(G - c)
constexpr uint32_t SMALL = 196608;
constexpr uint32_t RV_LATE = 32768;         // raw v tile of a 4-byte activation (free while T is formed)
constexpr uint32_t RV_EARLY = SMALL + 2560; // raw v tile of a 2-byte activation (loaded with the others)
constexpr uint32_t TDIAG = RV_EARLY + (CH + HALO) * D * 2;  // [4][16 s][16 r] diagonal blocks of T, transposed
constexpr uint32_t XS_C = RV_EARLY;  // [3][16][16] fp32 scratch of the off-diagonal blocks (the raw v tile is consumed)
constexpr int OFFDIAG_THREADS = 192;  // warps 0..5 form T's off-diagonal blocks, the rest the T-free phase-3 images
constexpr int NT = 512;
constexpr int QW = NT / 128;  // warps per TMEM lane quarter (a warp reaches lanes 32 (w % 4) .. + 31)
template <typename Act>
__host__ __device__ constexpr uint32_t tile_bytes() { return uint32_t((CH + HALO) * D * sizeof(Act)); }
// A 2-byte activation's v tile fits beside everything else and arrives with
// q, k and alpha; a 4-byte one is loaded once A and P have freed the images.
template <typename Act>
__host__ __device__ constexpr bool v_early() { return sizeof(Act) == 2; }
template <typename Act>
__host__ __device__ constexpr uint32_t RK() { return RQ + tile_bytes<Act>(); }
template <typename Act>
__host__ __device__ constexpr uint32_t RV() { return v_early<Act>() ? RV_EARLY : RV_LATE; }
// alpha: a 2-byte tile sits beside raw q and k; a 4-byte one lands in the G
// buffer itself (same [64][128] 4-byte layout), where G is formed in place
template <typename Act>
__host__ __device__ constexpr uint32_t RA() { return sizeof(Act) == 2 ? RK<Act>() + tile_bytes<Act>() : GG; }
template <typename Act>
__host__ __device__ constexpr uint32_t BYTES() { return TDIAG + 4 * 16 * 16 * 4; }
template <typename Act>
__host__ __device__ constexpr bool map_ok() {
    return RK<Act>() + tile_bytes<Act>() <= IN0 && (sizeof(Act) != 2 || RA<Act>() + CH * D * sizeof(Act) <= IN0) &&
           (v_early<Act>() || (RV_LATE >= A_F32 + 16384 && RV_LATE + tile_bytes<Act>() <= T_F32)) &&
           XS_C + 3 * 16 * 16 * 4 <= TDIAG &&
           SSQ >= RK<Act>() + tile_bytes<Act>() && (sizeof(Act) != 2 || SSQ >= RA<Act>() + CH * D * sizeof(Act)) &&
           (!v_early<Act>() || RV_EARLY + tile_bytes<Act>() <= TDIAG) && BYTES<Act>() + 1024 <= 232448 &&
           tile_bytes<Act>() % 128 == 0;
}
}  // namespace is

// One level of the blocked inverse of I + A (A stored transposed: A[s * CH +
// r] = A_rs; TD holds T's diagonal blocks transposed): the 4 - d blocks at
// distance d below the diagonal, T_ab = -T_aa sum_{b <= c < a} A_ac T_cb,
// by the first OFFDIAG_THREADS threads (named barrier 1; a level has at most
// 3 x 64 work items).  A thread owns 4 adjacent columns of one row, so each A
// value it loads feeds 4 FMAs and the T / X values arrive as 16-byte vectors;
// the 8 rows a warp covers read A and TD without bank conflicts.  XS holds the
// level's sums, block blk = b at [blk][16][16].
__device__ __forceinline__ void offdiag_sync() {
    asm volatile("bar.sync 1, %0;" :: "n"(is::OFFDIAG_THREADS) : "memory");
}
__device__ __forceinline__ void tri_offdiag(const float *A, float *T, float *XS, const float *TD, int tid, int d) {
    const int nblk = 4 - d;
    for (int e = tid; e < nblk * 64; e += is::OFFDIAG_THREADS) {
        const int blk = e >> 6, r = (e >> 2) & 15, c4 = (e & 3) * 4, a = blk + d, b = blk;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int s = 0; s < 16 * d; ++s) {
            const float av = A[(b * 16 + s) * CH + a * 16 + r];
            const float4 tv = ld4(T + (b * 16 + s) * CH + b * 16 + c4);
            acc.x = fmaf(av, tv.x, acc.x);
            acc.y = fmaf(av, tv.y, acc.y);
            acc.z = fmaf(av, tv.z, acc.z);
            acc.w = fmaf(av, tv.w, acc.w);
        }
        *reinterpret_cast<float4 *>(XS + (blk * 16 + r) * 16 + c4) = acc;
    }
    offdiag_sync();
    for (int e = tid; e < nblk * 64; e += is::OFFDIAG_THREADS) {
        const int blk = e >> 6, r = (e >> 2) & 15, c4 = (e & 3) * 4, a = blk + d, b = blk;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int s = 0; s < 16; ++s) {
            const float tv = -TD[(a * 16 + s) * 16 + r];  // T[a16 + r][a16 + s]
            const float4 xv = ld4(XS + (blk * 16 + s) * 16 + c4);
            acc.x = fmaf(tv, xv.x, acc.x);
            acc.y = fmaf(tv, xv.y, acc.y);
            acc.z = fmaf(tv, xv.z, acc.z);
            acc.w = fmaf(tv, xv.w, acc.w);
        }
        *reinterpret_cast<float4 *>(T + (a * 16 + r) * CH + b * 16 + c4) = acc;
    }
    offdiag_sync();
}

// 16 warps per CTA.  Grid mode: one CTA per (chunk, head) of a window.
// List mode (p.fb_list set): the CTAs walk the chunk-heads the fast kernel
// listed, one at a time.  Per chunk-head, TMA brings the raw q, k, v tiles of
// the chunk's 64 tokens plus the 3 before them (the conv halo) and the alpha
// tile; the kernel forms G, q^, k^ (conv + SiLU + L2) and v (conv + SiLU) in
// shared memory, so every operand build reads shared memory.  The record
// images that involve no MMA (exp(G) . q, K^, P) go to the record from
// registers; W is staged in shared memory and bulk-stored, Ut^T rows go to
// the record from tensor memory.
template <typename Act>
__global__ void __launch_bounds__(is::NT, 1) prefill_intra_generic_kernel(const PrefillParams p,
                                                                       const __grid_constant__ CUtensorMap tm_q,
                                                                       const __grid_constant__ CUtensorMap tm_k,
                                                                       const __grid_constant__ CUtensorMap tm_v,
                                                                       const __grid_constant__ CUtensorMap tm_a) {
    static_assert(is::map_ok<Act>(), "intra shared-memory map overlaps");
    static_assert(CH % (16 * is::QW) == 0 && is::NT >= 4 * D, "drain split / thread roles need these");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1 KiB-aligned, still shared
    float *cref = reinterpret_cast<float *>(sm + is::SMALL);  // [128] c = mid of the log-decay range
    float *beta = cref + D;                                    // [64]
    int *flag = reinterpret_cast<int *>(beta + CH);            // [1]
    float *ec = reinterpret_cast<float *>(sm + is::SMALL + 1536);  // [128] exp(c)
    float *elc = ec + D;                                           // [128] exp(G_last - c)
    uint32_t *tbase = reinterpret_cast<uint32_t *>(flag + 1);  // [1]
    uint64_t *bar_ld = reinterpret_cast<uint64_t *>(sm + is::SMALL + 1024);
    uint64_t *bar_mma = bar_ld + 1;
    uint64_t *bar_v = bar_ld + 2;
    constexpr uint32_t TILE = is::tile_bytes<Act>();
    const Act *rq = reinterpret_cast<const Act *>(sm + is::RQ);
    const Act *rk = reinterpret_cast<const Act *>(sm + is::RK<Act>());
    const Act *rv = reinterpret_cast<const Act *>(sm + is::RV<Act>());
    const Act *ra = reinterpret_cast<const Act *>(sm + is::RA<Act>());
    const float *QHs = reinterpret_cast<const float *>(sm + is::IN0);
    const float *VVs = reinterpret_cast<const float *>(sm + is::IN0);
    const float *KHs = reinterpret_cast<const float *>(sm + is::KH);
    const float *GGs = reinterpret_cast<const float *>(sm + is::GG);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);
    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_v, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tbase, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase;
    uint32_t mma_phase = 0;  // bar_mma completes once or twice per chunk-head
    uint32_t ph = 0;         // bar_ld and bar_v complete once per chunk-head
    bool ok = true;
    for (int it = 0; ok; ++it) {
    int g, h;
    if (p.fb_list) {
        const int idx = int(blockIdx.x) + it * int(gridDim.x);
        if (idx >= int(*p.fb_count)) break;
        const uint32_t e = p.fb_list[idx];
        g = int(e / uint32_t(p.H));
        h = int(e % uint32_t(p.H));
    } else {
        if (it > 0) break;
        g = p.chunk_base + int(blockIdx.x);
        h = int(blockIdx.y);
    }
    const ChunkMeta cm = p.chunks[g];
    if (cm.len <= 0) continue;  // a padding entry of a device-built table: no chunk here
    const SeqMeta sq = p.seqs[cm.seq];
    char *rec = rec_ptr(p, g, h);
    if (tid == 0) {
        *flag = 0;
        mbar_arrive_expect_tx(bar_ld, 2 * TILE + uint32_t(CH * D * sizeof(Act)));
        tma_load_3d(sm + is::RQ, &tm_q, bar_ld, 0, h, cm.row0 - HALO);
        tma_load_3d(sm + is::RK<Act>(), &tm_k, bar_ld, 0, h, cm.row0 - HALO);
        tma_load_3d(sm + is::RA<Act>(), &tm_a, bar_ld, 0, h, cm.row0);
        if constexpr (is::v_early<Act>()) {
            mbar_arrive_expect_tx(bar_v, TILE);
            tma_load_3d(sm + is::RV<Act>(), &tm_v, bar_v, 0, h, cm.row0 - HALO);
        }
    }
    if (tid < CH)
        beta[tid] = tid < cm.len ? to_f32(static_cast<const Act *>(p.beta)[size_t(cm.row0 + tid) * p.H + h]) : 0.f;
    // conv tail of this head (resumed sequences), and the conv taps of the
    // channel this thread convolves: q or k (stream qk, channel cc, tokens
    // 32 qh .. 32 qh + 31), and v (threads 64..447, three per channel, while
    // T is formed)
    const Act *tail = sq.has_init ? static_cast<const Act *>(p.tails) + size_t(sq.slot) * 3 * p.n_ch + h * D : nullptr;
    const int qk = (tid >> 7) & 1, cc = tid & (D - 1), qh = tid >> 8;
    const int vt = tid - 64, vc = vt & (D - 1), vh = vt >> 7;
    const bool v_thread = vt >= 0 && vt < 3 * D;
    const float4 w_qk = conv_taps<Act>(p, qk, h, cc);
    const float4 w_v = v_thread ? conv_taps<Act>(p, 2, h, vc) : make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    ok = __syncthreads_and(mbar_wait(bar_ld, ph, p.err));
    // q^ = L2(SiLU(conv(q))), k^ likewise: two threads per channel, 32 tokens
    // each, the values kept in registers.  The warp's 32 lanes are 32
    // channels of one (stream, half): a transpose-reduce gives each lane the
    // warp's sum of squares of one token, the 4 warps of the (stream, half)
    // add theirs through shared memory, and the scaled values are stored once.
    float *GGw = reinterpret_cast<float *>(sm + is::GG);
    float *QHw = reinterpret_cast<float *>(sm + is::IN0), *KHw = reinterpret_cast<float *>(sm + is::KH);
    float *ssq = reinterpret_cast<float *>(sm + is::SSQ);
    {
        float y[32];
        if (ok) {
            conv_silu_regs32<Act>(qk ? rk : rq, cc, w_qk, qh * (CH / 2), cm.pos0, cm.len,
                                  tail ? tail + qk * p.H * D + cc : nullptr, p.n_ch, y);
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) y[e] = 0.f;
        }
        float s2[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) s2[e] = y[e] * y[e];
        lane_transpose_sum<32, 16>(s2, lane);
        const int grp = (qk * 2 + qh) * 4;  // the 4 warps of this (stream, half): warp & 3 = channel quarter
        ssq[(grp + (warp & 3)) * 32 + lane] = s2[0];
        // ln of the 128 bf16 mantissas 1 + m/128, in the c buffer (written only after G)
        if (sizeof(Act) == 2 && tid < D) cref[tid] = logf(1.0f + float(tid) * (1.0f / 128.0f));
        __syncthreads();
        float *rn = ssq + 512 + warp * 32;  // this warp's 32 token norms
        rn[lane] = rsqrtf(ssq[grp * 32 + lane] + ssq[(grp + 1) * 32 + lane] + ssq[(grp + 2) * 32 + lane] +
                          ssq[(grp + 3) * 32 + lane] + p.eps_l2);
        __syncwarp();
        float *outp = (qk ? KHw : QHw) + qh * (CH / 2) * D + cc;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 r4 = ld4(rn + e);
            outp[(e + 0) * D] = y[e + 0] * r4.x;
            outp[(e + 1) * D] = y[e + 1] * r4.y;
            outp[(e + 2) * D] = y[e + 2] * r4.z;
            outp[(e + 3) * D] = y[e + 3] * r4.w;
        }
    }
    // G = cumulative log decay, thread = (channel gi, half gh of the chunk);
    // the second half adds the first half's total below.  (A 4-byte alpha
    // tile is the G buffer itself: element in, element out.)
    const int gi = tid & (D - 1), gh = tid >> 7;
    if (ok && tid < 2 * D) {  // all 32 loads, then all 32 logarithms, then the scan: one latency each
        const int t0 = gh * (CH / 2);
        Act av[CH / 2];
        float lg[CH / 2];
#pragma unroll
        for (int e = 0; e < CH / 2; ++e) av[e] = ra[(t0 + e) * D + gi];
#pragma unroll
        for (int b = 0; b < CH / 2; b += 8)
            log_alpha8(*reinterpret_cast<const Act(*)[8]>(av + b), cref, cm.len - (t0 + b),
                       *reinterpret_cast<float(*)[8]>(lg + b));
        float G = 0.f;
#pragma unroll
        for (int e = 0; e < CH / 2; ++e) {
            if (t0 + e < cm.len) G += fmaxf(lg[e], kLogAlphaMin);
            GGw[(t0 + e) * D + gi] = G;
        }
    }
    __syncthreads();
    if (ok && tid >= D && tid < 2 * D) {
        const float g31 = GGw[(CH / 2 - 1) * D + gi];
        float gv[CH / 2];
#pragma unroll
        for (int e = 0; e < CH / 2; ++e) gv[e] = GGw[(CH / 2 + e) * D + gi];
#pragma unroll
        for (int e = 0; e < CH / 2; ++e) GGw[(CH / 2 + e) * D + gi] = gv[e] + g31;
    }
    __syncthreads();
    if (ok && tid < D) {
        const float g0 = GGs[tid], gl = GGs[(CH - 1) * D + tid];
        const float c = 0.5f * (g0 + gl);
        cref[tid] = c;
        ec[tid] = expf(c);
        elc[tid] = expf(gl - c);
        at<float>(rec, Rec::GAM)[tid] = expf(gl);
        at<float>(rec, Rec::ELC)[tid] = 1.0f;  // this kernel's K^ image already holds exp(G_last - G)
        if (g0 - gl > kSafeSpanGeneric) atomicOr(flag, 1);
    }
    __syncthreads();
    const bool exact = *flag != 0;
    // Within the safe span every decay factor of the chunk derives from one
    // exponential per element, E = exp(G - c) in [e^-80, e^80]:
    //   exp(G_r - c), exp(c - G_s) = 1/E, exp(G) = E e^c, exp(G_last - G) = e^(G_last - c) / E.
    // G is replaced by E in place.  The exact path keeps G.
    float *EE = reinterpret_cast<float *>(sm + is::GG);
    if (ok && !exact) {
        // a thread's float4s all sit at channels 4 * tid mod D: all loads first
        const float4 c4 = ld4(cref + (4 * tid) % D);
#pragma unroll 1
        for (int k0 = 0; k0 < CH * D / 4 / is::NT; k0 += 2) {
            float4 g[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) g[k] = ld4(GGs + 4 * (tid + (k0 + k) * is::NT));
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                g[k].x = expf(g[k].x - c4.x);
                g[k].y = expf(g[k].y - c4.y);
                g[k].z = expf(g[k].z - c4.z);
                g[k].w = expf(g[k].w - c4.w);
                *reinterpret_cast<float4 *>(EE + 4 * (tid + (k0 + k) * is::NT)) = g[k];
            }
        }
        __syncthreads();
    }

    // ---- phase 1: X = [K exp(G - c); Q exp(G - c)], Kb = K exp(c - G) -> A, P
    if (ok && !exact) {
        // One pass over (row r, 8-channel chunk c) of k^, q^ and E, which are
        // read once: X rows r and 64 + r = k^ E and q^ E, Kb row r = k^ / E,
        // and the record's exp(G) . q row 64 + r of WQ = q^ (E e^c).
        unsigned char *wq_hi = reinterpret_cast<unsigned char *>(rec + Rec::WQ_HI);
        unsigned char *wq_lo = reinterpret_cast<unsigned char *>(rec + Rec::WQ_LO);
#pragma unroll 1
        for (int u = tid; u < CH * (D / 8); u += is::NT) {
            const int r = u / (D / 8), c = u % (D / 8), k0 = 8 * c;
            float kk[8], qq[8], ee[8], cc[8], x[8];
            ld8(KHs + r * D + k0, kk);
            ld8(QHs + r * D + k0, qq);
            ld8(EE + r * D + k0, ee);
            ld8(ec + k0, cc);
            uint4 vh, vl;
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = kk[e] * ee[e];
            split8(x, vh, vl);
            *reinterpret_cast<uint4 *>(sm + is::X_HI + sw128_chunk(r, c, 2 * CH)) = vh;
            *reinterpret_cast<uint4 *>(sm + is::X_LO + sw128_chunk(r, c, 2 * CH)) = vl;
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = qq[e] * ee[e];
            split8(x, vh, vl);
            *reinterpret_cast<uint4 *>(sm + is::X_HI + sw128_chunk(CH + r, c, 2 * CH)) = vh;
            *reinterpret_cast<uint4 *>(sm + is::X_LO + sw128_chunk(CH + r, c, 2 * CH)) = vl;
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = kk[e] * rcp_approx(ee[e]);  // ee in [e^-80, e^80]
            split8(x, vh, vl);
            *reinterpret_cast<uint4 *>(sm + is::KB_HI + sw128_chunk(r, c, CH)) = vh;
            *reinterpret_cast<uint4 *>(sm + is::KB_LO + sw128_chunk(r, c, CH)) = vl;
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = qq[e] * (ee[e] * cc[e]);
            split8(x, vh, vl);
            *reinterpret_cast<uint4 *>(wq_hi + sw128_chunk(CH + r, c, 2 * CH)) = vh;
            *reinterpret_cast<uint4 *>(wq_lo + sw128_chunk(CH + r, c, 2 * CH)) = vl;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            mma3(tm, sbase + is::X_HI, sbase + is::X_LO, sbase + is::KB_HI, sbase + is::KB_LO, 128, CH, D,
                 idesc_bf16_f32(128, CH), false);
            mma_commit(bar_mma);
        }
    }
    // chain images that need no MMA: exp(G) . q (WQ rows 64 + r; above when
    // !exact) and K^ = exp(G_last - G) . k (rows r)
    if (ok && exact) {
        build_image(reinterpret_cast<unsigned char *>(rec + Rec::WQ_HI), reinterpret_cast<unsigned char *>(rec + Rec::WQ_LO),
                    CH, 16, tid, is::NT, [&](int r, int k0, float(&x)[8]) {
                        float a[8], gg[8];
                        ld8(QHs + r * D + k0, a);
                        ld8(GGs + r * D + k0, gg);
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = a[e] * expf(gg[e]);
                    }, CH, 2 * CH);
    }
    if (ok) {
        build_image(reinterpret_cast<unsigned char *>(rec + Rec::KH_HI), reinterpret_cast<unsigned char *>(rec + Rec::KH_LO),
                    CH, 16, tid, is::NT, [&](int r, int k0, float(&x)[8]) {
                        float kv[8], gv[8];
                        ld8(KHs + r * D + k0, kv);
                        ld8(GGs + r * D + k0, gv);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            x[e] = kv[e] * (exact ? expf(GGs[(CH - 1) * D + k0 + e] - gv[e]) : elc[k0 + e] * rcp_approx(gv[e]));
                    });
    }
    __syncthreads();
    // ---- A (s < r, times beta_r) -> fp32 smem, stored transposed (A[s * CH + r]
    // = A_rs), P (s <= r) -> record images
    float *A = reinterpret_cast<float *>(sm + is::A_F32);
    unsigned char *phi = reinterpret_cast<unsigned char *>(rec + Rec::PP_HI);
    unsigned char *plo = reinterpret_cast<unsigned char *>(rec + Rec::PP_LO);
    if (!exact) {
        ok = __syncthreads_and(ok && mbar_wait(bar_mma, mma_phase, p.err));
        mma_phase ^= 1;
        tc_fence_after();
        const int m = (warp & 3) * 32 + lane;  // TMEM lane = row of X; the QW warps of a quarter split the columns
        const int cbase = (warp >> 2) * (CH / is::QW);
        if (ok) {
#pragma unroll 1
            for (int c0 = cbase; c0 < cbase + CH / is::QW; c0 += 16) {
                float v[16];
                tmem_ld16(tm + (uint32_t((warp & 3) * 32) << 16) + c0, v);
                tmem_wait_ld();
                if (m < CH) {  // A^T: the warp's lanes (rows r = m) store consecutive words
                    const float bm = beta[m];
#pragma unroll
                    for (int e = 0; e < 16; ++e) A[(c0 + e) * CH + m] = (c0 + e < m) ? bm * v[e] : 0.f;
                } else {
                    const int r = m - CH;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float x[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = (c0 + 8 * half + e <= r) ? v[8 * half + e] : 0.f;
                        uint4 vh, vl;
                        split8(x, vh, vl);
                        const uint32_t off = sw128_chunk(r, (c0 >> 3) + half, CH);
                        *reinterpret_cast<uint4 *>(phi + off) = vh;
                        *reinterpret_cast<uint4 *>(plo + off) = vl;
                    }
                }
            }
        }
    } else if (ok) {
        // exact per-element exponentials (chunks whose decay span is too wide)
        for (int e = tid; e < CH * CH; e += is::NT) {
            const int r = e / CH, s = e % CH;
            float a = 0.f, pq = 0.f;
            if (s <= r) {
                for (int i = 0; i < D; ++i) {
                    const float f = KHs[s * D + i] * expf(GGs[r * D + i] - GGs[s * D + i]);
                    a = fmaf(KHs[r * D + i], f, a);
                    pq = fmaf(QHs[r * D + i], f, pq);
                }
            }
            A[s * CH + r] = s < r ? beta[r] * a : 0.f;
            const float pv = s <= r ? pq : 0.f;
            const __nv_bfloat16 ph = __float2bfloat16_rn(pv);
            const __nv_bfloat16 pl = __float2bfloat16_rn(pv - __bfloat162float(ph));
            const uint32_t off = sw128_offset(r, s, CH);
            *reinterpret_cast<__nv_bfloat16 *>(phi + off) = ph;
            *reinterpret_cast<__nv_bfloat16 *>(plo + off) = pl;
        }
    }
    tc_fence_before();
    __syncthreads();  // q^ is consumed (the exact path reads it for P): v takes its place
    if constexpr (!is::v_early<Act>()) {
        if (tid == 0 && ok) {  // the phase-1 images are consumed: the raw v tile may land there
            mbar_arrive_expect_tx(bar_v, TILE);
            tma_load_3d(sm + is::RV<Act>(), &tm_v, bar_v, 0, h, cm.row0 - HALO);
        }
    }
    // ---- T = (I + A)^-1 (unit lower triangular), 16 x 16 blocks
    float *T = reinterpret_cast<float *>(sm + is::T_F32);
    float *XS = reinterpret_cast<float *>(sm + is::XS_C);
    float *TD = reinterpret_cast<float *>(sm + is::TDIAG);  // TD[(a16 + s) 16 + r] = T[a16 + r][a16 + s]
    for (int e = tid; e < CH * CH; e += is::NT) T[e] = 0.f;  // the blocks above the diagonal stay 0
    __syncthreads();
    // Diagonal 16 x 16 blocks by forward substitution, a lane per column with
    // the column in registers (fully unrolled): lanes 0-15 of warp w take
    // block 2w, lanes 16-31 block 2w + 1.  Rows above the lane's column come
    // out 0 by themselves (every earlier entry of the column is 0).
    if (warp < 2) {
        const int b0 = (warp * 2 + (lane >> 4)) * 16, c = lane & 15;
        float tc[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int s = 0; s < r; ++s) acc = fmaf(-A[(b0 + s) * CH + b0 + r], tc[s], acc);
            tc[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) T[(b0 + r) * CH + b0 + c] = tc[r];
#pragma unroll
        for (int r4 = 0; r4 < 16; r4 += 4)
            *reinterpret_cast<float4 *>(TD + (b0 + c) * 16 + r4) = make_float4(tc[r4], tc[r4 + 1], tc[r4 + 2], tc[r4 + 3]);
    }
    // meanwhile threads 64..447 form v = SiLU(conv(v raw)) in the q^ buffer,
    // three threads per channel (tokens 0..23, 24..47, 48..63)
    bool vok = true;
    if (v_thread) {
        // a late tile is only requested while ok; an early one is always in flight
        vok = (is::v_early<Act>() || ok) ? mbar_wait(bar_v, ph, p.err) : false;
        if (ok && vok)
            conv_silu_channel<Act>(rv, vc, w_v, vh * 24, vh < 2 ? 24 : CH - 48, cm.pos0, cm.len,
                                   tail ? tail + 2 * p.H * D + vc : nullptr, p.n_ch, reinterpret_cast<float *>(sm + is::IN0));
    }
    ok = __syncthreads_and(ok && vok);
    // ---- phase 3: W^T = (beta exp(G) . K)^T T^T and Ut^T = (beta V)^T T^T.
    // Warps 0..5 form T's blocks below the diagonal, by distance d, while the
    // other warps build the two operand images that do not involve T (the
    // off-diagonal levels have at most 192 work items).
    if (tid < is::OFFDIAG_THREADS) {
#pragma unroll 1
        for (int d = 1; d < 4; ++d) tri_offdiag(A, T, XS, TD, tid, d);
    } else if (ok) {
        const int t2 = tid - is::OFFDIAG_THREADS, n2 = is::NT - is::OFFDIAG_THREADS;
        build_image<true>(sm + is::AK_HI, sm + is::AK_LO, D, 8, t2, n2, [&](int i, int s0, float(&x)[8]) {
            const float cc = ec[i];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float gv = GGs[(s0 + e) * D + i];
                x[e] = beta[s0 + e] * (exact ? expf(gv) : gv * cc) * KHs[(s0 + e) * D + i];
            }
        });
        build_image<true>(sm + is::AV_HI, sm + is::AV_LO, D, 8, t2, n2, [&](int j, int s0, float(&x)[8]) {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = beta[s0 + e] * VVs[(s0 + e) * D + j];
        });
    }
    __syncthreads();
    if (ok) {
        build_image(sm + is::T_HI, sm + is::T_LO, CH, 8, tid, is::NT, [&](int r, int s0, float(&x)[8]) {
            ld8(T + r * CH + s0, x);
        });
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && ok) {
        const uint32_t id = idesc_bf16_f32(128, CH);
        mma3(tm + 64, sbase + is::AK_HI, sbase + is::AK_LO, sbase + is::T_HI, sbase + is::T_LO, D, CH, CH, id, false);
        mma3(tm + 128, sbase + is::AV_HI, sbase + is::AV_LO, sbase + is::T_HI, sbase + is::T_LO, D, CH, CH, id, false);
        mma_commit(bar_mma);
    }
    ok = __syncthreads_and(ok && mbar_wait(bar_mma, mma_phase, p.err));
    mma_phase ^= 1;
    tc_fence_after();
    // W (staged transposed from TMEM lane i into shared memory, then bulk-
    // stored as rows 0..63 of WQ) and Ut^T row j = i of the record: the warps
    // of a lane quarter split the 64 token columns
    unsigned char *whi = sm + is::IN0, *wlo = sm + is::IN0 + 16384;
    const int i = (warp & 3) * 32 + lane;
    const int cbase = (warp >> 2) * (CH / is::QW);
    if (ok) {
        float *UT = at<float>(rec, Rec::UT) + size_t(i) * CH;
#pragma unroll 1
        for (int c0 = cbase; c0 < cbase + CH / is::QW; c0 += 16) {
            float v[16], u[16];
            tmem_ld16(tm + (uint32_t((warp & 3) * 32) << 16) + 64 + c0, v);
            tmem_ld16(tm + (uint32_t((warp & 3) * 32) << 16) + 128 + c0, u);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int r = c0 + e;
                const __nv_bfloat16 wh = __float2bfloat16_rn(v[e]);
                const __nv_bfloat16 wl = __float2bfloat16_rn(v[e] - __bfloat162float(wh));
                const uint32_t off = sw128_offset(r, i, CH);
                *reinterpret_cast<__nv_bfloat16 *>(whi + off) = wh;
                *reinterpret_cast<__nv_bfloat16 *>(wlo + off) = wl;
            }
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4 *>(UT + 4 * ut_chunk(i, (c0 + e) >> 2)) = make_float4(u[e], u[e + 1], u[e + 2], u[e + 3]);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        // a 64-row image's K-block b holds the same bytes as rows 0..63 of K-block b of WQ
        bulk_store(rec + Rec::WQ_HI, whi, 8192);
        bulk_store(rec + Rec::WQ_HI + 16384, whi + 8192, 8192);
        bulk_store(rec + Rec::WQ_LO, wlo, 8192);
        bulk_store(rec + Rec::WQ_LO + 16384, wlo + 8192, 8192);
        bulk_commit();
        bulk_wait_read();  // shared memory is reused by the next chunk-head
    }
    ph ^= 1;
    tc_fence_before();
    __syncthreads();  // shared memory and TMEM are reused by the next chunk-head
    }  // chunk-heads
    if (warp == 0) tmem_dealloc(tm, 256);
}


}  // namespace

template <typename Act>
kda_status intra_generic_prepare() {
    return cudaFuncSetAttribute(prefill_intra_generic_kernel<Act>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(1024 + is::BYTES<Act>())) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

template <typename Act>
kda_status launch_intra_generic(const PrefillParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                                const CUtensorMap &mv, const CUtensorMap &ma, dim3 grid, cudaStream_t s) {
    const ProfScope prof(KDA_KERNEL_PREFILL_INTRA_EXACT, s);
    prefill_intra_generic_kernel<Act><<<grid, is::NT, 1024 + is::BYTES<Act>(), s>>>(p, mq, mk, mv, ma);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

template kda_status intra_generic_prepare<float>();
template kda_status intra_generic_prepare<__nv_bfloat16>();
template kda_status launch_intra_generic<float>(const PrefillParams &, const CUtensorMap &, const CUtensorMap &,
                                                const CUtensorMap &, const CUtensorMap &, dim3, cudaStream_t);
template kda_status launch_intra_generic<__nv_bfloat16>(const PrefillParams &, const CUtensorMap &, const CUtensorMap &,
                                                        const CUtensorMap &, const CUtensorMap &, dim3, cudaStream_t);

}  // namespace pf
}  // namespace kda
