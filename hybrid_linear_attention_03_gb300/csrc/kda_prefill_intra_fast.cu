// kda_prefill_intra_fast.cu -- the intra-chunk prefill kernel for bf16
// activations, one CTA (16 warps) per (chunk, head).
//
// "vLLM Kimi K3 지원", section "Fused Kernels 및 메타데이터 최적화", KDA Prefill
// bullet: prefill runs chunked (FlashKDA).  Per (chunk, head), with G_r the
// cumulative log decay per key channel and c the middle of its range over the
// chunk, E = exp(G - c), K~ = k^ E, Q~ = q^ E, K^ = k^ / E:
//   [A; P] = [K~; Q~] K^^T                       (A_rs times beta_r, s < r; P_rs, s <= r)
//   T = (I + A)^-1                                (blocked, CUDA cores)
//   W^T = diag(exp(c)) K~^T (T diag(beta))^T      Ut^T = V^T (T diag(beta))^T
//   (exp(G) . q)^T = diag(exp(c)) Q~^T            (an MMA with the identity)
// which is the generic kernel's arithmetic with W's factor exp(G) = E exp(c)
// split so that every operand is one of three images built once.
//
// Every image is built token-major, a thread holding 2 tokens x 8 channels
// in registers: conv + SiLU, the L2 norm (a 16-lane shuffle reduction over
// the head's channels), the decay factors and the bf16 hi / lo split all
// happen in registers, and each 16-byte chunk is stored once.  The products
// that need an image transposed read it MN-major (kda_sm100.cuh), so no
// column-wise pass over shared memory is needed.  The cumulative decay G is a
// per-warp prefix (one shuffle) plus a scan of the 16 warp totals.
//
// Phases (bar = CTA barrier):
//   TMA q, k, alpha (and v)  | identity image, beta, ln table
//   G, E (registers) bar scan bar
//   k pass: K~, K^ images    q pass: Q~ image                        bar
//   MMA [A; P] -> commit a;  MMA Q~^T -> commit t;  K^ image -> record (bulk)
//   v pass: v image (under the MMAs)
//   wait a: A^T -> smem, P -> record                                  bar
//   diagonal 16 x 16 blocks of T (2 warps) | wait t: Q^T rows -> record (14 warps)  bar
//   3 levels of off-diagonal blocks (2 bar each);  (T diag beta) image  bar
//   MMA W^T, Ut^T -> wait: W^T rows, Ut^T rows -> record
// A chunk whose decay span exceeds kSafeSpanFast is appended to the fallback
// list and left to the generic kernel.
//
// Shared memory (bytes from a 1 KiB-aligned base), 182 KiB, one CTA per SM:
//   RQ, RK, RA, RV  raw q, k (67 rows), alpha (64 rows), v (67 rows) tiles
//   VIMG            v image hi / lo [64 s][128 j], over RQ / RK after the q pass
//   X               [K~; Q~] image hi / lo [128][128]; the rows of Q~ in its
//                   first K block later hold the (T diag beta) image
//   KB              K^ image hi / lo [64][128]; after MMA 1, A^T and T fp32 [64][64]
//   IDN             identity [64][64] bf16
//   SCAN            warp totals of G; later TD (T's diagonal blocks, transposed)
//                   and XS (partial products of the off-diagonal levels)
//   SMALL           ln table, c, exp(c), G_0, beta, mbarriers
// Tensor memory (256 columns): [0, 64) [A; P], then W^T; [64, 128) Q~^T;
// [128, 192) Ut^T.
#include "kda_prefill.cuh"

namespace kda {
namespace pf {
namespace {

namespace fs {
constexpr int NT = 512;
constexpr uint32_t TILE = uint32_t((CH + HALO) * D * 2);  // one raw 67-row bf16 tile
constexpr uint32_t RQ = 0, RK = 17408, RA = 34816, RV = 51200;
constexpr uint32_t VIMG = 0, VIMG_LO = 16384;
constexpr uint32_t X = 68608, X_LO = X + 32768;
constexpr uint32_t KB = X + 65536, KB_LO = KB + 16384;
constexpr uint32_t AT = KB, TT = KB + 16384;
constexpr uint32_t TB = X + 8192, TB_LO = X_LO + 8192;
constexpr uint32_t IDN = KB + 32768;
constexpr uint32_t SCAN = IDN + 8192, TD = SCAN, XS = SCAN + 4096;
constexpr uint32_t SMALL = SCAN + 8192;
constexpr uint32_t LNM = SMALL, CREF = SMALL + 512, EC = SMALL + 1024, G0 = SMALL + 1536, BETA = SMALL + 2048;
constexpr uint32_t BARS = SMALL + 2304, TBASE = BARS + 64;
constexpr uint32_t BYTES = SMALL + 2560;
static_assert(RK >= RQ + TILE && RA >= RK + TILE && RV >= RA + CH * D * 2 && X >= RV + TILE, "raw tiles overlap");
static_assert(VIMG_LO + 16384 <= RA, "the v image overlaps the alpha tile");
static_assert(X % 1024 == 0 && KB % 1024 == 0 && IDN % 1024 == 0 && TB % 1024 == 0, "images need 1 KiB alignment");
static_assert(BYTES + 1024 <= 232448, "shared memory");
}  // namespace fs

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint4 lds16(const unsigned char *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ void unpack8(const uint4 u, float (&x)[8]) {
    x[0] = bf_lo(u.x); x[1] = bf_hi(u.x); x[2] = bf_lo(u.y); x[3] = bf_hi(u.y);
    x[4] = bf_lo(u.z); x[5] = bf_hi(u.z); x[6] = bf_lo(u.w); x[7] = bf_hi(u.w);
}

// ln(alpha) of 8 packed bf16 values, the generic kernel's log_alpha8 on a
// 16-byte register word (no trip through local memory).
__device__ __forceinline__ void log_alpha8_u4(const uint4 u, const float *lnm, int n_valid, float (&l)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    bool normal = true;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t b = (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu, ex = (b >> 7) & 0xFFu;
        normal = normal && (e >= n_valid || ((b >> 15) == 0 && ex != 0 && ex != 0xFFu));
    }
    if (__all_sync(0xffffffffu, normal)) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t b = (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
            l[e] = fmaf(float(int((b >> 7) & 0xFFu) - 127), 0.6931471805599453f, lnm[b & 0x7Fu]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) l[e] = logf(__uint_as_float(((w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16));
    }
}

// Causal conv (width 4, last tap on the current token) + SiLU of tokens r0
// and r0 + 1, channels ch0 .. ch0 + 7 of stream s (0 q, 1 k, 2 v), from a raw
// tile whose row t + 3 is token t.  Rows before the segment start come from
// the slot's conv tail (tail: the slot's tail at this head's channel 0 of
// stream 0) or are zero; tokens past the segment end give 0.
__device__ __forceinline__ void conv_pair(const unsigned char *tile, const PrefillParams &p, int s, int h, int ch0,
                                          int r0, int pos0, int len, const __nv_bfloat16 *tail, float (&y)[2][8]) {
    const uint4 *wp = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.conv_w) +
                                                      (size_t(s) * p.H * D + size_t(h) * D + ch0) * 4);
    uint4 w4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w4[i] = __ldg(wp + i);
    float x[5][8];
#pragma unroll
    for (int j = 0; j < 5; ++j) {
        const int row = r0 + j, pos = pos0 - HALO + row;
        uint4 u = make_uint4(0u, 0u, 0u, 0u);
        if (pos >= 0)
            u = lds16(tile + row * (D * 2) + ch0 * 2);
        else if (tail)
            u = *reinterpret_cast<const uint4 *>(tail + size_t(HALO + pos) * p.n_ch + size_t(s) * p.H * D + ch0);
        unpack8(u, x[j]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint4 t = w4[e >> 1];
        const uint32_t wa = (e & 1) ? t.z : t.x, wb = (e & 1) ? t.w : t.y;
        const float w0 = bf_lo(wa), w1 = bf_hi(wa), w2 = bf_lo(wb), w3 = bf_hi(wb);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float acc = w0 * x[q][e];
            acc = fmaf(w1, x[q + 1][e], acc);
            acc = fmaf(w2, x[q + 2][e], acc);
            acc = fmaf(w3, x[q + 3][e], acc);
            y[q][e] = r0 + q < len ? acc * sigmoid_fast(acc) : 0.f;
        }
    }
}

// Scales the pair's two token rows by 1 / sqrt(|row|^2 + eps): the 16 lanes
// sharing the tokens hold the head's 128 channels.
__device__ __forceinline__ void l2_pair(float (&y)[2][8], float eps) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(y[q][e], y[q][e], ss);
#pragma unroll
        for (int o = 8; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = rsqrtf(ss + eps);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[q][e] *= r;
    }
}

__device__ __forceinline__ void store_split(unsigned char *hi, unsigned char *lo, uint32_t off, const float (&x)[8]) {
    uint4 vh, vl;
    split8(x, vh, vl);
    *reinterpret_cast<uint4 *>(hi + off) = vh;
    *reinterpret_cast<uint4 *>(lo + off) = vl;
}

__global__ void __launch_bounds__(fs::NT, 1) prefill_intra_fast_kernel(const PrefillParams p,
                                                                    const __grid_constant__ CUtensorMap tm_q,
                                                                    const __grid_constant__ CUtensorMap tm_k,
                                                                    const __grid_constant__ CUtensorMap tm_v,
                                                                    const __grid_constant__ CUtensorMap tm_a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *lnm = reinterpret_cast<float *>(sm + fs::LNM);
    float *cref = reinterpret_cast<float *>(sm + fs::CREF);
    float *ec = reinterpret_cast<float *>(sm + fs::EC);
    float *g0s = reinterpret_cast<float *>(sm + fs::G0);
    float *beta = reinterpret_cast<float *>(sm + fs::BETA);
    uint64_t *bar_ld = reinterpret_cast<uint64_t *>(sm + fs::BARS);
    uint64_t *bar_v = bar_ld + 1, *bar_a = bar_ld + 2, *bar_t = bar_ld + 3, *bar_w = bar_ld + 4;
    uint32_t *tbase = reinterpret_cast<uint32_t *>(sm + fs::TBASE);
    float *scan = reinterpret_cast<float *>(sm + fs::SCAN);
    float *At = reinterpret_cast<float *>(sm + fs::AT);  // At[s * 64 + r] = A_rs
    float *T = reinterpret_cast<float *>(sm + fs::TT);   // T[r * 64 + s]
    float *TD = reinterpret_cast<float *>(sm + fs::TD);  // TD[(a * 16 + s) * 16 + r] = T[16 a + r][16 a + s]
    float *XS = reinterpret_cast<float *>(sm + fs::XS);
    const int g = p.chunk_base + blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ChunkMeta cm = p.chunks[g];
    if (cm.len <= 0) return;  // a padding entry of a device-built table: no chunk here
    const SeqMeta sq = p.seqs[cm.seq];
    char *rec = rec_ptr(p, g, h);
    const uint32_t sbase = smem_u32(sm);
    if (tid == 0) {
        for (int b = 0; b < 5; ++b) mbar_init(bar_ld + b, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_ld, 2 * fs::TILE + uint32_t(CH * D * 2));
        tma_load_3d(sm + fs::RQ, &tm_q, bar_ld, 0, h, cm.row0 - HALO);
        tma_load_3d(sm + fs::RK, &tm_k, bar_ld, 0, h, cm.row0 - HALO);
        tma_load_3d(sm + fs::RA, &tm_a, bar_ld, 0, h, cm.row0);
        mbar_arrive_expect_tx(bar_v, fs::TILE);
        tma_load_3d(sm + fs::RV, &tm_v, bar_v, 0, h, cm.row0 - HALO);
    }
    if (tid < CH)
        beta[tid] = tid < cm.len ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p.beta)[size_t(cm.row0 + tid) * p.H + h])
                                 : 0.f;
    if (tid < 128) lnm[tid] = logf(1.0f + float(tid) * (1.0f / 128.0f));  // ln of the bf16 mantissas 1 + m/128
    {   // identity [64 r][64 s]: chunk (r, c) holds s = 8c .. 8c + 7; bf16 1.0 is 0x3F80
        const int r = tid >> 3, c = tid & 7, e = r & 7;
        const uint32_t one = ((r >> 3) == c) ? ((r & 1) ? 0x3F800000u : 0x00003F80u) : 0u;
        *reinterpret_cast<uint4 *>(sm + fs::IDN + sw128_chunk(r, c, CH)) =
            make_uint4((e >> 1) == 0 ? one : 0u, (e >> 1) == 1 ? one : 0u, (e >> 1) == 2 ? one : 0u, (e >> 1) == 3 ? one : 0u);
    }
    if (warp == 0) tmem_alloc(tbase, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase;
    bool ok = __syncthreads_and(mbar_wait(bar_ld, 0, p.err));

    // This thread's unit: tokens r0, r0 + 1 (pair pr) x channels ch0 .. ch0 + 7.
    // A warp holds pairs 2 warp (lanes 0-15) and 2 warp + 1 (lanes 16-31).
    const int pr = 2 * warp + (lane >> 4), cb = lane & 15, r0 = 2 * pr, ch0 = 8 * cb;
    const __nv_bfloat16 *tail =
        sq.has_init ? static_cast<const __nv_bfloat16 *>(p.tails) + size_t(sq.slot) * 3 * p.n_ch + size_t(h) * D : nullptr;

    // ---- G = cumulative log decay, E = exp(G - c) --------------------------
    float gA[8], gB[8];
    {
        const uint4 a0 = lds16(sm + fs::RA + r0 * (D * 2) + ch0 * 2), a1 = lds16(sm + fs::RA + (r0 + 1) * (D * 2) + ch0 * 2);
        float l0[8], l1[8];
        log_alpha8_u4(a0, lnm, r0 < cm.len ? 8 : 0, l0);
        log_alpha8_u4(a1, lnm, r0 + 1 < cm.len ? 8 : 0, l1);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            l0[e] = r0 < cm.len ? fmaxf(l0[e], kLogAlphaMin) : 0.f;
            l1[e] = r0 + 1 < cm.len ? fmaxf(l1[e], kLogAlphaMin) : 0.f;
            gA[e] = l0[e];
            gB[e] = l0[e] + l1[e];
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {  // the odd pair adds the even pair's total
            const float t = __shfl_up_sync(0xffffffffu, gB[e], 16);
            if (lane >= 16) {
                gA[e] += t;
                gB[e] += t;
            }
        }
        if (lane >= 16) {  // this warp's total over its 4 tokens
            *reinterpret_cast<float4 *>(scan + warp * D + ch0) = make_float4(gB[0], gB[1], gB[2], gB[3]);
            *reinterpret_cast<float4 *>(scan + warp * D + ch0 + 4) = make_float4(gB[4], gB[5], gB[6], gB[7]);
        }
        if (warp == 0 && lane < 16) {  // G of token 0
            *reinterpret_cast<float4 *>(g0s + ch0) = make_float4(l0[0], l0[1], l0[2], l0[3]);
            *reinterpret_cast<float4 *>(g0s + ch0 + 4) = make_float4(l0[4], l0[5], l0[6], l0[7]);
        }
    }
    __syncthreads();
    int wide = 0;
    if (tid < D) {  // exclusive scan of the 16 warp totals of channel tid
        float t[16];
#pragma unroll
        for (int w = 0; w < 16; ++w) t[w] = scan[w * D + tid];
        float run = 0.f;
#pragma unroll
        for (int w = 0; w < 16; ++w) {
            scan[w * D + tid] = run;
            run += t[w];
        }
        const float gfirst = g0s[tid], c = 0.5f * (gfirst + run);
        cref[tid] = c;
        ec[tid] = expf(c);
        at<float>(rec, Rec::GAM)[tid] = expf(run);
        at<float>(rec, Rec::ELC)[tid] = expf(run - c);
        wide = gfirst - run > kSafeSpanFast;
    }
    const bool exact = __syncthreads_or(wide) != 0;
    if (!ok || exact) {
        // a chunk this kernel cannot take: the generic kernel's list gets it
        if (ok && tid == 0) p.fb_list[atomicAdd(p.fb_count, 1u)] = uint32_t(g) * uint32_t(p.H) + uint32_t(h);
        mbar_wait(bar_v, 0, p.err);  // no copy may land after the CTA is gone
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tm, 256);
        return;
    }
    float E0[8], E1[8];
    {
        float pre[8], cc[8];
        ld8(scan + warp * D + ch0, pre);
        ld8(cref + ch0, cc);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            E0[e] = ex2_approx((pre[e] + gA[e] - cc[e]) * kLog2e);
            E1[e] = ex2_approx((pre[e] + gB[e] - cc[e]) * kLog2e);
        }
    }

    // ---- k pass: K~ = k^ E (X rows r), K^ = k^ / E (KB rows r) ---------------
    {
        float y[2][8];
        conv_pair(sm + fs::RK, p, 1, h, ch0, r0, cm.pos0, cm.len, tail, y);
        l2_pair(y, p.eps_l2);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = y[q][e] * (q ? E1[e] : E0[e]);
            store_split(sm + fs::X, sm + fs::X_LO, sw128_chunk(r0 + q, cb, 2 * CH), x);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = y[q][e] * rcp_approx(q ? E1[e] : E0[e]);  // E in [e^-60, e^60]
            store_split(sm + fs::KB, sm + fs::KB_LO, sw128_chunk(r0 + q, cb, CH), x);
        }
    }
    // ---- q pass: Q~ = q^ E (X rows 64 + r) -----------------------------------
    {
        float y[2][8];
        conv_pair(sm + fs::RQ, p, 0, h, ch0, r0, cm.pos0, cm.len, tail, y);
        l2_pair(y, p.eps_l2);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = y[q][e] * (q ? E1[e] : E0[e]);
            store_split(sm + fs::X, sm + fs::X_LO, sw128_chunk(CH + r0 + q, cb, 2 * CH), x);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        const Operand xop{sbase + fs::X, sbase + fs::X_LO, false, 2 * CH * 128};
        const Operand kbop{sbase + fs::KB, sbase + fs::KB_LO, false, CH * 128};
        mma_split(tm, xop, kbop, D, idesc_bf16_f32(128, CH), 3, false);  // [A; P] (unmasked)
        mma_commit(bar_a);
        // Q~^T: Q~ (X rows 64..127) read MN-major times the identity; hi + lo is exact
        const Operand qt{sbase + fs::X + CH * 128, sbase + fs::X_LO + CH * 128, true, 2 * CH * 128};
        const Operand id{sbase + fs::IDN, sbase + fs::IDN, false, CH * 128};
        mma_split(tm + 64, qt, id, CH, idesc_bf16_f32(128, CH, true, false), 2, false);
        mma_commit(bar_t);
        // K^ image -> record (the chain's operand), while the MMAs run
        bulk_store(rec + Rec::KH_HI, sm + fs::KB, 16384);
        bulk_store(rec + Rec::KH_LO, sm + fs::KB_LO, 16384);
        bulk_commit();
    }
    // ---- v pass (under the MMAs): v image over the raw q, k tiles ------------
    bool okv = mbar_wait(bar_v, 0, p.err);
    if (okv) {
        float y[2][8];
        conv_pair(sm + fs::RV, p, 2, h, ch0, r0, cm.pos0, cm.len, tail, y);
#pragma unroll
        for (int q = 0; q < 2; ++q) store_split(sm + fs::VIMG, sm + fs::VIMG_LO, sw128_chunk(r0 + q, cb, CH), y[q]);
    }
    okv = okv && mbar_wait(bar_a, 0, p.err);
    if (tid == 0) bulk_wait_read();  // KB becomes A^T and T below
    ok = __syncthreads_and(okv);
    tc_fence_after();
    const int qd = warp & 3, cs = (warp >> 2) * 16;  // TMEM lane quarter, 16-column slice
    if (ok) {
        // ---- A^T (s < r, times beta_r) -> smem; P (s <= r) -> record --------
        float v[16];
        tmem_ld16(tm + (uint32_t(qd * 32) << 16) + cs, v);
        tmem_wait_ld();
        if (qd < 2) {
            const int r = qd * 32 + lane;
            const float bm = beta[r];
#pragma unroll
            for (int e = 0; e < 16; ++e) At[(cs + e) * CH + r] = (cs + e < r) ? bm * v[e] : 0.f;
        } else {
            const int r = (qd - 2) * 32 + lane;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = (cs + 8 * hh + e <= r) ? v[8 * hh + e] : 0.f;
                store_split(reinterpret_cast<unsigned char *>(rec + Rec::PP_HI), reinterpret_cast<unsigned char *>(rec + Rec::PP_LO),
                            sw128_chunk(r, (cs >> 3) + hh, CH), x);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    bool okt = true;
    if (ok && warp < 2) {
        // ---- diagonal 16 x 16 blocks of T by forward substitution: lane =
        // column c of block b, the column in registers
        const int b = tid >> 4, c = tid & 15, b16 = 16 * b;
        float tc[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int k = 0; k < r; ++k) acc = fmaf(-At[(b16 + k) * CH + b16 + r], tc[k], acc);
            tc[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) T[(b16 + r) * CH + b16 + c] = tc[r];
#pragma unroll
        for (int r4 = 0; r4 < 16; r4 += 4)
            *reinterpret_cast<float4 *>(TD + (b16 + c) * 16 + r4) = make_float4(tc[r4], tc[r4 + 1], tc[r4 + 2], tc[r4 + 3]);
    } else if (ok) {
        // ---- meanwhile (exp(G) . q)^T rows = exp(c_i) Q~^T -> record WQ block 1;
        // the 16 (quarter, slice) units over warps 2..15
        okt = mbar_wait(bar_t, 0, p.err);
        tc_fence_after();
        if (okt) {
            const int k0 = (qd >= 2) ? (warp - 2) >> 2 : (warp - 4) >> 2;
            const int nk = (qd < 2 && k0 == 2) ? 2 : 1;
            const int i = qd * 32 + lane;
            const float e_c = ec[i];
            for (int k = k0; k < k0 + nk; ++k) {
                float v[16];
                tmem_ld16(tm + (uint32_t(qd * 32) << 16) + 64 + 16 * k, v);
                tmem_wait_ld();
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = v[8 * hh + e] * e_c;
                    store_split(reinterpret_cast<unsigned char *>(rec + Rec::WQ_HI + Rec::WQ_BLOCK),
                                reinterpret_cast<unsigned char *>(rec + Rec::WQ_LO + Rec::WQ_BLOCK), sw128_chunk(i, 2 * k + hh, D), x);
                }
            }
        }
    }
    ok = __syncthreads_and(ok && okt);
    // ---- off-diagonal blocks, by distance d: T_ab = -T_aa sum_{b <= c < a} A_ac T_cb
    if (ok) {
#pragma unroll 1
        for (int d = 1; d < 4; ++d) {
            const int nblk = 4 - d;
            for (int e = tid; e < nblk * d * 64; e += fs::NT) {  // partial products A_ac T_cb
                const int q4 = (e & 3) * 4, r = (e >> 2) & 15, bt = e >> 6;
                const int blk = bt / d, c = blk + (bt - blk * d), a = blk + d;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float av = At[(16 * c + k) * CH + 16 * a + r];
                    const float4 tv = ld4(T + (16 * c + k) * CH + 16 * blk + q4);
                    acc.x = fmaf(av, tv.x, acc.x);
                    acc.y = fmaf(av, tv.y, acc.y);
                    acc.z = fmaf(av, tv.z, acc.z);
                    acc.w = fmaf(av, tv.w, acc.w);
                }
                *reinterpret_cast<float4 *>(XS + (bt * 16 + r) * 16 + q4) = acc;
            }
            __syncthreads();
            for (int e = tid; e < nblk * 64; e += fs::NT) {  // T_ab = -T_aa X_ab
                const int q4 = (e & 3) * 4, r = (e >> 2) & 15, blk = e >> 6, a = blk + d;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const float tv = -TD[(16 * a + k) * 16 + r];
                    float4 xv = ld4(XS + ((blk * d) * 16 + k) * 16 + q4);
                    for (int t = 1; t < d; ++t) {
                        const float4 x2 = ld4(XS + ((blk * d + t) * 16 + k) * 16 + q4);
                        xv.x += x2.x;
                        xv.y += x2.y;
                        xv.z += x2.z;
                        xv.w += x2.w;
                    }
                    acc.x = fmaf(tv, xv.x, acc.x);
                    acc.y = fmaf(tv, xv.y, acc.y);
                    acc.z = fmaf(tv, xv.z, acc.z);
                    acc.w = fmaf(tv, xv.w, acc.w);
                }
                *reinterpret_cast<float4 *>(T + (16 * a + r) * CH + 16 * blk + q4) = acc;
            }
            __syncthreads();
        }
        // ---- (T diag beta) image [64 r][64 s] (s <= r), over Q~'s first K block
        {
            const int r = tid >> 3, c = tid & 7;
            float t8[8], b8[8], x[8];
            ld8(T + r * CH + 8 * c, t8);
            ld8(beta + 8 * c, b8);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = (8 * c + e <= r) ? t8[e] * b8[e] : 0.f;
            store_split(sm + fs::TB, sm + fs::TB_LO, sw128_chunk(r, c, CH), x);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && ok) {
        // W^T / exp(c) = K~^T (T diag beta)^T and Ut^T = V^T (T diag beta)^T: K~ and V read MN-major
        const Operand kt{sbase + fs::X, sbase + fs::X_LO, true, 2 * CH * 128};
        const Operand vt{sbase + fs::VIMG, sbase + fs::VIMG_LO, true, CH * 128};
        const Operand tb{sbase + fs::TB, sbase + fs::TB_LO, false, CH * 128};
        const uint32_t id = idesc_bf16_f32(128, CH, true, false);
        mma_split(tm, kt, tb, CH, id, 3, false);
        mma_split(tm + 128, vt, tb, CH, id, 3, false);
        mma_commit(bar_w);
    }
    ok = __syncthreads_and(ok && mbar_wait(bar_w, 0, p.err));
    tc_fence_after();
    if (ok) {
        // ---- W^T row i (times exp(c_i)) and Ut^T row j = i -> record ---------
        const int i = qd * 32 + lane;
        float w[16], u[16];
        tmem_ld16(tm + (uint32_t(qd * 32) << 16) + cs, w);
        tmem_ld16(tm + (uint32_t(qd * 32) << 16) + 128 + cs, u);
        tmem_wait_ld();
        const float e_c = ec[i];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = w[8 * hh + e] * e_c;
            store_split(reinterpret_cast<unsigned char *>(rec + Rec::WQ_HI), reinterpret_cast<unsigned char *>(rec + Rec::WQ_LO),
                        sw128_chunk(i, (cs >> 3) + hh, D), x);
        }
        float *ut = at<float>(rec, Rec::UT) + size_t(i) * CH + cs;
#pragma unroll
        for (int e = 0; e < 16; e += 4) *reinterpret_cast<float4 *>(ut + e) = make_float4(u[e], u[e + 1], u[e + 2], u[e + 3]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

}  // namespace

kda_status intra_fast_prepare() {
    return cudaFuncSetAttribute(prefill_intra_fast_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                int(1024 + fs::BYTES)) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

kda_status launch_intra_fast(const PrefillParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                             const CUtensorMap &mv, const CUtensorMap &ma, dim3 grid, cudaStream_t s) {
    const ProfScope prof(KDA_KERNEL_PREFILL_INTRA, s);
    prefill_intra_fast_kernel<<<grid, fs::NT, 1024 + fs::BYTES, s>>>(p, mq, mk, mv, ma);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace pf
}  // namespace kda
