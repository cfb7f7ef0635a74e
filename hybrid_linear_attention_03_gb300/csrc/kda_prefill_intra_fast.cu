// kda_prefill_intra_fast.cu -- the intra-chunk prefill kernel for bf16
// activations, one CTA (16 warps) per (chunk, head).
//
// "vLLM Kimi K3 지원", section "Fused Kernels 및 메타데이터 최적화", KDA Prefill
// bullet: prefill runs chunked (FlashKDA).  Per (chunk, head), with G_r the
// cumulative log decay per key channel and c the middle of its range over the
// chunk, E = exp(G - c), K~ = k^ E, Q~ = q^ E, K^ = k^ / E:
//   [A; P] = [K~; Q~] K^^T                  (A_rs times beta_r, s < r; P_rs, s <= r)
//   T = (I + A)^-1                           (blocked, CUDA cores, kept transposed)
//   W = (T diag(beta)) K~ diag(exp(c))       Ut^T = V^T (T diag(beta))^T
//   exp(G) . q = Q~ diag(exp(c))
// which is the generic kernel's arithmetic with W's factor exp(G) = E exp(c)
// split so that every operand is one of three images built once.
//
// Every image is built token-major, a thread holding 2 tokens x 8 channels
// in registers: conv + SiLU, the L2 norm (a 16-lane shuffle reduction over
// the head's channels), the decay factors and the bf16 hi / lo split all
// happen in registers, and each 16-byte chunk is stored once.  The products
// that need an image transposed read it MN-major (kda_sm100.cuh), so no
// column-wise pass over shared memory is needed.  The cumulative decay G is a
// per-warp prefix (one shuffle) plus a scan of the 16 warp totals.  Record
// images leave through shared-memory staging and TMA bulk stores.
//
// Phases (bar = CTA barrier):
//   TMA alpha, then q, k, then v | beta
//   G, E (registers) bar scan bar
//   k pass: K~, K^ images    q pass: Q~ image, exp(G) . q rows -> record   bar
//   warp 0: K^ image -> record (bulk), MMA [A; P]; all warps: v image
//   wait: A^T -> smem, P -> staging, T^T zeroed                         bar
//   diagonal 16 x 16 blocks of T (2 warps)                               bar
//   2 levels of off-diagonal blocks (32-blocks, 2 bar each); (T diag beta)^T image  bar
//   MMA W, Ut^T -> wait: W rows, Ut^T rows -> staging -> record (bulk)
// A chunk whose decay span exceeds kSafeSpanFast is appended to the fallback
// list and left to the generic kernel.
//
// Shared memory (bytes from a 1 KiB-aligned base), about 174 KiB, one CTA per SM:
//   RQ, RK, RA, RV  raw q, k (67 rows), alpha (64 rows), v (67 rows) tiles; RV
//                   later stages the P image
//   VIMG            v image hi / lo [64 s][128 j], over RQ / RK after the q pass
//   X               [K~; Q~] image hi / lo [128][128]; the rows of Q~ in its
//                   first K block later hold the (T diag beta)^T image; after
//                   the last MMA, the W and Ut^T staging
//   KB              K^ image hi / lo [64][128]; after MMA 1, A^T and T^T fp32 [64][64]
//   SCAN            warp totals of G; later the level products
//   SMALL           c, exp(c), G_0, beta, mbarriers
// Tensor memory (256 columns): [0, 64) [A; P], then [0, 128) W (lanes 0..63);
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
constexpr uint32_t SCAN = KB + 32768;
constexpr uint32_t SMALL = SCAN + 8192;
constexpr uint32_t CREF = SMALL + 512, EC = SMALL + 1024, G0 = SMALL + 1536, BETA = SMALL + 2048;  // [SMALL, +512) free
constexpr uint32_t BARS = SMALL + 2304, TBASE = BARS + 64;
constexpr uint32_t PPS = RV;            // P image staging (hi, lo at +8192) once the v pass has consumed raw v
constexpr uint32_t BYTES = SMALL + 2560;
static_assert(RK >= RQ + TILE && RA >= RK + TILE && RV >= RA + CH * D * 2 && X >= RV + TILE, "raw tiles overlap");
static_assert(VIMG_LO + 16384 <= RA, "the v image overlaps the alpha tile");
static_assert(X % 1024 == 0 && KB % 1024 == 0 && TB % 1024 == 0, "images need 1 KiB alignment");
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

// ln(alpha) of 8 packed bf16 values in a 16-byte register word: PTX's
// lg2.approx (absolute error about 2^-22 in log2) times ln 2 while the warp's
// valid values are all positive normals, else logf.  Over a chunk the decay
// sums 64 of these, so the error stays near 1e-5 in the exponent.
__device__ __forceinline__ void log_alpha8_u4(const uint4 u, int n_valid, float (&l)[8]) {
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
            float lg;
            asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(__uint_as_float(b << 16)));
            l[e] = lg * 0.6931471805599453f;
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

// The rest of a one-chunk sequence from a zero state, after the Ut^T product
// (TMEM [128, 192)); K^ is on its way back from the record into KB (bar_qk,
// phase 1), P's hi image is in the P staging, exp(G_last - c) in the G_0 slot.
//   U = Ut: the U^T hi/lo image -> X;  the gate tile -> RA (rows of 256 B)
//   O^T = U^T P^T (one product) -> TMEM [0, 64);  (K^^T U)^T = U^T K^ -> [64, 192)
//   S^T = (K^^T U)^T diag(exp(G_last - c)) -> the slot (and checkpoint slots)
//   out = w_n . O / sqrt(mean O^2 + eps) . sigmoid(gate), staged over the
//   gate tile, then stored row by row (rows past the sequence untouched)
struct SoloChunk {
    int32_t seq, row0, len, ck_begin, ck_count, slot;
};
__device__ __forceinline__ void solo_tail(const PrefillParams &p, unsigned char *sm, uint32_t sbase, uint32_t tm,
                                       const SoloChunk cm, int h, bool ok) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, cs = (warp >> 2) * 16, j = qd * 32 + lane;  // TMEM lane = value channel j
    uint64_t *bar_qk = reinterpret_cast<uint64_t *>(sm + fs::BARS) + 1;
    uint64_t *bar_m1 = reinterpret_cast<uint64_t *>(sm + fs::BARS) + 3;
    const float *elc = reinterpret_cast<const float *>(sm + fs::G0);
    float *red = reinterpret_cast<float *>(sm + fs::SCAN);  // [4 lane quarters][64 tokens], then rs [64]
    uint32_t *fail = reinterpret_cast<uint32_t *>(sm + fs::SCAN + 2048);
    const size_t HD = size_t(p.H) * D;
    // the gate tile: 64 rows x 256 bytes, two 16-byte pieces a thread, coalesced
    uint4 gl[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int idx = tid + q * fs::NT, r = idx >> 4, c16 = idx & 15;
        gl[q] = r < cm.len ? *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.gate) +
                                                             (size_t(cm.row0 + r) * HD + size_t(h) * D) + c16 * 8)
                           : make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid == 0) *fail = 0u;
    if (ok) {  // U^T row j, tokens cs .. cs + 15 -> the hi / lo image rows (K-major, K = token)
        float u[16];
        tmem_ld16(tm + (uint32_t(qd * 32) << 16) + 128 + cs, u);
        tmem_wait_ld();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = u[8 * hh + e];
            store_split(sm + fs::X, sm + fs::X + 16384, sw128_chunk(j, (cs >> 3) + hh, D), x);
        }
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int idx = tid + q * fs::NT;
        *reinterpret_cast<uint4 *>(sm + fs::RA + (idx >> 4) * 256 + (idx & 15) * 16) = gl[q];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && ok) {
        if (mbar_wait(bar_qk, 1, p.err)) {
            const Operand u_img{sbase + fs::X, sbase + fs::X + 16384, false, D * 128};
            const Operand pp_img{sbase + fs::PPS, sbase + fs::PPS + 8192, false, CH * 128};
            const Operand kh_img{sbase + fs::KB, sbase + fs::KB_LO, true, CH * 128};
            mma_split(tm, u_img, pp_img, CH, idesc_bf16_f32(128, CH), 1, false);
            mma_split(tm + 64, u_img, kh_img, CH, idesc_bf16_f32(128, D, false, true), 3, false);
            mma_commit(bar_m1);
        } else {
            *fail = 1u;
        }
    }
    ok = __syncthreads_and(ok) && *fail == 0u;
    ok = __syncthreads_and(ok && mbar_wait(bar_m1, 1, p.err));
    tc_fence_after();
    float o[16];
    if (ok) {
        // S^T row j, key channels 32 cb .. 32 cb + 31
        const int cb = warp >> 2;
        float sv[2][16];
        tmem_ld16(tm + (uint32_t(qd * 32) << 16) + 64 + 32 * cb, sv[0]);
        tmem_ld16(tm + (uint32_t(qd * 32) << 16) + 64 + 32 * cb + 16, sv[1]);
        tmem_ld16(tm + (uint32_t(qd * 32) << 16) + cs, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) sv[e >> 4][e & 15] *= elc[32 * cb + e];
        const size_t head = size_t(D) * D, off = size_t(h) * head + size_t(j) * D + 32 * cb;
        float *dst = p.states + size_t(cm.slot) * p.H * head + off;
#pragma unroll
        for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4 *>(dst + e) =
                make_float4(sv[e >> 4][e & 15], sv[e >> 4][(e & 15) + 1], sv[e >> 4][(e & 15) + 2], sv[e >> 4][(e & 15) + 3]);
        for (int k = 0; k < cm.ck_count; ++k) {  // checkpoints at this chunk's end
            float *cd = p.states + size_t(p.ckpts[cm.ck_begin + k].dst_slot) * p.H * head + off;
#pragma unroll
            for (int e = 0; e < 32; e += 4)
                *reinterpret_cast<float4 *>(cd + e) =
                    make_float4(sv[e >> 4][e & 15], sv[e >> 4][(e & 15) + 1], sv[e >> 4][(e & 15) + 2], sv[e >> 4][(e & 15) + 3]);
        }
        // per token, the sum of O^2 over the warp's 32 channels: add the lane
        // pairs l, l ^ 16, then a transpose-reduce over 16 lanes leaves token
        // cs + (lane mod 16)'s in lane
        float a[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            a[e] = o[e] * o[e];
            a[e] += __shfl_xor_sync(0xffffffffu, a[e], 16);
        }
#pragma unroll
        for (int wd = 8; wd >= 1; wd >>= 1) {
            const bool up = (lane & wd) != 0;
#pragma unroll
            for (int e = 0; e < wd; ++e) {
                const float send = up ? a[e] : a[e + wd];
                const float keep = up ? a[e + wd] : a[e];
                a[e] = keep + __shfl_xor_sync(0xffffffffu, send, wd);
            }
        }
        if (lane < 16) red[qd * CH + cs + lane] = a[0];
    }
    __syncthreads();
    if (ok && tid < CH)
        red[4 * CH + tid] = rsqrtf(((red[tid] + red[CH + tid]) + (red[2 * CH + tid] + red[3 * CH + tid])) * (1.0f / D) +
                                   p.eps_rms);
    __syncthreads();
    if (ok) {  // y over the gate tile, in place (one thread per (token, channel))
        const float wn = __bfloat162float(static_cast<const __nv_bfloat16 *>(p.norm_w)[j]);
        uint16_t *gs = reinterpret_cast<uint16_t *>(sm + fs::RA) + j;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int r = cs + e;
            const float gv = __uint_as_float(uint32_t(gs[r * D]) << 16);
            gs[r * D] = __bfloat16_as_ushort(__float2bfloat16_rn(wn * (o[e] * red[4 * CH + r]) * sigmoid_tanh(gv)));
        }
    }
    __syncthreads();
    if (ok) {  // rows of the output, a warp per row, 8 bytes a lane
        for (int r = warp; r < cm.len; r += fs::NT / 32)
            *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(p.out) + (size_t(cm.row0 + r) * HD + size_t(h) * D) +
                                       lane * 4) = *reinterpret_cast<const uint2 *>(sm + fs::RA + r * 256 + lane * 8);
    }
    if (tid == 0) p.solo[size_t(cm.seq) * p.H + h] = ok ? 1 : 0;
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tm, 256);
}

// kSolo: the variant that also finishes one-chunk sequences from a zero
// state (p.solo set); the other has no such path (its code would slow the
// main path by about 2 %) and is launched for calls without them.
template <bool kSolo>
__global__ void __launch_bounds__(fs::NT, 1) prefill_intra_fast_kernel(const PrefillParams p,
                                                                    const __grid_constant__ CUtensorMap tm_q,
                                                                    const __grid_constant__ CUtensorMap tm_k,
                                                                    const __grid_constant__ CUtensorMap tm_v,
                                                                    const __grid_constant__ CUtensorMap tm_a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1 KiB-aligned base, kept a shared-memory pointer (offset, not an integer round trip)
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float *cref = reinterpret_cast<float *>(sm + fs::CREF);
    float *ec = reinterpret_cast<float *>(sm + fs::EC);
    float *g0s = reinterpret_cast<float *>(sm + fs::G0);
    float *beta = reinterpret_cast<float *>(sm + fs::BETA);
    uint64_t *bar_a_ld = reinterpret_cast<uint64_t *>(sm + fs::BARS);  // alpha tile
    uint64_t *bar_qk = bar_a_ld + 1, *bar_v = bar_a_ld + 2;          // q, k tiles; v tile
    uint64_t *bar_m1 = bar_a_ld + 3, *bar_m2 = bar_a_ld + 4;  // MMA groups
    uint32_t *tbase = reinterpret_cast<uint32_t *>(sm + fs::TBASE);
    float *scan = reinterpret_cast<float *>(sm + fs::SCAN);
    float *At = reinterpret_cast<float *>(sm + fs::AT);   // At[s * 64 + r] = A_rs
    float *Tt = reinterpret_cast<float *>(sm + fs::TT);   // Tt[s * 64 + r] = T_rs
    float *XS = reinterpret_cast<float *>(sm + fs::SCAN);        // level 1: [2][16 j][16 i]
    float *X2t = reinterpret_cast<float *>(sm + fs::SCAN + 2048);  // level 2: [32 j][32 i]
    const int g = p.chunk_base + blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // The tiles: alpha first (the decay pass needs it alone), then q, k, v
    // with the 3-row conv halo.  Inside one sequence (host-built tables) the
    // chunk's first row follows from g, so they are requested before the
    // chunk's fields arrive; otherwise as soon as those are here.
    auto load_tiles = [&](int row0) {
        for (int b = 0; b < 5; ++b) mbar_init(bar_a_ld + b, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(bar_a_ld, uint32_t(CH * D * 2));
        tma_load_3d(sm + fs::RA, &tm_a, bar_a_ld, 0, h, row0);
        mbar_arrive_expect_tx(bar_qk, 2 * fs::TILE);
        tma_load_3d(sm + fs::RK, &tm_k, bar_qk, 0, h, row0 - HALO);
        tma_load_3d(sm + fs::RQ, &tm_q, bar_qk, 0, h, row0 - HALO);
        mbar_arrive_expect_tx(bar_v, fs::TILE);
        tma_load_3d(sm + fs::RV, &tm_v, bar_v, 0, h, row0 - HALO);
    };
    const bool row_rule = p.row0_base != kNoRowBase;
    if (row_rule && tid == 0) load_tiles(p.row0_base + CH * g);
    const ChunkMeta cm = p.chunks[g];
    // warp 1 takes the tensor memory while the chunk's fields are on their
    // way (without a row rule, warp 0's lane 0 issues the tile loads as soon
    // as they are here)
    if (warp == 1) tmem_alloc(tbase, 256);
    if (cm.len <= 0) {  // a padding entry of a device-built table: no chunk here
        if (row_rule && tid == 0) {  // (host-built tables have none; no copy may land after the CTA is gone)
            mbar_wait(bar_a_ld, 0, p.err);
            mbar_wait(bar_qk, 0, p.err);
            mbar_wait(bar_v, 0, p.err);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == 1) tmem_dealloc(*tbase, 256);
        return;
    }
    const SeqMeta sq = p.seqs[cm.seq];
    char *rec = rec_ptr(p, g, h);
    // a one-chunk sequence from a zero state: U = Ut, so this CTA also forms
    // O = P U and the end state itself and the chain skips the sequence
    const bool solo = kSolo && sq.n_chunks == 1 && !sq.has_init;
    const uint32_t sbase = smem_u32(sm);
    if (!row_rule && tid == 0) load_tiles(cm.row0);
    // the head's conv taps (3 streams x 1 KiB, 24 lines) into L1 now: each
    // conv pass starts with every warp reading them, and consecutive CTAs on
    // an SM belong to other heads
    if (tid >= 64 && tid < 64 + 24)
        prefetch_l1(static_cast<const __nv_bfloat16 *>(p.conv_w) +
                    (size_t((tid - 64) >> 3) * p.H * D + size_t(h) * D) * 4 + ((tid - 64) & 7) * 64);
    // beta of the chunk's tokens: loaded now, stored to shared memory after
    // the decay pass (first read by the A drain), so the load is off the setup path
    const float beta_ld = tid < CH && tid < cm.len
                              ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p.beta)[size_t(cm.row0 + tid) * p.H + h])
                              : 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase;
    bool ok = __syncthreads_and(mbar_wait(bar_a_ld, 0, p.err));

    // This thread's unit: tokens r0, r0 + 1 (pair pr) x channels ch0 .. ch0 + 7.
    // A warp holds pairs 2 warp (lanes 0-15) and 2 warp + 1 (lanes 16-31).
    const int pr = tid >> 4, cb = tid & 15, r0 = 2 * pr, ch0 = 8 * cb;
    const __nv_bfloat16 *tail =
        sq.has_init ? static_cast<const __nv_bfloat16 *>(p.tails) + size_t(sq.slot) * 3 * p.n_ch + size_t(h) * D : nullptr;

    // ---- G = cumulative log decay, E = exp(G - c) --------------------------
    float gA[8], gB[8];
    {
        const uint4 a0 = lds16(sm + fs::RA + r0 * (D * 2) + ch0 * 2), a1 = lds16(sm + fs::RA + (r0 + 1) * (D * 2) + ch0 * 2);
        float l0[8], l1[8];
        log_alpha8_u4(a0, r0 < cm.len ? 8 : 0, l0);
        log_alpha8_u4(a1, r0 + 1 < cm.len ? 8 : 0, l1);
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
    if (tid < CH) beta[tid] = beta_ld;
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
        const float elc = expf(run - c);
        at<float>(rec, Rec::ELC)[tid] = elc;
        g0s[tid] = elc;  // kept for a one-chunk sequence's end state (G_0 is read above)
        wide = gfirst - run > kSafeSpanFast;
    }
    const bool exact = __syncthreads_or(wide) != 0;
    if (!ok || exact) {
        // a chunk this kernel cannot take: the generic kernel's list gets it
        if (ok && tid == 0) p.fb_list[atomicAdd(p.fb_count, 1u)] = uint32_t(g) * uint32_t(p.H) + uint32_t(h);
        if (kSolo && solo && tid == 0) p.solo[size_t(cm.seq) * p.H + h] = 0;  // the chain takes it
        mbar_wait(bar_qk, 0, p.err);  // no copy may land after the CTA is gone
        mbar_wait(bar_v, 0, p.err);
        tc_fence_before();
        __syncthreads();
        if (warp == 1) tmem_dealloc(tm, 256);
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
    ok = __syncthreads_and(mbar_wait(bar_qk, 0, p.err));

    // ---- k pass: K~ = k^ E (X rows r), K^ = k^ / E (KB rows r) ---------------
    if (ok) {
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
    // ---- q pass: Q~ = q^ E (X rows 64 + r); exp(G) . q = Q~ exp(c) -> record
    // WQ rows 64 + r, hi half only (it feeds only the output); a warp's lanes
    // cover whole rows, so the stores are coalesced
    if (ok) {
        float y[2][8], e_c[8];
        ld8(ec + ch0, e_c);
        conv_pair(sm + fs::RQ, p, 0, h, ch0, r0, cm.pos0, cm.len, tail, y);
        l2_pair(y, p.eps_l2);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = y[q][e] * (q ? E1[e] : E0[e]);
            store_split(sm + fs::X, sm + fs::X_LO, sw128_chunk(CH + r0 + q, cb, 2 * CH), x);
            uint4 vh, vl;
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] *= e_c[e];
            split8(x, vh, vl);
            *reinterpret_cast<uint4 *>(rec + Rec::WQ_HI + sw128_chunk(CH + r0 + q, cb, 2 * CH)) = vh;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) {
        // warp 0 issues the MMAs (the issuing lane stalls while the tensor core
        // works through them); the other warps form v meanwhile
        if (lane == 0 && ok) {
            // K^ image -> record (the chain's operand)
            bulk_store(rec + Rec::KH_HI, sm + fs::KB, 16384);
            bulk_store(rec + Rec::KH_LO, sm + fs::KB_LO, 16384);
            bulk_commit();
            const Operand xop{sbase + fs::X, sbase + fs::X_LO, false, 2 * CH * 128};
            const Operand kbop{sbase + fs::KB, sbase + fs::KB_LO, false, CH * 128};
            mma_split(tm, xop, kbop, D, idesc_bf16_f32(128, CH), 3, false);  // [A; P] (unmasked)
            mma_commit(bar_m1);
        }
        __syncwarp();
    }
    // ---- v pass under the MMAs: v image over the raw q, k tiles, one unit
    // (2 tokens x 8 channels) a thread; warp 0 takes its units once its lane
    // 0 has issued the MMAs (a second round for 32 units on the other warps
    // cost more than that wait)
    bool okv = mbar_wait(bar_v, 0, p.err);
    if (okv) {
        const int vpr = tid >> 4, vcb = tid & 15;
        float y[2][8];
        conv_pair(sm + fs::RV, p, 2, h, 8 * vcb, 2 * vpr, cm.pos0, cm.len, tail, y);
#pragma unroll
        for (int q = 0; q < 2; ++q) store_split(sm + fs::VIMG, sm + fs::VIMG_LO, sw128_chunk(2 * vpr + q, vcb, CH), y[q]);
    }
    okv = okv && mbar_wait(bar_m1, 0, p.err);
    if (tid == 0) bulk_wait_read();  // KB becomes A^T and T^T below
    ok = __syncthreads_and(ok && okv);
    tc_fence_after();
    const int qd = warp & 3, cs = (warp >> 2) * 16;  // TMEM lane quarter, 16-column slice
    if (ok) {
        // ---- A^T (s < r, times beta_r) -> smem; P (s <= r) -> staging (RV) -----
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
            for (int hh = 0; hh < 2; ++hh) {  // P feeds only the output: hi half
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = (cs + 8 * hh + e <= r) ? v[8 * hh + e] : 0.f;
                uint4 vh, vl;
                split8(x, vh, vl);
                *reinterpret_cast<uint4 *>(sm + fs::PPS + sw128_chunk(r, (cs >> 3) + hh, CH)) = vh;
            }
        }
        // T^T starts at zero: the blocks above the diagonal stay zero
        for (int e = tid; e < CH * CH / 4; e += fs::NT) reinterpret_cast<float4 *>(Tt)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        bulk_store(rec + Rec::PP_HI, sm + fs::PPS, 8192);
        bulk_commit();
    }
    if (ok && warp < 2) {
        // ---- diagonal 16 x 16 blocks of T by forward substitution: lane =
        // column c of block b, the column in registers -> T^T row 16 b + c
        const int b = tid >> 4, c = tid & 15, b16 = 16 * b;
        float tc[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = (r == c) ? 1.f : 0.f;
#pragma unroll
            for (int k = 0; k < r; ++k) acc = fmaf(-At[(b16 + k) * CH + b16 + r], tc[k], acc);
            tc[r] = acc;
        }
        float *dst = Tt + (b16 + c) * CH + b16;
#pragma unroll
        for (int r4 = 0; r4 < 16; r4 += 4)
            *reinterpret_cast<float4 *>(dst + r4) = make_float4(tc[r4], tc[r4 + 1], tc[r4 + 2], tc[r4 + 3]);
    }
    __syncthreads();
    if (ok) {
        // The level products are bound by shared-memory wavefronts: the operand
        // shared by a warp's lanes comes 4 k at a time as one 16-byte load.
        // ---- level 1: T_ab = -T_aa A_ab T_bb for (a, b) = (1, 0), (3, 2) ------
        {
            const int blk = tid >> 8, j = (tid >> 4) & 15, i = tid & 15;
            const int a16 = 16 * (2 * blk + 1), b16 = a16 - 16;
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < 16; k += 4) {
                const float4 tq = *reinterpret_cast<const float4 *>(Tt + (b16 + j) * CH + b16 + k);
                acc = fmaf(At[(b16 + k) * CH + a16 + i], tq.x, acc);
                acc = fmaf(At[(b16 + k + 1) * CH + a16 + i], tq.y, acc);
                acc = fmaf(At[(b16 + k + 2) * CH + a16 + i], tq.z, acc);
                acc = fmaf(At[(b16 + k + 3) * CH + a16 + i], tq.w, acc);
            }
            XS[blk * 256 + j * 16 + i] = acc;
            __syncthreads();
            float t = 0.f;
#pragma unroll
            for (int k = 0; k < 16; k += 4) {
                const float4 xq = *reinterpret_cast<const float4 *>(XS + blk * 256 + j * 16 + k);
                t = fmaf(Tt[(a16 + k) * CH + a16 + i], xq.x, t);
                t = fmaf(Tt[(a16 + k + 1) * CH + a16 + i], xq.y, t);
                t = fmaf(Tt[(a16 + k + 2) * CH + a16 + i], xq.z, t);
                t = fmaf(Tt[(a16 + k + 3) * CH + a16 + i], xq.w, t);
            }
            Tt[(b16 + j) * CH + a16 + i] = -t;
        }
        __syncthreads();
        // ---- level 2: T_21 = -T_22 A_21 T_11 on 32 x 32 blocks -----------------
        {
            const int i = lane, j0 = 2 * warp;
            float x0 = 0.f, x1 = 0.f;
            // T_11 is lower triangular: T_k,j0 and T_k,j0+1 vanish for k < j0
            // (the terms from j0 rounded down to a multiple of 4 add zeros)
            for (int k = j0 & ~3; k < 32; k += 4) {
                const float4 ta = *reinterpret_cast<const float4 *>(Tt + j0 * CH + k);
                const float4 tb = *reinterpret_cast<const float4 *>(Tt + (j0 + 1) * CH + k);
                const float a0 = At[k * CH + 32 + i], a1 = At[(k + 1) * CH + 32 + i];
                const float a2 = At[(k + 2) * CH + 32 + i], a3 = At[(k + 3) * CH + 32 + i];
                x0 = fmaf(a0, ta.x, x0); x1 = fmaf(a0, tb.x, x1);
                x0 = fmaf(a1, ta.y, x0); x1 = fmaf(a1, tb.y, x1);
                x0 = fmaf(a2, ta.z, x0); x1 = fmaf(a2, tb.z, x1);
                x0 = fmaf(a3, ta.w, x0); x1 = fmaf(a3, tb.w, x1);
            }
            X2t[j0 * 32 + i] = x0;
            X2t[(j0 + 1) * 32 + i] = x1;
            __syncthreads();
            float t0 = 0.f, t1 = 0.f;
#pragma unroll 2
            for (int k = 0; k < 32; k += 4) {
                const float4 xa = *reinterpret_cast<const float4 *>(X2t + j0 * 32 + k);
                const float4 xb = *reinterpret_cast<const float4 *>(X2t + (j0 + 1) * 32 + k);
                const float v0 = Tt[(32 + k) * CH + 32 + i], v1 = Tt[(33 + k) * CH + 32 + i];
                const float v2 = Tt[(34 + k) * CH + 32 + i], v3 = Tt[(35 + k) * CH + 32 + i];
                t0 = fmaf(v0, xa.x, t0); t1 = fmaf(v0, xb.x, t1);
                t0 = fmaf(v1, xa.y, t0); t1 = fmaf(v1, xb.y, t1);
                t0 = fmaf(v2, xa.z, t0); t1 = fmaf(v2, xb.z, t1);
                t0 = fmaf(v3, xa.w, t0); t1 = fmaf(v3, xb.w, t1);
            }
            Tt[j0 * CH + 32 + i] = -t0;
            Tt[(j0 + 1) * CH + 32 + i] = -t1;
        }
        __syncthreads();
        // ---- (T diag beta)^T image: row s holds beta_s T_rs for r = 0..63,
        // MMA 2's B operand read MN-major; over Q~'s first K block
        {
            const int s_ = tid >> 3, c = tid & 7;
            float t8[8], x[8];
            ld8(Tt + s_ * CH + 8 * c, t8);
            const float bs = beta[s_];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = t8[e] * bs;
            store_split(sm + fs::TB, sm + fs::TB_LO, sw128_chunk(s_, c, CH), x);
        }
    }
    if (tid == 0) bulk_wait_read();  // the staged P image is read before X is staged over
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0 && lane == 0 && ok) {
        // W diag(exp(-c)) = (T diag beta) K~: A = (T diag beta) read MN-major
        // with a zero block stride, so its second 64-row block re-reads the
        // first and TMEM lanes 64..127 hold W again (all 16 warps drain it);
        // B = K~ read MN-major.  Ut^T = V^T (T diag beta)^T: V and
        // (T diag beta)^T read MN-major.
        const Operand tba{sbase + fs::TB, sbase + fs::TB_LO, true, CH * 128};
        const Operand tba2{sbase + fs::TB, sbase + fs::TB_LO, true, 0};
        const Operand kt{sbase + fs::X, sbase + fs::X_LO, true, 2 * CH * 128};
        const Operand vt{sbase + fs::VIMG, sbase + fs::VIMG_LO, true, CH * 128};
        mma_split(tm, tba2, kt, CH, idesc_bf16_f32(128, D, true, true), 3, false);
        mma_split(tm + 128, vt, tba, CH, idesc_bf16_f32(128, CH, true, true), 3, false);
        mma_commit(bar_m2);
        if (solo) {  // K^ back from the record into KB (A^T and T^T are done with)
            bulk_wait();
            mbar_arrive_expect_tx(bar_qk, 32768);
            bulk_load(sm + fs::KB, rec + Rec::KH_HI, 32768, bar_qk);
        }
    }
    ok = __syncthreads_and(ok && mbar_wait(bar_m2, 0, p.err));
    tc_fence_after();
    if (kSolo && solo) {
        solo_tail(p, sm, sbase, tm, SoloChunk{cm.seq, cm.row0, cm.len, cm.ck_begin, cm.ck_count, sq.slot}, h, ok);
        return;
    }
    // ---- Ut^T row i -> staging in X_LO, on its way out while W is drained --
    if (ok) {
        const int i = qd * 32 + lane;
        float u[16];
        tmem_ld16(tm + (uint32_t(qd * 32) << 16) + 128 + cs, u);
        tmem_wait_ld();
        unsigned char *ut = sm + fs::X_LO + i * (CH * 4);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4 *>(ut + (ut_chunk(i, (cs >> 2) + q) << 4)) =
                make_float4(u[4 * q], u[4 * q + 1], u[4 * q + 2], u[4 * q + 3]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0 && ok) {
        bulk_store(rec + Rec::UT, sm + fs::X_LO, 32768);
        bulk_commit();
    }
    // ---- W row r (times exp(c_i)) -> staging in X ---------------------------
    if (ok) {  // W: token r in TMEM lanes r and 64 + r; 16 of the 128 key channels per warp
        const int r = (qd & 1) * 32 + lane, cw = (warp >> 2) * 32 + (qd >> 1) * 16;
        float w[16];
        tmem_ld16(tm + (uint32_t(qd * 32) << 16) + cw, w);
        tmem_wait_ld();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x[8], e_c[8];
            ld8(ec + cw + 8 * hh, e_c);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = w[8 * hh + e] * e_c[e];
            store_split(sm + fs::X, sm + fs::X + 16384, sw128_chunk(r, (cw >> 3) + hh, CH), x);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        // W rows 0..63 of each 64-wide K block of the WQ images
        bulk_store(rec + Rec::WQ_HI, sm + fs::X, 8192);
        bulk_store(rec + Rec::WQ_HI + 16384, sm + fs::X + 8192, 8192);
        bulk_store(rec + Rec::WQ_LO, sm + fs::X + 16384, 8192);
        bulk_store(rec + Rec::WQ_LO + 16384, sm + fs::X + 24576, 8192);
        bulk_commit();
        bulk_wait_read();  // shared memory stays until the copies have read it
    }
    if (warp == 1) tmem_dealloc(tm, 256);
}

}  // namespace

kda_status intra_fast_prepare() {
    const int bytes = int(1024 + fs::BYTES);
    return cudaFuncSetAttribute(prefill_intra_fast_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) ==
                       cudaSuccess &&
                   cudaFuncSetAttribute(prefill_intra_fast_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        bytes) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

kda_status launch_intra_fast(const PrefillParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                             const CUtensorMap &mv, const CUtensorMap &ma, dim3 grid, cudaStream_t s) {
    const ProfScope prof(KDA_KERNEL_PREFILL_INTRA, s);
    if (p.solo)
        prefill_intra_fast_kernel<true><<<grid, fs::NT, 1024 + fs::BYTES, s>>>(p, mq, mk, mv, ma);
    else
        prefill_intra_fast_kernel<false><<<grid, fs::NT, 1024 + fs::BYTES, s>>>(p, mq, mk, mv, ma);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace pf
}  // namespace kda
