// kda_prefill.cu -- chunked KDA prefill (WY / UT form) on TMA + tcgen05,
// d_k = d_v = 128, chunk C = 64.
//
// "vLLM Kimi K3 지원", section "Fused Kernels 및 메타데이터 최적화", KDA Prefill
// bullet: prefill runs chunked (FlashKDA).  Within a chunk of C tokens with
// cumulative log decay G_r = sum_{s<=r} log alpha_s (per key channel), the
// recurrence re-associates exactly into
//   A_rs = beta_r sum_i k_ri k_si exp(G_ri - G_si)  (s < r),  T = (I + A)^-1
//   W = T diag(beta) (exp(G) . K),    Ut = T diag(beta) V
//   P_rs = sum_i q_ri k_si exp(G_ri - G_si)  (s <= r)
// and, carried over chunks with the state S (d_k x d_v):
//   U = Ut - W S,   O = (exp(G) . Q) S + P U,
//   S <- Diag(exp(G_last)) S + sum_s (exp(G_last - G_s) . k_s) U_s^T.
// exp(G_r - G_s) is split around a per-channel reference c_i (the middle of
// the chunk's log-decay range): k_r exp(G_r - c) times k_s exp(c - G_s).
// Both factors stay in fp32 range while a channel's decay span over the chunk
// is at most 160; a chunk beyond that computes A and P with exact
// per-element exponentials instead.
//
// Every product that feeds the state runs on the tensor cores as three bf16
// MMAs (x = hi + lo with hi = bf16(x), lo = bf16(x - hi): hi*hi + hi*lo +
// lo*hi, fp32 accumulation in TMEM), which keeps about 16 mantissa bits.  All
// MMAs are M = 128 (the chunk-pair trick and transposed products below), with
// operands in the 128-byte-swizzle K-major layout (kda_sm100.cuh).
//
// Kernels (per window of chunks: intra on the caller's stream, then the
// window's chain on a high-priority side stream and its out on a third, so
// the chain and the norm of one window overlap intra of the next; the tails
// run on the caller's stream after the join):
//   meta   (device-built tables only, one CTA): sequence, chunk and
//          checkpoint tables from device arrays.
//   intra  (chunk, head): TMA loads the raw q, k, v, alpha tiles (with the
//          3-token conv halo); conv + SiLU, L2 of q and k, G, beta in shared
//          memory; [K exp(G-c); Q exp(G-c)] x (K exp(c-G))^T -> A, P (one
//          M=128 MMA); T = (I + A)^-1 on CUDA cores; W^T and Ut^T as M=128
//          MMAs; writes the chain's operand images.
//   chain  (sequence, head): sequential over chunks; S^T (fp32) lives in
//          TMEM; (W S)^T, (Q S)^T, (K^T U)^T and (P U)^T are MMAs; the next
//          chunk's operand images stream in by TMA bulk copies while the
//          current chunk computes; interval checkpoints; end state -> slot.
//   out    (chunk, head): gated RMSNorm of O -> out.
//   tails  checkpoint tails, then end tails -> slots.
#include "kda_internal.h"
#include "kda_sm100.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

namespace kda {

namespace {

using namespace sm100;

constexpr int D = 128;   // channels per head (d_k = d_v)
constexpr int CH = 64;   // chunk length
constexpr int HALO = 3;  // previous raw inputs the width-4 conv needs
constexpr float kLogAlphaMin = -100.0f;  // log(alpha) floor: alpha below e^-100 acts as e^-100
constexpr float kSafeSpan = 160.0f;      // max per-channel log-decay span for the split exponent
constexpr int kMaxWindows = 8;           // chunk windows overlapped across the streams
constexpr int kMinWindowChunks = 32;     // smallest window worth a separate chain launch

struct SeqMeta {
    int32_t row0, len, slot, has_init, chunk0, n_chunks;
};
struct ChunkMeta {
    int32_t seq, row0, len, pos0, ck_begin, ck_count;
};
struct CkptMeta {
    int32_t seq, token_pos, dst_slot, pad;
};

// Per (chunk, head) workspace record (bytes).  "img" = bf16 operand image in
// the 128-byte-swizzle K-major layout, [rows][K].
struct Rec {
    // [W; exp(G) . q]: one 128-row image [r | 64 + r][128 i] (W rows 0..63, Q rows 64..127)
    static constexpr size_t WQ_HI = 0;
    static constexpr size_t WQ_LO = WQ_HI + 32768;
    // [(exp(G_last - G) . k)^T; P]: one 192-row image [i | 128 + r][64] (K^T rows 0..127, P rows 128..191)
    static constexpr size_t KP_HI = WQ_LO + 32768;
    static constexpr size_t KP_LO = KP_HI + 24576;
    static constexpr size_t P_OFF = 16384;           // P rows start 16 KiB into a KP image
    static constexpr size_t GAM = KP_LO + 24576;     // fp32 [128] exp(G_last)
    static constexpr size_t UT = GAM + 1024;         // fp32 [64 r][128 j]  Ut
    static constexpr size_t OO = UT + 32768;         // fp32 [64 r][128 j]  O (pre-norm)
    static constexpr size_t BYTES = OO + 32768;
    static constexpr uint32_t B1_BYTES = uint32_t(KP_HI - WQ_HI);  // [W; Q] images
    static constexpr uint32_t B2_BYTES = uint32_t(UT - KP_HI);     // [K^T; P] images + gamma
};
static_assert(Rec::BYTES % 1024 == 0, "record keeps 1 KiB alignment");

struct PrefillParams {
    const SeqMeta *seqs;
    const ChunkMeta *chunks;
    const CkptMeta *ckpts;
    char *rec;  // [n_chunks][H] records
    float *states;
    void *tails;
    uint32_t *err;
    const void *q, *k, *v, *alpha, *beta, *gate;
    void *out;
    const void *conv_w, *norm_w;
    int32_t H, n_ch, n_seqs, n_chunks, n_ckpts;
    int32_t chunk_base;      // intra, out: global index of blockIdx.x == 0
    int32_t win_lo, win_hi;  // chain: global chunk range of this launch
    float eps_l2, eps_rms;
};

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }
// PTX's approximate 2^x and 1/x (flush-to-zero; relative errors of a few
// 1e-7 and about 1 ulp).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// sigma(x) = 1 / (1 + e^-x), with e^-x = 2^(-x log2 e): 0 for x below about
// -88, where 2^(-x log2 e) is +inf.
__device__ __forceinline__ float sigmoid_fast(float x) {
    return rcp_approx(1.0f + ex2_approx(-x * 1.4426950408889634f));
}

__device__ __forceinline__ char *rec_ptr(const PrefillParams &p, int g, int h) {
    return p.rec + (size_t(g) * p.H + h) * Rec::BYTES;
}

template <typename T>
__device__ __forceinline__ T *at(char *base, size_t off) {
    return reinterpret_cast<T *>(base + off);
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

__device__ __forceinline__ void ld8(const float *p, float (&x)[8]) {  // p 16-byte aligned
    const float4 a = ld4(p), b = ld4(p + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <typename Act>
__device__ __forceinline__ float4 act4(const Act *p);
// 4 values -> 4 consecutive activations (16-byte fp32 or 8-byte bf16 store, round to nearest even)
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
}
template <>
__device__ __forceinline__ float4 act4<float>(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
template <>
__device__ __forceinline__ float4 act4<__nv_bfloat16>(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}

// ln(alpha) of 8 values.  A positive normal bf16 value is 2^e (1 + m/128):
// its log is e ln 2 + ln(1 + m/128), the second term from a 128-entry table
// (lnm).  When any lane of the warp holds a zero, subnormal, negative or
// non-finite value among its n_valid leading ones (the tokens before the
// segment end, so that nothing past it can change a token's bits), the
// whole warp takes logf for these 8 (a warp-uniform
// branch keeps logf out of the common path); fp32 values always use logf.
__device__ __forceinline__ void log_alpha8(const float (&a)[8], const float *, int, float (&l)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) l[e] = logf(a[e]);
}
__device__ __forceinline__ void log_alpha8(const __nv_bfloat16 (&a)[8], const float *lnm, int n_valid, float (&l)[8]) {
    bool normal = true;  // only the n_valid leading values (tokens before the segment end) decide the path
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t b = __bfloat16_as_ushort(a[e]), ex = (b >> 7) & 0xFFu;
        normal = normal && (e >= n_valid || ((b >> 15) == 0 && ex != 0 && ex != 0xFFu));
    }
    if (__all_sync(0xffffffffu, normal)) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t b = __bfloat16_as_ushort(a[e]);
            l[e] = fmaf(float(int((b >> 7) & 0xFFu) - 127), 0.6931471805599453f, lnm[b & 0x7Fu]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) l[e] = logf(__bfloat162float(a[e]));
    }
}

// ======================================================= conv helper ====
// Causal conv (width 4, last tap on the current token) + SiLU of one channel
// c for tokens t0 .. t0 + n - 1 of the chunk (n a multiple of 8), from a raw
// tile whose row t + 3 is token t (row stride D).  Tile rows before the
// segment start come from the slot's conv tail (tail_c points at channel c's
// oldest tap; rows n_ch apart) when the sequence resumes, else they are zero.
// Tokens past the segment end give 0.  out[t * D + c] receives token t.  Raw
// values are loaded 8 tokens at a time so their latencies overlap.
template <typename Act>
__device__ __forceinline__ void conv_silu_channel(const Act *__restrict__ tile, int c, float4 w, int t0, int n, int pos0,
                                                  int len, const Act *__restrict__ tail_c, int n_ch,
                                                  float *__restrict__ out) {
    float x[3];
#pragma unroll
    for (int j = 0; j < HALO; ++j) {
        const int row = t0 + j, pos = pos0 - HALO + row;
        x[j] = pos >= 0 ? to_f32(tile[row * D + c]) : (tail_c ? to_f32(tail_c[size_t(HALO + pos) * n_ch]) : 0.f);
    }
    float x0 = x[0], x1 = x[1], x2 = x[2];
#pragma unroll 1
    for (int tb = t0; tb < t0 + n; tb += 8) {
        float xs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) xs[e] = to_f32(tile[(tb + e + HALO) * D + c]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float acc = w.x * x0;
            acc = fmaf(w.y, x1, acc);
            acc = fmaf(w.z, x2, acc);
            acc = fmaf(w.w, xs[e], acc);
            out[(tb + e) * D + c] = tb + e < len ? acc * sigmoid_fast(acc) : 0.f;
            x0 = x1;
            x1 = x2;
            x2 = xs[e];
        }
    }
}

// The same for exactly 32 tokens t0 .. t0 + 31, into registers (fully
// unrolled so y stays in registers): y[e] is token t0 + e.
template <typename Act>
__device__ __forceinline__ void conv_silu_regs32(const Act *__restrict__ tile, int c, float4 w, int t0, int pos0, int len,
                                                 const Act *__restrict__ tail_c, int n_ch, float (&y)[32]) {
    float x[3];
#pragma unroll
    for (int j = 0; j < HALO; ++j) {
        const int row = t0 + j, pos = pos0 - HALO + row;
        x[j] = pos >= 0 ? to_f32(tile[row * D + c]) : (tail_c ? to_f32(tail_c[size_t(HALO + pos) * n_ch]) : 0.f);
    }
    float x0 = x[0], x1 = x[1], x2 = x[2];
#pragma unroll
    for (int b = 0; b < 32; b += 8) {
        float xs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) xs[e] = to_f32(tile[(t0 + b + e + HALO) * D + c]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float acc = w.x * x0;
            acc = fmaf(w.y, x1, acc);
            acc = fmaf(w.z, x2, acc);
            acc = fmaf(w.w, xs[e], acc);
            y[b + e] = t0 + b + e < len ? acc * sigmoid_fast(acc) : 0.f;
            x0 = x1;
            x1 = x2;
            x2 = xs[e];
        }
    }
}

// Transpose-reduce of 32 values per lane across the warp: afterwards v[0] of
// lane l is the sum over all 32 lanes of their value l.  At the stage with
// xor-offset O the upper lane of each pair keeps the upper half of its
// values, so the live values halve every stage (31 shuffles in all).
template <int CNT, int O>
__device__ __forceinline__ void lane_transpose_sum(float *v, int lane) {
    if constexpr (O > 0) {
        constexpr int HALF = CNT / 2;
        const bool upper = (lane & O) != 0;
#pragma unroll
        for (int m = 0; m < HALF; ++m) {
            const float send = upper ? v[m] : v[m + HALF];
            const float keep = upper ? v[m + HALF] : v[m];
            v[m] = keep + __shfl_xor_sync(0xffffffffu, send, O);
        }
        lane_transpose_sum<HALF, O / 2>(v, lane);
    }
}

// Conv taps of channel c of stream s (0 q, 1 k, 2 v) of head h.
template <typename Act>
__device__ __forceinline__ float4 conv_taps(const PrefillParams &p, int s, int h, int c) {
    return act4(static_cast<const Act *>(p.conv_w) + size_t(s * p.H * D + h * D + c) * 4);
}

// ============================================================== intra ====
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

// Fills `rows` x (8 * chunks_per_row) elements of an image pair with f(row, k0, out8),
// storing 16-byte chunks at their swizzled offsets (shared or global memory).
// Row-major unit order (consecutive threads walk one row's chunks) suits f
// reading rows of a [row][K] array; chunk-major order (consecutive threads
// take consecutive rows of one chunk) suits f reading columns of a [K][row]
// array without shared-memory bank conflicts.  The loop is kept rolled: this
// kernel runs each phase once per CTA, so compact code (fewer instruction
// cache misses) measured faster than unrolled, batched loads.
template <bool kChunkMajor = false, typename F>
__device__ __forceinline__ void build_image(unsigned char *hi, unsigned char *lo, int rows, int chunks_per_row,
                                            int tid, int nthreads, F f, int row0 = 0, int total_rows = 0) {
    if (total_rows == 0) total_rows = rows;
#pragma unroll 1
    for (int u = tid; u < rows * chunks_per_row; u += nthreads) {
        const int r = kChunkMajor ? u % rows : u / chunks_per_row;
        const int c = kChunkMajor ? u / rows : u - r * chunks_per_row;
        float x[8];
        f(r, 8 * c, x);
        uint4 vh, vl;
        split8(x, vh, vl);
        const uint32_t off = sw128_chunk(row0 + r, c, total_rows);
        *reinterpret_cast<uint4 *>(hi + off) = vh;
        *reinterpret_cast<uint4 *>(lo + off) = vl;
    }
}

// Issues the three bf16 MMAs of a split product: D (+)= Ahi Bhi + Ahi Blo + Alo Bhi.
__device__ __forceinline__ void mma3(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo, int a_rows,
                                     int b_rows, int k_total, uint32_t idesc, bool accumulate) {
    const int ksteps = k_total / 16;
    for (int part = 0; part < 3; ++part) {
        const uint32_t a = part == 2 ? a_lo : a_hi;
        const uint32_t b = part == 1 ? b_lo : b_hi;
        for (int ks = 0; ks < ksteps; ++ks) {
            const int kb = ks >> 2, kk = ks & 3;
            const uint64_t ad = sdesc_sw128(a + uint32_t(kb * a_rows * 128 + kk * 32));
            const uint64_t bd = sdesc_sw128(b + uint32_t(kb * b_rows * 128 + kk * 32));
            mma_bf16(d, ad, bd, idesc, (accumulate || part > 0 || ks > 0) ? 1u : 0u);
        }
    }
}

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

// One CTA (16 warps) per (chunk, head).  TMA brings the raw q, k, v tiles of
// the chunk's 64 tokens plus the 3 before them (the conv halo) and the alpha
// tile; the kernel forms G, q^, k^ (conv + SiLU + L2) and v (conv + SiLU) in
// shared memory, so every operand build reads shared memory.  Images the
// chain needs that involve no MMA (exp(G).q, (exp(G_last - G).k)^T, P) go
// straight to the record from registers; the W image is staged and
// bulk-stored.
template <typename Act>
__global__ void __launch_bounds__(is::NT, 1) prefill_intra_kernel(const PrefillParams p,
                                                               const __grid_constant__ CUtensorMap tm_q,
                                                               const __grid_constant__ CUtensorMap tm_k,
                                                               const __grid_constant__ CUtensorMap tm_v,
                                                               const __grid_constant__ CUtensorMap tm_a) {
    static_assert(is::map_ok<Act>(), "intra shared-memory map overlaps");
    static_assert(CH % (16 * is::QW) == 0 && is::NT >= 4 * D, "drain split / thread roles need these");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
    const int g = p.chunk_base + blockIdx.x, h = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const ChunkMeta cm = p.chunks[g];
    if (cm.len <= 0) return;  // a padding entry of a device-built table: no chunk here
    const SeqMeta sq = p.seqs[cm.seq];
    char *rec = rec_ptr(p, g, h);
    const uint32_t sbase = smem_u32(sm);
    if (tid == 0) {
        *flag = 0;
        mbar_init(bar_ld, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_v, 1);
        fence_mbar_init();
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
    if (warp == 0) tmem_alloc(tbase, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase;
    bool ok = __syncthreads_and(mbar_wait(bar_ld, 0, p.err));
    uint32_t mma_phase = 0;
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
        if (g0 - gl > kSafeSpan) atomicOr(flag, 1);
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
        // read once: X rows r and 64 + r = k^ E and q^ E, Kb row r = k^ / E, and
        // the chain's exp(G) . q image row 64 + r = q^ (E e^c) in the record.
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
    // chain images that need no MMA: exp(G) . q (rows r; above when !exact) and
    // (exp(G_last - G) . k)^T (rows i)
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
        build_image<true>(reinterpret_cast<unsigned char *>(rec + Rec::KP_HI),
                    reinterpret_cast<unsigned char *>(rec + Rec::KP_LO), D, 8, tid, is::NT,
                    [&](int i, int r0, float(&x)[8]) {
                        const float gl = GGs[(CH - 1) * D + i], l = elc[i];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float gv = GGs[(r0 + e) * D + i];
                            x[e] = KHs[(r0 + e) * D + i] * (exact ? expf(gl - gv) : l * rcp_approx(gv));
                        }
                    });
    }
    __syncthreads();
    // ---- A (s < r, times beta_r) -> fp32 smem, stored transposed (A[s * CH + r]
    // = A_rs), P (s <= r) -> record images
    float *A = reinterpret_cast<float *>(sm + is::A_F32);
    unsigned char *phi = reinterpret_cast<unsigned char *>(rec + Rec::KP_HI + Rec::P_OFF);
    unsigned char *plo = reinterpret_cast<unsigned char *>(rec + Rec::KP_LO + Rec::P_OFF);
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
        vok = (is::v_early<Act>() || ok) ? mbar_wait(bar_v, 0, p.err) : false;
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
    __syncthreads();  // v is consumed: the W image staging takes its place
    tc_fence_after();
    if (tid == 0 && ok) {
        const uint32_t id = idesc_bf16_f32(128, CH);
        mma3(tm + 64, sbase + is::AK_HI, sbase + is::AK_LO, sbase + is::T_HI, sbase + is::T_LO, D, CH, CH, id, false);
        mma3(tm + 128, sbase + is::AV_HI, sbase + is::AV_LO, sbase + is::T_HI, sbase + is::T_LO, D, CH, CH, id, false);
        mma_commit(bar_mma);
    }
    ok = __syncthreads_and(ok && mbar_wait(bar_mma, mma_phase, p.err));
    tc_fence_after();
    unsigned char *whi = sm + is::IN0, *wlo = sm + is::IN0 + 16384;
    const int i = (warp & 3) * 32 + lane;  // TMEM lane: key channel i (W^T row) / value channel j (Ut^T row)
    const int cbase = (warp >> 2) * (CH / is::QW);
    if (ok) {
        float *UT = at<float>(rec, Rec::UT) + i;  // column j = i of Ut [r][j]
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
            for (int e = 0; e < 16; ++e) UT[(c0 + e) * D] = u[e];  // coalesced across the warp
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
        bulk_wait_read();  // shared memory may go; the write lands before the kernel completes
    }
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 256);
}

// ============================================================== chain ====
namespace cs {  // chain shared-memory map
constexpr uint32_t A1_HI = 0, A1_LO = 32768;             // S^T images [128 j][128 i]
constexpr uint32_t B1 = 65536;                            // [W; Q] hi/lo images (64 KiB)
constexpr uint32_t WQ_HI = B1, WQ_LO = B1 + 32768;
constexpr uint32_t B2 = 131072;                           // [K^T; P] hi/lo images, gamma
constexpr uint32_t KP_HI = B2, KP_LO = B2 + 24576, GAM = B2 + 49152;
constexpr uint32_t A2_HI = 181248, A2_LO = 181248 + 16384;  // U^T images [128 j][64 r]
constexpr uint32_t GCUR = A2_LO + 16384;                   // gamma of the current chunk
constexpr uint32_t BARS = GCUR + 512;
constexpr uint32_t BYTES = BARS + 512;
}  // namespace cs
static_assert(cs::B2 + Rec::B2_BYTES <= cs::A2_HI, "chain smem map overlaps");

// TMEM columns: [(W S)^T | (Q S)^T] [0,128), [(K^T U)^T | (P U)^T] [128,320), S^T [320,448)
__global__ void __launch_bounds__(256) prefill_chain_kernel(const PrefillParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar_b1 = reinterpret_cast<uint64_t *>(sm + cs::BARS);
    uint64_t *bar_b2 = bar_b1 + 1, *bar_m1 = bar_b1 + 2, *bar_m2 = bar_b1 + 3;
    uint32_t *tbase = reinterpret_cast<uint32_t *>(bar_b1 + 4);
    float *gcur = reinterpret_cast<float *>(sm + cs::GCUR);
    // 8 warps: warps w and w + 4 share TMEM lanes 32*(w % 4) .. +31 (value
    // channel j = TMEM lane) and split every row's columns between them.
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = (warp & 3) * 32 + lane, half = warp >> 2;
    const int h = blockIdx.x % p.H, n = blockIdx.x / p.H;
    const SeqMeta sq = p.seqs[n];
    if (sq.slot < 0) return;  // disabled by the device metadata check: leave every slot alone
    // The chunks of this sequence inside the launch's window [win_lo, win_hi).
    // A sequence with no chunks is settled by the window that starts at 0.
    const int c_lo = max(sq.chunk0, p.win_lo) - sq.chunk0;
    const int c_hi = min(sq.chunk0 + sq.n_chunks, p.win_hi) - sq.chunk0;
    if (c_hi <= c_lo && !(sq.n_chunks == 0 && p.win_lo == 0)) return;
    // A window that continues a sequence reads the state the previous window
    // left in the slot.
    const bool load_state = sq.has_init || c_lo > 0;
    const size_t head_elems = size_t(D) * D;
    float *slot_state = p.states + size_t(sq.slot) * p.H * head_elems + size_t(h) * head_elems;  // S^T [j][i]
    const uint32_t sbase = smem_u32(sm);
    if (tid == 0) {
        for (int b = 0; b < 4; ++b) mbar_init(bar_b1 + b, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tbase, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase, tl = tm + (uint32_t((warp & 3) * 32) << 16);
    if (tid == 0 && c_hi > c_lo) {
        const char *r0 = rec_ptr(p, sq.chunk0 + c_lo, h);
        mbar_arrive_expect_tx(bar_b1, Rec::B1_BYTES);
        bulk_load(sm + cs::B1, r0 + Rec::WQ_HI, Rec::B1_BYTES, bar_b1);
        mbar_arrive_expect_tx(bar_b2, Rec::B2_BYTES);
        bulk_load(sm + cs::B2, r0 + Rec::KP_HI, Rec::B2_BYTES, bar_b2);
    }
    const int sc0 = half * 64;  // this thread's 64 columns of the S^T row
    // S^T row j: fp32 into TMEM, hi/lo into the A1 images
    for (int c0 = sc0; c0 < sc0 + 64; c0 += 16) {
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; e += 4) {
            const float4 x = load_state ? ld4(slot_state + size_t(j) * D + c0 + e) : make_float4(0.f, 0.f, 0.f, 0.f);
            v[e] = x.x; v[e + 1] = x.y; v[e + 2] = x.z; v[e + 3] = x.w;
        }
        tmem_st16(tl + 320 + c0, v);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = v[8 * hh + e];
            uint4 vh, vl;
            split8(x, vh, vl);
            const uint32_t off = sw128_chunk(j, (c0 >> 3) + hh, D);
            *reinterpret_cast<uint4 *>(sm + cs::A1_HI + off) = vh;
            *reinterpret_cast<uint4 *>(sm + cs::A1_LO + off) = vl;
        }
    }
    tmem_wait_st();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    bool ok = true;
    const uint32_t id128 = idesc_bf16_f32(128, 2 * CH), id192 = idesc_bf16_f32(128, D + CH);
    const int uc0 = half * 32;  // this thread's 32 columns of the U / O rows
    for (int c = c_lo; c < c_hi && ok; ++c) {
        const int g = sq.chunk0 + c;
        char *rec = rec_ptr(p, g, h);
        const uint32_t par = uint32_t((c - c_lo) & 1);
        ok = __syncthreads_and(mbar_wait(bar_b1, par, p.err));
        if (!ok) break;
        if (tid == 0) {
            tc_fence_after();
            mma3(tm + 0, sbase + cs::A1_HI, sbase + cs::A1_LO, sbase + cs::WQ_HI, sbase + cs::WQ_LO, D, 2 * CH, D,
                 id128, false);
            mma_commit(bar_m1);
        }
        // Ut row entries (r = uc0 .. uc0 + 31, column j) while the MMAs run
        float ut[32];
        const float *UTg = reinterpret_cast<const float *>(rec + Rec::UT) + j;  // column j, coalesced
#pragma unroll
        for (int e = 0; e < 32; ++e) ut[e] = UTg[(uc0 + e) * D];
        ok = __syncthreads_and(mbar_wait(bar_m1, par, p.err));
        if (!ok) break;
        tc_fence_after();
        if (tid == 0 && c + 1 < c_hi) {  // W and Q images are consumed: stream in the next chunk's
            mbar_arrive_expect_tx(bar_b1, Rec::B1_BYTES);
            bulk_load(sm + cs::B1, rec_ptr(p, g + 1, h) + Rec::WQ_HI, Rec::B1_BYTES, bar_b1);
        }
        // U^T row j = Ut^T - (W S)^T  -> hi/lo images (this thread's 32 columns)
        {
            float v[2][16];
            tmem_ld16(tl + uc0, v[0]);
            tmem_ld16(tl + uc0 + 16, v[1]);
            tmem_wait_ld();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = ut[8 * cc + e] - v[cc >> 1][8 * (cc & 1) + e];
                uint4 vh, vl;
                split8(x, vh, vl);
                const uint32_t off = sw128_chunk(j, (uc0 >> 3) + cc, D);
                *reinterpret_cast<uint4 *>(sm + cs::A2_HI + off) = vh;
                *reinterpret_cast<uint4 *>(sm + cs::A2_LO + off) = vl;
            }
        }
        ok = __syncthreads_and(mbar_wait(bar_b2, par, p.err));
        if (!ok) break;
        if (half == 0) gcur[j] = reinterpret_cast<const float *>(sm + cs::GAM)[j];
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            mma3(tm + 128, sbase + cs::A2_HI, sbase + cs::A2_LO, sbase + cs::KP_HI, sbase + cs::KP_LO, D, D + CH, CH,
                 id192, false);
            mma_commit(bar_m2);
        }
        ok = __syncthreads_and(mbar_wait(bar_m2, par, p.err));
        if (!ok) break;
        tc_fence_after();
        if (tid == 0 && c + 1 < c_hi) {  // K^T, P images and gamma consumed
            mbar_arrive_expect_tx(bar_b2, Rec::B2_BYTES);
            bulk_load(sm + cs::B2, rec_ptr(p, g + 1, h) + Rec::KP_HI, Rec::B2_BYTES, bar_b2);
        }
        // O column j (rows uc0 .. uc0 + 31) = (Q S)^T + (P U)^T -> record, coalesced across the warp
        {
            float* O = reinterpret_cast<float *>(rec + Rec::OO);
            float v[2][16], w2[2][16];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                tmem_ld16(tl + 64 + uc0 + 16 * q, v[q]);
                tmem_ld16(tl + 256 + uc0 + 16 * q, w2[q]);
            }
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int e = 0; e < 16; ++e) O[(uc0 + 16 * q + e) * D + j] = v[q][e] + w2[q][e];
        }
        // S^T row j <- gamma . S^T row j + (K^T U)^T row j; refresh the A1 images
        const ChunkMeta cm = p.chunks[g];
        for (int c0 = sc0; c0 < sc0 + 64; c0 += 32) {  // 32 columns per TMEM round trip
            float s[2][16], ds[2][16];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                tmem_ld16(tl + 320 + c0 + 16 * q, s[q]);
                tmem_ld16(tl + 128 + c0 + 16 * q, ds[q]);
            }
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 2; ++q) {
#pragma unroll
                for (int e = 0; e < 16; ++e) s[q][e] = fmaf(gcur[c0 + 16 * q + e], s[q][e], ds[q][e]);
                tmem_st16(tl + 320 + c0 + 16 * q, s[q]);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = s[q][8 * hh + e];
                    uint4 vh, vl;
                    split8(x, vh, vl);
                    const uint32_t off = sw128_chunk(j, ((c0 + 16 * q) >> 3) + hh, D);
                    *reinterpret_cast<uint4 *>(sm + cs::A1_HI + off) = vh;
                    *reinterpret_cast<uint4 *>(sm + cs::A1_LO + off) = vl;
                }
                for (int k = 0; k < cm.ck_count; ++k) {
                    const CkptMeta ck = p.ckpts[cm.ck_begin + k];
                    float *dst = p.states + size_t(ck.dst_slot) * p.H * head_elems + size_t(h) * head_elems +
                                 size_t(j) * D + c0 + 16 * q;
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4 *>(dst + e) = make_float4(s[q][e], s[q][e + 1], s[q][e + 2], s[q][e + 3]);
                }
            }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    }
    // end state S^T row j (this thread's 64 columns) -> slot
    if (ok) {
        for (int c0 = sc0; c0 < sc0 + 64; c0 += 16) {
            float s[16];
            tmem_ld16(tl + 320 + c0, s);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4 *>(slot_state + size_t(j) * D + c0 + e) = make_float4(s[e], s[e + 1], s[e + 2], s[e + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// ================================================================ out ====
template <typename Act>
__global__ void __launch_bounds__(128) prefill_out_kernel(const PrefillParams p) {
    const int g = p.chunk_base + blockIdx.x, h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ChunkMeta cm = p.chunks[g];
    const float *O = reinterpret_cast<const float *>(rec_ptr(p, g, h) + Rec::OO);
    const Act *gate = static_cast<const Act *>(p.gate);
    Act *out = static_cast<Act *>(p.out);
    const size_t HD = size_t(p.H) * D;
    const Act *nwp = static_cast<const Act *>(p.norm_w) + lane * 4;  // no alignment asked of norm_w
    const float4 wn = make_float4(to_f32(nwp[0]), to_f32(nwp[1]), to_f32(nwp[2]), to_f32(nwp[3]));
    for (int t = warp; t < cm.len; t += 4) {
        const size_t base = size_t(cm.row0 + t) * HD + size_t(h) * D + lane * 4;
        const float4 o4 = ld4(O + t * D + lane * 4);
        const float4 g4 = act4(gate + base);
        float ss = fmaf(o4.x, o4.x, fmaf(o4.y, o4.y, fmaf(o4.z, o4.z, o4.w * o4.w)));
        for (int s = 16; s; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
        const float r = rsqrtf(ss * (1.0f / D) + p.eps_rms);
        store4(out + base, make_float4(wn.x * (o4.x * r) * sigmoid_f(g4.x), wn.y * (o4.y * r) * sigmoid_f(g4.y),
                                       wn.z * (o4.z * r) * sigmoid_f(g4.z), wn.w * (o4.w * r) * sigmoid_f(g4.w)));
    }
}

// ============================================================== tails ====
// Conv tail after `pos` tokens of a segment: raw inputs at pos-3 .. pos-1
// (before the segment: the slot's old tail, or zeros for a new sequence).
// One block per checkpoint request when ckpt_pass, else per sequence; the
// request pass runs first because it may read a sequence slot's old tail.
template <typename Act>
__global__ void __launch_bounds__(256) prefill_tails_kernel(const PrefillParams p, int ckpt_pass) {
    const int item = blockIdx.x;
    int seq, pos, dst;
    if (ckpt_pass) {
        const CkptMeta ck = p.ckpts[item];
        seq = ck.seq;
        pos = ck.token_pos;
        dst = ck.dst_slot;
    } else {
        seq = item;
        pos = p.seqs[item].len;
        dst = p.seqs[item].slot;
    }
    if (seq < 0 || dst < 0 || p.seqs[seq].slot < 0) return;  // disabled by the device metadata check
    const SeqMeta sq = p.seqs[seq];
    const Act *old = static_cast<const Act *>(p.tails) + size_t(sq.slot) * 3 * p.n_ch;
    Act *nt = static_cast<Act *>(p.tails) + size_t(dst) * 3 * p.n_ch;
    const int HD = p.H * D;
    for (int ch = threadIdx.x; ch < p.n_ch; ch += blockDim.x) {
        const int s = ch / HD, rem = ch - s * HD;
        const Act *src = static_cast<const Act *>(s == 0 ? p.q : (s == 1 ? p.k : p.v));
        Act x[3];
        for (int jj = 0; jj < 3; ++jj) {
            const int q = pos - 3 + jj;
            if (q >= 0) x[jj] = src[size_t(sq.row0 + q) * HD + rem];
            else x[jj] = sq.has_init ? old[size_t(3 + q) * p.n_ch + ch] : from_f32<Act>(0.f);
        }
        for (int jj = 0; jj < 3; ++jj) nt[size_t(jj) * p.n_ch + ch] = x[jj];
    }
}

// ============================================================ metadata ===
// Builds the sequence, chunk and checkpoint tables on the device from device
// arrays (one CTA), with the host builder's rules: cu_seqlens from 0 and
// non-decreasing within max_tokens; sequence slots and request slots in range
// and all distinct; a request's position in (0, len] and a multiple of the
// chunk or the sequence end.  Chunks beyond the real count (the grid is sized
// from bounds) get len 0.  On any violation the error word gets
// KDA_DEVERR_SLOT_RANGE / KDA_DEVERR_META and every table entry disables its
// item (slot -1, no chunks, no requests), so the call changes nothing.
struct MetaArgs {
    const int32_t *cu;
    const int32_t *slots;
    const uint8_t *has_init;
    const kda_ckpt_req *reqs;
    int32_t N, n_reqs, max_tokens, max_chunks, num_slots;
    SeqMeta *seqs;
    ChunkMeta *chunks;
    CkptMeta *ckpts;
    uint32_t *used;  // ceil(num_slots / 32) words of scratch
    uint32_t *err;
};
constexpr int kMetaThreads = 1024;

__device__ __forceinline__ bool mark_slot(uint32_t *used, int slot) {  // true if already marked
    const uint32_t bit = 1u << (slot & 31);
    return (atomicOr(used + (slot >> 5), bit) & bit) != 0;
}

// (seq, pos) of sorted request r is after (s, t)
__device__ __forceinline__ bool req_after(const CkptMeta &c, int s, int t) {
    return c.seq > s || (c.seq == s && c.token_pos > t);
}

__global__ void __launch_bounds__(kMetaThreads) prefill_meta_kernel(const MetaArgs a) {
    __shared__ int bad_meta, bad_slot, carry;
    __shared__ int scan[kMetaThreads];
    const int tid = threadIdx.x;
    if (tid == 0) {
        bad_meta = 0;
        bad_slot = 0;
        carry = 0;
    }
    for (int i = tid; i < (a.num_slots + 31) / 32; i += kMetaThreads) a.used[i] = 0u;
    __syncthreads();
    for (int s = tid; s < a.N; s += kMetaThreads) {
        const int lo = a.cu[s], hi = a.cu[s + 1], sl = a.slots[s];
        if ((s == 0 && lo != 0) || hi < lo || hi > a.max_tokens) bad_meta = 1;
        if (sl < 0 || sl >= a.num_slots) bad_slot = 1;
        else if (mark_slot(a.used, sl)) bad_meta = 1;
    }
    __syncthreads();  // sequence slots are marked before request slots are checked against them
    for (int r = tid; r < a.n_reqs; r += kMetaThreads) {
        const kda_ckpt_req q = a.reqs[r];
        if (q.seq < 0 || q.seq >= a.N) {
            bad_meta = 1;
            continue;
        }
        const int len = a.cu[q.seq + 1] - a.cu[q.seq];
        if (q.token_pos <= 0 || q.token_pos > len || (q.token_pos != len && q.token_pos % CH != 0)) bad_meta = 1;
        if (q.dst_slot < 0 || q.dst_slot >= a.num_slots) bad_slot = 1;
        else if (mark_slot(a.used, q.dst_slot)) bad_meta = 1;
    }
    __syncthreads();
    const bool ok = !bad_meta && !bad_slot;
    if (tid == 0 && !ok) atomicOr(a.err, (bad_slot ? KDA_DEVERR_SLOT_RANGE : 0u) | (bad_meta ? KDA_DEVERR_META : 0u));
    // sequences: chunk counts, exclusive prefix -> first chunk
    for (int base = 0; base < a.N; base += kMetaThreads) {
        const int s = base + tid;
        const int len = (ok && s < a.N) ? a.cu[s + 1] - a.cu[s] : 0;
        const int nch = (len + CH - 1) / CH;
        scan[tid] = nch;
        __syncthreads();
        for (int off = 1; off < kMetaThreads; off <<= 1) {
            const int v = tid >= off ? scan[tid - off] : 0;
            __syncthreads();
            scan[tid] += v;
            __syncthreads();
        }
        if (s < a.N) {
            SeqMeta m = {0, 0, -1, 0, 0, 0};
            if (ok) m = {a.cu[s], len, a.slots[s], a.has_init[s] ? 1 : 0, carry + scan[tid] - nch, nch};
            a.seqs[s] = m;
        }
        __syncthreads();
        if (tid == kMetaThreads - 1) carry += scan[tid];
        __syncthreads();
    }
    const int total_chunks = carry;
    // requests sorted by (sequence, position): rank of each among all
    for (int r = tid; r < a.n_reqs; r += kMetaThreads) {
        const kda_ckpt_req q = a.reqs[r];
        int rank = 0;
        for (int k = 0; k < a.n_reqs; ++k) {
            const kda_ckpt_req o = a.reqs[k];
            rank += (o.seq < q.seq || (o.seq == q.seq && (o.token_pos < q.token_pos || (o.token_pos == q.token_pos && k < r))))
                        ? 1 : 0;
        }
        CkptMeta c = {-1, 0, -1, 0};
        if (ok) c = {q.seq, q.token_pos, q.dst_slot, 0};
        a.ckpts[rank] = c;
    }
    __syncthreads();  // the tables above are read back below
    // chunks: owning sequence (the last one starting at or before g), rows, and its requests
    for (int g = tid; g < a.max_chunks; g += kMetaThreads) {
        ChunkMeta cm = {-1, 0, 0, 0, 0, 0};
        if (ok && g < total_chunks) {
            int lo = 0, hi = a.N - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (a.seqs[mid].chunk0 <= g) lo = mid;
                else hi = mid - 1;
            }
            const SeqMeta sq = a.seqs[lo];
            const int pos0 = (g - sq.chunk0) * CH, clen = min(CH, sq.len - pos0);
            // requests of this sequence at positions (pos0, pos0 + clen]: all at pos0 + clen
            int b = 0, e = a.n_reqs;
            while (b < e) {
                const int mid = (b + e) >> 1;
                if (req_after(a.ckpts[mid], lo, pos0)) e = mid;
                else b = mid + 1;
            }
            int f = b, e2 = a.n_reqs;
            while (f < e2) {
                const int mid = (f + e2) >> 1;
                if (req_after(a.ckpts[mid], lo, pos0 + clen)) e2 = mid;
                else f = mid + 1;
            }
            cm = {lo, sq.row0 + pos0, clen, pos0, b, f - b};
        }
        a.chunks[g] = cm;
    }
}

// ================================================================ host ===
size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
    size_t seqs, chunks, ckpts, rec, total;
};

WsLayout ws_layout(int N, long long n_chunks, long long n_reqs, int H);

// The device-built tables' workspace: ws_layout plus the slot bitmap the
// builder uses to find repeated slots (at the end).
struct WsLayoutDev {
    WsLayout L;
    size_t used, total;
};
WsLayoutDev ws_layout_dev(int N, long long max_chunks, long long n_reqs, int H, int num_slots) {
    WsLayoutDev d;
    d.L = ws_layout(N, max_chunks, n_reqs, H);
    d.used = align256(d.L.total);
    d.total = d.used + sizeof(uint32_t) * size_t((num_slots + 31) / 32);
    return d;
}

WsLayout ws_layout(int N, long long n_chunks, long long n_reqs, int H) {
    WsLayout L;
    L.seqs = 0;
    L.chunks = align256(L.seqs + sizeof(SeqMeta) * size_t(N));
    L.ckpts = align256(L.chunks + sizeof(ChunkMeta) * size_t(n_chunks));
    L.rec = (L.ckpts + sizeof(CkptMeta) * size_t(std::max<long long>(n_reqs, 1)) + 1023) / 1024 * 1024;
    L.total = L.rec + Rec::BYTES * size_t(n_chunks) * size_t(H);
    return L;
}

long long count_chunks(const int32_t *cu, int N) {
    long long n = 0;
    for (int s = 0; s < N; ++s) n += (cu[s + 1] - cu[s] + CH - 1) / CH;
    return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// Tensor map over a token-major [n_tok][H][128] activation tensor; the box
// is one head's 128 channels x `rows` tokens.
bool make_map(CUtensorMap *m, const void *base, int n_tok, int H, int esize, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(H), cuuint64_t(n_tok)};
    const cuuint64_t strides[2] = {cuuint64_t(D) * esize, cuuint64_t(H) * D * esize};
    const cuuint32_t box[3] = {cuuint32_t(D), 1u, cuuint32_t(rows)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = fn(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <typename K>
kda_status set_smem(K kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

template <typename Act>
constexpr size_t intra_smem() {
    return 1024 + is::BYTES<Act>();
}
constexpr size_t kChainSmem = 1024 + cs::BYTES;

// Per-device side streams (the chain's at the highest priority) and events
// for the windowed overlap of the chain and the gated norm with the per-chunk
// kernels.  Not memory: nothing here allocates device memory.
struct SideStream {
    cudaStream_t s = nullptr;  // chain (highest priority)
    cudaStream_t o = nullptr;  // gated norm of finished windows
    // [0, W): window w's intra done; [W, 2W): window w's chain done;
    // 2W: call start; 2W + 1, 2W + 2: chain / norm streams done
    cudaEvent_t ev[2 * kMaxWindows + 3] = {};
    bool ok = false;
};

SideStream *side_stream() {
    static SideStream per_dev[64];
    static std::once_flag once[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::call_once(once[dev], [dev] {
        SideStream &x = per_dev[dev];
        int lo = 0, hi = 0;
        if (cudaDeviceGetStreamPriorityRange(&lo, &hi) != cudaSuccess) return;
        if (cudaStreamCreateWithPriority(&x.s, cudaStreamNonBlocking, hi) != cudaSuccess) return;
        if (cudaStreamCreateWithPriority(&x.o, cudaStreamNonBlocking, lo) != cudaSuccess) return;
        for (auto &e : x.ev)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return;
        x.ok = true;
    });
    return per_dev[dev].ok ? &per_dev[dev] : nullptr;
}

template <typename Act>
kda_status launch_act(const PrefillParams &p0, const kda_io *io, int n_tok, int N, long long n_chunks, int n_reqs,
                      cudaStream_t stream) {
    kda_status st;
    if ((st = set_smem(prefill_intra_kernel<Act>, intra_smem<Act>())) != KDA_OK) return st;
    if ((st = set_smem(prefill_chain_kernel, kChainSmem)) != KDA_OK) return st;
    PrefillParams p = p0;
    CUtensorMap mq, mk, mv, ma;
    if (n_chunks > 0) {
        const int es = int(sizeof(Act));
        if (!make_map(&mq, io->q, n_tok, p.H, es, CH + HALO) || !make_map(&mk, io->k, n_tok, p.H, es, CH + HALO) ||
            !make_map(&mv, io->v, n_tok, p.H, es, CH + HALO) || !make_map(&ma, io->alpha, n_tok, p.H, es, CH))
            return KDA_ERR_CUDA;
    }
    // Windows of chunks: the chain of window w (one CTA per sequence and
    // head, on the side stream) and then the gated norm of its chunks run
    // while intra of window w + 1 fills the other SMs; events order each
    // chain launch after its window's records and the final join returns
    // everything to the caller's stream.
    // The side stream's events are shared by every caller of this device:
    // one call's record / wait sequence is enqueued as a whole.
    static std::mutex enqueue_mu;
    std::lock_guard<std::mutex> lock(enqueue_mu);
    SideStream *side = nullptr;
    int n_win = 1;
    if (n_chunks >= 2 * kMinWindowChunks) {
        side = side_stream();
        if (side) n_win = int(std::min<long long>(kMaxWindows, n_chunks / kMinWindowChunks));
    }
    const long long per = (n_chunks + n_win - 1) / n_win;
    cudaStream_t cs = side ? side->s : stream, os = side ? side->o : stream;
    constexpr int W = kMaxWindows;
    // An event call that fails after kernels are queued on the side streams:
    // join them to the caller's stream as far as the runtime still allows, so
    // nothing of this call runs after the caller's stream has moved past it
    // (the caller may free the workspace once it sees the error).
    auto fail = [&]() {
        if (side) {
            cudaEventRecord(side->ev[2 * W + 1], cs);
            cudaEventRecord(side->ev[2 * W + 2], os);
            cudaStreamWaitEvent(stream, side->ev[2 * W + 1], 0);
            cudaStreamWaitEvent(stream, side->ev[2 * W + 2], 0);
        }
        cudaGetLastError();
        return KDA_ERR_CUDA;
    };
    if (side) {  // the chain stream starts after everything already on the caller's stream
        if (cudaEventRecord(side->ev[2 * W], stream) != cudaSuccess ||
            cudaStreamWaitEvent(cs, side->ev[2 * W], 0) != cudaSuccess)
            return fail();
    }
    for (int w = 0; w < n_win; ++w) {
        const long long lo = std::min(n_chunks, w * per), hi = std::min(n_chunks, (w + 1) * per);
        if (hi > lo) {
            p.chunk_base = int(lo);
            const dim3 grid(unsigned(hi - lo), unsigned(p.H));
            const ProfScope prof(KDA_KERNEL_PREFILL_INTRA, stream);
            prefill_intra_kernel<Act><<<grid, is::NT, intra_smem<Act>(), stream>>>(p, mq, mk, mv, ma);
        }
        p.win_lo = int(lo);
        p.win_hi = (w + 1 == n_win) ? int(n_chunks) : int(hi);
        if (side) {
            if (cudaEventRecord(side->ev[w], stream) != cudaSuccess || cudaStreamWaitEvent(cs, side->ev[w], 0) != cudaSuccess)
                return fail();
        }
        {
            const ProfScope prof(KDA_KERNEL_PREFILL_CHAIN, cs);
            prefill_chain_kernel<<<unsigned(N) * p.H, 256, kChainSmem, cs>>>(p);
        }
        if (hi > lo) {  // gated norm of the window's chunks once their chain is done, off the chain's stream
            if (side) {
                if (cudaEventRecord(side->ev[W + w], cs) != cudaSuccess ||
                    cudaStreamWaitEvent(os, side->ev[W + w], 0) != cudaSuccess)
                    return fail();
            }
            PrefillParams po = p;
            po.chunk_base = int(lo);
            const ProfScope prof(KDA_KERNEL_PREFILL_OUT, os);
            prefill_out_kernel<Act><<<dim3(unsigned(hi - lo), unsigned(p.H)), 128, 0, os>>>(po);
        }
    }
    if (side) {
        if (cudaEventRecord(side->ev[2 * W + 1], cs) != cudaSuccess ||
            cudaEventRecord(side->ev[2 * W + 2], os) != cudaSuccess ||
            cudaStreamWaitEvent(stream, side->ev[2 * W + 1], 0) != cudaSuccess ||
            cudaStreamWaitEvent(stream, side->ev[2 * W + 2], 0) != cudaSuccess)
            return fail();
    }
    p.chunk_base = 0;
    {
        const ProfScope prof(KDA_KERNEL_PREFILL_TAILS, stream);
        if (n_reqs > 0) prefill_tails_kernel<Act><<<n_reqs, 256, 0, stream>>>(p, 1);
        prefill_tails_kernel<Act><<<N, 256, 0, stream>>>(p, 0);
    }
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

size_t prefill_workspace_bytes(const kda_pool *pool, const int32_t *cu_seqlens, int N, int chunk) {
    if (chunk != CH || pool->desc.d_k != D || pool->desc.d_v != D || N < 0) return 0;
    if (cu_seqlens[0] != 0) return 0;
    for (int s = 0; s < N; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return 0;
    // room for one checkpoint per chunk end and per sequence end, twice over
    const long long nc = count_chunks(cu_seqlens, N);
    return ws_layout(N, nc, 2 * (nc + N), pool->desc.num_heads).total;
}

// Launch parameters over the workspace's tables (written, or enqueued to be
// written, on the stream) and the kernels.  n_chunks sizes the grids; n_tok
// is the token extent of the activation arrays the tensor maps describe.
kda_status launch_tables(const kda_pool *pool, const kda_weights *w, const kda_io *io, char *ws, const WsLayout &L,
                         int N, int n_reqs, long long n_chunks, int n_tok, cudaStream_t stream) {
    PrefillParams p{};
    p.chunk_base = 0;
    p.win_lo = 0;
    p.win_hi = int(n_chunks);
    p.seqs = reinterpret_cast<const SeqMeta *>(ws + L.seqs);
    p.chunks = reinterpret_cast<const ChunkMeta *>(ws + L.chunks);
    p.ckpts = reinterpret_cast<const CkptMeta *>(ws + L.ckpts);
    p.rec = ws + L.rec;
    p.states = pool->states;
    p.tails = pool->tails;
    p.err = pool->err;
    p.q = io->q;
    p.k = io->k;
    p.v = io->v;
    p.alpha = io->alpha;
    p.beta = io->beta;
    p.gate = io->gate;
    p.out = io->out;
    p.conv_w = w->conv_w;
    p.norm_w = w->norm_w;
    p.H = pool->desc.num_heads;
    p.n_ch = pool->n_ch;
    p.n_seqs = N;
    p.n_chunks = int(n_chunks);
    p.n_ckpts = n_reqs;
    p.eps_l2 = w->eps_l2;
    p.eps_rms = w->eps_rms;
    if (pool->desc.act == KDA_BF16) return launch_act<__nv_bfloat16>(p, io, n_tok, N, n_chunks, n_reqs, stream);
    return launch_act<float>(p, io, n_tok, N, n_chunks, n_reqs, stream);
}

kda_status launch_prefill(const kda_pool *pool, const kda_weights *w, const kda_io *io, const int32_t *cu_seqlens,
                          const int32_t *slots, const uint8_t *has_initial_state, int N, int chunk,
                          const kda_ckpt_req *reqs, int n_reqs, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
    if (pool->desc.d_k != D || pool->desc.d_v != D || chunk != CH) return KDA_ERR_UNSUPPORTED;
    const int H = pool->desc.num_heads;
    const long long n_chunks = count_chunks(cu_seqlens, N);
    if (n_chunks > (1LL << 31) / std::max(H, 1)) return KDA_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(N, n_chunks, n_reqs, H);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % 256) != 0 || workspace_bytes < L.total)
        return KDA_ERR_WORKSPACE;
    // host metadata: sequences, chunks, checkpoint requests sorted by (seq, pos)
    std::vector<SeqMeta> seqs(static_cast<size_t>(N));
    std::vector<ChunkMeta> chunks;
    chunks.reserve(static_cast<size_t>(n_chunks));
    std::vector<CkptMeta> cks(static_cast<size_t>(n_reqs));
    for (int r = 0; r < n_reqs; ++r) cks[r] = {reqs[r].seq, reqs[r].token_pos, reqs[r].dst_slot, 0};
    std::sort(cks.begin(), cks.end(), [](const CkptMeta &a, const CkptMeta &b) {
        return a.seq != b.seq ? a.seq < b.seq : a.token_pos < b.token_pos;
    });
    size_t ck = 0;
    for (int s = 0; s < N; ++s) {
        const int len = cu_seqlens[s + 1] - cu_seqlens[s];
        const int nch = (len + CH - 1) / CH;
        seqs[s] = {cu_seqlens[s], len, slots[s], has_initial_state[s] ? 1 : 0, int(chunks.size()), nch};
        for (int c = 0; c < nch; ++c) {
            const int pos0 = c * CH, clen = std::min(CH, len - pos0);
            ChunkMeta cm = {s, cu_seqlens[s] + pos0, clen, pos0, int(ck), 0};
            while (ck < cks.size() && cks[ck].seq == s && cks[ck].token_pos <= pos0 + clen) {
                if (cks[ck].token_pos != pos0 + clen) return KDA_ERR_INVALID_ARG;
                ++cm.ck_count;
                ++ck;
            }
            chunks.push_back(cm);
        }
    }
    if (ck != cks.size()) return KDA_ERR_INVALID_ARG;
    char *ws = static_cast<char *>(workspace);
    {
        const ProfScope prof(KDA_KERNEL_PREFILL_META, stream);  // the host tables' copies to the device
        if (N > 0 && cudaMemcpyAsync(ws + L.seqs, seqs.data(), sizeof(SeqMeta) * seqs.size(),
                                     cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
        if (!chunks.empty() && cudaMemcpyAsync(ws + L.chunks, chunks.data(), sizeof(ChunkMeta) * chunks.size(),
                                               cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
        if (!cks.empty() && cudaMemcpyAsync(ws + L.ckpts, cks.data(), sizeof(CkptMeta) * cks.size(),
                                            cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    return launch_tables(pool, w, io, ws, L, N, n_reqs, n_chunks, cu_seqlens[N], stream);
}

size_t prefill_workspace_bytes_bound(const kda_pool *pool, int N, int max_tokens, int n_reqs, int chunk) {
    if (chunk != CH || pool->desc.d_k != D || pool->desc.d_v != D || N < 0 || max_tokens < 0 || n_reqs < 0) return 0;
    const long long mc = max_tokens / CH + N;
    return ws_layout_dev(N, mc, n_reqs, pool->desc.num_heads, pool->desc.num_slots).total;
}

kda_status launch_prefill_dev(const kda_pool *pool, const kda_weights *w, const kda_io *io, const int32_t *cu_seqlens,
                              const int32_t *slots, const uint8_t *has_initial_state, int N, int max_tokens,
                              int chunk, const kda_ckpt_req *reqs, int n_reqs, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
    if (pool->desc.d_k != D || pool->desc.d_v != D || chunk != CH) return KDA_ERR_UNSUPPORTED;
    const int H = pool->desc.num_heads;
    // every sequence adds at most one partial chunk to max_tokens / CH whole ones
    const long long max_chunks = max_tokens / CH + N;
    if (max_chunks > (1LL << 31) / std::max(H, 1)) return KDA_ERR_INVALID_ARG;
    const WsLayoutDev LD = ws_layout_dev(N, max_chunks, n_reqs, H, pool->desc.num_slots);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % 256) != 0 || workspace_bytes < LD.total)
        return KDA_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    MetaArgs a;
    a.cu = cu_seqlens;
    a.slots = slots;
    a.has_init = has_initial_state;
    a.reqs = reqs;
    a.N = N;
    a.n_reqs = n_reqs;
    a.max_tokens = max_tokens;
    a.max_chunks = int(max_chunks);
    a.num_slots = pool->desc.num_slots;
    a.seqs = reinterpret_cast<SeqMeta *>(ws + LD.L.seqs);
    a.chunks = reinterpret_cast<ChunkMeta *>(ws + LD.L.chunks);
    a.ckpts = reinterpret_cast<CkptMeta *>(ws + LD.L.ckpts);
    a.used = reinterpret_cast<uint32_t *>(ws + LD.used);
    a.err = pool->err;
    {
        const ProfScope prof(KDA_KERNEL_PREFILL_META, stream);
        prefill_meta_kernel<<<1, kMetaThreads, 0, stream>>>(a);
    }
    return launch_tables(pool, w, io, ws, LD.L, N, n_reqs, max_chunks, max_tokens, stream);
}

// ------------------------------------------------------ no-allocation entry --
// Fixed scratch for kda_prefill_chunked_noalloc: callers that cannot allocate
// device memory run the prefill in this array instead of a workspace of
// their own.  It lives in the module image, so every GPU that loads the
// library holds it until the process exits.  Host code must not use the
// array's name as a device address: the address comes from
// cudaGetSymbolAddress with the call's device current.  It is looked up on
// every call (a table lookup once the module is loaded), so a device reset
// that reloads the module at another address leaves no stale pointer behind;
// the first lookup on a device may load the module, which is why the first
// call should come before any stream capture.
static __device__ __align__(256) unsigned char g_prefill_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

kda_status launch_prefill_noalloc(const kda_pool *pool, const kda_weights *w, const kda_io *io,
                                  const int32_t *cu_seqlens, const int32_t *slots,
                                  const uint8_t *has_initial_state, int N, int chunk, const kda_ckpt_req *reqs,
                                  int n_reqs, cudaStream_t stream) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_prefill_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return KDA_ERR_CUDA;
    }
    // Every byte of the scratch is written before it is read, so nothing is
    // cleared; a call that needs more than the array returns KDA_ERR_WORKSPACE.
    return launch_prefill(pool, w, io, cu_seqlens, slots, has_initial_state, N, chunk, reqs, n_reqs, ptr,
                          KDA_NOALLOC_SCRATCH_BYTES, stream);
}

}  // namespace kda
