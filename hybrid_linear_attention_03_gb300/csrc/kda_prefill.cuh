// kda_prefill.cuh -- what the chunked-prefill translation units share: the
// chunk geometry, the host-built tables, the per (chunk, head) record that
// the intra-chunk kernels write and the chain reads, the launch parameters
// and the device helpers (conv, logarithms, operand images, split MMAs).
// Not part of the C ABI.
//
// The record of one (chunk, head) (bytes; "image" = bf16 operand tile in the
// 128-byte-swizzle layout of kda_sm100.cuh, hi = bf16(x), lo = bf16(x - hi)):
//   WQ   [W; exp(G) . q]: 128 token rows (W rows 0..63, exp(G) . q rows
//        64..127) x 128 key channels, K-major; the rows of exp(G) . q feed
//        only the output, so with bf16 outputs their lo half is not kept
//        (q_lo = 0) and the chain reads zeros there
//   KH   k^ exp(c - G) [64 tokens][128 key channels], token-major, read by
//        the chain MN-major; multiplied per channel by ELC it is
//        k^ exp(G_last - G)
//   PP   P [64 tokens r][64 tokens s], K-major: PP_HI; PP_LO only when q_lo
//   GAM  exp(G_last) per key channel;  ELC  exp(G_last - c) per key channel
//   UT   Ut^T fp32 [128 value channels][64 tokens]; in row j the 16-byte
//        chunk c (tokens 4c .. 4c + 3) sits at chunk position c ^ (j mod 16)
// 145 KiB in all.  O never reaches memory: the chain applies the gated norm
// to it and writes the layer output.
// Records live in a ring: chunk g, head h uses slot (g mod ring_chunks, h).
#pragma once

#include "kda_internal.h"
#include "kda_sm100.cuh"

#include <cudaTypedefs.h>

namespace kda {
namespace pf {

using namespace sm100;

constexpr int D = 128;   // channels per head (d_k = d_v)
constexpr int CH = 64;   // chunk length
constexpr int HALO = 3;  // previous raw inputs the width-4 conv needs
constexpr float kLogAlphaMin = -100.0f;  // log(alpha) floor: alpha below e^-100 acts as e^-100
// Largest per-channel log-decay span of a chunk that the split exponent
// exp(G_r - G_s) = exp(G_r - c) exp(c - G_s) handles.  The generic kernel
// keeps its products under 2^128 up to 160; the fast kernel also multiplies
// its exp(G - c) factors (up to e^60) by T in a 64-term sum, so it stops at
// 120 and hands wider chunks to the generic kernel.
constexpr float kSafeSpanGeneric = 160.0f;
constexpr float kSafeSpanFast = 120.0f;

struct SeqMeta {
    int32_t row0, len, slot, has_init, chunk0, n_chunks;
};
struct ChunkMeta {
    int32_t seq, row0, len, pos0, ck_begin, ck_count;
};
struct CkptMeta {
    int32_t seq, token_pos, dst_slot, pad;
};

struct Rec {
    static constexpr size_t WQ_HI = 0, WQ_LO = 32768;
    static constexpr size_t KH_HI = 65536, KH_LO = 81920;
    static constexpr size_t PP_HI = 98304;
    static constexpr size_t GAM = PP_HI + 8192, ELC = GAM + 512;
    static constexpr size_t PP_LO = GAM + 1024;
    static constexpr size_t UT = PP_LO + 8192;
    static constexpr size_t BYTES = UT + 32768;
    static constexpr uint32_t B1_BYTES = uint32_t(KH_HI - WQ_HI);     // WQ images
    static constexpr uint32_t B2_BYTES = uint32_t(UT - KH_HI);        // KH, PP hi, GAM, ELC, PP lo
    static constexpr uint32_t B2_BYTES_HI = uint32_t(PP_LO - KH_HI);  // the same without PP lo
};
static_assert(Rec::BYTES % 1024 == 0, "record keeps 1 KiB alignment");

struct PrefillParams {
    const SeqMeta *seqs;
    const ChunkMeta *chunks;
    const CkptMeta *ckpts;
    char *rec;  // the record ring: [ring_chunks][H] records
    float *states;
    void *tails;
    uint32_t *err;
    const void *q, *k, *v, *alpha, *beta, *gate;
    void *out;
    const void *conv_w, *norm_w;
    uint32_t *fb_count;      // chunk-heads the fast intra kernel hands to the generic one ...
    uint32_t *fb_list;       // ... as g * H + h
    uint8_t *solo;           // bf16: [n_seqs][H], 1 where the intra kernel finished a one-chunk
                             // sequence from a zero state itself (the chain skips it), else 0
    int32_t H, n_ch, n_seqs, n_chunks, n_ckpts;
    int32_t ring_chunks;     // chunks the record ring holds
    int32_t chunk_base;      // intra, out: global index of blockIdx.x == 0
    int32_t win_lo, win_hi;  // chain: global chunk range of this launch
    int32_t seq_base;        // chain: sequence of blockIdx.x / H == 0
    int32_t q_lo;            // the record keeps the lo halves of exp(G) . q and P (fp32 outputs)
    int32_t row0_base;       // intra: chunk g's first row is row0_base + C g (a window inside one
                             // sequence, host-built tables), or kNoRowBase
    float eps_l2, eps_rms;
};
constexpr int32_t kNoRowBase = -2147483647 - 1;

// Brings the cache line holding gsrc into this SM's L1.
__device__ __forceinline__ void prefetch_l1(const void *gsrc) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<uint64_t>(gsrc)) : "memory");
}

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
// sigma(x) = (1 + tanh(x / 2)) / 2 with PTX's approximate tanh (one
// operation; relative error about 2^-11): for bf16 results only.
// w . sigma(x) = hw + hw . tanh(x / 2) with hw = w / 2.
__device__ __forceinline__ float scaled_sigmoid_tanh(float x, float hw) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
    return fmaf(hw, t, hw);
}
__device__ __forceinline__ float sigmoid_tanh(float x) { return scaled_sigmoid_tanh(x, 0.5f); }

// Chunk position of tokens 4c .. 4c + 3 in row j of the record's Ut^T (the
// XOR spreads the rows a warp writes over all shared-memory banks).
__host__ __device__ __forceinline__ uint32_t ut_chunk(int j, int c) { return uint32_t(c ^ (j & 15)); }

__device__ __forceinline__ char *rec_ptr(const PrefillParams &p, int g, int h) {
    return p.rec + (size_t(g % p.ring_chunks) * p.H + h) * Rec::BYTES;
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

// Fills `rows` x (8 * chunks_per_row) elements of an image pair with f(row, k0, out8),
// storing 16-byte chunks at their swizzled offsets (shared or global memory).
// Row-major unit order (consecutive threads walk one row's chunks) suits f
// reading rows of a [row][K] array; chunk-major order (consecutive threads
// take consecutive rows of one chunk) suits f reading columns of a [K][row]
// array without shared-memory bank conflicts.  The loop is kept rolled: the
// generic kernel runs each phase once per chunk-head, so compact code (fewer
// instruction cache misses) measured faster than unrolled, batched loads.
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

// An MMA operand: hi and lo images (shared-memory addresses) in the
// 128-byte-swizzle layout, K-major or MN-major.  stride: K-major, the byte
// stride of its 64-wide K blocks (rows * 128); MN-major, its leading byte
// offset (the stride of its 64-element M / N blocks).
struct Operand {
    uint32_t hi, lo;
    bool mn;
    uint32_t stride;
};

// Descriptor of K step ks (16 K indices) of one image of an operand: a
// K-major start moves 32 bytes per step inside a 64-wide block and `stride`
// per block; an MN-major start moves 2048 bytes (two 8-row groups) per step.
__device__ __forceinline__ uint64_t op_desc(const Operand &o, uint32_t base, int ks) {
    if (o.mn) return sdesc_sw128_mn(base + uint32_t(ks) * 2048u, o.stride);
    return sdesc_sw128(base + uint32_t(ks >> 2) * o.stride + uint32_t(ks & 3) * 32u);
}

// One MMA group D (+)= A B^T over k_total / 16 K steps: nproducts = 1 issues
// hi.hi; 3 also hi.lo and lo.hi (the split product that keeps about 16
// mantissa bits); 2 issues hi.hi and lo.hi (exact when B holds 0 and 1).
__device__ __forceinline__ void mma_split(uint32_t d, const Operand &a, const Operand &b, int k_total, uint32_t idesc,
                                          int nproducts, bool accumulate) {
    const int ksteps = k_total / 16;
    for (int part = 0; part < nproducts; ++part) {
        const bool a_lo = (nproducts == 3 && part == 2) || (nproducts == 2 && part == 1);
        const bool b_lo = nproducts == 3 && part == 1;
        for (int ks = 0; ks < ksteps; ++ks)
            mma_bf16(d, op_desc(a, a_lo ? a.lo : a.hi, ks), op_desc(b, b_lo ? b.lo : b.hi, ks), idesc,
                     (accumulate || part > 0 || ks > 0) ? 1u : 0u);
    }
}

// Launchers of the intra-chunk kernels (kda_prefill_intra_*.cu).  grid:
// (chunks of the window, H) for a window of chunks starting at
// p.chunk_base; the generic kernel in list mode (p.fb_list set) takes a
// 1-D grid that walks the list.
kda_status intra_fast_prepare();
kda_status launch_intra_fast(const PrefillParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                             const CUtensorMap &mv, const CUtensorMap &ma, dim3 grid, cudaStream_t s);
template <typename Act>
kda_status intra_generic_prepare();
template <typename Act>
kda_status launch_intra_generic(const PrefillParams &p, const CUtensorMap &mq, const CUtensorMap &mk,
                                const CUtensorMap &mv, const CUtensorMap &ma, dim3 grid, cudaStream_t s);

}  // namespace pf
}  // namespace kda
