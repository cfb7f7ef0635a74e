// kda_prefill.cu -- chunked KDA prefill (WY / UT form), d_k = d_v = 128, C = 64.
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
// The exponent of exp(G_r - G_s) is split around a per-channel reference
// c_i (the middle of the chunk's log-decay range): k_r exp(G_r - c) times
// k_s exp(c - G_s).  Both factors stay inside fp32 range while the chunk's
// decay span per channel is below 160 (alpha around 0.08 or larger on
// average); a chunk beyond that takes an exact per-element path.
//
// Kernels (one stream, in order):
//   prep   (chunk, head): conv + SiLU, L2 of q and k, G, beta -> workspace
//   intra  (chunk, head): A, P, T, W, Ut                     -> workspace
//   chain  (sequence, head, d_v block): sequential over chunks: U, O, S;
//          interval checkpoints; end state -> slot
//   out    (chunk, head): gated RMSNorm of O -> out
//   tails  checkpoint tails, then end tails -> slots
#include "kda_internal.h"

#include <algorithm>
#include <cmath>
#include <mutex>
#include <vector>

namespace kda {

namespace {

constexpr int D = 128;     // channels per head (d_k = d_v)
constexpr int CH = 64;     // chunk length
constexpr int NB = 4;      // d_v blocks per head in the chain
constexpr int DB = D / NB; // value channels per chain CTA
constexpr float kLogAlphaMin = -100.0f;  // log(alpha) floor: alpha below e^-100 acts as e^-100
constexpr float kSafeSpan = 160.0f;      // max per-channel log-decay span for the split exponent

struct SeqMeta {
    int32_t row0, len, slot, has_init, chunk0, n_chunks;
};
struct ChunkMeta {
    int32_t seq, row0, len, pos0, ck_begin, ck_count;
};
struct CkptMeta {
    int32_t seq, token_pos, dst_slot, pad;
};

// Per (chunk, head) workspace record, fp32.
struct ChunkRec {
    static constexpr size_t QH = 0;                 // [64][128] L2-normalised q
    static constexpr size_t KH = QH + CH * D;       // [64][128] L2-normalised k
    static constexpr size_t VV = KH + CH * D;       // [64][128] conv'd v
    static constexpr size_t GG = VV + CH * D;       // [64][128] cumulative log decay
    static constexpr size_t WW = GG + CH * D;       // [64][128] W
    static constexpr size_t UT = WW + CH * D;       // [64][128] Ut
    static constexpr size_t OO = UT + CH * D;       // [64][128] O (pre-norm output)
    static constexpr size_t PP = OO + CH * D;       // [64][64]  P (zero above the diagonal)
    static constexpr size_t BB = PP + CH * CH;      // [64]      beta (0 on padding rows)
    static constexpr size_t FLOATS = BB + CH;
};

struct PrefillParams {
    const SeqMeta *seqs;
    const ChunkMeta *chunks;
    const CkptMeta *ckpts;
    float *rec;  // [n_chunks][H] ChunkRec
    float *states;
    void *tails;
    uint32_t *err;
    const void *q, *k, *v, *alpha, *beta, *gate;
    void *out;
    const void *conv_w, *norm_w;
    int32_t H, n_ch, n_seqs, n_chunks, n_ckpts;
    float eps_l2, eps_rms;
};

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

__device__ __forceinline__ float *rec_ptr(const PrefillParams &p, int g, int h) {
    return p.rec + (size_t(g) * p.H + h) * ChunkRec::FLOATS;
}

// ---------------------------------------------------------------- prep ----
template <typename Act>
__global__ void __launch_bounds__(D) prefill_prep_kernel(const PrefillParams p) {
    extern __shared__ __align__(16) float sm[];
    float *qs = sm;             // [64][128]
    float *ks = qs + CH * D;    // [64][128]
    float *rq = ks + CH * D;    // [64]
    float *rk = rq + CH;        // [64]
    const int g = blockIdx.x, h = blockIdx.y, i = threadIdx.x;
    const ChunkMeta cm = p.chunks[g];
    const SeqMeta sq = p.seqs[cm.seq];
    float *rec = rec_ptr(p, g, h);
    const Act *tail = static_cast<const Act *>(p.tails) + size_t(sq.slot) * 3 * p.n_ch;
    const Act *cw = static_cast<const Act *>(p.conv_w);
    const size_t HD = size_t(p.H) * D;
    for (int s = 0; s < 3; ++s) {
        const Act *src = static_cast<const Act *>(s == 0 ? p.q : (s == 1 ? p.k : p.v));
        const int ch = s * p.H * D + h * D + i;
        const float w0 = to_f32(cw[ch * 4 + 0]), w1 = to_f32(cw[ch * 4 + 1]);
        const float w2 = to_f32(cw[ch * 4 + 2]), w3 = to_f32(cw[ch * 4 + 3]);
        float x[3];
        for (int j = 0; j < 3; ++j) {
            const int pos = cm.pos0 - 3 + j;
            if (pos >= 0) x[j] = to_f32(src[size_t(sq.row0 + pos) * HD + size_t(h) * D + i]);
            else x[j] = sq.has_init ? to_f32(tail[size_t(3 + pos) * p.n_ch + ch]) : 0.f;
        }
        float *dst = s == 0 ? qs : (s == 1 ? ks : rec + ChunkRec::VV);
        for (int t = 0; t < CH; ++t) {
            float y = 0.f;
            if (t < cm.len) {
                const float xt = to_f32(src[size_t(cm.row0 + t) * HD + size_t(h) * D + i]);
                float acc = w0 * x[0];
                acc = fmaf(w1, x[1], acc);
                acc = fmaf(w2, x[2], acc);
                acc = fmaf(w3, xt, acc);
                y = acc * sigmoid_f(acc);
                x[0] = x[1];
                x[1] = x[2];
                x[2] = xt;
            }
            dst[t * D + i] = y;
        }
    }
    __syncthreads();
    const int warp = i >> 5, lane = i & 31;
    for (int t = warp; t < CH; t += D / 32) {
        float a = 0.f, b = 0.f;
        for (int c = lane; c < D; c += 32) {
            a = fmaf(qs[t * D + c], qs[t * D + c], a);
            b = fmaf(ks[t * D + c], ks[t * D + c], b);
        }
        for (int o = 16; o; o >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, o);
            b += __shfl_xor_sync(0xffffffffu, b, o);
        }
        if (lane == 0) {
            rq[t] = rsqrtf(a + p.eps_l2);
            rk[t] = rsqrtf(b + p.eps_l2);
        }
    }
    __syncthreads();
    const Act *al = static_cast<const Act *>(p.alpha);
    float G = 0.f;
    for (int t = 0; t < CH; ++t) {
        rec[ChunkRec::QH + t * D + i] = qs[t * D + i] * rq[t];
        rec[ChunkRec::KH + t * D + i] = ks[t * D + i] * rk[t];
        if (t < cm.len) G += fmaxf(logf(to_f32(al[size_t(cm.row0 + t) * HD + size_t(h) * D + i])), kLogAlphaMin);
        rec[ChunkRec::GG + t * D + i] = G;
    }
    if (i < CH)
        rec[ChunkRec::BB + i] =
            i < cm.len ? to_f32(static_cast<const Act *>(p.beta)[size_t(cm.row0 + i) * p.H + h]) : 0.f;
}

// ---------------------------------------------------------------- intra ---
// A, P, T = (I + A)^-1, W, Ut for one (chunk, head) on CUDA cores.
constexpr int LDK = D + 1;   // padded row of a [64][128] smem tile
constexpr int LDC = CH + 1;  // padded row of a [64][64] smem tile

__global__ void __launch_bounds__(256) prefill_intra_kernel(const PrefillParams p) {
    extern __shared__ __align__(16) float sm[];
    float *Ka = sm;               // [64][LDK]  k exp(G - c), later diag(beta) exp(G) k
    float *Kb = Ka + CH * LDK;    // [64][LDK]  k exp(c - G), later diag(beta) v
    float *Qa = Kb + CH * LDK;    // [64][LDK]  q exp(G - c)
    float *A = Qa + CH * LDK;     // [64][LDC]
    float *T = A + CH * LDC;      // [64][LDC]
    float *X = T + CH * LDC;      // [64][LDC] scratch for the block inverse
    float *cref = X + CH * LDC;   // [128]
    float *beta = cref + D;       // [64]
    int *flag = reinterpret_cast<int *>(beta + CH);
    const int g = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    float *rec = rec_ptr(p, g, h);
    const float *QH = rec + ChunkRec::QH, *KH = rec + ChunkRec::KH, *VV = rec + ChunkRec::VV,
                *GG = rec + ChunkRec::GG;
    if (tid == 0) *flag = 0;
    if (tid < CH) beta[tid] = rec[ChunkRec::BB + tid];
    __syncthreads();
    if (tid < D) {
        const float g0 = GG[tid], g1 = GG[(CH - 1) * D + tid];
        cref[tid] = 0.5f * (g0 + g1);
        if (g0 - g1 > kSafeSpan) atomicOr(flag, 1);
    }
    __syncthreads();
    const bool exact = *flag != 0;
    for (int e = tid; e < CH * D; e += 256) {
        const int r = e / D, i = e - r * D;
        const float gr = GG[e], c = cref[i];
        const float er = exact ? 1.f : expf(gr - c), es = exact ? 1.f : expf(c - gr);
        Ka[r * LDK + i] = KH[e] * er;
        Kb[r * LDK + i] = KH[e] * es;
        Qa[r * LDK + i] = QH[e] * er;
    }
    __syncthreads();
    // A (s < r, scaled by beta_r) and P (s <= r): 4 x 4 output block per thread
    {
        const int r0 = (tid >> 4) * 4, s0 = (tid & 15) * 4;
        float a[4][4] = {}, pp[4][4] = {};
        if (!exact) {
            for (int i = 0; i < D; ++i) {
                float kr[4], qr[4], ks[4];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    kr[m] = Ka[(r0 + m) * LDK + i];
                    qr[m] = Qa[(r0 + m) * LDK + i];
                    ks[m] = Kb[(s0 + m) * LDK + i];
                }
#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        a[m][n] = fmaf(kr[m], ks[n], a[m][n]);
                        pp[m][n] = fmaf(qr[m], ks[n], pp[m][n]);
                    }
            }
        } else {
            for (int i = 0; i < D; ++i)
#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int n = 0; n < 4; ++n) {
                        const int r = r0 + m, s = s0 + n;
                        if (s > r) continue;
                        const float f = expf(GG[r * D + i] - GG[s * D + i]) * Kb[s * LDK + i];
                        a[m][n] = fmaf(Ka[r * LDK + i], f, a[m][n]);
                        pp[m][n] = fmaf(Qa[r * LDK + i], f, pp[m][n]);
                    }
        }
        float *P = rec + ChunkRec::PP;
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 4; ++n) {
                const int r = r0 + m, s = s0 + n;
                A[r * LDC + s] = s < r ? beta[r] * a[m][n] : 0.f;
                P[r * CH + s] = s <= r ? pp[m][n] : 0.f;
            }
    }
    __syncthreads();
    // T = (I + A)^-1, unit lower triangular, by 16 x 16 blocks.
    // Diagonal blocks: forward substitution, one warp per block, lane = column
    // (each lane reads only the column it writes).
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int e = tid; e < CH * LDC; e += 256) T[e] = 0.f;
        __syncthreads();
        if (warp < 4 && lane < 16) {
            const int b0 = warp * 16, c = b0 + lane;
            for (int r = b0; r < b0 + 16; ++r) {
                float acc = (r == c) ? 1.f : 0.f;
                for (int s = c; s < r; ++s) acc = fmaf(-A[r * LDC + s], T[s * LDC + c], acc);
                T[r * LDC + c] = (r >= c) ? acc : 0.f;
            }
        }
        __syncthreads();
        // Off-diagonal blocks by distance d: T_ab = -T_aa sum_{b <= c < a} A_ac T_cb
        for (int d = 1; d < 4; ++d) {
            const int nblk = 4 - d;
            for (int e = tid; e < nblk * 256; e += 256) {
                const int blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
                const int a = blk + d, b = blk;
                float acc = 0.f;
                for (int s = b * 16; s < a * 16; ++s)
                    acc = fmaf(A[(a * 16 + r) * LDC + s], T[s * LDC + b * 16 + cc], acc);
                X[(a * 16 + r) * LDC + b * 16 + cc] = acc;
            }
            __syncthreads();
            for (int e = tid; e < nblk * 256; e += 256) {
                const int blk = e >> 8, r = (e >> 4) & 15, cc = e & 15;
                const int a = blk + d, b = blk;
                float acc = 0.f;
                for (int s = 0; s <= r; ++s)
                    acc = fmaf(-T[(a * 16 + r) * LDC + a * 16 + s], X[(a * 16 + s) * LDC + b * 16 + cc], acc);
                T[(a * 16 + r) * LDC + b * 16 + cc] = acc;
            }
            __syncthreads();
        }
    }
    // W = T diag(beta) (exp(G) . K),  Ut = T diag(beta) V
    for (int e = tid; e < CH * D; e += 256) {
        const int s = e / D, i = e - s * D;
        Ka[s * LDK + i] = beta[s] * expf(GG[e]) * KH[e];
        Kb[s * LDK + i] = beta[s] * VV[e];
    }
    __syncthreads();
    {
        const int r0 = (tid >> 4) * 4, i0 = (tid & 15) * 8;
        float w[4][8] = {}, u[4][8] = {};
        for (int s = 0; s < r0 + 4; ++s) {
            float t4[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) t4[m] = T[(r0 + m) * LDC + s];
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                const float kk = Ka[s * LDK + i0 + n], vv = Kb[s * LDK + i0 + n];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    w[m][n] = fmaf(t4[m], kk, w[m][n]);
                    u[m][n] = fmaf(t4[m], vv, u[m][n]);
                }
            }
        }
        float *W = rec + ChunkRec::WW, *U = rec + ChunkRec::UT;
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
            for (int n = 0; n < 8; ++n) {
                W[(r0 + m) * D + i0 + n] = w[m][n];
                U[(r0 + m) * D + i0 + n] = u[m][n];
            }
    }
}

// ---------------------------------------------------------------- chain ---
// One CTA per (sequence, head, d_v block of DB columns), sequential over the
// sequence's chunks.  S block [128][DB] lives in shared memory.
constexpr int LDS = DB + 1;

__global__ void __launch_bounds__(256) prefill_chain_kernel(const PrefillParams p) {
    extern __shared__ __align__(16) float sm[];
    float *S = sm;                 // [128][LDS]
    float *Wt = S + D * LDS;       // [64][LDK]  W
    float *Qt = Wt + CH * LDK;     // [64][LDK]  exp(G) . q
    float *Kt = Qt + CH * LDK;     // [64][LDK]  exp(G_last - G) . k
    float *P = Kt + CH * LDK;      // [64][LDC]
    float *U = P + CH * LDC;       // [64][LDS]
    float *gam = U + CH * LDS;     // [128]  exp(G_last)
    const int tid = threadIdx.x;
    const int jb = blockIdx.x % NB, h = (blockIdx.x / NB) % p.H, n = blockIdx.x / (NB * p.H);
    const SeqMeta sq = p.seqs[n];
    const size_t head_elems = size_t(D) * D;
    float *slot_state = p.states + size_t(sq.slot) * p.H * head_elems + size_t(h) * head_elems;  // [j][i]
    for (int e = tid; e < D * DB; e += 256) {
        const int j = e / D, i = e - j * D;  // coalesced over i
        S[i * LDS + j] = sq.has_init ? slot_state[size_t(jb * DB + j) * D + i] : 0.f;
    }
    __syncthreads();
    for (int c = 0; c < sq.n_chunks; ++c) {
        const int g = sq.chunk0 + c;
        float *rec = rec_ptr(p, g, h);
        const float *GG = rec + ChunkRec::GG;
        for (int e = tid; e < CH * D; e += 256) {
            const int r = e / D, i = e - r * D;
            const float gl = GG[(CH - 1) * D + i], gr = GG[e];
            Wt[r * LDK + i] = rec[ChunkRec::WW + e];
            Qt[r * LDK + i] = expf(gr) * rec[ChunkRec::QH + e];
            Kt[r * LDK + i] = expf(gl - gr) * rec[ChunkRec::KH + e];
        }
        for (int e = tid; e < CH * CH; e += 256) P[(e / CH) * LDC + (e % CH)] = rec[ChunkRec::PP + e];
        if (tid < D) gam[tid] = expf(GG[(CH - 1) * D + tid]);
        __syncthreads();
        // U = Ut - W S   (64 x DB, 8 outputs per thread)
        {
            const int r = tid >> 2, j0 = (tid & 3) * (DB / 4);
            float acc[DB / 4];
#pragma unroll
            for (int m = 0; m < DB / 4; ++m) acc[m] = rec[ChunkRec::UT + r * D + jb * DB + j0 + m];
            for (int i = 0; i < D; ++i) {
                const float wv = Wt[r * LDK + i];
#pragma unroll
                for (int m = 0; m < DB / 4; ++m) acc[m] = fmaf(-wv, S[i * LDS + j0 + m], acc[m]);
            }
#pragma unroll
            for (int m = 0; m < DB / 4; ++m) U[r * LDS + j0 + m] = acc[m];
        }
        __syncthreads();
        // O = Qt S + P U  -> workspace
        {
            const int r = tid >> 2, j0 = (tid & 3) * (DB / 4);
            float acc[DB / 4] = {};
            for (int i = 0; i < D; ++i) {
                const float qv = Qt[r * LDK + i];
#pragma unroll
                for (int m = 0; m < DB / 4; ++m) acc[m] = fmaf(qv, S[i * LDS + j0 + m], acc[m]);
            }
            for (int s = 0; s <= r; ++s) {
                const float pv = P[r * LDC + s];
#pragma unroll
                for (int m = 0; m < DB / 4; ++m) acc[m] = fmaf(pv, U[s * LDS + j0 + m], acc[m]);
            }
            float *O = rec + ChunkRec::OO;
#pragma unroll
            for (int m = 0; m < DB / 4; ++m) O[r * D + jb * DB + j0 + m] = acc[m];
        }
        __syncthreads();
        // S <- Diag(gamma) S + Kt^T U   (128 x DB, 16 outputs per thread)
        {
            const int i = tid >> 1, j0 = (tid & 1) * (DB / 2);
            float acc[DB / 2];
#pragma unroll
            for (int m = 0; m < DB / 2; ++m) acc[m] = gam[i] * S[i * LDS + j0 + m];
            for (int s = 0; s < CH; ++s) {
                const float kv = Kt[s * LDK + i];
#pragma unroll
                for (int m = 0; m < DB / 2; ++m) acc[m] = fmaf(kv, U[s * LDS + j0 + m], acc[m]);
            }
#pragma unroll
            for (int m = 0; m < DB / 2; ++m) S[i * LDS + j0 + m] = acc[m];
        }
        __syncthreads();
        const ChunkMeta cm = p.chunks[g];
        for (int q = 0; q < cm.ck_count; ++q) {
            const CkptMeta ck = p.ckpts[cm.ck_begin + q];
            float *dst = p.states + size_t(ck.dst_slot) * p.H * head_elems + size_t(h) * head_elems;
            for (int e = tid; e < D * DB; e += 256) {
                const int j = e / D, i = e - j * D;
                dst[size_t(jb * DB + j) * D + i] = S[i * LDS + j];
            }
        }
    }
    for (int e = tid; e < D * DB; e += 256) {
        const int j = e / D, i = e - j * D;
        slot_state[size_t(jb * DB + j) * D + i] = S[i * LDS + j];
    }
}

// ---------------------------------------------------------------- out -----
template <typename Act>
__global__ void __launch_bounds__(128) prefill_out_kernel(const PrefillParams p) {
    const int g = blockIdx.x, h = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ChunkMeta cm = p.chunks[g];
    const float *O = rec_ptr(p, g, h) + ChunkRec::OO;
    const Act *gate = static_cast<const Act *>(p.gate);
    const Act *nw = static_cast<const Act *>(p.norm_w);
    Act *out = static_cast<Act *>(p.out);
    const size_t HD = size_t(p.H) * D;
    for (int t = warp; t < cm.len; t += 4) {
        float o[4], ss = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            o[m] = O[t * D + lane * 4 + m];
            ss = fmaf(o[m], o[m], ss);
        }
        for (int s = 16; s; s >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, s);
        const float r = rsqrtf(ss * (1.0f / D) + p.eps_rms);
        const size_t base = size_t(cm.row0 + t) * HD + size_t(h) * D + lane * 4;
#pragma unroll
        for (int m = 0; m < 4; ++m)
            out[base + m] = from_f32<Act>(to_f32(nw[lane * 4 + m]) * (o[m] * r) * sigmoid_f(to_f32(gate[base + m])));
    }
}

// ---------------------------------------------------------------- tails ---
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
    const SeqMeta sq = p.seqs[seq];
    const Act *old = static_cast<const Act *>(p.tails) + size_t(sq.slot) * 3 * p.n_ch;
    Act *nt = static_cast<Act *>(p.tails) + size_t(dst) * 3 * p.n_ch;
    const int HD = p.H * D;
    for (int ch = threadIdx.x; ch < p.n_ch; ch += blockDim.x) {
        const int s = ch / HD, rem = ch - s * HD;
        const Act *src = static_cast<const Act *>(s == 0 ? p.q : (s == 1 ? p.k : p.v));
        Act x[3];
        for (int j = 0; j < 3; ++j) {
            const int q = pos - 3 + j;
            if (q >= 0) x[j] = src[size_t(sq.row0 + q) * HD + rem];
            else x[j] = sq.has_init ? old[size_t(3 + q) * p.n_ch + ch] : from_f32<Act>(0.f);
        }
        for (int j = 0; j < 3; ++j) nt[size_t(j) * p.n_ch + ch] = x[j];
    }
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct WsLayout {
    size_t seqs, chunks, ckpts, rec, total;
};

WsLayout ws_layout(int N, long long n_chunks, long long n_reqs, int H) {
    WsLayout L;
    L.seqs = 0;
    L.chunks = align256(L.seqs + sizeof(SeqMeta) * size_t(N));
    L.ckpts = align256(L.chunks + sizeof(ChunkMeta) * size_t(n_chunks));
    L.rec = align256(L.ckpts + sizeof(CkptMeta) * size_t(std::max<long long>(n_reqs, 1)));
    L.total = align256(L.rec + sizeof(float) * ChunkRec::FLOATS * size_t(n_chunks) * size_t(H));
    return L;
}

long long count_chunks(const int32_t *cu, int N) {
    long long n = 0;
    for (int s = 0; s < N; ++s) n += (cu[s + 1] - cu[s] + CH - 1) / CH;
    return n;
}

template <typename K>
kda_status set_smem(K kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes)) == cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}

constexpr size_t kPrepSmem = sizeof(float) * (2 * CH * D + 2 * CH);
constexpr size_t kIntraSmem = sizeof(float) * (3 * CH * LDK + 3 * CH * LDC + D + CH + 4);
constexpr size_t kChainSmem = sizeof(float) * (D * LDS + 3 * CH * LDK + CH * LDC + CH * LDS + D);

template <typename Act>
kda_status launch_act(const PrefillParams &p, int N, long long n_chunks, int n_reqs, cudaStream_t stream) {
    kda_status st;
    if ((st = set_smem(prefill_prep_kernel<Act>, kPrepSmem)) != KDA_OK) return st;
    if ((st = set_smem(prefill_intra_kernel, kIntraSmem)) != KDA_OK) return st;
    if ((st = set_smem(prefill_chain_kernel, kChainSmem)) != KDA_OK) return st;
    if (n_chunks > 0) {
        const dim3 grid(unsigned(n_chunks), unsigned(p.H));
        prefill_prep_kernel<Act><<<grid, D, kPrepSmem, stream>>>(p);
        prefill_intra_kernel<<<grid, 256, kIntraSmem, stream>>>(p);
    }
    prefill_chain_kernel<<<unsigned(N) * p.H * NB, 256, kChainSmem, stream>>>(p);
    if (n_chunks > 0) prefill_out_kernel<Act><<<dim3(unsigned(n_chunks), unsigned(p.H)), 128, 0, stream>>>(p);
    if (n_reqs > 0) prefill_tails_kernel<Act><<<n_reqs, 256, 0, stream>>>(p, 1);
    prefill_tails_kernel<Act><<<N, 256, 0, stream>>>(p, 0);
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
    if (N > 0 && cudaMemcpyAsync(ws + L.seqs, seqs.data(), sizeof(SeqMeta) * seqs.size(), cudaMemcpyHostToDevice,
                                 stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (!chunks.empty() && cudaMemcpyAsync(ws + L.chunks, chunks.data(), sizeof(ChunkMeta) * chunks.size(),
                                           cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (!cks.empty() && cudaMemcpyAsync(ws + L.ckpts, cks.data(), sizeof(CkptMeta) * cks.size(),
                                        cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return KDA_ERR_CUDA;
    PrefillParams p;
    p.seqs = reinterpret_cast<const SeqMeta *>(ws + L.seqs);
    p.chunks = reinterpret_cast<const ChunkMeta *>(ws + L.chunks);
    p.ckpts = reinterpret_cast<const CkptMeta *>(ws + L.ckpts);
    p.rec = reinterpret_cast<float *>(ws + L.rec);
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
    p.H = H;
    p.n_ch = pool->n_ch;
    p.n_seqs = N;
    p.n_chunks = int(n_chunks);
    p.n_ckpts = n_reqs;
    p.eps_l2 = w->eps_l2;
    p.eps_rms = w->eps_rms;
    if (pool->desc.act == KDA_BF16) return launch_act<__nv_bfloat16>(p, N, n_chunks, n_reqs, stream);
    return launch_act<float>(p, N, n_chunks, n_reqs, stream);
}

// ------------------------------------------------------ no-allocation entry --
// Fixed scratch for kda_prefill_chunked_noalloc: callers that cannot allocate
// device memory run the prefill in this array instead of a workspace of
// their own.  It lives in the module image, so every GPU that loads the
// library holds it until the process exits.  Host code must not use the
// array's name as a device address: the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
static __device__ __align__(256) unsigned char g_prefill_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

kda_status launch_prefill_noalloc(const kda_pool *pool, const kda_weights *w, const kda_io *io,
                                  const int32_t *cu_seqlens, const int32_t *slots,
                                  const uint8_t *has_initial_state, int N, int chunk, const kda_ckpt_req *reqs,
                                  int n_reqs, cudaStream_t stream) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static void *scratch[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
    void *ptr = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!scratch[dev]) {
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_prefill_noalloc_scratch) != cudaSuccess || !addr) {
                cudaGetLastError();
                return KDA_ERR_CUDA;
            }
            scratch[dev] = addr;
        }
        ptr = scratch[dev];
    }
    // Every byte of the scratch is written before it is read, so nothing is
    // cleared; a call that needs more than the array returns KDA_ERR_WORKSPACE.
    return launch_prefill(pool, w, io, cu_seqlens, slots, has_initial_state, N, chunk, reqs, n_reqs, ptr,
                          KDA_NOALLOC_SCRATCH_BYTES, stream);
}

}  // namespace kda
