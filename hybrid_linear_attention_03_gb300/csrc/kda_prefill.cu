// kda_prefill.cu -- chunked KDA prefill (WY / UT form) on TMA + tcgen05,
// d_k = d_v = 128, chunk C = 64: the chunk chain, the gated norm, the conv
// tails, the device metadata builder and the host-side schedule.
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
// The intra-chunk part (A, P, T, W, Ut) is kda_prefill_intra_fast.cu (bf16)
// and kda_prefill_intra_generic.cu (fp32, and chunks with a decay span too
// wide for the fast kernel's split exponent).  Every product that feeds the
// state runs on the tensor cores as three bf16 MMAs (x = hi + lo with
// hi = bf16(x), lo = bf16(x - hi): hi*hi + hi*lo + lo*hi, fp32 accumulation
// in TMEM), which keeps about 16 mantissa bits.
//
// Schedule: the chunks of a call are cut into windows.  Per window the intra
// kernel(s) run on the caller's stream, then the window's chain on a
// high-priority side stream, so the chain of one window overlaps the intra
// work of the next.  The per-(chunk, head) records live in a ring of two
// windows: window w + 2 reuses window w's records once its chain has run, so
// the workspace does not grow with the prompt.  The tails run on the caller's
// stream after the join.
//   meta   (device-built tables only, one CTA): sequence, chunk and
//          checkpoint tables from device arrays.
//   chain  (sequence, head): sequential over chunks; S^T (fp32) lives in
//          registers; the next chunk's operand images stream in by TMA bulk
//          copies while the current chunk computes; the gated RMSNorm of
//          each chunk's O -> out; interval checkpoints; end state -> slot.
//   tails  checkpoint tails, then end tails -> slots.
#include "kda_prefill.cuh"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

namespace kda {

namespace pf {
namespace {

constexpr int kRingWindows = 2;   // windows of records the ring holds
constexpr int kWindowChunks = 48; // chunks per window of a call long enough to be split
constexpr int kSplitChunks = 64;  // calls with fewer chunks run as one window
constexpr int kEventSlots = 8;    // per-window events, reused cyclically (more than kRingWindows + 1)

// ============================================================== chain ====
// bf16 value of a 16-bit shared-memory word
__device__ __forceinline__ float bf16_word(uint16_t w) { return __uint_as_float(uint32_t(w) << 16); }

namespace cs {  // chain shared-memory map
constexpr uint32_t A1_HI = 0, A1_LO = 32768;             // S^T images [128 j][128 i]
constexpr uint32_t B1 = 65536;                            // the record's WQ images (64 KiB)
constexpr uint32_t WQ_HI = B1, WQ_LO = B1 + 32768;
constexpr uint32_t B2 = 131072;                           // the record's KH, PP images, gamma, elc
constexpr uint32_t KH_HI = B2, KH_LO = B2 + uint32_t(Rec::KH_LO - Rec::KH_HI);
constexpr uint32_t PP_HI = B2 + uint32_t(Rec::PP_HI - Rec::KH_HI), PP_LO = B2 + uint32_t(Rec::PP_LO - Rec::KH_HI);
constexpr uint32_t GAM = B2 + uint32_t(Rec::GAM - Rec::KH_HI), ELC = B2 + uint32_t(Rec::ELC - Rec::KH_HI);
constexpr uint32_t A2_HI = 181248, A2_LO = 181248 + 16384;  // U^T images [128 j][64 r]
constexpr uint32_t GCUR = A2_LO + 16384;                   // gamma, elc of the current chunk [2][128]
constexpr uint32_t RED = GCUR + 1024;                      // per-warp sums of O^2 [4 lane quarters][64 tokens]
constexpr uint32_t BARS = RED + 1024;
// bf16 gate tile of a chunk (tokens [32 half][128 channels]): half 0 in the
// record's PP lo slot of B2 (never loaded for bf16 outputs), half 1 here
constexpr uint32_t GATE0 = PP_LO, GATE1 = (BARS + 512 + 1023) / 1024 * 1024;
constexpr uint32_t RS = GATE1 + 8192;                       // per warp: 1 / rms of its 32 tokens
constexpr uint32_t BYTES = RS + 1024;
}  // namespace cs
static_assert(cs::B2 + Rec::B2_BYTES <= cs::A2_HI, "chain smem map overlaps");
static_assert(cs::GATE0 + 8192 <= cs::B2 + Rec::B2_BYTES && cs::GATE0 >= cs::B2 + Rec::B2_BYTES_HI &&
                  cs::GATE0 % 1024 == 0,
              "gate half 0 sits in the PP lo slot");

// One CTA (8 warps) per (sequence, head), walking the window's chunks in
// order.  Thread (j, half) keeps S^T row j, columns 64 half .. + 63, in fp32
// registers.  TMEM columns: [(W S)^T | (Q S)^T] [0,128), (K^^T U)^T
// [128,256), (P U)^T [256,320).  Each step asks L2 for the record two chunks
// ahead, so the next step's bulk loads find it there.
//   stage 1  [(W S)^T | (Q S)^T] = S^T [W; Q]^T (the record's WQ, K-major)
//   U^T      = Ut^T - (W S)^T, split into hi / lo images
//   stage 2  (K^^T U)^T = U^T K^ (K^ read MN-major), (P U)^T = U^T P^T
//   S^T     <- S^T diag(gamma) + (K^^T U)^T diag(elc),  O^T = (Q S)^T + (P U)^T
//   out      = w_n . O / sqrt(mean_j O^2 + eps) . sigmoid(gate), per token
// Without the lo halves of Q and P (q_lo = 0, bf16 outputs) the Q rows of
// the WQ lo image stay zero in shared memory and (P U)^T takes one product.
// bf16: the chunk's gate tile arrives by two TMA loads (tm_g: a box of 32
// tokens) issued a step ahead, and each half of the outputs that the chunk
// fills replaces its gate half in place and leaves by a TMA store (tm_o);
// fp32, and the partial halves of a sequence's last chunk: each thread loads
// its 32 gate values or stores its outputs itself.
template <typename Act>
__global__ void __launch_bounds__(256) prefill_chain_kernel(const PrefillParams p,
                                                           const __grid_constant__ CUtensorMap tm_g,
                                                           const __grid_constant__ CUtensorMap tm_o) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1 KiB-aligned, still shared
    uint64_t *bar_b1 = reinterpret_cast<uint64_t *>(sm + cs::BARS);
    uint64_t *bar_b2 = bar_b1 + 1, *bar_m1 = bar_b1 + 2, *bar_m2 = bar_b1 + 3, *bar_g = bar_b1 + 4;
    uint32_t *tbase = reinterpret_cast<uint32_t *>(bar_b1 + 5);
    constexpr bool kGateTile = sizeof(Act) == 2;
    float *gcur = reinterpret_cast<float *>(sm + cs::GCUR);
    float *red = reinterpret_cast<float *>(sm + cs::RED);
    // 8 warps: warps w and w + 4 share TMEM lanes 32*(w % 4) .. +31 (value
    // channel j = TMEM lane) and split every row's columns between them.
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j = (warp & 3) * 32 + lane, half = warp >> 2;
    const int h = blockIdx.x % p.H, n = p.seq_base + blockIdx.x / p.H;
    const SeqMeta sq = p.seqs[n];
    if (sq.slot < 0) return;  // disabled by the device metadata check: leave every slot alone
    // The chunks of this sequence inside the launch's window [win_lo, win_hi).
    // A sequence with no chunks is settled by the window that starts at 0.
    const int c_lo = max(sq.chunk0, p.win_lo) - sq.chunk0;
    const int c_hi = min(sq.chunk0 + sq.n_chunks, p.win_hi) - sq.chunk0;
    if (c_hi <= c_lo && !(sq.n_chunks == 0 && p.win_lo == 0)) return;
    // a one-chunk sequence from a zero state that the intra kernel finished
    // (outputs, end state, checkpoints): nothing left here
    if (p.solo && sq.n_chunks == 1 && !sq.has_init && p.solo[size_t(n) * p.H + h]) return;
    // A window that continues a sequence reads the state the previous window
    // left in the slot.
    const bool load_state = sq.has_init || c_lo > 0;
    // a sequence that starts here from a zero state: its first step has
    // W S = Q S = 0, so that step skips stage 1 and the S image is built
    // only at its end
    const bool s_zero = !load_state;
    const size_t head_elems = size_t(D) * D;
    float *slot_state = p.states + size_t(sq.slot) * p.H * head_elems + size_t(h) * head_elems;  // S^T [j][i]
    const uint32_t sbase = smem_u32(sm);
    if (tid == 0) {
        for (int b = 0; b < 5; ++b) mbar_init(bar_b1 + b, 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(tbase, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase, tl = tm + (uint32_t((warp & 3) * 32) << 16);
    // the record's WQ images (without the Q rows' lo half unless q_lo) and
    // KH, PP, GAM, ELC (without PP lo unless q_lo) of chunk g
    const uint32_t b1_bytes = p.q_lo ? Rec::B1_BYTES : 32768u + 16384u;
    const uint32_t b2_bytes = p.q_lo ? Rec::B2_BYTES : Rec::B2_BYTES_HI;
    auto load_rec = [&](const char *r) {
        mbar_arrive_expect_tx(bar_b1, b1_bytes);
        if (p.q_lo) {
            bulk_load(sm + cs::B1, r + Rec::WQ_HI, Rec::B1_BYTES, bar_b1);
        } else {  // hi image, then the W rows (0..63) of both K blocks of the lo image
            bulk_load(sm + cs::WQ_HI, r + Rec::WQ_HI, 32768, bar_b1);
            bulk_load(sm + cs::WQ_LO, r + Rec::WQ_LO, 8192, bar_b1);
            bulk_load(sm + cs::WQ_LO + 16384, r + Rec::WQ_LO + 16384, 8192, bar_b1);
        }
        mbar_arrive_expect_tx(bar_b2, b2_bytes);
        bulk_load(sm + cs::B2, r + Rec::KH_HI, b2_bytes, bar_b2);
    };
    if (!p.q_lo) {  // the Q rows (64..127) of both K blocks of the WQ lo image stay zero
        for (int e = tid; e < 2 * 8192 / 16; e += 256) {
            const int kb = e >> 9, off = (e & 511) * 16;
            *reinterpret_cast<uint4 *>(sm + cs::WQ_LO + kb * 16384 + 8192 + off) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    const uint32_t ut_bytes = uint32_t(Rec::BYTES - Rec::UT);
    auto prefetch_rec = [&](const char *r) {  // into L2: the bulk loads and the Ut^T rows of a later step
        bulk_prefetch_l2(r + Rec::WQ_HI, p.q_lo ? Rec::B1_BYTES : 32768u);
        if (!p.q_lo) {
            bulk_prefetch_l2(r + Rec::WQ_LO, 8192);
            bulk_prefetch_l2(r + Rec::WQ_LO + 16384, 8192);
        }
        bulk_prefetch_l2(r + Rec::KH_HI, b2_bytes);
        bulk_prefetch_l2(r + Rec::UT, ut_bytes);
    };
    const size_t HD = size_t(p.H) * D;
    // bf16 gate tiles and output halves move through one thread: thread 0
    // loads the first chunk's gate tile, thread 32 the others (and stores
    // the outputs; its bulk group is waited on before they are overwritten)
    auto load_gate = [&](int row0) {
        mbar_arrive_expect_tx(bar_g, 2 * 8192);
        tma_load_3d(sm + cs::GATE0, &tm_g, bar_g, 0, h, row0);
        tma_load_3d(sm + cs::GATE1, &tm_g, bar_g, 0, h, row0 + 32);
    };
    auto store_out = [&](const ChunkMeta &m) {  // the staged (full) output halves of chunk m
        if (m.len >= 32) tma_store_3d(&tm_o, sm + cs::GATE0, 0, h, m.row0);
        if (m.len >= 64) tma_store_3d(&tm_o, sm + cs::GATE1, 0, h, m.row0 + 32);
        bulk_commit();
    };
    if (tid == 0 && c_hi > c_lo) {
        load_rec(rec_ptr(p, sq.chunk0 + c_lo, h));
        if (c_lo + 1 < c_hi) prefetch_rec(rec_ptr(p, sq.chunk0 + c_lo + 1, h));
        if (kGateTile) load_gate(p.chunks[sq.chunk0 + c_lo].row0);
    }
    const int sc0 = half * 64;  // this thread's 64 columns of the S^T row
    // S^T row j (64 columns) in registers; hi/lo into the A1 images
    float sr[64];
    const float *srow = slot_state + size_t(j) * D + sc0;
#pragma unroll
    for (int e = 0; e < 64; e += 4) {
        const float4 x = load_state ? ld4(srow + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        sr[e] = x.x; sr[e + 1] = x.y; sr[e + 2] = x.z; sr[e + 3] = x.w;
    }
    if (!s_zero) {
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = sr[8 * cc + e];
            uint4 vh, vl;
            split8(x, vh, vl);
            const uint32_t off = sw128_chunk(j, (sc0 >> 3) + cc, D);
            *reinterpret_cast<uint4 *>(sm + cs::A1_HI + off) = vh;
            *reinterpret_cast<uint4 *>(sm + cs::A1_LO + off) = vl;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    bool ok = true;
    const uint32_t id_s1 = idesc_bf16_f32(128, 2 * CH), id_kh = idesc_bf16_f32(128, D, false, true),
                   id_pp = idesc_bf16_f32(128, CH);
    const Operand s_img{sbase + cs::A1_HI, sbase + cs::A1_LO, false, D * 128};
    const Operand wq_img{sbase + cs::WQ_HI, sbase + cs::WQ_LO, false, 2 * CH * 128};
    const Operand u_img{sbase + cs::A2_HI, sbase + cs::A2_LO, false, D * 128};
    const Operand kh_img{sbase + cs::KH_HI, sbase + cs::KH_LO, true, CH * 128};
    const Operand pp_img{sbase + cs::PP_HI, sbase + cs::PP_LO, false, CH * 128};
    const int uc0 = half * 32;  // this thread's 32 columns of the U / O rows
    const float wn = to_f32(static_cast<const Act *>(p.norm_w)[j]);
    ChunkMeta pcm{};  // the previous chunk (its outputs still staged)
    for (int c = c_lo; c < c_hi && ok; ++c) {
        const int g = sq.chunk0 + c;
        char *rec = rec_ptr(p, g, h);
        const ChunkMeta cm = p.chunks[g];
        const uint32_t par = uint32_t((c - c_lo) & 1);
        const bool z = s_zero && c == c_lo;                            // S = 0: no stage 1
        const uint32_t par1 = uint32_t((c - c_lo - (s_zero ? 1 : 0)) & 1);  // stage-1 commits so far
        ok = __syncthreads_and(mbar_wait(bar_b1, par, p.err));
        if (!ok) break;
        if (kGateTile && tid == 32 && c > c_lo) {  // previous outputs out, this chunk's gate tile in
            store_out(pcm);
            bulk_wait_read();
            load_gate(cm.row0);
        }
        if (tid == 0) {
            tc_fence_after();
            if (!z) {
                mma_split(tm + 0, s_img, wq_img, D, id_s1, 3, false);
                mma_commit(bar_m1);
            }
            if (c + 2 < c_hi) prefetch_rec(rec_ptr(p, g + 2, h));
        }
        // Ut^T row j, entries r = uc0 .. uc0 + 31, while the MMAs run
        float ut[32];
        const float *UTg = reinterpret_cast<const float *>(rec + Rec::UT) + size_t(j) * CH;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
            const float4 x = ld4(UTg + 4 * ut_chunk(j, (uc0 + e) >> 2));
            ut[e] = x.x; ut[e + 1] = x.y; ut[e + 2] = x.z; ut[e + 3] = x.w;
        }
        if (!z) {
            ok = __syncthreads_and(mbar_wait(bar_m1, par1, p.err));
            if (!ok) break;
            tc_fence_after();
        }
        if (tid == 0 && c + 1 < c_hi) {  // W and Q images are consumed: stream in the next chunk's
            const char *rn = rec_ptr(p, g + 1, h);
            mbar_arrive_expect_tx(bar_b1, b1_bytes);
            if (p.q_lo) {
                bulk_load(sm + cs::B1, rn + Rec::WQ_HI, Rec::B1_BYTES, bar_b1);
            } else {
                bulk_load(sm + cs::WQ_HI, rn + Rec::WQ_HI, 32768, bar_b1);
                bulk_load(sm + cs::WQ_LO, rn + Rec::WQ_LO, 8192, bar_b1);
                bulk_load(sm + cs::WQ_LO + 16384, rn + Rec::WQ_LO + 16384, 8192, bar_b1);
            }
        }
        // U^T row j = Ut^T - (W S)^T  -> hi/lo images (this thread's 32 columns)
        {
            float v[2][16];
            if (z) {
#pragma unroll
                for (int e = 0; e < 16; ++e) v[0][e] = v[1][e] = 0.f;
            } else {
                tmem_ld16(tl + uc0, v[0]);
                tmem_ld16(tl + uc0 + 16, v[1]);
                tmem_wait_ld();
            }
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
        gcur[half * D + j] = reinterpret_cast<const float *>(sm + (half ? cs::ELC : cs::GAM))[j];
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            mma_split(tm + 128, u_img, kh_img, CH, id_kh, 3, false);
            mma_split(tm + 256, u_img, pp_img, CH, id_pp, p.q_lo ? 3 : 1, false);
            mma_commit(bar_m2);
        }
        // fp32: the gate logits of tokens uc0 .. uc0 + 31 at channel j, under the MMAs
        constexpr int kGt = kGateTile ? 1 : 32;
        float gt[kGt];
        if (!kGateTile) {
            const Act *gp = static_cast<const Act *>(p.gate) + size_t(cm.row0 + uc0) * HD + size_t(h) * D + j;
#pragma unroll
            for (int e = 0; e < kGt; ++e) gt[e] = uc0 + e < cm.len ? to_f32(gp[size_t(e) * HD]) : 0.f;
        }
        ok = __syncthreads_and(mbar_wait(bar_m2, par, p.err));
        if (!ok) break;
        tc_fence_after();
        if (tid == 0 && c + 1 < c_hi) {  // K^, P images, gamma and elc consumed
            mbar_arrive_expect_tx(bar_b2, b2_bytes);
            bulk_load(sm + cs::B2, rec_ptr(p, g + 1, h) + Rec::KH_HI, b2_bytes, bar_b2);
        }
        // O at channel j, tokens uc0 .. uc0 + 31 = (Q S)^T + (P U)^T, then the
        // gated RMSNorm over the head's channels -> out (coalesced across the warp)
        {
            float o[32];
            {
                float v[2][16], w2[2][16];
#pragma unroll
                for (int q = 0; q < 2; ++q) tmem_ld16(tl + 256 + uc0 + 16 * q, w2[q]);
                if (z) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[0][e] = v[1][e] = 0.f;
                } else {
#pragma unroll
                    for (int q = 0; q < 2; ++q) tmem_ld16(tl + 64 + uc0 + 16 * q, v[q]);
                }
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[16 * q + e] = v[q][e] + w2[q][e];
            }
            // w_n . sigma of the gate logits first: it needs no reduction, so
            // its MUFU work overlaps the shuffles below
            uint16_t *gs = reinterpret_cast<uint16_t *>(sm + (half ? cs::GATE1 : cs::GATE0)) + j;
            if (kGateTile) ok = mbar_wait(bar_g, par, p.err) && ok;
            float sg[32];
            const float hwn = 0.5f * wn;
#pragma unroll
            for (int e = 0; e < 32; ++e)
                sg[e] = kGateTile ? scaled_sigmoid_tanh(bf16_word(gs[e * D]), hwn) : wn * sigmoid_fast(gt[kGateTile ? 0 : e]);
            // per token, the sum of O^2 over this warp's 32 channels: a
            // transpose-reduce over the lanes leaves token uc0 + lane's in lane
            float a[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) a[e] = o[e] * o[e];
#pragma unroll
            for (int wd = 16; wd >= 1; wd >>= 1) {
                const bool up = (lane & wd) != 0;
#pragma unroll
                for (int e = 0; e < wd; ++e) {
                    const float send = up ? a[e] : a[e + wd];
                    const float keep = up ? a[e + wd] : a[e];
                    a[e] = keep + __shfl_xor_sync(0xffffffffu, send, wd);
                }
            }
            red[(warp & 3) * CH + uc0 + lane] = a[0];
            // the four warps of this half of the tokens (named barrier 1 + half)
            asm volatile("bar.sync %0, 128;" ::"r"(1 + half) : "memory");
            const float ss = (red[uc0 + lane] + red[CH + uc0 + lane]) + (red[2 * CH + uc0 + lane] + red[3 * CH + uc0 + lane]);
            // token uc0 + lane's 1 / rms, to every lane of the warp through its own slot
            float *rsw = reinterpret_cast<float *>(sm + cs::RS) + warp * 32;
            rsw[lane] = rsqrtf(ss * (1.0f / D) + p.eps_rms);
            __syncwarp();
            float rv[32];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 r4 = *reinterpret_cast<const float4 *>(rsw + e);
                rv[e] = r4.x; rv[e + 1] = r4.y; rv[e + 2] = r4.z; rv[e + 3] = r4.w;
            }
            if (kGateTile && uc0 + 32 <= cm.len) {  // a full half: staged over its gate tile for a TMA store
#pragma unroll
                for (int e = 0; e < 32; ++e) gs[e * D] = __bfloat16_as_ushort(__float2bfloat16_rn((o[e] * rv[e]) * sg[e]));
            } else {
                Act *op = static_cast<Act *>(p.out) + size_t(cm.row0 + uc0) * HD + size_t(h) * D + j;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float y = (o[e] * rv[e]) * sg[e];
                    if (uc0 + e < cm.len) op[size_t(e) * HD] = from_f32<Act>(y);
                }
            }
        }
        // S^T row j <- gamma . S^T row j + elc . (K^^T U)^T row j; refresh the A1 images
        {
            float ds[4][16];
#pragma unroll
            for (int q = 0; q < 4; ++q) tmem_ld16(tl + 128 + sc0 + 16 * q, ds[q]);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 64; ++e) sr[e] = fmaf(gcur[sc0 + e], sr[e], gcur[D + sc0 + e] * ds[e >> 4][e & 15]);
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = sr[8 * cc + e];
            uint4 vh, vl;
            split8(x, vh, vl);
            const uint32_t off = sw128_chunk(j, (sc0 >> 3) + cc, D);
            *reinterpret_cast<uint4 *>(sm + cs::A1_HI + off) = vh;
            *reinterpret_cast<uint4 *>(sm + cs::A1_LO + off) = vl;
        }
        for (int k = 0; k < cm.ck_count; ++k) {  // interval checkpoints of this chunk end
            const CkptMeta ck = p.ckpts[cm.ck_begin + k];
            float *dst = p.states + size_t(ck.dst_slot) * p.H * head_elems + size_t(h) * head_elems + size_t(j) * D + sc0;
#pragma unroll
            for (int e = 0; e < 64; e += 4) *reinterpret_cast<float4 *>(dst + e) = make_float4(sr[e], sr[e + 1], sr[e + 2], sr[e + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok);
        tc_fence_after();
        pcm = cm;
    }
    // end state S^T row j (this thread's 64 columns) -> slot
    if (ok) {
        float *drow = slot_state + size_t(j) * D + sc0;
#pragma unroll
        for (int e = 0; e < 64; e += 4) *reinterpret_cast<float4 *>(drow + e) = make_float4(sr[e], sr[e + 1], sr[e + 2], sr[e + 3]);
    }
    if (kGateTile && tid == 32) {  // the last chunk's outputs; every store done before the CTA leaves
        if (ok && c_hi > c_lo) store_out(pcm);
        bulk_wait();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// ============================================================== tails ====
// Conv tail after `pos` tokens of a segment: raw inputs at pos-3 .. pos-1
// (before the segment: the slot's old tail, or zeros for a new sequence).
// blockIdx.x is the checkpoint request when ckpt_pass, else the sequence; a
// thread moves 8 consecutive channels (16 or 32 bytes, one stream: H d is a
// multiple of 8) of the three rows, blockIdx.y the block of 256 x 8
// channels.  The request pass runs first because it may read a sequence
// slot's old tail.
template <typename Act>
__global__ void __launch_bounds__(256) prefill_tails_kernel(const PrefillParams p, int ckpt_pass) {
    const int item = blockIdx.x;
    const int ch = 8 * (int(blockIdx.y) * 256 + int(threadIdx.x));
    if (ch >= p.n_ch) return;
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
    constexpr int kWords = int(sizeof(Act)) / 2;  // 16-byte words per 8 values
    const uint4 *old = reinterpret_cast<const uint4 *>(static_cast<const Act *>(p.tails) + size_t(sq.slot) * 3 * p.n_ch + ch);
    uint4 *nt = reinterpret_cast<uint4 *>(static_cast<Act *>(p.tails) + size_t(dst) * 3 * p.n_ch + ch);
    const int HD = p.H * D, s = ch / HD, rem = ch - s * HD;
    const Act *src = static_cast<const Act *>(s == 0 ? p.q : (s == 1 ? p.k : p.v));
    const size_t row_words = size_t(p.n_ch) / 8 * kWords;  // one tail row in 16-byte words
    uint4 x[3][kWords];
#pragma unroll
    for (int jj = 0; jj < 3; ++jj) {
        const int q = pos - 3 + jj;
        const uint4 *from = q >= 0 ? reinterpret_cast<const uint4 *>(src + size_t(sq.row0 + q) * HD + rem)
                                   : (sq.has_init ? old + size_t(3 + q) * row_words : nullptr);
#pragma unroll
        for (int u = 0; u < kWords; ++u) x[jj][u] = from ? from[u] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int jj = 0; jj < 3; ++jj)
#pragma unroll
        for (int u = 0; u < kWords; ++u) nt[size_t(jj) * row_words + u] = x[jj][u];
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

// Workspace: the tables, the fast kernel's two fallback lists (counts, then
// g * H + h entries of one window each; windows alternate), the flags of the
// one-chunk sequences the fast kernel finished ([N][H] bytes), then the
// record ring.
struct WsLayout {
    size_t seqs, chunks, ckpts, fb, solo, rec, total;
    int window;        // chunks per window
    int ring_windows;  // windows the record ring holds
};

int preferred_window(long long n_chunks) {
    return n_chunks < kSplitChunks ? int(std::max<long long>(n_chunks, 1)) : kWindowChunks;
}

WsLayout ws_layout(int N, long long n_chunks, long long n_reqs, int H, int window) {
    WsLayout L;
    L.window = window;
    const long long n_win = std::max<long long>((n_chunks + window - 1) / window, 1);
    L.ring_windows = int(std::min<long long>(kRingWindows, n_win));
    L.seqs = 0;
    L.chunks = align256(L.seqs + sizeof(SeqMeta) * size_t(N));
    L.ckpts = align256(L.chunks + sizeof(ChunkMeta) * size_t(n_chunks));
    L.fb = align256(L.ckpts + sizeof(CkptMeta) * size_t(std::max<long long>(n_reqs, 1)));
    L.solo = align256(L.fb + 32 + 2 * sizeof(uint32_t) * size_t(window) * size_t(H));
    L.rec = (L.solo + size_t(N) * size_t(H) + 1023) / 1024 * 1024;
    L.total = L.rec + Rec::BYTES * size_t(L.ring_windows) * size_t(window) * size_t(H);
    return L;
}

// The device-built tables' workspace: ws_layout plus the slot bitmap the
// builder uses to find repeated slots (at the end).
struct WsLayoutDev {
    WsLayout L;
    size_t used, total;
};
WsLayoutDev ws_layout_dev(int N, long long max_chunks, long long n_reqs, int H, int num_slots, int window) {
    WsLayoutDev d;
    d.L = ws_layout(N, max_chunks, n_reqs, H, window);
    d.used = align256(d.L.total);
    d.total = d.used + sizeof(uint32_t) * size_t((num_slots + 31) / 32);
    return d;
}

// The largest window, at most the preferred one, whose workspace (total(w))
// fits in `bytes`; 0 if not even windows of one chunk fit.  Below a single
// window the ring holds two windows, so the size grows with the window.
template <typename F>
int fit_window(size_t bytes, long long n_chunks, F total) {
    const int pref = preferred_window(n_chunks);
    if (total(pref) <= bytes) return pref;
    int lo = 1, hi = int(std::min<long long>(pref - 1, std::max<long long>(n_chunks - 1, 1))), best = 0;
    while (lo <= hi) {
        const int mid = (lo + hi) / 2;
        if (total(mid) <= bytes) {
            best = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    return best;
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

constexpr size_t kChainSmem = 1024 + cs::BYTES;

// Per-device side streams (the chain's at the highest priority) and events
// for the windowed overlap of the chain and the gated norm with the intra
// kernels.  Not memory: nothing here allocates device memory.
struct SideStream {
    cudaStream_t s = nullptr;  // chain (highest priority)
    cudaEvent_t intra_done[kEventSlots] = {}, chain_done[kEventSlots] = {};
    cudaEvent_t start = nullptr, s_done = nullptr;
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
        for (int i = 0; i < kEventSlots; ++i)
            if (cudaEventCreateWithFlags(&x.intra_done[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&x.chain_done[i], cudaEventDisableTiming) != cudaSuccess)
                return;
        if (cudaEventCreateWithFlags(&x.start, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&x.s_done, cudaEventDisableTiming) != cudaSuccess)
            return;
        x.ok = true;
    });
    return per_dev[dev].ok ? &per_dev[dev] : nullptr;
}

// Sequences [lo, hi) whose chunks meet a window (host-built tables).
struct SeqRange {
    int lo, hi;
    int32_t row0_base;  // a window inside one sequence: chunk g starts at row row0_base + C g
};

template <typename Act>
kda_status launch_act(const PrefillParams &p0, const kda_io *io, int n_tok, int N, long long n_chunks, int n_reqs,
                      const WsLayout &L, const std::vector<SeqRange> *ranges, bool solo, cudaStream_t stream) {
    constexpr bool kFast = sizeof(Act) == 2;
    kda_status st;
    if ((st = kFast ? intra_fast_prepare() : KDA_OK) != KDA_OK) return st;
    if ((st = intra_generic_prepare<Act>()) != KDA_OK) return st;
    if ((st = set_smem(prefill_chain_kernel<Act>, kChainSmem)) != KDA_OK) return st;
    PrefillParams p = p0;
    p.ring_chunks = L.ring_windows * L.window;
    p.q_lo = kFast ? 0 : 1;  // exp(G) . q and P feed only the output: bf16 outputs keep their hi halves
    // only the bf16 intra kernel finishes one-chunk sequences itself, and
    // only its variant for calls that may have them
    if (!kFast || !solo) p.solo = nullptr;
    CUtensorMap mq, mk, mv, ma, mg, mo;
    std::memset(&mg, 0, sizeof(mg));  // fp32: the chain loads its gate values and stores its outputs itself
    std::memset(&mo, 0, sizeof(mo));
    if (n_chunks > 0) {
        const int es = int(sizeof(Act));
        if (!make_map(&mq, io->q, n_tok, p.H, es, CH + HALO) || !make_map(&mk, io->k, n_tok, p.H, es, CH + HALO) ||
            !make_map(&mv, io->v, n_tok, p.H, es, CH + HALO) || !make_map(&ma, io->alpha, n_tok, p.H, es, CH) ||
            (kFast && (!make_map(&mg, io->gate, n_tok, p.H, es, 32) || !make_map(&mo, io->out, n_tok, p.H, es, 32))))
            return KDA_ERR_CUDA;
    }
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const unsigned fb_ctas = unsigned(std::max(sms / 4, 1));  // generic kernel CTAs walking the fallback list
    const int W = L.window;
    const long long n_win = std::max<long long>((n_chunks + W - 1) / W, 1);
    // The side stream's events are shared by every caller of this device:
    // one call's record / wait sequence is enqueued as a whole.
    static std::mutex enqueue_mu;
    std::lock_guard<std::mutex> lock(enqueue_mu);
    SideStream *side = n_win >= 2 ? side_stream() : nullptr;
    cudaStream_t cs = side ? side->s : stream;
    // An event call that fails after kernels are queued on the side streams:
    // join them to the caller's stream as far as the runtime still allows, so
    // nothing of this call runs after the caller's stream has moved past it
    // (the caller may free the workspace once it sees the error).
    auto fail = [&]() {
        if (side) {
            cudaEventRecord(side->s_done, cs);
            cudaStreamWaitEvent(stream, side->s_done, 0);
        }
        cudaGetLastError();
        return KDA_ERR_CUDA;
    };
    // the fast kernel of window w lists the chunks it leaves to the generic
    // kernel in list w mod 2; the generic kernel walks it on the chain's stream
    // just before that window's chain, which then clears its count for window w + 2
    if (kFast && cudaMemsetAsync(p.fb_count, 0, 2 * sizeof(uint32_t), stream) != cudaSuccess) return KDA_ERR_CUDA;
    if (side) {  // the chain stream starts after everything already on the caller's stream
        if (cudaEventRecord(side->start, stream) != cudaSuccess || cudaStreamWaitEvent(cs, side->start, 0) != cudaSuccess)
            return fail();
    }
    for (long long w = 0; w < n_win; ++w) {
        const long long lo = std::min(n_chunks, w * W), hi = std::min(n_chunks, (w + 1) * W);
        const int ev = int(w % kEventSlots);
        // window w writes the records window w - kRingWindows used: after that window's chain
        if (side && w >= L.ring_windows &&
            cudaStreamWaitEvent(stream, side->chain_done[(w - L.ring_windows) % kEventSlots], 0) != cudaSuccess)
            return fail();
        PrefillParams pw = p;  // this window's fallback list and row rule
        pw.row0_base = ranges ? (*ranges)[size_t(w)].row0_base : kNoRowBase;
        pw.fb_count = p.fb_count + (w & 1);
        pw.fb_list = p.fb_list + size_t(w & 1) * size_t(W) * size_t(p.H);
        if (hi > lo) {
            p.chunk_base = int(lo);
            pw.chunk_base = int(lo);
            const dim3 grid(unsigned(hi - lo), unsigned(p.H));
            if (kFast) {
                if ((st = launch_intra_fast(pw, mq, mk, mv, ma, grid, stream)) != KDA_OK) return fail();
            } else {
                PrefillParams pg = p;
                pg.fb_list = nullptr;  // grid mode: one CTA per (chunk, head) of the window
                if ((st = launch_intra_generic<Act>(pg, mq, mk, mv, ma, grid, stream)) != KDA_OK) return fail();
            }
        }
        p.win_lo = int(lo);
        p.win_hi = int(hi);
        // the chain of window 0 also settles the sequences that have no chunks
        const SeqRange rg = (ranges && w > 0) ? (*ranges)[size_t(w)] : SeqRange{0, N, kNoRowBase};
        if (side) {
            if (cudaEventRecord(side->intra_done[ev], stream) != cudaSuccess ||
                cudaStreamWaitEvent(cs, side->intra_done[ev], 0) != cudaSuccess)
                return fail();
        }
        if (kFast && hi > lo) {
            if ((st = launch_intra_generic<Act>(pw, mq, mk, mv, ma, dim3(fb_ctas), cs)) != KDA_OK) return fail();
            if (cudaMemsetAsync(pw.fb_count, 0, sizeof(uint32_t), cs) != cudaSuccess) return fail();
        }
        if (rg.hi > rg.lo) {
            p.seq_base = rg.lo;
            const ProfScope prof(KDA_KERNEL_PREFILL_CHAIN, cs);
            prefill_chain_kernel<Act><<<unsigned(rg.hi - rg.lo) * unsigned(p.H), 256, kChainSmem, cs>>>(p, mg, mo);
        }
        if (side && cudaEventRecord(side->chain_done[ev], cs) != cudaSuccess) return fail();
    }
    if (side) {
        if (cudaEventRecord(side->s_done, cs) != cudaSuccess || cudaStreamWaitEvent(stream, side->s_done, 0) != cudaSuccess)
            return fail();
    }
    p.chunk_base = 0;
    {
        const ProfScope prof(KDA_KERNEL_PREFILL_TAILS, stream);
        const unsigned ch_blocks = unsigned((p.n_ch / 8 + 255) / 256);
        if (n_reqs > 0) prefill_tails_kernel<Act><<<dim3(unsigned(n_reqs), ch_blocks), 256, 0, stream>>>(p, 1);
        prefill_tails_kernel<Act><<<dim3(unsigned(N), ch_blocks), 256, 0, stream>>>(p, 0);
    }
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Launch parameters over the workspace's tables (written, or enqueued to be
// written, on the stream) and the kernels.  n_chunks sizes the grids; n_tok
// is the token extent of the activation arrays the tensor maps describe;
// solo picks the intra variant that finishes one-chunk sequences itself.
kda_status launch_tables(const kda_pool *pool, const kda_weights *w, const kda_io *io, char *ws, const WsLayout &L,
                         int N, int n_reqs, long long n_chunks, int n_tok, const std::vector<SeqRange> *ranges,
                         bool solo, cudaStream_t stream) {
    PrefillParams p{};
    p.chunk_base = 0;
    p.win_lo = 0;
    p.win_hi = int(n_chunks);
    p.seq_base = 0;
    p.row0_base = kNoRowBase;
    p.seqs = reinterpret_cast<const SeqMeta *>(ws + L.seqs);
    p.chunks = reinterpret_cast<const ChunkMeta *>(ws + L.chunks);
    p.ckpts = reinterpret_cast<const CkptMeta *>(ws + L.ckpts);
    p.fb_count = reinterpret_cast<uint32_t *>(ws + L.fb);  // [2]
    p.fb_list = p.fb_count + 8;                             // [2][window * H]
    p.solo = reinterpret_cast<uint8_t *>(ws + L.solo);      // [N][H]
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
    if (pool->desc.act == KDA_BF16)
        return launch_act<__nv_bfloat16>(p, io, n_tok, N, n_chunks, n_reqs, L, ranges, solo, stream);
    return launch_act<float>(p, io, n_tok, N, n_chunks, n_reqs, L, ranges, solo, stream);
}

}  // namespace
}  // namespace pf

using pf::CH;
using pf::D;

size_t prefill_workspace_bytes(const kda_pool *pool, const int32_t *cu_seqlens, int N, int chunk) {
    if (chunk != CH || pool->desc.d_k != D || pool->desc.d_v != D || N < 0) return 0;
    if (cu_seqlens[0] != 0) return 0;
    for (int s = 0; s < N; ++s)
        if (cu_seqlens[s + 1] < cu_seqlens[s]) return 0;
    // room for one checkpoint per chunk end and per sequence end, twice over
    const long long nc = pf::count_chunks(cu_seqlens, N);
    return pf::ws_layout(N, nc, 2 * (nc + N), pool->desc.num_heads, pf::preferred_window(nc)).total;
}

kda_status launch_prefill(const kda_pool *pool, const kda_weights *w, const kda_io *io, const int32_t *cu_seqlens,
                          const int32_t *slots, const uint8_t *has_initial_state, int N, int chunk,
                          const kda_ckpt_req *reqs, int n_reqs, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream) {
    using namespace pf;
    if (pool->desc.d_k != D || pool->desc.d_v != D || chunk != CH) return KDA_ERR_UNSUPPORTED;
    const int H = pool->desc.num_heads;
    const long long n_chunks = count_chunks(cu_seqlens, N);
    if (n_chunks > (1LL << 31) / std::max(H, 1)) return KDA_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % 256) != 0) return KDA_ERR_WORKSPACE;
    const int window =
        fit_window(workspace_bytes, n_chunks, [&](int wv) { return ws_layout(N, n_chunks, n_reqs, H, wv).total; });
    if (window == 0) return KDA_ERR_WORKSPACE;
    const WsLayout L = ws_layout(N, n_chunks, n_reqs, H, window);
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
    // the sequences whose chunks meet each window (their chunks are contiguous)
    const long long n_win = std::max<long long>((n_chunks + window - 1) / window, 1);
    std::vector<SeqRange> ranges(static_cast<size_t>(n_win), SeqRange{0, 0, kNoRowBase});
    for (long long wv = 0; wv < n_win; ++wv) {
        const long long lo = wv * window, hi = std::min(n_chunks, lo + window);
        if (hi <= lo) continue;
        const int s0 = chunks[size_t(lo)].seq, s1 = chunks[size_t(hi - 1)].seq;
        ranges[size_t(wv)] = {s0, s1 + 1, kNoRowBase};
        if (s0 == s1) {  // chunk g of sequence s starts at row cu_s + C (g - chunk0_s)
            const long long base = (long long)cu_seqlens[s0] - (long long)CH * seqs[size_t(s0)].chunk0;
            if (base > kNoRowBase && base <= INT32_MAX) ranges[size_t(wv)].row0_base = int32_t(base);
        }
    }
    char *ws = static_cast<char *>(workspace);
    {
        // the three tables laid out as in the workspace, then one copy
        const size_t end = cks.empty() ? L.chunks + sizeof(ChunkMeta) * chunks.size()
                                       : L.ckpts + sizeof(CkptMeta) * cks.size();
        std::vector<char> host(end, 0);
        if (N > 0) std::memcpy(host.data() + L.seqs, seqs.data(), sizeof(SeqMeta) * seqs.size());
        if (!chunks.empty()) std::memcpy(host.data() + L.chunks, chunks.data(), sizeof(ChunkMeta) * chunks.size());
        if (!cks.empty()) std::memcpy(host.data() + L.ckpts, cks.data(), sizeof(CkptMeta) * cks.size());
        const ProfScope prof(KDA_KERNEL_PREFILL_META, stream);  // the host tables' copy to the device
        if (end > 0 && cudaMemcpyAsync(ws, host.data(), end, cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    // the intra variant that finishes one-chunk sequences itself: where they
    // are at least a sixteenth of the chunks (elsewhere its path costs more
    // than the chain steps it saves)
    long long n_solo = 0;
    for (int s = 0; s < N; ++s) n_solo += (seqs[s].n_chunks == 1 && !seqs[s].has_init) ? 1 : 0;
    const bool solo = n_solo > 0 && 16 * n_solo >= n_chunks;
    return launch_tables(pool, w, io, ws, L, N, n_reqs, n_chunks, cu_seqlens[N], &ranges, solo, stream);
}

size_t prefill_workspace_bytes_bound(const kda_pool *pool, int N, int max_tokens, int n_reqs, int chunk) {
    if (chunk != CH || pool->desc.d_k != D || pool->desc.d_v != D || N < 0 || max_tokens < 0 || n_reqs < 0) return 0;
    const long long mc = max_tokens / CH + N;
    return pf::ws_layout_dev(N, mc, n_reqs, pool->desc.num_heads, pool->desc.num_slots, pf::preferred_window(mc)).total;
}

kda_status launch_prefill_dev(const kda_pool *pool, const kda_weights *w, const kda_io *io, const int32_t *cu_seqlens,
                              const int32_t *slots, const uint8_t *has_initial_state, int N, int max_tokens,
                              int chunk, const kda_ckpt_req *reqs, int n_reqs, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
    using namespace pf;
    if (pool->desc.d_k != D || pool->desc.d_v != D || chunk != CH) return KDA_ERR_UNSUPPORTED;
    const int H = pool->desc.num_heads;
    // every sequence adds at most one partial chunk to max_tokens / CH whole ones
    const long long max_chunks = max_tokens / CH + N;
    if (max_chunks > (1LL << 31) / std::max(H, 1)) return KDA_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % 256) != 0) return KDA_ERR_WORKSPACE;
    const int ns = pool->desc.num_slots;
    const int window = fit_window(workspace_bytes, max_chunks,
                                  [&](int wv) { return ws_layout_dev(N, max_chunks, n_reqs, H, ns, wv).total; });
    if (window == 0) return KDA_ERR_WORKSPACE;
    const WsLayoutDev LD = ws_layout_dev(N, max_chunks, n_reqs, H, ns, window);
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
    a.num_slots = ns;
    a.seqs = reinterpret_cast<SeqMeta *>(ws + LD.L.seqs);
    a.chunks = reinterpret_cast<ChunkMeta *>(ws + LD.L.chunks);
    a.ckpts = reinterpret_cast<CkptMeta *>(ws + LD.L.ckpts);
    a.used = reinterpret_cast<uint32_t *>(ws + LD.used);
    a.err = pool->err;
    {
        const ProfScope prof(KDA_KERNEL_PREFILL_META, stream);
        prefill_meta_kernel<<<1, kMetaThreads, 0, stream>>>(a);
    }
    // device tables: the one-chunk variant when sequences may average 16 chunks or fewer
    return launch_tables(pool, w, io, ws, LD.L, N, n_reqs, max_chunks, max_tokens, nullptr,
                         N > 0 && 16LL * N >= max_chunks, stream);
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
    // cleared; the windows of chunks shrink to fit the array, and a call whose
    // tables and smallest window do not fit returns KDA_ERR_WORKSPACE.
    return launch_prefill(pool, w, io, cu_seqlens, slots, has_initial_state, N, chunk, reqs, n_reqs, ptr,
                          KDA_NOALLOC_SCRATCH_BYTES, stream);
}

}  // namespace kda
