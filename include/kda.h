/*
 * kda.h -- C ABI of libkda: the KDA (Kimi Delta Attention) layer step on one
 * GB300 (sm_103a).
 *
 * The layer step, per sequence and per head h, for each token t:
 *   conv   y = silu(sum_{j<4} w[c][j] * x_{t-3+j}[c]) on every raw q, k, v
 *          channel c (depthwise causal conv of width 4, last tap on the
 *          current token, no bias; the 3 previous raw inputs are the slot's
 *          "conv tail")
 *   L2     q <- q / sqrt(|q|^2 + eps_l2), k <- k / sqrt(|k|^2 + eps_l2)
 *   update S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   read   o_t = S_t^T q_t
 *   norm   y_t = w_n * o_t / sqrt(mean(o_t^2) + eps_rms) * sigmoid(g_t)
 * Sources: "vLLM Kimi K3 지원" (agentlenshq.com), section "Kimi K3 아키텍처 개요"
 * (KDA: linear attention over a fixed-size recurrent state) and section
 * "Fused Kernels 및 메타데이터 최적화" (the decode step fuses causal conv,
 * recurrent update and RMSNorm in one launch; prefill runs chunked).  The
 * pages do not print the recurrence; the formula above is the KDA step this
 * library implements.
 *
 * Conventions shared by every entry point
 *   - Device memory is owned by the caller: the pool buffer, inputs, outputs
 *     and workspaces are plain device pointers.  The library allocates no
 *     device memory at run time (the no-allocation prefill's fixed scratch is
 *     a static array of the module image).  A pool handle owns host metadata
 *     only; a prefix cache handle owns host memory only.
 *   - Calls that take a stream are asynchronous on that stream.  A host-side
 *     argument error returns a status synchronously and enqueues nothing.
 *   - A fault found on the device (a slot index out of range) sets a bit of
 *     the pool's device error word and the affected item is skipped; read it
 *     with kda_poll_device_error.  No kernel traps.
 *   - Not thread-safe per pool unless the callers order their streams.
 *   - Activations, conv weights, norm weight and the conv tail share one
 *     dtype (pool "act": fp32 or bf16).  State is always fp32.
 *
 * Pool layout (one caller buffer of kda_state_pool_bytes bytes, 256-aligned):
 *   [0, 256)             header; the uint32 device error word at offset 0
 *   states               [num_slots][H][d_v][d_k] fp32: each head's state
 *                        stored transposed, S^T, row j = value channel j,
 *                        d_k key channels contiguous
 *   tails (256-aligned)  [num_slots][3][n_ch] act, n_ch = H*(2*d_k + d_v):
 *                        the 3 previous raw inputs, oldest first; channels
 *                        q (h*d_k+i), then k (H*d_k+h*d_k+i), then
 *                        v (2*H*d_k+h*d_v+j)
 *   A slot that holds zeros is the state of a new sequence.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KDA_API __attribute__((visibility("default")))
#else
#define KDA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA stream type (same object as cudaStream_t). */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad shape, bad dtype */
    KDA_ERR_SLOT_RANGE = 2,  /* a host-visible slot index outside [0, num_slots) */
    KDA_ERR_ALIAS = 3,       /* the same slot written twice, or read and written by different items */
    KDA_ERR_UNSUPPORTED = 4, /* a legal shape this build has no kernel for */
    KDA_ERR_CUDA = 5,        /* a CUDA runtime call failed */
    KDA_ERR_DEVICE = 6,      /* the device error word was set (kda_poll_device_error) */
    KDA_ERR_WORKSPACE = 7,   /* workspace missing, misaligned or too small */
    KDA_ERR_HOST_MEMORY = 8, /* a host allocation failed */
    KDA_ERR_TIMEOUT = 9      /* kda_stream_wait: the stream's work had not finished in time */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Device error word bits. */
#define KDA_DEVERR_SLOT_RANGE 0x1u /* a device-side slot index was out of range */
#define KDA_DEVERR_META 0x2u       /* prefill metadata inconsistent on the device */
#define KDA_DEVERR_TIMEOUT 0x4u    /* a bounded wait inside a kernel gave up */

typedef struct {
    int32_t num_slots;  /* > 0 */
    int32_t num_heads;  /* H > 0 */
    int32_t d_k;        /* key channels per head */
    int32_t d_v;        /* value channels per head */
    int32_t conv_width; /* must be 4 */
    int32_t act;        /* kda_dtype of activations, weights and conv tail */
} kda_pool_desc;

typedef struct {
    size_t header_offset; /* error word at this byte offset */
    size_t state_offset;  /* byte offset of slot 0's state */
    size_t state_slot_bytes;
    size_t tail_offset;   /* byte offset of slot 0's conv tail */
    size_t tail_slot_bytes;
    size_t total_bytes;
} kda_pool_layout;

/* Layer weights (device pointers, act dtype). */
typedef struct {
    const void *conv_w; /* [n_ch][4]: row c holds channel c's taps, tap 3 on the current token; 16-byte aligned */
    const void *norm_w; /* [d_v], shared by all heads */
    float eps_l2;       /* added under the root of the q/k L2 norm (1e-6) */
    float eps_rms;      /* added under the root of the RMSNorm (1e-5) */
} kda_weights;

/* Per-token tensors (device pointers, act dtype), token-major.  For decode a
 * token is a sequence of the batch; for verify token (b, t) is row b*T + t;
 * for prefill the sequences are packed back to back (cu_seqlens). */
typedef struct {
    const void *q;     /* [n_tok][H][d_k] raw projections (before the conv) */
    const void *k;     /* [n_tok][H][d_k] */
    const void *v;     /* [n_tok][H][d_v] */
    const void *alpha; /* [n_tok][H][d_k] decay values in (0, 1] */
    const void *beta;  /* [n_tok][H] write strengths in [0, 1] */
    const void *gate;  /* [n_tok][H][d_v] output-gate logits */
    void *out;         /* [n_tok][H][d_v] gated, normalised output */
} kda_io;

/* A state checkpoint taken inside a prefill: after the first token_pos tokens
 * of sequence seq's segment, copy its state and conv tail into dst_slot.
 * token_pos is > 0 and either a multiple of the chunk size or the segment
 * length. */
typedef struct {
    int32_t seq;
    int32_t token_pos;
    int32_t dst_slot;
} kda_ckpt_req;

typedef struct kda_pool kda_pool;

/* Bytes a pool with this description needs; 0 if the description is invalid.
 * Source: "vLLM Kimi K3 지원", section "하이브리드 KV-Cache 관리" (compact KDA
 * recurrent-state blocks next to the paged KV blocks) and the DSpark page's
 * FP32 state cache ("Kimi K3 ... 842 tok/s", section "시간은 어디에 쓰였나"). */
KDA_API size_t kda_state_pool_bytes(const kda_pool_desc *desc);

/* Wraps a caller-owned device buffer (>= kda_state_pool_bytes, 256-aligned)
 * as a slot pool.  Does not clear it: the caller zeroes the buffer (or the
 * slots it hands to new sequences).  On success *out owns host metadata only;
 * free it with kda_state_pool_destroy.  Errors: KDA_ERR_INVALID_ARG,
 * KDA_ERR_UNSUPPORTED (dims without a kernel), KDA_ERR_CUDA. */
KDA_API kda_status kda_state_pool_create(const kda_pool_desc *desc, void *dev_buf, size_t bytes,
                                 kda_pool **out);

/* Frees the handle (not the caller's buffer).  NULL is ignored. */
KDA_API void kda_state_pool_destroy(kda_pool *pool);

/* Launch options of a pool's kda_decode / kda_verify calls (flags of
 * kda_state_pool_set_flags; 0, the default, sets none).
 * KDA_POOL_OVERLAP_INPUTS: each launch starts under the preceding kernel on
 *   its stream (programmatic dependent launch) and reads its slot tables,
 *   beta, weights and token inputs before that kernel has completed; only the
 *   pool (state and conv tail) is read after it.  The caller guarantees that
 *   the preceding kernel on the stream writes none of those inputs, e.g. a
 *   chain of decode steps whose inputs were staged beforehand.  Without the
 *   flag every input is read after the preceding kernel has completed, so any
 *   kernel (a q/k/v projection) may produce the inputs right before the call.
 * Returns KDA_ERR_INVALID_ARG for a null pool or an unknown flag. */
#define KDA_POOL_OVERLAP_INPUTS 0x1u
KDA_API kda_status kda_state_pool_set_flags(kda_pool *pool, uint32_t flags);

/* Byte offsets of the pool regions (see the layout above). */
KDA_API kda_status kda_state_pool_layout(const kda_pool *pool, kda_pool_layout *out);

/* Host-side validation of slot tables before they are used on the device.
 * in_slots [n_in] and out_slots [n_out] are HOST arrays (either may be NULL
 * with its count 0).  Fails with KDA_ERR_SLOT_RANGE if an index is outside
 * [0, num_slots), with KDA_ERR_ALIAS if out_slots repeats a slot, if in_slots
 * repeats a slot, or if out slot i*per_item + t equals an in slot other than
 * in_slots[i] (per_item = n_out / n_in when n_in > 0).  Enqueues nothing. */
KDA_API kda_status kda_check_slots(const kda_pool *pool, const int32_t *in_slots, int32_t n_in,
                           const int32_t *out_slots, int32_t n_out);

/* One decode step for a batch of B sequences: token b of io advances the
 * state and conv tail of slot slots[b] in place and writes out[b].  slots is a
 * DEVICE array [B] (so the call can sit in a CUDA graph); an index outside the
 * pool sets KDA_DEVERR_SLOT_RANGE and that sequence is skipped.  Slots must be
 * distinct (check with kda_check_slots).  B = 0 is a no-op.
 * One launch: conv, L2, update, readout and gated norm are fused.
 * The launch may start while the preceding kernel on its stream finishes
 * (programmatic dependent launch); it reads nothing until that kernel has
 * completed, unless the pool has KDA_POOL_OVERLAP_INPUTS set (see
 * kda_state_pool_set_flags for that contract).
 * Source: "vLLM Kimi K3 지원", section "Fused Kernels 및 메타데이터 최적화",
 * KDA Decode bullet. */
KDA_API kda_status kda_decode(kda_pool *pool, const kda_weights *w, const kda_io *io,
                      const int32_t *slots, int32_t B, kda_stream_t stream);

/* Asks L2 to fetch the state and conv tail of slots[0..B) (a DEVICE array)
 * ahead of a kda_decode / kda_verify that reads them, for example one layer
 * early while other layers run: a decode whose state has left L2 otherwise
 * waits on a chain of round trips to HBM.  With w non-null the layer's conv
 * taps and norm weight are fetched too (w is checked like kda_decode's; NULL
 * fetches the slots only).  A hint: results never depend on it, it changes
 * no memory, and a slot outside the pool is skipped.  It pays while the
 * prefetched slots fit in L2 (129 MB; a slot is 4.3 MB at H = 64, d = 128,
 * bf16), so small batches.  One small kernel on `stream`; B = 0 is a no-op.
 * Errors: KDA_ERR_INVALID_ARG (null pool or slots, B < 0, bad weights),
 * KDA_ERR_CUDA.
 * Source: "vLLM Kimi K3 지원", section "Fused Kernels 및 메타데이터 최적화",
 * KDA Decode bullet (the decode step is bound by its repeated state traffic). */
KDA_API kda_status kda_state_prefetch(kda_pool *pool, const kda_weights *w, const int32_t *slots, int32_t B,
                                      kda_stream_t stream);

/* Speculative verify: B sequences each advance T draft tokens (1 <= T <= 16)
 * in one launch.  Token (b, t) is io row b*T + t.  Sequence b starts from slot
 * in_slots[b] (DEVICE [B]); after its token t the state and conv tail are
 * written to slot snap_slots[b*T + t] (DEVICE [B*T]) and the output to row
 * b*T + t.  in_slots[b] is read before any write, so it may equal any of its
 * own snapshot slots.  Rollback to an accepted length a (1 <= a <= T) is the
 * caller adopting snap_slots[b*T + a - 1]: no device work.  Snapshot slots
 * must be distinct and must not be another sequence's in slot.
 * Source: "vLLM Kimi K3 지원", section "DSpark를 이용한 Speculative Decoding", and
 * "vLLM Kimi-K3 DSpark 사전 해석 구현", section "추론 성능 및 기능" (8 draft
 * tokens per step). */
KDA_API kda_status kda_verify(kda_pool *pool, const kda_weights *w, const kda_io *io,
                      const int32_t *in_slots, const int32_t *snap_slots, int32_t B, int32_t T,
                      kda_stream_t stream);

/* Workspace bytes kda_prefill_chunked prefers for these sequence lengths
 * (cu_seqlens: HOST [N+1], nondecreasing from 0).  0 on invalid input.
 * The workspace holds the sequence, chunk and checkpoint tables and a ring
 * of per-(chunk, head) records (145 KiB each at d = 128) for two windows of
 * at most 48 chunks, so it is bounded by the window, not the prompt: about
 * 0.9 GB for any prompt length at H = 64 (the tables add 24 B per chunk). */
KDA_API size_t kda_prefill_workspace_bytes(const kda_pool *pool, const int32_t *cu_seqlens, int32_t N,
                                   int32_t chunk);

/* Chunked prefill of N packed sequences.  Sequence n owns io rows
 * [cu_seqlens[n], cu_seqlens[n+1]) and slot slots[n]; it starts from that
 * slot's state and tail when has_initial_state[n] != 0, else from zeros, and
 * leaves its end state and tail in the slot.  Chunks of `chunk` tokens (64)
 * are aligned to each segment's first token.  reqs[n_reqs] asks for state
 * checkpoints (see kda_ckpt_req); the destinations must be distinct, must
 * not be a slot of this call, and a sequence's end may be checkpointed too.
 * cu_seqlens, slots, has_initial_state and reqs are HOST arrays (checked
 * here: KDA_ERR_SLOT_RANGE, KDA_ERR_ALIAS, KDA_ERR_INVALID_ARG).
 * workspace: device, 256-aligned.  With kda_prefill_workspace_bytes bytes the
 * call runs in its preferred windows; a smaller workspace runs it in smaller
 * windows (down to one chunk), with the same results bit for bit, and one too
 * small for the tables plus a ring of one-chunk windows returns
 * KDA_ERR_WORKSPACE with nothing enqueued.
 * Source: "vLLM Kimi K3 지원", section "Fused Kernels 및 메타데이터 최적화",
 * KDA Prefill bullet (FlashKDA), and section "에이전틱 캐시 유지 정책"
 * (interval-based retention: checkpoints every 32K tokens and at prompt
 * boundaries). */
KDA_API kda_status kda_prefill_chunked(kda_pool *pool, const kda_weights *w, const kda_io *io,
                               const int32_t *cu_seqlens, const int32_t *slots,
                               const uint8_t *has_initial_state, int32_t N, int32_t chunk,
                               const kda_ckpt_req *reqs, int32_t n_reqs, void *workspace,
                               size_t workspace_bytes, kda_stream_t stream);

/* Size of the fixed scratch array behind kda_prefill_chunked_noalloc. */
#define KDA_NOALLOC_SCRATCH_BYTES (64u << 20)

/* kda_prefill_chunked without a caller workspace, for callers that cannot
 * allocate device memory: for example a plugin whose host runtime reserves
 * all device memory up front and hands none out, or a C caller with no
 * device allocator of its own.  The pages have no counterpart for this
 * entry point; it exists for such callers only.
 * Arguments, results and errors are those of kda_prefill_chunked, except
 * that the scratch is a fixed array of KDA_NOALLOC_SCRATCH_BYTES (64 MiB)
 * compiled into the library: every GPU that loads the library holds it
 * until the process exits, and no call allocates or frees device memory.
 * The call runs in the largest windows the array holds (see
 * kda_prefill_chunked's workspace), so prompts of any length fit at H = 64;
 * a call whose tables plus a ring of one-chunk windows exceed the array (at
 * d = 128, more than about 450 heads) returns KDA_ERR_WORKSPACE and enqueues
 * nothing.
 * Every call looks up the array's device address with the call's device
 * current (so a device reset that reloads the library's module leaves no
 * stale address behind).  The first lookup on a device may load the module:
 * make the first call on each device before any stream capture.
 * Every call uses the same array and leaves its contents behind; each call
 * writes every scratch byte it reads, so nothing needs clearing.  Calls that
 * overlap on one GPU (other streams, other threads) race on the array:
 * order them. */
KDA_API kda_status kda_prefill_chunked_noalloc(kda_pool *pool, const kda_weights *w, const kda_io *io,
                                               const int32_t *cu_seqlens, const int32_t *slots,
                                               const uint8_t *has_initial_state, int32_t N, int32_t chunk,
                                               const kda_ckpt_req *reqs, int32_t n_reqs, kda_stream_t stream);

/* kda_prefill_chunked with its metadata in DEVICE memory, for callers whose
 * sequence tables live on the GPU and for CUDA graph capture: the call
 * enqueues no host-to-device copy.  The sequence, chunk and checkpoint tables
 * are built on the stream by one kernel, with the rules kda_prefill_chunked
 * checks on the host.  Source: "vLLM Kimi K3 지원", section "Fused Kernels 및
 * 메타데이터 최적화", Metadata Builder bullet (the KDA metadata prepared by
 * one fused GPU kernel).
 * cu_seqlens: device int32 [N + 1]; slots: device int32 [N];
 * has_initial_state: device uint8 [N]; reqs: device kda_ckpt_req [n_reqs].
 * N, n_reqs: host counts.  max_tokens: host bound on cu_seqlens[N]; q, k, v,
 *   alpha, beta, gate and out must have max_tokens rows (rows past
 *   cu_seqlens[N] may be read, are never written and never affect results).
 * workspace: device, 256-aligned, >= kda_prefill_workspace_bytes_bound(pool,
 *   N, max_tokens, n_reqs, chunk) bytes (sized from the bounds, so the host
 *   needs no sequence lengths).
 * Host errors: those of kda_prefill_chunked that need no device data
 *   (KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE).
 * Device errors: cu_seqlens not starting at 0, decreasing or past max_tokens,
 *   a request at a bad sequence or position, or a repeated slot set
 *   KDA_DEVERR_META; a slot out of range sets KDA_DEVERR_SLOT_RANGE.  Either
 *   way the call then changes no slot and writes no output (read the error
 *   word with kda_poll_device_error).
 * Cost: the builder is one 1024-thread CTA; it ranks the requests by
 *   comparing every pair, so its time grows with n_reqs^2 / 1024 (a few
 *   microseconds for hundreds of requests). */
KDA_API size_t kda_prefill_workspace_bytes_bound(const kda_pool *pool, int32_t N, int32_t max_tokens, int32_t n_reqs,
                                                 int32_t chunk);
KDA_API kda_status kda_prefill_chunked_dev(kda_pool *pool, const kda_weights *w, const kda_io *io,
                                           const int32_t *cu_seqlens, const int32_t *slots,
                                           const uint8_t *has_initial_state, int32_t N, int32_t max_tokens,
                                           int32_t chunk, const kda_ckpt_req *reqs, int32_t n_reqs, void *workspace,
                                           size_t workspace_bytes, kda_stream_t stream);

/* Copies state and conv tail of src_slots[i] into dst_slots[i], bit-exact,
 * for i < n (HOST arrays).  Restoring a checkpoint is the same call with the
 * roles swapped.  dst slots must be distinct and must not appear among the
 * sources.  Source: "vLLM Kimi K3 지원", section "에이전틱 캐시 유지 정책". */
KDA_API kda_status kda_state_checkpoint(kda_pool *pool, const int32_t *src_slots,
                                const int32_t *dst_slots, int32_t n, kda_stream_t stream);

/* Request-level state transfer between a slot and host memory: the state
 * (fp32 [H][d_v][d_k], S^T per head) followed by the conv tail (act
 * [3][n_ch]), kda_state_slot_bytes() bytes in all, copied bit-exactly.  It is
 * the single-GPU side of moving a request's KDA state between prefill and
 * decode replicas.  Source: "vLLM Kimi K3 지원", section "Prefill/Decode 분리
 * (Disaggregation)" (request-level KDA state transfer).
 * host: HOST buffer of at least kda_state_slot_bytes(pool) bytes, owned by
 *       the caller; page-locked memory makes the copies asynchronous, other
 *       host memory makes them return once the data is staged.  The buffer
 *       must stay valid (and, for import, unchanged) until the stream has
 *       executed the copies.
 * Errors: KDA_ERR_INVALID_ARG (null pool / host, bytes too small),
 *         KDA_ERR_SLOT_RANGE (slot outside the pool), KDA_ERR_CUDA. */
KDA_API size_t kda_state_slot_bytes(const kda_pool *pool);
KDA_API kda_status kda_state_export(kda_pool *pool, int32_t slot, void *host, size_t bytes, kda_stream_t stream);
KDA_API kda_status kda_state_import(kda_pool *pool, int32_t slot, const void *host, size_t bytes,
                                    kda_stream_t stream);

/* ---- Prefix-state cache with second-hit admission (host only) ----------
 * Decides, per prompt, which saved KDA state to resume from and where to
 * save a new one.  Source: "vLLM Kimi K3 지원", section "하이브리드 KV-Cache
 * 관리" (KDA state blocks kept apart from prefix matching, so a shared
 * prompt reuses the saved state) and section "에이전틱 캐시 유지 정책"
 * (Marconi-style selective retention: a prefix's state is saved only on the
 * prefix's second hit).
 *
 * A prefix is the first i * block tokens of a prompt (block: a positive
 * multiple of the chunk length 64), so every saved state is a checkpoint at
 * a chunk end.  kda_prefix_cache_plan, for a prompt of n token ids:
 *   - counts one hit on each of its n / block prefixes;
 *   - hit_len / hit_slot: the longest saved prefix of at most n - 1 tokens
 *     (0 / -1 if none).  The caller copies hit_slot into the request's slot
 *     (kda_state_checkpoint) and prefills tokens [hit_len, n) with
 *     has_initial_state = 1;
 *   - admit_pos / admit_slot: at most one longer prefix with two or more hits
 *     and no saved state (-1 / -1 if none).  The caller adds the checkpoint
 *     request {seq, admit_pos - hit_len, admit_slot} to that prefill, which
 *     writes the state there.
 * Admission slots come from the cache's list, lowest free first; with none
 * free, the least recently counted saved prefix other than the reused one
 * gives its slot up (it stays tracked, unsaved, with its hits); with no such
 * prefix nothing is admitted.  Unsaved prefixes beyond max_tracked are
 * dropped, least recently counted first, at the end of each plan.  A saved
 * prefix keeps its tokens, so only an exact match resumes from it.
 * The slots are pool slots the caller sets aside for the cache; the device
 * copies and prefills that use a plan go on one stream (or are ordered by
 * the caller), which keeps a slot from being overwritten before an earlier
 * copy from it has run.  Not thread-safe.
 * Errors: KDA_ERR_INVALID_ARG (null pointer, negative count, block not a
 * positive multiple of 64; forget of a slot holding no saved prefix),
 * KDA_ERR_SLOT_RANGE (a negative slot), KDA_ERR_ALIAS (a slot listed twice),
 * KDA_ERR_HOST_MEMORY (a plan or forget that fails this way may leave the
 * cache partly updated: destroy it and start a new one). */
typedef struct kda_prefix_cache kda_prefix_cache;
typedef struct {
    int32_t hit_len, hit_slot, admit_pos, admit_slot;
} kda_prefix_plan;
typedef struct {
    int64_t plans, hits, admissions, evictions; /* hits: plans that reused a state */
    int64_t n_saved, n_unsaved, n_free;
} kda_prefix_cache_stats;
KDA_API kda_status kda_prefix_cache_create(int32_t block, const int32_t *slots, int32_t n_slots, int32_t max_tracked,
                                           kda_prefix_cache **out);
KDA_API void kda_prefix_cache_destroy(kda_prefix_cache *cache);
KDA_API kda_status kda_prefix_cache_plan(kda_prefix_cache *cache, const int32_t *tokens, int32_t n,
                                         kda_prefix_plan *out);
/* Gives up the state saved in `slot` (e.g. its prefill was abandoned): the
 * slot returns to the free list and the prefix stays tracked, unsaved. */
KDA_API kda_status kda_prefix_cache_forget(kda_prefix_cache *cache, int32_t slot);
KDA_API kda_status kda_prefix_cache_get_stats(const kda_prefix_cache *cache, kda_prefix_cache_stats *out);
/* Writes up to cap (prefix length, slot) pairs of the saved prefixes, least
 * recently counted first; returns how many there are (-1 on a bad argument). */
KDA_API int32_t kda_prefix_cache_saved(const kda_prefix_cache *cache, int32_t *lens, int32_t *slots, int32_t cap);

/* Waits for `stream`, reads the device error word into *flags (may be NULL)
 * and clears it.  Returns KDA_ERR_DEVICE if any bit was set, else KDA_OK. */
KDA_API kda_status kda_poll_device_error(kda_pool *pool, kda_stream_t stream, uint32_t *flags);

/* Host watchdog: waits for the work enqueued on `stream` (NULL: the legacy
 * default stream) by polling it, for at most timeout_s seconds, instead of
 * blocking without limit.  KDA_OK once it has finished; KDA_ERR_TIMEOUT if it
 * has not (the work is still in flight and may yet finish; the caller
 * decides); KDA_ERR_CUDA if the stream reports an error; KDA_ERR_INVALID_ARG
 * for a negative or non-finite limit.  Every wait inside the kernels is
 * bounded too, so a stream the library alone feeds always finishes. */
KDA_API kda_status kda_stream_wait(kda_stream_t stream, double timeout_s);

/* ---- Device-time profile of the library's own kernels -------------------
 * A measurement aid; the pages have no counterpart.  Between
 * kda_profile_start and kda_profile_stop every kernel this library launches
 * (outside stream capture) is bracketed by two CUDA events recorded on the
 * stream it is launched on, so each interval is that kernel's device time as
 * it ran in the caller's schedule.  kda_profile_stop waits for the events
 * and reports, per kernel kind, the launches timed and their summed time.
 * max_launches (1 .. 2^20) bounds the events created (two per launch);
 * launches beyond it are counted in `dropped` and not timed.  One profile
 * per process at a time; the events belong to the device current at
 * kda_profile_start, so profile launches on that device only.  The events
 * serialise the launches they bracket with their neighbours on the stream
 * (a timed step launch no longer overlaps the one before it).
 * Errors: KDA_ERR_INVALID_ARG (a bad limit, start while running, stop while
 * stopped), KDA_ERR_CUDA (event creation or timing failed). */
typedef enum {
    KDA_KERNEL_STEP = 0,       /* kda_decode / kda_verify */
    KDA_KERNEL_SLOT_COPY,      /* kda_state_checkpoint */
    KDA_KERNEL_PREFILL_META,   /* prefill tables: the device builder (kda_prefill_chunked_dev), or the
                                  copies of the host-built tables (kda_prefill_chunked) */
    KDA_KERNEL_PREFILL_INTRA,  /* intra-chunk prefill kernel with the decay factored around the chunk's
                                  midpoint (bf16 inputs: every chunk-head of a window) */
    KDA_KERNEL_PREFILL_CHAIN,  /* the chunk chain (state passing, gated norm of the outputs) */
    KDA_KERNEL_PREFILL_OUT,    /* unused (the chain applies the gated norm); keeps the values below */
    KDA_KERNEL_PREFILL_TAILS,  /* conv tails of checkpoints and ends */
    KDA_KERNEL_STATE_PREFETCH, /* kda_state_prefetch */
    KDA_KERNEL_PREFILL_INTRA_EXACT, /* intra-chunk prefill kernel with per-pair decay exponents (bf16
                                  inputs: the chunk-heads the factored kernel hands over; fp32 inputs:
                                  every chunk-head) */
    KDA_KERNEL_COUNT
} kda_kernel_kind;
typedef struct {
    int64_t launches[KDA_KERNEL_COUNT];
    double ms[KDA_KERNEL_COUNT];
    int64_t dropped;
} kda_profile;
KDA_API kda_status kda_profile_start(int32_t max_launches);
KDA_API kda_status kda_profile_stop(kda_profile *out);

/* Static text for a status code. */
KDA_API const char *kda_status_string(kda_status s);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
