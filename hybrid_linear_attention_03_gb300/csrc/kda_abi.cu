// kda_abi.cu -- the C ABI of libkda: argument checks, the pool handle and
// dispatch to the kernels.  Declarations and contracts are in include/kda.h.
#include "kda_internal.h"

#include <nvtx3/nvToolsExt.h>

#include <chrono>
#include <cmath>
#include <cstring>
#include <new>
#include <thread>
#include <unordered_map>
#include <vector>

namespace {

// An NVTX range over an entry point that enqueues device work, so a profiler
// timeline shows the library's calls around their kernels (a no-op unless a
// tool is attached).
struct CallRange {
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

constexpr size_t kAlign = 256;
constexpr size_t kHeaderBytes = 256;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int act_bytes(int32_t act) { return act == KDA_BF16 ? 2 : (act == KDA_F32 ? 4 : 0); }

struct Layout {
    size_t state_off, state_slot, tail_off, tail_slot, total;
    long long n_ch;
};

bool compute_layout(const kda_pool_desc *d, Layout *L) {
    if (!d || d->num_slots <= 0 || d->num_heads <= 0 || d->d_k <= 0 || d->d_v <= 0 ||
        d->conv_width != kda::kConvWidth || act_bytes(d->act) == 0)
        return false;
    const long long n_ch = 1LL * d->num_heads * (2LL * d->d_k + d->d_v);
    if (n_ch > (1LL << 30)) return false;
    L->n_ch = n_ch;
    L->state_slot = sizeof(float) * size_t(d->num_heads) * size_t(d->d_v) * size_t(d->d_k);
    L->tail_slot = size_t(kda::kConvWidth - 1) * size_t(n_ch) * size_t(act_bytes(d->act));
    L->state_off = kHeaderBytes;
    L->tail_off = align_up(L->state_off + L->state_slot * size_t(d->num_slots), kAlign);
    L->total = align_up(L->tail_off + L->tail_slot * size_t(d->num_slots), kAlign);
    return true;
}

bool valid_weights(const kda_weights *w) {
    return w && w->conv_w && w->norm_w && aligned(w->conv_w, 16) && std::isfinite(w->eps_l2) &&
           std::isfinite(w->eps_rms) && w->eps_l2 >= 0.f && w->eps_rms >= 0.f;
}

bool valid_io(const kda_io *io) {
    if (!io || !io->q || !io->k || !io->v || !io->alpha || !io->beta || !io->gate || !io->out) return false;
    const void *ptrs[] = {io->q, io->k, io->v, io->alpha, io->gate, io->out};
    for (const void *p : ptrs)
        if (!aligned(p, 16)) return false;
    return true;
}

}  // namespace

extern "C" {

size_t kda_state_pool_bytes(const kda_pool_desc *desc) {
    Layout L;
    return compute_layout(desc, &L) ? L.total : 0;
}

kda_status kda_state_pool_create(const kda_pool_desc *desc, void *dev_buf, size_t bytes, kda_pool **out) {
    if (!out) return KDA_ERR_INVALID_ARG;
    *out = nullptr;
    Layout L;
    if (!compute_layout(desc, &L) || !dev_buf || !aligned(dev_buf, kAlign) || bytes < L.total)
        return KDA_ERR_INVALID_ARG;
    // The kernels cover d_k == d_v in {16, 32, 64, 128}.
    const int D = desc->d_k;
    if (desc->d_v != D || (D != 16 && D != 32 && D != 64 && D != 128)) return KDA_ERR_UNSUPPORTED;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, dev_buf) != cudaSuccess) {
        cudaGetLastError();
        return KDA_ERR_INVALID_ARG;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return KDA_ERR_INVALID_ARG;
    kda_pool *p = new (std::nothrow) kda_pool;
    if (!p) return KDA_ERR_INVALID_ARG;
    p->desc = *desc;
    p->base = static_cast<char *>(dev_buf);
    p->bytes = bytes;
    p->err = reinterpret_cast<uint32_t *>(p->base);
    p->states = reinterpret_cast<float *>(p->base + L.state_off);
    p->tails = p->base + L.tail_off;
    p->slot_state_elems = L.state_slot / sizeof(float);
    p->slot_tail_elems = L.tail_slot / size_t(act_bytes(desc->act));
    p->n_ch = int(L.n_ch);
    p->act_bytes = act_bytes(desc->act);
    p->device = attr.device;
    p->flags = 0;
    *out = p;
    return KDA_OK;
}

kda_status kda_state_pool_set_flags(kda_pool *pool, uint32_t flags) {
    if (!pool || (flags & ~uint32_t(KDA_POOL_OVERLAP_INPUTS)) != 0) return KDA_ERR_INVALID_ARG;
    pool->flags = flags;
    return KDA_OK;
}

void kda_state_pool_destroy(kda_pool *pool) { delete pool; }

kda_status kda_state_pool_layout(const kda_pool *pool, kda_pool_layout *out) {
    if (!pool || !out) return KDA_ERR_INVALID_ARG;
    Layout L;
    compute_layout(&pool->desc, &L);
    out->header_offset = 0;
    out->state_offset = L.state_off;
    out->state_slot_bytes = L.state_slot;
    out->tail_offset = L.tail_off;
    out->tail_slot_bytes = L.tail_slot;
    out->total_bytes = L.total;
    return KDA_OK;
}

kda_status kda_check_slots(const kda_pool *pool, const int32_t *in_slots, int32_t n_in,
                           const int32_t *out_slots, int32_t n_out) {
    if (!pool || n_in < 0 || n_out < 0 || (n_in > 0 && !in_slots) || (n_out > 0 && !out_slots))
        return KDA_ERR_INVALID_ARG;
    if (n_in > 0 && n_out > 0 && n_out % n_in != 0) return KDA_ERR_INVALID_ARG;
    const int32_t ns = pool->desc.num_slots;
    for (int32_t i = 0; i < n_in; ++i)
        if (in_slots[i] < 0 || in_slots[i] >= ns) return KDA_ERR_SLOT_RANGE;
    for (int32_t i = 0; i < n_out; ++i)
        if (out_slots[i] < 0 || out_slots[i] >= ns) return KDA_ERR_SLOT_RANGE;
    std::vector<int32_t> owner_in(size_t(ns), -1), seen_out(size_t(ns), 0);
    for (int32_t i = 0; i < n_in; ++i) {
        if (owner_in[in_slots[i]] >= 0) return KDA_ERR_ALIAS;
        owner_in[in_slots[i]] = i;
    }
    const int32_t per = n_in > 0 ? n_out / n_in : 0;
    for (int32_t i = 0; i < n_out; ++i) {
        const int32_t s = out_slots[i];
        if (seen_out[s]) return KDA_ERR_ALIAS;
        seen_out[s] = 1;
        if (n_in > 0 && owner_in[s] >= 0 && owner_in[s] != i / per) return KDA_ERR_ALIAS;
    }
    return KDA_OK;
}

static kda_status run_step(kda_pool *pool, const kda_weights *w, const kda_io *io, const int32_t *in_slots,
                           const int32_t *snap_slots, int32_t B, int32_t T, kda_stream_t stream) {
    if (!pool || !valid_weights(w) || !valid_io(io) || B < 0 || T < 1 || T > kda::kMaxVerifyT)
        return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;
    if (!in_slots || !snap_slots) return KDA_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * pool->desc.num_heads * 8 > 0x7fffffffLL) return KDA_ERR_INVALID_ARG;
    kda::StepParams p;
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
    p.in_slots = in_slots;
    p.snap_slots = snap_slots;
    p.B = B;
    p.T = T;
    p.H = pool->desc.num_heads;
    p.num_slots = pool->desc.num_slots;
    p.n_ch = pool->n_ch;
    p.early_inputs = (pool->flags & KDA_POOL_OVERLAP_INPUTS) ? 1 : 0;
    p.eps_l2 = w->eps_l2;
    p.eps_rms = w->eps_rms;
    return kda::launch_step(pool, p, reinterpret_cast<cudaStream_t>(stream));
}

kda_status kda_decode(kda_pool *pool, const kda_weights *w, const kda_io *io, const int32_t *slots, int32_t B,
                      kda_stream_t stream) {
    const CallRange range("kda_decode");
    return run_step(pool, w, io, slots, slots, B, 1, stream);
}

kda_status kda_state_prefetch(kda_pool *pool, const kda_weights *w, const int32_t *slots, int32_t B,
                              kda_stream_t stream) {
    const CallRange range("kda_state_prefetch");
    if (!pool || B < 0 || (B > 0 && !slots) || (w && !valid_weights(w))) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;
    return kda::launch_state_prefetch(pool, w, slots, B, reinterpret_cast<cudaStream_t>(stream));
}

kda_status kda_verify(kda_pool *pool, const kda_weights *w, const kda_io *io, const int32_t *in_slots,
                      const int32_t *snap_slots, int32_t B, int32_t T, kda_stream_t stream) {
    const CallRange range("kda_verify");
    return run_step(pool, w, io, in_slots, snap_slots, B, T, stream);
}

size_t kda_prefill_workspace_bytes(const kda_pool *pool, const int32_t *cu_seqlens, int32_t N, int32_t chunk) {
    if (!pool || !cu_seqlens || N < 0) return 0;
    return kda::prefill_workspace_bytes(pool, cu_seqlens, N, chunk);
}

// Host checks shared by both prefill entry points.
static kda_status check_prefill_args(kda_pool *pool, const kda_weights *w, const kda_io *io,
                                     const int32_t *cu_seqlens, const int32_t *slots,
                                     const uint8_t *has_initial_state, int32_t N, int32_t chunk,
                                     const kda_ckpt_req *reqs, int32_t n_reqs) {
    if (!pool || !valid_weights(w) || !valid_io(io) || N < 0 || n_reqs < 0 || (n_reqs > 0 && !reqs) ||
        (N > 0 && (!cu_seqlens || !slots || !has_initial_state)))
        return KDA_ERR_INVALID_ARG;
    if (N == 0) return n_reqs == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    if (cu_seqlens[0] != 0) return KDA_ERR_INVALID_ARG;
    for (int32_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ERR_INVALID_ARG;
    const int32_t ns = pool->desc.num_slots;
    std::vector<uint8_t> used(size_t(ns), 0);
    for (int32_t n = 0; n < N; ++n) {
        if (slots[n] < 0 || slots[n] >= ns) return KDA_ERR_SLOT_RANGE;
        if (used[slots[n]]) return KDA_ERR_ALIAS;
        used[slots[n]] = 1;
    }
    for (int32_t r = 0; r < n_reqs; ++r) {
        const kda_ckpt_req &q = reqs[r];
        if (q.seq < 0 || q.seq >= N) return KDA_ERR_INVALID_ARG;
        const int32_t len = cu_seqlens[q.seq + 1] - cu_seqlens[q.seq];
        if (q.token_pos <= 0 || q.token_pos > len || (q.token_pos != len && chunk > 0 && q.token_pos % chunk != 0))
            return KDA_ERR_INVALID_ARG;
        if (q.dst_slot < 0 || q.dst_slot >= ns) return KDA_ERR_SLOT_RANGE;
        if (used[q.dst_slot]) return KDA_ERR_ALIAS;
        used[q.dst_slot] = 1;
    }
    return KDA_OK;
}

size_t kda_prefill_workspace_bytes_bound(const kda_pool *pool, int32_t N, int32_t max_tokens, int32_t n_reqs,
                                         int32_t chunk) {
    if (!pool) return 0;
    return kda::prefill_workspace_bytes_bound(pool, N, max_tokens, n_reqs, chunk);
}

kda_status kda_prefill_chunked_dev(kda_pool *pool, const kda_weights *w, const kda_io *io, const int32_t *cu_seqlens,
                                   const int32_t *slots, const uint8_t *has_initial_state, int32_t N,
                                   int32_t max_tokens, int32_t chunk, const kda_ckpt_req *reqs, int32_t n_reqs,
                                   void *workspace, size_t workspace_bytes, kda_stream_t stream) {
    const CallRange range("kda_prefill_chunked_dev");
    if (!pool || !valid_weights(w) || !valid_io(io) || N < 0 || n_reqs < 0 || max_tokens < 0 ||
        (n_reqs > 0 && !reqs) || (N > 0 && (!cu_seqlens || !slots || !has_initial_state)))
        return KDA_ERR_INVALID_ARG;
    if (N == 0) return n_reqs == 0 ? KDA_OK : KDA_ERR_INVALID_ARG;
    return kda::launch_prefill_dev(pool, w, io, cu_seqlens, slots, has_initial_state, N, max_tokens, chunk, reqs,
                                   n_reqs, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

kda_status kda_prefill_chunked_noalloc(kda_pool *pool, const kda_weights *w, const kda_io *io,
                                       const int32_t *cu_seqlens, const int32_t *slots,
                                       const uint8_t *has_initial_state, int32_t N, int32_t chunk,
                                       const kda_ckpt_req *reqs, int32_t n_reqs, kda_stream_t stream) {
    const CallRange range("kda_prefill_chunked_noalloc");
    const kda_status st = check_prefill_args(pool, w, io, cu_seqlens, slots, has_initial_state, N, chunk, reqs, n_reqs);
    if (st != KDA_OK || N == 0) return st;
    return kda::launch_prefill_noalloc(pool, w, io, cu_seqlens, slots, has_initial_state, N, chunk, reqs, n_reqs,
                                       reinterpret_cast<cudaStream_t>(stream));
}

kda_status kda_prefill_chunked(kda_pool *pool, const kda_weights *w, const kda_io *io, const int32_t *cu_seqlens,
                               const int32_t *slots, const uint8_t *has_initial_state, int32_t N, int32_t chunk,
                               const kda_ckpt_req *reqs, int32_t n_reqs, void *workspace, size_t workspace_bytes,
                               kda_stream_t stream) {
    const CallRange range("kda_prefill_chunked");
    const kda_status st = check_prefill_args(pool, w, io, cu_seqlens, slots, has_initial_state, N, chunk, reqs, n_reqs);
    if (st != KDA_OK || N == 0) return st;
    return kda::launch_prefill(pool, w, io, cu_seqlens, slots, has_initial_state, N, chunk, reqs, n_reqs,
                               workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

kda_status kda_state_checkpoint(kda_pool *pool, const int32_t *src_slots, const int32_t *dst_slots, int32_t n,
                                kda_stream_t stream) {
    const CallRange range("kda_state_checkpoint");
    if (!pool || n < 0 || (n > 0 && (!src_slots || !dst_slots))) return KDA_ERR_INVALID_ARG;
    if (n == 0) return KDA_OK;
    const int32_t ns = pool->desc.num_slots;
    std::vector<uint8_t> is_src(size_t(ns), 0), is_dst(size_t(ns), 0);
    for (int32_t i = 0; i < n; ++i) {
        if (src_slots[i] < 0 || src_slots[i] >= ns || dst_slots[i] < 0 || dst_slots[i] >= ns)
            return KDA_ERR_SLOT_RANGE;
        is_src[src_slots[i]] = 1;
    }
    for (int32_t i = 0; i < n; ++i) {
        if (is_dst[dst_slots[i]] || is_src[dst_slots[i]]) return KDA_ERR_ALIAS;
        is_dst[dst_slots[i]] = 1;
    }
    return kda::launch_slot_copy(pool, src_slots, dst_slots, n, reinterpret_cast<cudaStream_t>(stream));
}

size_t kda_state_slot_bytes(const kda_pool *pool) {
    if (!pool) return 0;
    return pool->slot_state_elems * sizeof(float) + pool->slot_tail_elems * size_t(pool->act_bytes);
}

static kda_status slot_transfer(kda_pool *pool, int32_t slot, void *host, size_t bytes, bool to_host,
                                kda_stream_t stream) {
    if (!pool || !host || bytes < kda_state_slot_bytes(pool)) return KDA_ERR_INVALID_ARG;
    if (slot < 0 || slot >= pool->desc.num_slots) return KDA_ERR_SLOT_RANGE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t sb = pool->slot_state_elems * sizeof(float), tb = pool->slot_tail_elems * size_t(pool->act_bytes);
    char *dst_state = reinterpret_cast<char *>(pool->states) + size_t(slot) * sb;
    char *dst_tail = static_cast<char *>(pool->tails) + size_t(slot) * tb;
    char *h = static_cast<char *>(host);
    const cudaError_t e1 = to_host ? cudaMemcpyAsync(h, dst_state, sb, cudaMemcpyDeviceToHost, s)
                                   : cudaMemcpyAsync(dst_state, h, sb, cudaMemcpyHostToDevice, s);
    if (e1 != cudaSuccess) return KDA_ERR_CUDA;
    const cudaError_t e2 = to_host ? cudaMemcpyAsync(h + sb, dst_tail, tb, cudaMemcpyDeviceToHost, s)
                                   : cudaMemcpyAsync(dst_tail, h + sb, tb, cudaMemcpyHostToDevice, s);
    return e2 == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status kda_state_export(kda_pool *pool, int32_t slot, void *host, size_t bytes, kda_stream_t stream) {
    const CallRange range("kda_state_export");
    return slot_transfer(pool, slot, host, bytes, true, stream);
}

kda_status kda_state_import(kda_pool *pool, int32_t slot, const void *host, size_t bytes, kda_stream_t stream) {
    const CallRange range("kda_state_import");
    return slot_transfer(pool, slot, const_cast<void *>(host), bytes, false, stream);
}

kda_status kda_poll_device_error(kda_pool *pool, kda_stream_t stream, uint32_t *flags) {
    if (!pool) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, pool->err, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(pool->err, 0, sizeof(word), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (flags) *flags = word;
    return word ? KDA_ERR_DEVICE : KDA_OK;
}

kda_status kda_stream_wait(kda_stream_t stream, double timeout_s) {
    if (!(timeout_s >= 0.0) || !std::isfinite(timeout_s)) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        const cudaError_t q = cudaStreamQuery(s);
        if (q == cudaSuccess) return KDA_OK;
        if (q != cudaErrorNotReady) {
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() > timeout_s)
            return KDA_ERR_TIMEOUT;
        std::this_thread::sleep_for(std::chrono::microseconds(20));
    }
}

const char *kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_SLOT_RANGE: return "slot index out of range";
        case KDA_ERR_ALIAS: return "slot aliasing";
        case KDA_ERR_UNSUPPORTED: return "unsupported shape";
        case KDA_ERR_CUDA: return "CUDA runtime error";
        case KDA_ERR_DEVICE: return "device error word set";
        case KDA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case KDA_ERR_HOST_MEMORY: return "host allocation failed";
        case KDA_ERR_TIMEOUT: return "the stream had not finished within the time limit";
    }
    return "unknown status";
}

}  // extern "C"
