"""Thin ctypes binding of libkda (include/kda.h): argument marshalling only.

Every entry point of the C ABI has a function of the same name here.  Tensors
are torch tensors (device memory and streams come from PyTorch); each call
passes their data pointers and the current CUDA stream to the library, where
all of the work runs in the hand-written sm_103a kernels.  There is no
fallback: if ``libkda.so`` is missing the first call raises.
"""

from __future__ import annotations

import ctypes
from pathlib import Path

import torch

_LIB_PATH = Path(__file__).resolve().parent / "_build" / "libkda.so"
_LIB = None

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_SLOT_RANGE = 2
KDA_ERR_ALIAS = 3
KDA_ERR_UNSUPPORTED = 4
KDA_ERR_CUDA = 5
KDA_ERR_DEVICE = 6
KDA_ERR_WORKSPACE = 7
KDA_ERR_HOST_MEMORY = 8
KDA_ERR_TIMEOUT = 9
KDA_F32 = 0
KDA_BF16 = 1
KDA_DEVERR_SLOT_RANGE = 0x1
KDA_DEVERR_META = 0x2
KDA_DEVERR_TIMEOUT = 0x4
KDA_POOL_OVERLAP_INPUTS = 0x1

# Every symbol include/kda.h declares.
EXPORTS = ("kda_state_pool_bytes", "kda_state_pool_create", "kda_state_pool_destroy", "kda_state_pool_layout",
           "kda_check_slots", "kda_decode", "kda_verify", "kda_prefill_workspace_bytes", "kda_prefill_chunked",
           "kda_state_checkpoint", "kda_poll_device_error", "kda_status_string", "kda_prefill_chunked_noalloc",
           "kda_state_slot_bytes", "kda_state_export", "kda_state_import", "kda_prefill_workspace_bytes_bound",
           "kda_prefill_chunked_dev", "kda_prefix_cache_create", "kda_prefix_cache_destroy", "kda_prefix_cache_plan",
           "kda_prefix_cache_forget", "kda_prefix_cache_get_stats", "kda_prefix_cache_saved", "kda_stream_wait",
           "kda_state_pool_set_flags", "kda_profile_start", "kda_profile_stop", "kda_state_prefetch")

# kda_kernel_kind
KERNEL_KINDS = ("step", "slot_copy", "prefill_meta", "prefill_intra", "prefill_chain", "prefill_out", "prefill_tails",
                "state_prefetch", "prefill_intra_exact")

KDA_NOALLOC_SCRATCH_BYTES = 64 << 20


class kda_pool_desc(ctypes.Structure):
    _fields_ = [("num_slots", ctypes.c_int32), ("num_heads", ctypes.c_int32), ("d_k", ctypes.c_int32),
                ("d_v", ctypes.c_int32), ("conv_width", ctypes.c_int32), ("act", ctypes.c_int32)]


class kda_pool_layout(ctypes.Structure):
    _fields_ = [("header_offset", ctypes.c_size_t), ("state_offset", ctypes.c_size_t),
                ("state_slot_bytes", ctypes.c_size_t), ("tail_offset", ctypes.c_size_t),
                ("tail_slot_bytes", ctypes.c_size_t), ("total_bytes", ctypes.c_size_t)]


class kda_weights(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("norm_w", ctypes.c_void_p), ("eps_l2", ctypes.c_float),
                ("eps_rms", ctypes.c_float)]


class kda_io(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("alpha", ctypes.c_void_p),
                ("beta", ctypes.c_void_p), ("gate", ctypes.c_void_p), ("out", ctypes.c_void_p)]


class kda_ckpt_req(ctypes.Structure):
    _fields_ = [("seq", ctypes.c_int32), ("token_pos", ctypes.c_int32), ("dst_slot", ctypes.c_int32)]


class kda_prefix_plan(ctypes.Structure):
    _fields_ = [("hit_len", ctypes.c_int32), ("hit_slot", ctypes.c_int32), ("admit_pos", ctypes.c_int32),
                ("admit_slot", ctypes.c_int32)]


class kda_prefix_cache_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("plans", "hits", "admissions", "evictions", "n_saved", "n_unsaved",
                                               "n_free")]


class kda_profile(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_int64 * len(KERNEL_KINDS)), ("ms", ctypes.c_double * len(KERNEL_KINDS)),
                ("dropped", ctypes.c_int64)]


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kda_status_string(status)} ({status})")


def lib_path() -> Path:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libkda.so (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not _LIB_PATH.exists():
            raise RuntimeError(f"{_LIB_PATH} is missing: build it first (python -m hybrid_linear_attention_03_gb300.build)")
        L = ctypes.CDLL(str(_LIB_PATH))
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        P = ctypes.POINTER
        L.kda_state_pool_bytes.argtypes = [P(kda_pool_desc)]
        L.kda_state_pool_bytes.restype = sz
        L.kda_state_pool_create.argtypes = [P(kda_pool_desc), vp, sz, P(vp)]
        L.kda_state_pool_create.restype = i32
        L.kda_state_pool_destroy.argtypes = [vp]
        L.kda_state_pool_destroy.restype = None
        L.kda_state_pool_set_flags.argtypes = [vp, ctypes.c_uint32]
        L.kda_state_pool_set_flags.restype = i32
        L.kda_state_pool_layout.argtypes = [vp, P(kda_pool_layout)]
        L.kda_state_pool_layout.restype = i32
        L.kda_check_slots.argtypes = [vp, vp, i32, vp, i32]
        L.kda_check_slots.restype = i32
        L.kda_decode.argtypes = [vp, P(kda_weights), P(kda_io), vp, i32, vp]
        L.kda_decode.restype = i32
        L.kda_state_prefetch.argtypes = [vp, vp, vp, i32, vp]
        L.kda_state_prefetch.restype = i32
        L.kda_verify.argtypes = [vp, P(kda_weights), P(kda_io), vp, vp, i32, i32, vp]
        L.kda_verify.restype = i32
        L.kda_prefill_workspace_bytes.argtypes = [vp, vp, i32, i32]
        L.kda_prefill_workspace_bytes.restype = sz
        L.kda_prefill_chunked.argtypes = [vp, P(kda_weights), P(kda_io), vp, vp, vp, i32, i32,
                                          P(kda_ckpt_req), i32, vp, sz, vp]
        L.kda_prefill_chunked.restype = i32
        L.kda_prefill_chunked_noalloc.argtypes = [vp, P(kda_weights), P(kda_io), vp, vp, vp, i32, i32,
                                                  P(kda_ckpt_req), i32, vp]
        L.kda_prefill_chunked_noalloc.restype = i32
        L.kda_state_checkpoint.argtypes = [vp, vp, vp, i32, vp]
        L.kda_state_checkpoint.restype = i32
        L.kda_prefill_workspace_bytes_bound.argtypes = [vp, i32, i32, i32, i32]
        L.kda_prefill_workspace_bytes_bound.restype = sz
        L.kda_prefill_chunked_dev.argtypes = [vp, P(kda_weights), P(kda_io), vp, vp, vp, i32, i32, i32, vp, i32,
                                              vp, sz, vp]
        L.kda_prefill_chunked_dev.restype = i32
        L.kda_state_slot_bytes.argtypes = [vp]
        L.kda_state_slot_bytes.restype = sz
        L.kda_state_export.argtypes = [vp, i32, vp, sz, vp]
        L.kda_state_export.restype = i32
        L.kda_state_import.argtypes = [vp, i32, vp, sz, vp]
        L.kda_state_import.restype = i32
        L.kda_poll_device_error.argtypes = [vp, vp, P(ctypes.c_uint32)]
        L.kda_poll_device_error.restype = i32
        L.kda_prefix_cache_create.argtypes = [i32, vp, i32, i32, P(vp)]
        L.kda_prefix_cache_create.restype = i32
        L.kda_prefix_cache_destroy.argtypes = [vp]
        L.kda_prefix_cache_destroy.restype = None
        L.kda_prefix_cache_plan.argtypes = [vp, vp, i32, P(kda_prefix_plan)]
        L.kda_prefix_cache_plan.restype = i32
        L.kda_prefix_cache_forget.argtypes = [vp, i32]
        L.kda_prefix_cache_forget.restype = i32
        L.kda_prefix_cache_get_stats.argtypes = [vp, P(kda_prefix_cache_stats)]
        L.kda_prefix_cache_get_stats.restype = i32
        L.kda_prefix_cache_saved.argtypes = [vp, vp, vp, i32]
        L.kda_prefix_cache_saved.restype = i32
        L.kda_stream_wait.argtypes = [vp, ctypes.c_double]
        L.kda_stream_wait.restype = i32
        L.kda_profile_start.argtypes = [i32]
        L.kda_profile_start.restype = i32
        L.kda_profile_stop.argtypes = [P(kda_profile)]
        L.kda_profile_stop.restype = i32
        L.kda_status_string.argtypes = [i32]
        L.kda_status_string.restype = ctypes.c_char_p
        _LIB = L
    return _LIB


def kda_stream_wait(stream=None, timeout_s: float = 60.0) -> int:
    """Waits at most timeout_s for the stream's work; KDA_OK or KDA_ERR_TIMEOUT
    (raises on any other status)."""
    st = lib().kda_stream_wait(_stream(stream), float(timeout_s))
    if st not in (KDA_OK, KDA_ERR_TIMEOUT):
        raise KdaError(st, "kda_stream_wait")
    return st


def kda_profile_start(max_launches: int = 4096) -> None:
    """Starts timing every kernel the library launches (CUDA events on the
    launching stream) on the current device."""
    _check(lib().kda_profile_start(int(max_launches)), "kda_profile_start")


def kda_profile_stop() -> dict:
    """Stops the profile: {kind: (launches, total ms)} plus "dropped"."""
    out = kda_profile()
    _check(lib().kda_profile_stop(ctypes.byref(out)), "kda_profile_stop")
    res = {k: (int(out.launches[i]), float(out.ms[i])) for i, k in enumerate(KERNEL_KINDS)}
    res["dropped"] = int(out.dropped)
    return res


def kda_status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != KDA_OK:
        raise KdaError(status, where)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dptr(t: torch.Tensor | None):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _host_i32(x):
    """A host int32 array for the C side (keeps the buffer alive in the tuple)."""
    t = torch.as_tensor(x, dtype=torch.int32).contiguous().cpu()
    return t, ctypes.c_void_p(t.data_ptr()) if t.numel() else None


def act_code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return KDA_BF16
    if dtype == torch.float32:
        return KDA_F32
    raise ValueError(f"unsupported activation dtype {dtype}")


def make_desc(num_slots, H, dk, dv, act: torch.dtype, conv_width=4) -> kda_pool_desc:
    return kda_pool_desc(num_slots, H, dk, dv, conv_width, act_code(act))


def kda_state_pool_bytes(desc: kda_pool_desc) -> int:
    return int(lib().kda_state_pool_bytes(ctypes.byref(desc)))


def kda_state_pool_create(desc: kda_pool_desc, buf: torch.Tensor) -> ctypes.c_void_p:
    h = ctypes.c_void_p()
    _check(lib().kda_state_pool_create(ctypes.byref(desc), _dptr(buf), buf.numel() * buf.element_size(),
                                       ctypes.byref(h)), "kda_state_pool_create")
    return h


def kda_state_pool_destroy(handle) -> None:
    if handle:
        lib().kda_state_pool_destroy(handle)


def kda_state_pool_set_flags(pool: "StatePool", flags: int) -> None:
    """Launch options of the pool's decode / verify calls (KDA_POOL_* flags)."""
    _check(lib().kda_state_pool_set_flags(pool.handle, int(flags)), "kda_state_pool_set_flags")


def kda_state_pool_layout(handle) -> kda_pool_layout:
    out = kda_pool_layout()
    _check(lib().kda_state_pool_layout(handle, ctypes.byref(out)), "kda_state_pool_layout")
    return out


def make_weights(conv_w: torch.Tensor, norm_w: torch.Tensor, eps_l2=1e-6, eps_rms=1e-5) -> kda_weights:
    """The struct holds raw device pointers; it also keeps the two tensors
    alive, so their memory cannot be handed to another tensor while the
    struct is in use."""
    w = kda_weights(conv_w.data_ptr(), norm_w.data_ptr(), float(eps_l2), float(eps_rms))
    w._tensors = (conv_w, norm_w)
    return w


def make_io(inp: dict, out: torch.Tensor) -> kda_io:
    """Raw pointers to the step's arrays; the struct keeps the tensors alive."""
    io = kda_io(inp["q"].data_ptr(), inp["k"].data_ptr(), inp["v"].data_ptr(), inp["alpha"].data_ptr(),
                inp["beta"].data_ptr(), inp["gate"].data_ptr(), out.data_ptr())
    io._tensors = (inp["q"], inp["k"], inp["v"], inp["alpha"], inp["beta"], inp["gate"], out)
    return io


class StatePool:
    """A slot pool over a torch-allocated device buffer (zero-filled)."""

    def __init__(self, num_slots, H, dk, dv, act: torch.dtype = torch.bfloat16, device="cuda"):
        self.desc = make_desc(num_slots, H, dk, dv, act)
        self.act = act
        self.H, self.dk, self.dv, self.num_slots = H, dk, dv, num_slots
        self.n_ch = H * (2 * dk + dv)
        nbytes = kda_state_pool_bytes(self.desc)
        if nbytes == 0:
            raise KdaError(KDA_ERR_INVALID_ARG, "kda_state_pool_bytes")
        self.buf = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.handle = kda_state_pool_create(self.desc, self.buf)
        self.layout = kda_state_pool_layout(self.handle)

    def states(self) -> torch.Tensor:
        """View [num_slots][H][d_v][d_k] fp32 (S^T per head)."""
        L = self.layout
        n = self.num_slots * L.state_slot_bytes
        return self.buf[L.state_offset:L.state_offset + n].view(torch.float32).view(
            self.num_slots, self.H, self.dv, self.dk)

    def tails(self) -> torch.Tensor:
        """View [num_slots][3][n_ch] act."""
        L = self.layout
        n = self.num_slots * L.tail_slot_bytes
        return self.buf[L.tail_offset:L.tail_offset + n].view(self.act).view(self.num_slots, 3, self.n_ch)

    def error_word(self) -> torch.Tensor:
        return self.buf[0:4].view(torch.int32)

    def close(self):
        kda_state_pool_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            if getattr(self, "handle", None):
                kda_state_pool_destroy(self.handle)
        except Exception:
            pass


def kda_check_slots(pool: StatePool, in_slots=None, out_slots=None) -> int:
    """Host-side check of slot tables; returns the kda_status (0 = ok)."""
    ti, pi = _host_i32(in_slots if in_slots is not None else [])
    to, po = _host_i32(out_slots if out_slots is not None else [])
    return int(lib().kda_check_slots(pool.handle, pi, ti.numel(), po, to.numel()))


def kda_decode(pool: StatePool, weights: kda_weights, io: kda_io, slots: torch.Tensor, B: int | None = None,
               stream=None) -> None:
    B = slots.numel() if B is None else B
    _check(lib().kda_decode(pool.handle, ctypes.byref(weights), ctypes.byref(io), _dptr(slots), int(B),
                            _stream(stream)), "kda_decode")


def kda_state_prefetch(pool: StatePool, slots: torch.Tensor, B: int | None = None, stream=None,
                       weights: kda_weights | None = None) -> None:
    """Hint: bring the slots' state and conv tail (and the weights, if given)
    into L2 ahead of a decode."""
    B = slots.numel() if B is None else B
    wp = ctypes.byref(weights) if weights is not None else None
    _check(lib().kda_state_prefetch(pool.handle, wp, _dptr(slots), int(B), _stream(stream)), "kda_state_prefetch")


def kda_verify(pool: StatePool, weights: kda_weights, io: kda_io, in_slots: torch.Tensor, snap_slots: torch.Tensor,
               B: int, T: int, stream=None) -> None:
    _check(lib().kda_verify(pool.handle, ctypes.byref(weights), ctypes.byref(io), _dptr(in_slots),
                            _dptr(snap_slots), int(B), int(T), _stream(stream)), "kda_verify")


def kda_prefill_workspace_bytes(pool: StatePool, cu_seqlens, chunk: int = 64) -> int:
    t, p = _host_i32(cu_seqlens)
    return int(lib().kda_prefill_workspace_bytes(pool.handle, p, t.numel() - 1, int(chunk)))


def kda_prefill_chunked(pool: StatePool, weights: kda_weights, io: kda_io, cu_seqlens, slots, has_initial_state,
                        chunk: int = 64, reqs=(), workspace: torch.Tensor | None = None, stream=None) -> None:
    tc, pc = _host_i32(cu_seqlens)
    ts, ps = _host_i32(slots)
    th = torch.as_tensor(has_initial_state, dtype=torch.uint8).contiguous().cpu()
    n_req = len(reqs)
    req_arr = (kda_ckpt_req * max(1, n_req))(*[kda_ckpt_req(int(a), int(b), int(c)) for a, b, c in reqs])
    ws_ptr = _dptr(workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().kda_prefill_chunked(pool.handle, ctypes.byref(weights), ctypes.byref(io), pc, ps,
                                     ctypes.c_void_p(th.data_ptr()), int(tc.numel() - 1), int(chunk),
                                     req_arr, int(n_req), ws_ptr, ws_bytes, _stream(stream)),
           "kda_prefill_chunked")


def kda_prefill_workspace_bytes_bound(pool: StatePool, n_seqs: int, max_tokens: int, n_reqs: int,
                                      chunk: int = 64) -> int:
    return int(lib().kda_prefill_workspace_bytes_bound(pool.handle, int(n_seqs), int(max_tokens), int(n_reqs),
                                                       int(chunk)))


def kda_prefill_chunked_dev(pool: StatePool, weights: kda_weights, io: kda_io, cu_seqlens: torch.Tensor,
                            slots: torch.Tensor, has_initial_state: torch.Tensor, max_tokens: int,
                            reqs: torch.Tensor | None, workspace: torch.Tensor, chunk: int = 64, stream=None) -> None:
    """kda_prefill_chunked with the metadata in device memory: cu_seqlens and
    slots int32, has_initial_state uint8, reqs int32 [n, 3] (seq, token_pos,
    dst_slot) or None, all CUDA tensors; the tables are built on the GPU."""
    for name, t, dt in (("cu_seqlens", cu_seqlens, torch.int32), ("slots", slots, torch.int32),
                        ("has_initial_state", has_initial_state, torch.uint8)):
        if not t.is_cuda or t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    n_req = 0 if reqs is None else int(reqs.shape[0])
    if reqs is not None and (not reqs.is_cuda or reqs.dtype != torch.int32 or tuple(reqs.shape[1:]) != (3,)
                             or not reqs.is_contiguous()):
        raise ValueError("reqs must be a contiguous CUDA int32 tensor of shape [n, 3]")
    _check(lib().kda_prefill_chunked_dev(pool.handle, ctypes.byref(weights), ctypes.byref(io), cu_seqlens.data_ptr(),
                                         slots.data_ptr(), has_initial_state.data_ptr(), int(cu_seqlens.numel() - 1),
                                         int(max_tokens), int(chunk), None if n_req == 0 else reqs.data_ptr(),
                                         n_req, _dptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream)),
           "kda_prefill_chunked_dev")


def kda_prefill_chunked_noalloc(pool: StatePool, weights: kda_weights, io: kda_io, cu_seqlens, slots,
                                has_initial_state, chunk: int = 64, reqs=(), stream=None) -> None:
    """kda_prefill_chunked for callers that cannot allocate device memory: the
    library's fixed 64 MiB scratch array stands in for the workspace."""
    tc, pc = _host_i32(cu_seqlens)
    ts, ps = _host_i32(slots)
    th = torch.as_tensor(has_initial_state, dtype=torch.uint8).contiguous().cpu()
    n_req = len(reqs)
    req_arr = (kda_ckpt_req * max(1, n_req))(*[kda_ckpt_req(int(a), int(b), int(c)) for a, b, c in reqs])
    _check(lib().kda_prefill_chunked_noalloc(pool.handle, ctypes.byref(weights), ctypes.byref(io), pc, ps,
                                             ctypes.c_void_p(th.data_ptr()), int(tc.numel() - 1), int(chunk),
                                             req_arr, int(n_req), _stream(stream)),
           "kda_prefill_chunked_noalloc")


def kda_state_checkpoint(pool: StatePool, src_slots, dst_slots, stream=None) -> None:
    ts, ps = _host_i32(src_slots)
    td, pd = _host_i32(dst_slots)
    if ts.numel() != td.numel():
        raise ValueError("src and dst slot lists differ in length")
    _check(lib().kda_state_checkpoint(pool.handle, ps, pd, int(ts.numel()), _stream(stream)),
           "kda_state_checkpoint")


def kda_state_slot_bytes(pool: StatePool) -> int:
    return int(lib().kda_state_slot_bytes(pool.handle))


def kda_state_export(pool: StatePool, slot: int, host: torch.Tensor, stream=None) -> None:
    """Copies slot `slot` (state, then conv tail) into the CPU uint8 tensor
    `host` (pin it for an asynchronous copy); bit-exact."""
    if host.device.type != "cpu" or not host.is_contiguous():
        raise ValueError("host must be a contiguous CPU tensor")
    _check(lib().kda_state_export(pool.handle, int(slot), host.data_ptr(), host.numel() * host.element_size(),
                                  _stream(stream)), "kda_state_export")


def kda_state_import(pool: StatePool, slot: int, host: torch.Tensor, stream=None) -> None:
    """Copies a buffer written by kda_state_export into slot `slot`; bit-exact."""
    if host.device.type != "cpu" or not host.is_contiguous():
        raise ValueError("host must be a contiguous CPU tensor")
    _check(lib().kda_state_import(pool.handle, int(slot), host.data_ptr(), host.numel() * host.element_size(),
                                  _stream(stream)), "kda_state_import")


def kda_poll_device_error(pool: StatePool, stream=None) -> tuple[int, int]:
    """Returns (status, flags); reading clears the device error word."""
    flags = ctypes.c_uint32(0)
    st = int(lib().kda_poll_device_error(pool.handle, _stream(stream), ctypes.byref(flags)))
    return st, int(flags.value)


def kda_prefix_cache_create(block: int, slots, max_tracked: int) -> ctypes.c_void_p:
    ts, ps = _host_i32(slots)
    h = ctypes.c_void_p()
    _check(lib().kda_prefix_cache_create(int(block), ps, int(ts.numel()), int(max_tracked), ctypes.byref(h)),
           "kda_prefix_cache_create")
    return h


def kda_prefix_cache_destroy(handle: ctypes.c_void_p) -> None:
    lib().kda_prefix_cache_destroy(handle)


def kda_prefix_cache_plan(handle: ctypes.c_void_p, tokens) -> tuple[int, int, int, int]:
    """(hit_len, hit_slot, admit_pos, admit_slot) for a prompt of token ids."""
    t, pt = _host_i32(tokens)
    out = kda_prefix_plan()
    _check(lib().kda_prefix_cache_plan(handle, pt, int(t.numel()), ctypes.byref(out)), "kda_prefix_cache_plan")
    return out.hit_len, out.hit_slot, out.admit_pos, out.admit_slot


def kda_prefix_cache_forget(handle: ctypes.c_void_p, slot: int) -> None:
    _check(lib().kda_prefix_cache_forget(handle, int(slot)), "kda_prefix_cache_forget")


def kda_prefix_cache_get_stats(handle: ctypes.c_void_p) -> dict:
    st = kda_prefix_cache_stats()
    _check(lib().kda_prefix_cache_get_stats(handle, ctypes.byref(st)), "kda_prefix_cache_get_stats")
    return {n: getattr(st, n) for n, _ in kda_prefix_cache_stats._fields_}


def kda_prefix_cache_saved(handle: ctypes.c_void_p) -> dict:
    """{slot: prefix length} of the saved prefixes."""
    n = lib().kda_prefix_cache_saved(handle, None, None, 0)
    lens = (ctypes.c_int32 * max(n, 1))()
    slots = (ctypes.c_int32 * max(n, 1))()
    m = lib().kda_prefix_cache_saved(handle, lens, slots, n)
    return {int(slots[i]): int(lens[i]) for i in range(m)}


class PrefixCache:
    """Owner of a kda_prefix_cache handle (destroyed with the object); the
    methods are the kda_prefix_cache_* functions above."""

    def __init__(self, block: int, slots, max_tracked: int):
        self.handle = kda_prefix_cache_create(block, slots, max_tracked)
        self.block = int(block)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value and _LIB is not None:
            _LIB.kda_prefix_cache_destroy(h)
            self.handle = None

    def plan(self, tokens) -> tuple[int, int, int, int]:
        return kda_prefix_cache_plan(self.handle, tokens)

    def forget(self, slot: int) -> None:
        kda_prefix_cache_forget(self.handle, slot)

    def stats(self) -> dict:
        return kda_prefix_cache_get_stats(self.handle)

    def saved(self) -> dict:
        return kda_prefix_cache_saved(self.handle)
