"""Python face of the double-precision CPU oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module.  It never imports the
CUDA package and the CUDA package never imports it; the two share nothing but
the seeded input generators.

The C file computes the KDA layer step of "vLLM Kimi K3 지원" (agentlenshq.com),
sections "Kimi K3 아키텍처 개요" and "Fused Kernels 및 메타데이터 최적화":
conv + SiLU, L2 norm of q and k, the delta-rule update with per-channel decay,
the readout and the sigmoid-gated RMSNorm.  This module builds it with gcc,
loads it with ctypes and adds the slot-pool semantics (decode, speculative
verify with per-token snapshots, chunked prefill with interval checkpoints,
slot copies) on top, all in float64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "kda_oracle.c"
BUILD_DIR = HERE / "_build"
LIB_PATH = BUILD_DIR / "libkda_oracle.so"

_dp = ctypes.POINTER(ctypes.c_double)


def compile_source(src: Path, out: Path) -> Path:
    """Compile an oracle C source into a shared library with gcc + OpenMP."""
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".{os.getpid()}.tmp.so")
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC",
           "-o", str(tmp), str(src), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> Path:
    """Build ``libkda_oracle.so`` if it is missing or older than its source."""
    if force or not LIB_PATH.exists() or LIB_PATH.stat().st_mtime < SRC.stat().st_mtime:
        compile_source(SRC, LIB_PATH)
    return LIB_PATH


def _ptr(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous float64"
    return a.ctypes.data_as(_dp)


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


class Oracle:
    """ctypes wrapper over one build of the oracle library."""

    def __init__(self, lib_path: Path | str | None = None):
        path = Path(lib_path) if lib_path is not None else build()
        self.lib = ctypes.CDLL(str(path))
        L = self.lib
        i, l, d = ctypes.c_int, ctypes.c_long, ctypes.c_double
        L.kdaref_conv_silu.argtypes = [i, l, i, _dp, _dp, _dp, _dp, _dp]
        L.kdaref_conv_silu.restype = None
        L.kdaref_l2norm_rows.argtypes = [l, i, _dp, d]
        L.kdaref_l2norm_rows.restype = None
        L.kdaref_gated_rmsnorm_rows.argtypes = [l, i, _dp, _dp, _dp, d, _dp]
        L.kdaref_gated_rmsnorm_rows.restype = None
        L.kdaref_core.argtypes = [i, i, i, i, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp]
        L.kdaref_core.restype = i
        L.kdaref_layer.argtypes = [i, i, i, i, i, d, d, i] + [_dp] * 13 + [i]
        L.kdaref_layer.restype = i
        L.kdaref_max_threads.argtypes = []
        L.kdaref_max_threads.restype = i

    def max_threads(self) -> int:
        return int(self.lib.kdaref_max_threads())

    # -- individual steps ---------------------------------------------------
    def conv_silu(self, x, conv_w, tail, want_hist=False):
        """a1 on x [L][n_ch]; returns (y, new_tail, hist_tail|None)."""
        x = _f64(x)
        conv_w = _f64(conv_w)
        tail = _f64(tail).copy()
        L, n_ch = x.shape
        W = conv_w.shape[1]
        assert conv_w.shape == (n_ch, W) and tail.shape == (W - 1, n_ch)
        y = np.zeros_like(x)
        hist = np.zeros((L, W - 1, n_ch)) if want_hist else None
        self.lib.kdaref_conv_silu(L, n_ch, W, _ptr(conv_w), _ptr(tail), _ptr(x), _ptr(y), _ptr(hist))
        return y, tail, hist

    def l2norm_rows(self, x, eps):
        x = _f64(x).copy()
        self.lib.kdaref_l2norm_rows(x.size // x.shape[-1], x.shape[-1], _ptr(x), float(eps))
        return x

    def gated_rmsnorm_rows(self, o, g, wn, eps):
        o, g, wn = _f64(o), _f64(g), _f64(wn)
        y = np.zeros_like(o)
        self.lib.kdaref_gated_rmsnorm_rows(o.size // o.shape[-1], o.shape[-1], _ptr(o), _ptr(g),
                                           _ptr(wn), float(eps), _ptr(y))
        return y

    def core(self, q, k, v, alpha, beta, S, chunk=0, want_hist=False):
        """a3 + a4 for one head on preprocessed inputs; returns (S_end, o, hist|None)."""
        q, k, v, alpha, beta = map(_f64, (q, k, v, alpha, beta))
        S = _f64(S).copy()
        L, dk = q.shape
        dv = v.shape[1]
        o = np.zeros((L, dv))
        hist = np.zeros((L, dk, dv)) if want_hist else None
        rc = self.lib.kdaref_core(L, dk, dv, int(chunk), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                  _ptr(beta), _ptr(S), _ptr(o), _ptr(hist))
        if rc != 0:
            raise RuntimeError("kdaref_core failed")
        return S, o, hist

    # -- the layer step -----------------------------------------------------
    def layer(self, inp, w, state, tail, chunk=0, want_hist=False, eps_l2=1e-6, eps_rms=1e-5,
              n_threads=0):
        """a1..a5 for one sequence.

        inp: dict q,k,v [L][H][d], alpha [L][H][dk], beta [L][H], gate [L][H][dv]
        w:   dict conv_w [n_ch][W], norm_w [dv]
        state [H][dk][dv], tail [W-1][n_ch] (not modified; new ones returned)
        returns (out [L][H][dv], state_end, tail_end, hist_state|None, hist_tail|None)
        """
        q, k, v = _f64(inp["q"]), _f64(inp["k"]), _f64(inp["v"])
        alpha, beta, gate = _f64(inp["alpha"]), _f64(inp["beta"]), _f64(inp["gate"])
        conv_w, norm_w = _f64(w["conv_w"]), _f64(w["norm_w"])
        L, H, dk = q.shape
        dv = v.shape[2]
        W = conv_w.shape[1]
        state = _f64(state).copy()
        tail = _f64(tail).copy()
        assert state.shape == (H, dk, dv) and tail.shape == (W - 1, H * (2 * dk + dv))
        out = np.zeros((L, H, dv))
        hs = np.zeros((L, H, dk, dv)) if want_hist else None
        ht = np.zeros((L, W - 1, H * (2 * dk + dv))) if want_hist else None
        rc = self.lib.kdaref_layer(L, H, dk, dv, W, float(eps_l2), float(eps_rms), int(chunk),
                                   _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(gate),
                                   _ptr(conv_w), _ptr(norm_w), _ptr(state), _ptr(tail), _ptr(out),
                                   _ptr(hs), _ptr(ht), int(n_threads))
        if rc != 0:
            raise RuntimeError("kdaref_layer failed")
        return out, state, tail, hs, ht


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT


class OraclePool:
    """The slot pool in float64: slot -> (state [H][dk][dv], tail [W-1][n_ch]).

    Mirrors the library's slot semantics: a slot never written holds a zero
    state and a zero tail ("vLLM Kimi K3 지원", section "하이브리드 KV-Cache 관리":
    compact per-request KDA state blocks; a new request starts from zero).
    """

    def __init__(self, H, dk, dv, W=4, eps_l2=1e-6, eps_rms=1e-5, oracle: Oracle | None = None):
        self.H, self.dk, self.dv, self.W = H, dk, dv, W
        self.n_ch = H * (2 * dk + dv)
        self.eps_l2, self.eps_rms = eps_l2, eps_rms
        self.o = oracle or default()
        self.slots: dict[int, tuple[np.ndarray, np.ndarray]] = {}

    def zero(self):
        return np.zeros((self.H, self.dk, self.dv)), np.zeros((self.W - 1, self.n_ch))

    def get(self, slot):
        S, t = self.slots.get(slot, self.zero())
        return S.copy(), t.copy()

    def put(self, slot, S, tail):
        self.slots[slot] = (np.array(S, dtype=np.float64), np.array(tail, dtype=np.float64))

    def run(self, slot, inp, w, chunk=0, fresh=False, want_hist=False, n_threads=0):
        """Advance one slot through a segment of tokens; returns out (and hist)."""
        S, t = self.zero() if fresh else self.get(slot)
        out, S, t, hs, ht = self.o.layer(inp, w, S, t, chunk=chunk, want_hist=want_hist,
                                         eps_l2=self.eps_l2, eps_rms=self.eps_rms,
                                         n_threads=n_threads)
        self.put(slot, S, t)
        return (out, hs, ht) if want_hist else out

    def checkpoint(self, src, dst):
        """Slot copy: every dst[i] receives src[i]'s state and tail."""
        snap = [self.get(s) for s in src]
        for d, (S, t) in zip(dst, snap):
            self.put(d, S, t)
