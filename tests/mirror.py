"""A GPU slot pool and an oracle slot pool driven through the same calls.

Each method runs one library entry point on the GPU pool and the matching
oracle computation on the float64 pool, and returns both outputs.  Only the
seeded inputs are shared; the oracle never reads anything the GPU produced.
"""

from __future__ import annotations

import numpy as np
import torch

from hybrid_linear_attention_03_gb300 import kda
from oracle import kda_oracle as ko

import helpers as hp


class Mirror:
    def __init__(self, num_slots, H, D, act, weights: dict, eps_l2=1e-6, eps_rms=1e-5):
        self.H, self.D, self.act = H, D, act
        self.gpu = kda.StatePool(num_slots, H, D, D, act)
        self.w_dev = hp.to_device(weights)
        self.w = kda.make_weights(self.w_dev["conv_w"], self.w_dev["norm_w"], eps_l2, eps_rms)
        self.ora = ko.OraclePool(H, D, D, 4, eps_l2, eps_rms)
        self.w_ora = hp.oracle_weights(weights)

    # -- entry points ---------------------------------------------------------
    def decode(self, slots, inp, stream=None):
        B = len(slots)
        dev = hp.to_device(inp)
        out = torch.empty(B, self.H, self.D, dtype=self.act, device="cuda")
        sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
        kda.kda_decode(self.gpu, self.w, kda.make_io(dev, out), sl, B, stream)
        ref = np.zeros((B, self.H, self.D))
        oi = hp.oracle_inputs(inp)
        for b, s in enumerate(slots):
            tok = {k: v[b:b + 1] for k, v in oi.items()}
            ref[b] = self.ora.run(int(s), tok, self.w_ora)[0]
        return out, ref

    def verify(self, in_slots, snap_slots, T, inp, stream=None):
        """snap_slots: [B][T]; inp rows b*T + t."""
        B = len(in_slots)
        dev = hp.to_device(inp)
        out = torch.empty(B * T, self.H, self.D, dtype=self.act, device="cuda")
        si = torch.tensor(in_slots, dtype=torch.int32, device="cuda")
        ss = torch.tensor(np.asarray(snap_slots).reshape(-1), dtype=torch.int32, device="cuda")
        kda.kda_verify(self.gpu, self.w, kda.make_io(dev, out), si, ss, B, T, stream)
        ref = np.zeros((B * T, self.H, self.D))
        oi = hp.oracle_inputs(inp)
        starts = [self.ora.get(int(s)) for s in in_slots]
        for b in range(B):
            tok = {k: v[b * T:(b + 1) * T] for k, v in oi.items()}
            S0, t0 = starts[b]
            o, _, _, hs, ht = self.ora.o.layer(tok, self.w_ora, S0, t0, want_hist=True,
                                               eps_l2=self.ora.eps_l2, eps_rms=self.ora.eps_rms)
            ref[b * T:(b + 1) * T] = o
            for t in range(T):
                self.ora.put(int(snap_slots[b][t]), hs[t], ht[t])
        return out, ref

    def checkpoint(self, src, dst):
        kda.kda_state_checkpoint(self.gpu, src, dst)
        self.ora.checkpoint(src, dst)

    # -- comparisons ------------------------------------------------------------
    def state_err(self, slot) -> float:
        g = hp.gpu_state_as_oracle(self.gpu.states()[slot])
        return hp.block_rel_err(g, self.ora.get(int(slot))[0], 2)

    def tail_equal(self, slot) -> bool:
        g = hp.f64(self.gpu.tails()[slot])
        return bool(np.array_equal(g, self.ora.get(int(slot))[1]))


class OracleMirror:
    """The oracle side of a Mirror alone, for tests that drive the GPU pools
    themselves: a float64 slot pool started from the GPU pool's states and
    tails (read once, before any GPU call of the test), and the layer weights.
    prefill_oracle accepts it in place of a Mirror."""

    def __init__(self, H, D, act, weights: dict, states=None, tails=None, eps_l2=1e-6, eps_rms=1e-5):
        self.H, self.D, self.act = H, D, act
        self.ora = ko.OraclePool(H, D, D, 4, eps_l2, eps_rms)
        self.w_ora = hp.oracle_weights(weights)
        if states is not None:
            for s in range(states.shape[0]):
                self.ora.put(s, hp.gpu_state_as_oracle(states[s]), hp.f64(tails[s]))

    def check_slots(self, pool, slots, tol=hp.STATE_TOL):
        """Every listed slot of the GPU pool against the oracle pool: state
        within tol (block relative error), conv tail bit for bit."""
        for s in slots:
            g = hp.gpu_state_as_oracle(pool.states()[int(s)])
            S, t = self.ora.get(int(s))
            err = hp.block_rel_err(g, S, 2)
            assert err <= tol, f"state of slot {s}: {err:.3e}"
            assert np.array_equal(hp.f64(pool.tails()[int(s)]), t), f"tail of slot {s}"


def prefill_gpu(m: Mirror, inp_dev: dict, lens, slots, has_init, reqs=(), stream=None):
    """Run kda_prefill_chunked on the mirror's GPU pool; returns the output."""
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out = torch.empty(int(cu[-1]), m.H, m.D, dtype=m.act, device="cuda")
    ws_bytes = kda.kda_prefill_workspace_bytes(m.gpu, cu)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device="cuda")
    kda.kda_prefill_chunked(m.gpu, m.w, kda.make_io(inp_dev, out), cu, slots, has_init, 64, reqs, ws, stream)
    if stream is not None:
        # the workspace was allocated on the current stream but is used on
        # `stream`: keep the caching allocator from reusing it before that
        # stream's prefill has finished
        ws.record_stream(stream)
    return out


def prefill_oracle(m: Mirror, inp: dict, lens, slots, has_init, reqs=()):
    """The same prefill on the oracle pool: each sequence runs from its slot
    (or from zeros), split at its checkpoint positions."""
    oi = hp.oracle_inputs(inp)
    cu = np.concatenate([[0], np.cumsum(lens)])
    out = np.zeros((int(cu[-1]), m.H, m.D))
    for n, (slot, init) in enumerate(zip(slots, has_init)):
        a, b = int(cu[n]), int(cu[n + 1])
        cuts = sorted({int(r[1]) for r in reqs if r[0] == n} | {b - a})
        S, t = m.ora.get(int(slot)) if init else m.ora.zero()
        pos = 0
        for c in cuts:
            if c > pos:
                part = {k: v[a + pos:a + c] for k, v in oi.items()}
                o, S, t, _, _ = m.ora.o.layer(part, m.w_ora, S, t, eps_l2=m.ora.eps_l2, eps_rms=m.ora.eps_rms)
                out[a + pos:a + c] = o
                pos = c
            for r in reqs:
                if r[0] == n and r[1] == c:
                    m.ora.put(int(r[2]), S, t)
        m.ora.put(int(slot), S, t)
    return out
