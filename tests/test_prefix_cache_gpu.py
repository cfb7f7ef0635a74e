"""Prompts served through the prefix-state cache on the GPU: a plan's reused
state is copied into the request's slot, only the rest of the prompt is
prefilled, and a second-hit prefix is saved by a checkpoint request of that
prefill.  Each request's outputs, end state and conv tail must equal, bit for
bit, a prefill of the whole prompt from a zero state (chunks stay aligned to
the sequence start, so the resumed run is the uninterrupted one)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from hybrid_linear_attention_03_gb300 import build as kbuild
from hybrid_linear_attention_03_gb300 import inputs as I
from hybrid_linear_attention_03_gb300 import kda

import helpers as hp

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kda.lib()


def _prefill(pool, wk, rows, slot, has_init, reqs=()):
    n = next(iter(rows.values())).shape[0]
    out = torch.empty(n, pool.H, D, dtype=pool.act, device="cuda")
    cu = np.array([0, n], dtype=np.int32)
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pool, cu), dtype=torch.uint8, device="cuda")
    kda.kda_prefill_chunked(pool, wk, kda.make_io(rows, out), cu, [slot], [has_init], 64, list(reqs), ws)
    return out


def test_requests_through_the_prefix_cache_equal_full_prefills():
    H, act, V = 2, torch.bfloat16, 211
    w = hp.to_device(I.layer_weights(81, H, D, D, 4, act))
    wk = kda.make_weights(w["conv_w"], w["norm_w"])
    # per-token activations: a prompt's rows depend on its token ids only, so
    # prompts with a common prefix share that prefix's rows
    vocab = hp.to_device(I.token_inputs(81, 0, V, H, D, D, 2.0, act))
    rng = np.random.default_rng(81)
    P = rng.integers(0, V, 200).tolist()
    Q = P[:130] + rng.integers(0, V, 70).tolist()
    S = P[:128] + rng.integers(0, V, 172).tolist()
    X = rng.integers(0, V, 100).tolist()
    prompts = [P, P, P, Q, P, S, X, X, P, Q + [5], S[:129]]
    cache_slots = [40, 41]
    served = kda.StatePool(64, H, D, D, act)
    full = kda.StatePool(64, H, D, D, act)
    cache = kda.PrefixCache(64, cache_slots, 1000)
    reused = admitted = 0
    for r, toks in enumerate(prompts):
        ids = torch.tensor(toks, device="cuda")
        rows = {k: v[ids].contiguous() for k, v in vocab.items()}
        ref = _prefill(full, wk, rows, r, 0)
        hit, hit_slot, apos, aslot = cache.plan(toks)
        if hit:
            kda.kda_state_checkpoint(served, [hit_slot], [r])
            reused += 1
        reqs = [(0, apos - hit, aslot)] if apos >= 0 else []
        admitted += bool(reqs)
        part = {k: v[hit:].contiguous() for k, v in rows.items()}
        out = _prefill(served, wk, part, r, 1 if hit else 0, reqs)
        torch.cuda.synchronize()
        assert torch.equal(out, ref[hit:]), f"request {r}"
        assert torch.equal(served.states()[r], full.states()[r]), f"request {r}: end state"
        assert torch.equal(served.tails()[r], full.tails()[r]), f"request {r}: conv tail"
    assert kda.kda_poll_device_error(served) == (kda.KDA_OK, 0)
    st = cache.stats()
    assert reused == st["hits"] >= 5 and admitted == st["admissions"] >= 4 and st["evictions"] >= 1
