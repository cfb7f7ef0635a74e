"""Parity at the full sizes of the five workloads, in the launch
configurations the benchmark times.  The oracle checks sampled heads or
sequences at full length (heads and sequences are independent); everything
else is checked by properties that hold at any size (finiteness, bit-exact
resume, bookkeeping)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from hybrid_linear_attention_03_gb300 import build as kbuild
from hybrid_linear_attention_03_gb300 import inputs as I
from hybrid_linear_attention_03_gb300 import kda
from oracle import kda_oracle as ko

import helpers as hp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kda.lib()


def _dev(x):
    return {k: v.cuda() for k, v in x.items()}


def _weights(wl):
    w = wl.weights()
    wd = _dev(w)
    return w, wd, kda.make_weights(wd["conv_w"], wd["norm_w"], wl.eps_l2, wl.eps_rms)


def _prefill(pool, wgt, inp_dev, lens, slots, init, reqs=()):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    out = torch.empty(int(cu[-1]), pool.H, pool.dv, dtype=pool.act, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pool, cu), dtype=torch.uint8, device="cuda")
    kda.kda_prefill_chunked(pool, wgt, kda.make_io(inp_dev, out), cu, slots, init, 64, reqs, ws)
    del ws
    return out


def _oracle_run(wl, w, inp, heads, S0=None, t0=None):
    """Oracle over `heads` only; returns (out [L][h][dv], S [h][dk][dv], tail)."""
    sub, wsub = hp.head_subset(inp, w, heads, wl.H, wl.dk, wl.dv)
    nh = len(heads)
    S = np.zeros((nh, wl.dk, wl.dv)) if S0 is None else S0
    t = np.zeros((3, nh * (2 * wl.dk + wl.dv))) if t0 is None else t0
    out, S, t, _, _ = ko.default().layer(hp.oracle_inputs(sub), hp.oracle_weights(wsub), S, t,
                                         eps_l2=wl.eps_l2, eps_rms=wl.eps_rms)
    return out, S, t


def _gpu_state(pool, slot, heads):
    return hp.gpu_state_as_oracle(pool.states()[slot][list(heads)])


def _gpu_tail(pool, slot, heads):
    chans = hp.conv_channels(heads, pool.H, pool.dk, pool.dv)
    return hp.f64(pool.tails()[slot])[:, chans]


def test_decode_b1_1000_steps_full():
    """Batch-1 decode: 512 warm tokens (chunked prefill), then 1000 chained
    decode steps; all 64 heads against the oracle."""
    wl = I.DECODE_B1
    w, wd, wgt = _weights(wl)
    pool = kda.StatePool(wl.num_slots, wl.H, wl.dk, wl.dv, wl.act)
    slot = int(I.integers(wl.seed, 0, 0, wl.num_slots - 1, 1)[0])
    warm = wl.tokens(0, wl.extra["warm"])
    _prefill(pool, wgt, _dev(warm), [wl.extra["warm"]], [slot], [0])
    steps = wl.extra["steps"]
    toks = wl.tokens(100, steps)
    td = _dev(toks)
    out = torch.empty(steps, wl.H, wl.dv, dtype=wl.act, device="cuda")
    st = torch.tensor([slot], dtype=torch.int32, device="cuda")
    for i in range(steps):
        kda.kda_decode(pool, wgt, kda.make_io({k: v[i:i + 1] for k, v in td.items()}, out[i:i + 1]), st, 1)
    heads = list(range(wl.H))
    _, S, t = _oracle_run(wl, w, warm, heads)
    ref, S, t = _oracle_run(wl, w, toks, heads, S, t)
    assert hp.block_rel_err(hp.f64(out), ref, 1) <= hp.OUT_TOL_BF16
    assert hp.block_rel_err(_gpu_state(pool, slot, heads), S, 2) <= hp.STATE_TOL
    assert np.array_equal(_gpu_tail(pool, slot, heads), t)
    assert kda.kda_poll_device_error(pool) == (kda.KDA_OK, 0)


def test_verify_b64_t8_full():
    """64 sequences x 8 drafts over a 512-slot shuffled table, each warmed by
    512 tokens; accepted lengths uniform in 1..8 adopt their snapshot.  Four
    seeded sequences are checked against the oracle on all heads; every
    adopted slot must hold its snapshot bit for bit."""
    wl = I.VERIFY_B64
    B, T, warm_n = wl.extra["B"], wl.extra["T"], wl.extra["warm"]
    w, wd, wgt = _weights(wl)
    pool = kda.StatePool(wl.num_slots, wl.H, wl.dk, wl.dv, wl.act)
    table = I.permutation(wl.seed, 0, wl.num_slots).reshape(B, T)
    ins = table[:, 0].copy()
    warm = [wl.tokens(b, warm_n) for b in range(B)]
    _prefill(pool, wgt, _dev(I.concat_inputs(warm)), [warm_n] * B, ins, [0] * B)
    drafts = wl.tokens(200, B * T)
    out = torch.empty(B * T, wl.H, wl.dv, dtype=wl.act, device="cuda")
    kda.kda_verify(pool, wgt, kda.make_io(_dev(drafts), out), torch.from_numpy(ins).cuda(),
                   torch.from_numpy(table.reshape(-1).copy()).cuda(), B, T)
    acc = I.integers(wl.seed, 1, 1, T, B)
    adopted = [int(table[b, acc[b] - 1]) for b in range(B)]
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    heads = list(range(wl.H))
    for b in [int(x) for x in I.integers(wl.seed, 2, 0, B - 1, 4)]:
        _, S, t = _oracle_run(wl, w, warm[b], heads)
        for tt in range(T):
            tok = {k: v[b * T + tt:b * T + tt + 1] for k, v in drafts.items()}
            ref, S, t = _oracle_run(wl, w, tok, heads, S, t)
            assert hp.block_rel_err(hp.f64(out[b * T + tt:b * T + tt + 1]), ref, 1) <= hp.OUT_TOL_BF16
            snap = int(table[b, tt])
            assert hp.block_rel_err(_gpu_state(pool, snap, heads), S, 2) <= hp.STATE_TOL, (b, tt)
            assert np.array_equal(_gpu_tail(pool, snap, heads), t)
        assert adopted[b] == int(table[b, acc[b] - 1])
    assert kda.kda_poll_device_error(pool) == (kda.KDA_OK, 0)


def test_prefill_32k_full():
    """One 32768-token sequence (64 heads, C = 64, alpha = sigmoid(N(3,1))):
    every output and the end state of two seeded heads against the oracle."""
    wl = I.PREFILL_32K
    L = wl.extra["L"]
    w, wd, wgt = _weights(wl)
    pool = kda.StatePool(wl.num_slots, wl.H, wl.dk, wl.dv, wl.act)
    toks = wl.tokens(300, L)
    out = _prefill(pool, wgt, _dev(toks), [L], [0], [0])
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all()
    heads = sorted({int(x) for x in I.integers(wl.seed, 3, 0, wl.H - 1, 2)})
    ref, S, t = _oracle_run(wl, w, toks, heads)
    assert hp.block_rel_err(hp.f64(out[:, heads]), ref, 1) <= hp.OUT_TOL_BF16
    assert hp.block_rel_err(_gpu_state(pool, 0, heads), S, 2) <= hp.STATE_TOL
    assert np.array_equal(_gpu_tail(pool, 0, heads), t)
    assert kda.kda_poll_device_error(pool) == (kda.KDA_OK, 0)


def test_mixed_step_full_with_checkpoints_and_resume():
    """8 varlen prefills (log-uniform 1K..64K) and 56 single-token decodes
    (each warmed by 512 tokens) over a 1024-slot pool; checkpoints every
    32768 tokens and at every sequence end; then 4 seeded sequences resume
    from their latest checkpoint and must reproduce the uninterrupted run bit
    for bit.  Two seeded heads of every sequence against the oracle."""
    wl = I.MIXED
    plan = I.mixed_plan(wl)
    lens, reqs = plan["lens"], plan["reqs"]
    w, wd, wgt = _weights(wl)
    pool = kda.StatePool(wl.num_slots, wl.H, wl.dk, wl.dv, wl.act)
    nd, warm_n = wl.extra["n_decode"], wl.extra["warm"]
    warm = [wl.tokens(b, warm_n) for b in range(nd)]
    _prefill(pool, wgt, _dev(I.concat_inputs(warm)), [warm_n] * nd, plan["dec_slots"], [0] * nd)
    # the mixed step: one prefill call + one decode call
    pf = [wl.tokens(300 + n, L) for n, L in enumerate(lens)]
    pf_cat = I.concat_inputs(pf)
    pf_dev = _dev(pf_cat)
    out_pf = _prefill(pool, wgt, pf_dev, lens, plan["pf_slots"], [0] * len(lens), reqs)
    dec = wl.tokens(400, nd)
    out_dec = torch.empty(nd, wl.H, wl.dv, dtype=wl.act, device="cuda")
    kda.kda_decode(pool, wgt, kda.make_io(_dev(dec), out_dec), torch.tensor(plan["dec_slots"], dtype=torch.int32,
                                                                            device="cuda"), nd)
    torch.cuda.synchronize()
    assert torch.isfinite(out_pf.float()).all() and torch.isfinite(out_dec.float()).all()

    heads = sorted({int(x) for x in I.integers(wl.seed, 3, 0, wl.H - 1, 2)})
    cu = np.concatenate([[0], np.cumsum(lens)])
    for n, L in enumerate(lens):
        S = t = None
        pos = 0
        for (sq, p_, dst) in [r for r in reqs if r[0] == n]:
            part = {k: v[pos:p_] for k, v in pf[n].items()}
            ref, S, t = _oracle_run(wl, w, part, heads, S, t)
            got = out_pf[int(cu[n]) + pos:int(cu[n]) + p_][:, heads]
            assert hp.block_rel_err(hp.f64(got), ref, 1) <= hp.OUT_TOL_BF16, (n, pos)
            assert hp.block_rel_err(_gpu_state(pool, dst, heads), S, 2) <= hp.STATE_TOL, (n, p_)
            assert np.array_equal(_gpu_tail(pool, dst, heads), t)
            pos = p_
        assert hp.block_rel_err(_gpu_state(pool, plan["pf_slots"][n], heads), S, 2) <= hp.STATE_TOL
    for b in range(0, nd, 11):  # a sample of the decodes
        _, S, t = _oracle_run(wl, w, warm[b], heads)
        ref, S, t = _oracle_run(wl, w, {k: v[b:b + 1] for k, v in dec.items()}, heads, S, t)
        assert hp.block_rel_err(hp.f64(out_dec[b:b + 1][:, heads]), ref, 1) <= hp.OUT_TOL_BF16
        assert hp.block_rel_err(_gpu_state(pool, plan["dec_slots"][b], heads), S, 2) <= hp.STATE_TOL

    # resume: restore the latest checkpoint of each picked sequence into a fresh slot
    nxt = plan["next_free"]
    for n in plan["resume"]:
        mine = [r for r in reqs if r[0] == n]
        inner = [r for r in mine if r[1] < lens[n]]
        ck = inner[-1] if inner else mine[-1]
        fresh = nxt
        nxt += 1
        kda.kda_state_checkpoint(pool, [ck[2]], [fresh])
        orig = plan["pf_slots"][n]
        if ck[1] < lens[n]:  # replay the rest of the prompt from the interval checkpoint
            rest = {k: v[ck[1]:].contiguous() for k, v in {k2: v2[int(cu[n]):int(cu[n + 1])] for k2, v2 in pf_dev.items()}.items()}
            o = _prefill(pool, wgt, rest, [lens[n] - ck[1]], [fresh], [1])
            assert torch.equal(o, out_pf[int(cu[n]) + ck[1]:int(cu[n + 1])])
        cont = _dev(wl.tokens(500 + n, 64))
        o1 = _prefill(pool, wgt, cont, [64], [orig], [1])
        o2 = _prefill(pool, wgt, cont, [64], [fresh], [1])
        torch.cuda.synchronize()
        assert torch.equal(o1, o2), f"resumed sequence {n} diverged"
        assert torch.equal(pool.states()[orig], pool.states()[fresh])
        assert torch.equal(pool.tails()[orig], pool.tails()[fresh])
    assert kda.kda_poll_device_error(pool) == (kda.KDA_OK, 0)
