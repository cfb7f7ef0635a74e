"""The chunked prefill with its sequence metadata in device memory
(kda_prefill_chunked_dev): its tables are built on the GPU, so it must match
the oracle (outputs, states and tails of every sequence and checkpoint slot),
give bit for bit what the host-metadata call gives, run inside a CUDA graph,
and reject bad metadata on the device without touching any slot or output."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from hybrid_linear_attention_03_gb300 import build as kbuild
from hybrid_linear_attention_03_gb300 import inputs as I
from hybrid_linear_attention_03_gb300 import kda

import helpers as hp
from mirror import OracleMirror, prefill_oracle

pytestmark = pytest.mark.gpu

D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kda.lib()


def _setup(act, seed, lens, max_extra=70, want_oracle=False):
    """Two identical pools (random warm states and tails), weights, inputs of
    max_tokens rows (the real tokens first, then padding rows); with
    want_oracle also an oracle pool holding the same start states."""
    H, num_slots = 2, 32
    w = I.layer_weights(seed, H, D, D, 4, act)
    w_dev = hp.to_device(w)
    wk = kda.make_weights(w_dev["conv_w"], w_dev["norm_w"])  # keeps the device tensors alive
    pools = [kda.StatePool(num_slots, H, D, D, act) for _ in range(2)]
    g = torch.Generator(device="cpu").manual_seed(seed)
    st = torch.randn(num_slots, H, D, D, generator=g) * 0.05
    tl = torch.randn(num_slots, 3, pools[0].n_ch, generator=g).to(act)
    for p in pools:
        p.states().copy_(st)
        p.tails().copy_(tl)
    n_tok = int(sum(lens))
    max_tokens = n_tok + max_extra
    inp_cpu = I.token_inputs(seed, 0, max_tokens, H, D, D, 2.0, act)
    inp = hp.to_device(inp_cpu)
    if want_oracle:
        om = OracleMirror(H, D, act, w, st, tl)
        real_cpu = {k: v[:n_tok] for k, v in inp_cpu.items()}
        return H, wk, pools, inp, n_tok, max_tokens, om, real_cpu
    return H, wk, pools, inp, n_tok, max_tokens


def _check_oracle(om, real_cpu, lens, slots, has_init, reqs, pool, out):
    """The device-metadata prefill against the oracle token loop: outputs of
    every real row, state and tail of every sequence and checkpoint slot."""
    ref = prefill_oracle(om, real_cpu, lens, slots, has_init, reqs)
    assert torch.isfinite(out.float()).all()
    err = hp.block_rel_err(hp.f64(out), ref, 1)
    assert err <= hp.prefill_out_tol(om.act), f"outputs: {err:.3e}"
    om.check_slots(pool, list(slots) + [r[2] for r in reqs])


def _run_dev(pool, wk, inp, lens, slots, has_init, reqs, max_tokens, out, stream=None):
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
    hi = torch.tensor(has_init, dtype=torch.uint8, device="cuda")
    rq = torch.tensor(reqs, dtype=torch.int32, device="cuda").reshape(-1, 3) if reqs else None
    ws = torch.empty(kda.kda_prefill_workspace_bytes_bound(pool, len(lens), max_tokens, len(reqs)),
                     dtype=torch.uint8, device="cuda")
    kda.kda_prefill_chunked_dev(pool, wk, kda.make_io(inp, out), cu, sl, hi, max_tokens, rq, ws, stream=stream)
    return cu, sl, hi, rq, ws


@pytest.mark.parametrize("act", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_device_tables_match_host_tables_bitexact(act):
    lens = [1, 2, 3, 63, 64, 65, 130, 0, 200]
    slots = [3, 9, 1, 4, 0, 7, 12, 30, 5]
    has_init = [0, 1, 1, 0, 1, 0, 1, 1, 0]
    reqs = [(5, 64, 20), (5, 65, 21), (6, 64, 22), (6, 128, 23), (8, 200, 24), (3, 63, 25), (0, 1, 26),
            (8, 64, 27)]
    H, wk, (pa, pb), inp, n_tok, max_tokens, om, real_cpu = _setup(act, 61, lens, want_oracle=True)
    real = {k: v[:n_tok].contiguous() for k, v in inp.items()}
    out_a = torch.full((n_tok, H, D), 7.0, dtype=act, device="cuda")
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pa, cu), dtype=torch.uint8, device="cuda")
    kda.kda_prefill_chunked(pa, wk, kda.make_io(real, out_a), cu, slots, has_init, 64, reqs, ws)
    out_b = torch.full((max_tokens, H, D), 7.0, dtype=act, device="cuda")
    _run_dev(pb, wk, inp, lens, slots, has_init, reqs, max_tokens, out_b)
    torch.cuda.synchronize()
    assert kda.kda_poll_device_error(pb) == (kda.KDA_OK, 0)
    assert torch.equal(out_b[:n_tok], out_a)
    assert torch.all(out_b[n_tok:] == 7.0), "rows past cu_seqlens[N] are never written"
    assert torch.equal(pb.states(), pa.states()) and torch.equal(pb.tails(), pa.tails())
    _check_oracle(om, real_cpu, lens, slots, has_init, reqs, pb, out_b[:n_tok])


def test_device_tables_inside_a_cuda_graph():
    """Long enough (66 chunks) that the call overlaps the chain and the norm on
    its side streams, which the graph captures too."""
    lens = [40, 4100, 64]
    slots, has_init, reqs = [2, 6, 11], [1, 0, 1], [(1, 4096, 20), (1, 4100, 21)]
    H, wk, (pa, pb), inp, n_tok, max_tokens = _setup(torch.bfloat16, 67, lens)
    start = pa.states().clone(), pa.tails().clone()
    out_a = torch.empty(max_tokens, H, D, dtype=torch.bfloat16, device="cuda")
    _run_dev(pa, wk, inp, lens, slots, has_init, reqs, max_tokens, out_a)
    torch.cuda.synchronize()
    out_b = torch.empty(max_tokens, H, D, dtype=torch.bfloat16, device="cuda")
    # the first call of this process has already set the kernels' attributes
    stream = torch.cuda.Stream()
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
    hi = torch.tensor(has_init, dtype=torch.uint8, device="cuda")
    rq = torch.tensor(reqs, dtype=torch.int32, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_bytes_bound(pb, 3, max_tokens, 2), dtype=torch.uint8, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kda.kda_prefill_chunked_dev(pb, wk, kda.make_io(inp, out_b), cu, sl, hi, max_tokens, rq, ws, stream=stream)
    # capture enqueued nothing: pb still holds the start state
    torch.cuda.synchronize()
    assert torch.equal(pb.states(), start[0])
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_b[:n_tok], out_a[:n_tok])
    assert torch.equal(pb.states(), pa.states()) and torch.equal(pb.tails(), pa.tails())


@pytest.mark.parametrize("case", ["slot_range", "repeated_slot", "mid_chunk_request", "decreasing_cu",
                                  "past_max_tokens"])
def test_bad_device_metadata_sets_the_error_word_and_changes_nothing(case):
    lens, slots, has_init, reqs = [70, 130], [1, 2], [1, 0], [(1, 64, 5)]
    H, wk, (pa, _), inp, n_tok, max_tokens = _setup(torch.bfloat16, 71, lens)
    if case == "slot_range":
        slots = [1, 32]
    elif case == "repeated_slot":
        reqs = [(1, 64, 1)]
    elif case == "mid_chunk_request":
        reqs = [(1, 65, 5)]
    before = pa.states().clone(), pa.tails().clone()
    out = torch.full((max_tokens, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    if case == "decreasing_cu":
        cu[1] = 250
    if case == "past_max_tokens":
        cu[2] = max_tokens + 1
    sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
    hi = torch.tensor(has_init, dtype=torch.uint8, device="cuda")
    rq = torch.tensor(reqs, dtype=torch.int32, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_bytes_bound(pa, 2, max_tokens, 1), dtype=torch.uint8, device="cuda")
    kda.kda_prefill_chunked_dev(pa, wk, kda.make_io(inp, out), cu, sl, hi, max_tokens, rq, ws)
    st, flags = kda.kda_poll_device_error(pa)
    expect = kda.KDA_DEVERR_SLOT_RANGE if case == "slot_range" else kda.KDA_DEVERR_META
    assert st == kda.KDA_ERR_DEVICE and flags & expect
    assert torch.equal(pa.states(), before[0]) and torch.equal(pa.tails(), before[1])
    assert torch.all(out == 7.0)


def test_device_metadata_host_errors():
    H, wk, (pa, _), inp, n_tok, max_tokens = _setup(torch.bfloat16, 73, [64])
    out = torch.empty(max_tokens, H, D, dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, 64], dtype=torch.int32, device="cuda")
    sl = torch.tensor([0], dtype=torch.int32, device="cuda")
    hi = torch.tensor([0], dtype=torch.uint8, device="cuda")
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_chunked_dev(pa, wk, kda.make_io(inp, out), cu, sl, hi, max_tokens, None, small)
    assert e.value.status == kda.KDA_ERR_WORKSPACE
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_chunked_dev(pa, wk, kda.make_io(inp, out), cu, sl, hi, -1, None, small)
    assert e.value.status == kda.KDA_ERR_INVALID_ARG
    assert kda.kda_poll_device_error(pa) == (kda.KDA_OK, 0)


@pytest.mark.parametrize("seed", [101, 202, 303])
def test_random_metadata_device_equals_host_bitexact(seed):
    """Seeded random batches: 1..9 sequences of 0..300 tokens, shuffled slots,
    random resume flags and checkpoint requests at random chunk ends and
    sequence ends.  Device-built tables must give the host-built tables'
    outputs, states and tails bit for bit."""
    rng = np.random.default_rng(seed)
    N = int(rng.integers(1, 10))
    lens = [int(x) for x in rng.integers(0, 301, N)]
    order = rng.permutation(32)
    slots = [int(x) for x in order[:N]]
    has_init = [int(x) for x in rng.integers(0, 2, N)]
    free = [int(x) for x in order[N:]]
    reqs = []
    for n, L in enumerate(lens):
        ends = sorted({p for p in range(64, L, 64)} | ({L} if L else set()))
        for pos in ends:
            if free and rng.random() < 0.4:
                reqs.append((n, pos, free.pop()))
    H, wk, (pa, pb), inp, n_tok, max_tokens, om, real_cpu = _setup(torch.bfloat16, seed, lens, want_oracle=True)
    real = {k: v[:n_tok].contiguous() for k, v in inp.items()}
    out_a = torch.full((max(n_tok, 1), H, D), 7.0, dtype=torch.bfloat16, device="cuda")[:n_tok]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ws = torch.empty(max(kda.kda_prefill_workspace_bytes(pa, cu), 256), dtype=torch.uint8, device="cuda")
    kda.kda_prefill_chunked(pa, wk, kda.make_io(real, out_a), cu, slots, has_init, 64, reqs, ws)
    out_b = torch.full((max_tokens, H, D), 7.0, dtype=torch.bfloat16, device="cuda")
    _run_dev(pb, wk, inp, lens, slots, has_init, reqs, max_tokens, out_b)
    torch.cuda.synchronize()
    assert kda.kda_poll_device_error(pb) == (kda.KDA_OK, 0)
    assert torch.equal(out_b[:n_tok], out_a)
    assert torch.all(out_b[n_tok:] == 7.0)
    assert torch.equal(pb.states(), pa.states()) and torch.equal(pb.tails(), pa.tails())
    _check_oracle(om, real_cpu, lens, slots, has_init, reqs, pb, out_b[:n_tok])
