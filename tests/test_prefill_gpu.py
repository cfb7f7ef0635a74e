"""GPU parity of the chunked prefill against the oracle (token loop), its
checkpoints and resume, and decode after prefill."""

from __future__ import annotations

import pytest
import torch

from hybrid_linear_attention_03_gb300 import build as kbuild
from hybrid_linear_attention_03_gb300 import inputs as I
from hybrid_linear_attention_03_gb300 import kda

import helpers as hp
from mirror import Mirror, prefill_gpu, prefill_oracle

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kda.lib()


def _check(m, out, ref, slots, reqs=()):
    assert torch.isfinite(out.float()).all()
    assert hp.block_rel_err(hp.f64(out), ref, 1) <= hp.prefill_out_tol(m.act)
    for s in list(slots) + [r[2] for r in reqs]:
        assert m.state_err(int(s)) <= hp.STATE_TOL, f"state of slot {s}"
        assert m.tail_equal(int(s)), f"tail of slot {s}"


@pytest.mark.parametrize("act", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_prefill_ragged_lengths_match_oracle(act):
    """Lengths around the chunk size (1, 2, 3, 63, 64, 65, 130, 200), half of
    them continuing a warmed slot, with checkpoints at chunk ends and ends."""
    H = 2
    lens = [1, 2, 3, 63, 64, 65, 130, 200]
    N = len(lens)
    m = Mirror(32, H, D, act, I.layer_weights(31, H, D, D, 4, act))
    slots = list(range(N))
    # warm the odd sequences' slots with a first prefill segment
    warm_lens = [0 if n % 2 == 0 else 37 + n for n in range(N)]
    warm = I.token_inputs(31, 0, sum(warm_lens), H, D, D, 2.0, act)
    out = prefill_gpu(m, hp.to_device(warm), warm_lens, slots, [0] * N)
    ref = prefill_oracle(m, warm, warm_lens, slots, [0] * N)
    _check(m, out, ref, slots)
    has_init = [n % 2 for n in range(N)]
    reqs = [(5, 64, 20), (5, 65, 21), (6, 64, 22), (6, 128, 23), (7, 200, 24), (3, 63, 25), (0, 1, 26)]
    inp = I.token_inputs(31, 1, sum(lens), H, D, D, 2.0, act)
    out = prefill_gpu(m, hp.to_device(inp), lens, slots, has_init, reqs)
    ref = prefill_oracle(m, inp, lens, slots, has_init, reqs)
    _check(m, out, ref, slots, reqs)
    assert kda.kda_poll_device_error(m.gpu) == (kda.KDA_OK, 0)


def test_prefill_resume_from_checkpoint_is_bitexact():
    """Prefill 320 tokens with a checkpoint at 192; restore it into a fresh
    slot and prefill the last 128 tokens from there: outputs, end state and
    tail equal the uninterrupted run bit for bit."""
    H, act, L, cut = 3, torch.bfloat16, 320, 192
    m = Mirror(8, H, D, act, I.layer_weights(41, H, D, D, 4, act))
    inp = hp.to_device(I.token_inputs(41, 0, L, H, D, D, 3.0, act))
    full = prefill_gpu(m, inp, [L], [0], [0], [(0, cut, 1)])
    kda.kda_state_checkpoint(m.gpu, [1], [2])
    rest = {k: v[cut:].contiguous() for k, v in inp.items()}
    part = prefill_gpu(m, rest, [L - cut], [2], [1])
    torch.cuda.synchronize()
    assert torch.equal(part, full[cut:])
    assert torch.equal(m.gpu.states()[2], m.gpu.states()[0])
    assert torch.equal(m.gpu.tails()[2], m.gpu.tails()[0])


def test_prefill_beta0_alpha1_keeps_state_bitexact():
    H, act, L = 2, torch.float32, 100
    m = Mirror(4, H, D, act, I.layer_weights(43, H, D, D, 4, act))
    g = torch.Generator(device="cpu").manual_seed(3)
    m.gpu.states()[1].copy_(torch.randn(H, D, D, generator=g))
    before = m.gpu.states()[1].clone()
    inp = I.token_inputs(43, 0, L, H, D, D, 2.0, act)
    inp["beta"].zero_()
    inp["alpha"].fill_(1.0)
    prefill_gpu(m, hp.to_device(inp), [L], [1], [1])
    torch.cuda.synchronize()
    assert torch.equal(m.gpu.states()[1], before)


def test_prefill_strong_decay_takes_exact_path():
    """alpha ~ 0.05 (log-decay span ~190 per chunk, past the split-exponent
    range): finite results that match the oracle."""
    H, act, L = 2, torch.float32, 150
    m = Mirror(4, H, D, act, I.layer_weights(47, H, D, D, 4, act))
    inp = I.token_inputs(47, 0, L, H, D, D, 2.0, act)
    inp["alpha"] = torch.full_like(inp["alpha"], 0.05)
    out = prefill_gpu(m, hp.to_device(inp), [L], [0], [0])
    ref = prefill_oracle(m, inp, [L], [0], [0])
    _check(m, out, ref, [0])


def test_prefill_alpha_edge_values():
    """bf16 alpha with exact zeros, subnormals, exact ones and 1 - 2^-8 mixed
    in: both ways the kernel takes log(alpha) (per-exponent table, and logf
    for zero / subnormal lanes) match the oracle, and alpha = 0 erases."""
    H, act, L = 2, torch.bfloat16, 150
    m = Mirror(4, H, D, act, I.layer_weights(59, H, D, D, 4, act))
    inp = I.token_inputs(59, 0, L, H, D, D, 2.0, act)
    a = inp["alpha"].float()
    idx = torch.arange(a.numel()).view_as(a)
    a = torch.where(idx % 7 == 0, torch.zeros_like(a), a)
    a = torch.where(idx % 11 == 0, torch.full_like(a, 5e-39), a)  # below the smallest normal, 1.18e-38
    a = torch.where(idx % 13 == 0, torch.ones_like(a), a)
    a = torch.where(idx % 17 == 0, torch.full_like(a, 1.0 - 2.0 ** -8), a)
    inp["alpha"] = a.to(act)
    assert (inp["alpha"].float() == 0).any() and ((inp["alpha"].float() > 0) & (inp["alpha"].float() < 1.18e-38)).any()
    out = prefill_gpu(m, hp.to_device(inp), [L], [0], [0])
    ref = prefill_oracle(m, inp, [L], [0], [0])
    _check(m, out, ref, [0])


def test_decode_after_prefill_equals_one_long_run():
    H, act = 4, torch.bfloat16
    m = Mirror(4, H, D, act, I.layer_weights(53, H, D, D, 4, act))
    inp = I.token_inputs(53, 0, 150, H, D, D, 2.0, act)
    prefill_gpu(m, hp.to_device(inp), [150], [3], [0])
    prefill_oracle(m, inp, [150], [3], [0])
    for step in range(5):
        o, r = m.decode([3], I.token_inputs(53, 10 + step, 1, H, D, D, 2.0, act))
        assert hp.block_rel_err(hp.f64(o), r, 1) <= hp.OUT_TOL_BF16
    assert m.state_err(3) <= hp.STATE_TOL and m.tail_equal(3)


def test_prefill_host_errors():
    H, act = 2, torch.bfloat16
    m = Mirror(8, H, D, act, I.layer_weights(2, H, D, D, 4, act))
    inp = hp.to_device(I.token_inputs(2, 0, 10, H, D, D, 2.0, act))
    out = torch.empty(10, H, D, dtype=act, device="cuda")
    io = kda.make_io(inp, out)
    ws = torch.empty(kda.kda_prefill_workspace_bytes(m.gpu, [0, 4, 10]), dtype=torch.uint8, device="cuda")
    cases = [
        (dict(cu=[0, 4, 10], slots=[1, 1], init=[0, 0]), kda.KDA_ERR_ALIAS),
        (dict(cu=[0, 4, 10], slots=[1, 9], init=[0, 0]), kda.KDA_ERR_SLOT_RANGE),
        (dict(cu=[0, 6, 4], slots=[1, 2], init=[0, 0]), kda.KDA_ERR_INVALID_ARG),
        (dict(cu=[0, 4, 10], slots=[1, 2], init=[0, 0], reqs=[(0, 3, 5)]), kda.KDA_ERR_INVALID_ARG),
        (dict(cu=[0, 4, 10], slots=[1, 2], init=[0, 0], reqs=[(1, 6, 2)]), kda.KDA_ERR_ALIAS),
        (dict(cu=[0, 4, 10], slots=[1, 2], init=[0, 0], reqs=[(1, 6, 5), (0, 4, 5)]), kda.KDA_ERR_ALIAS),
        (dict(cu=[0, 4, 10], slots=[1, 2], init=[0, 0], chunk=32), kda.KDA_ERR_UNSUPPORTED),
    ]
    for c, want in cases:
        with pytest.raises(kda.KdaError) as e:
            kda.kda_prefill_chunked(m.gpu, m.w, io, c["cu"], c["slots"], c["init"], c.get("chunk", 64),
                                    c.get("reqs", ()), ws)
        assert e.value.status == want, c
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_chunked(m.gpu, m.w, io, [0, 4, 10], [1, 2], [0, 0], 64, (), ws[:256])
    assert e.value.status == kda.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(m.gpu.states() == 0)


def test_prefill_across_chunk_windows_matches_oracle():
    """72 chunks (3 sequences) run as two chunk windows whose chain launches
    overlap the next window's per-chunk kernels; sequence 1 straddles the
    window boundary and continues from its slot.  Checkpoints on both sides."""
    H, act = 2, torch.bfloat16
    lens = [2000, 1500, 1000]
    m = Mirror(16, H, D, act, I.layer_weights(59, H, D, D, 4, act))
    inp = I.token_inputs(59, 0, sum(lens), H, D, D, 3.0, act)
    reqs = [(0, 1024, 8), (1, 192, 9), (1, 1408, 10), (1, 1500, 11), (2, 1000, 12)]
    out = prefill_gpu(m, hp.to_device(inp), lens, [0, 1, 2], [0, 0, 0], reqs)
    ref = prefill_oracle(m, inp, lens, [0, 1, 2], [0, 0, 0], reqs)
    _check(m, out, ref, [0, 1, 2], reqs)


def test_prefill_window_inside_a_sequence_that_starts_mid_batch():
    """114 chunks in windows of 48: the middle window (chunks 48..95) lies
    inside sequence 1, which starts at row 100, so each CTA there derives its
    tile rows from the chunk index (row 100 + 64 (g - 2)) instead of waiting
    for the chunk table.  Sequence 1 continues a warmed slot, with a
    checkpoint inside that window; the other two start from zero."""
    H, act = 2, torch.bfloat16
    lens = [100, 7000, 70]
    m = Mirror(16, H, D, act, I.layer_weights(61, H, D, D, 4, act))
    warm_lens = [0, 40, 0]
    warm = I.token_inputs(61, 0, sum(warm_lens), H, D, D, 3.0, act)
    out = prefill_gpu(m, hp.to_device(warm), warm_lens, [0, 1, 2], [0, 0, 0])
    ref = prefill_oracle(m, warm, warm_lens, [0, 1, 2], [0, 0, 0])
    _check(m, out, ref, [0, 1, 2])
    inp = I.token_inputs(61, 1, sum(lens), H, D, D, 3.0, act)
    reqs = [(0, 100, 8), (1, 3200, 9), (1, 7000, 10), (2, 70, 11)]
    out = prefill_gpu(m, hp.to_device(inp), lens, [0, 1, 2], [0, 1, 0], reqs)
    ref = prefill_oracle(m, inp, lens, [0, 1, 2], [0, 1, 0], reqs)
    _check(m, out, ref, [0, 1, 2], reqs)
    assert kda.kda_poll_device_error(m.gpu) == (kda.KDA_OK, 0)


def test_prefill_results_do_not_depend_on_batch_composition():
    """A sequence prefilled alone and inside a batch (between sequences whose
    lengths put its chunk ends mid-group) gives the same outputs, state and
    tail bit for bit: nothing past a segment's end reaches its tokens."""
    H, act = 2, torch.bfloat16
    m = Mirror(8, H, D, act, I.layer_weights(53, H, D, D, 4, act))
    X = I.token_inputs(53, 0, 100, H, D, D, 2.0, act)
    Y = I.token_inputs(53, 1, 37, H, D, D, 2.0, act)
    Z = I.token_inputs(53, 2, 50, H, D, D, 2.0, act)
    Z["alpha"][:5].zero_()  # zero and tiny alphas right after X's end
    Z["alpha"][5:9] = 1e-40
    alone = prefill_gpu(m, hp.to_device(X), [100], [0], [0])
    batch = {k: torch.cat([Y[k], X[k], Z[k]]) for k in X}
    out = prefill_gpu(m, hp.to_device(batch), [37, 100, 50], [1, 2, 3], [0, 0, 0])
    torch.cuda.synchronize()
    assert torch.equal(out[37:137], alone)
    assert torch.equal(m.gpu.states()[2], m.gpu.states()[0])
    assert torch.equal(m.gpu.tails()[2], m.gpu.tails()[0])


def test_stream_wait_reports_a_timeout_then_completion():
    """The host watchdog returns KDA_ERR_TIMEOUT while a long prefill is still
    in flight (a zero limit), then KDA_OK once it has finished."""
    H, act, L = 64, torch.bfloat16, 8192
    m = Mirror(2, H, D, act, I.layer_weights(59, H, D, D, 4, act))
    inp = hp.to_device(I.token_inputs(59, 0, L, H, D, D, 2.0, act))
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    prefill_gpu(m, inp, [L], [0], [0], stream=stream)
    assert kda.kda_stream_wait(stream, 0.0) == kda.KDA_ERR_TIMEOUT
    assert kda.kda_stream_wait(stream, 120.0) == kda.KDA_OK
    assert kda.kda_poll_device_error(m.gpu, stream) == (kda.KDA_OK, 0)


def test_one_chunk_sequences_from_zero_state_match_oracle():
    """One-chunk sequences that start from a zero state are finished inside
    the intra-chunk kernel when they make up a large share of a call (the
    chain skips them), and by the chain otherwise.  Both batches, with a
    checkpoint at a short sequence's end and a resumed short sequence among
    them, match the oracle."""
    H, act = 2, torch.bfloat16
    m = Mirror(48, H, D, act, I.layer_weights(41, H, D, D, 4, act))
    # many short sequences: the intra kernel finishes the new ones itself
    lens = [64, 17, 1, 64, 40, 63, 5, 64, 33, 2]
    N = len(lens)
    slots = list(range(N))
    has_init = [0] * N
    has_init[4] = 1  # a short continuation still goes through the chain
    warm = I.token_inputs(41, 0, 24, H, D, D, 2.0, act)
    prefill_gpu(m, hp.to_device(warm), [24], [4], [0])
    prefill_oracle(m, warm, [24], [4], [0])
    reqs = [(1, 17, 30), (7, 64, 31)]
    inp = I.token_inputs(41, 1, sum(lens), H, D, D, 2.0, act)
    out = prefill_gpu(m, hp.to_device(inp), lens, slots, has_init, reqs)
    ref = prefill_oracle(m, inp, lens, slots, has_init, reqs)
    _check(m, out, ref, slots, reqs)
    # one short sequence beside a long one: the chain takes both
    lens2 = [50, 2000]
    slots2 = [20, 21]
    inp2 = I.token_inputs(41, 2, sum(lens2), H, D, D, 2.0, act)
    out2 = prefill_gpu(m, hp.to_device(inp2), lens2, slots2, [0, 0], [(0, 50, 32)])
    ref2 = prefill_oracle(m, inp2, lens2, slots2, [0, 0], [(0, 50, 32)])
    _check(m, out2, ref2, slots2, [(0, 50, 32)])
    assert kda.kda_poll_device_error(m.gpu) == (kda.KDA_OK, 0)
