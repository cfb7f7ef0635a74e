"""GPU parity of the fused decode / speculative-verify kernel against the
oracle, bit-exact bookkeeping, and the host/device error paths."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from hybrid_linear_attention_03_gb300 import build as kbuild
from hybrid_linear_attention_03_gb300 import inputs as I
from hybrid_linear_attention_03_gb300 import kda

import helpers as hp
from mirror import Mirror

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kda.lib()


def _weights(seed, H, D, act):
    return I.layer_weights(seed, H, D, D, 4, act)


def _tokens(seed, idx, n, H, D, act, mu=2.0):
    return I.token_inputs(seed, idx, n, H, D, D, mu, act)


def test_tiny_fp32_decode_matches_oracle():
    """Tiny fp32 workload: 1 sequence, 2 heads, d = 16, 8 decode steps from zero."""
    wl = I.TINY_DECODE
    m = Mirror(wl.num_slots, wl.H, wl.dk, wl.act, wl.weights(), wl.eps_l2, wl.eps_rms)
    for step in range(wl.extra["steps"]):
        out, ref = m.decode([0], wl.tokens(100 + step, 1))
        assert hp.block_rel_err(hp.f64(out), ref, 1) <= hp.OUT_TOL_F32
    assert m.state_err(0) <= hp.STATE_TOL
    assert m.tail_equal(0)
    st, flags = kda.kda_poll_device_error(m.gpu)
    assert st == kda.KDA_OK and flags == 0


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_decode_chain_matches_oracle(D, act):
    """Chained decode steps on a scattered slot list: every step's output,
    then the end states and tails."""
    H = 3
    m = Mirror(16, H, D, act, _weights(7, H, D, act))
    slots = [9, 2, 14, 0, 5]
    for step in range(6):
        out, ref = m.decode(slots, _tokens(7, 10 + step, len(slots), H, D, act))
        assert hp.block_rel_err(hp.f64(out), ref, 1) <= hp.out_tol(act)
    for s in slots:
        assert m.state_err(s) <= hp.STATE_TOL
        assert m.tail_equal(s)
    for s in set(range(16)) - set(slots):
        assert torch.all(m.gpu.states()[s] == 0), "an untouched slot changed"


@pytest.mark.parametrize("B", [1, 12, 20, 40])
def test_verify_matches_oracle(B):
    """B sequences x T = 8 drafts (H = 8, d = 128, bf16).  Snapshots go to a
    shuffled table and each sequence's start slot doubles as its snapshot 0."""
    H, D, T, act = 8, 128, 8, torch.bfloat16
    ns = B * T
    m = Mirror(ns, H, D, act, _weights(11, H, D, act))
    table = I.permutation(11, B, ns).reshape(B, T)
    m.verify(table[:, 0], table, T, _tokens(11, 1, B * T, H, D, act))  # warm-up launch
    starts = table[:, T - 1].copy()
    taken = set(int(x) for x in starts)
    rest = [int(x) for x in I.permutation(11, 1000 + B, ns) if int(x) not in taken]
    table2 = np.array([[starts[b]] + rest[b * (T - 1):(b + 1) * (T - 1)] for b in range(B)], dtype=np.int32)
    assert kda.kda_check_slots(m.gpu, starts, table2.reshape(-1)) == kda.KDA_OK
    out, ref = m.verify(starts, table2, T, _tokens(11, 2, B * T, H, D, act))
    assert hp.block_rel_err(hp.f64(out), ref, 1) <= hp.OUT_TOL_BF16
    for s in table2.reshape(-1):
        assert m.state_err(int(s)) <= hp.STATE_TOL
        assert m.tail_equal(int(s))


@pytest.mark.parametrize("T", [1, 3, 16])
def test_verify_draft_counts_match_oracle(T):
    """The draft-count edges: one draft, an odd count and the maximum (16),
    3 sequences (H = 4, d = 128, bf16), each continuing from a warmed slot
    with its snapshots in a shuffled table."""
    H, D, B, act = 4, 128, 3, torch.bfloat16
    ns = 2 * B * T + B
    m = Mirror(ns, H, D, act, _weights(13, H, D, act))
    perm = [int(x) for x in I.permutation(13, T, ns)]
    warm_in, warm_snap = perm[:B], np.array(perm[B:B + B * T], dtype=np.int32).reshape(B, T)
    m.verify(warm_in, warm_snap, T, _tokens(13, 1, B * T, H, D, act))
    starts = warm_snap[:, T - 1].copy()
    rest = [x for x in perm if x not in set(int(v) for v in starts)][:B * T]
    table = np.array(rest, dtype=np.int32).reshape(B, T)
    assert kda.kda_check_slots(m.gpu, starts, table.reshape(-1)) == kda.KDA_OK
    out, ref = m.verify(starts, table, T, _tokens(13, 2, B * T, H, D, act))
    assert hp.block_rel_err(hp.f64(out), ref, 1) <= hp.OUT_TOL_BF16
    for s in table.reshape(-1):
        assert m.state_err(int(s)) <= hp.STATE_TOL
        assert m.tail_equal(int(s))


@pytest.mark.parametrize("D", [32, 64])
@pytest.mark.parametrize("act", [torch.float32, torch.bfloat16], ids=["f32", "bf16"])
def test_verify_other_head_sizes_match_oracle(D, act):
    """Verify (T = 5 drafts, 4 sequences, H = 3) at the smaller head sizes the
    step kernel is built for, in both activation dtypes."""
    H, B, T = 3, 4, 5
    ns = B * T + B
    m = Mirror(ns, H, D, act, _weights(17, H, D, act))
    perm = [int(x) for x in I.permutation(17, D, ns)]
    ins, table = perm[:B], np.array(perm[B:B + B * T], dtype=np.int32).reshape(B, T)
    m.verify(ins, table, T, _tokens(17, 1, B * T, H, D, act))  # from zero slots
    starts = table[:, T - 1].copy()  # each sequence continues from its last snapshot, which is also its snapshot 0
    rest = [x for x in perm if x not in set(int(v) for v in starts)]
    table2 = np.array([[int(starts[b])] + rest[b * (T - 1):(b + 1) * (T - 1)] for b in range(B)], dtype=np.int32)
    assert kda.kda_check_slots(m.gpu, starts, table2.reshape(-1)) == kda.KDA_OK
    out, ref = m.verify(starts, table2, T, _tokens(17, 2, B * T, H, D, act))
    tol = hp.out_tol(act)
    assert hp.block_rel_err(hp.f64(out), ref, 1) <= tol
    for s in table2.reshape(-1):
        assert m.state_err(int(s)) <= hp.STATE_TOL
        assert m.tail_equal(int(s))


def test_verify_snapshots_equal_decode_steps_bitexact():
    """Snapshot t of one verify launch equals t + 1 decode launches, bit for
    bit (state, tail and outputs)."""
    H, D, T, act = 4, 128, 8, torch.bfloat16
    pool = kda.StatePool(24, H, D, D, act)
    wd = hp.to_device(_weights(5, H, D, act))
    w = kda.make_weights(wd["conv_w"], wd["norm_w"])
    warm = hp.to_device(_tokens(5, 0, 2 * 8, H, D, act))
    o = torch.empty(16, H, D, dtype=act, device="cuda")
    kda.kda_verify(pool, w, kda.make_io(warm, o), torch.tensor([0, 1], dtype=torch.int32, device="cuda"),
                   torch.tensor([2, 3, 4, 5, 6, 7, 8, 0, 9, 10, 11, 12, 13, 14, 15, 1], dtype=torch.int32,
                                device="cuda"), 2, 8)
    kda.kda_state_checkpoint(pool, [0], [20])  # decode copy starts from the same state
    inp = hp.to_device(_tokens(5, 1, T, H, D, act))
    vo = torch.empty(T, H, D, dtype=act, device="cuda")
    snaps = torch.arange(2, 2 + T, dtype=torch.int32, device="cuda")
    kda.kda_verify(pool, w, kda.make_io(inp, vo), torch.tensor([0], dtype=torch.int32, device="cuda"), snaps, 1, T)
    one = torch.tensor([20], dtype=torch.int32, device="cuda")
    for t in range(T):
        tok = {k: v[t:t + 1] for k, v in inp.items()}
        do = torch.empty(1, H, D, dtype=act, device="cuda")
        kda.kda_decode(pool, w, kda.make_io(tok, do), one, 1)
        assert torch.equal(do[0], vo[t]), f"output differs at draft {t}"
        assert torch.equal(pool.states()[20], pool.states()[2 + t]), f"state differs at draft {t}"
        assert torch.equal(pool.tails()[20], pool.tails()[2 + t]), f"tail differs at draft {t}"


def test_batch_composition_is_bitexact():
    """A 2-draft verify of one sequence alone and the same verify inside a
    batch of 64 give identical bits: outputs, both snapshots and tails."""
    H, D, act, T = 8, 128, torch.bfloat16, 2
    pool = kda.StatePool(256, H, D, D, act)
    wd = hp.to_device(_weights(3, H, D, act))
    w = kda.make_weights(wd["conv_w"], wd["norm_w"])
    g = torch.Generator(device="cpu").manual_seed(0)
    pool.states()[:64].copy_(torch.randn(64, H, D, D, generator=g) * 0.05)
    pool.tails()[:64].copy_(torch.randn(64, 3, pool.n_ch, generator=g).to(act))
    kda.kda_state_checkpoint(pool, list(range(64)), list(range(64, 128)))
    inp = hp.to_device(_tokens(3, 0, 64 * T, H, D, act))
    big = torch.empty(64 * T, H, D, dtype=act, device="cuda")
    ins = torch.arange(64, dtype=torch.int32, device="cuda")
    snaps = torch.stack([ins + 128, ins], 1).reshape(-1).contiguous()  # draft 0 to a spare, draft 1 in place
    kda.kda_verify(pool, w, kda.make_io(inp, big), ins, snaps, 64, T)
    for b in (0, 17, 63):
        tok = {k: v[b * T:(b + 1) * T] for k, v in inp.items()}
        small = torch.empty(T, H, D, dtype=act, device="cuda")
        kda.kda_verify(pool, w, kda.make_io(tok, small), torch.tensor([64 + b], dtype=torch.int32, device="cuda"),
                       torch.tensor([192 + b, 64 + b], dtype=torch.int32, device="cuda"), 1, T)
        assert torch.equal(small, big[b * T:(b + 1) * T])
        assert torch.equal(pool.states()[64 + b], pool.states()[b])
        assert torch.equal(pool.states()[192 + b], pool.states()[128 + b])
        assert torch.equal(pool.tails()[64 + b], pool.tails()[b])


def test_rollback_adopts_snapshot_and_continues():
    """Accepted length a: adopting snapshot a - 1 and decoding on matches the
    oracle run of the first a drafts followed by the next token."""
    H, D, T, act, B = 4, 64, 8, torch.float32, 6
    m = Mirror(B * T + 8, H, D, act, _weights(21, H, D, act))
    table = I.permutation(21, 0, B * T).reshape(B, T)
    ins = table[:, 0].copy()
    m.verify(ins, table, T, _tokens(21, 1, B * T, H, D, act))
    acc = I.integers(21, 1, 1, T, B)
    adopted = [int(table[b, acc[b] - 1]) for b in range(B)]
    # the oracle's rollback: re-run the first a drafts from the start state
    out, ref = m.decode(adopted, _tokens(21, 2, B, H, D, act))
    assert hp.block_rel_err(hp.f64(out), ref, 1) <= hp.OUT_TOL_F32
    for s in adopted:
        assert m.state_err(s) <= hp.STATE_TOL and m.tail_equal(s)


def test_checkpoint_copy_is_bitexact():
    H, D, act = 2, 32, torch.bfloat16
    pool = kda.StatePool(8, H, D, D, act)
    g = torch.Generator(device="cpu").manual_seed(1)
    pool.states().copy_(torch.randn(8, H, D, D, generator=g))
    pool.tails().copy_(torch.randn(8, 3, pool.n_ch, generator=g).to(act))
    before = pool.states().clone(), pool.tails().clone()
    kda.kda_state_checkpoint(pool, [1, 4], [6, 0])
    torch.cuda.synchronize()
    assert torch.equal(pool.states()[6], before[0][1]) and torch.equal(pool.states()[0], before[0][4])
    assert torch.equal(pool.tails()[6], before[1][1]) and torch.equal(pool.tails()[0], before[1][4])
    for s in (1, 2, 3, 4, 5, 7):
        assert torch.equal(pool.states()[s], before[0][s])


def test_state_export_import_round_trip_continues_the_request():
    """A warmed slot exported to host memory and imported into another slot
    (the request moving between replicas) is bit-exact, and decoding from
    the imported copy gives the same outputs as decoding from the original."""
    H, D, act = 2, 32, torch.bfloat16
    m = Mirror(8, H, D, act, _weights(11, H, D, act))
    warm = hp.to_device(_tokens(11, 0, 6, H, D, act))
    out = torch.empty(1, H, D, dtype=act, device="cuda")
    for t in range(6):
        kda.kda_decode(m.gpu, m.w, kda.make_io({k: v[t:t + 1] for k, v in warm.items()}, out),
                       torch.tensor([2], dtype=torch.int32, device="cuda"), 1)
    nb = kda.kda_state_slot_bytes(m.gpu)
    assert nb == H * D * D * 4 + 3 * m.gpu.n_ch * 2
    host = torch.empty(nb, dtype=torch.uint8).pin_memory()
    kda.kda_state_export(m.gpu, 2, host)
    torch.cuda.synchronize()
    kda.kda_state_import(m.gpu, 5, host)
    torch.cuda.synchronize()
    assert torch.equal(m.gpu.states()[5], m.gpu.states()[2]) and torch.equal(m.gpu.tails()[5], m.gpu.tails()[2])
    nxt = hp.to_device(_tokens(11, 1, 3, H, D, act))
    for t in range(3):
        tok = {k: v[t:t + 1] for k, v in nxt.items()}
        oa = torch.empty(1, H, D, dtype=act, device="cuda")
        ob = torch.empty(1, H, D, dtype=act, device="cuda")
        kda.kda_decode(m.gpu, m.w, kda.make_io(tok, oa), torch.tensor([2], dtype=torch.int32, device="cuda"), 1)
        kda.kda_decode(m.gpu, m.w, kda.make_io(tok, ob), torch.tensor([5], dtype=torch.int32, device="cuda"), 1)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob)
    assert torch.equal(m.gpu.states()[5], m.gpu.states()[2])
    with pytest.raises(kda.KdaError) as e:
        kda.kda_state_export(m.gpu, 8, host)
    assert e.value.status == kda.KDA_ERR_SLOT_RANGE
    with pytest.raises(kda.KdaError) as e:
        kda.kda_state_import(m.gpu, 1, host[: nb - 1])
    assert e.value.status == kda.KDA_ERR_INVALID_ARG


def test_out_of_range_device_slot_sets_error_and_skips():
    H, D, act = 2, 16, torch.float32
    m = Mirror(4, H, D, act, _weights(2, H, D, act))
    inp = hp.to_device(_tokens(2, 0, 2, H, D, act))
    out = torch.full((2, H, D), 7.0, dtype=act, device="cuda")
    kda.kda_decode(m.gpu, m.w, kda.make_io(inp, out), torch.tensor([1, 99], dtype=torch.int32, device="cuda"), 2)
    st, flags = kda.kda_poll_device_error(m.gpu)
    assert st == kda.KDA_ERR_DEVICE and flags & kda.KDA_DEVERR_SLOT_RANGE
    assert torch.all(out[1] == 7.0), "the bad item must be skipped"
    assert kda.kda_poll_device_error(m.gpu) == (kda.KDA_OK, 0), "polling clears the word"
    ref = m.ora.run(1, {k: v[0:1] for k, v in hp.oracle_inputs(_tokens(2, 0, 2, H, D, act)).items()}, m.w_ora)
    assert hp.block_rel_err(hp.f64(out[0:1]), ref, 1) <= hp.OUT_TOL_F32


def test_host_argument_errors_enqueue_nothing():
    H, D, act = 2, 16, torch.float32
    pool = kda.StatePool(4, H, D, D, act)
    wd = hp.to_device(_weights(2, H, D, act))
    w = kda.make_weights(wd["conv_w"], wd["norm_w"])
    inp = hp.to_device(_tokens(2, 0, 4, H, D, act))
    out = torch.zeros(4, H, D, dtype=act, device="cuda")
    io = kda.make_io(inp, out)
    sl = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    for T in (0, 17):
        with pytest.raises(kda.KdaError) as e:
            kda.kda_verify(pool, w, io, sl, sl, 2, T)
        assert e.value.status == kda.KDA_ERR_INVALID_ARG
    bad = kda.kda_weights(0, w.norm_w, 1e-6, 1e-5)
    with pytest.raises(kda.KdaError):
        kda.kda_decode(pool, bad, io, sl, 2)
    bad_io = kda.make_io(inp, out)
    bad_io.q = inp["q"].data_ptr() + 4  # misaligned
    with pytest.raises(kda.KdaError):
        kda.kda_decode(pool, w, bad_io, sl, 2)
    kda.kda_decode(pool, w, io, sl, 0)  # B = 0 is a no-op
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(pool.states() == 0)
    assert kda.kda_check_slots(pool, [0, 4]) == kda.KDA_ERR_SLOT_RANGE
    assert kda.kda_check_slots(pool, [1, 1]) == kda.KDA_ERR_ALIAS
    assert kda.kda_check_slots(pool, [0, 1], [0, 2, 1, 2]) == kda.KDA_ERR_ALIAS
    assert kda.kda_check_slots(pool, [0, 1], [1, 2, 0, 3]) == kda.KDA_ERR_ALIAS
    assert kda.kda_check_slots(pool, [0, 1], [0, 2, 1, 3]) == kda.KDA_OK
    with pytest.raises(kda.KdaError) as e:
        kda.kda_state_checkpoint(pool, [0, 1], [2, 2])
    assert e.value.status == kda.KDA_ERR_ALIAS
    with pytest.raises(kda.KdaError) as e:
        kda.kda_state_checkpoint(pool, [0, 1], [1, 2])
    assert e.value.status == kda.KDA_ERR_ALIAS
    with pytest.raises(kda.KdaError) as e:
        kda.kda_state_checkpoint(pool, [0], [9])
    assert e.value.status == kda.KDA_ERR_SLOT_RANGE


@pytest.mark.parametrize("graph", [False, True], ids=["stream", "graph"])
def test_inputs_written_by_the_preceding_kernel(graph):
    """A torch kernel writes each step's inputs on the same stream right
    before kda_decode, as the q/k/v projection of a serving step does.  With
    the pool's default launch options the decode reads its inputs only after
    that kernel has completed, so every output and the end states match the
    oracle, on a plain stream and inside a captured CUDA graph.  The last
    producer before each decode is a 64 MiB copy whose final rows are q."""
    H, D, act, B, steps = 4, 128, torch.bfloat16, 8, 4
    m = Mirror(16, H, D, act, _weights(91, H, D, act))
    slots = [3, 7, 1, 12, 0, 9, 5, 14]
    sl = torch.tensor(slots, dtype=torch.int32, device="cuda")
    toks = [_tokens(91, 20 + s, B, H, D, act) for s in range(steps)]
    pad_rows = (64 << 20) // (H * D * 2)  # q's producer writes 64 MiB ahead of the real rows
    order = ("alpha", "beta", "gate", "v", "k", "q")  # q last: its copy is the kernel right before the decode
    big = {k: torch.full((pad_rows + B,) + tuple(toks[0][k].shape[1:]), float("nan"), dtype=act, device="cuda")
           if k == "q" else torch.full(tuple(toks[0][k].shape), float("nan"), dtype=act, device="cuda")
           for k in order}
    staged = []
    for t in toks:
        d = {k: t[k].cuda() for k in order}
        d["q"] = torch.cat([torch.zeros(pad_rows, H, D, dtype=act), t["q"]]).cuda()
        staged.append(d)
    view = {k: (big[k][pad_rows:] if k == "q" else big[k]) for k in order}
    outs = [torch.empty(B, H, D, dtype=act, device="cuda") for _ in range(steps)]
    ios = [kda.make_io(view, o) for o in outs]
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def run_all():
        for s in range(steps):
            for k in order:
                big[k].copy_(staged[s][k])
            kda.kda_decode(m.gpu, m.w, ios[s], sl, B, stream)

    if graph:
        m.decode([15], _tokens(91, 99, 1, H, D, act))  # the first launch sets attributes, outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run_all()
        torch.cuda.synchronize()
        assert torch.all(m.gpu.states()[slots] == 0), "capture enqueued nothing"
        g.replay()
    else:
        with torch.cuda.stream(stream):
            run_all()
    torch.cuda.synchronize()
    for s in range(steps):
        oi = hp.oracle_inputs(toks[s])
        ref = np.zeros((B, H, D))
        for b, slot in enumerate(slots):
            ref[b] = m.ora.run(slot, {k: v[b:b + 1] for k, v in oi.items()}, m.w_ora)[0]
        assert hp.block_rel_err(hp.f64(outs[s]), ref, 1) <= hp.OUT_TOL_BF16, f"step {s}"
    for slot in slots:
        assert m.state_err(slot) <= hp.STATE_TOL
        assert m.tail_equal(slot)
    assert kda.kda_poll_device_error(m.gpu) == (kda.KDA_OK, 0)


def test_state_prefetch_changes_nothing():
    """kda_state_prefetch is an L2 hint: a decode after it equals the same
    decode without it bit for bit, the pool is untouched by the prefetch
    itself (with and without the weights), and an out-of-range slot in its
    table is skipped silently."""
    H, D, act, B = 4, 128, torch.bfloat16, 3
    ma = Mirror(8, H, D, act, _weights(93, H, D, act))
    mb = Mirror(8, H, D, act, _weights(93, H, D, act))
    slots = [5, 0, 3]
    for m in (ma, mb):
        m.decode(slots, _tokens(93, 1, B, H, D, act))
    torch.cuda.synchronize()
    before = mb.gpu.states().clone(), mb.gpu.tails().clone()
    table = torch.tensor(slots + [99, -1], dtype=torch.int32, device="cuda")
    kda.kda_state_prefetch(mb.gpu, table)
    kda.kda_state_prefetch(mb.gpu, table, weights=mb.w)
    torch.cuda.synchronize()
    assert torch.equal(mb.gpu.states(), before[0]) and torch.equal(mb.gpu.tails(), before[1])
    assert kda.kda_poll_device_error(mb.gpu) == (kda.KDA_OK, 0)
    tok = _tokens(93, 2, B, H, D, act)
    out_a, _ = ma.decode(slots, tok)
    out_b, _ = mb.decode(slots, tok)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b)
    assert torch.equal(ma.gpu.states(), mb.gpu.states()) and torch.equal(ma.gpu.tails(), mb.gpu.tails())
