"""The prefill entry point that allocates nothing.

Some callers cannot allocate device memory (a plugin whose host runtime
reserves all device memory up front and hands none out, or a C caller with
no device allocator).  kda_prefill_chunked_noalloc serves them by running
the chunked prefill in a fixed 64 MiB scratch array compiled into the
library instead of a caller workspace.  Here it is called through the C ABI
twice in a row.  It runs the same deterministic kernels as
kda_prefill_chunked (which takes a workspace), so outputs, states and tails
must equal that call's bit for bit; the second call reuses the array the
first left behind, which shows that no stale scratch byte is read.  Both
calls are also held to the oracle within the tolerances every other GPU
test uses, and a request larger than the array must be refused.  This file
is collected last, so a run that stops at its first failure has already run
every other test.
"""

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
H, D, act = 2, 128, torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kda.lib()


def _pool_and_weights():
    pool = kda.StatePool(16, H, D, D, act)
    w_cpu = I.layer_weights(61, H, D, D, 4, act)
    w = {k: v.cuda() for k, v in w_cpu.items()}
    return pool, w, kda.make_weights(w["conv_w"], w["norm_w"]), w_cpu


def test_noalloc_prefill_matches_workspace_prefill_twice():
    lens = [5, 64, 130, 77]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    slots = [3, 0, 7, 11]
    reqs = [(2, 64, 12), (3, 77, 13)]
    pa, wa, wgt_a, w_cpu = _pool_and_weights()
    pb, wb, wgt_b, _ = _pool_and_weights()
    om = OracleMirror(H, D, act, w_cpu)  # both pools start from zeros, as the oracle pool does
    for call in range(2):  # the second call continues the first (and reuses the scratch)
        inp_cpu = I.token_inputs(61, call, int(cu[-1]), H, D, D, 3.0, act)
        inp = {k: v.cuda() for k, v in inp_cpu.items()}
        init = [call] * len(lens)
        out_a = torch.empty(int(cu[-1]), H, D, dtype=act, device="cuda")
        ws = torch.empty(kda.kda_prefill_workspace_bytes(pa, cu), dtype=torch.uint8, device="cuda")
        kda.kda_prefill_chunked(pa, wgt_a, kda.make_io(inp, out_a), cu, slots, init, 64, reqs, ws)
        out_b = torch.full((int(cu[-1]), H, D), float("nan"), dtype=act, device="cuda")
        kda.kda_prefill_chunked_noalloc(pb, wgt_b, kda.make_io(inp, out_b), cu, slots, init, 64, reqs)
        torch.cuda.synchronize()
        assert torch.equal(out_b, out_a), f"call {call}: outputs differ from the workspace prefill"
        for s in slots + [r[2] for r in reqs]:
            assert torch.equal(pb.states()[s], pa.states()[s]), f"call {call}: state of slot {s}"
            assert torch.equal(pb.tails()[s], pa.tails()[s]), f"call {call}: tail of slot {s}"
        ref = prefill_oracle(om, inp_cpu, lens, slots, init, reqs)
        err = hp.block_rel_err(hp.f64(out_b), ref, 1)
        assert err <= hp.OUT_TOL_BF16, f"call {call}: outputs vs the oracle {err:.3e}"
        om.check_slots(pb, slots + [r[2] for r in reqs])
    assert kda.kda_poll_device_error(pb) == (kda.KDA_OK, 0)


def test_noalloc_prefill_refuses_requests_beyond_the_scratch():
    """The scratch holds the tables and a ring of per-(chunk, head) records
    whose windows shrink to fit; a layer with so many heads that even one
    chunk's records exceed 64 MiB is refused, with nothing enqueued."""
    Hb = 480  # one chunk of 480 heads needs 480 records of 145 KiB: more than 64 MiB
    pool = kda.StatePool(2, Hb, D, D, act)
    w = {k: v.cuda() for k, v in I.layer_weights(61, Hb, D, D, 4, act).items()}
    wgt = kda.make_weights(w["conv_w"], w["norm_w"])
    L = 64
    assert kda.kda_prefill_workspace_bytes(pool, [0, L]) > kda.KDA_NOALLOC_SCRATCH_BYTES
    inp = {k: v.cuda() for k, v in I.token_inputs(61, 9, L, Hb, D, D, 3.0, act).items()}
    out = torch.zeros(L, Hb, D, dtype=act, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_chunked_noalloc(pool, wgt, kda.make_io(inp, out), [0, L], [0], [0])
    assert e.value.status == kda.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(pool.states() == 0)


def test_noalloc_prefill_of_a_long_prompt_runs_in_small_windows():
    """A prompt whose preferred workspace is larger than the scratch (4096
    tokens, 16 heads: 2 windows of 48 chunks x 16 heads of records, about
    218 MiB) runs in the scratch with smaller windows and equals the
    workspace prefill bit for bit."""
    Hs, L = 16, 4096
    pa = kda.StatePool(2, Hs, D, D, act)
    pb = kda.StatePool(2, Hs, D, D, act)
    w = {k: v.cuda() for k, v in I.layer_weights(67, Hs, D, D, 4, act).items()}
    wgt = kda.make_weights(w["conv_w"], w["norm_w"])
    cu = [0, L]
    assert kda.kda_prefill_workspace_bytes(pa, cu) > kda.KDA_NOALLOC_SCRATCH_BYTES
    inp = {k: v.cuda() for k, v in I.token_inputs(67, 0, L, Hs, D, D, 3.0, act).items()}
    out_a = torch.empty(L, Hs, D, dtype=act, device="cuda")
    ws = torch.empty(kda.kda_prefill_workspace_bytes(pa, cu), dtype=torch.uint8, device="cuda")
    kda.kda_prefill_chunked(pa, wgt, kda.make_io(inp, out_a), cu, [1], [0], 64, [(0, 2048, 0)], ws)
    out_b = torch.empty(L, Hs, D, dtype=act, device="cuda")
    kda.kda_prefill_chunked_noalloc(pb, wgt, kda.make_io(inp, out_b), cu, [1], [0], 64, [(0, 2048, 0)])
    torch.cuda.synchronize()
    assert torch.equal(out_b, out_a)
    assert torch.equal(pb.states(), pa.states()) and torch.equal(pb.tails(), pa.tails())
    assert kda.kda_poll_device_error(pb) == (kda.KDA_OK, 0)
