"""Guard bands: the pool, the prefill workspace and the outputs each sit in
the middle of a larger buffer whose 4 KiB bands hold a pattern.  Decode,
verify, chunked prefill with checkpoints, slot copies and state export /
import on the first and the last slots must leave every band untouched (an
out-of-bounds write shows up here without a memory checker)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from hybrid_linear_attention_03_gb300 import build as kbuild
from hybrid_linear_attention_03_gb300 import inputs as I
from hybrid_linear_attention_03_gb300 import kda

import helpers as hp

pytestmark = pytest.mark.gpu

BAND = 4096
PATTERN = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    kbuild.build()
    kda.lib()


def _banded(nbytes: int) -> tuple[torch.Tensor, torch.Tensor]:
    whole = torch.full((nbytes + 2 * BAND,), PATTERN, dtype=torch.uint8, device="cuda")
    return whole, whole[BAND:BAND + nbytes]


def _intact(whole: torch.Tensor) -> bool:
    return bool(torch.all(whole[:BAND] == PATTERN)) and bool(torch.all(whole[-BAND:] == PATTERN))


class BandedPool(kda.StatePool):
    """A slot pool created over the middle of a banded buffer."""

    def __init__(self, num_slots, H, dk, dv, act):
        self.desc = kda.make_desc(num_slots, H, dk, dv, act)
        self.act = act
        self.H, self.dk, self.dv, self.num_slots = H, dk, dv, num_slots
        self.n_ch = H * (2 * dk + dv)
        self.whole, self.buf = _banded(kda.kda_state_pool_bytes(self.desc))
        self.buf.zero_()
        self.handle = kda.kda_state_pool_create(self.desc, self.buf)
        self.layout = kda.kda_state_pool_layout(self.handle)


def _banded_out(rows: int, H: int, D: int, act) -> tuple[torch.Tensor, torch.Tensor]:
    per_row = H * D * torch.tensor([], dtype=act).element_size()
    whole, mid = _banded(rows * per_row)
    return whole, mid.view(act).view(rows, H, D)


@pytest.mark.parametrize("act", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_no_call_writes_outside_its_buffers(act):
    H, D, n_slots = 2, 128, 12
    last = n_slots - 1
    pool = BandedPool(n_slots, H, D, D, act)
    w_dev = hp.to_device(I.layer_weights(61, H, D, D, 4, act))
    w = kda.make_weights(w_dev["conv_w"], w_dev["norm_w"])
    torch.cuda.synchronize()

    # decode on the first and the last slot
    tok = hp.to_device(I.token_inputs(61, 0, 2, H, D, D, 2.0, act))
    o_whole, out = _banded_out(2, H, D, act)
    kda.kda_decode(pool, w, kda.make_io(tok, out), torch.tensor([0, last], dtype=torch.int32, device="cuda"), 2)

    # verify: 2 sequences x 3 drafts, snapshots into the last slots
    T = 3
    vt = hp.to_device(I.token_inputs(61, 1, 2 * T, H, D, D, 2.0, act))
    v_whole, vout = _banded_out(2 * T, H, D, act)
    ins = torch.tensor([0, last], dtype=torch.int32, device="cuda")
    snaps = torch.tensor([0, 5, 6, last, 7, 8], dtype=torch.int32, device="cuda")
    kda.kda_verify(pool, w, kda.make_io(vt, vout), ins, snaps, 2, T)

    # chunked prefill into the last slot (resuming it), a checkpoint into slot 0
    lens = [70, 131]
    pt = hp.to_device(I.token_inputs(61, 2, sum(lens), H, D, D, 2.0, act))
    p_whole, pout = _banded_out(sum(lens), H, D, act)
    cu = np.array([0, lens[0], sum(lens)], dtype=np.int32)
    ws_whole, ws = _banded(kda.kda_prefill_workspace_bytes(pool, cu))
    kda.kda_prefill_chunked(pool, w, kda.make_io(pt, pout), cu, [9, last], [0, 1], 64, [(1, 128, 0)], ws)

    # slot copy onto the last slot, export / import of the last slot
    kda.kda_state_checkpoint(pool, [9], [last])
    host = torch.empty(kda.kda_state_slot_bytes(pool), dtype=torch.uint8).pin_memory()
    kda.kda_state_export(pool, last, host)
    kda.kda_state_import(pool, 0, host)
    torch.cuda.synchronize()

    assert kda.kda_poll_device_error(pool) == (kda.KDA_OK, 0)
    for name, whole in (("pool", pool.whole), ("decode out", o_whole), ("verify out", v_whole),
                        ("prefill out", p_whole), ("workspace", ws_whole)):
        assert _intact(whole), f"a band around the {name} was written"
    assert torch.isfinite(pout.float()).all() and torch.isfinite(vout.float()).all()
