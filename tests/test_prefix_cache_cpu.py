"""The native prefix-state cache (libkda, host only) against the plain model
in oracle/prefix_policy.py: the hand-worked pins, identical plans on random
request streams, and its argument errors.  No GPU is involved."""

from __future__ import annotations

import ctypes
import random

import pytest

from hybrid_linear_attention_03_gb300 import build as kbuild
from hybrid_linear_attention_03_gb300 import kda
from oracle import prefix_policy as pp

import test_prefix_policy as pins


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kbuild.build()
    kda.lib()


class Native:
    """The library's cache behind the model's interface, so the same pins run on it."""

    class PrefixPolicy:
        def __init__(self, block, slots, max_tracked):
            self.c = kda.PrefixCache(block, slots, max_tracked)

        def plan(self, tokens):
            return self.c.plan(tokens)

        def forget(self, slot):
            try:
                self.c.forget(slot)
                return True
            except kda.KdaError as e:
                assert e.status == kda.KDA_ERR_INVALID_ARG
                return False

        def saved(self):
            return self.c.saved()

        def n_unsaved(self):
            return self.c.stats()["n_unsaved"]


@pytest.mark.parametrize("pin", pins.PINS, ids=lambda f: f.__name__)
def test_native_cache_meets_the_pins(pin):
    pin(Native)


@pytest.mark.parametrize("seed,block,n_slots,max_tracked", [(1, 64, 2, 1000), (2, 64, 5, 12), (3, 128, 1, 3),
                                                             (4, 192, 8, 0), (5, 64, 0, 50)])
def test_native_plans_equal_the_model_on_random_streams(seed, block, n_slots, max_tracked):
    rng = random.Random(seed)
    slots = rng.sample(range(1000), n_slots)
    model = pp.PrefixPolicy(block, slots, max_tracked)
    native = kda.PrefixCache(block, slots, max_tracked)
    bases = [[rng.randrange(1 << 31) for _ in range(rng.randrange(block, 6 * block))] for _ in range(5)]
    for step in range(600):
        if step % 37 == 36 and model.saved():
            s = rng.choice(sorted(model.saved()))
            assert model.forget(s)
            native.forget(s)
            continue
        b = rng.choice(bases)
        toks = b[:rng.randrange(0, len(b) + 1)] + [rng.randrange(1 << 31) for _ in range(rng.randrange(0, 2 * block))]
        assert native.plan(toks) == model.plan(toks), step
        assert native.saved() == model.saved(), step
        st = native.stats()
        assert st["n_unsaved"] == model.n_unsaved() and st["n_saved"] == len(model.saved())
        assert st["n_free"] == n_slots - st["n_saved"]
    st = native.stats()
    assert st["plans"] > 500 and st["admissions"] >= st["evictions"]


def test_native_cache_argument_errors():
    L = kda.lib()
    with pytest.raises(kda.KdaError) as e:
        kda.PrefixCache(0, [1], 10)
    assert e.value.status == kda.KDA_ERR_INVALID_ARG
    with pytest.raises(kda.KdaError) as e:
        kda.PrefixCache(96, [1], 10)
    assert e.value.status == kda.KDA_ERR_INVALID_ARG
    with pytest.raises(kda.KdaError) as e:
        kda.PrefixCache(64, [1, -2], 10)
    assert e.value.status == kda.KDA_ERR_SLOT_RANGE
    with pytest.raises(kda.KdaError) as e:
        kda.PrefixCache(64, [4, 4], 10)
    assert e.value.status == kda.KDA_ERR_ALIAS
    with pytest.raises(kda.KdaError) as e:
        kda.PrefixCache(64, [1], -1)
    assert e.value.status == kda.KDA_ERR_INVALID_ARG
    c = kda.PrefixCache(64, [1], 10)
    with pytest.raises(kda.KdaError) as e:
        c.forget(1)                                   # holds no saved prefix yet
    assert e.value.status == kda.KDA_ERR_INVALID_ARG
    out = kda.kda_prefix_plan()
    assert L.kda_prefix_cache_plan(c.handle, None, 5, ctypes.byref(out)) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_prefix_cache_plan(c.handle, None, 0, ctypes.byref(out)) == kda.KDA_OK
    assert (out.hit_len, out.hit_slot, out.admit_pos, out.admit_slot) == (0, -1, -1, -1)
    assert L.kda_prefix_cache_plan(None, None, 0, ctypes.byref(out)) == kda.KDA_ERR_INVALID_ARG
    assert L.kda_prefix_cache_saved(c.handle, None, None, 3) == -1
    assert c.stats()["plans"] == 1
