"""Pins of the plain prefix-retention model (oracle/prefix_policy.py).

Every expected plan below was worked out by hand from the rule: a prefix's
state is saved on its second hit, reused by later prompts that share it, and
the least recently used saved prefix gives its slot up when the cache is
full.  A mutation test checks that a planted mistake in the model fails one
of these pins.
"""

from __future__ import annotations

import random
import types
from pathlib import Path

import pytest

from oracle import prefix_policy as pp

B = 64
P = list(range(1000, 1200))                       # 200 tokens: 3 blocks
Q = P[:130] + list(range(5000, 5070))             # shares 2 blocks with P
S = P[:128] + list(range(9000, 9172))             # 300 tokens, shares 2 blocks
X = list(range(20000, 20100))                     # 100 tokens: 1 block
E = list(range(30000, 30128))                     # exactly 2 blocks


def pin_second_hit_and_reuse(mod):
    c = mod.PrefixPolicy(B, [7, 5], 1000)
    expect = [
        (P, (0, -1, -1, -1)),      # first sight: counted only
        (P, (0, -1, 192, 5)),      # second hit: save the 3-block prefix, lowest slot first
        (P, (192, 5, -1, -1)),     # reuse it
        (Q, (0, -1, 128, 7)),      # the shared 2-block prefix has 4 hits: save it
        (P, (192, 5, -1, -1)),
        (S, (128, 7, -1, -1)),     # reuse the shared 2 blocks; its own blocks are new
        (X, (0, -1, -1, -1)),
        (X, (0, -1, 64, 5)),       # full: the least recently used saved prefix (P, 3 blocks) gives up slot 5
        (P, (128, 7, 192, 5)),     # reuse 2 blocks, save 3 again; the victim is X, never the reused prefix
    ]
    for toks, want in expect:
        assert c.plan(toks) == want, (len(toks), want)
    assert c.saved() == {7: 128, 5: 192}
    assert c.forget(7) and not c.forget(7)
    assert c.saved() == {5: 192}
    assert c.plan(Q) == (0, -1, 192, 7)            # Q's own 3-block prefix reached 2 hits


def pin_one_token_left_and_no_victim(mod):
    c = mod.PrefixPolicy(B, [0], 1000)
    assert c.plan(E) == (0, -1, -1, -1)
    assert c.plan(E) == (0, -1, 128, 0)            # the whole prompt (2 blocks) is saved
    assert c.plan(E) == (0, -1, 64, 0)             # not reusable (no token left): 1 block takes the slot
    assert c.plan(E) == (64, 0, -1, -1)            # the only victim would be the reused prefix: no admission
    assert c.saved() == {0: 64}


def pin_short_and_empty_prompts(mod):
    c = mod.PrefixPolicy(B, [1, 2], 1000)
    for _ in range(3):
        assert c.plan([]) == (0, -1, -1, -1)
        assert c.plan(list(range(63))) == (0, -1, -1, -1)
    assert c.saved() == {} and c.n_unsaved() == 0
    assert c.plan(list(range(64))) == (0, -1, -1, -1)
    assert c.plan(list(range(64))) == (0, -1, 64, 1)
    assert c.plan(list(range(64))) == (0, -1, -1, -1)   # 64 tokens: a 1-block prefix leaves none to compute
    assert c.plan(list(range(65))) == (64, 1, -1, -1)


def pin_tracking_bound(mod):
    T = list(range(40000, 40320))                  # 5 blocks
    c = mod.PrefixPolicy(B, [3], 2)
    assert c.plan(T) == (0, -1, -1, -1)
    assert c.n_unsaved() == 2                      # only the 2 most recent (4 and 5 blocks) stay tracked
    assert c.plan(T) == (0, -1, 320, 3)            # 4 and 5 blocks have 2 hits, 1..3 start again at 1
    assert c.saved() == {3: 320} and c.n_unsaved() == 2
    # 5 blocks cannot be reused (no token left); 4 blocks (3 hits) takes the
    # only slot from 5 blocks, then is reused, and 5 blocks finds no victim
    assert c.plan(T) == (0, -1, 256, 3)
    assert c.saved() == {3: 256} and c.n_unsaved() == 2
    assert c.plan(T) == (256, 3, -1, -1)


PINS = [pin_second_hit_and_reuse, pin_one_token_left_and_no_victim, pin_short_and_empty_prompts,
        pin_tracking_bound]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_policy_pins(pin):
    pin(pp)


def test_policy_random_streams_keep_the_invariants():
    rng = random.Random(5)
    bases = [[rng.randrange(1 << 20) for _ in range(rng.randrange(64, 700))] for _ in range(6)]
    c = pp.PrefixPolicy(128, [9, 4, 11], 40)
    admitted = {}  # slot -> prefix saved there
    for _ in range(400):
        b = rng.choice(bases)
        toks = b[:rng.randrange(0, len(b) + 1)] + [rng.randrange(1 << 20) for _ in range(rng.randrange(0, 90))]
        hit, hs, ap, aslot = c.plan(toks)
        assert hit % 128 == 0 and hit <= max(0, len(toks) - 1)
        if hit:
            assert admitted[hs] == tuple(toks[:hit]), "reused state was saved for this exact prefix"
        else:
            assert hs == -1
        if ap >= 0:
            assert ap % 128 == 0 and hit < ap <= len(toks) and aslot in (9, 4, 11) and aslot != hs
            admitted[aslot] = tuple(toks[:ap])
        sv = c.saved()
        assert len(sv) <= 3 and set(sv) <= {9, 4, 11}
        assert c.n_unsaved() <= 40


MUTATIONS = [
    ("admit on the first hit", "if e[0] >= 2 and e[1] < 0:", "if e[0] >= 1 and e[1] < 0:"),
    ("reuse with no token left", "for i in range((n - 1) // B if n > 0 else 0, 0, -1):",
     "for i in range(n // B, 0, -1):"),
    ("evict the most recent", "_, victim = min(saved)", "_, victim = max(saved)"),
    ("highest free slot first", "slot = self.free.pop(0)", "slot = self.free.pop()"),
    ("may evict the reused prefix", "if e[1] >= 0 and p != keep]", "if e[1] >= 0]"),
    ("admit the shortest", "for i in range(nb, hit, -1):", "for i in range(hit + 1, nb + 1):"),
    ("count only up to the reused prefix", "for i in range(1, nb + 1):\n            e = self.entries.setdefault",
     "for i in range(1, hit + 1):\n            e = self.entries.setdefault"),
    ("drop the most recent unsaved", "for _, p in unsaved[:max(0, len(unsaved) - self.max_tracked)]:",
     "for _, p in unsaved[min(len(unsaved), self.max_tracked):]:"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_policy_mistake_fails_a_pin(name, old, new):
    src = Path(pp.__file__).read_text()
    assert src.count(old) == 1, name
    mod = types.ModuleType("mutant_policy")
    exec(compile(src.replace(old, new), "mutant_policy", "exec"), mod.__dict__)
    failed = 0
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, KeyError, IndexError):
            failed += 1
    assert failed > 0, f"no pin notices: {name}"
