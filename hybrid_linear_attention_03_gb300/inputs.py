"""Seeded synthetic inputs and the named workloads of the KDA layer step.

This module draws input values only; it holds none of the layer's arithmetic.
It is the one module that both the CUDA side (bench, GPU tests) and the
oracle side (tests, CPU baseline) use, so that both read the same values.

Value recipe (every workload): raw q, k, v ~ N(0, 1); conv weights
~ N(0, 0.25); alpha = sigmoid(N(mu, 1)) per key channel with mu = 2, or 3 for
the long-prefill workloads; beta = sigmoid(N(0, 1)) per (token, head); output
gate logits ~ N(0, 1); RMSNorm weight = 1 + N(0, 0.1).  N(m, s) names the
mean and the standard deviation.  Draws are float32 from numpy's PCG64
(``default_rng``) keyed by a SeedSequence of (seed, purpose, index), then
cast to the activation dtype with round-to-nearest-even.

Shapes follow the pages' serving setting ("vLLM Kimi K3 지원", section
"하이브리드 KV-Cache 관리": per-request KDA state blocks in a slot pool;
section "DSpark를 이용한 Speculative Decoding" and the DSpark page, section
"추론 성능 및 기능": 8 draft tokens per verify step; section "에이전틱 캐시 유지
정책": state checkpoints every 32K tokens and at prompt ends).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 1000

# purposes in the SeedSequence key
_P_WEIGHTS, _P_TOKENS, _P_TABLES = 0, 1, 2


def _rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(x) for x in key]))


def _sigmoid64(x: np.ndarray) -> np.ndarray:
    # input-distribution transform (alpha, beta are drawn as sigmoid(normal))
    return 1.0 / (1.0 + np.exp(-x.astype(np.float64)))


def _cast(a: np.ndarray, act: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(act)


def layer_weights(seed: int, H: int, dk: int, dv: int, W: int = 4,
                  act: torch.dtype = torch.bfloat16) -> dict[str, torch.Tensor]:
    """conv_w [H*(2*dk+dv)][W] (q channels, then k, then v) and norm_w [dv]."""
    rng = _rng(seed, _P_WEIGHTS)
    conv_w = rng.normal(0.0, 0.25, size=(H * (2 * dk + dv), W)).astype(np.float32)
    norm_w = (1.0 + rng.normal(0.0, 0.1, size=(dv,))).astype(np.float32)
    return {"conv_w": _cast(conv_w, act), "norm_w": _cast(norm_w, act)}


def token_inputs(seed: int, index: int, n_tok: int, H: int, dk: int, dv: int,
                 alpha_mu: float = 2.0, act: torch.dtype = torch.bfloat16) -> dict[str, torch.Tensor]:
    """One segment of tokens: q,k [n][H][dk], v [n][H][dv], alpha [n][H][dk],
    beta [n][H], gate [n][H][dv], all on the CPU in ``act``.  ``index`` tells
    independent segments (sequences, steps) apart."""
    rng = _rng(seed, _P_TOKENS, index)
    out = {}
    out["q"] = _cast(rng.standard_normal((n_tok, H, dk), dtype=np.float32), act)
    out["k"] = _cast(rng.standard_normal((n_tok, H, dk), dtype=np.float32), act)
    out["v"] = _cast(rng.standard_normal((n_tok, H, dv), dtype=np.float32), act)
    out["alpha"] = _cast(_sigmoid64(rng.normal(alpha_mu, 1.0, size=(n_tok, H, dk)).astype(np.float32)), act)
    out["beta"] = _cast(_sigmoid64(rng.standard_normal((n_tok, H), dtype=np.float32)), act)
    out["gate"] = _cast(rng.standard_normal((n_tok, H, dv), dtype=np.float32), act)
    return out


def concat_inputs(parts: list[dict[str, torch.Tensor]]) -> dict[str, torch.Tensor]:
    return {k: torch.cat([p[k] for p in parts], dim=0) for k in parts[0]}


def slice_inputs(inp: dict[str, torch.Tensor], a: int, b: int) -> dict[str, torch.Tensor]:
    return {k: v[a:b] for k, v in inp.items()}


def permutation(seed: int, index: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n) (shuffled slot tables)."""
    return _rng(seed, _P_TABLES, index).permutation(n).astype(np.int32)


def integers(seed: int, index: int, low: int, high: int, size) -> np.ndarray:
    """Seeded integers in [low, high] inclusive (accepted lengths, picks)."""
    return _rng(seed, _P_TABLES, index).integers(low, high + 1, size=size).astype(np.int64)


def uniforms(seed: int, index: int, size) -> np.ndarray:
    return _rng(seed, _P_TABLES, index).random(size)


@dataclass(frozen=True)
class Workload:
    """A named workload: shapes, pool size and the value recipe's seed."""
    name: str
    index: int                  # seed = SEED_BASE + index
    H: int
    dk: int
    dv: int
    act: torch.dtype
    alpha_mu: float
    num_slots: int
    W: int = 4
    eps_l2: float = 1e-6
    eps_rms: float = 1e-5
    extra: dict = field(default_factory=dict)

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    def weights(self) -> dict[str, torch.Tensor]:
        return layer_weights(self.seed, self.H, self.dk, self.dv, self.W, self.act)

    def tokens(self, index: int, n_tok: int) -> dict[str, torch.Tensor]:
        return token_inputs(self.seed, index, n_tok, self.H, self.dk, self.dv, self.alpha_mu, self.act)


# The five workloads.  Token-segment indices: 0..63 warm-up segments of the
# decode/verify sequences, 100 + step for decode steps, 200 + b for verify
# drafts, 300 + i for prefill sequences, 400 + i for mixed-step decodes.
TINY_DECODE = Workload("tiny_decode_fp32_b1_h2_d16_8steps", 0, H=2, dk=16, dv=16, act=torch.float32,
                       alpha_mu=2.0, num_slots=4, extra={"B": 1, "steps": 8})
DECODE_B1 = Workload("decode_b1_h64_d128_1000steps", 1, H=64, dk=128, dv=128, act=torch.bfloat16,
                     alpha_mu=2.0, num_slots=256, extra={"B": 1, "steps": 1000, "warm": 512})
VERIFY_B64 = Workload("verify_b64_t8_h64_d128", 2, H=64, dk=128, dv=128, act=torch.bfloat16,
                      alpha_mu=2.0, num_slots=512, extra={"B": 64, "T": 8, "warm": 512})
PREFILL_32K = Workload("prefill_l32768_h64_d128_c64", 3, H=64, dk=128, dv=128, act=torch.bfloat16,
                       alpha_mu=3.0, num_slots=4, extra={"L": 32768, "chunk": 64})
MIXED = Workload("mixed_8prefill_1k_64k_56decode_h64_d128", 4, H=64, dk=128, dv=128, act=torch.bfloat16,
                 alpha_mu=3.0, num_slots=1024,
                 extra={"n_prefill": 8, "n_decode": 56, "warm": 512, "interval": 32768,
                        "resume": 4, "chunk": 64})
# batch-64 single-token decode over the shapes of the verify workload
DECODE_B64 = Workload("decode_b64_h64_d128", 2, H=64, dk=128, dv=128, act=torch.bfloat16,
                      alpha_mu=2.0, num_slots=512, extra={"B": 64, "warm": 512})

WORKLOADS = {w.name: w for w in (TINY_DECODE, DECODE_B1, VERIFY_B64, PREFILL_32K, MIXED, DECODE_B64)}


def mixed_prefill_lengths(wl: Workload = MIXED) -> list[int]:
    """Prefill lengths of the mixed workload: floor(1024 * 64**u), u ~ U[0,1)
    (log-uniform in [1K, 64K])."""
    u = uniforms(wl.seed, 0, wl.extra["n_prefill"])
    return [int(np.floor(1024.0 * 64.0 ** x)) for x in u]


def mixed_plan(wl: Workload = MIXED) -> dict:
    """Slots and checkpoint requests of the mixed workload: decodes in slots
    0..n_decode-1, prefills next, then one fresh slot per checkpoint request
    (every `interval` tokens from the sequence start, and each sequence end)."""
    lens = mixed_prefill_lengths(wl)
    nd, npf, iv = wl.extra["n_decode"], wl.extra["n_prefill"], wl.extra["interval"]
    dec_slots = list(range(nd))
    pf_slots = list(range(nd, nd + npf))
    reqs, nxt = [], nd + npf
    for n, L in enumerate(lens):
        for pos in sorted(set(list(range(iv, L, iv)) + [L])):
            reqs.append((n, pos, nxt))
            nxt += 1
    resume = [int(x) for x in permutation(wl.seed, 5, npf)[:wl.extra["resume"]]]
    return {"lens": lens, "dec_slots": dec_slots, "pf_slots": pf_slots, "reqs": reqs, "next_free": nxt,
            "resume": resume}
