"""Shared test helpers: tolerance metric, conversions between the GPU pool's
layout and the oracle's, and a mirrored GPU/oracle pool driver."""

from __future__ import annotations

import numpy as np
import torch

# Tolerances (max relative error per block, see block_rel_err).
STATE_TOL = 1e-4      # fp32 state
OUT_TOL_BF16 = 2e-2   # bf16 outputs
OUT_TOL_F32 = 1e-4    # fp32 outputs of the decode / verify step (fp32 CUDA-core arithmetic)
# fp32 outputs of the chunked prefill.  Its products run on the tensor cores
# as three bf16 products of hi/lo splits, which keep about 16 mantissa bits:
# each product term carries a relative error near 2^-17 (7.6e-6), a 128-term
# sum about sqrt(128) times that relative to the row's largest value
# (8.6e-5), and O = Q S + P U adds two such sums after the state itself was
# re-split in the same way; 5e-4 bounds that with margin.  The state keeps
# the 1e-4 bound.
OUT_TOL_F32_PREFILL = 5e-4


def block_rel_err(x, ref, block_dims: int) -> float:
    """max over blocks of max|x - ref| / max|ref|, a block being the trailing
    ``block_dims`` axes (one (token, head) output row, or one (slot, head)
    state matrix)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    if x.size == 0:
        return 0.0
    axes = tuple(range(x.ndim - block_dims, x.ndim))
    num = np.max(np.abs(x - ref), axis=axes)
    den = np.max(np.abs(ref), axis=axes)
    den = np.where(den == 0.0, 1.0, den)
    return float(np.max(num / den))


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_inputs(inp: dict) -> dict:
    return {k: f64(v) for k, v in inp.items()}


def oracle_weights(w: dict) -> dict:
    return {k: f64(v) for k, v in w.items()}


def gpu_state_as_oracle(states_slot: torch.Tensor) -> np.ndarray:
    """GPU slot state [H][d_v][d_k] (S^T) -> oracle S [H][d_k][d_v]."""
    return f64(states_slot).transpose(0, 2, 1)


def to_device(inp: dict, device="cuda") -> dict:
    return {k: v.to(device).contiguous() for k, v in inp.items()}


def out_tol(act: torch.dtype) -> float:
    return OUT_TOL_BF16 if act == torch.bfloat16 else OUT_TOL_F32


def prefill_out_tol(act: torch.dtype) -> float:
    return OUT_TOL_BF16 if act == torch.bfloat16 else OUT_TOL_F32_PREFILL


def head_subset(inp: dict, w: dict, heads, H: int, dk: int, dv: int):
    """Slices per-token inputs and weights down to `heads` (heads are
    independent, so the oracle can check a sample of them at full length)."""
    heads = list(heads)
    sub = {k: v[:, heads] for k, v in inp.items()}
    chans = conv_channels(heads, H, dk, dv)
    return sub, {"conv_w": w["conv_w"][chans], "norm_w": w["norm_w"]}


def conv_channels(heads, H: int, dk: int, dv: int) -> np.ndarray:
    """Conv-channel indices (q, then k, then v) of the given heads."""
    q = [h * dk + i for h in heads for i in range(dk)]
    k = [H * dk + h * dk + i for h in heads for i in range(dk)]
    v = [2 * H * dk + h * dv + j for h in heads for j in range(dv)]
    return np.array(q + k + v)
