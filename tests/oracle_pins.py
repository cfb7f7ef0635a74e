"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` takes an ``Oracle`` (any build of ``oracle/kda_oracle.c``) and
raises AssertionError when the build disagrees with

* a library routine: ``torch.nn.functional.conv1d`` / ``silu`` /
  ``normalize`` / ``rms_norm`` and ``torch.autograd`` (float64);
* a closed form of the recurrence (zero state, beta = 0, alpha = 0, alpha = 1,
  unit key with beta = 1);
* an invariant (chunked == token loop, split run == one run, permutations of
  key or value channels, head independence, linearity in v);
* a differently-organised brute force (the state written as an explicit
  product of transition matrices).

The same pins run against deliberately broken builds of the oracle in
``test_oracle_mutations.py``; every planted mistake must fail at least one.
The recurrence is the KDA step of "vLLM Kimi K3 지원" (agentlenshq.com), sections
"Kimi K3 아키텍처 개요" (linear attention with a fixed-size recurrent state) and
"Fused Kernels 및 메타데이터 최적화" (conv, recurrent update and RMSNorm fused
into one decode step).
"""

from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

TOL = 1e-11


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol * scale, f"{what}: max abs err {err:.3e} (scale {scale:.3e})"


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _core_inputs(rng, L, dk, dv, unit_k=True):
    q = _unit(rng.standard_normal((L, dk)))
    k = _unit(rng.standard_normal((L, dk))) if unit_k else rng.standard_normal((L, dk))
    v = rng.standard_normal((L, dv))
    alpha = 1.0 / (1.0 + np.exp(-rng.normal(1.0, 1.0, (L, dk))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    return q, k, v, alpha, beta


def _layer_inputs(rng, L, H, dk, dv, W=4):
    inp = {
        "q": rng.standard_normal((L, H, dk)),
        "k": rng.standard_normal((L, H, dk)),
        "v": rng.standard_normal((L, H, dv)),
        "alpha": 1.0 / (1.0 + np.exp(-rng.normal(1.5, 1.0, (L, H, dk)))),
        "beta": 1.0 / (1.0 + np.exp(-rng.standard_normal((L, H)))),
        "gate": rng.standard_normal((L, H, dv)),
    }
    n_ch = H * (2 * dk + dv)
    w = {"conv_w": rng.normal(0.0, 0.5, (n_ch, W)), "norm_w": 1.0 + rng.normal(0.0, 0.1, dv)}
    S0 = rng.standard_normal((H, dk, dv)) * 0.3
    tail0 = rng.standard_normal((W - 1, n_ch))
    return inp, w, S0, tail0


# ----------------------------------------------------------------- a1 conv --

def pin_conv_matches_torch_conv1d(o):
    """a1 == F.silu(F.conv1d(cat(tail, x), w, groups=C)); the tail advances."""
    rng = _rng(1)
    L, n_ch, W = 7, 5, 4
    x = rng.standard_normal((L, n_ch))
    w = rng.standard_normal((n_ch, W))
    tail = rng.standard_normal((W - 1, n_ch))
    y, new_tail, hist = o.conv_silu(x, w, tail, want_hist=True)
    seq = torch.from_numpy(np.concatenate([tail, x], 0).T.copy())[None]  # [1][C][W-1+L]
    ref = F.silu(F.conv1d(seq, torch.from_numpy(w)[:, None, :], groups=n_ch))[0].T.numpy()
    _close(y, ref, what="conv+silu vs torch conv1d")
    full = np.concatenate([tail, x], 0)
    _close(new_tail, full[-(W - 1):], what="tail after the segment")
    for t in range(L):
        _close(hist[t], full[t + 1:t + W], what=f"tail after token {t}")


def pin_conv_identity_taps(o):
    """Taps [0,0,0,1] make the conv the identity, so a1 is SiLU alone."""
    rng = _rng(2)
    x = rng.standard_normal((5, 3))
    w = np.zeros((3, 4))
    w[:, 3] = 1.0
    y, _, _ = o.conv_silu(x, w, rng.standard_normal((3, 3)))
    _close(y, F.silu(torch.from_numpy(x)).numpy(), what="identity conv")


# ------------------------------------------------------------------- a2 L2 --

def pin_l2norm_matches_normalize(o):
    """With eps = 0 the L2 step is torch's normalize; eps sits under the root."""
    rng = _rng(3)
    x = rng.standard_normal((4, 6))
    _close(o.l2norm_rows(x, 0.0), F.normalize(torch.from_numpy(x), dim=-1).numpy(), what="l2 eps=0")
    z = np.zeros((1, 4))
    z[0, 1] = 3.0  # norm 3
    eps = 0.75
    _close(o.l2norm_rows(z, eps)[0, 1], 3.0 / np.sqrt(9.0 + eps), what="l2 eps under the root")


# ------------------------------------------------------------- a5 gated norm --

def pin_gated_norm_matches_rms_norm(o):
    """a5 == F.rms_norm(o, weight=w_n, eps) * sigmoid(g)."""
    rng = _rng(4)
    x = rng.standard_normal((5, 8)) * 3.0
    g = rng.standard_normal((5, 8))
    wn = 1.0 + rng.normal(0.0, 0.3, 8)
    eps = 0.3
    ref = F.rms_norm(torch.from_numpy(x), (8,), weight=torch.from_numpy(wn), eps=eps) * torch.sigmoid(torch.from_numpy(g))
    _close(o.gated_rmsnorm_rows(x, g, wn, eps), ref.numpy(), what="gated rms norm")


# ----------------------------------------------------------- a3 / a4 core --

def pin_update_is_gradient_step(o):
    """One token of a3 is one gradient step of the delta rule:
    S_t = St - beta * d/dSt (1/2 |St^T k - v|^2), St = Diag(alpha) S_{t-1}
    (torch.autograd, float64; d_k != d_v so a transposed operand fails)."""
    rng = _rng(5)
    dk, dv = 5, 3
    q, k, v, alpha, beta = _core_inputs(rng, 1, dk, dv, unit_k=False)
    S0 = rng.standard_normal((dk, dv))
    S1, _, _ = o.core(q, k, v, alpha, beta, S0)
    St = (torch.from_numpy(alpha[0])[:, None] * torch.from_numpy(S0)).requires_grad_(True)
    loss = 0.5 * torch.sum((St.T @ torch.from_numpy(k[0]) - torch.from_numpy(v[0])) ** 2)
    (grad,) = torch.autograd.grad(loss, St)
    _close(S1, (St - float(beta[0]) * grad).detach().numpy(), what="delta-rule gradient step")


def pin_unit_key_recall(o):
    """beta = 1 and |k| = 1: the new state recalls v exactly, S_t^T k = v, for
    any alpha and start state; reading out with q = k returns v."""
    rng = _rng(6)
    dk, dv = 6, 4
    _, k, v, alpha, _ = _core_inputs(rng, 3, dk, dv)
    beta = np.ones(3)
    S0 = rng.standard_normal((dk, dv))
    S, out, hist = o.core(k, k, v, alpha, beta, S0, want_hist=True)
    for t in range(3):
        _close(hist[t].T @ k[t], v[t], what=f"S_t^T k_t = v_t at t={t}")
        _close(out[t], v[t], what=f"readout with q = k at t={t}")


def pin_beta0_alpha1_identity(o):
    """beta = 0 and alpha = 1 leave the state unchanged; o = S^T q."""
    rng = _rng(7)
    dk, dv = 5, 4
    q, k, v, _, _ = _core_inputs(rng, 4, dk, dv)
    S0 = rng.standard_normal((dk, dv))
    S, out, _ = o.core(q, k, v, np.ones((4, dk)), np.zeros(4), S0)
    assert np.array_equal(S, S0), "state moved with beta = 0, alpha = 1"
    _close(out, q @ S0, what="readout of an unchanged state")


def pin_alpha0_erases(o):
    """alpha = 0 erases the history: S_t = beta k v^T."""
    rng = _rng(8)
    dk, dv = 5, 4
    q, k, v, _, beta = _core_inputs(rng, 1, dk, dv, unit_k=False)
    S, _, _ = o.core(q, k, v, np.zeros((1, dk)), beta, rng.standard_normal((dk, dv)))
    _close(S, beta[0] * np.outer(k[0], v[0]), what="alpha = 0")


def pin_beta0_decay_only(o):
    """beta = 0: S_L = Diag(prod_t alpha_t) S_0 (key rows decay, nothing is written)."""
    rng = _rng(9)
    dk, dv, L = 5, 3, 6
    q, k, v, alpha, _ = _core_inputs(rng, L, dk, dv)
    S0 = rng.standard_normal((dk, dv))
    S, _, _ = o.core(q, k, v, alpha, np.zeros(L), S0)
    _close(S, np.prod(alpha, axis=0)[:, None] * S0, what="decay only")


def pin_zero_state_closed_form(o):
    """From S_0 = 0: S_1 = beta k v^T and o_1 = beta (q.k) v."""
    rng = _rng(10)
    dk, dv = 5, 3
    q, k, v, alpha, beta = _core_inputs(rng, 1, dk, dv, unit_k=False)
    S, out, _ = o.core(q, k, v, alpha, beta, np.zeros((dk, dv)))
    _close(S, beta[0] * np.outer(k[0], v[0]), what="S_1 from zero")
    _close(out[0], beta[0] * float(q[0] @ k[0]) * v[0], what="o_1 from zero")


def pin_brute_force_transition_product(o):
    """Tiny brute force organised differently: S_t written as the product of
    explicit transition matrices M_t = (I - beta_t k_t k_t^T) Diag(alpha_t)
    applied to S_0 plus the injected terms, S_t = M_t..M_1 S_0 +
    sum_s M_t..M_{s+1} beta_s k_s v_s^T; o_t = S_t^T q_t."""
    rng = _rng(11)
    dk, dv, L = 3, 2, 5
    q, k, v, alpha, beta = _core_inputs(rng, L, dk, dv, unit_k=False)
    S0 = rng.standard_normal((dk, dv))
    _, out, hist = o.core(q, k, v, alpha, beta, S0, want_hist=True)
    M = [(np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(alpha[t]) for t in range(L)]
    for t in range(L):
        prod = np.eye(dk)
        for s in range(t, -1, -1):
            prod = prod @ M[s]
        St = prod @ S0
        for s in range(t + 1):
            P = np.eye(dk)
            for r in range(t, s, -1):
                P = P @ M[r]
            St = St + P @ (beta[s] * np.outer(k[s], v[s]))
        _close(hist[t], St, what=f"transition product state t={t}")
        _close(out[t], St.T @ q[t], what=f"transition product readout t={t}")


def pin_v_linearity(o):
    """From a zero state, scaling every v by c scales S and o by c."""
    rng = _rng(12)
    dk, dv, L = 4, 3, 5
    q, k, v, alpha, beta = _core_inputs(rng, L, dk, dv)
    S_a, o_a, _ = o.core(q, k, v, alpha, beta, np.zeros((dk, dv)))
    S_b, o_b, _ = o.core(q, k, 2.5 * v, alpha, beta, np.zeros((dk, dv)))
    _close(S_b, 2.5 * S_a, what="linearity S")
    _close(o_b, 2.5 * o_a, what="linearity o")


def pin_chunked_equals_token_loop(o):
    """The chunked (WY/UT) form equals the token loop, ragged last chunk included."""
    rng = _rng(13)
    dk, dv, L = 6, 5, 11
    q, k, v, alpha, beta = _core_inputs(rng, L, dk, dv)
    S0 = rng.standard_normal((dk, dv))
    S_r, o_r, _ = o.core(q, k, v, alpha, beta, S0)
    for C in (1, 4, 11, 16):
        S_c, o_c, _ = o.core(q, k, v, alpha, beta, S0, chunk=C)
        _close(S_c, S_r, what=f"chunked C={C} state")
        _close(o_c, o_r, what=f"chunked C={C} readout")


# ---------------------------------------------------------------- layer --

def pin_layer_first_token_closed_form(o):
    """From a zero state and tail, token 1 through the layer is
    y = w_n * rms_norm(beta (q.k) v) * sigmoid(g), where q, k, v are
    normalize(silu(w[:, W-1] x)) (v not normalised)."""
    rng = _rng(14)
    H, dk, dv, W = 2, 4, 3, 4
    inp, w, _, _ = _layer_inputs(rng, 1, H, dk, dv, W)
    n_ch = H * (2 * dk + dv)
    out, S, _, _, _ = o.layer(inp, w, np.zeros((H, dk, dv)), np.zeros((W - 1, n_ch)), eps_l2=0.0, eps_rms=1e-5)
    last = torch.from_numpy(w["conv_w"][:, W - 1])
    for h in range(H):
        qx = F.silu(last[h * dk:(h + 1) * dk] * torch.from_numpy(inp["q"][0, h]))
        kx = F.silu(last[H * dk + h * dk:H * dk + (h + 1) * dk] * torch.from_numpy(inp["k"][0, h]))
        vx = F.silu(last[2 * H * dk + h * dv:2 * H * dk + (h + 1) * dv] * torch.from_numpy(inp["v"][0, h]))
        qn, kn = F.normalize(qx, dim=0), F.normalize(kx, dim=0)
        b = float(inp["beta"][0, h])
        _close(S[h], (b * torch.outer(kn, vx)).numpy(), what=f"layer S_1 head {h}")
        o1 = b * torch.dot(qn, kn) * vx
        y = F.rms_norm(o1, (dv,), weight=torch.from_numpy(w["norm_w"]), eps=1e-5) * torch.sigmoid(torch.from_numpy(inp["gate"][0, h]))
        _close(out[0, h], y.numpy(), what=f"layer y_1 head {h}")


def pin_layer_split_equals_one_run(o):
    """Running L1 tokens then L2 tokens from the saved state and tail gives
    exactly the single run of L1 + L2 tokens (decode after prefill)."""
    rng = _rng(15)
    H, dk, dv = 2, 4, 3
    inp, w, S0, t0 = _layer_inputs(rng, 9, H, dk, dv)
    out, S, t, _, _ = o.layer(inp, w, S0, t0)
    a = {k2: v2[:4] for k2, v2 in inp.items()}
    b = {k2: v2[4:] for k2, v2 in inp.items()}
    oa, Sa, ta, _, _ = o.layer(a, w, S0, t0)
    ob, Sb, tb, _, _ = o.layer(b, w, Sa, ta)
    assert np.array_equal(np.concatenate([oa, ob]), out), "split run output differs"
    assert np.array_equal(Sb, S) and np.array_equal(tb, t), "split run state differs"


def pin_layer_history_is_prefix_run(o):
    """The per-token history (verify snapshots) equals the end state of the
    prefix run of t + 1 tokens."""
    rng = _rng(16)
    H, dk, dv, L = 2, 3, 4, 5
    inp, w, S0, t0 = _layer_inputs(rng, L, H, dk, dv)
    out, S, t, hs, ht = o.layer(inp, w, S0, t0, want_hist=True)
    for n in range(1, L + 1):
        part = {k2: v2[:n] for k2, v2 in inp.items()}
        _, Sn, tn, _, _ = o.layer(part, w, S0, t0)
        assert np.array_equal(hs[n - 1], Sn) and np.array_equal(ht[n - 1], tn), f"history at {n}"


def pin_layer_chunked_equals_token_loop(o):
    """The layer in chunked form equals the layer as a token loop."""
    rng = _rng(17)
    H, dk, dv, L = 2, 5, 4, 13
    inp, w, S0, t0 = _layer_inputs(rng, L, H, dk, dv)
    out_r, S_r, t_r, _, _ = o.layer(inp, w, S0, t0)
    out_c, S_c, t_c, _, _ = o.layer(inp, w, S0, t0, chunk=4)
    _close(out_c, out_r, what="layer chunked out")
    _close(S_c, S_r, what="layer chunked state")
    assert np.array_equal(t_c, t_r)


def pin_layer_heads_independent(o):
    """Heads do not interact: the H-head run equals H one-head runs."""
    rng = _rng(18)
    H, dk, dv, L, W = 3, 4, 3, 5, 4
    inp, w, S0, t0 = _layer_inputs(rng, L, H, dk, dv, W)
    out, S, _, _, _ = o.layer(inp, w, S0, t0)
    for h in range(H):
        chans = np.r_[h * dk:(h + 1) * dk, H * dk + h * dk:H * dk + (h + 1) * dk,
                      2 * H * dk + h * dv:2 * H * dk + (h + 1) * dv]
        ih = {"q": inp["q"][:, h:h + 1], "k": inp["k"][:, h:h + 1], "v": inp["v"][:, h:h + 1],
              "alpha": inp["alpha"][:, h:h + 1], "beta": inp["beta"][:, h:h + 1], "gate": inp["gate"][:, h:h + 1]}
        wh = {"conv_w": w["conv_w"][chans], "norm_w": w["norm_w"]}
        oh, Sh, _, _, _ = o.layer(ih, wh, S0[h:h + 1], t0[:, chans])
        _close(oh[:, 0], out[:, h], what=f"head {h} out")
        _close(Sh[0], S[h], what=f"head {h} state")


def pin_layer_value_permutation(o):
    """Permuting the value channels (v, gate, w_n, v conv rows) permutes the
    state columns and y."""
    rng = _rng(19)
    H, dk, dv, L = 1, 4, 5, 4
    inp, w, S0, t0 = _layer_inputs(rng, L, H, dk, dv)
    out, S, _, _, _ = o.layer(inp, w, S0, t0)
    p = rng.permutation(dv)
    ip = dict(inp)
    ip["v"] = inp["v"][:, :, p]
    ip["gate"] = inp["gate"][:, :, p]
    vch = 2 * dk + p
    order = np.r_[np.arange(2 * dk), vch]
    wp = {"conv_w": w["conv_w"][order], "norm_w": w["norm_w"][p]}
    op, Sp, _, _, _ = o.layer(ip, wp, S0[:, :, p], t0[:, order])
    _close(op, out[:, :, p], what="value permutation y")
    _close(Sp, S[:, :, p], what="value permutation state")


def pin_layer_key_permutation(o):
    """Permuting the key channels (q, k, alpha and their conv rows) permutes
    the state rows and leaves y unchanged."""
    rng = _rng(20)
    H, dk, dv, L = 1, 5, 3, 4
    inp, w, S0, t0 = _layer_inputs(rng, L, H, dk, dv)
    out, S, _, _, _ = o.layer(inp, w, S0, t0)
    p = rng.permutation(dk)
    ip = dict(inp)
    for name in ("q", "k", "alpha"):
        ip[name] = inp[name][:, :, p]
    order = np.r_[p, dk + p, 2 * dk + np.arange(dv)]
    wp = {"conv_w": w["conv_w"][order], "norm_w": w["norm_w"]}
    op, Sp, _, _, _ = o.layer(ip, wp, S0[:, p, :], t0[:, order])
    _close(op, out, what="key permutation y")
    _close(Sp, S[:, p, :], what="key permutation state")


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
