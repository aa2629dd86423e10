"""Pins for the CPU oracle: checks against facts fixed by the mathematics.

Nothing here compares the oracle with itself. Each test pins it to something
independent of its own code: hand-derived values, central finite differences,
closed forms of special cases, conservation laws of the softmax gradient, and
a textbook materialised attention built from PyTorch float64 library routines
(softmax, tril/triu masks, repeat_interleave, autograd).

Definitions followed: "mlx-bun 0.0.4: package/src/model/flash-attention.ts"
(forward shader; backward passes 1-3; manualSdpa) and "R/ag_flash_attn.R"
(ggmlR; causal mask builder).
"""
import math
import os
import re
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.txt")


# ----------------------------------------------------------------- helpers
def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def loss(q, k, v, do, scale, causal, window):
    o, _ = oracle.attn_fwd(q, k, v, scale, causal, window)
    return float(np.sum(o * do))


def _eval(expr: str) -> float:
    expr = expr.strip()
    if expr in ("inf", "+inf"):
        return math.inf
    if expr == "-inf":
        return -math.inf
    if not re.fullmatch(r"[0-9ln()./*+\- ]+", expr):
        raise ValueError(f"bad golden expression {expr!r}")
    return float(eval(expr, {"__builtins__": {}}, {"ln": math.log}))


def load_golden():
    cases, cur = [], None
    for raw in open(GOLDEN):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        key, _, val = line.partition(":")
        key = key.strip()
        if key == "case":
            cur = {"name": val.strip()}
        elif key == "end":
            cases.append(cur)
            cur = None
        elif key == "dims":
            cur["dims"] = [int(x) for x in val.split()]
        elif key == "params":
            p = dict(kv.split("=") for kv in val.split())
            cur["scale"] = float(Fraction(p["scale"]))
            cur["causal"] = bool(int(p["causal"]))
            cur["window"] = int(p["window"])
        else:
            cur[key] = np.array([_eval(x) for x in val.split(",")])
    return cases


GOLDEN_CASES = load_golden()


# ------------------------------------------------------------ golden cases
@pytest.mark.parametrize("case", GOLDEN_CASES, ids=[c["name"] for c in GOLDEN_CASES])
def test_hand_derived_cases(case):
    B, Hq, Hkv, Tq, Tkv, D = case["dims"]
    q = case["q"].reshape(B, Hq, Tq, D)
    k = case["k"].reshape(B, Hkv, Tkv, D)
    v = case["v"].reshape(B, Hkv, Tkv, D)
    do = case["do"].reshape(B, Hq, Tq, D)
    sc, ca, w = case["scale"], case["causal"], case["window"]
    o, lse = oracle.attn_fwd(q, k, v, sc, ca, w)
    np.testing.assert_allclose(o.ravel(), case["o"], rtol=0, atol=1e-12)
    finite = np.isfinite(case["lse"])
    assert np.array_equal(np.isfinite(lse.ravel()), finite)
    np.testing.assert_allclose(lse.ravel()[finite], case["lse"][finite], rtol=0, atol=1e-12)
    assert np.all(lse.ravel()[~finite] == -np.inf)
    g = oracle.attn_bwd(q, k, v, do, sc, ca, w)
    np.testing.assert_allclose(g["dq"].ravel(), case["dq"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["dk"].ravel(), case["dk"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["dv"].ravel(), case["dv"], rtol=0, atol=1e-12)


# ------------------------------------------------------ finite differences
FD_CASES = [
    # (Hq, Hkv, Tq, Tkv, D, causal, window)
    (2, 1, 5, 5, 3, False, 0),
    (2, 1, 5, 5, 3, True, 0),
    (2, 1, 6, 6, 4, True, 2),
    (2, 1, 5, 5, 2, False, 2),
    (2, 2, 4, 6, 3, True, 0),      # Tq != Tkv, top-left causal
    (2, 1, 6, 3, 2, True, 2),      # fully masked rows present
]


@pytest.mark.parametrize("Hq,Hkv,Tq,Tkv,D,causal,window", FD_CASES)
def test_gradients_match_central_differences(Hq, Hkv, Tq, Tkv, D, causal, window):
    """Pin dQ/dK/dV to central differences of L = sum(O * dO) in double."""
    seed = hash((Hq, Hkv, Tq, Tkv, D, causal, window)) % 1000
    q = rand((1, Hq, Tq, D), seed)
    k = rand((1, Hkv, Tkv, D), seed + 1)
    v = rand((1, Hkv, Tkv, D), seed + 2)
    do = rand((1, Hq, Tq, D), seed + 3)
    scale = 0.7
    g = oracle.attn_bwd(q, k, v, do, scale, causal, window)
    h = 1e-5
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            lp = loss(q, k, v, do, scale, causal, window)
            x[idx] = old - h
            lm = loss(q, k, v, do, scale, causal, window)
            x[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        err = np.abs(fd - g[name]).max() / max(1.0, np.abs(fd).max())
        assert err < 1e-7, (name, err)


# --------------------------------------------- textbook library cross-check
def torch_reference(q, k, v, do, scale, causal, window):
    """Materialised attention from PyTorch float64 library routines + autograd."""
    q = torch.tensor(q, requires_grad=True)
    k = torch.tensor(k, requires_grad=True)
    v = torch.tensor(v, requires_grad=True)
    Hq, Hkv = q.shape[1], k.shape[1]
    Tq, Tkv = q.shape[2], k.shape[2]
    ke = k.repeat_interleave(Hq // Hkv, dim=1)
    ve = v.repeat_interleave(Hq // Hkv, dim=1)
    ones = torch.ones(Tq, Tkv, dtype=torch.bool)
    keep = ones.clone()
    if causal:
        keep &= ones.tril(0)
    if window:
        past = ones.tril(0)                      # key at or before the query
        near = ones.triu(-(window - 1))          # key within window-1 of the query
        keep &= ~past | near
    s = (q @ ke.transpose(-1, -2)) * scale
    s = s.masked_fill(~keep, -math.inf)
    lse = torch.logsumexp(s, dim=-1)
    full = torch.isfinite(lse)
    p = torch.softmax(s, dim=-1)
    p = torch.where(full[..., None], p, torch.zeros_like(p))
    o = p @ ve
    (o * torch.tensor(do)).sum().backward()
    return o.detach().numpy(), lse.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


LIB_CASES = [
    (1, 4, 1, 17, 17, 8, True, 0),
    (2, 4, 2, 13, 21, 5, False, 0),
    (1, 8, 2, 19, 19, 6, True, 5),
    (1, 2, 2, 12, 12, 4, False, 3),
    (1, 2, 1, 9, 4, 3, True, 3),         # fully masked rows
    (2, 6, 3, 1, 7, 4, False, 0),        # single query row
]


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Tkv,D,causal,window", LIB_CASES)
def test_matches_textbook_library_attention(B, Hq, Hkv, Tq, Tkv, D, causal, window):
    rng = np.random.default_rng(B * 1000 + Tq * 10 + Tkv)
    q = rng.standard_normal((B, Hq, Tq, D))
    k = rng.standard_normal((B, Hkv, Tkv, D))
    v = rng.standard_normal((B, Hkv, Tkv, D))
    do = rng.standard_normal((B, Hq, Tq, D))
    scale = 1 / math.sqrt(D)
    o_t, lse_t, dq_t, dk_t, dv_t = torch_reference(q, k, v, do, scale, causal, window)
    o, lse = oracle.attn_fwd(q, k, v, scale, causal, window)
    g = oracle.attn_bwd(q, k, v, do, scale, causal, window)
    np.testing.assert_allclose(o, o_t, atol=1e-12)
    assert np.array_equal(lse == -np.inf, lse_t == -np.inf)
    fin = np.isfinite(lse_t)
    np.testing.assert_allclose(lse[fin], lse_t[fin], atol=1e-12)
    np.testing.assert_allclose(g["dq"], np.nan_to_num(dq_t), atol=1e-11)
    np.testing.assert_allclose(g["dk"], dk_t, atol=1e-11)
    np.testing.assert_allclose(g["dv"], dv_t, atol=1e-11)


# ------------------------------------------------ closed forms and invariants
def test_causal_row0_is_first_value_row():
    """Causal row 0 sees only key 0: O[0] = V[g, 0], LSE[0] = scale * q0.k0."""
    q, k, v = rand((2, 4, 9, 5), 1), rand((2, 2, 9, 5), 2), rand((2, 2, 9, 5), 3)
    o, lse = oracle.attn_fwd(q, k, v, 0.3, True, 0)
    for b in range(2):
        for h in range(4):
            g = h // 2
            np.testing.assert_allclose(o[b, h, 0], v[b, g, 0], atol=1e-14)
            np.testing.assert_allclose(lse[b, h, 0], 0.3 * q[b, h, 0] @ k[b, g, 0], atol=1e-14)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 4), (False, 3)])
def test_uniform_scores_closed_form(causal, window):
    """Q = 0: every allowed score is 0, so O_i = mean of the allowed V rows,
    LSE_i = ln(#allowed), and dQ_i = (s/n_i) sum_j (dO_i.(V_j - Vbar_i)) K_j."""
    T, D, s = 11, 3, 0.5
    q = np.zeros((1, 2, T, D))
    k, v, do = rand((1, 1, T, D), 4), rand((1, 1, T, D), 5), rand((1, 2, T, D), 6)
    o, lse = oracle.attn_fwd(q, k, v, s, causal, window)
    g = oracle.attn_bwd(q, k, v, do, s, causal, window)
    for h in range(2):
        for i in range(T):
            # the allowed keys, enumerated straight from the mask's wording
            keys = [j for j in range(T)
                    if not (causal and j > i) and not (window and i >= j and i - j >= window)]
            n = len(keys)
            vbar = v[0, 0, keys].mean(axis=0)
            np.testing.assert_allclose(o[0, h, i], vbar, atol=1e-14)
            np.testing.assert_allclose(lse[0, h, i], math.log(n), atol=1e-14)
            dq = sum((do[0, h, i] @ (v[0, 0, j] - vbar)) * k[0, 0, j] for j in keys) * s / n
            np.testing.assert_allclose(g["dq"][0, h, i], dq, atol=1e-13)
    if causal and window:
        # a causal window W lets row i see exactly min(i + 1, W) keys
        np.testing.assert_allclose(lse[0, 0], np.log(np.minimum(np.arange(T) + 1, window)),
                                   atol=1e-14)


@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 5)])
def test_softmax_gradient_conservation(causal, window):
    """Each row of dS sums to 0, so sum_j dK[b,g,j,:] = 0; each allowed row of P
    sums to 1, so sum_j dV[b,g,j,:] = sum over the group's rows of dO."""
    q, k, v = rand((2, 6, 13, 4), 7), rand((2, 2, 13, 4), 8), rand((2, 2, 13, 4), 9)
    do = rand((2, 6, 13, 4), 10)
    g = oracle.attn_bwd(q, k, v, do, 0.6, causal, window)
    np.testing.assert_allclose(g["dk"].sum(axis=2), 0.0, atol=1e-12)
    want = do.reshape(2, 2, 3, 13, 4).sum(axis=(2, 3))
    np.testing.assert_allclose(g["dv"].sum(axis=2), want, atol=1e-12)


def test_dvector_equals_rowsum_p_dp():
    """D_i = sum_d dO_i O_i equals sum_j P_ij (dO_i . V_j), with P rebuilt from
    the oracle's LSE and scores computed here."""
    q, k, v, do = rand((1, 2, 10, 4), 11), rand((1, 1, 10, 4), 12), rand((1, 1, 10, 4), 13), rand((1, 2, 10, 4), 14)
    s = 0.8
    g = oracle.attn_bwd(q, k, v, do, s, True, 0)
    for h in range(2):
        S = s * q[0, h] @ k[0, 0].T
        P = np.where(np.tril(np.ones((10, 10))) > 0, np.exp(S - g["lse"][0, h][:, None]), 0.0)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-13)
        dP = do[0, h] @ v[0, 0].T
        np.testing.assert_allclose(g["dvec"][0, h], (P * dP).sum(axis=1), atol=1e-12)
        np.testing.assert_allclose(g["dvec"][0, h], (do[0, h] * g["o"][0, h]).sum(axis=1), atol=1e-13)


def test_constant_values_give_zero_q_k_gradients():
    """All V rows equal: O = v for every row, and dP_ij = D_i so dQ = dK = 0."""
    q, k, do = rand((1, 4, 8, 3), 15), rand((1, 2, 8, 3), 16), rand((1, 4, 8, 3), 17)
    v = np.broadcast_to(np.array([0.3, -1.2, 2.0]), (1, 2, 8, 3)).copy()
    o, _ = oracle.attn_fwd(q, k, v, 0.5, True, 0)
    np.testing.assert_allclose(o, np.broadcast_to(v[0, 0, 0], o.shape), atol=1e-14)
    g = oracle.attn_bwd(q, k, v, do, 0.5, True, 0)
    np.testing.assert_allclose(g["dq"], 0.0, atol=1e-13)
    np.testing.assert_allclose(g["dk"], 0.0, atol=1e-13)


def test_single_key():
    """Tkv = 1: O = V, LSE = S, dV = sum of the group's dO, dQ = dK = 0."""
    q, k, v, do = rand((2, 4, 5, 3), 18), rand((2, 2, 1, 3), 19), rand((2, 2, 1, 3), 20), rand((2, 4, 5, 3), 21)
    o, lse = oracle.attn_fwd(q, k, v, 0.9, False, 0)
    g = oracle.attn_bwd(q, k, v, do, 0.9, False, 0)
    for b in range(2):
        for h in range(4):
            np.testing.assert_allclose(o[b, h], np.broadcast_to(v[b, h // 2, 0], (5, 3)), atol=1e-14)
            np.testing.assert_allclose(lse[b, h], 0.9 * q[b, h] @ k[b, h // 2, 0], atol=1e-14)
    np.testing.assert_allclose(g["dv"][:, :, 0], do.reshape(2, 2, 2, 5, 3).sum(axis=(2, 3)), atol=1e-13)
    np.testing.assert_allclose(g["dq"], 0.0, atol=1e-14)
    np.testing.assert_allclose(g["dk"], 0.0, atol=1e-14)


def test_no_nan_and_fully_masked_rows():
    """Causal window with Tq > Tkv leaves rows with no allowed key: their O is
    0, LSE is -inf, dQ is 0; every other LSE is finite; nothing is NaN."""
    q, k, v, do = rand((1, 2, 12, 4), 22), rand((1, 1, 5, 4), 23), rand((1, 1, 5, 4), 24), rand((1, 2, 12, 4), 25)
    W = 3
    o, lse = oracle.attn_fwd(q, k, v, 0.5, True, W)
    g = oracle.attn_bwd(q, k, v, do, 0.5, True, W)
    dead = np.arange(12) - (5 - 1) >= W
    for arr in (o, g["dq"], g["dk"], g["dv"]):
        assert not np.isnan(arr).any()
    assert np.all(lse[..., dead] == -np.inf) and np.all(np.isfinite(lse[..., ~dead]))
    assert np.all(o[:, :, dead] == 0) and np.all(g["dq"][:, :, dead] == 0)


def test_row_range_restriction_is_exact_where_promised():
    """Rows [lo, hi) reproduce the full result on those rows; dK/dV are exact
    for key rows whose allowed query rows all lie in the range."""
    q, k, v, do = rand((1, 4, 24, 4), 26), rand((1, 2, 24, 4), 27), rand((1, 2, 24, 4), 28), rand((1, 4, 24, 4), 29)
    full = oracle.attn_bwd(q, k, v, do, 0.4, True, 6)
    lo = 16
    part = oracle.attn_bwd(q, k, v, do, 0.4, True, 6, row_lo=lo, row_hi=24)
    np.testing.assert_allclose(part["dq"][:, :, lo:], full["dq"][:, :, lo:], atol=1e-14)
    np.testing.assert_allclose(part["o"][:, :, lo:], full["o"][:, :, lo:], atol=1e-14)
    # causal: key j is seen by rows i >= j only, so keys >= lo are complete
    np.testing.assert_allclose(part["dk"][:, :, lo:], full["dk"][:, :, lo:], atol=1e-13)
    np.testing.assert_allclose(part["dv"][:, :, lo:], full["dv"][:, :, lo:], atol=1e-13)
    o, lse = oracle.attn_fwd(q, k, v, 0.4, True, 6, row_lo=3, row_hi=9)
    np.testing.assert_allclose(o[:, :, 3:9], full["o"][:, :, 3:9], atol=1e-14)
    assert np.isnan(o[:, :, :3]).all() and np.isnan(lse[:, :, 9:]).all()
