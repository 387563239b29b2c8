"""Pins for the float64 oracle: closed forms, finite differences, a brute-force torch
float64 evaluation, invariants, and planted mistakes that each pin must catch.

CPU only. None of these tests touches the CUDA library.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import logsumexp, softmax

from oracle import flce_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(BT=9, H=5, V=7, seed=0, n_ignored=2, bias=True, scale=0.7):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((BT, H))
    W = rng.standard_normal((V, H)) * scale
    b = rng.standard_normal(V) * 0.3 if bias else None
    t = rng.integers(0, V, BT)
    ign = rng.permutation(BT)[:n_ignored]
    t[ign] = -100
    g = rng.uniform(0.5, 1.5, BT)
    return X, W, b, t, g


# --------------------------------------------------------------------------- closed forms

@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_uniform_logits_give_log_V(reduction):
    """W = 0 and no bias: every logit is 0, so loss = lse = ln V, pred = 0, dX = 0, and
    dW[v] = sum_i c_i (1/V - [v = t_i]) X_i."""
    BT, H, V = 11, 4, 13
    rng = np.random.default_rng(1)
    X = rng.standard_normal((BT, H))
    W = np.zeros((V, H))
    t = rng.integers(0, V, BT)
    t[[2, 7]] = -100
    g = rng.uniform(0.5, 1.5, BT) if reduction == "none" else np.array([0.8])
    r = orc.flce_oracle(X, W, t, reduction=reduction, grad_out=g)
    lab = t != -100
    n = lab.sum()
    assert np.allclose(r["lse_tok"][lab], math.log(V), rtol=0, atol=1e-14)
    assert np.allclose(r["loss_tok"][lab], math.log(V), rtol=0, atol=1e-14)
    assert np.all(r["pred_tok"][lab] == 0)
    assert np.all(r["dX"] == 0)
    c = {"mean": 0.8 / n, "sum": 0.8, "none": None}[reduction]
    cw = np.where(lab, g if reduction == "none" else c, 0.0)
    expect = np.zeros((V, H))
    for i in range(BT):
        if lab[i]:
            expect += cw[i] * np.outer(np.full(V, 1.0 / V) - np.eye(V)[t[i]], X[i])
    assert np.allclose(r["dW"], expect, rtol=0, atol=1e-13)
    if reduction == "mean":
        assert abs(r["loss"] - math.log(V)) < 1e-14


def test_zero_input_closed_form():
    """X = 0, W random, no bias: s = 0, loss = ln V, dX_i = c_i (mean_v W_v - W_{t_i}),
    and dW = 0."""
    BT, H, V = 6, 3, 9
    rng = np.random.default_rng(2)
    W = rng.standard_normal((V, H))
    X = np.zeros((BT, H))
    t = rng.integers(0, V, BT)
    r = orc.flce_oracle(X, W, t, reduction="sum")
    assert np.allclose(r["loss_tok"], math.log(V), atol=1e-14)
    expect = W.mean(axis=0)[None, :] - W[t]
    assert np.allclose(r["dX"], expect, atol=1e-14)
    assert np.all(r["dW"] == 0)


def test_bias_only_logits_match_logsumexp():
    """W = 0 with a bias: loss_i = logsumexp(b) - b_{t_i} (scipy), dbias = sum_i c_i
    (softmax(b) - onehot(t_i))."""
    BT, H, V = 5, 2, 17
    rng = np.random.default_rng(3)
    b = rng.standard_normal(V) * 2
    X = rng.standard_normal((BT, H))
    W = np.zeros((V, H))
    t = rng.integers(0, V, BT)
    r = orc.flce_oracle(X, W, t, bias=b, reduction="sum")
    assert np.allclose(r["loss_tok"], logsumexp(b) - b[t], atol=1e-13)
    assert np.allclose(r["lse_tok"], logsumexp(b), atol=1e-13)
    sm = softmax(b)
    expect = sum(sm - np.eye(V)[ti] for ti in t)
    assert np.allclose(r["dbias"], expect, atol=1e-13)
    assert np.all(r["pred_tok"] == np.argmax(b))


def test_two_class_softplus():
    """V = 2: cross entropy is softplus(s_other - s_target) = log(1 + exp(d))."""
    X = np.array([[1.5, -0.5], [0.25, 2.0], [-1.0, -1.0]])
    W = np.array([[0.3, -0.7], [1.1, 0.4]])
    t = np.array([0, 1, 1])
    r = orc.flce_oracle(X, W, t, reduction="none")
    s = X @ W.T
    d = s[np.arange(3), 1 - t] - s[np.arange(3), t]
    assert np.allclose(r["loss_tok"], np.log1p(np.exp(d)), atol=1e-15)


def test_hand_computed_three_logits():
    """H = 1, x = 1, W = [1, 2, 3]^T, target 2: loss = log(1 + e^-1 + e^-2), written out
    by hand; dX = sum_v p_v v - 3 with p = (1, e, e^2) / (1 + e + e^2)."""
    X = np.array([[1.0]])
    W = np.array([[1.0], [2.0], [3.0]])
    r = orc.flce_oracle(X, W, np.array([2]), reduction="mean")
    e = math.e
    assert abs(r["loss"] - math.log(1 + 1 / e + 1 / e ** 2)) < 1e-15
    den = 1 + e + e * e
    assert abs(r["dX"][0, 0] - ((1 + 2 * e + 3 * e * e) / den - 3.0)) < 1e-15
    assert r["pred_tok"][0] == 2 and r["acc_tok"][0] == 1.0


def test_dominant_logit_drives_loss_to_zero():
    X = np.array([[1.0, 0.0]])
    W = np.array([[0.0, 0.0], [20.0, 0.0], [0.0, 0.0]])
    r = orc.flce_oracle(X, W, np.array([1]), reduction="sum")
    # loss = log(1 + 2 e^-20); lse - s_t is exact to one ulp of 20 (3.6e-15)
    assert 0.0 < r["loss"] < 1e-8
    assert abs(r["loss"] - math.log1p(2 * math.exp(-20))) < 1e-14


def test_argmax_tie_takes_lowest_index():
    """Exact ties (duplicated W rows) resolve to the lowest vocabulary index."""
    rng = np.random.default_rng(4)
    W = rng.standard_normal((8, 3))
    W[5] = W[2]
    X = W[2:3] * 10.0  # row 2 (and its copy 5) dominates
    r = orc.flce_oracle(X, W, np.array([5]), reduction="none")
    assert r["pred_tok"][0] == 2
    assert r["acc_tok"][0] == 0.0


# --------------------------------------------------------------- finite differences

def _objective(X, W, b, t, reduction, z, g):
    r = orc.flce_oracle(X, W, t, bias=b, reduction=reduction, z_loss_scale=z,
                        grad_out=g, want_dX=False, want_dW=False)
    if reduction == "none":
        return float(np.sum(g * r["loss"]))
    return float(g[0] * r["loss"])


def _fd_errors(reduction, z, seed=5):
    X, W, b, t, g = _problem(seed=seed)
    gg = g if reduction == "none" else np.array([1.3])
    r = orc.flce_oracle(X, W, t, bias=b, reduction=reduction, z_loss_scale=z, grad_out=gg)
    h = 1e-6
    errs = []
    for name, arr, grad in (("X", X, r["dX"]), ("W", W, r["dW"]), ("b", b, r["dbias"])):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            fp = _objective(X, W, b, t, reduction, z, gg)
            arr[idx] = old - h
            fm = _objective(X, W, b, t, reduction, z, gg)
            arr[idx] = old
            num[idx] = (fp - fm) / (2 * h)
        errs.append(np.max(np.abs(num - grad)) / max(1e-3, np.max(np.abs(num))))
    return max(errs)


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("z", [0.0, 0.3])
def test_finite_differences(reduction, z):
    assert _fd_errors(reduction, z) < 1e-7


# ---------------------------------------------------- brute force through torch float64

def _torch_reference(X, W, b, t, reduction, z, g):
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True) if b is not None else None
    tt = torch.tensor(t, dtype=torch.int64)
    logits = F.linear(Xt, Wt, bt)
    ce = F.cross_entropy(logits, tt, ignore_index=-100, reduction="none")
    lab = tt != -100
    lse = torch.logsumexp(logits, dim=-1)
    per = ce + torch.where(lab, z * lse * lse, torch.zeros_like(lse))
    if reduction == "mean":
        loss = per.sum() / lab.sum()
        (loss * float(g[0])).backward()
    elif reduction == "sum":
        loss = per.sum()
        (loss * float(g[0])).backward()
    else:
        loss = per
        (per * torch.tensor(g)).sum().backward()
    return (loss.detach().numpy(), Xt.grad.numpy(), Wt.grad.numpy(),
            None if bt is None else bt.grad.numpy(), logits.argmax(-1).numpy())


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("z,bias", [(0.0, False), (1e-4, True), (0.2, True)])
def test_matches_torch_float64(reduction, z, bias):
    X, W, b, t, g = _problem(BT=40, H=16, V=50, seed=6, n_ignored=9, bias=bias, scale=1.0)
    gg = g if reduction == "none" else np.array([0.9])
    r = orc.flce_oracle(X, W, t, bias=b, reduction=reduction, z_loss_scale=z, grad_out=gg)
    loss, dX, dW, db, am = _torch_reference(X, W, b, t, reduction, z, gg)
    lab = t != -100
    if reduction == "none":
        assert np.allclose(r["loss"], loss, atol=1e-12)
    else:
        assert abs(r["loss"] - float(loss)) < 1e-12
    assert np.allclose(r["dX"], dX, atol=1e-12)
    assert np.allclose(r["dW"], dW, atol=1e-12)
    if bias:
        assert np.allclose(r["dbias"], db, atol=1e-12)
    assert np.all(r["pred_tok"][lab] == am[lab])


# ------------------------------------------------------------------------ invariants

def test_gradient_rows_sum_to_zero_without_z():
    """With z = 0, sum_v dS_iv = 0 for every row, so sum_v dW[v,:] = 0 and sum dbias = 0."""
    X, W, b, t, g = _problem(BT=30, H=6, V=40, seed=7, n_ignored=5)
    r = orc.flce_oracle(X, W, t, bias=b, reduction="mean")
    assert np.allclose(r["dW"].sum(axis=0), 0.0, atol=1e-14)
    assert abs(r["dbias"].sum()) < 1e-14


def test_shift_invariance():
    """Adding a constant to every logit of a row (through the bias) changes neither the
    cross entropy nor dX (z = 0)."""
    X, W, b, t, g = _problem(BT=12, H=4, V=10, seed=8)
    r0 = orc.flce_oracle(X, W, t, bias=b, reduction="none")
    r1 = orc.flce_oracle(X, W, t, bias=b + 3.25, reduction="none")
    assert np.allclose(r0["loss"], r1["loss"], atol=1e-12)
    assert np.allclose(r0["dX"], r1["dX"], atol=1e-12)
    assert np.all(r0["pred_tok"] == r1["pred_tok"])


def test_mean_is_sum_over_labelled_count():
    X, W, b, t, g = _problem(BT=20, H=5, V=12, seed=9, n_ignored=6)
    rm = orc.flce_oracle(X, W, t, bias=b, reduction="mean", z_loss_scale=0.01)
    rs = orc.flce_oracle(X, W, t, bias=b, reduction="sum", z_loss_scale=0.01)
    rn = orc.flce_oracle(X, W, t, bias=b, reduction="none", z_loss_scale=0.01)
    n = (t != -100).sum()
    assert abs(rm["loss"] - rs["loss"] / n) < 1e-13
    assert abs(rs["loss"] - rn["loss"].sum()) < 1e-12
    assert np.allclose(rm["dX"] * n, rs["dX"], atol=1e-12)
    assert np.allclose(rm["dW"] * n, rs["dW"], atol=1e-12)


def test_ignored_rows_match_golden_and_nan_does_not_leak():
    """Ignored rows give the outputs the pages list, and a NaN in an ignored row of X
    reaches no output (Liger-Kernel PR #1554, Details item 1 and Tests)."""
    with open(os.path.join(GOLDEN, "ignored_row_outputs.json")) as f:
        gold = json.load(f)
    X, W, b, t, g = _problem(BT=15, H=4, V=9, seed=10, n_ignored=5)
    ign = t == -100
    Xn = X.copy()
    Xn[ign] = np.nan
    r0 = orc.flce_oracle(X, W, t, bias=b, reduction="none", z_loss_scale=0.1, grad_out=g)
    r1 = orc.flce_oracle(Xn, W, t, bias=b, reduction="none", z_loss_scale=0.1, grad_out=g)
    for k in ("loss", "z_loss_tok", "acc_tok", "lse_tok"):
        assert np.array_equal(r0[k], r1[k])
    assert np.array_equal(r0["dW"], r1["dW"]) and np.array_equal(r0["dbias"], r1["dbias"])
    assert np.all(np.isfinite(r1["dW"])) and np.all(np.isfinite(r1["dX"]))
    assert np.all(r1["loss_tok"][ign] == gold["loss_tok"])
    assert np.all(r1["z_loss_tok"][ign] == gold["z_loss_tok"])
    assert np.all(r1["acc_tok"][ign] == gold["acc_tok"])
    assert np.all(r1["pred_tok"][ign] == gold["pred_tok"])
    assert np.all(r1["dX"][ign] == gold["dX_row"])


def test_all_rows_ignored_mean_is_zero():
    X, W, b, t, g = _problem(BT=6, H=3, V=5, seed=11, n_ignored=0)
    t[:] = -100
    r = orc.flce_oracle(X, W, t, bias=b, reduction="mean")
    assert r["loss"] == 0.0 and r["n_labelled"] == 0
    assert np.all(r["dX"] == 0) and np.all(r["dW"] == 0) and np.all(r["dbias"] == 0)


def test_out_of_range_target_is_flagged_and_ignored():
    X, W, b, t, g = _problem(BT=6, H=3, V=5, seed=12, n_ignored=0)
    t2 = t.copy()
    t2[3] = 5  # == V
    r = orc.flce_oracle(X, W, t2, bias=b, reduction="sum")
    assert r["out_of_range"] and r["n_labelled"] == 5 and r["pred_tok"][3] == -1
    t3 = t.copy()
    t3[3] = -100
    r3 = orc.flce_oracle(X, W, t3, bias=b, reduction="sum")
    assert abs(r["loss"] - r3["loss"]) < 1e-14 and not r3["out_of_range"]


def test_sampled_rows_agree_with_full_oracle():
    X, W, b, t, g = _problem(BT=33, H=8, V=70, seed=13, n_ignored=7)
    full = orc.flce_oracle(X, W, t, bias=b, reduction="none", z_loss_scale=1e-3, grad_out=g)
    rows = np.array([0, 4, 5, 17, 32])
    part = orc.flce_oracle_rows(X, W, t, rows, bias=b, reduction="none",
                                z_loss_scale=1e-3, grad_out=g)
    for k in ("loss_tok", "lse_tok", "pred_tok", "acc_tok", "z_loss_tok"):
        assert np.allclose(part[k], full[k][rows], atol=1e-13)
    assert np.allclose(part["dX"], full["dX"][rows], atol=1e-13)


# ---------------------------------------------- planted mistakes: each pin must catch one

def test_planted_mistakes_are_caught(monkeypatch):
    """Plant a mistake in the oracle (dropped z-term, wrong one-hot sign, BT instead of N
    as the mean divisor) and check that the pins above would fail."""
    base = _fd_errors("mean", 0.3)
    assert base < 1e-7

    orig = orc.rows_grad_logits

    def no_z(p, t, lse, c, z):
        return orig(p, t, lse, c, 0.0)

    monkeypatch.setattr(orc, "rows_grad_logits", no_z)
    assert _fd_errors("mean", 0.3) > 1e-3
    monkeypatch.setattr(orc, "rows_grad_logits", orig)

    def plus_onehot(p, t, lse, c, z):
        d = p * (1.0 + 2.0 * z * lse)[:, None]
        d[np.arange(p.shape[0]), t] += 1.0
        return d * c[:, None]

    monkeypatch.setattr(orc, "rows_grad_logits", plus_onehot)
    assert _fd_errors("sum", 0.0) > 1e-3
    monkeypatch.setattr(orc, "rows_grad_logits", orig)

    orig_scales = orc.grad_scales

    def bt_divisor(mask, reduction, grad_out):
        c = orig_scales(mask, reduction, grad_out)
        if reduction == "mean":
            c = c * mask.sum() / mask.shape[0]
        return c

    monkeypatch.setattr(orc, "grad_scales", bt_divisor)
    assert _fd_errors("mean", 0.0) > 1e-3


# --------------------------------------------------------------------------- argmax tie band

def _fp32_dot(x, w, order):
    """x . w in fp32: each product rounded to fp32, summed one term at a time in `order`."""
    acc = np.float32(0.0)
    for h in order:
        acc = np.float32(acc + np.float32(np.float32(x[h]) * np.float32(w[h])))
    return acc


def test_argmax_tie_band_bounds_fp32_logit_error():
    """The band accepts an argmax mismatch only where fp32 evaluation could produce one.
    (1) Logits of bf16-exact values evaluated in fp32 (sequential, reversed and numpy's own
    order, then an fp32 bias add) stay within one logit's share of the band (half of it) of
    the float64 value on 240 random row / vocabulary pairs. (2) The worst case the bound is
    written for, reached: x = w = (2^12, 1, ..., 1) summed left to right in fp32 keeps
    rounding 2^24 + 1 back to 2^24, an error of H - 1, which the band covers and a bound
    without its factor H (u times the absolute dot product) would not."""
    rng = np.random.default_rng(5)
    H = 512
    X = torch.from_numpy(rng.standard_normal((8, H))).to(torch.bfloat16).double().numpy()
    W = torch.from_numpy(rng.standard_normal((30, H)) * 0.05).to(torch.bfloat16).double().numpy()
    b = torch.from_numpy(rng.standard_normal(30) * 0.3).to(torch.bfloat16).double().numpy()
    bmax = float(np.max(np.abs(b)))
    for i in range(X.shape[0]):
        absdot = orc._absdot_max(np.abs(X[i:i + 1]), W)[0]
        half_band = orc.argmax_tie_band(absdot, bmax, H) / 2.0
        for v in range(W.shape[0]):
            exact = float(X[i] @ W[v]) + b[v]
            for order in (range(H), range(H - 1, -1, -1), None):
                d = (X[i].astype(np.float32) @ W[v].astype(np.float32) if order is None
                     else _fp32_dot(X[i], W[v], order))
                got = float(np.float32(d + np.float32(b[v])))
                assert abs(got - exact) <= half_band, (i, v, order)
    x = np.ones(H)
    x[0] = 4096.0
    exact = float(x @ x)
    err = abs(float(_fp32_dot(x, x, range(H))) - exact)
    assert err == H - 1
    absdot = float(np.abs(x) @ np.abs(x))
    assert err <= orc.argmax_tie_band(absdot, 0.0, H) / 2.0
    assert err > 2.0 ** -23 * absdot  # what a bound without the factor H would allow


def test_vocabulary_blocks_match_torch_float64():
    """The oracle converts and multiplies W in vocabulary blocks of 32768 rows
    (logits_rows, dX_rows, _absdot_max). At V = 70000 (three blocks, a ragged last one) the
    blocked evaluation must equal torch's float64 cross entropy + autograd over the whole
    vocabulary, and the blocked max |x|.|w| the unblocked one; the target and argmax of some
    rows are placed in the second and third blocks."""
    rng = np.random.default_rng(21)
    BT, H, V = 6, 8, 70000
    X = rng.standard_normal((BT, H))
    W = rng.standard_normal((V, H)) * 0.3
    b = rng.standard_normal(V) * 0.1
    t = np.array([5, 32767, 32768, 65535, 69999, -100])
    W[40000] = 3.0 * X[1] / np.linalg.norm(X[1])   # row 1's argmax in the second block
    W[69000] = 3.0 * X[2] / np.linalg.norm(X[2])   # row 2's argmax in the last block
    for red in ("mean", "none"):
        g = np.linspace(0.5, 1.5, BT) if red == "none" else np.array([1.3])
        r = orc.flce_oracle(X, W, t, bias=b, reduction=red, z_loss_scale=1e-3, grad_out=g)
        loss, dX, dW, db, am = _torch_reference(X, W, b, t, red, 1e-3, g)
        assert np.allclose(r["loss"], loss, rtol=1e-12, atol=1e-12)
        assert np.allclose(r["dX"], dX, rtol=1e-10, atol=1e-13)
        assert np.allclose(r["dW"], dW, rtol=1e-10, atol=1e-15)
        assert np.allclose(r["dbias"], db, rtol=1e-10, atol=1e-15)
        lab = t != -100
        assert np.array_equal(r["pred_tok"][lab], am[lab])
    assert r["pred_tok"][1] == 40000 and r["pred_tok"][2] == 69000
    xa = np.abs(X)
    assert np.allclose(orc._absdot_max(xa, W), (xa @ np.abs(W).T).max(axis=1), rtol=1e-14)
    assert np.allclose(orc._absdot_max(xa, W, v_block=1000), orc._absdot_max(xa, W), rtol=1e-14)
