"""Pins for the float64 JSD / KL distillation oracle (CPU only): identical distributions,
closed forms, finite differences, torch float64 kl_div and autograd, symmetry at
beta = 0.5, the log 2 bound, and planted mistakes the pins must catch."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import jsd_oracle as jo


def _problem(BT=7, Hs=5, Ht=4, V=9, seed=0, n_ignored=2, scale=0.8):
    rng = np.random.default_rng(seed)
    Xs = rng.standard_normal((BT, Hs))
    Ws = rng.standard_normal((V, Hs)) * scale
    Xt = rng.standard_normal((BT, Ht))
    Wt = rng.standard_normal((V, Ht)) * scale
    lab = rng.integers(0, V, BT)
    lab[rng.permutation(BT)[:n_ignored]] = -100
    g = rng.uniform(0.5, 1.5, BT)
    return Xs, Ws, Xt, Wt, lab, g


@pytest.mark.parametrize("beta", [0.0, 0.3, 0.5, 1.0])
def test_identical_distributions_give_zero(beta):
    """Teacher = student (same rows, same head): every divergence is 0 and so is every
    gradient."""
    Xs, Ws, _, _, lab, _ = _problem(seed=1)
    r = jo.jsd_oracle(Xs, Ws, Xs, Ws, lab, beta=beta, temperature=1.7, reduction="sum")
    assert abs(r["loss"]) < 1e-14
    assert np.max(np.abs(r["dX"])) < 1e-14 and np.max(np.abs(r["dW"])) < 1e-14


def test_two_point_closed_form():
    """V = 2 with logits (0, a) against (0, b): KL between two Bernoulli distributions,
    written out by hand."""
    Xs = np.array([[1.0]])
    Ws = np.array([[0.0], [0.7]])
    Xt = np.array([[1.0]])
    Wt = np.array([[0.0], [-0.4]])
    q1 = 1 / (1 + math.exp(-0.7))
    p1 = 1 / (1 + math.exp(0.4))
    kl_pq = p1 * math.log(p1 / q1) + (1 - p1) * math.log((1 - p1) / (1 - q1))
    kl_qp = q1 * math.log(q1 / p1) + (1 - q1) * math.log((1 - q1) / (1 - p1))
    assert abs(jo.jsd_oracle(Xs, Ws, Xt, Wt, None, beta=0.0, reduction="sum")["loss"] - kl_pq) < 1e-15
    assert abs(jo.jsd_oracle(Xs, Ws, Xt, Wt, None, beta=1.0, reduction="sum")["loss"] - kl_qp) < 1e-15
    m1 = 0.5 * (p1 + q1)
    js = 0.5 * (p1 * math.log(p1 / m1) + (1 - p1) * math.log((1 - p1) / (1 - m1))) + \
        0.5 * (q1 * math.log(q1 / m1) + (1 - q1) * math.log((1 - q1) / (1 - m1)))
    assert abs(jo.jsd_oracle(Xs, Ws, Xt, Wt, None, beta=0.5, reduction="sum")["loss"] - js) < 1e-15


def test_symmetry_and_bound_at_half():
    """JSD_0.5 is symmetric in teacher and student and at most log 2."""
    Xs, Ws, Xt, Wt, lab, _ = _problem(seed=2, scale=3.0)
    a = jo.jsd_oracle(Xs, Ws, Xt, Wt, lab, beta=0.5, reduction="none")["loss"]
    b = jo.jsd_oracle(Xt, Wt, Xs, Ws, lab, beta=0.5, reduction="none")["loss"]
    assert np.allclose(a, b, atol=1e-14)
    assert np.all(a <= math.log(2) + 1e-15) and np.all(a >= 0)


def _objective(Xs, Ws, Xt, Wt, lab, beta, T, reduction, g):
    r = jo.jsd_oracle(Xs, Ws, Xt, Wt, lab, beta=beta, temperature=T, reduction=reduction,
                      grad_out=g, want_dX=False, want_dW=False)
    return float(np.sum(g * r["loss"])) if reduction == "none" else float(g[0] * r["loss"])


def _fd_error(beta, T, reduction, seed=3):
    Xs, Ws, Xt, Wt, lab, g = _problem(seed=seed)
    gg = g if reduction == "none" else np.array([1.3])
    r = jo.jsd_oracle(Xs, Ws, Xt, Wt, lab, beta=beta, temperature=T, reduction=reduction, grad_out=gg)
    h = 1e-6
    errs = []
    for arr, grad in ((Xs, r["dX"]), (Ws, r["dW"])):
        num = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            o = arr[i]
            arr[i] = o + h
            fp = _objective(Xs, Ws, Xt, Wt, lab, beta, T, reduction, gg)
            arr[i] = o - h
            fm = _objective(Xs, Ws, Xt, Wt, lab, beta, T, reduction, gg)
            arr[i] = o
            num[i] = (fp - fm) / (2 * h)
        errs.append(np.max(np.abs(num - grad)) / max(1e-3, np.max(np.abs(num))))
    return max(errs)


@pytest.mark.parametrize("beta", [0.0, 0.25, 0.5, 1.0])
@pytest.mark.parametrize("T,reduction", [(1.0, "mean"), (2.0, "none"), (0.7, "sum")])
def test_finite_differences(beta, T, reduction):
    assert _fd_error(beta, T, reduction) < 1e-7


@pytest.mark.parametrize("beta", [0.0, 0.4, 1.0])
def test_matches_torch_float64(beta):
    Xs, Ws, Xt, Wt, lab, _ = _problem(BT=30, Hs=12, Ht=10, V=40, seed=4, n_ignored=6, scale=1.0)
    T = 1.5
    xs = torch.tensor(Xs, requires_grad=True)
    ws = torch.tensor(Ws, requires_grad=True)
    lq = F.log_softmax(xs @ ws.T / T, dim=-1)
    lp = F.log_softmax(torch.tensor(Xt) @ torch.tensor(Wt).T / T, dim=-1)
    keep = torch.tensor(lab != -100)
    if beta == 0.0:
        per = F.kl_div(lq, lp, reduction="none", log_target=True).sum(-1)        # KL(P || Q)
    elif beta == 1.0:
        per = F.kl_div(lp, lq, reduction="none", log_target=True).sum(-1)        # KL(Q || P)
    else:
        lm = torch.log(beta * lp.exp() + (1 - beta) * lq.exp())
        per = beta * F.kl_div(lm, lp, reduction="none", log_target=True).sum(-1) + \
            (1 - beta) * F.kl_div(lm, lq, reduction="none", log_target=True).sum(-1)
    loss = per[keep].sum() / keep.sum()
    loss.backward()
    r = jo.jsd_oracle(Xs, Ws, Xt, Wt, lab, beta=beta, temperature=T, reduction="mean")
    assert abs(r["loss"] - float(loss.detach())) < 1e-12
    assert np.allclose(r["dX"], xs.grad.numpy(), atol=1e-12)
    assert np.allclose(r["dW"], ws.grad.numpy(), atol=1e-12)


def test_ignored_rows_and_nan_isolation():
    Xs, Ws, Xt, Wt, lab, g = _problem(BT=12, seed=5, n_ignored=4)
    ign = lab == -100
    Xs2, Xt2 = Xs.copy(), Xt.copy()
    Xs2[ign] = np.nan
    Xt2[ign] = np.nan
    a = jo.jsd_oracle(Xs, Ws, Xt, Wt, lab, beta=0.5, reduction="none")
    b = jo.jsd_oracle(Xs2, Ws, Xt2, Wt, lab, beta=0.5, reduction="none")
    assert np.array_equal(a["loss"], b["loss"]) and np.array_equal(a["dW"], b["dW"])
    assert np.all(b["loss"][ign] == 0) and np.all(b["dX"][ign] == 0)


def test_planted_mistakes_are_caught(monkeypatch):
    """Drop the mean-subtraction of the softmax Jacobian, or the 1/T chain factor: the
    finite-difference pin must fail."""
    assert _fd_error(0.5, 2.0, "mean") < 1e-7
    orig = jo.jsd_rows

    def no_center(zs, zt, beta):
        loss, dz = orig(zs, zt, beta)
        logQ = jo._log_softmax(zs)
        M = beta * np.exp(jo._log_softmax(zt)) + (1 - beta) * np.exp(logQ)
        return loss, np.exp(logQ) * (1 - beta) * (logQ - np.log(M))

    monkeypatch.setattr(jo, "jsd_rows", no_center)
    assert _fd_error(0.5, 2.0, "mean") > 1e-3
    monkeypatch.setattr(jo, "jsd_rows", orig)

    def times_T(zs, zt, beta):
        loss, dz = orig(zs, zt, beta)
        return loss, dz * 2.0

    monkeypatch.setattr(jo, "jsd_rows", times_T)
    assert _fd_error(0.5, 2.0, "sum") > 1e-3
