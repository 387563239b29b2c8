"""Float64 CPU oracle for fused linear JSD / KL distillation, forward and backward.

TEST INFRASTRUCTURE, like flce_oracle: only the test suite, the smoke check and bench.py's
CPU legs may import it; the product never does, and it imports nothing from the product.

The pages name this sibling op without defining it: the commit page of Liger-Kernel v0.8.3
lists a "fused linear KL" loss with its own chunk policy, and "Liger-Kernel PR #1554: skip
ignore_index rows" (Results) lists test_fused_linear_jsd.py::test_correctness_with_ignore_index.
The reading taken here is the generalised Jensen-Shannon divergence between a teacher and a
student distribution over the vocabulary, both produced by a linear head:

    z_s = X_s W_s^T / T,  z_t = X_t W_t^T / T          (student, teacher logits; T > 0)
    Q = softmax(z_s),     P = softmax(z_t)
    0 < beta < 1:  loss_i = beta KL(P || M) + (1 - beta) KL(Q || M),  M = beta P + (1-beta) Q
    beta = 0:      loss_i = KL(P || Q)      (forward KL, teacher -> student)
    beta = 1:      loss_i = KL(Q || P)      (reverse KL)

Rows whose label is ignore_index take no part (as in the cross-entropy op). Only the
student receives gradients. With g_v = dloss_i/dQ_v up to a constant,

    beta in (0,1): g_v = (1 - beta) log(Q_v / M_v)     beta = 1: g_v = log(Q_v / P_v)
    dloss_i/dz_s = Q * (g - sum_u Q_u g_u)             beta = 0: dloss_i/dz_s = Q - P
    dS = c_i dloss_i/dz_s / T,   dX_s = dS W_s,   dW_s += dS^T X_s

with c_i the upstream gradient factor (g/N for mean, g for sum, g_i for none). Pins live
in tests/test_jsd_oracle.py (identical distributions, finite differences, torch float64
kl_div and autograd, symmetry at beta = 0.5, the log 2 bound).
"""

from __future__ import annotations

import numpy as np

from .flce_oracle import grad_scales


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def _log_softmax(z):
    m = z.max(axis=1, keepdims=True)
    return z - (m + np.log(np.exp(z - m).sum(axis=1, keepdims=True)))


def jsd_rows(zs, zt, beta):
    """Per-row loss and dloss/dz_s for student / teacher logits (already divided by T)."""
    logQ = _log_softmax(zs)
    logP = _log_softmax(zt)
    Q = np.exp(logQ)
    P = np.exp(logP)
    if beta == 0.0:
        loss = (P * (logP - logQ)).sum(axis=1)
        dz = Q - P
    elif beta == 1.0:
        loss = (Q * (logQ - logP)).sum(axis=1)
        g = logQ - logP
        dz = Q * (g - (Q * g).sum(axis=1, keepdims=True))
    else:
        M = beta * P + (1.0 - beta) * Q
        logM = np.log(M)
        loss = beta * (P * (logP - logM)).sum(axis=1) + (1.0 - beta) * (Q * (logQ - logM)).sum(axis=1)
        g = (1.0 - beta) * (logQ - logM)
        dz = Q * (g - (Q * g).sum(axis=1, keepdims=True))
    return loss, dz


def jsd_oracle(Xs, Ws, Xt, Wt, labels=None, beta=0.5, temperature=1.0, ignore_index=-100,
               reduction="mean", grad_out=None, want_dX=True, want_dW=True, row_block=64):
    """Full float64 fused linear JSD. Returns loss (scalar or [BT]), loss_tok [BT],
    n_labelled, mask, dX [BT,Hs] or None, dW [V,Hs] or None."""
    Xs = np.asarray(Xs)
    BT, Hs = Xs.shape
    V = np.asarray(Ws).shape[0]
    if labels is None:
        mask = np.ones(BT, dtype=bool)
    else:
        mask = np.asarray(labels, dtype=np.int64) != ignore_index
    c = grad_scales(mask, reduction, grad_out)
    rows = np.nonzero(mask)[0]
    n = rows.shape[0]
    T = float(temperature)
    Ws64 = _f64(Ws)
    Wt64 = _f64(Wt)
    loss_tok = np.zeros(BT)
    dX = np.zeros((BT, Hs)) if want_dX else None
    dW = np.zeros((V, Hs)) if want_dW else None
    for k0 in range(0, n, row_block):
        blk = rows[k0:k0 + row_block]
        xs = _f64(Xs[blk])
        zs = xs @ Ws64.T / T
        zt = _f64(np.asarray(Xt)[blk]) @ Wt64.T / T
        loss, dz = jsd_rows(zs, zt, beta)
        loss_tok[blk] = loss
        dS = dz * (c[blk] / T)[:, None]
        if want_dX:
            dX[blk] = dS @ Ws64
        if want_dW:
            dW += dS.T @ xs
    if reduction == "none":
        red = loss_tok.copy()
    elif reduction == "mean":
        red = float(loss_tok[mask].sum() / n) if n > 0 else 0.0
    else:
        red = float(loss_tok[mask].sum())
    return {"loss": red, "loss_tok": loss_tok, "n_labelled": int(n), "mask": mask, "dX": dX, "dW": dW}
