"""Float64 CPU oracle for fused linear cross entropy (FLCE), forward and backward.

TEST INFRASTRUCTURE. Only the test suite (``tests/``), the smoke check in
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import or run this module. The product path (the CUDA library and its
Python binding) never imports it, and this module imports nothing from the product.

What it computes
----------------
The pages describe one op: a language-model head projection followed by cross entropy,
computed chunk by chunk so that the full [tokens, vocabulary] logits never exist at once
("Reduce FLCE weight-gradient allocation overhead across FP16, BF16, and FP32", section
"Background and motivation"). The forward runs the logits, grad_input and grad_weight
products in one call ("Liger-Kernel PR #1554: skip ignore_index rows", Summary), so the
gradients are produced together with the loss. Rows whose target equals ``ignore_index``
add nothing to the loss or to any gradient (PR #1554, Summary); they still receive
per-token outputs: zero loss, zero z-loss, zero accuracy, predicted token -1 and a zero
grad_input row (PR #1554, Details item 1). A NaN stored in an ignored row must reach no
output (PR #1554, Tests, ``test_ignored_rows_do_not_enter_projection``). The weight
gradient is accumulated into the caller's destination, ``dW += G^T X`` (issue "Reduce
FLCE weight-gradient allocation overhead", section "Proposed direction").

The pages print no formula for the loss itself; this module takes the textbook
definition of softmax cross entropy plus a squared-logsumexp z-loss. For each labelled
row i with target t_i (float64 throughout, inputs upcast exactly):

    s_v   = sum_h X[i,h] W[v,h] + b_v                      (logits of row i)
    lse_i = log sum_v exp(s_v)          (evaluated as M + log sum exp(s_v - M))
    loss_i = (lse_i - s_{t_i}) + z * lse_i^2      z-loss_i = z * lse_i^2
    pred_i = argmax_v s_v (lowest index on exact ties)    acc_i = [pred_i == t_i]
    dS_v  = c_i * (p_v * (1 + 2 z lse_i) - [v == t_i]),  p_v = exp(s_v - lse_i)
    dX_i  = sum_v dS_v W[v]      dW += dS^T X      dbias += sum_i dS

c_i is the upstream gradient of the returned loss with respect to loss_i: ``g / N`` for
``mean`` (N = number of labelled rows), ``g`` for ``sum``, ``g_i`` for ``none``, where g
is the scalar upstream gradient (1 when not given) and g_i the per-token one.

Readings where the pages are silent:
  * z-loss is ``z * lse^2``, added to the loss and also reported on its own.
  * ``mean`` divides by the number of labelled rows; with none labelled the loss is 0
    and every gradient is 0.
  * A labelled target outside [0, V) is treated as ignored and flagged.
  * lse of an ignored row is reported as 0.
  * ``mean``/``sum`` reduce z-loss and accuracy the same way as the loss.

Parity of this oracle is pinned in ``tests/test_oracle.py`` by closed forms, central
finite differences, a brute-force evaluation through torch's float64 ``cross_entropy``
with autograd, and invariants (zero-sum gradient rows, shift invariance, NaN isolation).
"""

from __future__ import annotations

import numpy as np

REDUCTIONS = ("mean", "sum", "none")


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def labelled_rows(targets, ignore_index, V):
    """Return (mask, out_of_range) for a target vector.

    mask[i] is True for rows that enter the loss (PR #1554, Summary: rows whose target is
    ignore_index add nothing). A target that is neither ignore_index nor in [0, V) is
    treated as ignored and reported through ``out_of_range`` (a reading: the pages do not
    cover it).
    """
    t = np.asarray(targets, dtype=np.int64)
    not_ignored = t != ignore_index
    in_range = (t >= 0) & (t < V)
    mask = not_ignored & in_range
    out_of_range = bool(np.any(not_ignored & ~in_range))
    return mask, out_of_range


def grad_scales(mask, reduction, grad_out):
    """Upstream gradient c_i of the returned loss with respect to loss_i, per row.

    ``reduction="none"`` takes a per-token upstream gradient (PR #1554, Tests:
    ``test_correctness_ignored_rows`` with a per-token upstream gradient); ``mean`` and
    ``sum`` take a scalar one. Ignored rows get 0.
    """
    if reduction not in REDUCTIONS:
        raise ValueError(f"reduction must be one of {REDUCTIONS}")
    BT = mask.shape[0]
    n = int(mask.sum())
    if reduction == "none":
        g = np.ones(BT) if grad_out is None else np.asarray(grad_out, np.float64).reshape(BT)
        c = np.where(mask, g, 0.0)
    else:
        g = 1.0 if grad_out is None else float(np.asarray(grad_out, np.float64).reshape(-1)[0])
        if reduction == "mean":
            scale = g / n if n > 0 else 0.0
        else:
            scale = g
        c = np.where(mask, scale, 0.0)
    return c


def logits_rows(x_rows, W, bias=None, v_block=32768):
    """s = x_rows @ W^T + b in float64, for a few rows, over all V (W converted per block)."""
    x = _f64(x_rows)
    V = W.shape[0]
    out = np.empty((x.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, v_block):
        v1 = min(V, v0 + v_block)
        out[:, v0:v1] = x @ _f64(W[v0:v1]).T
    if bias is not None:
        out += _f64(bias)[None, :]
    return out


def rows_forward(s, t, z):
    """Per-row forward statistics from float64 logits s [n, V] and targets t [n].

    Returns lse, loss, z-loss, pred, acc, p (softmax) for each row.
    """
    n = s.shape[0]
    M = s.max(axis=1)
    lse = M + np.log(np.exp(s - M[:, None]).sum(axis=1))
    ar = np.arange(n)
    s_t = s[ar, t]
    zl = z * lse * lse
    loss = (lse - s_t) + zl
    pred = s.argmax(axis=1).astype(np.int64)  # numpy returns the first maximum
    acc = (pred == t).astype(np.float64)
    p = np.exp(s - lse[:, None])
    return lse, loss, zl, pred, acc, p


def rows_grad_logits(p, t, lse, c, z):
    """dS = c_i (p (1 + 2 z lse_i) - onehot(t_i)) for a block of rows."""
    dS = p * (1.0 + 2.0 * z * lse)[:, None]
    dS[np.arange(p.shape[0]), t] -= 1.0
    dS *= c[:, None]
    return dS


def dX_rows(dS, W, v_block=32768):
    """dX_i = sum_v dS_iv W[v] in float64, W converted per vocabulary block."""
    V, H = W.shape
    out = np.zeros((dS.shape[0], H), dtype=np.float64)
    for v0 in range(0, V, v_block):
        v1 = min(V, v0 + v_block)
        out += dS[:, v0:v1] @ _f64(W[v0:v1])
    return out


def flce_oracle(X, W, targets, bias=None, ignore_index=-100, reduction="mean",
                z_loss_scale=0.0, grad_out=None, want_dX=True, want_dW=True,
                row_block=64):
    """Full float64 FLCE forward + backward. Returns a dict of float64/int64 arrays.

    Keys: loss, z_loss, acc (reduced per ``reduction``: scalars for mean/sum, [BT] for
    none), lse_tok, loss_tok, z_loss_tok, acc_tok, pred_tok ([BT] per token), n_labelled,
    out_of_range, dX ([BT,H] or None), dW ([V,H] or None, the contribution of this call),
    dbias ([V] or None).
    """
    X = np.asarray(X)
    W = np.asarray(W)
    BT, H = X.shape
    V = W.shape[0]
    z = float(z_loss_scale)
    t_all = np.asarray(targets, dtype=np.int64)
    mask, oor = labelled_rows(t_all, ignore_index, V)
    c = grad_scales(mask, reduction, grad_out)
    rows = np.nonzero(mask)[0]
    n = rows.shape[0]

    loss_tok = np.zeros(BT)
    zl_tok = np.zeros(BT)
    lse_tok = np.zeros(BT)
    acc_tok = np.zeros(BT)
    pred_tok = np.full(BT, -1, dtype=np.int64)
    dX = np.zeros((BT, H)) if want_dX else None
    dW = np.zeros((V, H)) if want_dW else None
    db = np.zeros(V) if (want_dW and bias is not None) else None

    for k0 in range(0, n, row_block):
        blk = rows[k0:k0 + row_block]
        t = t_all[blk]
        xb = _f64(X[blk])
        s = logits_rows(xb, W, bias)
        lse, loss, zl, pred, acc, p = rows_forward(s, t, z)
        loss_tok[blk] = loss
        zl_tok[blk] = zl
        lse_tok[blk] = lse
        acc_tok[blk] = acc
        pred_tok[blk] = pred
        if want_dX or want_dW:
            dS = rows_grad_logits(p, t, lse, c[blk], z)
            if want_dX:
                dX[blk] = dX_rows(dS, W)
            if want_dW:
                dW += dS.T @ xb
                if db is not None:
                    db += dS.sum(axis=0)

    if reduction == "none":
        loss, zl_out, acc_out = loss_tok.copy(), zl_tok.copy(), acc_tok.copy()
    else:
        div = float(n) if (reduction == "mean" and n > 0) else 1.0
        if reduction == "mean" and n == 0:
            loss, zl_out, acc_out = 0.0, 0.0, 0.0
        else:
            loss = float(loss_tok[mask].sum() / div)
            zl_out = float(zl_tok[mask].sum() / div)
            acc_out = float(acc_tok[mask].sum() / div)
    return {
        "loss": loss, "z_loss": zl_out, "acc": acc_out,
        "loss_tok": loss_tok, "z_loss_tok": zl_tok, "lse_tok": lse_tok,
        "acc_tok": acc_tok, "pred_tok": pred_tok,
        "n_labelled": int(n), "out_of_range": oor, "mask": mask,
        "dX": dX, "dW": dW, "dbias": db,
    }


def flce_oracle_rows(X, W, targets, rows, bias=None, ignore_index=-100, reduction="mean",
                     z_loss_scale=0.0, grad_out=None, want_dX=True):
    """Per-row oracle outputs for a sample of rows of a large problem.

    The loss, lse, prediction and dX of a row depend only on that row's logits and on its
    upstream gradient c_i (which needs only the labelled count), so each sampled row is
    evaluated exactly as in :func:`flce_oracle`. Returns a dict of arrays indexed like
    ``rows``; ignored rows get the ignored-row outputs.
    """
    X = np.asarray(X)
    W = np.asarray(W)
    V = W.shape[0]
    H = X.shape[1]
    z = float(z_loss_scale)
    t_all = np.asarray(targets, dtype=np.int64)
    mask, _ = labelled_rows(t_all, ignore_index, V)
    c = grad_scales(mask, reduction, grad_out)
    rows = np.asarray(rows, dtype=np.int64)
    k = rows.shape[0]
    out = {
        "loss_tok": np.zeros(k), "z_loss_tok": np.zeros(k), "lse_tok": np.zeros(k),
        "acc_tok": np.zeros(k), "pred_tok": np.full(k, -1, dtype=np.int64),
        "dX": np.zeros((k, H)) if want_dX else None,
        "logit_gap": np.full(k, np.inf), "logit_absdot": np.zeros(k),
    }
    sel = np.nonzero(mask[rows])[0]
    if sel.size:
        r = rows[sel]
        t = t_all[r]
        xb = _f64(X[r])
        s = logits_rows(xb, W, bias)
        lse, loss, zl, pred, acc, p = rows_forward(s, t, z)
        out["loss_tok"][sel] = loss
        out["z_loss_tok"][sel] = zl
        out["lse_tok"][sel] = lse
        out["acc_tok"][sel] = acc
        out["pred_tok"][sel] = pred
        srt = np.sort(s, axis=1)
        out["logit_gap"][sel] = srt[:, -1] - srt[:, -2] if s.shape[1] > 1 else np.inf
        out["logit_absdot"][sel] = _absdot_max(np.abs(xb), W)
        if want_dX:
            dS = rows_grad_logits(p, t, lse, c[r], z)
            out["dX"][sel] = dX_rows(dS, W)
    return out


def _absdot_max(xa, W, v_block=32768):
    """max_v sum_h |x_h| |W[v,h]| per row (used for the fp32 argmax error bound)."""
    V = W.shape[0]
    m = np.zeros(xa.shape[0])
    for v0 in range(0, V, v_block):
        v1 = min(V, v0 + v_block)
        m = np.maximum(m, (xa @ np.abs(_f64(W[v0:v1])).T).max(axis=1))
    return m


def argmax_tie_band(absdot, bias_absmax, H):
    """Worst-case fp32 logit error bound delta_i for the argmax comparison.

    Two logits of one row are each computed as an fp32 dot product of length H followed by
    one bias addition; the standard bound for a dot product summed in any order is
    |fl(x.y) - x.y| <= gamma_H sum |x_h y_h| with gamma_H = H u / (1 - H u) (Higham,
    Accuracy and Stability of Numerical Algorithms, section 3.1), and the bias addition
    adds at most u (|x.y| + |b|). u is taken as 2^-23, twice the fp32 unit roundoff, so
    that the bound also covers accumulators that truncate instead of rounding to nearest.
    A row whose two largest float64 logits are further apart than the sum of the two
    logits' bounds has an argmax that any such fp32 evaluation must reproduce exactly.
    """
    u = 2.0 ** -23
    gam = H * u / (1.0 - H * u)
    one = gam * absdot + u * (absdot + bias_absmax)
    return 2.0 * one


def flce_oracle_dW(X, W, targets, bias=None, ignore_index=-100, reduction="mean",
                   z_loss_scale=0.0, grad_out=None, row_block=64):
    """dW (and dbias) of one call, float64, for problems whose labelled rows are few.

    Identical arithmetic to :func:`flce_oracle`, returned without the dX work.
    """
    r = flce_oracle(X, W, targets, bias=bias, ignore_index=ignore_index,
                    reduction=reduction, z_loss_scale=z_loss_scale, grad_out=grad_out,
                    want_dX=False, want_dW=True, row_block=row_block)
    return r["dW"], r["dbias"]
