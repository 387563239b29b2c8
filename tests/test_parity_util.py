"""CPU checks of the argmax acceptance rule the GPU parity tests use (parity_util.pred_ok):
the fp32 spread it allows covers what real fp32 evaluations of bf16 logits do, and it
rejects a prediction that is wrong by more than rounding."""

import numpy as np
import torch

from oracle import flce_oracle as orc
from parity_util import fp32_logit_spread, max_argmax_mismatches, pred_ok


def _bf16(a):
    return torch.from_numpy(a).to(torch.bfloat16).double().numpy()


def test_spread_covers_blas_fp32_logits():
    """Four times the spread of a logit bounds the deviation of the float32 BLAS product
    (another summation order) from the float64 value, on 300 random head-shaped logits
    (H = 4096, x ~ N(0,1), w ~ N(0, 0.02^2), as in the Llama-shaped workloads)."""
    rng = np.random.default_rng(11)
    H = 4096
    X = _bf16(rng.standard_normal((10, H)))
    W = _bf16(rng.standard_normal((30, H)) * 0.02)
    s32 = X.astype(np.float32) @ W.astype(np.float32).T
    s64 = X @ W.T
    worst = 0.0
    for i in range(X.shape[0]):
        for v in range(W.shape[0]):
            sp = fp32_logit_spread(X[i], W[v])
            assert sp > 0.0
            worst = max(worst, abs(float(s32[i, v]) - s64[i, v]) / (4.0 * sp))
    assert worst <= 1.0, worst


def test_spread_is_far_below_the_worst_case_band():
    """The realistic spread is orders of magnitude tighter than the worst-case band."""
    rng = np.random.default_rng(12)
    H = 4096
    x = _bf16(rng.standard_normal(H))
    W = _bf16(rng.standard_normal((4, H)) * 0.02)
    band = orc.argmax_tie_band(orc._absdot_max(np.abs(x[None, :]), W)[0], 0.0, H)
    for v in range(4):
        assert 8.0 * fp32_logit_spread(x, W[v]) < band / 100.0


def test_pred_ok_rejects_a_wrong_index_and_accepts_a_true_tie():
    rng = np.random.default_rng(13)
    H, V = 256, 64
    X = _bf16(rng.standard_normal((3, H)))
    W = _bf16(rng.standard_normal((V, H)) * 0.05)
    W[40] = W[7]  # rows 7 and 40 give identical logits
    X[2] = 0.0
    X[2, :8] = 1.0
    W[7, :8] = 4.0  # row 2: logit 32 at columns 7 and 40, the rest small
    W[40, :8] = 4.0
    s = X @ W.T
    orc_pred = s.argmax(axis=1)
    assert orc_pred[2] == 7
    mask = np.ones(3, dtype=bool)
    rows = np.arange(3)
    # the runner-up of row 0 (below the maximum by more than rounding) is not a tie: rejected
    order = np.argsort(s[0])[::-1]
    second = next(v for v in order if s[0, v] < s[0, order[0]] - 1e-3)
    bad = orc_pred.copy()
    bad[0] = second
    ok, where = pred_ok(bad, orc_pred, X, W, None, rows, mask)
    assert not ok and where == 0
    # the higher index of an exact tie: accepted and counted
    tie = orc_pred.copy()
    tie[2] = 40
    rep = []
    ok, n = pred_ok(tie, orc_pred, X, W, None, rows, mask, report=rep)
    assert ok and n == 1 and rep[0][0] == 2 and rep[0][1] == 0.0
    # an ignored row must predict -1 exactly
    ok, where = pred_ok(tie, orc_pred, X, W, None, rows, np.array([True, True, False]))
    assert not ok and where == 2


def test_mismatch_cap():
    assert max_argmax_mismatches(8176) == 3
    assert max_argmax_mismatches(32768) == 10
