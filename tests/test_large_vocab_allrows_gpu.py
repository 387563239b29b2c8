"""The large-vocabulary long-context workload (BT = 32768, H = 5376, V = 262144, Zipf(1.1)
targets, every row labelled) against the float64 oracle on every row, in the launch
configuration the benchmark times: the workload's 1.5 GiB workspace cap, which gives
2688-row chunks, so the call runs 13 chunks and dW is accumulated across all of them
("feat(flce): expose direct chunk-size control via LIGER_FLCE_CHUNK_SIZE", Details table:
the BT = 32768, H = 5376, V = 262144 rows).

Compared: lse, per-token loss and prediction of all 32768 rows (the oracle's row-blocked
float64 forward over the whole vocabulary, 92 TFLOP); dW on 256 sampled vocabulary rows
accumulated over all 32768 rows, i.e. across every chunk of the call (a dropped or doubled
chunk changes it by a thirteenth); dX on 4 sampled rows of every 1024-row block. The call
uses reduction "none" with an upstream gradient of ones, which gives every row the
gradient factor of the workload's "sum" (c_i = 1) and returns every per-token loss; the
reduced "sum" call is compared with the sum of those per-token losses.
"""

import concurrent.futures as cf

import numpy as np
import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import flce
from linear_cross_entropy_logits_gb300 import inputs as I
from oracle import flce_oracle as orc
from parity_util import TOL, max_argmax_mismatches, pred_ok, rel_fro

pytestmark = pytest.mark.gpu

BLOCK = 1024


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    flce.load()


def _rows_forward_threaded(s, t, z, pool, parts=16):
    """orc.rows_forward over row slices in parallel threads (the oracle is row-independent;
    numpy's elementwise passes release the GIL)."""
    n = s.shape[0]
    cuts = np.linspace(0, n, parts + 1).astype(int)
    futs = [pool.submit(orc.rows_forward, s[a:b], t[a:b], z) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    res = [f.result() for f in futs]
    return [np.concatenate([r[k] for r in res], axis=0) for k in range(6)]


def test_large_vocab_every_row_and_dW_across_chunks():
    sp = I.spec("large_vocab")
    inp = I.generate(sp, seed=0)
    BT, H, V = sp["BT"], sp["H"], sp["V"]
    z = sp.get("z", 0.0)
    cap = sp["workspace_cap"]
    R = flce.chunk_rows(BT, H, V, torch.bfloat16, flce.workspace_size(BT, H, V, torch.bfloat16, cap))
    assert R == 2688 and -(-BT // R) == 13
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    dW = torch.zeros(V, H, dtype=torch.float32, device="cuda")
    ones = torch.ones(BT, device="cuda")
    out = flce.fwd_bwd(d["X"], d["W"], d["targets"], None, reduction="none", z_loss_scale=z,
                       grad_out=ones, want_dX=True, want_dW=True, dW=dW, budget_bytes=cap)
    assert out["status_code"] == flce.FLCE_OK
    red = flce.fwd_bwd(d["X"], d["W"], d["targets"], None, reduction="sum", z_loss_scale=z,
                       want_dX=False, want_dW=False, budget_bytes=cap)
    assert red["status_code"] == flce.FLCE_OK
    lse = out["lse"].cpu().numpy()
    loss = out["loss"].cpu().numpy()
    pred = out["pred"].cpu().numpy()
    tot = float(np.sum(loss.astype(np.float64)))
    assert abs(float(red["loss"][0]) - tot) <= 1e-5 * abs(tot)

    rng = np.random.default_rng(2024)
    t = inp["targets"].numpy()
    # sampled vocabulary rows: the most frequent Zipf targets (ranks 1..32), and random ones
    vs = np.unique(np.concatenate([np.arange(32), rng.choice(V, size=224, replace=False)]))
    dW_got = dW[torch.from_numpy(vs).cuda()].cpu().numpy()
    dx_rows = np.sort(np.concatenate([k0 + rng.choice(BLOCK, size=4, replace=False)
                                      for k0 in range(0, BT, BLOCK)]))
    dX_got = out["dX"][torch.from_numpy(dx_rows).cuda()].float().cpu().numpy()
    del out, red, dW, d
    torch.cuda.empty_cache()

    X = I.to_numpy_exact(inp["X"])
    W64 = I.to_numpy_exact(inp["W"]).astype(np.float64)
    del inp
    c = np.ones(BT)
    dW_ref = np.zeros((vs.size, H))
    # the device balances the labelled rows over the chunks: cdiv(N, R) chunks of r_eff rows,
    # r_eff = cdiv(N, chunks) rounded up to 128
    n_chunks = -(-BT // R)
    r_eff = -(-(-(-BT // n_chunks)) // 128) * 128
    dW_part = np.zeros((n_chunks, vs.size, H))
    dX_ref = np.zeros((dx_rows.size, H))
    worst_lse = worst_loss = 0.0
    n_mis = 0
    tol = TOL["bf16"]
    with cf.ThreadPoolExecutor(16) as pool:
        for k0 in range(0, BT, BLOCK):
            r = np.arange(k0, min(BT, k0 + BLOCK))
            x64 = np.asarray(X[r], np.float64)
            s = x64 @ W64.T
            o_lse, o_loss, _, o_pred, _, p = _rows_forward_threaded(s, t[r], z, pool)
            del s
            dS = orc.rows_grad_logits(p, t[r], o_lse, c[r], z)
            del p
            for k in np.unique(r // r_eff):
                m = (r // r_eff) == k
                dW_part[k] += dS[m][:, vs].T @ x64[m]

            sel = np.nonzero(np.isin(r, dx_rows))[0]
            dX_ref[np.searchsorted(dx_rows, r[sel])] = dS[sel] @ W64
            del dS
            worst_lse = max(worst_lse, float(np.max(np.abs(lse[r] - o_lse) / np.abs(o_lse))))
            worst_loss = max(worst_loss, float(np.max(np.abs(loss[r] - o_loss) /
                                                      np.maximum(np.abs(o_loss), 1e-3))))
            ok, k = pred_ok(pred[r], o_pred, X, W64, None, r, np.ones(r.size, bool))
            assert ok, f"argmax mismatch outside the fp32 spread at row {k}"
            n_mis += k
    dW_ref = dW_part.sum(axis=0)
    print(f"large vocab: lse rel {worst_lse:.2e}, loss rel {worst_loss:.2e}, argmax near-tie "
          f"mismatches {n_mis} of {BT} rows, dW(256 rows) rel-Frobenius {rel_fro(dW_got, dW_ref):.2e}, "
          f"dX({dx_rows.size} rows) {rel_fro(dX_got, dX_ref):.2e}")
    assert worst_lse <= tol["loss"], f"lse rel err {worst_lse}"
    assert worst_loss <= tol["loss"], f"per-token loss rel err {worst_loss}"
    assert n_mis <= max_argmax_mismatches(BT)
    assert rel_fro(dW_got, dW_ref) <= tol["grad"], f"dW rel-Frobenius {rel_fro(dW_got, dW_ref)}"
    assert rel_fro(dX_got, dX_ref) <= tol["grad"], f"dX rel-Frobenius {rel_fro(dX_got, dX_ref)}"
    # the comparison would catch a dropped or doubled chunk: each chunk's share of the
    # sampled dW rows is far above the tolerance
    for k in range(n_chunks):
        share = np.linalg.norm(dW_part[k]) / np.linalg.norm(dW_ref)
        assert share > 10 * tol["grad"], (k, share)
