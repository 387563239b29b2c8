"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI binding,
run the float64 oracle on the same seeded inputs, and compare with the stated tolerances.

Tolerances (fixed by the method's contract, not tuned to results):
  * bf16/fp16 inputs: loss and per-token loss/lse relative error <= 2e-3; dX and dW
    relative Frobenius error <= 1e-2.
  * fp32 inputs: all of the above <= 1e-5.
  * Prediction and ignored-row mask: bit exact, except on rows whose two largest oracle
    logits are closer than the fp32 evaluation bound (oracle.argmax_tie_band), where
    either of the tied indices is accepted.
"""

import numpy as np
import torch

from linear_cross_entropy_logits_gb300 import flce
from linear_cross_entropy_logits_gb300 import inputs as I
from oracle import flce_oracle as orc

TOL = {"bf16": dict(loss=2e-3, grad=1e-2), "f16": dict(loss=2e-3, grad=1e-2),
       "f32": dict(loss=1e-5, grad=1e-5)}


def rel_fro(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def to_dev(inp, dev="cuda"):
    return {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()}


def run_gpu(inp, sp, dW_init=None, flags=0, workspace_bytes=None, budget_bytes=0, **kw):
    d = to_dev(inp)
    dW = None
    if sp.get("want_dW", True):
        dW = (dW_init.clone().cuda() if dW_init is not None else
              torch.zeros(sp["V"], sp["H"], dtype=torch.float32, device="cuda"))
    ws = None
    if workspace_bytes is not None:
        ws = torch.empty(workspace_bytes, dtype=torch.uint8, device="cuda")
    go = d["grad_out"]
    if sp["reduction"] != "none" and sp.get("grad_scalar") is not None:
        go = torch.tensor([sp["grad_scalar"]], dtype=torch.float32, device="cuda")
    out = flce.fwd_bwd(d["X"], d["W"], d["targets"], d["bias"], reduction=sp["reduction"],
                       z_loss_scale=sp.get("z", 0.0), grad_out=go, want_dX=sp.get("want_dX", True),
                       want_dW=sp.get("want_dW", True), dW=dW, workspace=ws,
                       budget_bytes=budget_bytes, flags=flags, **kw)
    torch.cuda.synchronize()
    res = {}
    for k, v in out.items():
        if torch.is_tensor(v) and k != "workspace":
            res[k] = v.detach().float().cpu().numpy() if v.dtype in (torch.bfloat16, torch.float16) \
                else v.detach().cpu().numpy()
        else:
            res[k] = v
    return res


def run_oracle(inp, sp):
    X = I.to_numpy_exact(inp["X"])
    W = I.to_numpy_exact(inp["W"])
    b = I.to_numpy_exact(inp["bias"])
    g = inp["grad_out"].numpy() if inp["grad_out"] is not None else None
    if sp["reduction"] != "none" and sp.get("grad_scalar") is not None:
        g = np.array([sp["grad_scalar"]])
    return orc.flce_oracle(X, W, inp["targets"].numpy(), bias=b, reduction=sp["reduction"],
                           z_loss_scale=sp.get("z", 0.0), grad_out=g,
                           want_dX=sp.get("want_dX", True), want_dW=sp.get("want_dW", True))


def pred_ok(gpu_pred, orc_pred, X, W, b, rows, targets_mask):
    """Bit-exact predictions except within the fp32 tie band of a row."""
    bad = np.nonzero(gpu_pred != orc_pred)[0]
    if bad.size == 0:
        return True, 0
    H = X.shape[1]
    bmax = 0.0 if b is None else float(np.max(np.abs(b)))
    for j in bad:
        r = rows[j]
        if not targets_mask[j]:
            return False, int(r)
        s = orc.logits_rows(np.asarray(X[r:r + 1], np.float64), W, b)[0]
        absdot = orc._absdot_max(np.abs(np.asarray(X[r:r + 1], np.float64)), W)[0]
        band = orc.argmax_tie_band(absdot, bmax, H)
        if s[gpu_pred[j]] < s.max() - band:
            return False, int(r)
    return True, int(bad.size)


def compare_full(g, o, inp, sp):
    """Element-by-element comparison of every output against the oracle."""
    dt = sp["dtype"]
    tol = TOL[dt]
    BT = sp["BT"]
    mask = o["mask"]
    assert int(g["n_labelled"][0]) == o["n_labelled"]
    # ignored-row outputs, bit exact
    assert np.all(g["pred"][~mask] == -1)
    assert np.all(g["lse"][~mask] == 0.0)
    if sp["reduction"] == "none":
        assert np.all(g["loss"][~mask] == 0.0)
        assert np.all(g["acc"][~mask] == 0.0)
        assert np.all(g["z_loss"][~mask] == 0.0)
        ref = o["loss"]
        den = np.maximum(np.abs(ref), 1e-3)
        err = np.max(np.abs(g["loss"] - ref) / den)
        assert err <= tol["loss"], f"per-token loss rel err {err}"
        zerr = np.max(np.abs(g["z_loss"] - o["z_loss"]) / np.maximum(np.abs(o["z_loss"]), 1e-6))
        assert zerr <= max(tol["loss"], 1e-4) or np.max(np.abs(o["z_loss"])) < 1e-6
    else:
        ref = o["loss"]
        err = abs(float(g["loss"][0]) - ref) / max(abs(ref), 1e-6)
        assert err <= tol["loss"], f"loss rel err {err}"
        zref = o["z_loss"]
        assert abs(float(g["z_loss"][0]) - zref) <= tol["loss"] * max(abs(zref), 1e-6) + 1e-7
    lse_err = np.max(np.abs(g["lse"][mask] - o["lse_tok"][mask]) /
                     np.maximum(np.abs(o["lse_tok"][mask]), 1e-3)) if mask.any() else 0.0
    assert lse_err <= tol["loss"], f"lse rel err {lse_err}"
    X = I.to_numpy_exact(inp["X"])
    W = I.to_numpy_exact(inp["W"])
    b = I.to_numpy_exact(inp["bias"])
    rows = np.arange(BT)
    ok, nties = pred_ok(g["pred"], o["pred_tok"], X, W, b, rows, mask)
    assert ok, f"argmax mismatch outside the tie band at row {nties}"
    # accuracy follows the prediction
    exp_acc = (g["pred"] == inp["targets"].numpy()).astype(np.float64) * mask
    if sp["reduction"] == "none":
        assert np.array_equal(g["acc"], exp_acc.astype(np.float32))
    if sp.get("want_dX", True):
        e = rel_fro(g["dX"], o["dX"])
        assert e <= tol["grad"], f"dX rel-Frobenius {e}"
        assert np.all(g["dX"][~mask] == 0.0)
    if sp.get("want_dW", True):
        e = rel_fro(g["dW"], o["dW"])
        assert e <= tol["grad"], f"dW rel-Frobenius {e}"
        if inp["bias"] is not None:
            e = rel_fro(g["dbias"], o["dbias"])
            assert e <= tol["grad"], f"dbias rel-Frobenius {e}"
    return nties
