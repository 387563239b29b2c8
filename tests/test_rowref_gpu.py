"""GPU parity of the row-reference form of the bf16 tensor-core path.

By default a bf16 tensor-core call with gradients and no dbias stores exp(s) in the slab
and normalises each row with one scale (no pass over the slab). Rows outside the window
(|row max| > 60, or a row scale outside exp(+-70)) make the device redo their chunk with
per-tile maxima. Every case here is compared element by element with the float64 oracle,
and with the per-tile form forced by FLCE_FLAG_NO_ROW_REF. The window flag is read back
from the workspace's control record (int32 word 6 of the record at offset 0: the flag of
the last chunk), to check which form ran.
"""

import numpy as np
import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import flce
from linear_cross_entropy_logits_gb300 import inputs as I
from parity_util import compare_full, rel_fro, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

FB_WORD = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    flce.load()


def _run(inp, sp, flags=0, budget_bytes=0):
    """run_gpu plus the last chunk's window flag."""
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    nbytes = flce.workspace_size(sp["BT"], sp["H"], sp["V"], I.TORCH_DTYPES[sp["dtype"]], budget_bytes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    g = run_gpu(inp, sp, flags=flags, workspace_bytes=None, budget_bytes=budget_bytes)
    # a second call into our own workspace, only to read the flag the call leaves behind
    dW = torch.zeros(sp["V"], sp["H"], dtype=torch.float32, device="cuda") if sp.get("want_dW", True) else None
    go = d["grad_out"] if sp["reduction"] == "none" else None
    flce.fwd_bwd(d["X"], d["W"], d["targets"], d["bias"], reduction=sp["reduction"],
                 z_loss_scale=sp.get("z", 0.0), grad_out=go, want_dW=sp.get("want_dW", True), dW=dW,
                 workspace=ws, flags=flags)
    torch.cuda.synchronize()
    fb = int(ws[:32].view(torch.int32)[FB_WORD].item())
    return g, fb


CASES = [
    ("bf16_mean_ragged", "llama1b", dict(BT=300, H=192, V=3000, w_std=0.2, ignore="random", n_ignored=40)),
    ("bf16_z_prompt_first", "llama8b", dict(BT=1024, H=256, V=2304, w_std=0.1, labelled_fraction=0.5, z=1e-2)),
    ("bf16_none_grad_out", "llama1b", dict(BT=260, H=136, V=1300, w_std=0.2, reduction="none",
                                           grad_out="uniform", ignore="random", n_ignored=30)),
    ("bf16_frozen_bias_dX_only", "frozen_head", dict(BT=400, H=128, V=5000, w_std=0.15, bias_std=0.3,
                                                     n_ignored=200)),
]


@pytest.mark.parametrize("name,base,ov", CASES, ids=[c[0] for c in CASES])
def test_row_reference_matches_oracle_and_tile_form(name, base, ov):
    sp = I.spec(base, **ov)
    inp = I.generate(sp, seed=11)
    o = run_oracle(inp, sp)
    g_ref, fb = _run(inp, sp)
    assert fb == 0 and g_ref["status_code"] == flce.FLCE_OK
    g_tile, _ = _run(inp, sp, flags=flce.FLAG_NO_ROW_REF)
    compare_full(g_ref, o, inp, sp)
    compare_full(g_tile, o, inp, sp)
    assert np.array_equal(g_ref["pred"], g_tile["pred"])
    assert rel_fro(g_ref["dX"], g_tile["dX"]) < 1e-2


@pytest.mark.parametrize("H", [256, 4096])
def test_large_logits_fall_back_per_tile(H):
    """Row maxima far above the window (X scaled so that |s| reaches ~100): the chunk is
    redone with per-tile maxima and still matches the oracle (H = 4096: on the wide forward
    tile)."""
    sp = I.spec("llama1b", BT=300, H=H, V=3000, x_std=4.0, w_std=6.4 / H ** 0.5, ignore="random",
                n_ignored=20)
    inp = I.generate(sp, seed=12)
    o = run_oracle(inp, sp)
    assert np.max(o["lse_tok"]) > 80.0
    g, fb = _run(inp, sp)
    assert fb == 1 and g["status_code"] == flce.FLCE_OK
    compare_full(g, o, inp, sp)


def test_very_negative_logits_fall_back():
    """Every logit below -60 (bias shifted by -100, dX only): the window's lower side."""
    sp = I.spec("frozen_head", BT=256, H=128, V=2000, w_std=0.1, bias_std=0.1, n_ignored=50)
    inp = I.generate(sp, seed=13)
    inp["bias"] = (inp["bias"].float() - 100.0).to(torch.bfloat16)
    o = run_oracle(inp, sp)
    g, fb = _run(inp, sp)
    assert fb == 1
    compare_full(g, o, inp, sp)


def test_tiny_upstream_gradient_falls_back():
    """A per-token upstream gradient of 1e-35 on some rows puts their row scale below the
    window (the pre-scaled Xc rows would leave the bf16 normal range)."""
    sp = I.spec("llama1b", BT=200, H=128, V=1500, w_std=0.2, reduction="none", grad_out="uniform",
                ignore="random", n_ignored=10)
    inp = I.generate(sp, seed=14)
    inp["grad_out"][::7] = 1e-35
    o = run_oracle(inp, sp)
    g, fb = _run(inp, sp)
    assert fb == 1
    compare_full(g, o, inp, sp)


def test_one_chunk_of_many_falls_back():
    """128-row chunks; one row of one middle chunk gets logits far above the window. Only
    that chunk is redone (the flag is reset per chunk: the last chunk's flag is 0) and the
    whole result matches the oracle and the per-tile form."""
    sp = I.spec("llama8b", BT=1024, H=128, V=1500, w_std=0.2, labelled_fraction=0.75, z=1e-3)
    inp = I.generate(sp, seed=15)
    lab = np.nonzero(inp["targets"].numpy() != I.IGNORE_INDEX)[0]
    r = int(lab[len(lab) // 2])
    inp["X"][r] = (inp["X"][r].float() * 60.0).to(torch.bfloat16)
    budget = flce.workspace_size(128, sp["H"], sp["V"], torch.bfloat16, 0) + 16 * sp["BT"] + 4096
    assert flce.chunk_rows(sp["BT"], sp["H"], sp["V"], torch.bfloat16, budget) == 128
    o = run_oracle(inp, sp)
    assert o["lse_tok"][r] > 60.0
    g, fb = _run(inp, sp, budget_bytes=budget)
    assert fb == 0
    compare_full(g, o, inp, sp)
    g_tile, _ = _run(inp, sp, flags=flce.FLAG_NO_ROW_REF, budget_bytes=budget)
    assert rel_fro(g["dW"], g_tile["dW"]) < 1e-2
