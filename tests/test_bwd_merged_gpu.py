"""The merged dX + dW launch (one persistent kernel over a device-wide work queue, used by
tensor-core calls with both gradients whose chunks hold 2048 rows or more) against the
float64 oracle, element by element, at sizes with ragged tails in every dimension; and bit
for bit against the same call run as two launches (FLCE_FLAG_SEPARATE_BWD): which pair
draws which work item must not change a single bit. The products are the grad_input and
grad_weight GEMMs of "Liger-Kernel PR #1554: skip ignore_index rows" (Summary), dW
accumulated into the caller's buffer ("Reduce FLCE weight-gradient allocation overhead
across FP16, BF16, and FP32", Proposed direction)."""

import numpy as np
import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import flce
from linear_cross_entropy_logits_gb300 import inputs as I
from parity_util import TOL, compare_full, rel_fro, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    flce.load()


def _chunk_rows(sp, budget):
    dt = I.TORCH_DTYPES[sp["dtype"]]
    return flce.chunk_rows(sp["BT"], sp["H"], sp["V"], dt,
                           flce.workspace_size(sp["BT"], sp["H"], sp["V"], dt, budget))


@pytest.mark.parametrize("reduction,z", [("mean", 1e-4), ("sum", 0.0)])
def test_merged_matches_oracle_one_chunk(reduction, z):
    # 4500 rows, 380 of them ignored at random: one chunk of 4608 rows (>= 2048: merged)
    sp = I.spec("frozen_head", BT=4500, H=200, V=5000, w_std=0.1, bias_std=None, n_ignored=380,
                reduction=reduction, grad_out=None, want_dW=True, z=z)
    assert _chunk_rows(sp, 0) >= 2048
    inp = I.generate(sp, seed=61)
    compare_full(run_gpu(inp, sp), run_oracle(inp, sp), inp, sp)


def test_merged_matches_oracle_three_chunks():
    # 9000 labelled rows in a workspace of 4096-row chunks: three chunks, each merged
    sp = I.spec("llama1b", BT=9000, H=136, V=3100, w_std=0.15, z=1e-3)
    inp = I.generate(sp, seed=62)
    budget = flce.workspace_size(sp["BT"], sp["H"], sp["V"], torch.bfloat16, 0)
    for b in range(budget, 0, -(1 << 16)):
        if _chunk_rows(sp, b) == 4096:
            budget = b
            break
    assert _chunk_rows(sp, budget) == 4096
    compare_full(run_gpu(inp, sp, budget_bytes=budget), run_oracle(inp, sp), inp, sp)


def test_merged_same_dtype_dW():
    sp = I.spec("llama1b", BT=4300, H=96, V=2600, w_std=0.2, reduction="sum")
    inp = I.generate(sp, seed=63)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    init = (torch.randn(sp["V"], sp["H"], generator=torch.Generator().manual_seed(64)) * 0.01).to(torch.bfloat16)
    dW = init.clone().cuda()
    out = flce.fwd_bwd(d["X"], d["W"], d["targets"], None, reduction="sum", dW=dW)
    assert out["status_code"] == flce.FLCE_OK
    o = run_oracle(inp, sp)
    assert rel_fro(out["dW"].float().cpu().numpy() - init.float().numpy(), o["dW"]) <= TOL["bf16"]["grad"]
    assert rel_fro(out["dX"].float().cpu().numpy(), o["dX"]) <= TOL["bf16"]["grad"]


@pytest.mark.parametrize("dw_dtype", ["f32", "same", "overwrite"])
def test_merged_equals_two_launches_bitwise(dw_dtype):
    sp = I.spec("llama8b", BT=5120, H=512, V=8000, w_std=0.05, labelled_fraction=0.9, z=1e-4)
    inp = I.generate(sp, seed=65)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    res = []
    for flags in (0, flce.FLAG_SEPARATE_BWD):
        dt = torch.float32 if dw_dtype == "f32" else torch.bfloat16
        dW = torch.full((sp["V"], sp["H"]), 0.25, dtype=dt, device="cuda")
        f = flags | (flce.FLAG_DW_OVERWRITE if dw_dtype == "overwrite" else 0)
        out = flce.fwd_bwd(d["X"], d["W"], d["targets"], None, reduction="mean", z_loss_scale=sp["z"],
                           dW=dW, flags=f)
        assert out["status_code"] == flce.FLCE_OK
        res.append((out["dX"].clone(), out["dW"].clone(), out["loss"].clone()))
    for a, b in zip(res[0], res[1]):
        assert torch.equal(a, b)
