"""Which row chunks run. The pages pin their op's row skipping with 0 / 1 / 8 / 24 / 40
ignored rows of 40 giving 3 / 3 / 2 / 1 / 0 logits GEMMs at 16-row chunks, because that op
skips only chunks whose rows are all ignored ("Liger-Kernel PR #1554: skip ignore_index
rows", Tests). Here every ignored row is compacted away first and the device runs
cdiv(N_labelled, R) chunks, so the same pattern appears scaled to 128-row units (R = 2048
rows of a 40-unit call), and a partly ignored unit costs less rather than the same. The
chunk count is read back from the workspace's control record (int32 word 1 of the record
at offset 0), and every output is compared with the float64 oracle."""

import numpy as np
import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import flce
from linear_cross_entropy_logits_gb300 import inputs as I
from parity_util import compare_full, run_oracle

pytestmark = pytest.mark.gpu

N_CHUNKS_WORD = 1
UNIT = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    flce.load()


@pytest.mark.parametrize("ignored_units,ignored_rows,chunks", [
    (0, 0, 3), (1, 0, 3), (8, 0, 2), (24, 0, 1), (40, 0, 0),
    (0, 1, 3),        # one ignored row: still three chunks (5119 rows)
    (8, 1, 2),        # 4095 labelled rows: two chunks, not three
])
def test_chunks_follow_the_labelled_count(ignored_units, ignored_rows, chunks):
    BT = 40 * UNIT
    sp = I.spec("llama1b", BT=BT, H=64, V=1000, w_std=0.3, ignore="random", n_ignored=0)
    inp = I.generate(sp, seed=40 + ignored_units)
    t = inp["targets"].numpy().copy()
    t[:ignored_units * UNIT] = I.IGNORE_INDEX
    t[BT - ignored_rows:] = I.IGNORE_INDEX
    inp["targets"] = torch.from_numpy(t)
    R = 16 * UNIT
    ws_bytes = flce.workspace_size(R, sp["H"], sp["V"], torch.bfloat16, 0) + 16 * BT + 4096
    assert flce.chunk_rows(BT, sp["H"], sp["V"], torch.bfloat16, ws_bytes) == R
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    dW = torch.zeros(sp["V"], sp["H"], dtype=torch.float32, device="cuda")
    out = flce.fwd_bwd(d["X"], d["W"], d["targets"], None, reduction="mean", dW=dW, workspace=ws)
    torch.cuda.synchronize()
    assert out["status_code"] == flce.FLCE_OK
    ctrl = ws[:32].view(torch.int32).cpu().numpy()
    n_lab = int((t != I.IGNORE_INDEX).sum())
    assert int(ctrl[0]) == n_lab
    assert int(ctrl[N_CHUNKS_WORD]) == chunks == -(-n_lab // R)
    g = {k: (v.float().cpu().numpy() if v.dtype in (torch.bfloat16, torch.float16) else v.cpu().numpy())
         for k, v in out.items() if torch.is_tensor(v) and k != "workspace"}
    g["dW"] = dW.cpu().numpy()
    compare_full(g, run_oracle(inp, sp), inp, sp)
