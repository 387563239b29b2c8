"""Transient memory of one call stays flat in BT (the memory concern of "feat(flce): expose
direct chunk-size control via LIGER_FLCE_CHUNK_SIZE", Summary and Details table: the
logits slab grew with BT there). The library allocates nothing: with every buffer
supplied by the caller, torch's allocator sees no allocation during the call, and the
workspace for a fixed budget differs between BT values only by 16 bytes per row."""

import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import flce
from linear_cross_entropy_logits_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    flce.load()


def test_transient_flat_in_BT():
    H, V = 1024, 32000
    budget = 256 << 20
    ws_sizes = {}
    for BT in (8192, 16384, 32768):
        sp = I.spec("llama1b", BT=BT, H=H, V=V, w_std=0.05)
        inp = I.generate(sp, seed=50)
        dev = torch.device("cuda")
        X, W, t = inp["X"].to(dev), inp["W"].to(dev), inp["targets"].to(dev)
        ws_bytes = flce.workspace_size(BT, H, V, torch.bfloat16, budget)
        assert 0 < ws_bytes <= budget
        ws_sizes[BT] = ws_bytes
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        outs = {"loss": torch.empty(1, device=dev), "z_loss": torch.empty(1, device=dev),
                "acc": torch.empty(1, device=dev), "lse": torch.empty(BT, device=dev),
                "pred": torch.empty(BT, dtype=torch.int64, device=dev),
                "n_labelled": torch.empty(1, dtype=torch.int32, device=dev),
                "status": torch.zeros(1, dtype=torch.int32, device=dev),
                "dX": torch.empty_like(X)}
        dW = torch.zeros(V, H, device=dev)
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        o = flce.fwd_bwd(X, W, t, None, dW=dW, workspace=ws, outputs=outs, check=False)
        torch.cuda.synchronize()
        assert torch.cuda.max_memory_allocated() - base == 0
        st = flce.load().flce_get_status(outs["status"].data_ptr(), None, None)
        assert st == flce.FLCE_OK
        del X, W, t, ws, outs, dW, o
        torch.cuda.empty_cache()
    rows = {BT: flce.chunk_rows(BT, H, V, torch.bfloat16, s) for BT, s in ws_sizes.items()}
    assert len(set(rows.values())) == 1
    for a, b in ((8192, 16384), (16384, 32768)):
        assert abs((ws_sizes[b] - ws_sizes[a]) - 16 * (b - a)) <= 4 * 256
