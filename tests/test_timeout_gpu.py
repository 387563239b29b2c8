"""Bounded pipeline waits (GPU). With FLCE_FLAG_DEBUG_STALL the tensor-core forward GEMM
leaves one pipeline stage of each CTA unfilled — a barrier that nothing completes — so its
waits run out after wait_timeout_ms. The call must report FLCE_ERR_TIMEOUT (no trap, no
hang), and the context must stay usable: the next normal call gives the same result as a
normal call before it."""

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


@pytest.mark.parametrize("H", [256, 4096])  # 256 x 256 and 256 x 512 forward tiles
def test_stalled_pipeline_reports_timeout_and_context_survives(H):
    sp = I.spec("llama1b", BT=512, H=H, V=4000, w_std=3.2 / H ** 0.5, ignore="random", n_ignored=64)
    inp = I.generate(sp, seed=30)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}

    def call(**kw):
        return flce.fwd_bwd(d["X"], d["W"], d["targets"], None, reduction="mean", **kw)

    before = call()
    assert before["status_code"] == flce.FLCE_OK
    stalled = call(flags=flce.FLAG_DEBUG_STALL, wait_timeout_ms=200)
    assert stalled["status_code"] == flce.FLCE_ERR_TIMEOUT
    after = call()
    assert after["status_code"] == flce.FLCE_OK
    for k in ("loss", "lse", "pred", "dX", "dW"):
        assert torch.equal(before[k], after[k]), k


def test_stalled_merged_backward_reports_timeout_and_context_survives():
    """The same for the merged dX + dW launch (a 2304-row chunk takes it): a stage of its
    first work item is armed but never filled, every role of both CTAs leaves the work
    queue through its bounded waits, and the next call is normal."""
    sp = I.spec("llama1b", BT=2304, H=256, V=4000, w_std=0.2, ignore="random", n_ignored=100)
    inp = I.generate(sp, seed=31)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    assert flce.chunk_rows(sp["BT"], sp["H"], sp["V"], torch.bfloat16,
                           flce.workspace_size(sp["BT"], sp["H"], sp["V"], torch.bfloat16, 0)) >= 2048

    def call(**kw):
        return flce.fwd_bwd(d["X"], d["W"], d["targets"], None, reduction="mean", **kw)

    before = call()
    assert before["status_code"] == flce.FLCE_OK
    stalled = call(flags=flce.FLAG_DEBUG_STALL_BWD, wait_timeout_ms=200)
    assert stalled["status_code"] == flce.FLCE_ERR_TIMEOUT
    after = call()
    assert after["status_code"] == flce.FLCE_OK
    for k in ("loss", "lse", "pred", "dX", "dW"):
        assert torch.equal(before[k], after[k]), k
