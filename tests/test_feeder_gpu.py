"""The double-buffered host feeder: each step sees exactly its own inputs although the copy
of step k+1 overlaps step k (three distinct input sets, losses equal to direct calls)."""

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


def test_feeder_steps_see_their_own_inputs():
    from linear_cross_entropy_logits_gb300.feeder import DoubleBufferedInputs
    sp = I.spec("llama8b", BT=1024, H=256, V=4000, seq_len=256)
    W = I.generate(sp, seed=0)["W"].cuda()
    hosts = []
    for seed in (1, 2, 3, 4, 5):
        inp = I.generate(sp, seed=seed)
        hosts.append({"X": inp["X"].pin_memory(), "t": inp["targets"].pin_memory()})
    direct = []
    for h in hosts:
        out = flce.fwd_bwd(h["X"].cuda(), W, h["t"].cuda(), reduction="sum", want_dW=False)
        direct.append(float(out["loss"][0]))
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream(dev)
    feed = DoubleBufferedInputs(hosts[0], dev)
    outs = {"loss": torch.empty(1, device=dev)}
    got = [torch.empty(1).pin_memory() for _ in hosts]
    slot = feed.stage(hosts[0])
    for k in range(len(hosts)):
        nxt = feed.stage(hosts[k + 1]) if k + 1 < len(hosts) else None
        dv = feed.acquire(slot, stream)
        flce.fwd_bwd(dv["X"], W, dv["t"], reduction="sum", want_dW=False, outputs=outs, check=False)
        feed.release(slot, stream)
        got[k].copy_(outs["loss"], non_blocking=True)
        slot = nxt
    torch.cuda.synchronize()
    assert [float(g[0]) for g in got] == direct
