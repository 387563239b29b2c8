"""flce_fwd_bwd and the fused linear JSD op inside a CUDA graph: a call enqueues only
kernels and memsets on the caller's stream (no host synchronisation, no allocation when the
caller passes every buffer), so it can be captured once and replayed. Replays give bit-identical outputs to eager calls,
including a replay after the captured inputs were overwritten in place."""

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


def _buffers(sp, dev):
    BT, H, V = sp["BT"], sp["H"], sp["V"]
    ws = torch.empty(flce.workspace_size(BT, H, V, torch.bfloat16, 0), dtype=torch.uint8, device=dev)
    outs = {"loss": torch.empty(1, device=dev), "z_loss": torch.empty(1, device=dev),
            "acc": torch.empty(1, device=dev), "lse": torch.empty(BT, device=dev),
            "pred": torch.empty(BT, dtype=torch.int64, device=dev),
            "n_labelled": torch.empty(1, dtype=torch.int32, device=dev),
            "status": torch.zeros(1, dtype=torch.int32, device=dev),
            "dX": torch.empty(BT, H, dtype=torch.bfloat16, device=dev)}
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    return ws, outs, dW


@pytest.mark.parametrize("flags", [0, "overwrite"])
def test_capture_and_replay(flags):
    sp = I.spec("llama8b", BT=2048, H=256, V=5000, seq_len=512, w_std=0.1, labelled_fraction=0.75,
                z=1e-3)
    dev = torch.device("cuda")
    a = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in I.generate(sp, seed=41).items()}
    b = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in I.generate(sp, seed=42).items()}
    fl = flce.FLAG_DW_OVERWRITE if flags == "overwrite" else 0
    X = a["X"].clone()
    t = a["targets"].clone()
    ws, outs, dW = _buffers(sp, dev)

    def call(Xc, tc, o, w, d):
        if not fl:
            d.zero_()
        flce.fwd_bwd(Xc, a["W"], tc, None, reduction="mean", z_loss_scale=sp["z"], dW=d, workspace=w,
                     outputs=o, flags=fl, check=False)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(X, t, outs, ws, dW)  # warm-up outside the capture (planner and launch caches)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(X, t, outs, ws, dW)

    for inp in (a, b):
        X.copy_(inp["X"])
        t.copy_(inp["targets"])
        g.replay()
        torch.cuda.synchronize()
        ws2, ref, dW2 = _buffers(sp, dev)
        call(inp["X"], inp["targets"], ref, ws2, dW2)
        torch.cuda.synchronize()
        for k in ("loss", "z_loss", "acc", "lse", "pred", "n_labelled", "dX"):
            assert torch.equal(outs[k], ref[k]), k
        assert torch.equal(dW, dW2)
        assert int(outs["status"][0]) == 0


def test_distillation_capture_and_replay():
    """The fused linear JSD op (beta 0.5, so its elementwise kernel keeps the log ratio in
    dynamic shared memory) captured once and replayed: bit-identical to eager calls."""
    sp = dict(I.DISTILL, BT=640, Hs=256, Ht=512, V=3000, w_std=0.1, ignore="random", n_ignored=40)
    dev = torch.device("cuda")
    a = {k: v.to(dev) for k, v in I.generate_distill(sp, seed=43).items()}
    b = {k: v.to(dev) for k, v in I.generate_distill(sp, seed=44).items()}
    BT, Hs, Ht, V = sp["BT"], sp["Hs"], sp["Ht"], sp["V"]
    Xs, Xt, lab = a["Xs"].clone(), a["Xt"].clone(), a["labels"].clone()

    def bufs():
        ws = torch.empty(flce.jsd_workspace_size(BT, Hs, Ht, V, torch.bfloat16, 0), dtype=torch.uint8,
                         device=dev)
        o = {"loss": torch.empty(1, device=dev), "n_labelled": torch.empty(1, dtype=torch.int32, device=dev),
             "status": torch.zeros(1, dtype=torch.int32, device=dev),
             "dX": torch.empty(BT, Hs, dtype=torch.bfloat16, device=dev)}
        return ws, o, torch.empty(V, Hs, dtype=torch.float32, device=dev)

    def call(xs, xt, lb, o, w, d):
        d.zero_()
        flce.fused_linear_jsd(xs, a["Ws"], xt, a["Wt"], lb, beta=0.5, temperature=1.0, reduction="mean",
                              dW=d, workspace=w, outputs=o, check=False)

    ws, outs, dW = bufs()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(Xs, Xt, lab, outs, ws, dW)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(Xs, Xt, lab, outs, ws, dW)
    for inp in (a, b):
        Xs.copy_(inp["Xs"])
        Xt.copy_(inp["Xt"])
        lab.copy_(inp["labels"])
        g.replay()
        torch.cuda.synchronize()
        ws2, ref, dW2 = bufs()
        call(inp["Xs"], inp["Xt"], inp["labels"], ref, ws2, dW2)
        torch.cuda.synchronize()
        for k in ("loss", "n_labelled", "dX"):
            assert torch.equal(outs[k], ref[k]), k
        assert torch.equal(dW, dW2)
        assert int(outs["status"][0]) == 0
