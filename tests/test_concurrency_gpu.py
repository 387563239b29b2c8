"""Calls from several host threads, each on its own CUDA stream with its own workspace and
outputs, run concurrently on the GPU and give bit-for-bit the results of the same calls made
one after another. The library keeps no per-call state outside the caller's buffers (its only
globals are per-device launch caches), so calls on independent streams may overlap."""

import threading

import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import flce
from linear_cross_entropy_logits_gb300 import inputs as I
from parity_util import compare_full, run_oracle

pytestmark = pytest.mark.gpu

OUT_KEYS = ("loss", "z_loss", "acc", "lse", "pred", "dX", "dW")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    flce.load()


def _problem(seed, path):
    sp = I.spec("llama8b", BT=1536, H=384, V=9000, w_std=0.1, labelled_fraction=0.75, z=1e-3)
    if path == "simt":
        sp = I.spec("llama8b", BT=384, H=96, V=2100, w_std=0.2, labelled_fraction=0.75, z=1e-3,
                    seq_len=128)
    inp = I.generate(sp, seed=seed)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    BT, H, V = sp["BT"], sp["H"], sp["V"]
    dev = torch.device("cuda")
    o = {"loss": torch.empty(1, device=dev), "z_loss": torch.empty(1, device=dev),
         "acc": torch.empty(1, device=dev), "lse": torch.empty(BT, device=dev),
         "pred": torch.empty(BT, dtype=torch.int64, device=dev),
         "n_labelled": torch.empty(1, dtype=torch.int32, device=dev),
         "status": torch.zeros(1, dtype=torch.int32, device=dev),
         "dX": torch.empty_like(d["X"])}
    dW = torch.zeros(V, H, dtype=torch.float32, device=dev)
    # a workspace of two 128-row chunks, so each call runs several chunks
    wb = flce.workspace_size(256, H, V, torch.bfloat16, 0) + 16 * BT + 4096
    ws = torch.empty(wb, dtype=torch.uint8, device=dev)
    return sp, inp, d, o, dW, ws


def _call(p, stream, flags):
    sp, _, d, o, dW, ws = p
    with torch.cuda.stream(stream):  # the zero fill is ordered before the call on `stream`
        dW.zero_()
        flce.fwd_bwd(d["X"], d["W"], d["targets"], d["bias"], reduction=sp["reduction"],
                     z_loss_scale=sp["z"], want_dW=True, dW=dW, workspace=ws, outputs=o,
                     flags=flags, check=False, stream=stream)


def _snapshot(p):
    _, _, _, o, dW, _ = p
    r = {k: o[k].detach().cpu().clone() for k in OUT_KEYS if k != "dW"}
    r["dW"] = dW.detach().cpu().clone()
    return r


@pytest.mark.parametrize("path", ["tc", "simt"])
def test_concurrent_streams_match_serial_calls(path):
    flags = flce.FLAG_FORCE_SIMT if path == "simt" else 0
    probs = [_problem(seed, path) for seed in range(4)]
    # serial: one call after another on the current stream
    serial = []
    for p in probs:
        _call(p, torch.cuda.current_stream(), flags)
        torch.cuda.synchronize()
        serial.append(_snapshot(p))
    # clear every output, then the same calls from four threads on four streams
    for p in probs:
        for k in OUT_KEYS:
            if k != "dW":
                p[3][k].fill_(-7)
        p[4].fill_(-7.0)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in probs]
    start = threading.Barrier(len(probs))
    errors = []

    def worker(i):
        try:
            start.wait()
            for _ in range(3):  # repeated calls keep the streams busy at the same time
                _call(probs[i], streams[i], flags)
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(probs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i, p in enumerate(probs):
        assert int(p[3]["status"][0]) == 0
        got = _snapshot(p)
        for k in OUT_KEYS:
            assert torch.equal(got[k], serial[i][k]), (i, k)
    # and the concurrent results are the oracle's
    sp, inp = probs[0][0], probs[0][1]
    g = {k: (v.float().numpy() if v.dtype in (torch.bfloat16, torch.float16) else v.numpy())
         for k, v in _snapshot(probs[0]).items()}
    g["n_labelled"] = probs[0][3]["n_labelled"].cpu().numpy()
    compare_full(g, run_oracle(inp, sp), inp, sp)
