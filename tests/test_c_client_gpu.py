"""The C ABI used from plain C (tests/c/flce_c_client.c): no PyTorch on the call path. The
test builds the client with nvcc against include/flce.h and the in-tree libflce.so, feeds
it a seeded problem through a file, and checks its outputs against the float64 oracle."""

import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import inputs as I
from parity_util import TOL, pred_ok, rel_fro, run_oracle

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "linear_cross_entropy_logits_gb300")


@pytest.fixture(scope="module")
def client(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    exe = str(tmp_path_factory.mktemp("c") / "flce_c_client")
    subprocess.run([B.nvcc(), "-O2", "-x", "c", os.path.join(ROOT, "tests", "c", "flce_c_client.c"),
                    "-o", exe, "-I", os.path.join(ROOT, "include"), "-L", PKG, "-lflce", "-lcudart",
                    "-Xlinker", "-rpath=" + PKG], check=True)
    return exe


def test_c_client_matches_oracle(client, tmp_path):
    sp = I.spec("llama8b", BT=600, H=192, V=3000, seq_len=300, w_std=0.2, labelled_fraction=0.8, z=1e-3)
    inp = I.generate(sp, seed=51)
    BT, H, V = sp["BT"], sp["H"], sp["V"]
    src = tmp_path / "in.bin"
    with open(src, "wb") as f:
        np.array([BT, H, V], dtype=np.int64).tofile(f)
        np.array([sp["z"]], dtype=np.float32).tofile(f)
        np.array([0], dtype=np.int64).tofile(f)  # FLCE_MEAN
        inp["X"].view(torch.int16).numpy().tofile(f)
        inp["W"].view(torch.int16).numpy().tofile(f)
        inp["targets"].numpy().astype(np.int64).tofile(f)
    out = tmp_path / "out.bin"
    r = subprocess.run([client, str(src), str(out)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    raw = open(out, "rb").read()
    off = 0

    def take(dtype, n):
        nonlocal off
        a = np.frombuffer(raw, dtype=dtype, count=n, offset=off)
        off += a.nbytes
        return a
    status = int(take(np.int32, 1)[0])
    loss = float(take(np.float32, 1)[0])
    lse = take(np.float32, BT)
    pred = take(np.int64, BT)
    dX = torch.from_numpy(take(np.int16, BT * H).copy()).view(torch.bfloat16).float().numpy().reshape(BT, H)
    dW = take(np.float32, V * H).reshape(V, H)
    assert status == 0
    o = run_oracle(inp, sp)
    tol = TOL["bf16"]
    assert abs(loss - o["loss"]) <= tol["loss"] * abs(o["loss"])
    m = o["mask"]
    assert np.all(lse[~m] == 0) and np.all(pred[~m] == -1)
    assert np.max(np.abs(lse[m] - o["lse_tok"][m]) / np.abs(o["lse_tok"][m])) <= tol["loss"]
    ok, _ = pred_ok(pred, o["pred_tok"], I.to_numpy_exact(inp["X"]), I.to_numpy_exact(inp["W"]), None,
                    np.arange(BT), m)
    assert ok
    assert rel_fro(dX, o["dX"]) <= tol["grad"] and rel_fro(dW, o["dW"]) <= tol["grad"]
