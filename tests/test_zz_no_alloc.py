"""GPU test of flce_fwd_bwd_noalloc, the entry point for callers that cannot allocate
device memory (a framework that owns all device memory through its own pool, code that
must not allocate after start-up, a foreign-function layer that forwards only the op's
inputs and outputs). It runs the same fused forward+backward out of a fixed scratch array
compiled into the library instead of a caller workspace.

The file is named so that pytest collects it last. It passes run alone in a fresh process
and after the other tests: two calls in a row (different problems, sharing the one
scratch array) must each match flce_fwd_bwd on the same inputs, within the tolerances of
the parity tests; once a first call has set the device up, a call leaves the device's
free memory unchanged; a problem too large for the scratch is rejected before any launch.
"""

import ctypes

import numpy as np
import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import flce
from linear_cross_entropy_logits_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    return flce.load()


def _rel_fro(a, b):
    a = a.double()
    b = b.double()
    return float((a - b).norm() / max(float(b.norm()), 1e-30))


def _noalloc_call(lib, d, sp, dW):
    """Fill flce_args with the inputs and freshly allocated outputs (the caller's own
    buffers) and no workspace; call the scratch-free entry point."""
    BT, H, V = sp["BT"], sp["H"], sp["V"]
    nl = BT if sp["reduction"] == "none" else 1
    dev = d["X"].device
    o = {"loss": torch.empty(nl, device=dev), "z_loss": torch.empty(nl, device=dev),
         "acc": torch.empty(nl, device=dev), "lse": torch.empty(BT, device=dev),
         "pred": torch.empty(BT, dtype=torch.int64, device=dev),
         "n_labelled": torch.empty(1, dtype=torch.int32, device=dev),
         "status": torch.zeros(1, dtype=torch.int32, device=dev),
         "dX": torch.empty_like(d["X"]), "dW": dW,
         "dbias": torch.zeros(V, device=dev) if d["bias"] is not None else None}
    a = flce.FlceArgs()
    a.BT, a.H, a.V = BT, H, V
    a.in_dtype = flce.DTYPES[d["X"].dtype]
    a.reduction = flce.REDUCTIONS[sp["reduction"]]
    a.X, a.W = d["X"].data_ptr(), d["W"].data_ptr()
    a.bias = d["bias"].data_ptr() if d["bias"] is not None else None
    a.targets = d["targets"].data_ptr()
    a.ignore_index = I.IGNORE_INDEX
    a.z_loss_scale = sp.get("z", 0.0)
    a.grad_out = d["grad_out"].data_ptr() if (d["grad_out"] is not None and sp["reduction"] == "none") else None
    a.want_dX, a.want_dW, a.dW_dtype = 1, 1, 0
    for k in ("loss", "z_loss", "acc", "lse", "pred", "n_labelled", "status"):
        setattr(a, k, o[k].data_ptr())
    a.dX, a.dW = o["dX"].data_ptr(), o["dW"].data_ptr()
    a.dbias = o["dbias"].data_ptr() if o["dbias"] is not None else None
    a.workspace, a.workspace_bytes, a.profile = None, 0, None
    s = torch.cuda.current_stream()
    rc = lib.flce_fwd_bwd_noalloc(ctypes.byref(a), ctypes.c_void_p(s.cuda_stream))
    assert rc == flce.FLCE_OK, flce.status_string(rc)
    st = lib.flce_get_status(ctypes.c_void_p(o["status"].data_ptr()), None, ctypes.c_void_p(s.cuda_stream))
    assert st == flce.FLCE_OK, flce.status_string(st)
    return o


PROBLEMS = [
    # a 128-row chunk of this vocabulary takes ~16 MB, so the 128 MiB scratch holds 1024
    # rows and the 1236 labelled rows run in two chunks
    I.spec("frozen_head", BT=1536, H=320, V=60000, w_std=0.1, bias_std=0.2, n_ignored=300,
           reduction="mean", grad_out=None, want_dW=True, z=1e-3),
    I.spec("llama8b", BT=1024, H=256, V=8000, w_std=0.15, labelled_fraction=0.5, z=1e-4),
]


def test_noalloc_matches_fwd_bwd_on_two_calls(lib):
    for i, sp in enumerate(PROBLEMS):
        inp = I.generate(sp, seed=20 + i)
        d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
        ref = flce.fwd_bwd(d["X"], d["W"], d["targets"], d["bias"], reduction=sp["reduction"],
                           z_loss_scale=sp.get("z", 0.0))
        assert ref["status_code"] == flce.FLCE_OK
        dW = torch.zeros(sp["V"], sp["H"], dtype=torch.float32, device="cuda")
        got = _noalloc_call(lib, d, sp, dW)
        torch.cuda.synchronize()
        rl, gl = float(ref["loss"][0]), float(got["loss"][0])
        assert abs(gl - rl) <= 2e-3 * abs(rl)
        assert int(got["n_labelled"][0]) == int(ref["n_labelled"][0])
        assert torch.equal(got["pred"], ref["pred"])
        assert torch.allclose(got["lse"], ref["lse"], rtol=2e-3, atol=0)
        assert _rel_fro(got["dX"], ref["dX"]) <= 1e-2
        assert _rel_fro(got["dW"], ref["dW"]) <= 1e-2
        if d["bias"] is not None:
            assert _rel_fro(got["dbias"], ref["dbias"]) <= 1e-2


def test_noalloc_call_allocates_no_device_memory(lib):
    """The point of the entry point: once a first call on the device has looked up the
    scratch array's address (and loaded the kernels), a call allocates no device memory.
    The caller's buffers are allocated before the measurement; free device memory is read
    before and after a second call of the same problem."""
    sp = PROBLEMS[1]
    inp = I.generate(sp, seed=30)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    dW = torch.zeros(sp["V"], sp["H"], dtype=torch.float32, device="cuda")
    first = _noalloc_call(lib, d, sp, dW)
    torch.cuda.synchronize()
    a = flce.FlceArgs()
    # rebuild the same call with the same (already allocated) output buffers
    BT, H, V = sp["BT"], sp["H"], sp["V"]
    a.BT, a.H, a.V = BT, H, V
    a.in_dtype = flce.DTYPES[d["X"].dtype]
    a.reduction = flce.REDUCTIONS[sp["reduction"]]
    a.X, a.W, a.bias = d["X"].data_ptr(), d["W"].data_ptr(), None
    a.targets = d["targets"].data_ptr()
    a.ignore_index = I.IGNORE_INDEX
    a.z_loss_scale = sp.get("z", 0.0)
    a.grad_out = None
    a.want_dX, a.want_dW, a.dW_dtype = 1, 1, 0
    for k in ("loss", "z_loss", "acc", "lse", "pred", "n_labelled", "status"):
        setattr(a, k, first[k].data_ptr())
    a.dX, a.dW, a.dbias = first["dX"].data_ptr(), dW.data_ptr(), None
    a.workspace, a.workspace_bytes, a.profile = None, 0, None
    loss1 = float(first["loss"][0])
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    s = torch.cuda.current_stream()
    rc = lib.flce_fwd_bwd_noalloc(ctypes.byref(a), ctypes.c_void_p(s.cuda_stream))
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert rc == flce.FLCE_OK, flce.status_string(rc)
    assert free1 == free0, f"device memory changed by {free0 - free1} bytes"
    assert float(first["loss"][0]) == loss1  # same inputs, same result


def test_noalloc_rejects_problems_beyond_the_scratch(lib):
    # one 128-row chunk of a 600k vocabulary needs ~150 MB of slab alone
    big = np.zeros(1, dtype=np.uint8)  # any non-null host address; nothing is dereferenced
    a = flce.FlceArgs()
    a.BT, a.H, a.V = 256, 64, 600_000
    a.in_dtype, a.reduction = 1, 0
    a.X = a.W = a.targets = a.loss = big.ctypes.data
    a.want_dX = a.want_dW = 0
    a.workspace, a.workspace_bytes, a.profile = None, 0, None
    assert lib.flce_fwd_bwd_noalloc(ctypes.byref(a), None) == flce.FLCE_ERR_SCRATCH_LIMIT
    a.V = 1000
    a.workspace = big.ctypes.data
    assert lib.flce_fwd_bwd_noalloc(ctypes.byref(a), None) == flce.FLCE_ERR_INVALID_ARG
