"""Host-side checks of the C-ABI library: it builds, loads without a GPU, exports every
symbol include/flce.h declares, its struct layout matches the binding, the workspace
planner keeps the transient flat in BT, and invalid arguments are rejected on the host
before any CUDA call."""

import ctypes
import os
import re
import subprocess
import sys
import tempfile

import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import flce

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "flce.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return flce.load()


def _declared():
    txt = open(HEADER).read()
    return re.findall(r"FLCE_API\s+[\w\s\*]+?\b(flce_\w+)\s*\(", txt)


def test_header_declares_the_binding_symbols():
    assert sorted(_declared()) == sorted(flce.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", flce.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (flce_\w+)", out))
    for name in _declared():
        assert name in exported, name
        assert hasattr(lib, name)
    assert lib.flce_abi_version() == 2


@pytest.mark.parametrize("cls,cname", [(flce.FlceArgs, "flce_args"), (flce.FlceJsdArgs, "flce_jsd_args")])
def test_struct_layout_matches_c(lib, cls, cname):
    fields = [f for f, _ in cls._fields_]
    src = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void){",
           f'printf("%zu\\n", sizeof({cname}));']
    src += [f'printf("%zu\\n", offsetof({cname}, {f}));' for f in fields]
    src.append("return 0;}")
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write("\n".join(src))
        subprocess.run(["gcc", "-std=c99", "-o", exe, c], check=True)
        vals = [int(x) for x in subprocess.run([exe], capture_output=True, text=True,
                                               check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(cls)
    for f, off in zip(fields, vals[1:]):
        assert getattr(cls, f).offset == off, f


@pytest.mark.parametrize("H,V,dt", [(4096, 128256, torch.bfloat16), (5376, 262144, torch.bfloat16),
                                    (2048, 128256, torch.bfloat16), (64, 1000, torch.float32)])
def test_workspace_flat_in_BT(lib, H, V, dt):
    """With a fixed budget the workspace differs between BT values only by the 16 bytes
    per row of the compaction index and per-row loss terms."""
    budget = int(1.5 * 2 ** 30)
    sizes = {BT: flce.workspace_size(BT, H, V, dt, budget) for BT in (8192, 16384, 32768)}
    rows = {BT: flce.chunk_rows(BT, H, V, dt, sizes[BT]) for BT in sizes}
    for BT, s in sizes.items():
        assert 0 < s <= budget
        assert rows[BT] % 128 == 0 and rows[BT] >= 128
    if len(set(rows.values())) == 1:
        d = sizes[32768] - sizes[16384]
        assert abs(d - 16 * 16384) <= 4 * 256


def test_large_vocab_workspace_fits_the_cap(lib):
    cap = int(1.5 * 2 ** 30)
    s = flce.workspace_size(32768, 5376, 262144, torch.bfloat16, cap)
    assert 0 < s <= cap
    assert flce.chunk_rows(32768, 5376, 262144, torch.bfloat16, s) >= 2048


def test_workspace_too_small(lib):
    assert flce.workspace_size(1024, 4096, 128256, torch.bfloat16, 1 << 20) == 0
    assert flce.chunk_rows(1024, 4096, 128256, torch.bfloat16, 1 << 20) == 0


def _args(**kw):
    a = flce.FlceArgs()
    a.BT, a.H, a.V = 16, 64, 100
    a.in_dtype, a.reduction = 1, 0
    a.X, a.W, a.targets, a.loss = 0x1000, 0x2000, 0x3000, 0x4000
    a.workspace, a.workspace_bytes = 0x100000, 1 << 30
    a.want_dX, a.dX = 0, None
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(X=None), flce.FLCE_ERR_INVALID_ARG),
    (dict(W=None), flce.FLCE_ERR_INVALID_ARG),
    (dict(targets=None), flce.FLCE_ERR_INVALID_ARG),
    (dict(loss=None), flce.FLCE_ERR_INVALID_ARG),
    (dict(workspace=None), flce.FLCE_ERR_INVALID_ARG),
    (dict(BT=0), flce.FLCE_ERR_INVALID_ARG),
    (dict(H=-1), flce.FLCE_ERR_INVALID_ARG),
    (dict(in_dtype=7), flce.FLCE_ERR_INVALID_ARG),
    (dict(reduction=3), flce.FLCE_ERR_INVALID_ARG),
    (dict(z_loss_scale=-1.0), flce.FLCE_ERR_INVALID_ARG),
    (dict(z_loss_scale=float("nan")), flce.FLCE_ERR_INVALID_ARG),
    (dict(want_dX=1, dX=None), flce.FLCE_ERR_INVALID_ARG),
    (dict(want_dW=1, dW=None), flce.FLCE_ERR_INVALID_ARG),
    (dict(want_dW=1, dW=0x5000, dW_dtype=2), flce.FLCE_ERR_UNSUPPORTED),
    (dict(in_dtype=0, want_dW=1, dW=0x5000, dW_dtype=1), flce.FLCE_ERR_UNSUPPORTED),
    (dict(X=0x1008), flce.FLCE_ERR_INVALID_ARG),
    (dict(workspace=0x100010), flce.FLCE_ERR_INVALID_ARG),
    (dict(workspace_bytes=1024), flce.FLCE_ERR_WORKSPACE),
])
def test_host_validation_rejects_before_any_cuda_call(lib, kw, code):
    a = _args(**kw)
    assert flce.raw_call(a, 0) == code


def test_null_args_pointer(lib):
    assert lib.flce_fwd_bwd(None, None) == flce.FLCE_ERR_INVALID_ARG


def test_torch_custom_op_registers():
    """The torch integration imports without a GPU and registers its custom op."""
    from linear_cross_entropy_logits_gb300 import torch_ops
    assert hasattr(torch.ops.flce_gb300, "fused_linear_cross_entropy")
    assert callable(torch_ops.fused_linear_cross_entropy)


def _jsd_args(**kw):
    a = flce.FlceJsdArgs()
    a.BT, a.Hs, a.Ht, a.V = 16, 64, 32, 100
    a.in_dtype, a.reduction = 1, 0
    a.Xs, a.Ws, a.Xt, a.Wt, a.loss = 0x1000, 0x2000, 0x3000, 0x4000, 0x5000
    a.beta, a.temperature = 0.5, 1.0
    a.workspace, a.workspace_bytes = 0x100000, 1 << 30
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(Xt=None), flce.FLCE_ERR_INVALID_ARG),
    (dict(beta=1.5), flce.FLCE_ERR_INVALID_ARG),
    (dict(beta=-0.1), flce.FLCE_ERR_INVALID_ARG),
    (dict(temperature=0.0), flce.FLCE_ERR_INVALID_ARG),
    (dict(Ht=0), flce.FLCE_ERR_INVALID_ARG),
    (dict(want_dX=1, dX=None), flce.FLCE_ERR_INVALID_ARG),
    (dict(want_dW=1, dW=0x6000, dW_dtype=2), flce.FLCE_ERR_UNSUPPORTED),
    (dict(workspace_bytes=2048), flce.FLCE_ERR_WORKSPACE),
])
def test_jsd_host_validation(lib, kw, code):
    a = _jsd_args(**kw)
    assert lib.flce_fused_linear_jsd(ctypes.byref(a), None) == code


def test_jsd_workspace_flat_in_BT(lib):
    s = {BT: flce.jsd_workspace_size(BT, 2048, 4096, 128256, torch.bfloat16, int(1.5 * 2 ** 30))
         for BT in (8192, 16384)}
    assert 0 < s[8192] <= int(1.5 * 2 ** 30)
    assert abs((s[16384] - s[8192]) - 16 * 8192) <= 4 * 256


def test_plan_describe(lib):
    """The host-side plan text: chunk rows and tiles as the planner computes them, snprintf
    length semantics (the NULL / 0 query gives the full length, a short buffer truncates),
    and -1 for an invalid call."""
    BT, H, V = 8192, 4096, 128256
    wb = flce.workspace_size(BT, H, V, torch.bfloat16, 0)
    R = flce.chunk_rows(BT, H, V, torch.bfloat16, wb)
    txt = flce.describe_plan(BT, H, V, torch.bfloat16, wb)
    assert f"chunk rows R={R}," in txt and "cdiv(BT,R)=1 " in txt
    assert "vocabulary tiles: 501 x 256 columns" in txt
    assert f"forward {((R + 255) // 256) * 251} tiles of 256x512" in txt  # H >= 4096: wide tile
    t2 = flce.describe_plan(BT, 2048, V, torch.bfloat16)
    assert "forward " in t2 and "tiles of 256x256;" in t2
    assert "dW 4008 tiles of 256x512" in txt and "dX and dW in one launch" in txt
    # chunks under 2048 rows: dW on 256x256 tiles, two launches
    small_ws = flce.workspace_size(BT, H, V, torch.bfloat16, 1 << 29)
    t3 = flce.describe_plan(BT, H, V, torch.bfloat16, small_ws)
    assert flce.chunk_rows(BT, H, V, torch.bfloat16, small_ws) < 2048
    assert "dX and dW in two launches" in t3 and "tiles of 256x256; dX and dW" in t3
    assert "workspace slab   at" in txt and str(R * 128256 * 2) in txt
    n = lib.flce_plan_describe(BT, H, V, 1, wb, None, 0)
    assert n == len(txt.encode())
    buf = ctypes.create_string_buffer(16)
    assert lib.flce_plan_describe(BT, H, V, 1, wb, buf, 16) == n
    assert buf.value.decode() == txt[:15]
    # fp32 and a workspace that forces 128-row chunks
    small = flce.workspace_size(128, 64, 1000, torch.float32, 0) + 16 * 1000 + 4096
    t32 = flce.describe_plan(1000, 64, 1000, torch.float32, small)
    assert "chunk rows R=128," in t32 and "cdiv(BT,R)=8 " in t32 and "SIMT fp32-FMA" in t32
    assert lib.flce_plan_describe(0, H, V, 1, wb, None, 0) == -1
    assert lib.flce_plan_describe(BT, H, V, 7, wb, None, 0) == -1
    assert lib.flce_plan_describe(BT, H, V, 1, 1024, None, 0) == -1


@pytest.mark.parametrize("kw,code", [
    (dict(), flce.FLCE_ERR_INVALID_ARG),                    # a caller workspace is given
    (dict(workspace=None), flce.FLCE_ERR_INVALID_ARG),      # ... or its size
    (dict(workspace=None, workspace_bytes=0, BT=0), flce.FLCE_ERR_INVALID_ARG),
    (dict(workspace=None, workspace_bytes=0, in_dtype=7), flce.FLCE_ERR_INVALID_ARG),
    (dict(workspace=None, workspace_bytes=0, H=4096, V=10_000_000), flce.FLCE_ERR_SCRATCH_LIMIT),
])
def test_noalloc_host_rejections(lib, kw, code):
    """The scratch-only entry point refuses a caller workspace and problems whose 128-row
    chunk exceeds its fixed scratch, on the host, before any CUDA call."""
    a = _args(**kw)
    assert lib.flce_fwd_bwd_noalloc(ctypes.byref(a), None) == code
    assert lib.flce_fwd_bwd_noalloc(None, None) == flce.FLCE_ERR_INVALID_ARG


@pytest.mark.gpu
def test_trace_prints_the_plan_of_each_call(tmp_path):
    """FLCE_TRACE=1: a real call prints its plan and path to stderr (a child process, so the
    switch is read fresh); without it nothing is printed."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    code = (
        "import torch\n"
        "from linear_cross_entropy_logits_gb300 import flce\n"
        "flce.load()\n"
        "X = torch.randn(256, 128, device='cuda').bfloat16()\n"
        "W = (0.05 * torch.randn(1000, 128, device='cuda')).bfloat16()\n"
        "t = torch.randint(0, 1000, (256,), device='cuda')\n"
        "o = flce.fwd_bwd(X, W, t, None)\n"
        "torch.cuda.synchronize()\n"
        "assert o['status_code'] == flce.FLCE_OK\n")
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    on = subprocess.run([sys.executable, "-c", code], env=dict(env, FLCE_TRACE="1"), capture_output=True,
                        text=True, timeout=600)
    assert on.returncode == 0, on.stderr
    assert "flce plan: BT=256 H=128 V=1000 dtype=bf16" in on.stderr
    assert "GEMMs on tcgen05; gradient form row-reference" in on.stderr
    off = subprocess.run([sys.executable, "-c", code], env=dict(env, FLCE_TRACE="0"), capture_output=True,
                         text=True, timeout=600)
    assert off.returncode == 0, off.stderr
    assert "flce plan:" not in off.stderr
