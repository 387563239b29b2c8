"""GPU parity of the CUDA path (through the C ABI) against the float64 oracle, element by
element, at sizes the oracle finishes in seconds that span several tiles and ragged tails,
plus the method's edge cases. Both GEMM back-ends are covered: the tcgen05 tensor-core
kernels (bf16/fp16) and the SIMT fp32-FMA kernels (fp32, and bf16 when forced)."""

import numpy as np
import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import flce
from linear_cross_entropy_logits_gb300 import inputs as I
from parity_util import compare_full, rel_fro, run_gpu, run_oracle, TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()
    flce.load()


# Small problems: (name, base workload, overrides)
SMALL = [
    ("bf16_mean_ragged", "llama1b", dict(BT=300, H=192, V=3000, w_std=0.2, ignore="random",
                                          n_ignored=40)),
    ("bf16_sum_bias_z", "large_vocab", dict(BT=260, H=520, V=1300, w_std=0.1, bias_std=0.5,
                                             z=0.01, targets="uniform", ignore="random",
                                             n_ignored=31)),
    ("bf16_prompt_first", "llama8b", dict(BT=1024, H=256, V=2304, w_std=0.1,
                                          labelled_fraction=0.5)),
    ("bf16_none_frozen_bias", "frozen_head", dict(BT=400, H=128, V=5000, w_std=0.15,
                                                   bias_std=0.3, n_ignored=200)),
    ("f16_mean", "llama1b", dict(BT=256, H=320, V=2000, dtype="f16", w_std=0.1,
                                 ignore="random", n_ignored=5)),
    ("bf16_tiny_H64", "llama1b", dict(BT=130, H=64, V=1000, w_std=0.3, ignore="random",
                                      n_ignored=3)),
    # H >= 4096: the forward runs on 256 x 512 tiles (ragged last tile: 12 of 13 sub-tiles)
    ("bf16_wide_fwd_H4096", "llama1b", dict(BT=300, H=4096, V=3100, w_std=0.03, ignore="random",
                                            n_ignored=40)),
    ("f16_wide_fwd_H4096_bias", "frozen_head", dict(BT=260, H=4096, V=2000, dtype="f16", w_std=0.03,
                                                    bias_std=0.3, n_ignored=30)),
]


def _spec(base, ov):
    sp = I.spec(base, **ov)
    return sp


@pytest.mark.parametrize("name,base,ov", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("path", ["tc", "simt"])
def test_small_parity(name, base, ov, path):
    sp = _spec(base, ov)
    inp = I.generate(sp, seed=0)
    o = run_oracle(inp, sp)
    g = run_gpu(inp, sp, flags=flce.FLAG_FORCE_SIMT if path == "simt" else 0)
    assert g["status_code"] == flce.FLCE_OK
    compare_full(g, o, inp, sp)


def test_config1_tiny_fp32_full():
    """BT=128, H=64, V=1000 fp32, 13 rows ignored, mean: every output element against the
    oracle at 1e-5."""
    sp = I.spec("tiny_fp32")
    inp = I.generate(sp, seed=0)
    o = run_oracle(inp, sp)
    g = run_gpu(inp, sp)
    assert g["status_code"] == flce.FLCE_OK
    assert int(g["n_labelled"][0]) == 115
    compare_full(g, o, inp, sp)


def test_fp32_none_with_bias_and_z():
    sp = I.spec("tiny_fp32", BT=200, H=96, V=700, bias_std=0.2, reduction="none",
                grad_out="uniform", z=0.05, n_ignored=20)
    inp = I.generate(sp, seed=3)
    compare_full(run_gpu(inp, sp), run_oracle(inp, sp), inp, sp)


def _ws_for_rows(BT, H, V, dt, R):
    return flce.workspace_size(R, H, V, dt, 0) + 16 * BT + 4096


@pytest.mark.parametrize("path", ["tc", "simt"])
def test_multichunk(path):
    """A workspace that holds 128 rows forces several chunks (uneven last chunk); the
    result must match the oracle and the single-chunk result."""
    sp = I.spec("llama8b", BT=1024, H=128, V=1500, w_std=0.2, labelled_fraction=0.75,
                z=1e-3)
    inp = I.generate(sp, seed=1)
    flags = flce.FLAG_FORCE_SIMT if path == "simt" else 0
    wb = _ws_for_rows(sp["BT"], sp["H"], sp["V"], torch.bfloat16, 128)
    assert flce.chunk_rows(sp["BT"], sp["H"], sp["V"], torch.bfloat16, wb) == 128
    g1 = run_gpu(inp, sp, flags=flags, workspace_bytes=wb)
    g2 = run_gpu(inp, sp, flags=flags)
    o = run_oracle(inp, sp)
    compare_full(g1, o, inp, sp)
    compare_full(g2, o, inp, sp)
    assert rel_fro(g1["dW"], g2["dW"]) < 1e-5
    assert rel_fro(g1["dX"], g2["dX"]) < 1e-5


def test_deterministic():
    sp = I.spec("llama1b", BT=512, H=256, V=3000, w_std=0.2, ignore="random", n_ignored=50)
    inp = I.generate(sp, seed=2)
    a = run_gpu(inp, sp)
    b = run_gpu(inp, sp)
    for k in ("loss", "lse", "pred", "dX", "dW"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("path", ["tc", "simt"])
def test_nan_in_ignored_rows_does_not_leak(path):
    """A NaN stored in an ignored row reaches no output; results equal the clean run bit
    for bit (Liger-Kernel PR #1554, Tests: test_ignored_rows_do_not_enter_projection)."""
    sp = I.spec("frozen_head", BT=256, H=128, V=1200, w_std=0.2, n_ignored=100,
                reduction="sum", want_dW=True, grad_out=None)
    inp = I.generate(sp, seed=4)
    flags = flce.FLAG_FORCE_SIMT if path == "simt" else 0
    clean = run_gpu(inp, sp, flags=flags)
    ign = inp["targets"] == I.IGNORE_INDEX
    Xn = inp["X"].clone()
    Xn[ign] = float("nan")
    dirty = run_gpu(dict(inp, X=Xn), sp, flags=flags)
    for k in ("loss", "lse", "pred", "dX", "dW", "dbias", "z_loss", "acc"):
        assert np.array_equal(clean[k], dirty[k], equal_nan=False), k
    assert np.all(np.isfinite(dirty["dW"])) and np.all(np.isfinite(dirty["dX"]))


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_all_rows_ignored(reduction):
    sp = I.spec("llama1b", BT=200, H=64, V=500, ignore="all", reduction=reduction,
                bias_std=0.1)
    inp = I.generate(sp, seed=5)
    g = run_gpu(inp, sp)
    assert g["status_code"] == flce.FLCE_OK
    assert int(g["n_labelled"][0]) == 0
    assert np.all(g["loss"] == 0) and np.all(g["pred"] == -1) and np.all(g["lse"] == 0)
    assert np.all(g["dX"] == 0) and np.all(g["dW"] == 0) and np.all(g["dbias"] == 0)


def test_single_labelled_row_and_target_edges():
    sp = I.spec("llama1b", BT=150, H=72, V=777, w_std=0.3, ignore="none")
    inp = I.generate(sp, seed=6)
    t = inp["targets"]
    t[:] = I.IGNORE_INDEX
    t[77] = sp["V"] - 1
    o = run_oracle(inp, sp)
    compare_full(run_gpu(inp, sp), o, inp, sp)
    t[:] = 0
    t[1::2] = sp["V"] - 1
    compare_full(run_gpu(inp, sp), run_oracle(inp, sp), inp, sp)


def test_out_of_range_target_sets_status_and_is_ignored():
    sp = I.spec("llama1b", BT=128, H=64, V=300, w_std=0.3, ignore="random", n_ignored=4)
    inp = I.generate(sp, seed=7)
    inp["targets"][10] = sp["V"]
    inp["targets"][11] = -5
    g = run_gpu(inp, sp)
    assert g["status_code"] == flce.FLCE_ERR_TARGET_RANGE
    o = run_oracle(inp, sp)
    assert o["out_of_range"]
    compare_full(g, o, inp, sp)


def test_dW_accumulates_into_destination():
    sp = I.spec("llama1b", BT=300, H=128, V=900, w_std=0.2, ignore="random", n_ignored=30)
    inp = I.generate(sp, seed=8)
    init = torch.randn(sp["V"], sp["H"], generator=torch.Generator().manual_seed(9))
    g = run_gpu(inp, sp, dW_init=init)
    o = run_oracle(inp, sp)
    assert rel_fro(g["dW"] - init.numpy(), o["dW"]) <= TOL["bf16"]["grad"]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("path", ["tc", "simt"])
def test_same_dtype_dW_accumulation(dt, path):
    """dW and dbias accumulated in the input dtype ("Reduce FLCE weight-gradient allocation
    overhead across FP16, BF16, and FP32", support matrix: same-dtype FP16/BF16 direct
    accumulation). The tensor-core path adds G^T X, rounded to the input dtype, into dW in
    the L2 (a second rounding); the SIMT path rounds dW_init + G^T X once."""
    sp = I.spec("frozen_head", BT=300, H=136, V=2100, dtype=dt, w_std=0.15, bias_std=0.3,
                n_ignored=60, reduction="sum", grad_out=None, want_dW=True, z=1e-3)
    inp = I.generate(sp, seed=12)
    tdt = I.TORCH_DTYPES[dt]
    init = (torch.randn(sp["V"], sp["H"], generator=torch.Generator().manual_seed(13)) * 0.01).to(tdt)
    binit = (torch.randn(sp["V"], generator=torch.Generator().manual_seed(14)) * 0.01).to(tdt)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    dW = init.clone().cuda()
    db = binit.clone().cuda()
    out = flce.fwd_bwd(d["X"], d["W"], d["targets"], d["bias"], reduction="sum", z_loss_scale=sp["z"],
                       dW=dW, dbias=db, flags=flce.FLAG_FORCE_SIMT if path == "simt" else 0)
    assert out["status_code"] == flce.FLCE_OK
    o = run_oracle(inp, sp)
    got_dW = out["dW"].float().cpu().numpy() - init.float().numpy()
    got_db = out["dbias"].float().cpu().numpy() - binit.float().numpy()
    assert out["dW"].dtype == tdt and out["dbias"].dtype == tdt
    assert rel_fro(got_dW, o["dW"]) <= TOL[dt]["grad"]
    assert rel_fro(got_db, o["dbias"]) <= TOL[dt]["grad"]
    assert rel_fro(out["dX"].float().cpu().numpy(), o["dX"]) <= TOL[dt]["grad"]


def test_grad_scalar_scales_gradients():
    sp = I.spec("llama1b", BT=128, H=64, V=640, w_std=0.2, ignore="random", n_ignored=8,
                grad_scalar=0.37, z=0.02)
    inp = I.generate(sp, seed=10)
    compare_full(run_gpu(inp, sp), run_oracle(inp, sp), inp, sp)


def test_guard_bands_untouched():
    """Canary bands around every output and around the workspace stay intact (the
    stand-in for an out-of-bounds checker)."""
    sp = I.spec("frozen_head", BT=300, H=192, V=1700, w_std=0.2, n_ignored=90,
                reduction="none", want_dW=True)
    inp = I.generate(sp, seed=11)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    BT, H, V = sp["BT"], sp["H"], sp["V"]
    G = 4096
    sentinel = 0x5A

    def guarded(n, dtype):
        esz = torch.empty(0, dtype=dtype).element_size()
        raw = torch.full((n * esz + 2 * G,), sentinel, dtype=torch.uint8, device="cuda")
        return raw, raw[G:G + n * esz].view(dtype)

    bufs = {
        "loss": guarded(BT, torch.float32), "z_loss": guarded(BT, torch.float32),
        "acc": guarded(BT, torch.float32), "lse": guarded(BT, torch.float32),
        "pred": guarded(BT, torch.int64), "dX": guarded(BT * H, torch.bfloat16),
    }
    dW_raw, dW = guarded(V * H, torch.float32)
    dW.zero_()
    db_raw, db = guarded(V, torch.float32)
    db.zero_()
    wsb = flce.workspace_size(BT, H, V, torch.bfloat16, 0)
    ws_raw = torch.full((wsb + 2 * G,), sentinel, dtype=torch.uint8, device="cuda")
    ws = ws_raw[G:G + wsb]
    outs = {k: (v[1].view(BT, H) if k == "dX" else v[1]) for k, v in bufs.items()}
    o = flce.fwd_bwd(d["X"], d["W"], d["targets"], d["bias"], reduction="none",
                     grad_out=d["grad_out"], dW=dW.view(V, H), dbias=db, workspace=ws,
                     outputs=outs)
    torch.cuda.synchronize()
    assert o["status_code"] == flce.FLCE_OK
    for raw in [b[0] for b in bufs.values()] + [dW_raw, db_raw, ws_raw]:
        assert torch.all(raw[:G] == sentinel) and torch.all(raw[-G:] == sentinel)


@pytest.mark.parametrize("H", [136, 520])
def test_wide_dw_tile_ragged(H):
    """Chunks of at least 4096 rows take the 256 x 512 dW tile; H = 136 leaves the second
    256-column sub-tile wholly past the output, H = 520 a third sub-tile partly past it.
    Every output against the oracle."""
    sp = I.spec("llama1b", BT=4300, H=H, V=1300, w_std=0.2, ignore="random", n_ignored=100)
    inp = I.generate(sp, seed=21)
    assert flce.chunk_rows(sp["BT"], H, sp["V"], torch.bfloat16,
                           flce.workspace_size(sp["BT"], H, sp["V"], torch.bfloat16, 0)) >= 4096
    compare_full(run_gpu(inp, sp), run_oracle(inp, sp), inp, sp)


@pytest.mark.parametrize("path", ["tc", "simt"])
@pytest.mark.parametrize("dw_dt", ["f32", "same"])
@pytest.mark.parametrize("labelled", ["some", "none"])
def test_dw_overwrite(path, dw_dt, labelled):
    """FLCE_FLAG_DW_OVERWRITE: dW and dbias (pre-filled with NaN) receive exactly this call's
    gradient over several chunks (the first chunk stores, later ones add); with no labelled
    row they come back zero."""
    sp = I.spec("frozen_head", BT=700, H=136, V=1500, w_std=0.15, bias_std=0.3, n_ignored=70,
                reduction="sum", grad_out=None, want_dW=True, z=1e-3,
                ignore="random" if labelled == "some" else "all")
    inp = I.generate(sp, seed=23)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    adt = torch.float32 if dw_dt == "f32" else torch.bfloat16
    dW = torch.full((sp["V"], sp["H"]), float("nan"), dtype=adt, device="cuda")
    db = torch.full((sp["V"],), float("nan"), dtype=adt, device="cuda")
    budget = flce.workspace_size(128, sp["H"], sp["V"], torch.bfloat16, 0) + 16 * sp["BT"] + 4096
    flags = flce.FLAG_DW_OVERWRITE | (flce.FLAG_FORCE_SIMT if path == "simt" else 0)
    out = flce.fwd_bwd(d["X"], d["W"], d["targets"], d["bias"], reduction="sum", z_loss_scale=sp["z"],
                       dW=dW, dbias=db, budget_bytes=budget, flags=flags)
    assert out["status_code"] == flce.FLCE_OK
    o = run_oracle(inp, sp)
    gw = dW.float().cpu().numpy()
    gb = db.float().cpu().numpy()
    if labelled == "none":
        assert np.all(gw == 0) and np.all(gb == 0)
    else:
        assert np.all(np.isfinite(gw)) and np.all(np.isfinite(gb))
        assert rel_fro(gw, o["dW"]) <= TOL["bf16"]["grad"]
        assert rel_fro(gb, o["dbias"]) <= TOL["bf16"]["grad"]


def test_overwrite_row_reference_wide_tile():
    """The same flag on the row-reference, 256x512-tile dW path (no bias, >= 4096 rows)."""
    sp = I.spec("llama1b", BT=4300, H=136, V=1300, w_std=0.2, ignore="random", n_ignored=100)
    inp = I.generate(sp, seed=24)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}
    for adt in (torch.float32, torch.bfloat16):
        dW = torch.full((sp["V"], sp["H"]), float("nan"), dtype=adt, device="cuda")
        out = flce.fwd_bwd(d["X"], d["W"], d["targets"], None, dW=dW, flags=flce.FLAG_DW_OVERWRITE)
        assert out["status_code"] == flce.FLCE_OK
        assert rel_fro(dW.float().cpu().numpy(), run_oracle(inp, sp)["dW"]) <= TOL["bf16"]["grad"]


@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16, torch.float16])
def test_scale_by(dt):
    """flce_scale_by: x *= g on the device; bit-identical no-op when g == 1."""
    x = (torch.randn(100003, generator=torch.Generator().manual_seed(3)) * 3).to(dt).cuda()
    ref = x.clone()
    flce.scale_by(x, torch.ones(1, device="cuda"))
    assert torch.equal(x, ref)
    flce.scale_by(x, torch.full((1,), 0.375, device="cuda"))
    assert torch.equal(x, (ref.float() * 0.375).to(dt))


@pytest.mark.parametrize("BT,n_ignored", [(4864, 0), (6400, 0)])
def test_dx_three_and_four_way_k_splits(BT, n_ignored):
    """On 76 pairs, 19 dX pair tiles (4864 rows, H <= 512) take four K splits and 25 tiles
    (6400 rows) three: splits 0-1 add into one zeroed fp32 buffer, 2-3 into a second, so
    the result is bit-identical run to run, and it matches the oracle."""
    sp = I.spec("llama1b", BT=BT, H=256, V=2000, w_std=0.2, ignore="none")
    inp = I.generate(sp, seed=25)
    a = run_gpu(inp, sp)
    b = run_gpu(inp, sp)
    assert np.array_equal(a["dX"], b["dX"]) and np.array_equal(a["dW"], b["dW"])
    compare_full(a, run_oracle(inp, sp), inp, sp)


@pytest.mark.parametrize("BT,H,V", [(1, 64, 1000), (50, 8, 7), (37, 16, 300), (130, 24, 5),
                                    (257, 72, 257)])
@pytest.mark.parametrize("path", ["tc", "simt"])
def test_tiny_shapes(BT, H, V, path):
    """Shapes far below one tile in every dimension (one row; V = 5 or 7 columns of a
    256-column tile; H = 8 or 24, under one 64-deep k-block) and just past tile edges
    (257): every output against the oracle, on both GEMM back-ends."""
    sp = I.spec("llama1b", BT=BT, H=H, V=V, w_std=0.5, ignore="none" if BT < 10 else "random",
                n_ignored=BT // 7)
    inp = I.generate(sp, seed=27 + BT)
    g = run_gpu(inp, sp, flags=flce.FLAG_FORCE_SIMT if path == "simt" else 0)
    assert g["status_code"] == flce.FLCE_OK
    compare_full(g, run_oracle(inp, sp), inp, sp)


@pytest.mark.parametrize("BT,H,V", [(1, 24, 9), (45, 40, 300)])
def test_tiny_shapes_fp32(BT, H, V):
    sp = I.spec("tiny_fp32", BT=BT, H=H, V=V, ignore="none" if BT < 10 else "random", n_ignored=5)
    inp = I.generate(sp, seed=28 + BT)
    compare_full(run_gpu(inp, sp), run_oracle(inp, sp), inp, sp)


@pytest.mark.parametrize("n_lab", [1, 127, 128, 129, 1000, 20000])
def test_mean_and_sum_equal_the_sum_of_per_token_values(n_lab):
    """The mean / sum outputs are the float64 sum of the per-token loss, z-loss and
    accuracy that reduction "none" returns for the same rows (the rows' values do not depend
    on the reduction), rounded once to fp32: checked at labelled counts around the final
    reduction's 128-block split (one row, one row per block, a ragged last block, many rows
    per block)."""
    BT = n_lab + 7
    base = dict(BT=BT, H=64, V=500, w_std=0.3, z=1e-3, ignore="random", n_ignored=7, want_dW=False)
    none = run_gpu(I.generate(I.spec("llama1b", reduction="none", **base), seed=11),
                   I.spec("llama1b", reduction="none", **base))
    lab = I.generate(I.spec("llama1b", reduction="none", **base), seed=11)["targets"].numpy() != I.IGNORE_INDEX
    assert int(lab.sum()) == n_lab
    for red in ("sum", "mean"):
        sp = I.spec("llama1b", reduction=red, **base)
        g = run_gpu(I.generate(sp, seed=11), sp)
        d = 1.0 if red == "sum" else float(n_lab)
        for k in ("loss", "z_loss", "acc"):
            want = np.float32(np.sum(none[k][lab].astype(np.float64)) / d)
            got = np.float32(g[k][0])
            assert abs(got - want) <= 2 * np.spacing(np.abs(want)) + 1e-30, (red, k, got, want)


def test_simt_dx_tile_sizes_give_the_same_bits():
    """fp32 inputs: one 2432-row chunk runs the SIMT dX GEMM on 128x128 tiles (8 x 19 of
    them), 128-row chunks on 64x64 tiles (few output tiles); every dX element sums its k in
    the same order either way, so dX, lse and the per-token loss are bit-identical, and both
    match the oracle."""
    sp = I.spec("tiny_fp32", BT=2432, H=1024, V=500, reduction="none", want_dW=False,
                n_ignored=0)
    inp = I.generate(sp, seed=12)
    wb = _ws_for_rows(sp["BT"], sp["H"], sp["V"], torch.float32, 128)
    assert flce.chunk_rows(sp["BT"], sp["H"], sp["V"], torch.float32, wb) == 128
    one = run_gpu(inp, sp)
    many = run_gpu(inp, sp, workspace_bytes=wb)
    for k in ("dX", "lse", "loss", "pred"):
        assert np.array_equal(one[k], many[k]), k
    compare_full(one, run_oracle(inp, sp), inp, sp)
