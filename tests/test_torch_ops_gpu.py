"""The torch integration (custom op + autograd Function) on the GPU: gradients through
loss.backward() match the float64 oracle for every reduction with a trained and a frozen
head, and torch.compile(fullgraph=True) gives the eager results (the pages check that
compiled results equal eager: "Liger-Kernel PR #1554", Details item 6)."""

import numpy as np
import pytest
import torch

from linear_cross_entropy_logits_gb300 import build as B
from linear_cross_entropy_logits_gb300 import inputs as I
from parity_util import TOL, rel_fro, run_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build()


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("frozen", [False, True])
def test_autograd_matches_oracle(reduction, frozen):
    from linear_cross_entropy_logits_gb300.torch_ops import fused_linear_cross_entropy
    sp = I.spec("frozen_head", BT=320, H=128, V=3000, w_std=0.15, bias_std=0.2, n_ignored=70,
                reduction=reduction, grad_out="uniform", want_dW=not frozen, z=1e-3)
    inp = I.generate(sp, seed=40)
    X = inp["X"].cuda().requires_grad_(True)
    W = inp["W"].cuda().requires_grad_(not frozen)
    b = inp["bias"].cuda().requires_grad_(not frozen)
    t = inp["targets"].cuda()
    loss = fused_linear_cross_entropy(X, W, t, b, reduction=reduction, z_loss_scale=sp["z"],
                                      accum_dtype=torch.float32)
    g = inp["grad_out"].cuda()
    if reduction == "none":
        (loss * g).sum().backward()
        go = inp["grad_out"]
    else:
        (loss * 0.7).backward()
        go = None
    sp2 = dict(sp, grad_scalar=0.7) if reduction != "none" else sp
    o = run_oracle(dict(inp, grad_out=go) if reduction == "none" else dict(inp, grad_out=None), sp2)
    tol = TOL["bf16"]
    if reduction == "none":
        ref = o["loss"]
        assert np.max(np.abs(loss.detach().cpu().numpy() - ref) / np.maximum(np.abs(ref), 1e-3)) <= tol["loss"]
    else:
        assert abs(float(loss.detach()) - o["loss"]) <= tol["loss"] * abs(o["loss"])
    assert rel_fro(X.grad.float().cpu().numpy(), o["dX"]) <= tol["grad"]
    if not frozen:
        assert rel_fro(W.grad.float().cpu().numpy(), o["dW"]) <= tol["grad"]
        assert rel_fro(b.grad.float().cpu().numpy(), o["dbias"]) <= tol["grad"]
    else:
        assert W.grad is None and b.grad is None


def test_compile_matches_eager():
    from linear_cross_entropy_logits_gb300.torch_ops import fused_linear_cross_entropy
    sp = I.spec("llama8b", BT=512, H=256, V=4000, w_std=0.15, z=1e-4)
    inp = I.generate(sp, seed=41)
    A = (torch.randn(256, 256, generator=torch.Generator().manual_seed(42)) * 0.05).to(torch.bfloat16)

    def step(x, a, w, t):
        h = x @ a
        return fused_linear_cross_entropy(h, w, t, z_loss_scale=1e-4)

    res = []
    for fn in (step, torch.compile(step, fullgraph=True)):
        x = inp["X"].cuda()
        a = A.cuda().requires_grad_(True)
        w = inp["W"].cuda().requires_grad_(True)
        loss = fn(x, a, w, inp["targets"].cuda())
        loss.backward()
        res.append((loss.detach().float().cpu(), a.grad.float().cpu(), w.grad.float().cpu()))
    for e, c in zip(res[0], res[1]):
        assert torch.equal(e, c)


def test_autograd_upstream_gradient_scales():
    """(2.5 * loss).backward(): the gradients computed in the forward are scaled on the
    device by the upstream gradient (and left untouched when it is 1)."""
    from linear_cross_entropy_logits_gb300.torch_ops import fused_linear_cross_entropy
    sp = I.spec("llama1b", BT=300, H=192, V=3000, w_std=0.2, ignore="random", n_ignored=40)
    inp = I.generate(sp, seed=31)
    o = run_oracle(inp, sp)
    for scale in (1.0, 2.5):
        X = inp["X"].cuda().requires_grad_(True)
        W = inp["W"].cuda().requires_grad_(True)
        loss = fused_linear_cross_entropy(X, W, inp["targets"].cuda(), accum_dtype=torch.float32)
        (scale * loss).backward()
        assert rel_fro(X.grad.float().cpu().numpy(), scale * o["dX"]) <= TOL["bf16"]["grad"]
        assert rel_fro(W.grad.float().cpu().numpy(), scale * o["dW"]) <= TOL["bf16"]["grad"]



def test_second_backward_through_a_retained_graph():
    """loss.backward(retain_graph=True) with an upstream gradient of 2.5, then again with 1:
    the in-place scaling of the op's gradient buffers must not compound (each backward
    adds its own scale times the gradient)."""
    from linear_cross_entropy_logits_gb300.torch_ops import fused_linear_cross_entropy
    sp = I.spec("llama1b", BT=300, H=192, V=3000, w_std=0.2, ignore="random", n_ignored=40)
    inp = I.generate(sp, seed=32)
    o = run_oracle(inp, sp)
    X = inp["X"].cuda().requires_grad_(True)
    W = inp["W"].cuda().requires_grad_(True)
    loss = fused_linear_cross_entropy(X, W, inp["targets"].cuda(), accum_dtype=torch.float32)
    loss.backward(torch.tensor(2.5, device="cuda"), retain_graph=True)
    loss.backward()
    assert rel_fro(X.grad.float().cpu().numpy(), 3.5 * o["dX"]) <= TOL["bf16"]["grad"]
    assert rel_fro(W.grad.float().cpu().numpy(), 3.5 * o["dW"]) <= TOL["bf16"]["grad"]


def test_autograd_grad_twice_keeps_the_first_result():
    """torch.autograd.grad(..., retain_graph=True) twice: the tensors the first call
    returned keep their values (the second call's gradients are fresh tensors), and each
    call's gradients are its own upstream gradient times the oracle's."""
    from linear_cross_entropy_logits_gb300.torch_ops import fused_linear_cross_entropy
    sp = I.spec("llama1b", BT=300, H=192, V=3000, w_std=0.2, ignore="random", n_ignored=40)
    inp = I.generate(sp, seed=33)
    o = run_oracle(inp, sp)
    X = inp["X"].cuda().requires_grad_(True)
    W = inp["W"].cuda().requires_grad_(True)
    loss = fused_linear_cross_entropy(X, W, inp["targets"].cuda(), accum_dtype=torch.float32)
    gx1, gw1 = torch.autograd.grad(loss, (X, W), torch.tensor(2.5, device="cuda"), retain_graph=True)
    keep_x, keep_w = gx1.clone(), gw1.clone()
    gx2, gw2 = torch.autograd.grad(loss, (X, W), torch.tensor(-0.5, device="cuda"), retain_graph=True)
    assert torch.equal(gx1, keep_x) and torch.equal(gw1, keep_w)
    assert gx2.data_ptr() != gx1.data_ptr() and gw2.data_ptr() != gw1.data_ptr()
    assert rel_fro(gx1.float().cpu().numpy(), 2.5 * o["dX"]) <= TOL["bf16"]["grad"]
    assert rel_fro(gw1.float().cpu().numpy(), 2.5 * o["dW"]) <= TOL["bf16"]["grad"]
    assert rel_fro(gx2.float().cpu().numpy(), -0.5 * o["dX"]) <= TOL["bf16"]["grad"]
    assert rel_fro(gw2.float().cpu().numpy(), -0.5 * o["dW"]) <= TOL["bf16"]["grad"]


def test_second_backward_after_a_zero_upstream_gradient_raises():
    """A first backward with upstream gradient 0 leaves nothing to rescale from: a second
    backward through the retained graph raises instead of returning inf/NaN gradients; so
    does one after the first gradients were modified in place (autograd's version check on
    the saved buffers)."""
    from linear_cross_entropy_logits_gb300.torch_ops import fused_linear_cross_entropy
    sp = I.spec("llama1b", BT=200, H=128, V=2000, w_std=0.2)
    inp = I.generate(sp, seed=34)
    X = inp["X"].cuda().requires_grad_(True)
    W = inp["W"].cuda().requires_grad_(True)
    loss = fused_linear_cross_entropy(X, W, inp["targets"].cuda(), accum_dtype=torch.float32)
    torch.autograd.grad(loss, (X, W), torch.tensor(0.0, device="cuda"), retain_graph=True)
    with pytest.raises(RuntimeError, match="upstream gradient was 0"):
        torch.autograd.grad(loss, (X, W), torch.tensor(1.0, device="cuda"), retain_graph=True)
    loss = fused_linear_cross_entropy(X, W, inp["targets"].cuda(), accum_dtype=torch.float32)
    gx, gw = torch.autograd.grad(loss, (X, W), retain_graph=True)
    # dX comes back in X's dtype, so autograd hands out the op's own buffer (the fp32 dW
    # is cast to W's dtype on the way out, a copy)
    gx.mul_(3.0)
    with pytest.raises(RuntimeError, match="modified by an inplace operation"):
        torch.autograd.grad(loss, (X, W), retain_graph=True)
