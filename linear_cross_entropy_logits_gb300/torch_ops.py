"""PyTorch integration: a torch.library custom op over the C ABI and an autograd Function.

The op runs the fused forward+backward in one call, so the gradients are produced in the
forward (as the pages' op does: "Liger-Kernel PR #1554: skip ignore_index rows", Summary:
the forward runs the logits, grad_input and grad_weight GEMMs) and the backward only
applies the upstream gradient:

  * mean / sum: the gradients are linear in the scalar upstream gradient g, so the forward
    computes them for g = 1 and the backward scales them by g;
  * none with a frozen head (W, bias without grad): dX row i is linear in g_i, so the
    backward scales the rows;
  * none with a trained head: dW mixes rows with their own g_i, so the backward calls the
    fused op again with the per-token upstream gradient.

The custom op has a fake (meta) implementation, so torch.compile traces it as one opaque op
(no graph break) and compiled results equal eager ones. Marshalling only: every step of the
computation runs in libflce.so.
"""

from __future__ import annotations

from typing import Optional

import torch

from . import flce

_REDUCTIONS = ("mean", "sum", "none")


@torch.library.custom_op("flce_gb300::fused_linear_cross_entropy", mutates_args=())
def fused_linear_cross_entropy_op(X: torch.Tensor, W: torch.Tensor, targets: torch.Tensor,
                                  bias: Optional[torch.Tensor], grad_out: Optional[torch.Tensor],
                                  ignore_index: int, reduction: str, z_loss_scale: float,
                                  want_dX: bool, want_dW: bool, dW_fp32: bool
                                  ) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor,
                                             torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor]:
    """(loss, z_loss, acc, lse, pred, dX, dW, dbias); dX/dW/dbias are empty when not wanted."""
    V, H = W.shape
    dW_dtype = torch.float32 if dW_fp32 else W.dtype
    # fresh gradient buffers, written (not accumulated) by the op: no zero fill
    dW = torch.empty(V, H, dtype=dW_dtype, device=X.device) if want_dW else None
    db = torch.empty(V, dtype=dW_dtype, device=X.device) if (want_dW and bias is not None) else None
    out = flce.fwd_bwd(X.contiguous(), W.contiguous(), targets.contiguous(),
                       None if bias is None else bias.contiguous(), ignore_index=ignore_index,
                       reduction=reduction, z_loss_scale=z_loss_scale, grad_out=grad_out,
                       want_dX=want_dX, want_dW=want_dW, dW=dW, dbias=db, check=False,
                       flags=flce.FLAG_DW_OVERWRITE)
    empty = X.new_empty(0)
    return (out["loss"], out["z_loss"], out["acc"], out["lse"], out["pred"],
            out["dX"] if want_dX else empty, dW if want_dW else empty.float(),
            db if db is not None else empty.float())


@fused_linear_cross_entropy_op.register_fake
def _(X, W, targets, bias, grad_out, ignore_index, reduction, z_loss_scale, want_dX, want_dW,
      dW_fp32):
    BT, H = X.shape
    V = W.shape[0]
    nl = BT if reduction == "none" else 1
    f32 = dict(dtype=torch.float32, device=X.device)
    dW_dtype = torch.float32 if dW_fp32 else W.dtype
    return (X.new_empty(nl, **{"dtype": torch.float32}), X.new_empty(nl, **{"dtype": torch.float32}),
            X.new_empty(nl, **{"dtype": torch.float32}), torch.empty(BT, **f32),
            torch.empty(BT, dtype=torch.int64, device=X.device),
            X.new_empty(BT, H) if want_dX else X.new_empty(0),
            torch.empty(V, H, dtype=dW_dtype, device=X.device) if want_dW else torch.empty(0, **f32),
            torch.empty(V, dtype=dW_dtype, device=X.device) if (want_dW and bias is not None)
            else torch.empty(0, **f32))


class FusedLinearCrossEntropy(torch.autograd.Function):
    """loss = CE(X W^T + b, targets) (+ z-loss) with ignore_index rows skipped; see module
    docstring for how the backward uses the gradients computed in the forward."""

    @staticmethod
    def forward(ctx, X, W, targets, bias, ignore_index, reduction, z_loss_scale, dW_fp32):
        if reduction not in _REDUCTIONS:
            raise ValueError(f"reduction must be one of {_REDUCTIONS}")
        need_x = ctx.needs_input_grad[0]
        need_w = ctx.needs_input_grad[1] or (bias is not None and ctx.needs_input_grad[3])
        loss, z, acc, lse, pred, dX, dW, db = fused_linear_cross_entropy_op(
            X, W, targets, bias, None, ignore_index, reduction, z_loss_scale,
            need_x, need_w, dW_fp32)
        ctx.reduction = reduction
        ctx.args = (ignore_index, z_loss_scale, dW_fp32)
        ctx.need = (need_x, need_w)
        if reduction == "none" and need_w:
            ctx.save_for_backward(X, W, targets, bias)   # recomputed with g_i in backward
        else:
            ctx.save_for_backward(dX, dW, db)
        ctx.has_bias = bias is not None
        ctx.mark_non_differentiable(z, acc, lse, pred)
        return loss, z, acc, lse, pred

    @staticmethod
    def backward(ctx, g_loss, *unused):
        need_x, need_w = ctx.need
        if ctx.reduction == "none" and need_w:
            X, W, targets, bias = ctx.saved_tensors
            ignore_index, z, dW_fp32 = ctx.args
            _, _, _, _, _, dX, dW, db = fused_linear_cross_entropy_op(
                X, W, targets, bias, g_loss.float().contiguous(), ignore_index, "none", z,
                need_x, True, dW_fp32)
        else:
            dX, dW, db = ctx.saved_tensors
            if ctx.reduction == "none":
                dX = dX * g_loss.to(dX.dtype)[:, None] if need_x else dX
            elif torch.compiler.is_compiling():
                # traced backward (torch.compile): plain tensor ops
                g = g_loss.reshape(())
                dX = dX * g.to(dX.dtype) if need_x else dX
                dW = dW * g.to(dW.dtype) if need_w else dW
                db = db * g.to(db.dtype) if (need_w and ctx.has_bias) else db
            else:
                g = g_loss.reshape(1).float().contiguous()
                prev = getattr(ctx, "applied_scale", None)
                if prev is None:
                    # eager, first backward: scale the op's own gradient buffers in place on
                    # the device and hand them out; nothing is done (no pass over dW) when
                    # the upstream gradient is exactly 1
                    ctx.applied_scale = g.clone()
                    if need_x:
                        flce.scale_by(dX, g)
                    if need_w:
                        flce.scale_by(dW, g)
                        if ctx.has_bias:
                            flce.scale_by(db, g)
                else:
                    # a later backward through a retained graph: the buffers were handed
                    # out scaled by the first upstream gradient, and whoever holds them
                    # (torch.autograd.grad's result, a hook) must keep what they got, so
                    # the new gradients are fresh tensors scaled by the ratio (if the handed
                    # out buffers were modified in place since, autograd's own check on the
                    # saved tensors raises before this backward runs)
                    if float(prev) == 0.0:
                        raise RuntimeError(
                            "fused_linear_cross_entropy: a second backward through a retained "
                            "graph cannot follow a first backward whose upstream gradient was 0")
                    r = (g / prev).contiguous()
                    dX = dX.clone() if need_x else dX
                    dW = dW.clone() if need_w else dW
                    db = db.clone() if (need_w and ctx.has_bias) else db
                    if need_x:
                        flce.scale_by(dX, r)
                    if need_w:
                        flce.scale_by(dW, r)
                        if ctx.has_bias:
                            flce.scale_by(db, r)
        return (dX if need_x else None, dW if need_w else None, None,
                db if (need_w and ctx.has_bias) else None, None, None, None, None)


def fused_linear_cross_entropy(X, W, targets, bias=None, *, ignore_index=-100, reduction="mean",
                               z_loss_scale=0.0, accum_dtype=None, return_extras=False):
    """Differentiable fused linear cross entropy. X [BT,H], W [V,H] (bf16/fp16/fp32, same
    dtype), targets int64 [BT]. ``accum_dtype=torch.float32`` accumulates dW/dbias in fp32
    (the pages' accum_dtype path); by default they come out in W's dtype. Returns the loss,
    or (loss, z_loss, accuracy, lse, pred) when ``return_extras``."""
    dW_fp32 = accum_dtype == torch.float32 or W.dtype == torch.float32
    outs = FusedLinearCrossEntropy.apply(X, W, targets, bias, ignore_index, reduction,
                                         float(z_loss_scale), dW_fp32)
    loss = outs[0] if reduction == "none" else outs[0].reshape(())
    if return_extras:
        return (loss,) + tuple(outs[1:])
    return loss
