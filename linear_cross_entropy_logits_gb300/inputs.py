"""Seeded synthetic inputs for the fused linear cross entropy workloads.

This module only draws random numbers and lays out target masks. It holds none of the
method's arithmetic, and it is the one module that both the CUDA path's callers and the
float64 oracle's tests take inputs from.

Every draw comes from one ``torch.Generator`` seeded with ``seed``, in a fixed order:
targets, ignored-row mask, X, W, bias, upstream gradient. bf16/fp16 values are rounded to
nearest-even from fp32 draws; the oracle receives exactly those rounded values.

Workloads (shapes after the pages' model heads):
  * ``tiny_fp32``   BT=128, H=64, V=1000, fp32, X~N(0,1), W~N(0,1/H), 13 rows ignored at
                    random, mean, dX and dW.
  * ``llama1b``     Llama-3.2-1B head: BT=8192, H=2048, V=128256, bf16, W~N(0,0.02^2), all
                    rows labelled, uniform targets, mean, dX and fp32 dW.
  * ``llama8b``     Llama-3.1-8B head: BT=8192, H=4096, V=128256, bf16, 16 sequences of 512
                    rows, each prompt-first (the leading round((1-f)*512) rows ignored) plus
                    its last row ignored, mean, z-loss 1e-4, dX and fp32 dW. ``f`` is the
                    labelled fraction (1.0, 0.75, 0.5, 0.25, 0.1).
  * ``large_vocab`` BT=32768, H=5376, V=262144, bf16, all labelled, Zipf(1.1) targets (rank
                    k maps to token k-1), sum, dX and fp32 dW.
  * ``frozen_head`` BT=16384, H=4096, V=151936, bf16, bias~N(0,0.01^2), 8192 rows ignored at
                    random, none with a per-token upstream gradient ~U(0.5,1.5), dX only.
  * ``llama2_7b``   a 32000-token head: BT=16384, H=4096, V=32000, bf16 (or fp32 / fp16 by
                    override), W~N(0,0.02^2), all rows labelled, uniform targets, mean, dX and
                    fp32 dW.
  * ``distill``     fused linear JSD distillation: student Llama-3.2-1B-shaped head (Hs=2048)
                    against a Llama-3.1-8B-shaped teacher head (Ht=4096), V=128256,
                    BT=8192, bf16, W~N(0,0.02^2), all rows labelled, beta=0.5, T=1, mean,
                    student dX and fp32 dW. Drawn by generate_distill: labels, X_s, W_s,
                    X_t, W_t.
"""

from __future__ import annotations

import math

import numpy as np
import torch

IGNORE_INDEX = -100

WORKLOADS = {
    "tiny_fp32": dict(BT=128, H=64, V=1000, dtype="f32", x_std=1.0, w_std=1.0 / 8.0,
                      bias_std=None, targets="uniform", ignore="random", n_ignored=13,
                      reduction="mean", z=0.0, want_dW=True),
    "llama1b": dict(BT=8192, H=2048, V=128256, dtype="bf16", x_std=1.0, w_std=0.02,
                    bias_std=None, targets="uniform", ignore="none", reduction="mean",
                    z=0.0, want_dW=True),
    "llama8b": dict(BT=8192, H=4096, V=128256, dtype="bf16", x_std=1.0, w_std=0.02,
                    bias_std=None, targets="uniform", ignore="prompt_first", seq_len=512,
                    labelled_fraction=1.0, reduction="mean", z=1e-4, want_dW=True),
    "large_vocab": dict(BT=32768, H=5376, V=262144, dtype="bf16", x_std=1.0, w_std=0.02,
                        bias_std=None, targets="zipf", zipf_s=1.1, ignore="none",
                        reduction="sum", z=0.0, want_dW=True,
                        workspace_cap=int(1.5 * 2 ** 30)),
    "frozen_head": dict(BT=16384, H=4096, V=151936, dtype="bf16", x_std=1.0, w_std=0.02,
                        bias_std=0.01, targets="uniform", ignore="random", n_ignored=8192,
                        reduction="none", grad_out="uniform", z=0.0, want_dW=False),
    "llama2_7b": dict(BT=16384, H=4096, V=32000, dtype="bf16", x_std=1.0, w_std=0.02,
                      bias_std=None, targets="uniform", ignore="none", reduction="mean",
                      z=0.0, want_dW=True),
}

DISTILL = dict(name="distill", BT=8192, Hs=2048, Ht=4096, V=128256, dtype="bf16", x_std=1.0,
               w_std=0.02, ignore="none", beta=0.5, temperature=1.0, reduction="mean",
               want_dW=True)

TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def spec(name, **overrides):
    """A workload spec by name, with fields overridden (e.g. smaller shapes for tests)."""
    s = dict(WORKLOADS[name])
    s["name"] = name
    s.update(overrides)
    return s


def prompt_first_length(seq_len, labelled_fraction):
    """Leading ignored rows per sequence: round-half-up of (1 - f) * seq_len."""
    return int(math.floor((1.0 - labelled_fraction) * seq_len + 0.5))


def _zipf_targets(g, BT, V, s):
    u = torch.rand(BT, generator=g, dtype=torch.float64).numpy()
    k = np.arange(1, V + 1, dtype=np.float64)
    cdf = np.cumsum(k ** (-s))
    cdf /= cdf[-1]
    idx = np.searchsorted(cdf, u, side="left")
    return torch.from_numpy(np.minimum(idx, V - 1).astype(np.int64))


def generate(sp, seed=0):
    """Draw one workload's inputs on the CPU. Returns a dict of CPU tensors:
    X [BT,H], W [V,H] (in the workload dtype), bias [V] or None, targets int64 [BT],
    grad_out (fp32 [BT] for reduction none with a drawn gradient, else None)."""
    BT, H, V = sp["BT"], sp["H"], sp["V"]
    dt = TORCH_DTYPES[sp["dtype"]]
    g = torch.Generator().manual_seed(seed)

    # 1. targets
    if sp.get("targets", "uniform") == "zipf":
        targets = _zipf_targets(g, BT, V, sp.get("zipf_s", 1.1))
    else:
        targets = torch.randint(0, V, (BT,), generator=g, dtype=torch.int64)

    # 2. ignored-row mask
    mode = sp.get("ignore", "none")
    if mode == "random":
        k = sp["n_ignored"]
        perm = torch.randperm(BT, generator=g)[:k]
        targets[perm] = IGNORE_INDEX
    elif mode == "prompt_first":
        L = sp.get("seq_len", 512)
        p = prompt_first_length(L, sp.get("labelled_fraction", 1.0))
        pos = torch.arange(BT) % L
        targets[(pos < p) | (pos == L - 1)] = IGNORE_INDEX
    elif mode == "all":
        targets[:] = IGNORE_INDEX
    elif mode != "none":
        raise ValueError(f"unknown ignore mode {mode}")

    # 3. X, 4. W, 5. bias
    X = (torch.randn(BT, H, generator=g) * sp.get("x_std", 1.0)).to(dt)
    W = (torch.randn(V, H, generator=g) * sp["w_std"]).to(dt)
    bias = None
    if sp.get("bias_std") is not None:
        bias = (torch.randn(V, generator=g) * sp["bias_std"]).to(dt)

    # 6. upstream gradient
    grad_out = None
    if sp.get("grad_out") == "uniform":
        grad_out = torch.rand(BT, generator=g) + 0.5
    return {"X": X, "W": W, "bias": bias, "targets": targets, "grad_out": grad_out}


def generate_distill(sp=None, seed=0):
    """Draw one distillation problem on the CPU: labels int64 [BT] (ignored rows per
    ``ignore``/``n_ignored``), Xs [BT,Hs], Ws [V,Hs], Xt [BT,Ht], Wt [V,Ht]."""
    sp = dict(DISTILL, **(sp or {}))
    BT, V = sp["BT"], sp["V"]
    dt = TORCH_DTYPES[sp["dtype"]]
    g = torch.Generator().manual_seed(seed)
    labels = torch.randint(0, V, (BT,), generator=g, dtype=torch.int64)
    if sp.get("ignore") == "random":
        labels[torch.randperm(BT, generator=g)[:sp["n_ignored"]]] = IGNORE_INDEX
    Xs = (torch.randn(BT, sp["Hs"], generator=g) * sp["x_std"]).to(dt)
    Ws = (torch.randn(V, sp["Hs"], generator=g) * sp["w_std"]).to(dt)
    Xt = (torch.randn(BT, sp["Ht"], generator=g) * sp["x_std"]).to(dt)
    Wt = (torch.randn(V, sp["Ht"], generator=g) * sp["w_std"]).to(dt)
    return {"labels": labels, "Xs": Xs, "Ws": Ws, "Xt": Xt, "Wt": Wt}


def to_numpy_exact(t):
    """Exact float32/float64 numpy copy of a CPU tensor (bf16/fp16 values are exact in
    fp32)."""
    if t is None:
        return None
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.float()
    return t.numpy()
