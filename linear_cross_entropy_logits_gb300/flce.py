"""Thin ctypes binding of libflce.so (the C ABI in include/flce.h).

Argument marshalling only: torch tensors supply device memory and the current CUDA stream;
every step of the computation runs in the library's kernels. If the library has not been
built the first call raises, there is no fallback.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libflce.so")

FLCE_OK, FLCE_ERR_INVALID_ARG, FLCE_ERR_UNSUPPORTED, FLCE_ERR_TARGET_RANGE = 0, 1, 2, 3
FLCE_ERR_WORKSPACE, FLCE_ERR_CUDA, FLCE_ERR_TIMEOUT, FLCE_ERR_SCRATCH_LIMIT = 4, 5, 6, 7
NOALLOC_SCRATCH_BYTES = 128 << 20
REDUCTIONS = {"mean": 0, "sum": 1, "none": 2}
DTYPES = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}
FLAG_FORCE_SIMT = 0x1
FLAG_NO_ROW_REF = 0x2
FLAG_DW_OVERWRITE = 0x4
FLAG_SEPARATE_BWD = 0x8
FLAG_DEBUG_STALL = 0x100
FLAG_DEBUG_STALL_BWD = 0x200
EXPORTED = ("flce_workspace_size", "flce_chunk_rows", "flce_fwd_bwd", "flce_fwd_bwd_noalloc",
            "flce_get_status",
            "flce_profile_create", "flce_profile_reset", "flce_profile_destroy",
            "flce_profile_read", "flce_last_cuda_error", "flce_status_string", "flce_abi_version",
            "flce_jsd_workspace_size", "flce_fused_linear_jsd", "flce_scale_by",
            "flce_plan_describe")
STAGES = ("prologue", "gather", "fwd", "finalize", "gpass", "dx", "dw", "reduce", "bwd")


class FlceArgs(ctypes.Structure):
    """Mirror of ``flce_args`` (field order and C types must match include/flce.h)."""
    _fields_ = [
        ("BT", ctypes.c_int64), ("H", ctypes.c_int64), ("V", ctypes.c_int64),
        ("in_dtype", ctypes.c_int32), ("reduction", ctypes.c_int32),
        ("X", ctypes.c_void_p), ("W", ctypes.c_void_p), ("bias", ctypes.c_void_p),
        ("targets", ctypes.c_void_p), ("ignore_index", ctypes.c_int64),
        ("z_loss_scale", ctypes.c_float), ("grad_out", ctypes.c_void_p),
        ("want_dX", ctypes.c_int32), ("want_dW", ctypes.c_int32), ("dW_dtype", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("loss", ctypes.c_void_p), ("z_loss", ctypes.c_void_p), ("acc", ctypes.c_void_p),
        ("lse", ctypes.c_void_p), ("pred", ctypes.c_void_p), ("n_labelled", ctypes.c_void_p),
        ("dX", ctypes.c_void_p), ("dW", ctypes.c_void_p), ("dbias", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("status", ctypes.c_void_p), ("wait_timeout_ms", ctypes.c_uint32),
        ("profile", ctypes.c_void_p),
    ]


class FlceJsdArgs(ctypes.Structure):
    """Mirror of ``flce_jsd_args`` (field order and C types must match include/flce.h)."""
    _fields_ = [
        ("BT", ctypes.c_int64), ("Hs", ctypes.c_int64), ("Ht", ctypes.c_int64), ("V", ctypes.c_int64),
        ("in_dtype", ctypes.c_int32), ("reduction", ctypes.c_int32),
        ("Xs", ctypes.c_void_p), ("Ws", ctypes.c_void_p), ("Xt", ctypes.c_void_p), ("Wt", ctypes.c_void_p),
        ("labels", ctypes.c_void_p), ("ignore_index", ctypes.c_int64),
        ("beta", ctypes.c_float), ("temperature", ctypes.c_float), ("grad_out", ctypes.c_void_p),
        ("want_dX", ctypes.c_int32), ("want_dW", ctypes.c_int32), ("dW_dtype", ctypes.c_int32),
        ("flags", ctypes.c_uint32),
        ("loss", ctypes.c_void_p), ("n_labelled", ctypes.c_void_p), ("dX", ctypes.c_void_p),
        ("dW", ctypes.c_void_p), ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("status", ctypes.c_void_p), ("wait_timeout_ms", ctypes.c_uint32),
        ("profile", ctypes.c_void_p),
    ]


_lib = None


def load(path: str | None = None):
    """Load libflce.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with linear_cross_entropy_logits_gb300.build.build()")
    lib = ctypes.CDLL(p)
    lib.flce_workspace_size.restype = ctypes.c_size_t
    lib.flce_workspace_size.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_int32, ctypes.c_size_t]
    lib.flce_chunk_rows.restype = ctypes.c_int64
    lib.flce_chunk_rows.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_int32, ctypes.c_size_t]
    lib.flce_plan_describe.restype = ctypes.c_int64
    lib.flce_plan_describe.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_int32, ctypes.c_size_t,
                                                              ctypes.c_char_p, ctypes.c_size_t]
    lib.flce_fwd_bwd.restype = ctypes.c_int32
    lib.flce_fwd_bwd.argtypes = [ctypes.POINTER(FlceArgs), ctypes.c_void_p]
    lib.flce_fwd_bwd_noalloc.restype = ctypes.c_int32
    lib.flce_fwd_bwd_noalloc.argtypes = [ctypes.POINTER(FlceArgs), ctypes.c_void_p]
    lib.flce_get_status.restype = ctypes.c_int32
    lib.flce_get_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    lib.flce_status_string.restype = ctypes.c_char_p
    lib.flce_status_string.argtypes = [ctypes.c_int32]
    lib.flce_abi_version.restype = ctypes.c_int32
    lib.flce_last_cuda_error.restype = ctypes.c_char_p
    lib.flce_last_cuda_error.argtypes = []
    lib.flce_scale_by.restype = ctypes.c_int32
    lib.flce_scale_by.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                  ctypes.c_void_p]
    lib.flce_jsd_workspace_size.restype = ctypes.c_size_t
    lib.flce_jsd_workspace_size.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int32, ctypes.c_size_t]
    lib.flce_fused_linear_jsd.restype = ctypes.c_int32
    lib.flce_fused_linear_jsd.argtypes = [ctypes.POINTER(FlceJsdArgs), ctypes.c_void_p]
    lib.flce_profile_create.restype = ctypes.c_void_p
    lib.flce_profile_create.argtypes = []
    lib.flce_profile_reset.restype = None
    lib.flce_profile_reset.argtypes = [ctypes.c_void_p]
    lib.flce_profile_destroy.restype = None
    lib.flce_profile_destroy.argtypes = [ctypes.c_void_p]
    lib.flce_profile_read.restype = ctypes.c_int32
    lib.flce_profile_read.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_float),
                                      ctypes.POINTER(ctypes.c_int32), ctypes.c_int32]
    _lib = lib
    return lib


class FlceError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        msg = f"{where}: {status_string(code)}"
        if code == FLCE_ERR_CUDA:
            msg += f" ({load().flce_last_cuda_error().decode()})"
        super().__init__(msg)


def status_string(code: int) -> str:
    return load().flce_status_string(int(code)).decode()


def workspace_size(BT, H, V, dtype=torch.bfloat16, budget_bytes=0) -> int:
    return int(load().flce_workspace_size(BT, H, V, DTYPES[dtype], budget_bytes))


def chunk_rows(BT, H, V, dtype, workspace_bytes) -> int:
    return int(load().flce_chunk_rows(BT, H, V, DTYPES[dtype], workspace_bytes))


def describe_plan(BT, H, V, dtype=torch.bfloat16, workspace_bytes=None, budget_bytes=0) -> str:
    """The library's text plan of a call (chunk rows, workspace regions, GEMM tiles) for a
    workspace of ``workspace_bytes`` (default: the planner's size for ``budget_bytes``)."""
    lib = load()
    wb = workspace_size(BT, H, V, dtype, budget_bytes) if workspace_bytes is None else workspace_bytes
    n = int(lib.flce_plan_describe(BT, H, V, DTYPES[dtype], wb, None, 0))
    if n < 0:
        raise FlceError(FLCE_ERR_INVALID_ARG, "flce_plan_describe")
    buf = ctypes.create_string_buffer(n + 1)
    lib.flce_plan_describe(BT, H, V, DTYPES[dtype], wb, buf, n + 1)
    return buf.value.decode()


class Profiler:
    """Per-stage device time of the calls that are given this profiler (CUDA events
    recorded by the library on the launching stream)."""

    def __init__(self):
        self._lib = load()
        self.handle = self._lib.flce_profile_create()
        if not self.handle:
            raise MemoryError("flce_profile_create")

    def reset(self):
        self._lib.flce_profile_reset(self.handle)

    def read(self):
        n = len(STAGES)
        ms = (ctypes.c_float * n)()
        cnt = (ctypes.c_int32 * n)()
        rc = self._lib.flce_profile_read(self.handle, ms, cnt, n)
        if rc != FLCE_OK:
            raise FlceError(rc, "flce_profile_read")
        return {s: (float(ms[i]), int(cnt[i])) for i, s in enumerate(STAGES)}

    def close(self):
        if self.handle:
            self._lib.flce_profile_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _ptr(t):
    return None if t is None else t.data_ptr()


def fwd_bwd(X, W, targets, bias=None, *, ignore_index=-100, reduction="mean",
            z_loss_scale=0.0, grad_out=None, want_dX=True, want_dW=True, dW=None, dbias=None,
            workspace=None, workspace_bytes=None, budget_bytes=0, outputs=None, flags=0,
            wait_timeout_ms=0, check=True, stream=None, profiler=None):
    """Fused linear cross entropy forward + backward on X's device.

    X [BT,H] and W [V,H] share a dtype (fp32, bf16 or fp16); targets int64 [BT]. dW/dbias
    are accumulated into when given (fp32, or X's dtype for same-dtype accumulation), else
    allocated as fp32 zeros. Returns a dict of
    tensors: loss, z_loss, acc (reduced per ``reduction``), lse, pred, n_labelled, dX, dW,
    dbias, and the status code when ``check`` is set (which synchronises the stream).
    ``outputs`` may carry preallocated output tensors under the same keys.
    """
    lib = load()
    if X.device.type != "cuda":
        raise ValueError("X must be a CUDA tensor")
    BT, H = X.shape
    V = W.shape[0]
    dev = X.device
    red = REDUCTIONS[reduction]
    o = dict(outputs or {})
    nl = BT if reduction == "none" else 1
    if o.get("loss") is None:
        o["loss"] = torch.empty(nl, dtype=torch.float32, device=dev)
    if o.get("z_loss") is None:
        o["z_loss"] = torch.empty(nl, dtype=torch.float32, device=dev)
    if o.get("acc") is None:
        o["acc"] = torch.empty(nl, dtype=torch.float32, device=dev)
    if o.get("lse") is None:
        o["lse"] = torch.empty(BT, dtype=torch.float32, device=dev)
    if o.get("pred") is None:
        o["pred"] = torch.empty(BT, dtype=torch.int64, device=dev)
    if o.get("n_labelled") is None:
        o["n_labelled"] = torch.empty(1, dtype=torch.int32, device=dev)
    if o.get("status") is None:
        o["status"] = torch.zeros(1, dtype=torch.int32, device=dev)
    if want_dX and o.get("dX") is None:
        o["dX"] = torch.empty_like(X)
    dW_dt = torch.float32 if dW is None else dW.dtype
    if want_dW and dW is None:
        dW = torch.zeros(V, H, dtype=dW_dt, device=dev)
    if want_dW and bias is not None and dbias is None:
        dbias = torch.zeros(V, dtype=dW_dt, device=dev)
    if workspace is None:
        nbytes = workspace_bytes or workspace_size(BT, H, V, X.dtype, budget_bytes)
        if nbytes == 0:
            raise FlceError(FLCE_ERR_WORKSPACE, "workspace_size")
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    wbytes = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    if grad_out is not None and not torch.is_tensor(grad_out):
        grad_out = torch.tensor([float(grad_out)], dtype=torch.float32, device=dev)

    a = FlceArgs()
    a.BT, a.H, a.V = BT, H, V
    a.in_dtype = DTYPES[X.dtype]
    a.reduction = red
    a.X, a.W, a.bias = _ptr(X), _ptr(W), _ptr(bias)
    a.targets = _ptr(targets)
    a.ignore_index = ignore_index
    a.z_loss_scale = z_loss_scale
    a.grad_out = _ptr(grad_out)
    a.want_dX, a.want_dW = int(bool(want_dX)), int(bool(want_dW))
    a.dW_dtype = DTYPES[dW_dt]
    a.flags = flags
    a.loss, a.z_loss, a.acc = _ptr(o["loss"]), _ptr(o["z_loss"]), _ptr(o["acc"])
    a.lse, a.pred, a.n_labelled = _ptr(o["lse"]), _ptr(o["pred"]), _ptr(o["n_labelled"])
    a.dX = _ptr(o.get("dX")) if want_dX else None
    a.dW = _ptr(dW) if want_dW else None
    a.dbias = _ptr(dbias) if (want_dW and bias is not None) else None
    a.workspace, a.workspace_bytes = _ptr(workspace), wbytes
    a.status = _ptr(o["status"])
    a.wait_timeout_ms = wait_timeout_ms
    a.profile = profiler.handle if profiler is not None else None
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    rc = lib.flce_fwd_bwd(ctypes.byref(a), ctypes.c_void_p(s.cuda_stream))
    if rc != FLCE_OK:
        raise FlceError(rc, "flce_fwd_bwd")
    o["dW"], o["dbias"] = dW, dbias
    o["workspace"] = workspace
    if check:
        o["status_code"] = int(lib.flce_get_status(ctypes.c_void_p(_ptr(o["status"])), None,
                                                   ctypes.c_void_p(s.cuda_stream)))
    return o


def jsd_workspace_size(BT, Hs, Ht, V, dtype=torch.bfloat16, budget_bytes=0) -> int:
    return int(load().flce_jsd_workspace_size(BT, Hs, Ht, V, DTYPES[dtype], budget_bytes))


def fused_linear_jsd(Xs, Ws, Xt, Wt, labels=None, *, beta=0.5, temperature=1.0, ignore_index=-100,
                     reduction="mean", grad_out=None, want_dX=True, want_dW=True, dW=None,
                     workspace=None, budget_bytes=0, flags=0, check=True, stream=None, profiler=None,
                     outputs=None):
    """Fused linear JSD / KL distillation forward + backward (student gradients only).
    Returns a dict with loss, n_labelled, dX, dW (and status_code when ``check``)."""
    lib = load()
    BT, Hs = Xs.shape
    Ht = Xt.shape[1]
    V = Ws.shape[0]
    dev = Xs.device
    nl = BT if reduction == "none" else 1
    o = dict(outputs or {})
    if o.get("loss") is None:
        o["loss"] = torch.empty(nl, dtype=torch.float32, device=dev)
    if o.get("n_labelled") is None:
        o["n_labelled"] = torch.empty(1, dtype=torch.int32, device=dev)
    if o.get("status") is None:
        o["status"] = torch.zeros(1, dtype=torch.int32, device=dev)
    if want_dX and o.get("dX") is None:
        o["dX"] = torch.empty_like(Xs)
    if want_dW and dW is None:
        dW = torch.zeros(V, Hs, dtype=torch.float32, device=dev)
    if workspace is None:
        nbytes = jsd_workspace_size(BT, Hs, Ht, V, Xs.dtype, budget_bytes)
        if nbytes == 0:
            raise FlceError(FLCE_ERR_WORKSPACE, "jsd_workspace_size")
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if grad_out is not None and not torch.is_tensor(grad_out):
        grad_out = torch.tensor([float(grad_out)], dtype=torch.float32, device=dev)
    a = FlceJsdArgs()
    a.BT, a.Hs, a.Ht, a.V = BT, Hs, Ht, V
    a.in_dtype = DTYPES[Xs.dtype]
    a.reduction = REDUCTIONS[reduction]
    a.Xs, a.Ws, a.Xt, a.Wt = _ptr(Xs), _ptr(Ws), _ptr(Xt), _ptr(Wt)
    a.labels = _ptr(labels)
    a.ignore_index = ignore_index
    a.beta, a.temperature = beta, temperature
    a.grad_out = _ptr(grad_out)
    a.want_dX, a.want_dW = int(bool(want_dX)), int(bool(want_dW))
    a.dW_dtype = DTYPES[dW.dtype] if dW is not None else 0
    a.flags = flags
    a.loss, a.n_labelled = _ptr(o["loss"]), _ptr(o["n_labelled"])
    a.dX = _ptr(o.get("dX")) if want_dX else None
    a.dW = _ptr(dW) if want_dW else None
    a.workspace, a.workspace_bytes = _ptr(workspace), workspace.numel()
    a.status = _ptr(o["status"])
    a.profile = profiler.handle if profiler is not None else None
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    rc = lib.flce_fused_linear_jsd(ctypes.byref(a), ctypes.c_void_p(s.cuda_stream))
    if rc != FLCE_OK:
        raise FlceError(rc, "flce_fused_linear_jsd")
    o["dW"] = dW
    if check:
        o["status_code"] = int(lib.flce_get_status(ctypes.c_void_p(_ptr(o["status"])), None,
                                                   ctypes.c_void_p(s.cuda_stream)))
    return o


def scale_by(x, g, stream=None):
    """x *= g in place (x: contiguous CUDA tensor, fp32/bf16/fp16; g: one-element fp32 CUDA
    tensor), skipped on the device when g == 1."""
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    rc = load().flce_scale_by(ctypes.c_void_p(x.data_ptr()), x.numel(), DTYPES[x.dtype],
                              ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(s.cuda_stream))
    if rc != FLCE_OK:
        raise FlceError(rc, "flce_scale_by")
    return x


def raw_call(args: FlceArgs, stream_handle: int) -> int:
    """Call flce_fwd_bwd with a prepared FlceArgs (for callers that manage every buffer)."""
    return int(load().flce_fwd_bwd(ctypes.byref(args), ctypes.c_void_p(stream_handle)))
