"""FlashAttention-2 exact multi-head attention on GB300 (sm_103a).

A thin Python binding over ``libfa2.so``, whose C ABI is declared in
``include/fa2.h``. This module only marshals arguments: every step of the
forward and backward pass runs in the library's CUDA kernels. PyTorch is used
for device memory, streams and the autograd hook, nothing else. There is no
CPU or PyTorch fallback: if the library is missing or a call fails, an
exception is raised.

Tensors are contiguous ``[B, H, N, d]`` CUDA tensors of dtype float16 or
bfloat16 (``d`` in {64, 128}); the logsumexp is float32 ``[B, H, N]``.
"""

from __future__ import annotations

import ctypes
import math
from pathlib import Path

import torch

__all__ = [
    "FA2Error",
    "load_library",
    "forward",
    "forward_instrumented",
    "forward_kv_outer",
    "step_host",
    "backward",
    "bwd_workspace_size",
    "device_status",
    "attention",
    "fwd_grid",
    "fwd_block_work",
    "fwd_schedule",
    "bwd_grid",
    "bwd_block_work",
    "status_string",
]

_LIB_PATH = Path(__file__).resolve().parent / "libfa2.so"
_lib = None

_c_int_p = ctypes.POINTER(ctypes.c_int)


class FA2Error(RuntimeError):
    """A libfa2 call returned a status other than FA2_OK."""

    def __init__(self, func: str, code: int):
        self.code = code
        extra = ""
        if code == 5:  # FA2_ERR_CUDA: name the underlying CUDA error
            extra = f", cuda error {load_library().fa2_last_cuda_error()}"
        super().__init__(f"{func} failed: {status_string(code)} ({code}{extra})")


def load_library() -> ctypes.CDLL:
    """Load libfa2.so (built by ``exact_attention_64_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not _LIB_PATH.exists():
        raise RuntimeError(
            f"{_LIB_PATH} is not built; run `python -m exact_attention_64_gb300.build` "
            "(or __graft_entry__.build())"
        )
    lib = ctypes.CDLL(str(_LIB_PATH))
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sigs = {
        "fa2_fwd": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]),
        "fa2_fwd_instrumented": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp]),
        "fa2_fwd_split": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz, vp]),
        "fa2_fwd_qk": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]),
        "fa2_bwd_qk": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]),
        "fa2_fwd_split_workspace_size": (sz, [i, i, i, i, i]),
        "fa2_fwd_kv_outer": (i, [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]),
        "fa2_fwd_kv_outer_workspace_size": (sz, [i, i, i, i]),
        "fa2_step_host": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, sz,
                              vp]),
        "fa2_step_host_workspace_size": (sz, [i, i, i, i, i]),
        "fa2_num_splits": (i, [i, i, i, i, i, i]),
        "fa2_bwd_workspace_size": (sz, [i, i, i, i]),
        "fa2_bwd_atomic_workspace_size": (sz, [i, i, i, i]),
        "fa2_bwd": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]),
        "fa2_bwd_atomic": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz,
                               vp]),
        "fa2_bwd_timed": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp,
                              vp]),
        "fa2_bwd_atomic_timed": (i, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp,
                                     sz, vp, vp]),
        "fa2_get_device_status": (i, [vp]),
        "fa2_status_string": (ctypes.c_char_p, [i]),
        "fa2_fwd_grid": (i, [i, i, i, _c_int_p, _c_int_p]),
        "fa2_fwd_block_work": (i, [i, i, i, _c_int_p, _c_int_p, _c_int_p]),
        "fa2_fwd_schedule": (i, [i, i, i, i, i, _c_int_p, _c_int_p, _c_int_p]),
        "fa2_bwd_grid": (i, [i, i, i, i, _c_int_p, _c_int_p, _c_int_p]),
        "fa2_bwd_block_work": (i, [i, i, i, i, _c_int_p, _c_int_p, _c_int_p, _c_int_p]),
        "fa2_debug_arm_fault": (i, [i, i]),
        "fa2_last_cuda_error": (i, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().fa2_status_string(int(code)).decode()


def _check(func: str, code: int) -> None:
    if code != 0:
        raise FA2Error(func, code)


_DTYPES = {torch.float16: 0, torch.bfloat16: 1}


def _stream_ptr(dev: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _shape(q: torch.Tensor):
    if q.dim() != 4:
        raise ValueError("expected a [B, H, N, d] tensor")
    return tuple(int(x) for x in q.shape)


def _check_tensor(name, t, shape, dtype, device):
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name} must have shape {tuple(shape)} and dtype {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_host(name, t, shape, dtype):
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name} must have shape {tuple(shape)} and dtype {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def num_splits(B: int, H: int, N: int, d: int, causal: bool, num_sms: int) -> int:
    """The K/V split count ``fa2_fwd_split`` would use for this shape on a GPU
    with ``num_sms`` SMs (host-only rule of the library)."""
    return int(load_library().fa2_num_splits(B, H, N, d, int(bool(causal)), num_sms))


def forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
            num_splits: int | str = "auto"):
    """O = softmax(scale * Q K^T [+ causal mask]) V and its logsumexp L.

    ``num_splits`` > 1 cuts each worker's K/V range into that many parts run by
    separate CTAs and merges them (fa2_fwd_split); "auto" (the default) takes
    the library's rule for this GPU (fa2_num_splits), which keeps 1 unless the
    unsplit launch leaves the SMs underused; 1 always runs fa2_fwd. k and v
    may have their own length N_k (fa2_fwd_qk, never split; causal mask
    top-left: query i sees keys 0..i). Returns (o, lse): o like q, lse
    float32 [B, H, N] (natural log).
    """
    B, H, N, d = _shape(q)
    Nk = _shape(k)[2]
    dt = q.dtype
    if dt not in _DTYPES:
        raise ValueError("q must be float16 or bfloat16")
    dev = q.device
    _check_tensor("q", q, (B, H, N, d), dt, dev)
    for name, t in (("k", k), ("v", v)):
        _check_tensor(name, t, (B, H, Nk, d), dt, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    _check_tensor("out", out, (B, H, N, d), dt, dev)
    _check_tensor("lse", lse, (B, H, N), torch.float32, dev)
    lib = load_library()
    if Nk != N:
        if num_splits not in (1, "auto"):
            raise ValueError("a K/V split needs equal query and key lengths")
        code = lib.fa2_fwd_qk(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr(), B, H, N, Nk, d, int(bool(causal)), float(scale),
                              _DTYPES[dt], _stream_ptr(dev))
        _check("fa2_fwd_qk", code)
        return out, lse
    if num_splits == "auto":
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        num_splits = int(lib.fa2_num_splits(B, H, N, d, int(bool(causal)), sms))
    num_splits = int(num_splits)
    if num_splits > 1:
        nbytes = lib.fa2_fwd_split_workspace_size(B, H, N, d, num_splits)
        if nbytes == 0:
            raise FA2Error("fa2_fwd_split_workspace_size", 1)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        code = lib.fa2_fwd_split(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 lse.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                 _DTYPES[dt], num_splits, ws.data_ptr(), nbytes, _stream_ptr(dev))
        _check("fa2_fwd_split", code)
        return out, lse
    code = lib.fa2_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, H, N, d, int(bool(causal)), float(scale), _DTYPES[dt], _stream_ptr(dev))
    _check("fa2_fwd", code)
    return out, lse


def forward_kv_outer(q, k, v, causal: bool = False, scale: float | None = None):
    """The same (o, lse) as ``forward``, computed in the FlashAttention-1 loop
    order (fa2_fwd_kv_outer: K/V blocks outer, the running O, m, l of every
    query block read from and written back to HBM at each step). For
    measuring the loop order; ``forward`` is the fast path."""
    B, H, N, d = _shape(q)
    dt = q.dtype
    if dt not in _DTYPES:
        raise ValueError("q must be float16 or bfloat16")
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t, (B, H, N, d), dt, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lib = load_library()
    nbytes = lib.fa2_fwd_kv_outer_workspace_size(B, H, N, d)
    if nbytes == 0:
        raise FA2Error("fa2_fwd_kv_outer_workspace_size", 1)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    code = lib.fa2_fwd_kv_outer(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                lse.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                _DTYPES[dt], ws.data_ptr(), nbytes, _stream_ptr(dev))
    _check("fa2_fwd_kv_outer", code)
    return out, lse


def step_host(q, k, v, do, causal: bool = False, scale: float | None = None,
              heads_per_chunk: int = 0, device=None, out=None, workspace=None):
    """Forward + backward on host (CPU) tensors through fa2_step_host: the
    copies to and from ``device`` overlap the kernels, chunk by chunk of heads.
    Inputs should be pinned. Returns host tensors (o, lse, dq, dk, dv); with
    ``out`` = that 5-tuple of host tensors, writes into them. Synchronises
    the device's current stream before returning."""
    B, H, N, d = _shape(q)
    dt = q.dtype
    if dt not in _DTYPES:
        raise ValueError("q must be float16 or bfloat16")
    for name, t in (("q", q), ("k", k), ("v", v), ("do", do)):
        _check_host(name, t, (B, H, N, d), dt)
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        pin = q.is_pinned()
        o, dq, dk, dv = (torch.empty(q.shape, dtype=dt, pin_memory=pin) for _ in range(4))
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    else:
        o, lse, dq, dk, dv = out
    for name, t in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_host(name, t, (B, H, N, d), dt)
    _check_host("lse", lse, (B, H, N), torch.float32)
    lib = load_library()
    nbytes = lib.fa2_step_host_workspace_size(B, H, N, d, int(heads_per_chunk))
    if nbytes == 0:
        raise FA2Error("fa2_step_host_workspace_size", 1)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        code = lib.fa2_step_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                 o.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                 dv.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                 _DTYPES[dt], int(heads_per_chunk), workspace.data_ptr(),
                                 workspace.numel(), _stream_ptr(dev))
        _check("fa2_step_host", code)
        torch.cuda.current_stream(dev).synchronize()
    return o, lse, dq, dk, dv


def forward_instrumented(q, k, v, causal=False, scale=None):
    """``forward`` that also returns, per forward CTA (grid order), the number of
    K/V tiles it loaded (an int32 CUDA tensor)."""
    B, H, N, d = _shape(q)
    dev = q.device
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    gx, gy, gz = fwd_grid(B, H, N)[0]
    counts = torch.full((gx * gy * gz,), -1, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    lib = load_library()
    code = lib.fa2_fwd_instrumented(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                    _DTYPES[q.dtype], counts.data_ptr(), _stream_ptr(dev))
    _check("fa2_fwd_instrumented", code)
    return out, lse, counts


def bwd_workspace_size(B: int, H: int, N: int, d: int, atomic: bool = False) -> int:
    lib = load_library()
    if atomic:
        return int(lib.fa2_bwd_atomic_workspace_size(B, H, N, d))
    return int(lib.fa2_bwd_workspace_size(B, H, N, d))


def backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None,
             dq=None, dk=None, dv=None, workspace=None, atomic: bool = False):
    """Gradients (dq, dk, dv) of the attention output given dO. k and v may
    have their own length N_k (fa2_bwd_qk). ``atomic`` runs fa2_bwd_atomic,
    the column-worker variant with fp32 dQ reduce-adds (equal lengths only)."""
    B, H, N, d = _shape(q)
    Nk = _shape(k)[2]
    dt = q.dtype
    if dt not in _DTYPES:
        raise ValueError("q must be float16 or bfloat16")
    dev = q.device
    for name, t in (("q", q), ("o", o), ("do", do)):
        _check_tensor(name, t, (B, H, N, d), dt, dev)
    for name, t in (("k", k), ("v", v)):
        _check_tensor(name, t, (B, H, Nk, d), dt, dev)
    _check_tensor("lse", lse, (B, H, N), torch.float32, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_tensor("dq", dq, (B, H, N, d), dt, dev)
    for name, t in (("dk", dk), ("dv", dv)):
        _check_tensor(name, t, (B, H, Nk, d), dt, dev)
    need = bwd_workspace_size(B, H, N, d, atomic)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    lib = load_library()
    if atomic:
        if Nk != N:
            raise ValueError("fa2_bwd_atomic needs equal query and key lengths")
        code = lib.fa2_bwd_atomic(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                  dv.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                  _DTYPES[dt], workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), _stream_ptr(dev))
        _check("fa2_bwd_atomic", code)
        return dq, dk, dv
    if Nk != N:
        code = lib.fa2_bwd_qk(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), B, H, N, Nk, d, int(bool(causal)), float(scale),
                              _DTYPES[dt], workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream_ptr(dev))
        _check("fa2_bwd_qk", code)
        return dq, dk, dv
    code = lib.fa2_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                       int(bool(causal)), float(scale), _DTYPES[dt], workspace.data_ptr(),
                       workspace.numel() * workspace.element_size(), _stream_ptr(dev))
    _check("fa2_bwd", code)
    return dq, dk, dv


def device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    lib = load_library()
    s = ctypes.c_void_p(stream.cuda_stream if stream is not None else
                        torch.cuda.current_stream().cuda_stream)
    return int(lib.fa2_get_device_status(s))


def _ints(n):
    return [ctypes.c_int(0) for _ in range(n)]


def fwd_grid(B: int, H: int, N: int):
    """((grid_x, grid_y, grid_z), rows_per_cta) of the forward launch."""
    g = (ctypes.c_int * 3)()
    rows = ctypes.c_int(0)
    _check("fa2_fwd_grid", load_library().fa2_fwd_grid(B, H, N, g, ctypes.byref(rows)))
    return (g[0], g[1], g[2]), rows.value


def fwd_block_work(block_x: int, N: int, causal: bool):
    """(row_begin, row_end, kv_tiles) of forward row block ``block_x``."""
    a, b, c = _ints(3)
    _check("fa2_fwd_block_work", load_library().fa2_fwd_block_work(
        block_x, N, int(bool(causal)), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c)))
    return a.value, b.value, c.value


def fwd_schedule(B: int, H: int, N: int, causal: bool, num_sms: int):
    """(num_ctas, cta_of_block, pos_of_block) of the unsplit forward's
    persistent grid on ``num_sms`` multiprocessors; the lists are in
    ``fwd_grid`` order (row block fastest, then batch, then head)."""
    n = load_library()
    nb = B * H * fwd_grid(1, 1, N)[0][0]
    g = ctypes.c_int()
    cta = (ctypes.c_int * nb)()
    pos = (ctypes.c_int * nb)()
    _check("fa2_fwd_schedule", n.fa2_fwd_schedule(B, H, N, int(bool(causal)), num_sms,
                                                  ctypes.byref(g), cta, pos))
    return g.value, list(cta), list(pos)


def bwd_grid(B: int, H: int, N: int, d: int):
    """((grid_x, grid_y, grid_z), keys_per_cta, q_rows_per_tile) of the dK/dV launch."""
    g = (ctypes.c_int * 3)()
    kp, qr = _ints(2)
    _check("fa2_bwd_grid", load_library().fa2_bwd_grid(B, H, N, d, g, ctypes.byref(kp),
                                                        ctypes.byref(qr)))
    return (g[0], g[1], g[2]), kp.value, qr.value


def bwd_block_work(block_x: int, N: int, d: int, causal: bool):
    """(key_begin, key_end, q_tile_begin, q_tile_end) of dK/dV column block ``block_x``."""
    a, b, c, e = _ints(4)
    _check("fa2_bwd_block_work", load_library().fa2_bwd_block_work(
        block_x, N, d, int(bool(causal)), ctypes.byref(a), ctypes.byref(b), ctypes.byref(c),
        ctypes.byref(e)))
    return a.value, b.value, c.value, e.value


class _FA2Function(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale):
        o, lse = forward(q, k, v, causal=causal, scale=scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale = causal, scale
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = backward(q, k, v, o, lse, do.contiguous(), causal=ctx.causal,
                              scale=ctx.scale)
        return dq, dk, dv, None, None


def attention(q, k, v, causal: bool = False, scale: float | None = None):
    """Differentiable FlashAttention-2 (forward and backward in libfa2)."""
    return _FA2Function.apply(q, k, v, causal, scale)
