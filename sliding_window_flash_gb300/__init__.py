"""Python binding of libswa.so: causal sliding-window attention with grouped-query heads for
training, forward and backward, hand-written for GB300 (sm_103a).

The binding only marshals arguments: torch tensors become device pointers and the current CUDA
stream becomes ``cudaStream_t``; every step of the computation runs in the library's kernels.
PyTorch owns all device memory (outputs and the backward workspace are allocated here with torch).
There is no fallback: if libswa.so is missing or the device is not sm_103, the calls raise.

    o, lse = swa_attn_fwd(q, k, v, window, scale)
    dq, dk, dv = swa_attn_bwd(q, k, v, o, do, lse, window, scale)
    out = SlidingWindowAttention.apply(q, k, v, window, scale)   # autograd wrapper

Layout: q, o, do, dq [B, Hq, Lq, D]; k, v, dk, dv [B, Hkv, Lk, D], all contiguous and of one
dtype (bf16, fp16, or fp32 with bf16 tensor-core operands); lse [B, Hq, Lq] fp32.
D in {64, 128, 256}; Hq % Hkv == 0; Lq <= Lk (the queries are the last Lq key positions).
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

__all__ = [
    "load",
    "library_path",
    "SwaError",
    "swa_attn_fwd",
    "swa_attn_bwd",
    "swa_attn_bwd_workspace_bytes",
    "swa_attn_bwd_fused_workspace_bytes",
    "swa_attn_f32_workspace_bytes",
    "swa_attn_fwd_bwd_host",
    "swa_attn_host_workspace_bytes",
    "swa_attn_bwd_phases",
    "swa_check_device",
    "SlidingWindowAttention",
    "STATUS",
]

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libswa.so"
_lib: Optional[ctypes.CDLL] = None

STATUS = {
    0: "SWA_OK",
    1: "SWA_ERR_INVALID_ARG",
    2: "SWA_ERR_UNSUPPORTED",
    3: "SWA_ERR_MISALIGNED",
    4: "SWA_ERR_CUDA",
    5: "SWA_ERR_DEVICE_TIMEOUT",
    6: "SWA_ERR_WORKSPACE",
    7: "SWA_ERR_DEVICE_LAYOUT",
}

# Every symbol include/swa_attn.h declares, with its ctypes signature.
_c_int, _c_float, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
SIGNATURES = {
    "swa_attn_fwd": (_c_int, [_vp] * 5 + [_c_int] * 6 + [_c_float, _vp]),
    "swa_attn_fwd_f16": (_c_int, [_vp] * 5 + [_c_int] * 6 + [_c_float, _vp]),
    "swa_attn_fwd_ex": (_c_int, [_vp] * 5 + [_c_int] * 8 + [_c_float, _c_int, _vp]),
    "swa_attn_bwd_workspace_bytes": (ctypes.c_size_t, [_c_int] * 4),
    "swa_attn_bwd": (
        _c_int,
        [_vp] * 9 + [_c_int] * 6 + [_c_float, _vp, ctypes.c_size_t, _vp],
    ),
    "swa_attn_bwd_f16": (
        _c_int,
        [_vp] * 9 + [_c_int] * 6 + [_c_float, _vp, ctypes.c_size_t, _vp],
    ),
    "swa_attn_bwd_ex": (
        _c_int,
        [_vp] * 9 + [_c_int] * 8 + [_c_float, _c_int, _vp, ctypes.c_size_t, _vp],
    ),
    "swa_attn_f32_workspace_bytes": (ctypes.c_size_t, [_c_int] * 6),
    "swa_attn_fwd_f32": (_c_int, [_vp] * 5 + [_c_int] * 8 + [_c_float, _vp, ctypes.c_size_t, _vp]),
    "swa_attn_bwd_f32": (_c_int, [_vp] * 9 + [_c_int] * 8 + [_c_float, _vp, ctypes.c_size_t, _vp]),
    "swa_attn_host_workspace_bytes": (ctypes.c_size_t, [_c_int] * 6),
    "swa_attn_fwd_bwd_host": (
        _c_int,
        [_vp] * 9 + [_c_int] * 6 + [_c_float, _c_int, _vp, ctypes.c_size_t, _vp],
    ),
    "swa_attn_bwd_preprocess": (_c_int, [_vp] * 3 + [_c_int] * 4 + [_vp]),
    "swa_attn_bwd_dkdv": (_c_int, [_vp] * 8 + [_c_int] * 6 + [_c_float, _vp]),
    "swa_attn_bwd_dq": (_c_int, [_vp] * 7 + [_c_int] * 6 + [_c_float, _vp]),
    "swa_attn_bwd_noalloc": (_c_int, [_vp] * 9 + [_c_int] * 6 + [_c_float, _vp]),
    "swa_attn_bwd_fused_workspace_bytes": (ctypes.c_size_t, [_c_int] * 4),
    "swa_attn_bwd_fused": (
        _c_int,
        [_vp] * 9 + [_c_int] * 8 + [_c_float, _c_int, _vp, ctypes.c_size_t, _vp],
    ),
    "swa_attn_bwd_fused_preprocess": (_c_int, [_vp] * 3 + [ctypes.c_size_t] + [_c_int] * 4 + [_vp]),
    "swa_attn_bwd_fused_dkdv": (
        _c_int,
        [_vp] * 8 + [ctypes.c_size_t] + [_c_int] * 6 + [_c_float, _vp],
    ),
    "swa_attn_bwd_fused_dq": (_c_int, [_vp] * 2 + [ctypes.c_size_t] + [_c_int] * 4 + [_c_float, _vp]),
    "swa_strerror": (ctypes.c_char_p, [_c_int]),
    "swa_check_device": (_c_int, [_vp]),
    "swa_selftest_wait_timeout": (_c_int, [_vp]),
    "swa_version": (_c_int, []),
}


class SwaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = STATUS.get(code, f"status {code}")
        if _lib is not None:
            msg = _lib.swa_strerror(code).decode()
        super().__init__(f"{where}: {msg}")


def library_path() -> str:
    return os.path.join(_PKG_DIR, _LIB_NAME)


def load() -> ctypes.CDLL:
    """Load libswa.so (built in-tree by ``sliding_window_flash_gb300.build``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} not found: build it with `python -m sliding_window_flash_gb300.build` "
            "(there is no CPU or PyTorch fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _stream_handle(device) -> int:
    import torch

    return torch.cuda.current_stream(device).cuda_stream


def _check_tensor(t, name, shape, dtype):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _dims(q, k):
    """(B, Hq, Hkv, Lq, Lk, D) of q [B, Hq, Lq, D] and k [B, Hkv, Lk, D]."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be 4-D [B, H, L, D]")
    B, Hq, Lq, D = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    return B, Hq, Hkv, Lq, Lk, D


def _scale(scale, D):
    return float(scale) if scale is not None else 1.0 / math.sqrt(D)


def _elem_dtype(q):
    """Element type of a call, taken from q: bf16, fp16 (the *_f16 entry points) or fp32 (the
    *_f32 entry points: operands rounded to bf16 on the device, results widened to fp32)."""
    import torch

    if q.dtype not in (torch.bfloat16, torch.float16, torch.float32):
        raise TypeError(f"q must be bfloat16, float16 or float32, got {q.dtype}")
    return q.dtype


def swa_attn_f32_workspace_bytes(B: int, Hq: int, Hkv: int, Lq: int, Lk: int, D: int) -> int:
    return int(load().swa_attn_f32_workspace_bytes(B, Hq, Hkv, Lq, Lk, D))


def _f32_workspace(workspace, B, Hq, Hkv, Lq, Lk, D, device):
    import torch

    n = swa_attn_f32_workspace_bytes(B, Hq, Hkv, Lq, Lk, D)
    if workspace is None:
        workspace = torch.empty(n, dtype=torch.uint8, device=device)
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def swa_attn_fwd(q, k, v, window: int, scale: Optional[float] = None, out=None, lse=None,
                 causal: bool = True, workspace=None):
    """Forward: returns (o [B,Hq,Lq,D] in q's dtype (bf16, fp16 or fp32), lse [B,Hq,Lq] fp32).

    q [B,Hq,Lq,D], k and v [B,Hkv,Lk,D] with Lq <= Lk: the queries are the last Lq positions of the
    keys.  causal=False selects the two-sided window |pos - j| < window.  fp32 calls use a device
    workspace of swa_attn_f32_workspace_bytes (allocated here unless given).
    """
    import torch

    lib = load()
    B, Hq, Hkv, Lq, Lk, D = _dims(q, k)
    dt = _elem_dtype(q)
    _check_tensor(q, "q", (B, Hq, Lq, D), dt)
    _check_tensor(k, "k", (B, Hkv, Lk, D), dt)
    _check_tensor(v, "v", (B, Hkv, Lk, D), dt)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Lq), dtype=torch.float32, device=q.device)
    _check_tensor(out, "out", (B, Hq, Lq, D), dt)
    _check_tensor(lse, "lse", (B, Hq, Lq), torch.float32)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr())
    f16 = dt == torch.float16
    st = _stream_handle(q.device)
    if dt == torch.float32:
        name = "swa_attn_fwd_f32"
        ws = _f32_workspace(workspace, B, Hq, Hkv, Lq, Lk, D, q.device)
        rc = lib.swa_attn_fwd_f32(*ptrs, B, Hq, Hkv, Lq, Lk, D, int(window), int(bool(causal)),
                                  _scale(scale, D), *ws, st)
    elif Lq == Lk and causal:
        name = "swa_attn_fwd_f16" if f16 else "swa_attn_fwd"
        rc = getattr(lib, name)(*ptrs, B, Hq, Hkv, Lq, D, int(window), _scale(scale, D), st)
    else:
        name = "swa_attn_fwd_ex"
        rc = lib.swa_attn_fwd_ex(*ptrs, B, Hq, Hkv, Lq, Lk, D, int(window), int(bool(causal)),
                                 _scale(scale, D), int(f16), st)
    if rc != 0:
        raise SwaError(rc, name)
    return out, lse


def swa_attn_bwd_workspace_bytes(B: int, Hq: int, N: int, D: int) -> int:
    return int(load().swa_attn_bwd_workspace_bytes(B, Hq, N, D))


def swa_attn_bwd_fused_workspace_bytes(B: int, Hq: int, Lq: int, D: int) -> int:
    return int(load().swa_attn_bwd_fused_workspace_bytes(B, Hq, Lq, D))


def swa_attn_bwd(q, k, v, o, do, lse, window: int, scale: Optional[float] = None,
                 dq=None, dk=None, dv=None, workspace=None, causal: bool = True,
                 fused: bool = False) -> Tuple:
    """Backward of sum(do * o): returns (dq, dk, dv) in q's dtype (bf16, fp16 or fp32), dk/dv
    summed over each kv group.  Shapes, window and workspace as in swa_attn_fwd.

    bf16 / fp16: ``fused=False`` (default) runs the split, bit-reproducible swa_attn_bwd /
    swa_attn_bwd_ex (workspace of swa_attn_bwd_workspace_bytes), the faster path on GB300;
    ``fused=True`` runs swa_attn_bwd_fused (one kernel for dK, dV and dQ; workspace of
    swa_attn_bwd_fused_workspace_bytes; dQ's fp32 additions run in a varying order).  fp32 tensors
    always take the split path."""
    import torch

    lib = load()
    B, Hq, Hkv, Lq, Lk, D = _dims(q, k)
    dt = _elem_dtype(q)
    for t, name, hs, L in ((q, "q", Hq, Lq), (k, "k", Hkv, Lk), (v, "v", Hkv, Lk), (o, "o", Hq, Lq),
                           (do, "do", Hq, Lq)):
        _check_tensor(t, name, (B, hs, L, D), dt)
    _check_tensor(lse, "lse", (B, Hq, Lq), torch.float32)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, name, hs, L in ((dq, "dq", Hq, Lq), (dk, "dk", Hkv, Lk), (dv, "dv", Hkv, Lk)):
        _check_tensor(t, name, (B, hs, L, D), dt)
    ptrs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(), lse.data_ptr(),
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr())
    f16 = dt == torch.float16
    st = _stream_handle(q.device)
    if dt == torch.float32:
        name = "swa_attn_bwd_f32"
        ws = _f32_workspace(workspace, B, Hq, Hkv, Lq, Lk, D, q.device)
        rc = lib.swa_attn_bwd_f32(*ptrs, B, Hq, Hkv, Lq, Lk, D, int(window), int(bool(causal)),
                                  _scale(scale, D), *ws, st)
        if rc != 0:
            raise SwaError(rc, name)
        return dq, dk, dv
    if fused:
        ws_bytes = int(lib.swa_attn_bwd_fused_workspace_bytes(B, Hq, Lq, D))
    else:
        ws_bytes = int(lib.swa_attn_bwd_workspace_bytes(B, Hq, Lq, D))
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    if fused:
        name = "swa_attn_bwd_fused"
        rc = lib.swa_attn_bwd_fused(*ptrs, B, Hq, Hkv, Lq, Lk, D, int(window), int(bool(causal)),
                                    _scale(scale, D), int(f16), *ws, st)
    elif Lq == Lk and causal:
        name = "swa_attn_bwd_f16" if f16 else "swa_attn_bwd"
        rc = getattr(lib, name)(*ptrs, B, Hq, Hkv, Lq, D, int(window), _scale(scale, D), *ws, st)
    else:
        name = "swa_attn_bwd_ex"
        rc = lib.swa_attn_bwd_ex(*ptrs, B, Hq, Hkv, Lq, Lk, D, int(window), int(bool(causal)),
                                 _scale(scale, D), int(f16), *ws, st)
    if rc != 0:
        raise SwaError(rc, name)
    return dq, dk, dv


def swa_attn_bwd_phases(q, k, v, o, do, lse, window: int, scale: Optional[float] = None,
                        dq=None, dk=None, dv=None, delta=None, between=None, fused: bool = False,
                        workspace=None) -> Tuple:
    """The backward as its three C-ABI phases on the current stream: split (preprocess, dK/dV,
    dQ; ``delta`` is the Delta buffer) or, with ``fused=True``, the fused backward's (preprocess
    with the accumulator zeroed, the fused dK/dV/dQ kernel, dQ from the accumulator;
    ``workspace`` as for swa_attn_bwd_fused).  Same kernels and results as swa_attn_bwd.
    ``between(i)`` (optional) is called before phase i and after the last one (i = 0..3), e.g. to
    record CUDA events around each kernel.
    """
    if fused:
        return _fused_phases(q, k, v, o, do, lse, window, scale, dq, dk, dv, workspace, between)
    import torch

    lib = load()
    B, Hq, Hkv, N, Lk, D = _dims(q, k)
    if Lk != N:
        raise ValueError("the phase entry points take equal query and key lengths")
    sc = _scale(scale, D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if delta is None:
        delta = torch.empty((B, Hq, N), dtype=torch.float32, device=q.device)
    for t, name, hs in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq),
                        (dq, "dq", Hq), (dk, "dk", Hkv), (dv, "dv", Hkv)):
        _check_tensor(t, name, (B, hs, N, D), torch.bfloat16)
    _check_tensor(lse, "lse", (B, Hq, N), torch.float32)
    _check_tensor(delta, "delta", (B, Hq, N), torch.float32)
    st = _stream_handle(q.device)
    mark = between or (lambda i: None)
    mark(0)
    rc = lib.swa_attn_bwd_preprocess(o.data_ptr(), do.data_ptr(), delta.data_ptr(), B, Hq, N, D, st)
    if rc != 0:
        raise SwaError(rc, "swa_attn_bwd_preprocess")
    mark(1)
    rc = lib.swa_attn_bwd_dkdv(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), lse.data_ptr(),
                               delta.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, N, D,
                               int(window), sc, st)
    if rc != 0:
        raise SwaError(rc, "swa_attn_bwd_dkdv")
    mark(2)
    rc = lib.swa_attn_bwd_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(), lse.data_ptr(),
                             delta.data_ptr(), dq.data_ptr(), B, Hq, Hkv, N, D, int(window), sc, st)
    if rc != 0:
        raise SwaError(rc, "swa_attn_bwd_dq")
    mark(3)
    return dq, dk, dv


def _fused_phases(q, k, v, o, do, lse, window, scale, dq, dk, dv, workspace, between):
    import torch

    lib = load()
    B, Hq, Hkv, N, Lk, D = _dims(q, k)
    if Lk != N:
        raise ValueError("the phase entry points take equal query and key lengths")
    sc = _scale(scale, D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, name, hs in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (o, "o", Hq), (do, "do", Hq),
                        (dq, "dq", Hq), (dk, "dk", Hkv), (dv, "dv", Hkv)):
        _check_tensor(t, name, (B, hs, N, D), torch.bfloat16)
    _check_tensor(lse, "lse", (B, Hq, N), torch.float32)
    n = int(lib.swa_attn_bwd_fused_workspace_bytes(B, Hq, N, D))
    if workspace is None:
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device)
    ws = (workspace.data_ptr(), workspace.numel() * workspace.element_size())
    st = _stream_handle(q.device)
    mark = between or (lambda i: None)
    mark(0)
    rc = lib.swa_attn_bwd_fused_preprocess(o.data_ptr(), do.data_ptr(), *ws, B, Hq, N, D, st)
    if rc != 0:
        raise SwaError(rc, "swa_attn_bwd_fused_preprocess")
    mark(1)
    rc = lib.swa_attn_bwd_fused_dkdv(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                     lse.data_ptr(), dk.data_ptr(), dv.data_ptr(), *ws, B, Hq, Hkv,
                                     N, D, int(window), sc, st)
    if rc != 0:
        raise SwaError(rc, "swa_attn_bwd_fused_dkdv")
    mark(2)
    rc = lib.swa_attn_bwd_fused_dq(dq.data_ptr(), *ws, B, Hq, N, D, sc, st)
    if rc != 0:
        raise SwaError(rc, "swa_attn_bwd_fused_dq")
    mark(3)
    return dq, dk, dv


def swa_attn_host_workspace_bytes(B: int, Hq: int, Hkv: int, N: int, D: int,
                                  units_per_chunk: int) -> int:
    return int(load().swa_attn_host_workspace_bytes(B, Hq, Hkv, N, D, units_per_chunk))


def default_units_per_chunk(B: int, Hkv: int) -> int:
    """About sixteen chunks of (batch, kv head) groups per call (on the N=32768 layer, one group
    per chunk with three buffer sets measured fastest: 5.56 ms against 6.2-6.7 ms for 2-4)."""
    return max(1, -(-(B * Hkv) // 16))


def swa_attn_fwd_bwd_host(q, k, v, do, window: int, scale: Optional[float] = None,
                          outs=None, units_per_chunk: Optional[int] = None, workspace=None,
                          device=None) -> Tuple:
    """Forward and backward of one layer whose tensors live in host memory (equal lengths, causal
    window): returns (o, lse, dq, dk, dv) as host tensors, filled asynchronously on the current
    stream of `device` (synchronize before reading them).

    q, do [B,Hq,N,D] and k, v [B,Hkv,N,D] are CPU tensors, pinned for the copies to overlap the
    kernels; `outs` (o, lse, dq, dk, dv) are pinned CPU tensors allocated here unless given.  The
    library copies (batch, kv head) groups in chunks and runs the same kernels on each chunk while
    the next one is copied in and the previous one out.
    """
    import torch

    lib = load()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    B, Hq, Hkv, N, Lk, D = _dims(q, k)
    dt = q.dtype
    if dt != torch.bfloat16:
        raise TypeError("the host pipeline takes bf16 tensors")
    for t, name, hs in ((q, "q", Hq), (k, "k", Hkv), (v, "v", Hkv), (do, "do", Hq)):
        if t.device.type != "cpu" or t.dtype != dt or tuple(t.shape) != (B, hs, N, D) or \
                not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU {dt} tensor [B, {hs}, N, D]")
    if outs is None:
        outs = (torch.empty_like(q).pin_memory(),
                torch.empty((B, Hq, N), dtype=torch.float32).pin_memory(),
                torch.empty_like(q).pin_memory(), torch.empty_like(k).pin_memory(),
                torch.empty_like(v).pin_memory())
    U = default_units_per_chunk(B, Hkv) if units_per_chunk is None else int(units_per_chunk)
    n = swa_attn_host_workspace_bytes(B, Hq, Hkv, N, D, U)
    if workspace is None:
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
    ptrs = [t.data_ptr() for t in (q, k, v, do)] + [t.data_ptr() for t in outs]
    rc = lib.swa_attn_fwd_bwd_host(*ptrs, B, Hq, Hkv, N, D, int(window), _scale(scale, D), U,
                                   workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(),
                                   _stream_handle(dev))
    if rc != 0:
        raise SwaError(rc, "swa_attn_fwd_bwd_host")
    return tuple(outs)


def swa_check_device(device=None) -> None:
    """Synchronize the current stream and raise if a kernel's bounded wait ran out."""
    import torch

    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    rc = load().swa_check_device(_stream_handle(dev))
    if rc != 0:
        raise SwaError(rc, "swa_check_device")


def _make_autograd():
    import torch

    class SlidingWindowAttention(torch.autograd.Function):
        """o = attention(q, k, v) under a sliding window (causal unless causal=False); saves only
        (o, lse) for the backward."""

        @staticmethod
        def forward(ctx, q, k, v, window: int, scale: Optional[float] = None, causal: bool = True):
            o, lse = swa_attn_fwd(q, k, v, window, scale, causal=causal)
            ctx.save_for_backward(q, k, v, o, lse)
            ctx.window, ctx.scale, ctx.causal = window, scale, causal
            return o

        @staticmethod
        def backward(ctx, do):
            q, k, v, o, lse = ctx.saved_tensors
            dq, dk, dv = swa_attn_bwd(q, k, v, o, do.contiguous(), lse, ctx.window, ctx.scale,
                                      causal=ctx.causal)
            return dq, dk, dv, None, None, None

    return SlidingWindowAttention


class _LazyAutograd:
    _cls = None

    def __getattr__(self, name):
        if _LazyAutograd._cls is None:
            _LazyAutograd._cls = _make_autograd()
        return getattr(_LazyAutograd._cls, name)


SlidingWindowAttention = _LazyAutograd()
