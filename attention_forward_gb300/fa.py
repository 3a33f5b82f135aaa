"""ctypes binding of libfa_gb300.so -- argument marshalling only.

Every function here has the name of the C entry point it calls (declared in
include/fa.h).  Tensors are torch tensors used as device (or pinned host)
memory; all computation happens in the library's CUDA kernels.  There is no
fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                         "libfa_gb300.so")
_lib = None

FA_F16, FA_BF16 = 0, 1
FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED = 0, 1, 2
FA_ERR_CUDA, FA_ERR_WORKSPACE, FA_ERR_TIMEOUT = 3, 4, 5
FA_FLAG_NO_LPT = 0x1
FA_FLAG_ALWAYS_RESCALE = 0x2
FA_FLAG_EXACT_MAX = 0x4
FA_FLAG_PAIR = 0x8
FA_FLAG_SINGLE_CTA = 0x10
FA_FLAG_CORRECTION_WG = 0x20
FA_FLAG_PAIR64 = 0x40
FA_FLAG_OVERLAP_PREVIOUS = 0x80
FA_FLAG_TEST_STALL = 0x100
FA_FLAG_TAIL_SPLIT = 0x200
FA_FLAG_D64_THREE_STAGE = 0x400

_DTYPE = {torch.float16: FA_F16, torch.bfloat16: FA_BF16}


class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {fa_status_string(status)} (status {status})")


def lib_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load the library; raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = load_path(_LIB_PATH)
    return _lib


def load_path(path: str) -> ctypes.CDLL:
    """Load a build of the library from ``path`` (the in-tree one, or
    another build of the same sources, e.g. a variant compared against it
    in a paired measurement).  Each build loads as its own module, with its
    own device state."""
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(path)
    vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, ci, vp]
    L.fa_fwd.restype = ci
    L.fa_workspace_bytes.argtypes = [ci, ci, ci, ci, ci, ci]
    L.fa_workspace_bytes.restype = sz
    L.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci, ci,
                            ctypes.c_uint, ci, vp, sz, vp]
    L.fa_fwd_ex.restype = ci
    L.fa_host_staging_bytes.argtypes = [ci, ci, ci, ci, ci]
    L.fa_host_staging_bytes.restype = sz
    L.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, cf, ci,
                              ci, vp, sz, vp]
    L.fa_fwd_host.restype = ci
    L.fa_fwd_decode_static.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf,
                                       ci, vp]
    L.fa_fwd_decode_static.restype = ci
    L.fa_release_workspaces.argtypes = []
    L.fa_release_workspaces.restype = ci
    L.fa_get_device_status.argtypes = [vp]
    L.fa_get_device_status.restype = ci
    L.fa_set_watchdog_ns.argtypes = [ctypes.c_ulonglong]
    L.fa_set_watchdog_ns.restype = None
    L.fa_status_string.argtypes = [ci]
    L.fa_status_string.restype = ctypes.c_char_p
    L.fa_prefill_uses_pairs.argtypes = [ci, ci, ci, ci, ci, ci, ctypes.c_uint, ci]
    L.fa_prefill_uses_pairs.restype = ci
    L.fa_ex2_approx.argtypes = [vp, vp, ci, vp]
    L.fa_ex2_approx.restype = ci
    L.fa_prefill_tail_items.argtypes = [ci, ci, ci, ci, ci, ci, ci, ctypes.c_uint]
    L.fa_prefill_tail_items.restype = ci
    L.fa_version.argtypes = []
    L.fa_version.restype = ci
    return L


def _stream_handle(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _shape(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, H, S, D]")
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    if k.shape != (B, H, Skv, D) or v.shape != (B, H, Skv, D):
        raise ValueError("k and v must be [B, H, Skv, D] matching q")
    if q.dtype not in _DTYPE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share dtype float16 or bfloat16")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    return B, H, Sq, Skv, D


def _outputs(q, out, lse):
    B, H, Sq, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous():
        raise ValueError("out must match q")
    if lse.shape != (B, H, Sq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be float32 [B, H, Sq]")
    return out, lse


def _check(status: int, what: str) -> None:
    if status != FA_OK:
        raise FAError(status, what)


def fa_fwd(q, k, v, causal: bool = False, scale: float | None = None,
           out=None, lse=None, stream=None, lib=None):
    """O, LSE = attention(q, k, v) on the library's kernels.  Returns (o, lse).
    ``lib``: another loaded build (load_path); default the in-tree one."""
    B, H, Sq, Skv, D = _shape(q, k, v)
    out, lse = _outputs(q, out, lse)
    sc = float(D) ** -0.5 if scale is None else float(scale)
    st = (lib or load()).fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                       lse.data_ptr(), B, H, Sq, Skv, D, sc, int(bool(causal)),
                       _DTYPE[q.dtype], _stream_handle(stream))
    _check(st, "fa_fwd")
    return out, lse


def fa_workspace_bytes(B: int, H: int, Sq: int, Skv: int, D: int,
                       num_splits: int = 0) -> int:
    return int(load().fa_workspace_bytes(B, H, Sq, Skv, D, num_splits))


def fa_fwd_ex(q, k, v, causal: bool = False, scale: float | None = None,
              flags: int = 0, num_splits: int = 0, workspace=None, out=None,
              lse=None, stream=None, lib=None):
    """fa_fwd with flags, an explicit decode split count and a caller-owned
    workspace tensor (any dtype, on the device)."""
    B, H, Sq, Skv, D = _shape(q, k, v)
    out, lse = _outputs(q, out, lse)
    sc = float(D) ** -0.5 if scale is None else float(scale)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr = workspace.data_ptr()
        ws_bytes = workspace.numel() * workspace.element_size()
    st = (lib or load()).fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                          out.data_ptr(), lse.data_ptr(), B, H, Sq, Skv, D, sc,
                          int(bool(causal)), _DTYPE[q.dtype], int(flags),
                          int(num_splits), ws_ptr, ws_bytes,
                          _stream_handle(stream))
    _check(st, "fa_fwd_ex")
    return out, lse


def fa_host_staging_bytes(B: int, H: int, Sq: int, Skv: int, D: int) -> int:
    return int(load().fa_host_staging_bytes(B, H, Sq, Skv, D))


def fa_fwd_host(q_h, k_h, v_h, staging, causal: bool = False,
                scale: float | None = None, out_h=None, lse_h=None,
                stream=None):
    """The forward pass on HOST tensors (pinned for full bandwidth): the
    library copies them into ``staging`` (a device tensor of at least
    fa_host_staging_bytes bytes), runs, and copies O and LSE back into
    ``out_h`` / ``lse_h`` (host).  Asynchronous on ``stream``."""
    B, H, Sq, Skv, D = _shape(q_h, k_h, v_h)
    if out_h is None:
        out_h = torch.empty_like(q_h, pin_memory=q_h.is_pinned())
    if lse_h is None:
        lse_h = torch.empty((B, H, Sq), dtype=torch.float32,
                            pin_memory=q_h.is_pinned())
    sc = float(D) ** -0.5 if scale is None else float(scale)
    st = load().fa_fwd_host(q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(),
                            out_h.data_ptr(), lse_h.data_ptr(), B, H, Sq, Skv,
                            D, sc, int(bool(causal)), _DTYPE[q_h.dtype],
                            staging.data_ptr(),
                            staging.numel() * staging.element_size(),
                            _stream_handle(stream))
    _check(st, "fa_fwd_host")
    return out_h, lse_h


def fa_fwd_decode_static(q, k, v, scale: float | None = None, out=None,
                         lse=None, stream=None):
    """Decode (Sq == 1) without any device allocation: the split partials go
    to the library's static device scratch.  Calls whose GPU work overlaps
    share that scratch and race.  Returns (o, lse)."""
    B, H, Sq, Skv, D = _shape(q, k, v)
    if Sq != 1:
        raise ValueError("fa_fwd_decode_static takes one query row per head")
    out, lse = _outputs(q, out, lse)
    sc = float(D) ** -0.5 if scale is None else float(scale)
    st = load().fa_fwd_decode_static(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                     out.data_ptr(), lse.data_ptr(), B, H, Skv,
                                     D, sc, _DTYPE[q.dtype],
                                     _stream_handle(stream))
    _check(st, "fa_fwd_decode_static")
    return out, lse


def fa_release_workspaces() -> None:
    """Synchronises the device and frees the workspaces fa_fwd keeps for it."""
    _check(load().fa_release_workspaces(), "fa_release_workspaces")


def fa_get_device_status(stream=None) -> int:
    """Synchronises the stream; returns and clears the device status word."""
    return int(load().fa_get_device_status(_stream_handle(stream)))


def fa_set_watchdog_ns(ns: int) -> None:
    load().fa_set_watchdog_ns(int(ns))


def fa_status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def fa_prefill_uses_pairs(B: int, H: int, Sq: int, Skv: int, D: int, causal: bool,
                          flags: int = 0, num_splits: int = 0) -> bool:
    return bool(load().fa_prefill_uses_pairs(B, H, Sq, Skv, D, int(bool(causal)), flags,
                                              num_splits))


def fa_prefill_tail_items(B: int, H: int, Sq: int, Skv: int, D: int, causal: bool,
                          dtype=torch.bfloat16, flags: int = 0) -> int:
    """Pair items that fa_fwd_ex with these arguments splits into key
    quarters (FA_FLAG_TAIL_SPLIT); 0 if none."""
    return int(load().fa_prefill_tail_items(B, H, Sq, Skv, D, int(bool(causal)),
                                             _DTYPE[dtype], flags))


def fa_ex2_approx(x, stream=None):
    """2^x on the device with the kernels' exponential instruction (x: a
    contiguous float32 CUDA tensor).  Returns a new tensor."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    y = torch.empty_like(x)
    _check(load().fa_ex2_approx(x.data_ptr(), y.data_ptr(), x.numel(),
                                _stream_handle(stream)), "fa_ex2_approx")
    return y


def fa_version() -> int:
    return int(load().fa_version())
