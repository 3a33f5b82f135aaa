"""CPU oracle for the attention forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never links, loads or
calls it, and it never imports the CUDA library.

Contents
  attn_oracle.c   the fp64 three-step oracle and the fp32 same-precision floor
                  reference (compiled to ``liboracle.so`` by :func:`build`)
  online.py       fp64 restatement of the tiled online-softmax algorithm and
                  of the split-KV combine, used to pin the identity the
                  kernels rely on and to show that the parity gate catches
                  planted mistakes
  gate.py         the parity gate (tolerance rule)

All functions here take and return numpy arrays.  Inputs are the 16-bit values
widened exactly to fp32/fp64 by the caller.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math"]
_lock = threading.Lock()
_lib = None

FMT_F16 = 0
FMT_BF16 = 1


def compile_oracle(src: str, out: str) -> None:
    """Compile an oracle C source into a shared object with gcc."""
    cmd = ["gcc", *_CFLAGS, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` if missing or older than its source."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH) or
                 os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            compile_oracle(_SRC, tmp)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    c_long, c_int, c_double, c_float = (ctypes.c_long, ctypes.c_int,
                                        ctypes.c_double, ctypes.c_float)
    vp = ctypes.c_void_p
    lib.oracle_attention_rows.argtypes = [vp, vp, vp, c_long, c_long, c_long,
                                          c_long, c_long, c_double, c_int, vp,
                                          c_long, vp, vp, c_int]
    lib.oracle_attention_rows.restype = c_int
    lib.floor_attention_rows.argtypes = [vp, vp, vp, c_long, c_long, c_long,
                                         c_long, c_long, c_float, c_int, c_int,
                                         vp, c_long, vp, vp, c_int]
    lib.floor_attention_rows.restype = c_int
    lib.oracle_probs.argtypes = [vp, vp, c_long, c_long, c_long, c_double,
                                 c_int, vp]
    lib.oracle_probs.restype = c_int
    lib.oracle_round_fmt.argtypes = [vp, c_long, c_int]
    lib.oracle_round_fmt.restype = None
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if needed).  ``path`` loads
    another build of an oracle source instead (used by the mutation tests)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _c32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _rows_arg(rows, total):
    if rows is None:
        return None, total
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    return r, r.size


def attention(q, k, v, scale: float, causal: bool, rows=None,
              nthreads: int | None = None, lib: ctypes.CDLL | None = None):
    """fp64 oracle.  q [B,H,Sq,D], k/v [B,H,Skv,D].

    Returns (o, lse).  With ``rows=None``: o [B,H,Sq,D], lse [B,H,Sq].  With
    ``rows`` (flat indices into [B,H,Sq]): o [n,D], lse [n]."""
    q, k, v = _c64(q), _c64(k), _c64(v)
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    assert k.shape == (B, H, Skv, D) and v.shape == (B, H, Skv, D)
    r, n = _rows_arg(rows, B * H * Sq)
    o = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    L = lib or load()
    rc = L.oracle_attention_rows(_ptr(q), _ptr(k), _ptr(v), B, H, Sq, Skv, D,
                                 float(scale), int(bool(causal)),
                                 None if r is None else _ptr(r), n, _ptr(o),
                                 _ptr(lse), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows failed ({rc})")
    if rows is None:
        return o.reshape(B, H, Sq, D), lse.reshape(B, H, Sq)
    return o, lse


def floor_attention(q, k, v, scale: float, causal: bool, fmt: int, rows=None,
                    nthreads: int | None = None, lib: ctypes.CDLL | None = None):
    """fp32 same-precision floor reference (fmt: FMT_F16 or FMT_BF16); same
    shapes and conventions as :func:`attention`."""
    q, k, v = _c32(q), _c32(k), _c32(v)
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    r, n = _rows_arg(rows, B * H * Sq)
    o = np.empty((n, D), np.float32)
    lse = np.empty((n,), np.float32)
    L = lib or load()
    rc = L.floor_attention_rows(_ptr(q), _ptr(k), _ptr(v), B, H, Sq, Skv, D,
                                float(np.float32(scale)), int(bool(causal)),
                                int(fmt), None if r is None else _ptr(r), n,
                                _ptr(o), _ptr(lse),
                                nthreads or default_threads())
    if rc != 0:
        raise RuntimeError(f"floor_attention_rows failed ({rc})")
    if rows is None:
        return o.reshape(B, H, Sq, D), lse.reshape(B, H, Sq)
    return o, lse


def probs(q2, k2, scale: float, causal: bool, lib: ctypes.CDLL | None = None):
    """Normalised probabilities P [Sq,Skv] of one head (q2 [Sq,D], k2 [Skv,D])."""
    q2, k2 = _c64(q2), _c64(k2)
    Sq, D = q2.shape
    Skv = k2.shape[0]
    P = np.empty((Sq, Skv), np.float64)
    L = lib or load()
    rc = L.oracle_probs(_ptr(q2), _ptr(k2), Sq, Skv, D, float(scale),
                        int(bool(causal)), _ptr(P))
    if rc != 0:
        raise RuntimeError(f"oracle_probs failed ({rc})")
    return P


def round_fmt(x, fmt: int, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Round fp32 values to fp16 (FMT_F16) or bf16 (FMT_BF16), ties to even."""
    a = _c32(x).copy()
    L = lib or load()
    L.oracle_round_fmt(_ptr(a), a.size, int(fmt))
    return a
