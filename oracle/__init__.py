"""Double-precision CPU oracle for the attention forward pass (TEST INFRASTRUCTURE).

This package is the checker the CUDA path is compared against.  Only the test
suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it; the library under ``online_softmax_tiling_gb300`` never does, and
this package imports nothing from it.

The arithmetic lives in ``attention_oracle.c`` (plain C, IEEE double, no fast
math); this module only builds it with gcc and marshals numpy arrays.  See the
C file's header for the definition it follows and the passages it cites:
[QS] "用 CuTe 读懂 FlashAttention：一次 forward 的完整流程" (sections "先固定一个例子",
"第四步：更新 online softmax", "causal 模式在哪一步生效", "最后：归一化并写回 O") and
[YT] "CUDA 算子工程" ch. 14, sections 14.1 and 14.5.

Every routine is pinned by ``tests/test_oracle.py``; none is "parity unpinned"
except the value given to a row with no valid key (O = 0, LSE = -inf), which no
page fixes and no workload reaches.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attention_oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")

FP16 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None


def build(source: str = SOURCE, output: str = LIBRARY, force: bool = False) -> str:
    """Compile the oracle with gcc (IEEE double: -O2, no -ffast-math)."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    tmp = output + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
           "-fPIC", "-shared", "-o", tmp, source, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle shared library."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    dp = ctypes.POINTER(ctypes.c_double)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.oracle_decode16.argtypes = [u16p, ctypes.c_int, dp, i64]
    lib.oracle_decode16.restype = None
    lib.oracle_attention_f64.argtypes = [dp, dp, dp, i64, i64, i64, i64, ctypes.c_double,
                                         ctypes.c_int, dp, dp]
    lib.oracle_attention_f64.restype = ctypes.c_int
    lib.oracle_attention_rows16.argtypes = [u16p, u16p, u16p, ctypes.c_int, i64, i64, i64, i64,
                                            ctypes.c_double, ctypes.c_int, i64p, i64,
                                            dp, dp, dp, ctypes.c_int]
    lib.oracle_attention_rows16.restype = ctypes.c_int
    lib.oracle_blocked_head.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double,
                                        ctypes.c_int, i64, dp, dp, dp, dp, dp, dp, dp]
    lib.oracle_blocked_head.restype = ctypes.c_int
    lib.oracle_version.argtypes = []
    lib.oracle_version.restype = ctypes.c_int
    return lib


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctype))
    return a.ctypes.data_as(ctypes.POINTER(ctype))


NO_MASK, TOP_LEFT, BOTTOM_RIGHT = 0, 1, 2


def _mask(causal) -> int:
    """False/0: no mask; True/1: top-left causal; 2: bottom-right causal."""
    m = int(causal)
    if m not in (NO_MASK, TOP_LEFT, BOTTOM_RIGHT):
        raise ValueError(f"mask mode {causal!r}")
    return m


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def decode16(bits: np.ndarray, dtype: int, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Widen raw fp16 / bf16 bit patterns (uint16) to float64 exactly."""
    lib = lib or load()
    src = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(src.shape, dtype=np.float64)
    lib.oracle_decode16(_ptr(src, ctypes.c_uint16), int(dtype), _ptr(out, ctypes.c_double),
                        src.size)
    return out


def attention(q, k, v, scale: float, causal: bool = False, lib: ctypes.CDLL | None = None):
    """Plain definition on float64 inputs; returns (O, LSE).

    q: [..., Nq, d]; k, v: [..., Nk, d] with the same leading dimensions.
    """
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    if (q.ndim < 2 or k.shape != v.shape or q.shape[:-2] != k.shape[:-2]
            or q.shape[-1] != k.shape[-1]):
        raise ValueError("q: [..., Nq, d]; k, v: [..., Nk, d]")
    Nq, Nk, d = q.shape[-2], k.shape[-2], q.shape[-1]
    BH = int(np.prod(q.shape[:-2])) if q.ndim > 2 else 1
    o = np.empty(q.shape, dtype=np.float64)
    lse = np.empty(q.shape[:-1], dtype=np.float64)
    rc = lib.oracle_attention_f64(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                  _ptr(v, ctypes.c_double), BH, Nq, Nk, d, float(scale),
                                  _mask(causal), _ptr(o, ctypes.c_double),
                                  _ptr(lse, ctypes.c_double))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_f64 failed ({rc})")
    return o, lse


def attention_rows16(q16, k16, v16, dtype: int, scale: float, causal: bool, rows,
                     nthreads: int | None = None, with_spread: bool = False,
                     lib: ctypes.CDLL | None = None):
    """Plain definition for selected query rows of 16-bit inputs.

    q16: uint16 bit patterns [B, H, Nq, d] (or [BH, Nq, d]); k16, v16: the
    same with Nk rows.  causal: mask mode (False, True = top-left, 2 =
    bottom-right).  rows: flat row indices ``bh * Nq + i``.  Returns
    (O [nrows, d], LSE [nrows]) in float64, plus spread [nrows, d] =
    sum_j P_ij |v_jc - O_ic| when ``with_spread`` (the sensitivity of O to
    relative errors in the weights).
    """
    lib = lib or load()
    q16 = np.ascontiguousarray(q16, dtype=np.uint16)
    k16 = np.ascontiguousarray(k16, dtype=np.uint16)
    v16 = np.ascontiguousarray(v16, dtype=np.uint16)
    if k16.shape != v16.shape or q16.shape[:-2] != k16.shape[:-2] or q16.shape[-1] != k16.shape[-1]:
        raise ValueError("q: [..., Nq, d]; k, v: [..., Nk, d]")
    Nq, Nk, d = q16.shape[-2], k16.shape[-2], q16.shape[-1]
    BH = q16.size // (Nq * d)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    order = np.argsort(rows, kind="stable")          # group rows of one head together
    srows = np.ascontiguousarray(rows[order])
    o = np.empty((srows.size, d), dtype=np.float64)
    lse = np.empty(srows.size, dtype=np.float64)
    spread = np.empty((srows.size, d), dtype=np.float64) if with_spread else None
    if nthreads is None:
        nthreads = len(os.sched_getaffinity(0))
    rc = lib.oracle_attention_rows16(_ptr(q16, ctypes.c_uint16), _ptr(k16, ctypes.c_uint16),
                                     _ptr(v16, ctypes.c_uint16), int(dtype), BH, Nq, Nk, d,
                                     float(scale), _mask(causal),
                                     _ptr(srows, ctypes.c_int64), srows.size,
                                     _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                                     _ptr(spread, ctypes.c_double), int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows16 failed ({rc})")
    out_o = np.empty_like(o)
    out_lse = np.empty_like(lse)
    out_o[order] = o
    out_lse[order] = lse
    if with_spread:
        out_s = np.empty_like(spread)
        out_s[order] = spread
        return out_o, out_lse, out_s
    return out_o, out_lse


def blocked_head(q, k, v, scale: float, causal: bool, block_n: int, trace: bool = False,
                 lib: ctypes.CDLL | None = None):
    """The online-softmax recurrence for one head: q [Nq, d], k, v [Nk, d] float64.

    Returns (O, LSE) or, with ``trace=True``, (O, LSE, trace) where trace is a
    dict of per-block states: m, l, alpha [nblk, Nq], u [nblk, Nq, d] and
    e [nblk, Nq, block_n].
    """
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    Nq, d = q.shape
    Nk = k.shape[0]
    nblk = (Nk + block_n - 1) // block_n
    o = np.empty((Nq, d), dtype=np.float64)
    lse = np.empty(Nq, dtype=np.float64)
    tr = None
    if trace:
        tr = {"m": np.empty((nblk, Nq)), "l": np.empty((nblk, Nq)),
              "alpha": np.empty((nblk, Nq)), "u": np.empty((nblk, Nq, d)),
              "e": np.empty((nblk, Nq, block_n))}
    rc = lib.oracle_blocked_head(
        _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
        Nq, Nk, d, float(scale), _mask(causal), int(block_n),
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
        _ptr(tr["m"] if tr else None, ctypes.c_double),
        _ptr(tr["l"] if tr else None, ctypes.c_double),
        _ptr(tr["alpha"] if tr else None, ctypes.c_double),
        _ptr(tr["u"] if tr else None, ctypes.c_double),
        _ptr(tr["e"] if tr else None, ctypes.c_double))
    if rc != 0:
        raise RuntimeError(f"oracle_blocked_head failed ({rc})")
    return (o, lse, tr) if trace else (o, lse)
