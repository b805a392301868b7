"""fp64 CPU oracle for the FlashAttention-2 forward pass.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product library
never does, and it shares no code with the CUDA path.  The attention
arithmetic lives in ``attn_ref.c`` (plain three-pass softmax attention in
double precision, "Flash Attention 全解析(上)" section 1.2, with the per-row
logsumexp of "FlashAttention 怎么做?online softmax 怎么更新?",
FlashAttention-2 follow-up); this module compiles it with gcc and marshals
numpy arrays through ctypes.  ``merge`` (the same page's ring-attention
merge of partial results) is written here in numpy float64.

``attention_backward`` gives the gradients of the same definition with
respect to Q, K and V (the chain rule written out in ``attn_ref.c``; the
pages name the backward pass but print no formulas).

Parity pins (checked by the CPU test suite): the pages' worked online-softmax
example, an independent library routine (torch's float64 CPU attention) on
tiny shapes, closed forms (uniform weights when K = 0, a single kept key,
causal row 0), invariants (convexity of O, LSE bounds, permutation
invariance) and brute-force enumeration on tiny shapes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile attn_ref.c into liboracle.so next to it (gcc, portable flags)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    finally:
        if os.path.exists(tmp):
            os.remove(tmp)
    return _LIB_PATH


class Oracle:
    """The oracle functions bound to one compiled copy of attn_ref.c."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_attention_rows.argtypes = [p, p, p, i64, i64, i64, i64, i64, ctypes.c_int,
                                              ctypes.c_float, p, i64, p, p, ctypes.c_int]
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_attention.argtypes = [p, p, p, i64, i64, i64, i64, i64, ctypes.c_int,
                                         ctypes.c_float, p, p, ctypes.c_int]
        self.typed = hasattr(lib, "oracle_attention_rows_typed")
        if self.typed:
            lib.oracle_attention_rows_typed.restype = ctypes.c_int
            lib.oracle_attention_rows_typed.argtypes = [p, p, p, i64, i64, i64, i64, i64, ctypes.c_int,
                                                        ctypes.c_float, ctypes.c_int, p, i64, p, p,
                                                        ctypes.c_int]
            lib.oracle_widen.restype = ctypes.c_double
            lib.oracle_widen.argtypes = [ctypes.c_uint16, ctypes.c_int]
        self.has_backward = hasattr(lib, "oracle_attention_backward")
        if self.has_backward:
            lib.oracle_attention_backward.restype = ctypes.c_int
            lib.oracle_attention_backward.argtypes = [p, p, p, p, i64, i64, i64, i64, i64,
                                                      ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                                      p, i64, p, p, p, p, p, p, ctypes.c_int]
        self.lib = lib
        self.path = lib_path

    def attention(self, Q, K, V, causal: bool, scale: float, nthreads: int | None = None,
                  dtype: str = "bf16"):
        """Exact attention of every row.  Q [B,H,Nq,d], K/V [B,H,Nk,d] 16-bit
        patterns of `dtype` ("bf16" or "fp16").

        Returns (O [B,H,Nq,d] float64, LSE [B,H,Nq] float64).
        """
        if dtype != "bf16":
            B, H, Nq = np.shape(Q)[:3]
            d = np.shape(Q)[3]
            O, L = self.attention_rows(Q, K, V, causal, scale, np.arange(B * H * Nq), nthreads, dtype)
            return O.reshape(B, H, Nq, d), L.reshape(B, H, Nq)
        Q, K, V = _bits(Q), _bits(K), _bits(V)
        B, H, Nq, d = Q.shape
        Nk = K.shape[2]
        if K.shape != (B, H, Nk, d) or V.shape != K.shape:
            raise ValueError("shape mismatch")
        O = np.empty((B, H, Nq, d), dtype=np.float64)
        LSE = np.empty((B, H, Nq), dtype=np.float64)
        rc = self.lib.oracle_attention(_ptr(Q), _ptr(K), _ptr(V), B, H, Nq, Nk, d,
                                       int(bool(causal)), float(scale), _ptr(O), _ptr(LSE),
                                       nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_attention failed with code {rc}")
        return O, LSE

    def attention_rows(self, Q, K, V, causal: bool, scale: float, rows,
                       nthreads: int | None = None, dtype: str = "bf16"):
        """Exact attention of selected rows.

        ``rows`` holds flattened row ids (b*H + h)*Nq + i.  Returns
        (O [len(rows), d] float64, LSE [len(rows)] float64) in the order given.
        """
        Q, K, V = _bits(Q), _bits(K), _bits(V)
        B, H, Nq, d = Q.shape
        Nk = K.shape[2]
        if K.shape != (B, H, Nk, d) or V.shape != K.shape:
            raise ValueError("shape mismatch")
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows.shape[0]
        O = np.empty((n, d), dtype=np.float64)
        LSE = np.empty((n,), dtype=np.float64)
        code = _DTYPES[dtype]
        if code == 0 and not self.typed:
            rc = self.lib.oracle_attention_rows(_ptr(Q), _ptr(K), _ptr(V), B, H, Nq, Nk, d,
                                                int(bool(causal)), float(scale), _ptr(rows), n,
                                                _ptr(O), _ptr(LSE), nthreads or default_threads())
        else:
            rc = self.lib.oracle_attention_rows_typed(_ptr(Q), _ptr(K), _ptr(V), B, H, Nq, Nk, d,
                                                      int(bool(causal)), float(scale), code,
                                                      _ptr(rows), n, _ptr(O), _ptr(LSE),
                                                      nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_attention_rows failed with code {rc}")
        return O, LSE


    def attention_backward(self, Q, K, V, dO, causal: bool, scale: float, heads=None,
                           nthreads: int | None = None, dtype: str = "bf16",
                           magnitudes: bool = False):
        """Gradients of the attention definition for upstream gradient dO.

        Q, dO [B,H,Nq,d] and K, V [B,H,Nk,d] are 16-bit patterns of `dtype`.
        ``heads`` lists flattened head ids b*H + h (default: all, in order).
        Returns (dQ [n,Nq,d], dK [n,Nk,d], dV [n,Nk,d]) float64 for the n heads,
        followed by (M_dQ, M_dK, M_dV), the per-element sums of absolute
        terms, when ``magnitudes`` is true.
        """
        Q, K, V, dO = _bits(Q), _bits(K), _bits(V), _bits(dO)
        B, H, Nq, d = Q.shape
        Nk = K.shape[2]
        if K.shape != (B, H, Nk, d) or V.shape != K.shape or dO.shape != Q.shape:
            raise ValueError("shape mismatch")
        hl = np.arange(B * H, dtype=np.int64) if heads is None else np.ascontiguousarray(heads, dtype=np.int64)
        n = hl.shape[0]
        out = [np.empty((n, N, d), dtype=np.float64) for N in (Nq, Nk, Nk)]
        mags = [np.empty((n, N, d), dtype=np.float64) for N in (Nq, Nk, Nk)] if magnitudes else None
        mp = [_ptr(a) for a in mags] if magnitudes else [None, None, None]
        rc = self.lib.oracle_attention_backward(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, H, Nq, Nk, d,
                                                int(bool(causal)), float(scale), _DTYPES[dtype],
                                                _ptr(hl), n, _ptr(out[0]), _ptr(out[1]), _ptr(out[2]),
                                                mp[0], mp[1], mp[2], nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"oracle_attention_backward failed with code {rc}")
        return tuple(out) + (tuple(mags) if magnitudes else ())

    def widen(self, bits: int, dtype: str) -> float:
        """The oracle's exact widening of one 16-bit pattern to double."""
        return self.lib.oracle_widen(bits, _DTYPES[dtype])


_DTYPES = {"bf16": 0, "fp16": 1}


def compile_source(src_path: str, out_path: str) -> str:
    """Compile a copy of the oracle source (used by the tests' planted-mistake checks)."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-o", out_path, src_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


def _default() -> Oracle:
    global _lib
    if _lib is None:
        _lib = Oracle(build())
    return _lib


def _bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16 or a.ndim != 4:
        raise TypeError("oracle inputs are [B,H,N,d] uint16 arrays of bf16 bit patterns")
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def default_threads() -> int:
    return os.cpu_count() or 1


def attention(Q, K, V, causal: bool, scale: float, nthreads: int | None = None, dtype: str = "bf16"):
    """Exact attention of every row (see ``Oracle.attention``)."""
    return _default().attention(Q, K, V, causal, scale, nthreads, dtype)


def attention_rows(Q, K, V, causal: bool, scale: float, rows, nthreads: int | None = None,
                   dtype: str = "bf16"):
    """Exact attention of selected rows (see ``Oracle.attention_rows``)."""
    return _default().attention_rows(Q, K, V, causal, scale, rows, nthreads, dtype)


def attention_backward(Q, K, V, dO, causal: bool, scale: float, heads=None,
                       nthreads: int | None = None, dtype: str = "bf16", magnitudes: bool = False):
    """Gradients of the attention definition (see ``Oracle.attention_backward``)."""
    return _default().attention_backward(Q, K, V, dO, causal, scale, heads, nthreads, dtype,
                                         magnitudes)


def widen(bits: int, dtype: str) -> float:
    """The oracle's exact widening of one 16-bit pattern (see ``Oracle.widen``)."""
    return _default().widen(bits, dtype)


def merge(O_parts, LSE_parts):
    """Merge of results over disjoint key subsets, in float64.

    "FlashAttention 怎么做?online softmax 怎么更新?" (ring-attention question):
    L = log(e^L1 + e^L2), O = e^(L1-L) O1 + e^(L2-L) O2, applied here to any
    number of parts: L = log sum_p e^(L_p), O = sum_p e^(L_p - L) O_p.  A part
    with L_p = -inf has no kept key and contributes nothing; a row whose
    parts are all -inf gets O = 0, L = -inf.

    O_parts [P, ..., d], LSE_parts [P, ...] -> (O [..., d], LSE [...]).
    """
    O_parts = np.asarray(O_parts, dtype=np.float64)
    L = np.asarray(LSE_parts, dtype=np.float64)
    m = np.max(L, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.where(np.isfinite(L), np.exp(L - m_safe[None]), 0.0)
    s = np.sum(w, axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, s, 1.0)), -np.inf)
    coef = np.where(finite[None], w / np.where(finite, s, 1.0)[None], 0.0)
    O = np.sum(coef[..., None] * O_parts, axis=0)
    return O, lse
