"""Python face of the fp64 CPU oracle (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  It builds ``oracle/liboracle.so`` from
``oracle.c`` with gcc (OpenMP over rows) and composes the layer from the C
pieces with plain numpy fp64 arithmetic:

  * ``router``      - logits, scores, brute-force top-k, weights, near-tie gap;
  * ``expert``      - one dense SwiGLU expert from its boundary blob;
  * ``layer``       - router + selected experts + weighted combine (+ shared);
  * ``rmsnorm_bf16``/``stack`` - the residual stack x += moe(rmsnorm(x)).

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against hand-expanded matrices, closed forms, brute force and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

SOFTMAX, SIGMOID = 0, 1
RVQ, INT4 = 1, 2

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile liboracle.so (plain C, fp64, OpenMP) if missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        L.oracle_matrix_bytes.restype = ctypes.c_longlong
        L.oracle_matrix_bytes.argtypes = [ctypes.c_int] * 3
        L.oracle_expert_bytes.restype = ctypes.c_longlong
        L.oracle_expert_bytes.argtypes = [ctypes.c_int] * 3
        L.oracle_dense.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, _dp]
        L.oracle_matvec.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                    ctypes.c_int, _dp, _dp]
        L.oracle_expert.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                    ctypes.c_int, _dp, _dp, _dp]
        L.oracle_router.argtypes = [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_void_p,
                                                         _dp, _dp, _ip, _dp, _dp]
        L.oracle_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _d(a):
    return a.ctypes.data_as(_dp)


def threads() -> int:
    return lib().oracle_threads()


def matrix_bytes(wfmt, rows, K):
    return lib().oracle_matrix_bytes(wfmt, rows, K)


def expert_bytes(wfmt, H, F):
    return lib().oracle_expert_bytes(wfmt, H, F)


def dense(wfmt, rows, K, block) -> np.ndarray:
    """Dense fp64 [rows, K] matrix of one boundary-format matrix block."""
    block = np.ascontiguousarray(block, dtype=np.uint8)
    W = np.empty((rows, K), dtype=np.float64)
    rc = lib().oracle_dense(wfmt, rows, K, block.ctypes.data, _d(W))
    if rc:
        raise ValueError("oracle_dense: bad shape")
    return W


def matvec(wfmt, rows, K, block, x) -> np.ndarray:
    block = np.ascontiguousarray(block, dtype=np.uint8)
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    y = np.empty((x.shape[0], rows), dtype=np.float64)
    rc = lib().oracle_matvec(wfmt, rows, K, block.ctypes.data, x.shape[0], _d(x), _d(y))
    if rc:
        raise ValueError("oracle_matvec: bad shape")
    return y


def expert(wfmt, H, F, blob, x, want_h=False):
    """SwiGLU expert on rows of x [n, H] (fp64); returns y [n, H] (and h)."""
    blob = np.ascontiguousarray(blob, dtype=np.uint8)
    if blob.size != expert_bytes(wfmt, H, F):
        raise ValueError("blob size %d != %d" % (blob.size, expert_bytes(wfmt, H, F)))
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float64)
    n = x.shape[0]
    y = np.empty((n, H), dtype=np.float64)
    h = np.empty((n, F), dtype=np.float64)
    rc = lib().oracle_expert(wfmt, H, F, blob.ctypes.data, n, _d(x), _d(h), _d(y))
    if rc:
        raise ValueError("oracle_expert failed (%d)" % rc)
    return (y, h) if want_h else y


def router(x_bf16_bits, Wr, k, kind):
    """Router for T tokens: returns dict(logits, scores, idx, w, gap)."""
    xb = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    Wr = np.ascontiguousarray(Wr, dtype=np.float32)
    T, H = xb.shape
    E = Wr.shape[0]
    out = dict(logits=np.empty((T, E)), scores=np.empty((T, E)),
               idx=np.empty((T, k), dtype=np.int32), w=np.empty((T, k)),
               gap=np.empty(T))
    rc = lib().oracle_router(T, H, E, k, kind, xb.ctypes.data, Wr.ctypes.data,
                             _d(out["logits"]), _d(out["scores"]),
                             out["idx"].ctypes.data_as(_ip), _d(out["w"]), _d(out["gap"]))
    if rc:
        raise ValueError("oracle_router failed (%d)" % rc)
    return out


def bf16_bits(x) -> np.ndarray:
    """Round float values (fp64 or fp32) to bf16 bits: to fp32 then to bf16,
    both round-to-nearest-even (fp32 is the precision the kernels work in)."""
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_value(bits) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def layer(x_bf16_bits, Wr, k, kind, get_blob, wfmt, H, F, shared_blob=None, shared_F=0):
    """One MoE layer on T tokens.

    ``get_blob(e)`` returns expert e's boundary blob; only selected experts
    are requested.  Returns dict(y [T,H] fp64, idx, w, gap, scores).
    Combine: y_t = sum_j w_tj * y_{idx_tj}(x_t), j in rank order, then the
    shared expert (weight 1) is added last.
    """
    r = router(x_bf16_bits, Wr, k, kind)
    x = bf16_value(x_bf16_bits)
    T = x.shape[0]
    y = np.zeros((T, H))
    cache = {}
    for t in range(T):
        for j in range(k):
            e = int(r["idx"][t, j])
            if e not in cache:
                cache[e] = get_blob(e)
            y[t] += r["w"][t, j] * expert(wfmt, H, F, cache[e], x[t:t + 1])[0]
    if shared_blob is not None:
        y += expert(wfmt, H, shared_F, shared_blob, x)
    r["y"] = y
    return r


def rmsnorm_bf16(x, eps=1e-6) -> np.ndarray:
    """xn = bf16(x / sqrt(mean(x^2) + eps)), per row, no gain; bf16 bits."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return bf16_bits(x / np.sqrt(ms + eps))


def stack(x0, layers, eps=1e-6, on_layer=None):
    """Residual stack: for each layer, xn = rmsnorm_bf16(x); x += moe(xn).

    ``layers`` is a list of callables xn_bits -> layer-result dict.  x stays
    fp64 throughout.  Returns the final x and the per-layer results.
    """
    x = np.array(x0, dtype=np.float64)
    res = []
    for li, fn in enumerate(layers):
        xn = rmsnorm_bf16(x, eps)
        r = fn(xn)
        r["xn"] = xn
        x = x + r["y"]
        res.append(r)
        if on_layer is not None:
            on_layer(li, x, r)
    return x, res
