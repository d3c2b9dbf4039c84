"""Python binding of the C ABI in include/moe.h (argument marshalling only).

Every step of the layer runs in ``libmoe.so``'s CUDA kernels; PyTorch provides device
memory and streams.  The library is built in-tree by ``build.py``; importing this module
fails loudly if it is missing or cannot be loaded (there is no CPU fallback).
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIBMOE = os.path.join(PKG, "libmoe.so")

OK, EINVAL, ENOMEM, EBUDGET, ECUDA, ESTATE, ETIMEOUT, ENOTFOUND, EIO = range(9)
ROUTER_SOFTMAX, ROUTER_SIGMOID = 0, 1
W_RVQ3, W_INT4 = 1, 2


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, strerror(status), status))


class Config(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("ffn", ctypes.c_int),
        ("num_experts", ctypes.c_int), ("top_k", ctypes.c_int), ("shared_ffn", ctypes.c_int),
        ("router", ctypes.c_int), ("wfmt", ctypes.c_int), ("max_tokens", ctypes.c_int),
        ("hbm_cache_bytes", ctypes.c_ulonglong),
        ("pool_file", ctypes.c_char_p), ("host_cache_bytes", ctypes.c_ulonglong),
    ]


class FileTierStats(ctypes.Structure):
    _fields_ = [("slots", ctypes.c_ulonglong), ("stride", ctypes.c_ulonglong), ("direct", ctypes.c_int),
                ("reads", ctypes.c_ulonglong), ("read_bytes", ctypes.c_ulonglong),
                ("ram_hits", ctypes.c_ulonglong), ("ram_misses", ctypes.c_ulonglong), ("read_ms", ctypes.c_double)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class Stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_ulonglong) for n in (
        "forwards", "tokens", "lookups", "hits", "misses", "bytes_expert_touched",
        "bytes_router", "bytes_h2d", "record_bytes", "cache_slots")] + [("h2d_ms", ctypes.c_double)] + [
        (n, ctypes.c_ulonglong) for n in ("prefetches", "prefetch_hits", "file_reads", "file_read_bytes",
                                          "ram_hits", "ram_misses")] + [
        ("file_read_ms", ctypes.c_double), ("file_direct", ctypes.c_int), ("launches", ctypes.c_ulonglong)]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


_lib = None


def lib():
    """Load libmoe.so (raises if it is missing: build it with build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBMOE):
        raise RuntimeError("libmoe.so is not built (%s); run routed_expert_ffn_03_gb300.build.build()" % LIBMOE)
    L = ctypes.CDLL(LIBMOE)
    vp, i, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_ulonglong
    L.moe_create.argtypes = [ctypes.POINTER(Config), i, ctypes.POINTER(vp)]
    L.moe_register_router.argtypes = [vp, i, vp]
    L.moe_register_expert.argtypes = [vp, i, i, vp, ctypes.c_size_t]
    L.moe_expert_blob_bytes.argtypes = [i, i, i]
    L.moe_expert_blob_bytes.restype = ctypes.c_size_t
    L.moe_forward.argtypes = [vp, i, vp, vp, i, vp]
    L.moe_get_routing.argtypes = [vp, i, vp, vp, ctypes.POINTER(i)]
    L.moe_forward_residual.argtypes = [vp, i, vp, vp, vp, vp, i, ctypes.c_float, vp]
    L.moe_route_noalloc.argtypes = [vp, vp, i, i, i, i, i, vp, vp, vp]
    L.moe_residual_rmsnorm.argtypes = [vp, vp, vp, vp, i, ctypes.c_float, vp]
    L.moe_stats.argtypes = [vp, ctypes.POINTER(Stats)]
    L.moe_reset_stats.argtypes = [vp]
    L.moe_destroy.argtypes = [vp]
    L.moe_strerror.argtypes = [i]
    L.moe_strerror.restype = ctypes.c_char_p
    L.moe_profile.argtypes = [vp, i]
    L.moe_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i)]
    L.moe_debug_fail_copies.argtypes = [vp, i]
    L.moe_set_readahead.argtypes = [vp, i]
    L.moe_debug_wait_timeout.argtypes = [vp, u64, vp, ctypes.POINTER(i)]
    L.moe_filetier_create.argtypes = [ctypes.c_char_p, ctypes.c_size_t, ctypes.c_longlong, u64, ctypes.POINTER(vp)]
    L.moe_filetier_write.argtypes = [vp, ctypes.c_longlong, vp]
    L.moe_filetier_fetch.argtypes = [vp, ctypes.POINTER(ctypes.c_longlong), i, ctypes.POINTER(vp),
                                     ctypes.POINTER(i)]
    L.moe_filetier_info.argtypes = [vp, ctypes.POINTER(FileTierStats)]
    L.moe_filetier_destroy.argtypes = [vp]
    L.moe_filetier_destroy.restype = None
    L.moe_rvq_block_split.argtypes = [i, i, i, ctypes.POINTER(i), ctypes.POINTER(i)]
    L.moe_rvq_block_split.restype = ctypes.c_int
    for name in ("moe_create", "moe_register_router", "moe_register_expert", "moe_forward",
                 "moe_get_routing", "moe_residual_rmsnorm", "moe_stats", "moe_reset_stats",
                 "moe_destroy", "moe_debug_fail_copies", "moe_debug_wait_timeout",
                 "moe_profile", "moe_profile_read", "moe_forward_residual", "moe_route_noalloc",
                 "moe_set_readahead", "moe_filetier_create", "moe_filetier_write", "moe_filetier_fetch",
                 "moe_filetier_info"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def strerror(status: int) -> str:
    return lib().moe_strerror(status).decode()


def expert_blob_bytes(wfmt: int, hidden: int, ffn: int) -> int:
    return int(lib().moe_expert_blob_bytes(wfmt, hidden, ffn))


def _ptr(t):
    """Address of a torch tensor or numpy array (or an int address)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def rvq_block_split(u_n: int, ntask: int, grid: int):
    """The RVQ lookup kernel's task ranges (moe_rvq_block_split): lists t0, t1 of `grid`
    blocks for u_n units of ntask tasks, grid < u_n < 2 grid.  Host code; raises ValueError
    outside that range."""
    t0 = (ctypes.c_int * grid)()
    t1 = (ctypes.c_int * grid)()
    if lib().moe_rvq_block_split(u_n, ntask, grid, t0, t1) != 0:
        raise ValueError("moe_rvq_block_split(%d, %d, %d)" % (u_n, ntask, grid))
    return list(t0), list(t1)


def route_noalloc(x_bf16, W, T, H, E, k, router, idx, w, stream=None):
    """Routing without allocation (moe_route_noalloc): x bf16 [T,H], W fp32 [E,H] and the
    outputs idx int32 [T,k], w fp32 [T,k] are device tensors.  Raises MoeError."""
    st = lib().moe_route_noalloc(_ptr(x_bf16), _ptr(W), T, H, E, k, router, _ptr(idx), _ptr(w), _stream(stream))
    if st != OK:
        raise MoeError(st, "moe_route_noalloc")


class FileTier:
    """The RAM + file tier on its own (moe_filetier_*): host memory only, no GPU."""

    def __init__(self, path, rec_bytes, n_keys, ram_bytes):
        h = ctypes.c_void_p()
        st = lib().moe_filetier_create(str(path).encode(), rec_bytes, n_keys, ram_bytes, ctypes.byref(h))
        if st != OK:
            raise MoeError(st, "moe_filetier_create")
        self._h = h
        self.rec_bytes = rec_bytes

    def write(self, key, rec):
        """rec: a contiguous numpy uint8 array of rec_bytes."""
        assert rec.nbytes == self.rec_bytes
        st = lib().moe_filetier_write(self._h, key, rec.ctypes.data)
        if st != OK:
            raise MoeError(st, "moe_filetier_write")

    def fetch(self, keys):
        """Returns (list of record bytes copies, list of RAM slots)."""
        n = len(keys)
        karr = (ctypes.c_longlong * n)(*keys)
        out = (ctypes.c_void_p * n)()
        slots = (ctypes.c_int * n)()
        st = lib().moe_filetier_fetch(self._h, karr, n, out, slots)
        if st != OK:
            raise MoeError(st, "moe_filetier_fetch")
        recs = [ctypes.string_at(out[i], self.rec_bytes) for i in range(n)]
        return recs, list(slots)

    def info(self):
        s = FileTierStats()
        st = lib().moe_filetier_info(self._h, ctypes.byref(s))
        if st != OK:
            raise MoeError(st, "moe_filetier_info")
        return s.as_dict()

    def close(self):
        if self._h:
            lib().moe_filetier_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Context:
    """One stack of MoE layers on one GPU (wraps moe_ctx)."""

    def __init__(self, num_layers, hidden, ffn, num_experts, top_k, wfmt, router=ROUTER_SOFTMAX,
                 shared_ffn=0, max_tokens=1, hbm_cache_bytes=0, device=0, pool_file=None, host_cache_bytes=0):
        self.cfg = Config(num_layers, hidden, ffn, num_experts, top_k, shared_ffn, router, wfmt,
                          max_tokens, hbm_cache_bytes,
                          pool_file.encode() if pool_file else None, host_cache_bytes)
        self.device = device
        h = ctypes.c_void_p()
        st = lib().moe_create(ctypes.byref(self.cfg), device, ctypes.byref(h))
        if st != OK:
            raise MoeError(st, "moe_create")
        self._h = h

    # -- lifetime
    def close(self):
        if getattr(self, "_h", None):
            lib().moe_destroy(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, st, what):
        if st != OK:
            raise MoeError(st, what)

    # -- registration
    def register_router(self, layer, w):
        """w: fp32 [E, H] (numpy array or torch tensor, host or this device)."""
        self._check(lib().moe_register_router(self._h, layer, _ptr(w)), "moe_register_router")

    def register_expert(self, layer, expert, blob, nbytes=None):
        """blob: uint8 boundary-format blob (numpy/torch, host or device); expert -1 = shared."""
        if nbytes is None:
            nbytes = blob.numel() if hasattr(blob, "numel") else blob.nbytes
        self._check(lib().moe_register_expert(self._h, layer, expert, _ptr(blob), nbytes),
                    "moe_register_expert")

    # -- compute
    def forward(self, layer, x_bf16, out, T=None, stream=None):
        """x_bf16: int16/bfloat16 cuda tensor [T, H]; out: float32 cuda tensor [T, H]."""
        if T is None:
            T = x_bf16.shape[0]
        self._check(lib().moe_forward(self._h, layer, _ptr(x_bf16), _ptr(out), T, _stream(stream)),
                    "moe_forward")

    def forward_residual(self, layer, x, y_prev, xn, y, T=None, eps=1e-6, stream=None):
        """Fused stack step: x += y_prev (if given); xn = bf16(rmsnorm(x)); y = layer(xn)."""
        if T is None:
            T = x.shape[0]
        self._check(lib().moe_forward_residual(self._h, layer, _ptr(x), _ptr(y_prev), _ptr(xn), _ptr(y), T,
                                               float(eps), _stream(stream)), "moe_forward_residual")

    def residual_rmsnorm(self, x, y, xn, T=None, eps=1e-6, stream=None):
        if T is None:
            T = x.shape[0]
        self._check(lib().moe_residual_rmsnorm(self._h, _ptr(x), _ptr(y), _ptr(xn), T,
                                               float(eps), _stream(stream)),
                    "moe_residual_rmsnorm")

    def get_routing(self, layer):
        import numpy as np
        k, maxT = self.cfg.top_k, self.cfg.max_tokens
        idx = np.zeros((maxT, k), dtype=np.int32)
        w = np.zeros((maxT, k), dtype=np.float32)
        T = ctypes.c_int(0)
        self._check(lib().moe_get_routing(self._h, layer, idx.ctypes.data, w.ctypes.data,
                                          ctypes.byref(T)), "moe_get_routing")
        return idx[:T.value].copy(), w[:T.value].copy()

    def stats(self):
        s = Stats()
        self._check(lib().moe_stats(self._h, ctypes.byref(s)), "moe_stats")
        return s.as_dict()

    def stats_status(self):
        """(status, stats) without raising: for tests of sticky errors."""
        s = Stats()
        st = lib().moe_stats(self._h, ctypes.byref(s))
        return st, s.as_dict()

    def reset_stats(self):
        self._check(lib().moe_reset_stats(self._h), "moe_reset_stats")

    # -- measurement
    def set_readahead(self, enable=True):
        """Streamed contexts: predict the next layer's experts and start their copies early."""
        self._check(lib().moe_set_readahead(self._h, 1 if enable else 0), "moe_set_readahead")

    def profile(self, enable=True):
        self._check(lib().moe_profile(self._h, 1 if enable else 0), "moe_profile")

    def profile_read(self):
        """(ms[router, gateup, down, combine] summed over recorded layers, n_layers)."""
        ms = (ctypes.c_double * 4)()
        n = ctypes.c_int(0)
        self._check(lib().moe_profile_read(self._h, ms, ctypes.byref(n)), "moe_profile_read")
        return list(ms), n.value

    # -- failure injection (host side)
    def debug_fail_copies(self, n):
        self._check(lib().moe_debug_fail_copies(self._h, n), "moe_debug_fail_copies")

    def debug_wait_timeout(self, cycles, stream=None):
        st = ctypes.c_int(-1)
        self._check(lib().moe_debug_wait_timeout(self._h, cycles, _stream(stream), ctypes.byref(st)),
                    "moe_debug_wait_timeout")
        return st.value
