"""Device-side fill of the seeded synthetic expert blobs (same bytes as synth.synth).

Large workloads generate their expert blobs on the GPU: the integer byte fields (RVQ
codes, int4 nibbles and scales) come from ``libsynthgen.so`` (SplitMix64 counter
streams, bit-identical to ``synth.byte_stream`` / ``synth.int4_scales_bits``); the RVQ
codebooks, which need normal draws, are made on the host by ``synth.rvq_codebook`` and
copied.  Input generation only.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import synth as S

_HERE = os.path.dirname(os.path.abspath(__file__))
LIBSYNTH = os.path.join(_HERE, "libsynthgen.so")
_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIBSYNTH):
            raise RuntimeError("libsynthgen.so is not built (%s)" % LIBSYNTH)
        L = ctypes.CDLL(LIBSYNTH)
        L.synth_fill_bytes.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.synth_fill_scales.argtypes = [ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
        L.synth_fill_bytes.restype = ctypes.c_int
        L.synth_fill_scales.restype = ctypes.c_int
        _lib = L
    return _lib


def fill_bytes(key: int, dst_ptr: int, nbytes: int, stream: int = 0):
    rc = lib().synth_fill_bytes(ctypes.c_uint64(key), dst_ptr, nbytes, stream)
    if rc:
        raise RuntimeError("synth_fill_bytes failed (%d)" % rc)


def fill_scales(key: int, dst_ptr: int, n: int, stream: int = 0):
    rc = lib().synth_fill_scales(ctypes.c_uint64(key), dst_ptr, n, stream)
    if rc:
        raise RuntimeError("synth_fill_scales failed (%d)" % rc)


def make_expert_blob_device(seed, layer, expert, wfmt, hidden, ffn, out, stream=0, codebooks=None):
    """Write the boundary blob of one expert into ``out`` (a uint8 CUDA tensor).

    ``codebooks`` (optional) is a dict matrix -> uint8 host array of the 3 fp16
    codebooks, to reuse host draws; otherwise they are generated here.
    """
    import torch
    base = out.data_ptr()
    off = 0
    for m, (rows, K) in enumerate(S.matrix_shapes(hidden, ffn)):
        if wfmt == S.RVQ:
            if codebooks is not None and m in codebooks:
                cb = codebooks[m]
            else:
                cb = np.concatenate([S.rvq_codebook(S.stream_key(seed, layer, expert, m, S.FIELD_CODEBOOK + s), s)
                                     .view(np.uint8).ravel() for s in range(S.RVQ_STAGES)])
            out[off:off + cb.size].copy_(torch.from_numpy(cb), non_blocking=False)
            off += cb.size
            n = rows * (K // S.RVQ_GROUP) * S.RVQ_STAGES
            fill_bytes(S.stream_key(seed, layer, expert, m, S.FIELD_CODES), base + off, n, stream)
            off += n
        else:
            n = rows * K // 2
            fill_bytes(S.stream_key(seed, layer, expert, m, S.FIELD_NIBBLES), base + off, n, stream)
            off += n
            ns = rows * (K // S.INT4_GROUP)
            fill_scales(S.stream_key(seed, layer, expert, m, S.FIELD_SCALES), base + off, ns, stream)
            off += 2 * ns
    assert off == S.expert_blob_bytes(wfmt, hidden, ffn)
    return out
