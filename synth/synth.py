"""Counter-based seeded generator and boundary-format blob builders.

Every random number here is a pure function of (seed, tags, index), so any
expert's record can be regenerated on its own, in any order, on the host
(this module) or on the device (``synth/csrc/synth_gen.cu`` fills the bulk
byte fields with the identical byte stream).

Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used counter-style: the i-th
draw of a stream with key ``k`` is ``mix64(k + (i+1)*GAMMA)``, where ``mix64``
is the SplitMix64 output function with the constants published for it.
Streams are separated by ``derive(key, tag) = mix64(key ^ TAGMUL*(tag+1))``.

Distributions (the workload recipe of the routed expert FFN):
  * byte fields (RVQ codes, int4 nibbles): the little-endian bytes of the
    draws, so every code is uniform on 0..255 and every nibble on 0..15;
  * int4 group scales: fp16 value (1024 + k) * 2**-18 with k = draw >> 54,
    i.e. uniform on [2**-8, 2**-7) and exactly representable;
  * normals: Box-Muller on pairs of 53-bit uniforms (host only: codebooks,
    router weights, inputs), rounded once to the stored type.
"""
from __future__ import annotations

import math

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB
TAGMUL = 0xD1B54A32D192ED03
ROOT = 0x243F6A8885A308D3
MASK64 = (1 << 64) - 1

# stream tags
TAG_LAYER, TAG_INPUT, TAG_CENTROID, TAG_TRACE = 1, 2, 3, 4
TAG_ROUTER, TAG_EXPERT = 10, 11
FIELD_CODES, FIELD_CODEBOOK, FIELD_NIBBLES, FIELD_SCALES = 100, 200, 300, 400

RVQ = 1      # 3 bits/weight residual VQ, 8-weight groups, 3 stages
INT4 = 2     # int4 symmetric, 128-weight groups, fp16 scales
RVQ_GROUP, RVQ_STAGES, RVQ_CODES = 8, 3, 256
INT4_GROUP = 128
CODEBOOK_STD = (0.02, 0.01, 0.005)   # std of stage s = 0.02 * 0.5**s

__all__ = [
    "mix64", "derive", "draws", "byte_stream", "normals", "root_key",
    "layer_key", "expert_key", "matrix_shapes", "matrix_block_bytes",
    "expert_blob_bytes", "rvq_codebook", "int4_scales_bits",
    "make_expert_blob", "make_router", "make_tokens", "make_domain_trace",
    "f32_to_bf16_bits", "bf16_bits_to_f32", "RVQ", "INT4", "RVQ_GROUP",
    "RVQ_STAGES", "RVQ_CODES", "INT4_GROUP", "CODEBOOK_STD",
    "FIELD_CODES", "FIELD_CODEBOOK", "FIELD_NIBBLES", "FIELD_SCALES",
    "rvq_codebook_bytes", "stream_key",
]


# --------------------------------------------------------------------------
# SplitMix64, counter style
# --------------------------------------------------------------------------
def _mix64_scalar(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX1) & MASK64
    z = ((z ^ (z >> 27)) * MIX2) & MASK64
    return z ^ (z >> 31)


def mix64(z):
    """SplitMix64 output function on a python int or a numpy uint64 array."""
    if isinstance(z, (int, np.integer)):
        return _mix64_scalar(int(z))
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX2)
        return z ^ (z >> np.uint64(31))


def derive(key: int, tag: int) -> int:
    return _mix64_scalar(int(key) ^ ((TAGMUL * (int(tag) + 1)) & MASK64))


def draws(key: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of the stream ``key`` (uint64)."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + i * np.uint64(GAMMA))


def byte_stream(key: int, nbytes: int) -> np.ndarray:
    """Bytes 0..nbytes-1 of stream ``key``: draw p//8, byte p%8 (little end)."""
    nd = (nbytes + 7) // 8
    d = draws(key, 0, nd).astype("<u8", copy=False)
    return d.view(np.uint8)[:nbytes].copy()


def normals(key: int, n: int) -> np.ndarray:
    """n standard normals (float64) by Box-Muller on draws (2i, 2i+1)."""
    m = (n + 1) // 2
    d = draws(key, 0, 2 * m)
    u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * math.pi * u2)
    z[1::2] = r * np.sin(2.0 * math.pi * u2)
    return z[:n]


def root_key(seed: int) -> int:
    return derive(ROOT, seed)


def layer_key(seed: int, layer: int) -> int:
    return derive(derive(root_key(seed), TAG_LAYER), layer)


def expert_key(seed: int, layer: int, expert: int) -> int:
    """expert = -1 names the always-on shared expert."""
    return derive(derive(layer_key(seed, layer), TAG_EXPERT), expert + 1)


def stream_key(seed: int, layer: int, expert: int, matrix: int, field: int) -> int:
    return derive(derive(expert_key(seed, layer, expert), matrix), field)


# --------------------------------------------------------------------------
# bf16 helpers (round to nearest even; inputs here are finite)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(a) -> np.ndarray:
    b = np.asarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# Boundary blob format
# --------------------------------------------------------------------------
def matrix_shapes(hidden: int, ffn: int):
    """(rows, K) of gate, up, down; K is the input dim that groups run along."""
    return [(ffn, hidden), (ffn, hidden), (hidden, ffn)]


def rvq_codebook_bytes() -> int:
    return RVQ_STAGES * RVQ_CODES * RVQ_GROUP * 2


def matrix_block_bytes(wfmt: int, rows: int, K: int) -> int:
    if wfmt == RVQ:
        assert K % RVQ_GROUP == 0
        return rvq_codebook_bytes() + rows * (K // RVQ_GROUP) * RVQ_STAGES
    if wfmt == INT4:
        assert K % INT4_GROUP == 0
        return rows * K // 2 + rows * (K // INT4_GROUP) * 2
    raise ValueError(wfmt)


def expert_blob_bytes(wfmt: int, hidden: int, ffn: int) -> int:
    return sum(matrix_block_bytes(wfmt, r, k) for r, k in matrix_shapes(hidden, ffn))


def rvq_codebook(key: int, stage: int) -> np.ndarray:
    """fp16 [256, 8] codebook of one stage, entries ~ N(0, std_s)."""
    z = normals(key, RVQ_CODES * RVQ_GROUP) * CODEBOOK_STD[stage]
    return z.astype(np.float16).reshape(RVQ_CODES, RVQ_GROUP)


def int4_scales_bits(key: int, n: int) -> np.ndarray:
    """fp16 bit patterns of n scales (1024 + k) * 2**-18, k = draw >> 54."""
    k = (draws(key, 0, n) >> np.uint64(54)).astype(np.uint16)
    return (np.uint16(7 << 10) | k).astype(np.uint16)


def make_expert_blob(seed: int, layer: int, expert: int, wfmt: int,
                     hidden: int, ffn: int) -> np.ndarray:
    """The boundary blob (uint8) of one expert.

    RVQ, per matrix in the order gate [F,H], up [F,H], down [H,F]:
      fp16 codebooks [3][256][8] (stage 0, 1, 2), then
      uint8 codes [rows][K/8][3] (stage order 0, 1, 2 within a group).
    INT4, per matrix in the same order:
      uint8 nibbles [rows][K/2] (low nibble = even input index, two's
      complement q in [-8, 7]), then fp16 scales [rows][K/128].
    """
    parts = []
    for m, (rows, K) in enumerate(matrix_shapes(hidden, ffn)):
        if wfmt == RVQ:
            for s in range(RVQ_STAGES):
                cb = rvq_codebook(stream_key(seed, layer, expert, m, FIELD_CODEBOOK + s), s)
                parts.append(cb.view(np.uint8).ravel())
            n = rows * (K // RVQ_GROUP) * RVQ_STAGES
            parts.append(byte_stream(stream_key(seed, layer, expert, m, FIELD_CODES), n))
        elif wfmt == INT4:
            parts.append(byte_stream(stream_key(seed, layer, expert, m, FIELD_NIBBLES), rows * K // 2))
            sb = int4_scales_bits(stream_key(seed, layer, expert, m, FIELD_SCALES), rows * (K // INT4_GROUP))
            parts.append(sb.view(np.uint8))
        else:
            raise ValueError(wfmt)
    blob = np.concatenate(parts)
    assert blob.size == expert_blob_bytes(wfmt, hidden, ffn)
    return blob


def make_router(seed: int, layer: int, num_experts: int, hidden: int) -> np.ndarray:
    """Router weights fp32 [E, H], entries ~ N(0, 1/H) (variance 1/H)."""
    z = normals(derive(layer_key(seed, layer), TAG_ROUTER), num_experts * hidden)
    return (z / math.sqrt(hidden)).astype(np.float32).reshape(num_experts, hidden)


def make_tokens(seed: int, stream: int, T: int, hidden: int) -> np.ndarray:
    """T inputs x ~ N(0,1), rounded to bf16 (returned as float32 values)."""
    z = normals(derive(derive(root_key(seed), TAG_INPUT), stream), T * hidden)
    return bf16_bits_to_f32(f32_to_bf16_bits(z.astype(np.float32))).reshape(T, hidden)


def make_domain_trace(seed: int, t0: int, T: int, hidden: int,
                      n_domains: int = 4, period: int = 256) -> np.ndarray:
    """Domain-local token process: x_t = c_d(t) + 0.5 N(0,1), bf16.

    Centroids c_d ~ N(0,1)^H are fixed by the seed; d(t) = (t // period) mod
    n_domains, so the domain switches round-robin every ``period`` tokens.
    """
    ck = derive(root_key(seed), TAG_CENTROID)
    cent = [normals(derive(ck, d), hidden) for d in range(n_domains)]
    tk = derive(root_key(seed), TAG_TRACE)
    out = np.empty((T, hidden), dtype=np.float32)
    for i in range(T):
        t = t0 + i
        d = (t // period) % n_domains
        out[i] = (cent[d] + 0.5 * normals(derive(tk, t), hidden)).astype(np.float32)
    return bf16_bits_to_f32(f32_to_bf16_bits(out))
