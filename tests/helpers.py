"""Shared test utilities: building seeded layers, running the CUDA path through the C
ABI binding, running the oracle on the same inputs, and the acceptance checks.

Acceptance (the spec bar of this layer):
  * expert indices identical to the oracle's, except tokens whose oracle gap between
    the k-th and (k+1)-th score is below 1e-5 (counted, and left out of the output check
    only if the selections differ);
  * max |y_gpu - y_ref| <= 1e-3 * max(1, RMS(y_ref)).
"""
from __future__ import annotations

import math
import os

import numpy as np

import synth as S

TOL_REL = 1e-3
NEAR_TIE = 1e-5

# Near-ties seen by compare(), one entry per call: (test id, tokens, tokens whose oracle
# gap between the k-th and (k+1)-th score is below NEAR_TIE, of those the ones whose
# selection differed).  The session summary prints them (tests/conftest.py).
NEAR_TIE_LOG = []
# 1-ulp bf16 differences of the stack step's normalised input allowed by check_rmsnorm_bf16
# (test id, elements compared, elements at a rounding tie).
NORM_TIE_LOG = []


def _test_id():
    return os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0] or "-"


class LayerSpec:
    def __init__(self, H, F, E, k, wfmt, router=0, shared=False, seed=0, layers=1):
        self.H, self.F, self.E, self.k = H, F, E, k
        self.wfmt, self.router, self.shared, self.seed, self.layers = wfmt, router, shared, seed, layers

    def blob(self, layer, e):
        return S.make_expert_blob(self.seed, layer, e, self.wfmt, self.H, self.F)

    def router_w(self, layer):
        return S.make_router(self.seed, layer, self.E, self.H)


def make_context(spec, max_tokens, hbm_cache_bytes=0, register=True, order=None, pool_file=None,
                 host_cache_bytes=0):
    import routed_expert_ffn_03_gb300 as M
    ctx = M.Context(spec.layers, spec.H, spec.F, spec.E, spec.k, spec.wfmt, router=spec.router,
                    shared_ffn=spec.F if spec.shared else 0, max_tokens=max_tokens,
                    hbm_cache_bytes=hbm_cache_bytes, pool_file=pool_file, host_cache_bytes=host_cache_bytes)
    if register:
        for l in range(spec.layers):
            ctx.register_router(l, spec.router_w(l))
            experts = list(range(spec.E)) + ([-1] if spec.shared else [])
            if order is not None:
                experts = [experts[i] for i in order]
            for e in experts:
                ctx.register_expert(l, e, spec.blob(l, e))
    return ctx


def x_tokens(seed, stream, T, H):
    """bf16 bits (uint16) [T, H] of x ~ N(0,1)."""
    return S.f32_to_bf16_bits(S.make_tokens(seed, stream, T, H))


def gpu_forward(ctx, layer, xbits, stream=None):
    import torch
    T, H = xbits.shape
    x = torch.from_numpy(xbits.view(np.int16).copy()).cuda()
    out = torch.empty((T, H), dtype=torch.float32, device="cuda")
    ctx.forward(layer, x, out, T, stream=stream)
    torch.cuda.synchronize()
    idx, w = ctx.get_routing(layer)
    return out.cpu().numpy().astype(np.float64), idx, w


def oracle_forward(spec, layer, xbits, blobs=None):
    from oracle import oracle as O
    cache = {} if blobs is None else blobs
    def get(e):
        if e not in cache:
            cache[e] = spec.blob(layer, e)
        return cache[e]
    shared = get(-1) if spec.shared else None
    return O.layer(xbits, spec.router_w(layer), spec.k, spec.router, get, spec.wfmt, spec.H, spec.F,
                   shared, spec.F if spec.shared else 0)


def compare(ref, y, idx, w=None):
    """Returns a dict of the acceptance figures; asserts the bar."""
    T = y.shape[0]
    ties = flips = 0
    checked = []
    for t in range(T):
        same = np.array_equal(idx[t], ref["idx"][t])
        if ref["gap"][t] < NEAR_TIE:
            ties += 1
            if not same:
                flips += 1
                continue
        else:
            assert same, "token %d: expert ids %s != oracle %s (gap %.3g)" % (
                t, idx[t], ref["idx"][t], ref["gap"][t])
        checked.append(t)
    assert checked, "every token was a near-tie"
    yr = ref["y"][checked]
    rms = math.sqrt(float(np.mean(yr * yr)))
    err = float(np.max(np.abs(y[checked] - yr)))
    bound = TOL_REL * max(1.0, rms)
    assert err <= bound, "max|dy| %.3g > %.3g (rms %.3g)" % (err, bound, rms)
    if w is not None:
        np.testing.assert_allclose(w[checked], ref["w"][checked], rtol=1e-5, atol=1e-6)
    NEAR_TIE_LOG.append((_test_id(), T, ties, flips))
    return dict(err=err, bound=bound, rms=rms, near_ties=ties, near_tie_flips=flips, tokens=T)


# Relative distance from a bf16 rounding midpoint inside which the GPU's fp32 norm may
# round the other way.  The GPU sums x^2 in fp32 along a chain of at most ~40 additions
# (per-thread batches, then warp and block trees), so the mean square carries a relative
# error below ~40 u (u = 2^-24); 1/sqrt of it (a few ulp) and the product x * inv add a
# few u more: about 25 u on the normalised value.  2^-18 = 64 u leaves a margin.
NORM_TIE_REL = 2.0 ** -18


def check_rmsnorm_bf16(x32, xn_bits, eps=1e-6):
    """The stack step's normalised input against the oracle, on the same fp32 residual.

    x32: fp32 [T, H] residual the GPU normalised; xn_bits: the GPU's bf16 bits.  Bit
    equality with oracle.rmsnorm_bf16(x32) is required, with one exception: a 1-ulp
    difference (same sign, adjacent bf16 values) where the exact value x / sqrt(mean(x^2)
    + eps) lies within NORM_TIE_REL of the midpoint of the two bf16 values, i.e. where fp32
    rounding inside the norm decides a bf16 rounding tie.  Returns the count of those."""
    from oracle import oracle as O
    x64 = np.asarray(x32, dtype=np.float32).astype(np.float64)
    ref = O.rmsnorm_bf16(x64, eps)
    got = np.asarray(xn_bits).view(np.uint16)
    diff = ref != got
    n = int(diff.sum())
    if n:
        v = (x64 / np.sqrt(np.mean(x64 * x64, axis=-1, keepdims=True) + eps))[diff]
        a, b = ref[diff].astype(np.int64), got[diff].astype(np.int64)
        assert np.all((a & 0x8000) == (b & 0x8000)), "bf16 sign differs from the oracle"
        assert np.all(np.abs(a - b) == 1), "bf16 differs from the oracle by more than one ulp"
        lo = np.minimum(a, b)
        mid = 0.5 * (O.bf16_value(lo.astype(np.uint16)) + O.bf16_value((lo + 1).astype(np.uint16)))
        far = np.abs(v - mid) > NORM_TIE_REL * np.abs(v)
        assert not far.any(), "a 1-ulp bf16 difference away from a rounding tie: value %r, midpoint %r" % (
            v[far][:4], mid[far][:4])
    NORM_TIE_LOG.append((_test_id(), int(diff.size), n))
    return n


def register_device(spec, ctxs):
    """Register every router and expert of spec into each context of ctxs, the expert
    blobs made by the device generator (same bytes as spec.blob, faster at full sizes),
    each blob made once."""
    import torch
    from synth import device as D
    blob = torch.empty(S.expert_blob_bytes(spec.wfmt, spec.H, spec.F), dtype=torch.uint8, device="cuda")
    experts = list(range(spec.E)) + ([-1] if spec.shared else [])
    for l in range(spec.layers):
        W = spec.router_w(l)
        for c in ctxs:
            c.register_router(l, W)
        for e in experts:
            D.make_expert_blob_device(spec.seed, l, e, spec.wfmt, spec.H, spec.F, blob)
            for c in ctxs:
                c.register_expert(l, e, blob)
    torch.cuda.synchronize()
    return ctxs
