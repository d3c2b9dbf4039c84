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

import numpy as np

import synth as S

TOL_REL = 1e-3
NEAR_TIE = 1e-5


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
    ties = 0
    checked = []
    for t in range(T):
        same = np.array_equal(idx[t], ref["idx"][t])
        if ref["gap"][t] < NEAR_TIE:
            ties += 1
            if not same:
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
    return dict(err=err, bound=bound, rms=rms, near_ties=ties, tokens=T)
