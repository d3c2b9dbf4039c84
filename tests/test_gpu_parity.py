"""GPU parity of the whole layer (C ABI) against the fp64 oracle, small shapes.

Shapes span several tiles and ragged tails: rows not multiples of 32, k-slices with
fewer groups than the tile, E below and above 32 / 256, T = 1, 3, 4, 32, both router
kinds, the shared expert, both weight formats.
"""
import numpy as np
import pytest

import synth as S
from tests.helpers import LayerSpec, compare, gpu_forward, make_context, oracle_forward, x_tokens

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from routed_expert_ffn_03_gb300 import build
    build.build()


def _run(spec, T, stream_id=0):
    ctx = make_context(spec, max_tokens=T)
    try:
        xb = x_tokens(spec.seed + 100, stream_id, T, spec.H)
        y, idx, w = gpu_forward(ctx, 0, xb)
        ref = oracle_forward(spec, 0, xb)
        return compare(ref, y, idx, w)
    finally:
        ctx.close()


def test_tiny_config_rvq_top2_softmax():
    """1 layer, H=256, F=512, 8 experts, top-2 softmax renormalised, T=4, RVQ-3bit."""
    r = _run(LayerSpec(256, 512, 8, 2, S.RVQ, router=0, seed=0), T=4)
    assert r["tokens"] == 4


@pytest.mark.parametrize("H,F,E,k,T,router,shared", [
    (72, 40, 5, 2, 1, 0, False),        # rows and K far below one tile
    (264, 200, 33, 3, 3, 1, True),      # ragged k-slice (33 groups), E > 32, sigmoid + shared
    (520, 96, 7, 7, 4, 0, False),       # k = E
    (128, 64, 300, 8, 2, 1, False),     # E > 256
    (256, 136, 16, 4, 32, 0, True),     # T = 32 with shared expert (dense tcgen05 groups)
    (512, 384, 4, 2, 16, 1, True),      # T = 16: most experts take the dense path
    (264, 200, 3, 3, 40, 0, False),     # 40 tokens on every expert: split into 2 dense groups
    (64, 48, 1, 1, 5, 1, False),        # a single expert, k = 1 (weight 1 for both score kinds)
    (128, 96, 12, 3, 256, 0, True),     # the largest T (256): many dense groups
    (2048, 64, 40, 4, 5, 0, True),      # router clusters of 2 slices
    (2560, 128, 24, 3, 40, 1, False),   # clusters of 3 (a ragged slice), two 32-token staging groups
    (8448, 64, 40, 4, 3, 1, False),     # 9 slices: the router without clusters
    # one token: the router writes the logits only, the RVQ kernels route (both many-block
    # router kernels)
    (2048, 64, 40, 4, 1, 0, True),      # clusters of 2 slices, shared expert
    (8448, 64, 40, 4, 1, 1, False),     # 9 slices
    (128, 64, 300, 8, 1, 1, True),      # E > 256, sigmoid + shared
    (264, 200, 33, 3, 1, 0, True),      # ragged k-slice, clusters of one slice
    (256, 64, 64, 32, 1, 1, True),      # k = 32, the most the kernels route: 33 passes with the shared one
    (256, 64, 600, 8, 1, 0, False),     # E > 512: the router routes by itself (32 keys per lane)
])
def test_rvq_odd_shapes(H, F, E, k, T, router, shared):
    _run(LayerSpec(H, F, E, k, S.RVQ, router=router, shared=shared, seed=H + F + E), T)


@pytest.mark.parametrize("H,F,E,k,T,router,shared", [
    (128, 128, 4, 2, 1, 0, False),      # one group per row
    (384, 640, 6, 2, 1, 0, False),      # 3 and 5 groups: ragged 4-group k-slices
    (512, 384, 9, 3, 3, 1, True),       # sigmoid + shared, T = 3
    (256, 256, 40, 4, 4, 0, False),     # one pass carries 4 tokens when they share an expert
    (256, 128, 8, 2, 32, 1, True),      # T = 32: experts with > 4 tokens take several passes
    (128, 128, 1, 1, 3, 0, False),      # a single expert, k = 1
    (256, 256, 12, 3, 256, 1, True),    # the largest T (256): up to 4 tokens per pass, many passes
    (2304, 256, 20, 2, 3, 0, False),    # router clusters of 3 slices, the last ragged
])
def test_int4_odd_shapes(H, F, E, k, T, router, shared):
    _run(LayerSpec(H, F, E, k, S.INT4, router=router, shared=shared, seed=H + F + E), T)


def test_device_generator_matches_host():
    import torch
    from synth import device as D
    for wfmt, H, F in ((S.RVQ, 64, 40), (S.INT4, 256, 128)):
        host = S.make_expert_blob(5, 2, 3, wfmt, H, F)
        dev = torch.empty(host.size, dtype=torch.uint8, device="cuda")
        D.make_expert_blob_device(5, 2, 3, wfmt, H, F, dev)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(dev.cpu().numpy(), host)


def _int4_wide_scale_blob(spec, layer, e, rng):
    """The generator's int4 blob of expert e with every fp16 group scale replaced by a
    random positive value over 20 binades: subnormal (2^-24 and up) to 2^-4, plus zeros.
    The activations stay far inside fp16's range (the kernels carry them as fp16 hi + lo)."""
    blob = spec.blob(layer, e).copy()
    off = 0
    for rows, K in S.matrix_shapes(spec.H, spec.F):
        nb = rows * K // 2
        ns = rows * (K // S.INT4_GROUP)
        expo = rng.integers(0, 12, ns).astype(np.uint16)          # 0 = subnormal, 11 = 2^-4
        mant = rng.integers(0, 1024, ns).astype(np.uint16)
        bits = (expo << 10) | mant
        bits[rng.random(ns) < 0.02] = 0                           # some zero scales
        blob[off + nb:off + nb + 2 * ns] = bits.view(np.uint8)
        off += nb + 2 * ns
    assert off == blob.size
    return blob


@pytest.mark.parametrize("T", [1, 3])
def test_int4_scales_over_the_fp16_range(T):
    """int4 group scales from fp16 subnormals to 2^-4 (the generator's own scales sit in
    [2^-8, 2^-7)): every group's sum is scaled by its own fp16 value on the GPU as in the
    oracle."""
    import routed_expert_ffn_03_gb300 as M
    spec = LayerSpec(512, 384, 6, 2, S.INT4, router=0, seed=91)
    rng = np.random.default_rng(91)
    blobs = {e: _int4_wide_scale_blob(spec, 0, e, rng) for e in range(spec.E)}
    ctx = M.Context(1, spec.H, spec.F, spec.E, spec.k, spec.wfmt, router=spec.router, max_tokens=T)
    try:
        ctx.register_router(0, spec.router_w(0))
        for e in range(spec.E):
            ctx.register_expert(0, e, blobs[e])
        xb = x_tokens(spec.seed, 5, T, spec.H)
        y, idx, w = gpu_forward(ctx, 0, xb)
        r = compare(oracle_forward(spec, 0, xb, dict(blobs)), y, idx, w)
        assert r["rms"] > 0
    finally:
        ctx.close()
