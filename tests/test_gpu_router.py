"""Router selection with exactly equal logits, on the GPU.

The top-k order is logits descending with equal logits taken by ascending expert id (the
oracle's stable order).  Router rows that are equal give bit-equal logits on both sides,
so these cases fix the GPU's choice exactly, with no near-tie allowance: rows
W[e] = c_e * u with u exact in a few bits and c_e a small integer level, so the logit of
expert e is c_e * (u . x) and every level is a run of exact ties.  The cases cover few
candidates at the selection threshold, between 32 and 64 of them, and more than 64 (every
logit equal), and the three router kernels (one block, clusters of slices, more than 8
slices), with several tokens (the router's own top-k) and with one (the top-k taken in the
RVQ expert kernels, except behind the one-block router).
"""
import numpy as np
import pytest

import synth as S
from tests.helpers import LayerSpec, compare, gpu_forward, oracle_forward, x_tokens

pytestmark = pytest.mark.gpu


def _levels_router(seed, E, H, n_levels):
    rng = np.random.default_rng(seed)
    u = rng.integers(-8, 9, size=H).astype(np.float32) / np.float32(16.0)
    c = rng.integers(0, n_levels, size=E) if n_levels > 0 else np.zeros(E, dtype=np.int64)
    return (c[:, None].astype(np.float32) * u[None, :]).astype(np.float32), c, u


def _expected(c, s, k):
    """top-k ids of logits c * s, descending, equal logits by ascending id."""
    E = len(c)
    key = [(-(int(c[e]) * s), e) for e in range(E)]
    return [e for _, e in sorted(key)[:k]]


@pytest.mark.parametrize("H,E,k,n_levels,router,T", [
    (256, 32, 8, 4, 0, 3),       # one-block router, 4 levels of about 8
    (1024, 128, 16, 16, 0, 2),   # cluster router (1 slice), about 8 per level: 20-40 candidates
    (2048, 96, 16, 3, 1, 2),     # clusters of 2 slices, 32 per level: 28 and 38 candidates
    (1024, 256, 8, 2, 1, 2),     # 2 levels of about 128: more than 64 candidates
    (1024, 40, 4, 0, 0, 2),      # every logit 0: 40 candidates, ids 0..3
    (7168, 384, 16, 0, 0, 1),    # every logit 0, 384 experts, clusters of 7 slices
    (8448, 72, 8, 6, 1, 2),      # 9 slices (no clusters), 12 per level
    # one token: a router of many blocks writes the logits only and the RVQ kernels take
    # the top-k; the one-block router still routes by itself
    (256, 32, 8, 4, 0, 1),       # one-block router
    (1024, 256, 8, 2, 1, 1),     # clusters, more than 64 candidates
    (8448, 72, 8, 6, 1, 1),      # 9 slices (no clusters)
])
def test_exact_ties_take_the_lower_id(H, E, k, n_levels, router, T):
    import routed_expert_ffn_03_gb300 as M
    spec = LayerSpec(H, 64, E, k, S.RVQ, router=router, seed=H + E)
    W, c, u = _levels_router(H * 7 + E, E, H, n_levels)
    xb = x_tokens(spec.seed, 3, T, H)
    ctx = M.Context(1, H, spec.F, E, k, spec.wfmt, router=router, max_tokens=T)
    try:
        ctx.register_router(0, W)
        for e in range(E):
            ctx.register_expert(0, e, spec.blob(0, e))
        y, idx, w = gpu_forward(ctx, 0, xb)
    finally:
        ctx.close()
    from oracle import oracle as O
    x = O.bf16_value(xb)
    blobs = {}
    ref = O.layer(xb, W, k, router, lambda e: blobs.setdefault(e, spec.blob(0, e)), spec.wfmt, H, spec.F)
    for t in range(T):
        s = float(np.dot(u.astype(np.float64), x[t]))
        assert s != 0.0
        exp = _expected(c, s, k)
        assert list(ref["idx"][t]) == exp, (t, list(ref["idx"][t]), exp)
        assert list(idx[t]) == exp, (t, list(idx[t]), exp)
    compare(ref, y, idx, w)
