"""moe_route_noalloc: the routing entry point that allocates nothing.

It serves callers that cannot allocate device memory when they route (for example code
recording a CUDA graph, or an engine whose pool owns the free memory); its scratch is a
fixed device array inside the library.  The checks: its expert ids and weights equal the
ones the regular entry point (moe_forward, read back with moe_get_routing) produces for
the same inputs, on two calls in a row, and the ids equal the oracle's (near-ties
excepted).  The shapes take every router kernel through the shared array: the one-block
router, the cluster router with one and with three blocks per SM, and the router with
global partials for more than 8 slices of H.  Two calls queued back to back on one stream
before a single synchronise check that a call's scratch clearing is ordered after the
previous call.  Kept in a file of its own, collected last.
"""
import numpy as np
import pytest

import synth as S
from tests.helpers import NEAR_TIE, LayerSpec, make_context, x_tokens

pytestmark = pytest.mark.gpu

SHAPES = [
    # H, E, k, router, T
    (512, 16, 4, 0, 3),      # one block (E * slices <= 32)
    (512, 40, 5, 1, 3),      # clusters of one slice
    (7168, 384, 16, 0, 1),   # clusters of 7 slices, grid above two blocks per SM
    (9216, 64, 6, 1, 3),     # 9 slices: global partials and tickets
]


def _forward_routing(spec, xbs, T):
    """Routing of moe_forward for each input in xbs (one context)."""
    import torch
    ctx = make_context(spec, max_tokens=T)
    out = torch.empty((T, spec.H), dtype=torch.float32, device="cuda")
    refs = []
    try:
        for xb in xbs:
            x = torch.from_numpy(xb.view(np.int16).copy()).cuda()
            ctx.forward(0, x, out, T)
            torch.cuda.synchronize()
            refs.append(ctx.get_routing(0))
    finally:
        ctx.close()
    return refs


def _check_oracle(spec, xb, idx):
    from oracle import oracle as O
    r = O.router(xb, spec.router_w(0), spec.k, spec.router)
    for t in range(xb.shape[0]):
        if r["gap"][t] >= NEAR_TIE:
            np.testing.assert_array_equal(idx[t], r["idx"][t])


@pytest.mark.parametrize("H,E,k,router,T", SHAPES)
def test_route_noalloc_matches_forward(H, E, k, router, T):
    import torch
    import routed_expert_ffn_03_gb300 as M
    from routed_expert_ffn_03_gb300 import build
    build.build()
    spec = LayerSpec(H, 64, E, k, S.RVQ, router=router, seed=31 + router + H + E)
    xb = x_tokens(spec.seed, 1, T, spec.H)
    (idx_ref, w_ref), = _forward_routing(spec, [xb], T)
    _check_oracle(spec, xb, idx_ref)
    x = torch.from_numpy(xb.view(np.int16).copy()).cuda()
    W = torch.from_numpy(spec.router_w(0)).cuda()
    for _ in range(2):                         # two calls in a row share the scratch
        idx = torch.full((T, spec.k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((T, spec.k), dtype=torch.float32, device="cuda")
        M.route_noalloc(x, W, T, spec.H, spec.E, spec.k, router, idx, w)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref)
        np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("H,E,k,router,T", [SHAPES[1], SHAPES[3]])
def test_route_noalloc_back_to_back_on_one_stream(H, E, k, router, T):
    """Two calls with different inputs queued on one stream, one synchronise after both:
    each call's routing lands in its own output buffers and equals moe_forward's."""
    import torch
    import routed_expert_ffn_03_gb300 as M
    spec = LayerSpec(H, 64, E, k, S.RVQ, router=router, seed=77 + H + E)
    xbs = [x_tokens(spec.seed, i, T, spec.H) for i in (3, 4)]
    refs = _forward_routing(spec, xbs, T)
    W = torch.from_numpy(spec.router_w(0)).cuda()
    xs = [torch.from_numpy(xb.view(np.int16).copy()).cuda() for xb in xbs]
    idxs = [torch.full((T, spec.k), -1, dtype=torch.int32, device="cuda") for _ in xbs]
    ws = [torch.zeros((T, spec.k), dtype=torch.float32, device="cuda") for _ in xbs]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    for x, idx, w in zip(xs, idxs, ws):
        M.route_noalloc(x, W, T, spec.H, spec.E, spec.k, router, idx, w, stream=stream)
    torch.cuda.synchronize()
    for (idx_ref, w_ref), idx, w in zip(refs, idxs, ws):
        np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref)
        np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-5, atol=1e-6)
    assert not np.array_equal(refs[0][0], refs[1][0])


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    import routed_expert_ffn_03_gb300 as M
    x = torch.zeros((256, 16384), dtype=torch.int16, device="cuda")
    W = torch.zeros((1024, 16384), dtype=torch.float32, device="cuda")
    idx = torch.zeros((256, 8), dtype=torch.int32, device="cuda")
    w = torch.zeros((256, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(M.MoeError) as ei:
        M.route_noalloc(x, W, 256, 16384, 1024, 8, 0, idx, w)
    assert ei.value.status == M.EINVAL
