"""moe_route_noalloc: the routing entry point that allocates nothing.

It serves callers that cannot allocate device memory when they route (for example code
recording a CUDA graph, or an engine whose pool owns the free memory); its scratch is a
fixed device array inside the library.  The check: its expert ids and weights equal the
ones the regular entry point (moe_forward, read back with moe_get_routing) produces for
the same inputs, on two calls in a row.  Kept in a file of its own, collected last.
"""
import numpy as np
import pytest

import synth as S
from tests.helpers import LayerSpec, make_context, x_tokens

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("router", [0, 1])
def test_route_noalloc_matches_forward(router):
    import torch
    import routed_expert_ffn_03_gb300 as M
    from routed_expert_ffn_03_gb300 import build
    build.build()
    spec = LayerSpec(512, 128, 40, 5, S.INT4, router=router, seed=31 + router)
    T = 3
    ctx = make_context(spec, max_tokens=T)
    xb = x_tokens(spec.seed, 1, T, spec.H)
    x = torch.from_numpy(xb.view(np.int16).copy()).cuda()
    out = torch.empty((T, spec.H), dtype=torch.float32, device="cuda")
    ctx.forward(0, x, out, T)
    torch.cuda.synchronize()
    idx_ref, w_ref = ctx.get_routing(0)
    ctx.close()
    W = torch.from_numpy(spec.router_w(0)).cuda()
    for _ in range(2):                         # two calls in a row share the scratch
        idx = torch.full((T, spec.k), -1, dtype=torch.int32, device="cuda")
        w = torch.zeros((T, spec.k), dtype=torch.float32, device="cuda")
        M.route_noalloc(x, W, T, spec.H, spec.E, spec.k, router, idx, w)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref)
        np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=1e-5, atol=1e-6)


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
