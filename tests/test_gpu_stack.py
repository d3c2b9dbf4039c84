"""The residual stack step on the GPU against the oracle, at full layer sizes.

Every layer of the benchmarked stacks runs moe_forward_residual:
    x += y_prev;  xn = bf16(x / sqrt(mean(x^2) + 1e-6));  y = layer(xn)
("x += moe(rmsnorm(x))", the Mixtral-shaped workload; the same stack form for the
DeepSeek-V3-shaped one, with no norm gain).  Teacher-forced, layer by layer, on three
layers at T = 1 and T = 4 (the norm runs inside the router kernel for both):
  * the residual: x after the call equals fp32(x_before + y_prev) bit for bit;
  * the normalised input: xn equals the oracle's bf16(rmsnorm(x)) on that same x bit for
    bit, except 1-ulp differences at a bf16 rounding tie (tests/helpers.py
    check_rmsnorm_bf16), which are counted and reported;
  * the layer: y against the oracle layer applied to the GPU's own xn, with the expert ids
    and the 1e-3 max(1, RMS) bound of tests/helpers.py compare.
"""
import numpy as np
import pytest

import synth as S
from tests.helpers import LayerSpec, check_rmsnorm_bf16, compare, oracle_forward, register_device

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.mark.parametrize("name,spec", [
    ("mixtral", LayerSpec(4096, 14336, 8, 2, S.INT4, router=0, seed=41, layers=3)),
    ("dsv3", LayerSpec(7168, 2048, 256, 8, S.RVQ, router=1, shared=True, seed=42, layers=3)),
])
def test_stack_step_matches_oracle(name, spec):
    import torch
    import routed_expert_ffn_03_gb300 as M
    ctx = M.Context(spec.layers, spec.H, spec.F, spec.E, spec.k, spec.wfmt, router=spec.router,
                    shared_ffn=spec.F if spec.shared else 0, max_tokens=4)
    try:
        register_device(spec, [ctx])
        blobs = [dict() for _ in range(spec.layers)]
        ties = 0
        for T in (1, 4):
            x0 = S.bf16_bits_to_f32(S.f32_to_bf16_bits(S.make_tokens(spec.seed, 7 + T, T, spec.H)))
            x = torch.from_numpy(x0.copy()).cuda()
            y = torch.zeros((T, spec.H), dtype=torch.float32, device="cuda")
            xn = torch.zeros((T, spec.H), dtype=torch.int16, device="cuda")
            prev_x, prev_y = x0, None
            for l in range(spec.layers):
                ctx.forward_residual(l, x, None if l == 0 else y, xn, y, T, eps=EPS)
                torch.cuda.synchronize()
                x_l = x.cpu().numpy()
                xn_l = xn.cpu().numpy().view(np.uint16)
                y_l = y.cpu().numpy().astype(np.float64)
                idx, w = ctx.get_routing(l)
                expect_x = prev_x if prev_y is None else (prev_x + prev_y).astype(np.float32)
                np.testing.assert_array_equal(x_l, expect_x)
                ties += check_rmsnorm_bf16(x_l, xn_l, EPS)
                r = compare(oracle_forward(spec, l, xn_l, blobs[l]), y_l, idx, w)
                print(name, "T=%d layer %d" % (T, l), r)
                prev_x, prev_y = x_l, y_l.astype(np.float32)
        print(name, "bf16 rounding ties in xn:", ties)
    finally:
        ctx.close()
