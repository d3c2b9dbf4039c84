"""GPU parity at the workloads' full layer sizes, one layer each, in the launch
configuration the benchmark uses (one block per SM, whole-layer forward through the C
ABI).  Expert blobs are registered from the device generator; the oracle reads the same
bytes generated on the host (the two generators are bit-identical, tested elsewhere)."""
import numpy as np
import pytest

import synth as S
from tests.helpers import LayerSpec, compare, gpu_forward, oracle_forward, x_tokens

pytestmark = pytest.mark.gpu


def _register_device(spec, max_tokens):
    import torch
    import routed_expert_ffn_03_gb300 as M
    from synth import device as D
    ctx = M.Context(1, spec.H, spec.F, spec.E, spec.k, spec.wfmt, router=spec.router,
                    shared_ffn=spec.F if spec.shared else 0, max_tokens=max_tokens)
    ctx.register_router(0, spec.router_w(0))
    blob = torch.empty(S.expert_blob_bytes(spec.wfmt, spec.H, spec.F), dtype=torch.uint8, device="cuda")
    for e in list(range(spec.E)) + ([-1] if spec.shared else []):
        D.make_expert_blob_device(spec.seed, 0, e, spec.wfmt, spec.H, spec.F, blob)
        ctx.register_expert(0, e, blob)
    torch.cuda.synchronize()
    return ctx


@pytest.mark.parametrize("name,spec,Ts,trace", [
    ("mixtral", LayerSpec(4096, 14336, 8, 2, S.INT4, router=0, seed=0), (1, 4), "iid"),
    ("dsv3", LayerSpec(7168, 2048, 256, 8, S.RVQ, router=1, shared=True, seed=0), (1, 4, 32), "iid"),
    ("wide", LayerSpec(7168, 1536, 384, 16, S.RVQ, router=0, seed=0), (1,), "domain"),
])
def test_full_layer(name, spec, Ts, trace):
    ctx = _register_device(spec, max(Ts))
    try:
        for T in Ts:
            if trace == "domain":
                xb = S.f32_to_bf16_bits(S.make_domain_trace(0, 300, T, spec.H))
            else:
                xb = x_tokens(7, T, T, spec.H)
            y, idx, w = gpu_forward(ctx, 0, xb)
            r = compare(oracle_forward(spec, 0, xb), y, idx, w)
            print(name, T, r)
    finally:
        ctx.close()
