"""Streaming tier and failure handling on the GPU.

The expert cache and the streamed copies change timing only: outputs must be the same
bits as the all-resident run, for any cache size, registration order and expert
labelling ("Introducing WARP", section "How WARP keeps the model out of RAM": the real
choice still comes from the router, prediction changes timing and not results).  Failure
cases are injected on the host; the device-side wait limit is exercised on a flag that
nothing sets.
"""
import numpy as np
import pytest

import synth as S
from tests.helpers import LayerSpec, make_context, x_tokens

pytestmark = pytest.mark.gpu


def _stack_run(ctx, spec, xbits_seq):
    """Feed tokens through all layers with the residual RMS-norm stack; return per-token
    final x (float32) and the per-layer routing."""
    import torch
    T, H = xbits_seq.shape[1], spec.H
    outs, routes = [], []
    x = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    y = torch.zeros_like(x)
    xn = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    for xb in xbits_seq:
        x.copy_(torch.from_numpy(S.bf16_bits_to_f32(xb)))
        for l in range(spec.layers):
            ctx.residual_rmsnorm(x, None if l == 0 else y, xn)
            ctx.forward(l, xn, y, T)
            routes.append(ctx.get_routing(l)[0])
        ctx.residual_rmsnorm(x, y, xn)
        torch.cuda.synchronize()
        outs.append(x.cpu().numpy().copy())
    return np.stack(outs), routes


SPEC = LayerSpec(512, 256, 32, 4, S.RVQ, router=0, seed=21, layers=4)
SPEC4 = LayerSpec(512, 256, 32, 4, S.INT4, router=1, shared=True, seed=22, layers=3)


def _tokens(spec, n, T=1):
    return np.stack([x_tokens(spec.seed, i, T, spec.H) for i in range(n)])


@pytest.mark.parametrize("spec", [SPEC, SPEC4])
def test_file_tier_streamed_equals_resident_bitwise(spec, tmp_path):
    """Experts in a file behind a RAM cache of 2k + 1 records, behind an HBM cache of 2k
    slots: VRAM, then RAM, then the file; the results are those of the all-resident run."""
    import os
    seq = _tokens(spec, 10)
    ref_ctx = make_context(spec, 1)
    ref, ref_routes = _stack_run(ref_ctx, spec, seq)
    ref_ctx.close()
    probe = make_context(spec, 1, hbm_cache_bytes=1 << 40, register=False)
    rb = probe.stats()["record_bytes"]
    probe.close()
    stride = (rb + 4095) // 4096 * 4096
    path = str(tmp_path / "experts.bin")
    for readahead in (0, 1):
        ctx = make_context(spec, 1, hbm_cache_bytes=2 * spec.k * rb, pool_file=path,
                           host_cache_bytes=(2 * spec.k + 1) * stride)
        assert os.path.getsize(path) == spec.layers * spec.E * stride
        ctx.set_readahead(bool(readahead))
        out, routes = _stack_run(ctx, spec, seq)
        st = ctx.stats()
        ctx.close()
        assert not os.path.exists(path)          # the context removes its file
        assert st["misses"] > 0 and st["ram_misses"] > 0 and st["file_reads"] == st["ram_misses"]
        assert st["file_read_bytes"] == st["file_reads"] * stride
        np.testing.assert_array_equal(out, ref)
        for a, b in zip(routes, ref_routes):
            np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("spec", [SPEC, SPEC4])
def test_streamed_equals_resident_bitwise(spec):
    import routed_expert_ffn_03_gb300 as M
    seq = _tokens(spec, 12)
    rec = M.expert_blob_bytes(spec.wfmt, spec.H, spec.F)
    ref_ctx = make_context(spec, 1)
    ref, ref_routes = _stack_run(ref_ctx, spec, seq)
    ref_ctx.close()
    # record size in the kernel layout: ask a context
    probe = make_context(spec, 1, hbm_cache_bytes=1 << 40, register=False)
    rb = probe.stats()["record_bytes"]
    probe.close()
    for slots in (2 * spec.k, 2 * spec.k + 3, 4 * spec.k):
        ctx = make_context(spec, 1, hbm_cache_bytes=slots * rb)
        out, routes = _stack_run(ctx, spec, seq)
        st = ctx.stats()
        ctx.close()
        assert st["cache_slots"] == slots
        assert st["misses"] > 0 and st["hits"] + st["misses"] == st["lookups"]
        assert all(np.array_equal(a, b) for a, b in zip(routes, ref_routes))
        np.testing.assert_array_equal(out, ref)
    assert rec > 0


def test_registration_order_does_not_matter():
    seq = _tokens(SPEC, 4)
    a = make_context(SPEC, 1)
    ra, _ = _stack_run(a, SPEC, seq)
    a.close()
    order = list(np.random.default_rng(3).permutation(SPEC.E))
    b = make_context(SPEC, 1, order=order)
    rb_, _ = _stack_run(b, SPEC, seq)
    b.close()
    np.testing.assert_array_equal(ra, rb_)


def test_expert_relabelling_with_router_rows():
    """Expert e' = perm[e]: blobs and router rows permuted together give the same output."""
    import routed_expert_ffn_03_gb300 as M
    import torch
    spec = LayerSpec(256, 128, 12, 3, S.INT4, router=1, seed=9)
    perm = np.random.default_rng(5).permutation(spec.E)   # new id n holds old expert perm[n]
    xb = x_tokens(9, 0, 3, spec.H)
    outs = []
    for relabel in (False, True):
        ctx = M.Context(1, spec.H, spec.F, spec.E, spec.k, spec.wfmt, router=spec.router, max_tokens=3)
        W = spec.router_w(0)
        ctx.register_router(0, W[perm] if relabel else W)
        for n in range(spec.E):
            ctx.register_expert(0, n, spec.blob(0, int(perm[n]) if relabel else n))
        x = torch.from_numpy(xb.view(np.int16).copy()).cuda()
        out = torch.empty((3, spec.H), dtype=torch.float32, device="cuda")
        ctx.forward(0, x, out)
        torch.cuda.synchronize()
        idx, _ = ctx.get_routing(0)
        outs.append((out.cpu().numpy(), idx))
        ctx.close()
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(perm[outs[1][1]], outs[0][1])


def test_cache_below_two_k_records_is_refused():
    import routed_expert_ffn_03_gb300 as M
    with pytest.raises(M.MoeError) as ei:
        make_context(SPEC, 1, hbm_cache_bytes=1000, register=False)
    assert ei.value.status == M.EBUDGET


@pytest.mark.parametrize("spec", [SPEC, SPEC4])
def test_multi_token_streamed_equals_resident_bitwise(spec, tmp_path):
    """T = 4: a forward may pin min(E, 4 k) experts, so the HBM cache needs that many
    slots (one fewer is refused at create).  With exactly that many, and with the file
    tier's RAM cache (2 k + 1 records) smaller than a forward's misses (read in chunks),
    the results are those of the all-resident run."""
    import routed_expert_ffn_03_gb300 as M
    T = 4
    seq = _tokens(spec, 6, T)
    ref_ctx = make_context(spec, T)
    ref, ref_routes = _stack_run(ref_ctx, spec, seq)
    ref_ctx.close()
    probe = make_context(spec, T, hbm_cache_bytes=1 << 40, register=False)
    rb = probe.stats()["record_bytes"]
    probe.close()
    need = max(2 * spec.k, min(spec.E, T * spec.k))
    with pytest.raises(M.MoeError) as ei:
        make_context(spec, T, hbm_cache_bytes=(need - 1) * rb, register=False)
    assert ei.value.status == M.EBUDGET
    stride = (rb + 4095) // 4096 * 4096
    for pool_file in (None, str(tmp_path / "experts.bin")):
        ctx = make_context(spec, T, hbm_cache_bytes=need * rb, pool_file=pool_file,
                           host_cache_bytes=(2 * spec.k + 1) * stride if pool_file else 0)
        out, routes = _stack_run(ctx, spec, seq)
        st = ctx.stats()
        ctx.close()
        assert st["misses"] > 0
        np.testing.assert_array_equal(out, ref)
        for a, b in zip(routes, ref_routes):
            np.testing.assert_array_equal(a, b)


def test_forward_before_registration_and_bad_args():
    import torch
    import routed_expert_ffn_03_gb300 as M
    ctx = make_context(SPEC, 2, register=False)
    x = torch.zeros((2, SPEC.H), dtype=torch.int16, device="cuda")
    out = torch.zeros((2, SPEC.H), dtype=torch.float32, device="cuda")
    with pytest.raises(M.MoeError) as ei:
        ctx.forward(0, x, out, 1)
    assert ei.value.status == M.ESTATE
    with pytest.raises(M.MoeError) as ei:
        ctx.forward(0, x, out, 3)            # T > max_tokens
    assert ei.value.status == M.EINVAL
    with pytest.raises(M.MoeError) as ei:
        ctx.forward(SPEC.layers, x, out, 1)  # layer out of range
    assert ei.value.status == M.EINVAL
    with pytest.raises(M.MoeError) as ei:
        ctx.register_expert(0, 0, np.zeros(10, dtype=np.uint8))
    assert ei.value.status == M.EINVAL
    with pytest.raises(M.MoeError) as ei:
        ctx.get_routing(0)
    assert ei.value.status == M.ENOTFOUND
    ctx.close()


def test_failed_miss_copy_is_sticky():
    import torch
    import routed_expert_ffn_03_gb300 as M
    probe = make_context(SPEC, 1, hbm_cache_bytes=1 << 40, register=False)
    rb = probe.stats()["record_bytes"]
    probe.close()
    ctx = make_context(SPEC, 1, hbm_cache_bytes=2 * SPEC.k * rb)
    x = torch.from_numpy(x_tokens(1, 0, 1, SPEC.H).view(np.int16).copy()).cuda()
    out = torch.zeros((1, SPEC.H), dtype=torch.float32, device="cuda")
    ctx.debug_fail_copies(1)
    with pytest.raises(M.MoeError) as ei:
        ctx.forward(0, x, out, 1)
    assert ei.value.status == M.ECUDA
    with pytest.raises(M.MoeError) as ei:     # sticky: the next call fails too
        ctx.forward(0, x, out, 1)
    assert ei.value.status == M.ECUDA
    st, _ = ctx.stats_status()
    assert st == M.ECUDA
    ctx.close()


def test_bounded_device_wait_reports_timeout():
    ctx = make_context(SPEC, 1, register=False)
    import routed_expert_ffn_03_gb300 as M
    assert ctx.debug_wait_timeout(100000) == M.ETIMEOUT
    st, _ = ctx.stats_status()               # the check does not poison the context
    assert st == M.OK
    ctx.close()


# wide rows: the single-block router (8 experts x 4 slices), the cluster router (16
# experts x 7 slices, a cluster per expert group) and the one for more than 8 slices
SPEC_H4K = LayerSpec(4096, 256, 8, 2, S.INT4, router=0, seed=23, layers=2)
SPEC_H7K = LayerSpec(7168, 256, 16, 4, S.RVQ, router=0, seed=24, layers=2)
SPEC_H9K = LayerSpec(8448, 128, 24, 4, S.RVQ, router=1, seed=25, layers=2)


@pytest.mark.parametrize("spec,T", [(SPEC, 1), (SPEC4, 1), (SPEC_H4K, 1), (SPEC_H7K, 1), (SPEC_H7K, 4),
                                    (SPEC_H9K, 1), (SPEC_H9K, 3)])
def test_fused_stack_step_equals_separate_calls(spec, T):
    """moe_forward_residual == moe_residual_rmsnorm + moe_forward, bit for bit."""
    import torch
    ctx = make_context(spec, T)
    seq = _tokens(spec, 5, T)
    ref, _ = _stack_run(ctx, spec, seq)
    outs = []
    H = spec.H
    x = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    y = torch.zeros_like(x)
    xn = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    for xb in seq:
        x.copy_(torch.from_numpy(S.bf16_bits_to_f32(xb)))
        for l in range(spec.layers):
            ctx.forward_residual(l, x, None if l == 0 else y, xn, y, T)
        ctx.residual_rmsnorm(x, y, xn)
        torch.cuda.synchronize()
        outs.append(x.cpu().numpy().copy())
    ctx.close()
    np.testing.assert_array_equal(np.stack(outs), ref)


def _fused_run(ctx, spec, xbits_seq):
    import torch
    T, H = xbits_seq.shape[1], spec.H
    outs = []
    x = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    y = torch.zeros_like(x)
    xn = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    for xb in xbits_seq:
        x.copy_(torch.from_numpy(S.bf16_bits_to_f32(xb)))
        for l in range(spec.layers):
            ctx.forward_residual(l, x, None if l == 0 else y, xn, y, T)
        ctx.residual_rmsnorm(x, y, xn)
        torch.cuda.synchronize()
        outs.append(x.cpu().numpy().copy())
    return np.stack(outs)


@pytest.mark.parametrize("spec", [SPEC, SPEC4])
def test_readahead_changes_timing_not_bits(spec):
    """Read-ahead copies of predicted experts (right or wrong) leave every bit as the
    resident run's, including when a miss or another prediction evicts a slot whose
    read-ahead copy is still in flight (the smallest cache)."""
    seq = _tokens(spec, 12)
    ref_ctx = make_context(spec, 1)
    ref, ref_routes = _stack_run(ref_ctx, spec, seq)
    ref_f = _fused_run(ref_ctx, spec, seq)
    ref_ctx.close()
    probe = make_context(spec, 1, hbm_cache_bytes=1 << 40, register=False)
    rb = probe.stats()["record_bytes"]
    probe.close()
    for slots in (2 * spec.k, 3 * spec.k, 4 * spec.k):
        ctx = make_context(spec, 1, hbm_cache_bytes=slots * rb)
        ctx.set_readahead(True)
        out, routes = _stack_run(ctx, spec, seq)
        out_f = _fused_run(ctx, spec, seq)
        st = ctx.stats()
        ctx.close()
        assert all(np.array_equal(a, b) for a, b in zip(routes, ref_routes))
        np.testing.assert_array_equal(out, ref)
        np.testing.assert_array_equal(out_f, ref_f)
        assert st["prefetches"] > 0
        assert 0 <= st["prefetch_hits"] <= st["prefetches"]
        assert st["hits"] + st["misses"] == st["lookups"]
        assert st["bytes_h2d"] == (st["misses"] + st["prefetches"]) * rb
        assert st["h2d_ms"] > 0


def test_readahead_arguments():
    import routed_expert_ffn_03_gb300 as M
    from routed_expert_ffn_03_gb300.moe import lib
    res = make_context(SPEC, 1, register=False)
    with pytest.raises(M.MoeError) as ei:       # nothing to read ahead into: all resident
        res.set_readahead(True)
    assert ei.value.status == M.EINVAL
    res.set_readahead(False)
    res.close()
    probe = make_context(SPEC, 1, hbm_cache_bytes=1 << 40, register=False)
    rb = probe.stats()["record_bytes"]
    probe.close()
    ctx = make_context(SPEC, 1, hbm_cache_bytes=2 * SPEC.k * rb, register=False)
    assert lib().moe_set_readahead(ctx._h, 2) == M.EINVAL
    assert lib().moe_set_readahead(ctx._h, -1) == M.EINVAL
    assert lib().moe_set_readahead(None, 1) == M.EINVAL
    ctx.set_readahead(True)
    ctx.set_readahead(False)
    ctx.close()


def test_engine_lru_matches_the_host_replay():
    """The cache's hits and misses equal a host replay of the same routing trace through
    the LRU rules the hit-rate sweep uses (record granularity, ascending ids, current layer
    kept)."""
    import os
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    probe = make_context(SPEC, 1, hbm_cache_bytes=1 << 40, register=False)
    rb = probe.stats()["record_bytes"]
    probe.close()
    seq = _tokens(SPEC, 16)
    for slots in (2 * SPEC.k, 3 * SPEC.k + 1):
        ctx = make_context(SPEC, 1, hbm_cache_bytes=slots * rb)
        _, routes = _stack_run(ctx, SPEC, seq)
        st = ctx.stats()
        ctx.close()
        trace = [(i % SPEC.layers, r[0]) for i, r in enumerate(routes)]
        rate = bench.lru_hit_rate(trace, slots, SPEC.k)
        assert st["lookups"] == sum(len(set(r[0])) for r in routes)
        assert st["hits"] == round(rate * st["lookups"])


def test_launch_count_in_stats():
    """moe_stats counts the kernels the forward calls queue: router, gate/up, down and
    combine per layer (7 when the dense path serves experts with many tokens), one per
    residual RMS norm."""
    import torch
    spec = LayerSpec(256, 128, 8, 2, S.RVQ, router=0, seed=41)
    for T, per_forward in ((1, 4), (16, 7)):
        ctx = make_context(spec, T)
        try:
            ctx.reset_stats()
            xb = x_tokens(41, 0, T, spec.H)
            x = torch.from_numpy(xb.view(np.int16).copy()).cuda()
            out = torch.empty((T, spec.H), dtype=torch.float32, device="cuda")
            ctx.forward(0, x, out, T)
            xr = torch.zeros((T, spec.H), dtype=torch.float32, device="cuda")
            xn = torch.zeros((T, spec.H), dtype=torch.int16, device="cuda")
            ctx.residual_rmsnorm(xr, out, xn, T)
            torch.cuda.synchronize()
            assert ctx.stats()["launches"] == per_forward + 1
            ctx.reset_stats()
            assert ctx.stats()["launches"] == 0
        finally:
            ctx.close()
