"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each test fixes one part of the oracle to something independent of its own
code: a hand-expanded matrix, a closed form, brute force over all subsets, a
library routine in a special case, or an invariant of the method (relabelling
experts, k = E with a flat router, k = 1).  A plausible slip in the oracle (a
dropped stage, a swapped nibble, a wrong scale group, an inverted sort, a
missing renormalisation, the wrong SwiGLU operand) fails at least one test.
"""
import itertools
import math

import numpy as np
import pytest
from scipy.special import expit, softmax

import synth as S
from oracle import oracle as O

RVQ, INT4 = O.RVQ, O.INT4


# ---------------------------------------------------------------- builders
def rvq_block(codebooks, codes):
    """Boundary matrix block: fp16 [3][256][8] codebooks then u8 [rows][G][3]."""
    cb = np.asarray(codebooks, dtype=np.float16).reshape(3, 256, 8)
    cd = np.asarray(codes, dtype=np.uint8)
    return np.concatenate([cb.view(np.uint8).ravel(), cd.ravel()])


def int4_block(q, scales):
    """Boundary matrix block: nibbles [rows][K/2] (low = even k), fp16 scales."""
    q = np.asarray(q, dtype=np.int64)
    u = (q & 0xF).astype(np.uint8)
    packed = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    sc = np.asarray(scales, dtype=np.float16)
    return np.concatenate([packed.ravel(), sc.view(np.uint8).ravel()])


def bits(x):
    return S.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


# ---------------------------------------------------------------- RVQ decode
def test_rvq_hand_expanded():
    """Two rows, two 8-weight groups, values in sixteenths (exact in fp16)."""
    cb = np.zeros((3, 256, 8))
    cb[0, 1] = np.arange(1, 9) / 16.0
    cb[0, 2] = -1 / 16.0
    cb[1, 5] = np.array([1, 0, 1, 0, 1, 0, 1, 0]) / 16.0
    cb[2, 3] = np.array([0, 0, 0, 0, 0, 0, 0, 1]) / 16.0
    codes = [[[1, 0, 3], [2, 0, 0]],
             [[2, 5, 0], [1, 0, 3]]]
    W = O.dense(RVQ, 2, 16, rvq_block(cb, codes))
    # written out by hand (units of 1/16)
    expect = np.array([
        [1, 2, 3, 4, 5, 6, 7, 9, -1, -1, -1, -1, -1, -1, -1, -1],
        [0, -1, 0, -1, 0, -1, 0, -1, 1, 2, 3, 4, 5, 6, 7, 9],
    ]) / 16.0
    np.testing.assert_array_equal(W, expect)


def test_rvq_single_stage_is_plain_vq():
    """Stages 1 and 2 all zero: each group is one codebook row (plain VQ)."""
    rng = np.random.default_rng(1)
    cb = np.zeros((3, 256, 8))
    cb[0] = rng.normal(0, 0.02, (256, 8)).astype(np.float16)
    rows, K = 5, 64
    codes = rng.integers(0, 256, (rows, K // 8, 3))
    W = O.dense(RVQ, rows, K, rvq_block(cb, codes))
    vq = cb[0][codes[:, :, 0]].reshape(rows, K)      # table lookup
    np.testing.assert_array_equal(W, vq)


def test_rvq_stages_add():
    """Each stage contributes additively: W(all) = W(s0) + W(s1) + W(s2)."""
    rng = np.random.default_rng(2)
    cb = rng.normal(0, 0.02, (3, 256, 8)).astype(np.float16).astype(np.float64)
    rows, K = 4, 32
    codes = rng.integers(0, 256, (rows, K // 8, 3))
    W = O.dense(RVQ, rows, K, rvq_block(cb, codes))
    parts = []
    for s in range(3):
        c = np.zeros_like(cb)
        c[s] = cb[s]
        parts.append(O.dense(RVQ, rows, K, rvq_block(c, codes)))
    np.testing.assert_allclose(W, parts[0] + parts[1] + parts[2], rtol=0, atol=1e-15)


def test_half_decode_all_finite_patterns():
    """The oracle's fp16 decode equals numpy's for every finite fp16 value."""
    allbits = np.arange(65536, dtype=np.uint16)
    vals = allbits.view(np.float16)
    finite = allbits[np.isfinite(vals)]
    n = finite.size
    per = 256 * 8
    for start in range(0, n, per):
        chunk = finite[start:start + per]
        cb = np.zeros((3, 256, 8), dtype=np.uint16)
        cb0 = np.zeros(per, dtype=np.uint16)
        cb0[:chunk.size] = chunk
        cb[0] = cb0.reshape(256, 8)
        codes = np.zeros((256, 1, 3), dtype=np.uint8)
        codes[:, 0, 0] = np.arange(256)
        blk = np.concatenate([cb.view(np.uint8).ravel(), codes.ravel()])
        W = O.dense(RVQ, 256, 8, blk)
        expect = cb0.view(np.float16).astype(np.float64).reshape(256, 8)
        np.testing.assert_array_equal(W, expect)


# ---------------------------------------------------------------- int4 decode
@pytest.mark.parametrize("c", [-8, -5, -1, 0, 1, 3, 7])
def test_int4_constant_codes_closed_form(c):
    """All q = c, one scale s: g_r = c * s * sum(x) for every row."""
    rows, K = 3, 256
    s = 0.0068359375                       # exact in fp16
    blk = int4_block(np.full((rows, K), c), np.full((rows, K // 128), s))
    x = np.random.default_rng(c + 10).normal(size=K)
    g = O.matvec(INT4, rows, K, blk, x)[0]
    np.testing.assert_allclose(g, np.full(rows, c * s * x.sum()), rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("k", [0, 1, 126, 127, 128, 255])
def test_int4_nibble_order_and_group(k):
    """One nonzero q at input k: it lands at column k, scaled by group k//128."""
    rows, K = 2, 256
    q = np.zeros((rows, K), dtype=np.int64)
    q[1, k] = -3
    sc = np.array([[0.25, 0.5], [0.125, 2.0]])
    W = O.dense(INT4, rows, K, int4_block(q, sc))
    expect = np.zeros((rows, K))
    expect[1, k] = -3 * sc[1, k // 128]
    np.testing.assert_array_equal(W, expect)


def test_int4_nibble_byte_layout_by_hand():
    """Byte 0x9F holds q(even) = 0xF = -1 and q(odd) = 0x9 = -7."""
    nib = np.zeros(64, dtype=np.uint8)
    nib[0] = 0x9F
    nib[1] = 0x70          # q2 = 0, q3 = 7
    blk = np.concatenate([nib, np.array([1.0], dtype=np.float16).view(np.uint8)])
    W = O.dense(INT4, 1, 128, blk)
    np.testing.assert_array_equal(W[0, :4], [-1, -7, 0, 7])
    assert not W[0, 4:].any()


# ---------------------------------------------------------------- router
def _brute_topk(scores, k):
    """Best k-subset by total score, ordered by score desc (ties: lower id)."""
    E = scores.size
    best = max(itertools.combinations(range(E), k), key=lambda c: sum(scores[i] for i in c))
    return sorted(best, key=lambda i: (-scores[i], i))


@pytest.mark.parametrize("kind", [O.SOFTMAX, O.SIGMOID])
@pytest.mark.parametrize("E,k", [(6, 1), (6, 3), (7, 4), (5, 5)])
def test_router_brute_force(kind, E, k):
    rng = np.random.default_rng(E * 10 + k + kind)
    H, T = 24, 5
    x = bits(rng.normal(size=(T, H)))
    Wr = rng.normal(0, 1 / math.sqrt(H), (E, H)).astype(np.float32)
    r = O.router(x, Wr, k, kind)
    xv = S.bf16_bits_to_f32(x).astype(np.float64)
    logits = xv @ Wr.astype(np.float64).T                  # library matmul
    np.testing.assert_allclose(r["logits"], logits, rtol=1e-12, atol=1e-12)
    for t in range(T):
        sc = softmax(logits[t]) if kind == O.SOFTMAX else expit(logits[t])
        np.testing.assert_allclose(r["scores"][t], sc, rtol=1e-12)
        sel = _brute_topk(sc, k)
        assert list(r["idx"][t]) == sel
        if kind == O.SOFTMAX:
            w = softmax(logits[t][sel])                    # renormalised over k
        else:
            w = expit(logits[t][sel]) / expit(logits[t][sel]).sum()
        np.testing.assert_allclose(r["w"][t], w, rtol=1e-12)
        if k < E:
            srt = np.sort(sc)[::-1]
            assert r["gap"][t] == pytest.approx(srt[k - 1] - srt[k], abs=1e-15)


def test_router_ties_prefer_lower_id():
    """Equal scores (a zero router) are ranked by ascending expert id."""
    E, H = 6, 8
    x = bits(np.ones((1, H)))
    r = O.router(x, np.zeros((E, H), np.float32), 3, O.SOFTMAX)
    assert list(r["idx"][0]) == [0, 1, 2]
    np.testing.assert_allclose(r["w"][0], [1 / 3] * 3)
    assert r["gap"][0] == 0.0


def test_router_two_expert_softmax_is_logistic():
    """Top-2 of 2 renormalised softmax: w0 = logistic(l0 - l1)."""
    H = 4
    x = bits(np.array([[1.0, 0.0, 0.0, 0.0]]))
    Wr = np.zeros((2, H), np.float32)
    Wr[0, 0], Wr[1, 0] = 0.75, -0.5
    r = O.router(x, Wr, 2, O.SOFTMAX)
    assert list(r["idx"][0]) == [0, 1]
    assert r["w"][0, 0] == pytest.approx(1 / (1 + math.exp(-1.25)), rel=1e-14)


# ---------------------------------------------------------------- SwiGLU expert
def _int4_expert_blob(H, F, cg, cu, cd, sg, su, sd):
    return np.concatenate([
        int4_block(np.full((F, H), cg), np.full((F, H // 128), sg)),
        int4_block(np.full((F, H), cu), np.full((F, H // 128), su)),
        int4_block(np.full((H, F), cd), np.full((H, F // 128), sd)),
    ])


def test_swiglu_closed_form():
    """Constant matrices: g = cg sg X, u = cu su X, y = cd sd F silu(g) u."""
    H, F = 128, 256
    cg, cu, cd, sg, su, sd = 3, -2, 5, 0.0078125, 0.015625, 0.001953125
    blob = _int4_expert_blob(H, F, cg, cu, cd, sg, su, sd)
    x = np.random.default_rng(5).normal(size=(2, H))
    y, h = O.expert(INT4, H, F, blob, x, want_h=True)
    for t in range(2):
        X = x[t].sum()
        g, u = cg * sg * X, cu * su * X
        ht = g * expit(g) * u                               # silu from scipy
        np.testing.assert_allclose(h[t], np.full(F, ht), rtol=1e-12)
        np.testing.assert_allclose(y[t], np.full(H, cd * sd * F * ht), rtol=1e-11)


def test_swiglu_zero_gate_gives_zero():
    H, F = 64, 32
    blob = S.make_expert_blob(7, 0, 0, S.RVQ, H, F).copy()
    # zero the three gate codebooks -> gate matrix == 0 -> h == 0 -> y == 0
    blob[:3 * 256 * 8 * 2] = 0
    y = O.expert(RVQ, H, F, blob, np.random.default_rng(0).normal(size=(3, H)))
    assert not y.any()


def test_expert_equals_dense_numpy():
    """The expert equals numpy's dense linear algebra on the decoded matrices."""
    H, F = 64, 96
    blob = S.make_expert_blob(3, 1, 2, S.RVQ, H, F)
    mb = O.matrix_bytes(RVQ, F, H)
    Wg = O.dense(RVQ, F, H, blob[:mb])
    Wu = O.dense(RVQ, F, H, blob[mb:2 * mb])
    Wd = O.dense(RVQ, H, F, blob[2 * mb:])
    x = np.random.default_rng(1).normal(size=(4, H))
    g, u = x @ Wg.T, x @ Wu.T
    y_np = (g * expit(g) * u) @ Wd.T
    np.testing.assert_allclose(O.expert(RVQ, H, F, blob, x), y_np, rtol=1e-11, atol=1e-14)


# ---------------------------------------------------------------- layer invariants
def _tiny_layer(wfmt, E=5, H=128, F=128, seed=11):
    blobs = {e: S.make_expert_blob(seed, 0, e, wfmt, H, F) for e in range(E)}
    return blobs, H, F


@pytest.mark.parametrize("kind", [O.SOFTMAX, O.SIGMOID])
@pytest.mark.parametrize("wfmt", [RVQ, INT4])
def test_flat_router_all_experts_is_mean(kind, wfmt):
    """k = E and W_r = 0: uniform weights 1/E, so y is the mean of experts."""
    E = 5
    blobs, H, F = _tiny_layer(wfmt, E)
    xb = bits(np.random.default_rng(3).normal(size=(2, H)))
    r = O.layer(xb, np.zeros((E, H), np.float32), E, kind, blobs.__getitem__, wfmt, H, F)
    xv = S.bf16_bits_to_f32(xb).astype(np.float64)
    mean = sum(O.expert(wfmt, H, F, blobs[e], xv) for e in range(E)) / E
    np.testing.assert_allclose(r["y"], mean, rtol=1e-12, atol=1e-15)


def test_top1_is_single_expert():
    E = 5
    blobs, H, F = _tiny_layer(RVQ, E)
    rng = np.random.default_rng(4)
    xb = bits(rng.normal(size=(3, H)))
    Wr = rng.normal(0, 1 / math.sqrt(H), (E, H)).astype(np.float32)
    r = O.layer(xb, Wr, 1, O.SOFTMAX, blobs.__getitem__, RVQ, H, F)
    xv = S.bf16_bits_to_f32(xb).astype(np.float64)
    for t in range(3):
        assert r["w"][t, 0] == 1.0
        np.testing.assert_array_equal(r["y"][t], O.expert(RVQ, H, F, blobs[r["idx"][t, 0]], xv[t:t + 1])[0])


@pytest.mark.parametrize("kind", [O.SOFTMAX, O.SIGMOID])
def test_expert_relabelling_invariance(kind):
    """Permuting expert ids together with the router rows leaves y unchanged."""
    E = 6
    blobs, H, F = _tiny_layer(INT4, E)
    rng = np.random.default_rng(6)
    xb = bits(rng.normal(size=(4, H)))
    Wr = rng.normal(0, 1 / math.sqrt(H), (E, H)).astype(np.float32)
    perm = rng.permutation(E)                      # new id n holds old expert perm[n]
    r0 = O.layer(xb, Wr, 3, kind, blobs.__getitem__, INT4, H, F)
    r1 = O.layer(xb, Wr[perm], 3, kind, lambda n: blobs[perm[n]], INT4, H, F)
    np.testing.assert_allclose(r1["y"], r0["y"], rtol=1e-13, atol=1e-15)
    np.testing.assert_array_equal(perm[r1["idx"]], r0["idx"])


def test_shared_expert_added_with_weight_one():
    E = 4
    blobs, H, F = _tiny_layer(RVQ, E)
    shared = S.make_expert_blob(11, 0, -1, S.RVQ, H, 64)
    rng = np.random.default_rng(8)
    xb = bits(rng.normal(size=(2, H)))
    Wr = rng.normal(0, 1 / math.sqrt(H), (E, H)).astype(np.float32)
    r0 = O.layer(xb, Wr, 2, O.SIGMOID, blobs.__getitem__, RVQ, H, F)
    r1 = O.layer(xb, Wr, 2, O.SIGMOID, blobs.__getitem__, RVQ, H, F, shared, 64)
    xv = S.bf16_bits_to_f32(xb).astype(np.float64)
    np.testing.assert_allclose(r1["y"] - r0["y"], O.expert(RVQ, H, 64, shared, xv), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(r0["w"].sum(axis=1), 1.0, rtol=1e-14)


# ---------------------------------------------------------------- stack pieces
def test_rmsnorm_closed_form():
    xn = O.rmsnorm_bf16(np.array([[3.0, 4.0]]), eps=0.0)
    # mean square 12.5 -> 3/sqrt(12.5), 4/sqrt(12.5), then bf16
    expect = np.array([3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], dtype=np.float32)
    np.testing.assert_array_equal(xn[0], S.f32_to_bf16_bits(expect))
    assert abs(S.bf16_bits_to_f32(xn)[0, 0] - 0.8485) < 4e-3


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 is halfway between bf16 1.0 and 1 + 2^-7: rounds to even (1.0)
    assert O.bf16_bits(np.array([1 + 2 ** -8]))[0] == 0x3F80
    assert O.bf16_bits(np.array([1 + 3 * 2 ** -8]))[0] == 0x3F82
    assert O.bf16_bits(np.array([-2.0]))[0] == 0xC000


# ---------------------------------------------------------------- formats
def _golden_sizes():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "record_sizes.txt")
    rows = []
    for line in open(path):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def test_record_sizes_golden():
    for name, fmt, H, F, nbytes, nexp, approx in _golden_sizes():
        wfmt = RVQ if fmt == "rvq" else INT4
        H, F, nbytes, nexp = int(H), int(F), int(nbytes), int(nexp)
        assert O.expert_bytes(wfmt, H, F) == nbytes, name
        assert S.expert_blob_bytes(wfmt, H, F) == nbytes, name
        if approx != "-":
            assert abs(nbytes * nexp / 1e9 - float(approx)) / float(approx) < 0.03, name


def test_rvq_is_three_bits_per_weight():
    """Code bytes are exactly 3 bits per weight (codebooks extra, 36 KB/expert)."""
    H, F = 7168, 1536
    code_bytes = O.expert_bytes(RVQ, H, F) - 3 * 3 * 256 * 8 * 2
    assert code_bytes * 8 == 3 * (3 * H * F)


# ---------------------------------------------------------------- combine and stack in closed form
SG, SU, SD = 2.0 ** -7, 2.0 ** -6, 2.0 ** -9      # exact fp16 scales


def _const_expert_value(X, F, cg, cu, cd, sg=SG, su=SU, sd=SD):
    """Every output row of an int4 expert whose gate/up/down codes are the constants cg, cu,
    cd (one scale per matrix), on an input whose entries sum to X: g = cg sg X, u = cu su X
    in every row, h = silu(g) u, y = cd sd F h (silu from scipy's logistic)."""
    g, u = cg * sg * X, cu * su * X
    return cd * sd * F * (g * expit(g) * u)


@pytest.mark.parametrize("kind", [O.SOFTMAX, O.SIGMOID])
def test_weighted_combine_unequal_weights_closed_form(kind):
    """k = 2 of 3 experts with unequal weights: y = w_a y_a + w_b y_b written out by hand.

    Router row e is a_e at input 0 and zero elsewhere, and x = (1, 0.5, 0, ...), so the
    logits are exactly a = (0.5, -0.25, 1.0): expert 2 ranks first, expert 0 second.
    Softmax renormalised over the two: w = (1, e^-0.5) / (1 + e^-0.5); sigmoid normalised:
    w = (s(1), s(0.5)) / (s(1) + s(0.5)).  The three experts have different constant codes,
    so pairing a weight with the wrong expert, or the wrong rank order, changes y."""
    H = F = 128
    consts = {0: (3, -2, 5), 1: (-1, 4, 2), 2: (2, 3, -4)}
    blobs = {e: _int4_expert_blob(H, F, *c, SG, SU, SD) for e, c in consts.items()}
    x = np.zeros((1, H))
    x[0, 0], x[0, 1] = 1.0, 0.5
    X = 1.5
    Wr = np.zeros((3, H), np.float32)
    Wr[:, 0] = [0.5, -0.25, 1.0]
    r = O.layer(bits(x), Wr, 2, kind, blobs.__getitem__, INT4, H, F)
    if kind == O.SOFTMAX:
        w_first = 1.0 / (1.0 + math.exp(-0.5))
    else:
        s1, s05 = 1 / (1 + math.exp(-1.0)), 1 / (1 + math.exp(-0.5))
        w_first = s1 / (s1 + s05)
    w_second = 1.0 - w_first
    assert list(r["idx"][0]) == [2, 0]
    np.testing.assert_allclose(r["w"][0], [w_first, w_second], rtol=1e-14)
    y2 = _const_expert_value(X, F, *consts[2])
    y0 = _const_expert_value(X, F, *consts[0])
    expect = w_first * y2 + w_second * y0
    np.testing.assert_allclose(r["y"][0], np.full(H, expect), rtol=1e-12)
    # the pin separates the right pairing from the swapped one by far more than its tolerance
    assert abs((w_second * y2 + w_first * y0) - expect) > 1e-3 * abs(expect)


def test_stack_two_layers_closed_form():
    """Two layers of one constant-code int4 expert each (k = 1, weight 1), written out by hand.

    x0 = 2 s with s = +1 on the first 80 of 128 entries and -1 on the rest.  Layer 0 sees
    xn0 = bf16(x0 / sqrt(4 + eps)) = s exactly, so X0 = 32 and y0 is the constant v0; then
    x1 = 2 s + v0 has two distinct values a+, a-, mean square 4 + v0^2 + 2*2*v0*32/128, and
    layer 1 sees their bf16-rounded normalised values, X1 = 80 n+ + 48 n-; y1 = v1 and
    x2 = x1 + v1.  A wrong layer order, a dropped residual or a norm of the wrong x fails."""
    H = F = 128
    eps = 1e-6
    s = np.where(np.arange(H) < 80, 1.0, -1.0)
    c0, c1 = (3, -2, 5), (-1, 4, 7)
    blob0 = _int4_expert_blob(H, F, *c0, SG, SU, SD)
    blob1 = _int4_expert_blob(H, F, *c1, SG, SU, 2.0 ** -7)
    one = np.ones((1, H), np.float32)
    layers = [lambda xn: O.layer(xn, one, 1, O.SOFTMAX, lambda e: blob0, INT4, H, F),
              lambda xn: O.layer(xn, one, 1, O.SOFTMAX, lambda e: blob1, INT4, H, F)]
    x_final, res = O.stack((2.0 * s)[None, :], layers, eps=eps)

    np.testing.assert_array_equal(res[0]["xn"][0], bits(s))
    v0 = _const_expert_value(32.0, F, *c0)
    ms1 = 4.0 + v0 * v0 + 2 * 2.0 * v0 * 32.0 / 128.0
    n_plus = float(S.bf16_bits_to_f32(bits(np.float32((2.0 + v0) / math.sqrt(ms1 + eps)))))
    n_minus = float(S.bf16_bits_to_f32(bits(np.float32((-2.0 + v0) / math.sqrt(ms1 + eps)))))
    np.testing.assert_array_equal(res[1]["xn"][0], bits(np.where(s > 0, n_plus, n_minus)))
    v1 = _const_expert_value(80 * n_plus + 48 * n_minus, F, *c1, sd=2.0 ** -7)
    assert abs(v0) > 0.1 and abs(v1) > 0.01
    np.testing.assert_allclose(x_final[0], 2.0 * s + v0 + v1, rtol=1e-12, atol=1e-14)
