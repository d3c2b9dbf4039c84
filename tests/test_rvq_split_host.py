"""The RVQ lookup kernel's block split, on the host (moe_rvq_block_split runs the same
functions as the kernel): every task is taken by exactly one block, ranges inside a unit
start and end at rounds of 16 tasks unless the equal task ranges were cheaper, no block
costs more than under equal task ranges
(cost = rounds of 16 tasks plus one table build per unit touched), and the DeepSeek-V3
gate/up case (252 units of 64 tasks over 152 blocks) gives the groups of 3 blocks over 5
units worked out by hand."""
import pytest

SEG, RND, NW = 7, 8, 16   # the kernel's cost units: a table build, a round of 16 tasks


@pytest.fixture(scope="module")
def M():
    from routed_expert_ffn_03_gb300 import build
    build.build()
    import routed_expert_ffn_03_gb300 as M
    return M


def cost(t0, t1, n):
    c, i = 0, t0
    while i < t1:
        u = i // n
        e = min(t1, (u + 1) * n)
        c += SEG + RND * (-(-(e - i) // NW))
        i = e
    return c


@pytest.mark.parametrize("grid", [152, 148, 16, 7, 2])
@pytest.mark.parametrize("n", [64, 48, 224, 16, 17, 1])
def test_split_is_a_partition_on_round_boundaries(M, grid, n):
    for u_n in range(grid + 1, 2 * grid):
        t0, t1 = M.rvq_block_split(u_n, n, grid)
        assert t0[0] == 0 and t1[-1] == u_n * n
        assert all(t1[b] == t0[b + 1] for b in range(grid - 1))
        assert all(a <= b for a, b in zip(t0, t1))
        eq_t0 = [u_n * n * b // grid for b in range(grid)]
        if t0 != eq_t0:   # grouped: a block starts at a unit start or whole rounds into it
            assert all((a % n) % NW == 0 for a in t0), (u_n, n, grid)
        eq = max(cost(u_n * n * b // grid, u_n * n * (b + 1) // grid, n) for b in range(grid))
        got = max(cost(a, b, n) for a, b in zip(t0, t1))
        assert got <= eq, (u_n, n, grid, got, eq)


def test_deepseek_v3_gate_up_split(M):
    t0, t1 = M.rvq_block_split(252, 64, 152)
    # 50 groups of 3 blocks over 5 units (320 tasks): unit 0 and 3 rounds of unit 1; the
    # last round of unit 1, unit 2 and the first round of unit 3; the rest of unit 3 and
    # unit 4.  Then 2 blocks over the last 2 units, one each.
    for g in range(50):
        base = 320 * g
        assert (t0[3 * g], t1[3 * g]) == (base, base + 112)
        assert (t0[3 * g + 1], t1[3 * g + 1]) == (base + 112, base + 208)
        assert (t0[3 * g + 2], t1[3 * g + 2]) == (base + 208, base + 320)
    assert (t0[150], t1[150], t0[151], t1[151]) == (16000, 16064, 16064, 16128)


def test_outside_the_range_is_refused(M):
    for u_n in (152, 304, 0):
        with pytest.raises(ValueError):
            M.rvq_block_split(u_n, 64, 152)
