"""The RAM + file tier of the streamed expert store on its own (host code, no GPU):
records round-trip through the file, the RAM cache evicts the least recently used
record, a write drops the stale RAM copy, and the argument checks."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def M():
    from routed_expert_ffn_03_gb300 import build
    build.build()
    import routed_expert_ffn_03_gb300 as M
    return M


def _recs(n, nbytes, seed=0):
    rng = np.random.default_rng(seed)
    return [rng.integers(0, 256, size=nbytes, dtype=np.uint8) for _ in range(n)]


def test_round_trip_and_lru(M, tmp_path):
    rec = 5000
    recs = _recs(10, rec)
    ft = M.FileTier(tmp_path / "pool.bin", rec, 10, 3 * 8192)
    try:
        info = ft.info()
        assert info["slots"] == 3 and info["stride"] == 8192 and info["direct"] in (0, 1)
        for k, r in enumerate(recs):
            ft.write(k, r)
        got, slots = ft.fetch([0, 1, 2])
        assert [bytes(r) for r in recs[:3]] == got
        assert sorted(slots) == [0, 1, 2]
        assert ft.info()["reads"] == 3
        got, s1 = ft.fetch([1])                 # hit: 1 becomes the most recent
        assert got[0] == bytes(recs[1]) and s1[0] == slots[1]
        assert ft.info()["reads"] == 3 and ft.info()["ram_hits"] == 1
        got, s3 = ft.fetch([3])                 # evicts 0, the least recently used
        assert got[0] == bytes(recs[3]) and s3[0] == slots[0]
        got, s0 = ft.fetch([0])                 # 0 is read again and evicts 2
        assert got[0] == bytes(recs[0]) and s0[0] == slots[2]
        info = ft.info()
        assert info["reads"] == 5 and info["ram_misses"] == 5 and info["read_bytes"] == 5 * 8192
        got, _ = ft.fetch([1, 3, 0])            # all resident
        assert got == [bytes(recs[1]), bytes(recs[3]), bytes(recs[0])]
        assert ft.info()["reads"] == 5
    finally:
        ft.close()


def test_write_drops_the_ram_copy(M, tmp_path):
    rec = 4096
    a, b = _recs(2, rec, seed=1)
    ft = M.FileTier(tmp_path / "pool.bin", rec, 4, 2 * 4096)
    try:
        ft.write(2, a)
        assert ft.fetch([2])[0][0] == bytes(a)
        ft.write(2, b)
        assert ft.fetch([2])[0][0] == bytes(b)
        assert ft.info()["reads"] == 2
        assert ft.fetch([3])[0][0] == bytes(rec)   # never written: zeros
    finally:
        ft.close()


def test_parallel_batch(M, tmp_path):
    rec = (1 << 20) + 100
    recs = _recs(48, rec, seed=2)
    ft = M.FileTier(tmp_path / "pool.bin", rec, 48, 32 * ((rec + 4095) // 4096 * 4096))
    try:
        for k, r in enumerate(recs):
            ft.write(k, r)
        keys = list(range(40, 8, -1))          # 32 keys, one batch, read on the reader threads
        got, slots = ft.fetch(keys)
        assert got == [bytes(recs[k]) for k in keys]
        assert len(set(slots)) == 32
        keys2 = list(range(0, 16))             # half hits (9..15), half misses evicting the oldest
        got, _ = ft.fetch(keys2)
        assert got == [bytes(recs[k]) for k in keys2]
        assert ft.info()["ram_hits"] == 7
    finally:
        ft.close()


def test_argument_checks(M, tmp_path):
    with pytest.raises(M.MoeError) as e:
        M.FileTier(tmp_path / "p.bin", 5000, 4, 4096)        # RAM below one record
    assert e.value.status == M.EBUDGET
    with pytest.raises(M.MoeError) as e:
        M.FileTier(tmp_path / "no_such_dir" / "p.bin", 5000, 4, 8192)
    assert e.value.status == M.EIO
    ft = M.FileTier(tmp_path / "p.bin", 5000, 4, 2 * 8192)
    try:
        with pytest.raises(M.MoeError) as e:
            ft.fetch([0, 1, 2])                               # more keys than slots
        assert e.value.status == M.EINVAL
        with pytest.raises(M.MoeError) as e:
            ft.fetch([4])                                     # key out of range
        assert e.value.status == M.EINVAL
        with pytest.raises(M.MoeError) as e:
            ft.write(-1, np.zeros(5000, dtype=np.uint8))
        assert e.value.status == M.EINVAL
    finally:
        ft.close()
