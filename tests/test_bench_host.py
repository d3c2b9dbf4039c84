"""Host-side logic of the measurement script: the LRU replay behind the hit-rate sweep."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def test_lru_replay_small_cases():
    import bench
    tr = [(0, [0, 1]), (0, [0, 1]), (0, [2, 3]), (0, [0, 1])]
    assert bench.lru_hit_rate(tr, 2, 2) == pytest.approx(2 / 8)   # [2,3] evicts both
    assert bench.lru_hit_rate(tr, 4, 2) == pytest.approx(4 / 8)
    assert bench.lru_hit_rate(tr, 4, 1) == pytest.approx(2 / 4)   # top-1 of each list
    # least recently used goes first: 0 is touched again, so 1 is evicted by 2
    tr = [(0, [0, 1]), (0, [0]), (1, [2])]
    assert bench.lru_hit_rate(tr + [(0, [0])], 2, 2) == pytest.approx(2 / 5)
    assert bench.lru_hit_rate(tr + [(0, [1])], 2, 2) == pytest.approx(1 / 5)


def test_lru_replay_keeps_the_current_layer():
    import bench
    # 2 slots, a layer that needs both: its own first expert is never the victim
    tr = [(0, [5]), (1, [7, 8]), (1, [7, 8])]
    assert bench.lru_hit_rate(tr, 2, 2) == pytest.approx(2 / 5)
