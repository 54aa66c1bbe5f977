"""Host-side report arithmetic used by bench.py (CPU only): the per-shard
closed forms agree with the planner, the shard positions with the oracle's
position map, and the synchronous ring time is the sum of per-step maxima."""
import pytest

import ring_sequence_parallelism_gb300 as ra
from ring_sequence_parallelism_gb300 import report


@pytest.mark.parametrize("layout", ["contiguous", "striped", "zigzag"])
@pytest.mark.parametrize("P,n", [(1, 256), (4, 256), (8, 1024), (16, 8192)])
def test_closed_forms_match_planner(layout, P, n):
    att = ra.RingAttention(1, 2, P * n, 64, P, causal=True, layout=layout)
    pairs, _ = att.shard_work()
    att.close()
    assert [2 * x for x in report.shard_pairs_closed_form(layout, n, P)] == pairs


@pytest.mark.parametrize("layout,lid", [("contiguous", 0), ("striped", 1), ("zigzag", 2)])
def test_shard_positions_match_oracle(orc, layout, lid):
    P, n = 4, 12
    seen = []
    for r in range(P):
        pos = report.shard_positions(layout, n, P, r)
        assert pos == [orc.position(lid, n, P, r, i) for i in range(n)]
        seen += pos
    assert sorted(seen) == list(range(P * n))


def test_synchronous_ring_time():
    # step 0: shards take 1 and 3 ms, step 1: 2 and 2 ms -> 3 + 2
    assert report.synchronous_ring_ms([[1.0, 3.0], [2.0, 2.0]]) == 5.0
    assert report.imbalance([2.0, 8.0]) == 4.0
