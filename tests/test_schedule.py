"""Host logic of the ring schedule (agmm_ring_chunks), checked against the
Pallas TPU kernel's own index formulas and against exact coverage.

tpu_inference "all_gather_matmul.py", _do_o_local_copy: at outer offset s the
left half goes to output block left_o_idx = 2*((my_id + s) mod P) and the right
half to right_o_idx = 2*((my_id - s + P) mod P) + 1, each block being
m_per_device // 2 rows (m_per_device_per_direction)."""
import itertools

import pytest

import all_gather_gemm_agmm_gb300 as agmm


def chunks(P, m, my_id, bh, whole=False):
    return agmm.ring_chunks(P, m, my_id, bh, whole)


def halves_in_order(ch):
    """Collapse chunks into (shard, first src row, rows) runs in visit order."""
    runs = []
    for s, r0, v in zip(ch["shard"], ch["src_row"], ch["valid"]):
        if runs and runs[-1][0] == s and runs[-1][1] + runs[-1][2] == r0 and runs[-1][2] % 1 == 0:
            runs[-1][2] += v
        else:
            runs.append([s, r0, v])
    return runs


@pytest.mark.parametrize("P", range(1, 9))
def test_matches_pallas_output_offsets(agmm_lib, P):
    for m in (2, 8, 16, 64, 256):
        h = m // 2
        for my_id in range(P):
            ch = chunks(P, m, my_id, 128)
            # group chunk runs by ring step: left half then right half
            per = -(-h // 128) + -(-(m - h) // 128)
            for s in range(P):
                step = [(ch["shard"][c], ch["src_row"][c], ch["out_row"][c], ch["valid"][c])
                        for c in range(s * per, (s + 1) * per)]
                left = [t for t in step if t[1] < h]
                right = [t for t in step if t[1] >= h]
                left_o_idx = ((my_id + s) % P) * 2
                right_o_idx = ((my_id - s + P) % P) * 2 + 1
                assert left[0][2] == h * left_o_idx
                assert right[0][2] == h * right_o_idx
                assert sum(t[3] for t in left) == h and sum(t[3] for t in right) == m - h


@pytest.mark.parametrize("whole", [False, True])
@pytest.mark.parametrize("P,m,bh", [(1, 1, 8), (1, 7, 8), (2, 16, 8), (3, 5, 8), (4, 64, 32), (8, 1000, 128),
                                    (8, 1000, 8), (5, 333, 16), (8, 4096, 128), (7, 129, 64), (2, 3, 128)])
def test_every_row_exactly_once(agmm_lib, P, m, bh, whole):
    for my_id in range(P):
        ch = chunks(P, m, my_id, bh, whole)
        seen = {}
        for s, r0, o0, v in zip(ch["shard"], ch["src_row"], ch["out_row"], ch["valid"]):
            assert 1 <= v <= bh
            assert o0 == s * m + r0
            for r in range(v):
                key = o0 + r
                assert key not in seen
                seen[key] = True
        assert sorted(seen) == list(range(P * m))


def test_ring_order_and_direction(agmm_lib):
    # step 0 starts at my_id; left halves walk +1, right halves walk -1
    P, m = 5, 10
    for my_id in range(P):
        ch = chunks(P, m, my_id, 8)
        lefts = [s for s, r0 in zip(ch["shard"], ch["src_row"]) if r0 == 0]
        rights = [s for s, r0 in zip(ch["shard"], ch["src_row"]) if r0 == m // 2]
        assert lefts == [(my_id + s) % P for s in range(P)]
        assert rights == [(my_id - s) % P for s in range(P)]


def test_odd_and_single_row_shards(agmm_lib):
    ch = chunks(3, 1, 2, 8)  # left halves are empty: only right halves of one row
    assert ch["valid"] == [1, 1, 1] and ch["src_row"] == [0, 0, 0]
    assert ch["shard"] == [2, 1, 0]
    ch = chunks(2, 5, 0, 8)  # left 2 rows, right 3 rows
    assert list(zip(ch["src_row"], ch["valid"])) == [(0, 2), (2, 3), (0, 2), (2, 3)]


@pytest.mark.parametrize("P", range(1, 9))
def test_whole_shard_first_visit_order(agmm_lib, P):
    # Whole shards in the order the bidirectional ring first delivers them:
    # step 0 my_id, step s the shards my_id+s (left halves) and my_id-s (right).
    for my_id in range(P):
        ch = chunks(P, 10, my_id, 8, whole=True)
        order = [s for s, r0 in zip(ch["shard"], ch["src_row"]) if r0 == 0]
        want, seen = [], set()
        for s in range(P):
            for shard in ((my_id + s) % P, (my_id - s) % P):
                if shard not in seen:
                    seen.add(shard)
                    want.append(shard)
        assert order == want
