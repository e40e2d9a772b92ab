"""The split-KV planner's algorithm on the host (mla_decode_plan_host): schedule properties.

The device planner runs the same integer arithmetic; test_gpu_plan.py checks
that both write identical bytes.
"""

import numpy as np
import pytest

import workloads as W

m = pytest.importorskip("mla_decode_attention_02_gb300")

def _check_schedule(seq_lens, s_q, units, max_pages=None):
    seq_lens = [int(x) for x in seq_lens]
    if max_pages is None:
        max_pages = max((L + 63) // 64 for L in seq_lens)
    r = m.plan_host(seq_lens, s_q=s_q, max_pages_per_seq=max_pages, num_units=units)
    h, items, ub = r["header"], r["items"], r["unit_begin"]
    min_split = int(h["min_split"])          # the planner's shortest piece (a tuning constant)
    assert min_split >= 1
    R = len(seq_lens) * s_q
    assert h["num_rows"] == R and h["num_units"] == units and h["num_items"] == len(items)
    assert h["num_items"] <= h["max_items"]
    # every row is covered exactly once, in order, by page-aligned pieces
    parts_seen = []
    by_row = {}
    for row, j0, j1, part in items.tolist():
        by_row.setdefault(row, []).append((j0, j1, part))
    assert sorted(by_row) == list(range(R)) or h["status"] != 0
    for row in range(R):
        b, t = divmod(row, s_q)
        vis = seq_lens[b] - s_q + 1 + t
        pieces = by_row[row]
        assert r["row_nparts"][row] == len(pieces)
        assert pieces[0][0] == 0 and pieces[-1][1] == vis
        for (a0, a1, _), (c0, c1, _) in zip(pieces, pieces[1:]):
            assert a1 == c0
        for j0, j1, part in pieces:
            assert j0 % 64 == 0 and j1 > j0
            if len(pieces) > 1:
                assert (j1 - j0 + 63) // 64 >= min_split
        if len(pieces) == 1:
            assert pieces[0][2] == -1 and r["row_part0"][row] == -1
        else:
            parts = [p for _, _, p in pieces]
            assert parts == list(range(parts[0], parts[0] + len(parts)))
            assert r["row_part0"][row] == parts[0]
            parts_seen += parts
    assert sorted(parts_seen) == list(range(h["num_parts"]))
    # items are grouped by unit, units non-decreasing, unit_begin consistent
    unit = r["item_unit"]
    assert np.all(np.diff(unit) >= 0) and (len(unit) == 0 or (unit[0] >= 0 and unit[-1] < units))
    assert ub[0] == 0 and ub[-1] == len(items) and np.all(np.diff(ub) >= 0)
    for u in range(units):
        assert np.all(unit[ub[u]:ub[u + 1]] == u)
    # balance: every unit's load (pages + per-item cost) stays near the target; the
    # per-item cost (a tuning constant of the planner) follows from the header's total
    row_pages = [(seq_lens[r // s_q] - s_q + 1 + r % s_q + 63) // 64 for r in range(R)]
    busy_rows = sum(1 for x in row_pages if x > 0)
    if h["status"] != 0 or busy_rows == 0:
        return r, None
    item_cost = (h["total_cost"] - sum(row_pages)) // busy_rows
    assert h["total_cost"] == sum(row_pages) + item_cost * busy_rows and item_cost >= 1
    load = np.zeros(units, dtype=np.int64)
    for (row, j0, j1, part), u in zip(items.tolist(), unit.tolist()):
        load[u] += (j1 - j0 + 63) // 64 + item_cost
    bound = h["target"] + 2 * (min_split + item_cost)
    assert load.max() <= bound, (load.max(), h["target"])
    return r, load


@pytest.mark.parametrize("name", ["tiny", "uniform", "mtp", "mixed", "long", "long1m"])
@pytest.mark.parametrize("units", [1, 7, 74, 76, 148])
def test_workload_schedules(name, units):
    w = W.workload(name)
    _check_schedule(w.seq_lens, w.s_q, units)


def test_random_schedules():
    rng = np.random.default_rng(3)
    for _ in range(300):
        B = int(rng.integers(1, 70))
        s_q = int(rng.integers(1, 3))
        kind = rng.integers(0, 3)
        if kind == 0:
            lens = rng.integers(s_q, 3000, size=B)
        elif kind == 1:
            lens = np.where(rng.random(B) < 0.4, rng.integers(10000, 40000, size=B),
                            rng.integers(s_q, 600, size=B))
        else:
            lens = rng.integers(s_q, 200, size=B)
        units = int(rng.integers(1, 160))
        _check_schedule(lens, s_q, units)


def test_mixed_is_balanced():
    """The long/short mix that stalled FlashDecoding gets an even schedule."""
    w = W.workload("mixed")
    r, load = _check_schedule(w.seq_lens, 1, 74)
    assert load.max() / load.mean() < 1.15
    # long rows are split, short rows are not
    long_rows = [i for i, L in enumerate(w.seq_lens) if L == 20480]
    assert all(r["row_nparts"][i] >= 2 for i in long_rows)


def test_deterministic():
    w = W.workload("mtp")
    a = m.plan_host(w.seq_lens, s_q=2, max_pages_per_seq=128, num_units=74)
    b = m.plan_host(w.seq_lens, s_q=2, max_pages_per_seq=128, num_units=74)
    for k in a:
        if k != "header":
            np.testing.assert_array_equal(a[k], b[k])
    assert a["header"] == b["header"]


def test_invalid_rows_flagged():
    r = m.plan_host([1, 5, 700], s_q=2, max_pages_per_seq=10, num_units=4)
    assert r["header"]["status"] & m.MLA_DEV_BAD_SEQ_LEN
    assert r["row_nparts"][0] == 0 and r["row_nparts"][1] == 0   # seq_len 1 < s_q
    assert r["row_nparts"][4] == 0                               # 700 > 10 pages
    assert r["row_nparts"][2] >= 1


def test_bad_problem_rejected():
    with pytest.raises(m.MLAError) as e:
        m.plan_host([10], s_q=3, max_pages_per_seq=1, num_units=1)
    assert e.value.status == 2
    with pytest.raises(m.MLAError):
        m.plan_host([10], s_q=1, max_pages_per_seq=0, num_units=1)


def test_cost_line_is_token_major():
    """Every request's token 0, then every request's token 1: the two tokens of a request lie half
    a line apart, and for s_q = 1 the line is row order."""
    w = W.workload("mtp")
    B = w.batch
    r = m.plan_host(w.seq_lens, s_q=2, max_pages_per_seq=128, num_units=76)
    pos = r["row_pos"]
    line = [(k % B) * 2 + k // B for k in range(2 * B)]
    assert np.all(np.diff(pos[line]) > 0)
    # each request's token 1 runs on the unit half the GPU away from its token 0
    items, unit = r["items"], r["item_unit"]
    first_unit = {}
    for (row, _, _, _), u in zip(items.tolist(), unit.tolist()):
        first_unit.setdefault(row, u)
    gaps = [first_unit[2 * b + 1] - first_unit[2 * b] for b in range(B)]
    assert all(36 <= g <= 40 for g in gaps), sorted(set(gaps))
    r1 = m.plan_host(w.seq_lens[:64], s_q=1, max_pages_per_seq=128, num_units=76)
    assert np.all(np.diff(r1["row_pos"]) > 0)
