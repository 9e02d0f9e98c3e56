"""Pins of the oracle's routing plan: brute-force enumeration on tiny inputs and
invariants on larger ones."""
import numpy as np
import pytest

import moe_inputs as mi
from oracle import plan as P


def _brute(ids, off, El):
    M, k = ids.shape
    slots = [(int(ids[t, j]) - off, t * k + j) for t in range(M) for j in range(k)
             if 0 <= int(ids[t, j]) - off < El]
    slots.sort()          # by (local expert, slot index)
    counts = [sum(1 for l, _ in slots if l == e) for e in range(El)]
    padded = [0]
    for c in counts:
        padded.append(padded[-1] + (c + 127) // 128 * 128)
    rows = {}
    for e in range(El):
        mine = [s for l, s in slots if l == e]
        for i, s in enumerate(mine):
            rows[s] = padded[e] + i
    return counts, padded, rows


@pytest.mark.parametrize("seed", range(20))
def test_plan_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    M = int(rng.integers(1, 9))
    E = int(rng.integers(2, 12))
    k = int(rng.integers(1, E + 1))
    off = int(rng.integers(0, 3))
    El = int(rng.integers(1, E + 1))
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    ids[rng.random(ids.shape) < 0.15] = -1
    p = P.make_plan(ids, off, El)
    counts, padded, rows = _brute(ids, off, El)
    assert p["counts"].tolist() == counts
    assert p["padded_offsets"].tolist() == padded
    t2r = p["token_to_row"].ravel()
    for s in range(M * k):
        assert t2r[s] == rows.get(s, -1)
    r2s = p["row_to_slot"]
    for s, r in rows.items():
        assert r2s[r] == s
    assert (r2s >= 0).sum() == len(rows)
    assert p["capacity"] >= padded[-1]


def test_plan_invariants_prefill_skewed():
    cfg = mi.CONFIGS["prefill_skewed"]
    ids, _ = mi.routing(cfg)
    p = P.make_plan(ids, 0, cfg.E)
    counts, padded = p["counts"], p["padded_offsets"]
    assert counts.sum() == ids.size
    assert np.all(np.diff(padded) % 128 == 0)
    assert np.all(np.diff(padded) >= counts)
    assert np.all(np.diff(padded) < counts + 128)
    r2s, t2r = p["row_to_slot"], p["token_to_row"].ravel()
    real = r2s >= 0
    # row_to_slot o token_to_row is the identity on routed slots, and back
    assert np.array_equal(t2r[r2s[real]], np.nonzero(real)[0])
    assert np.array_equal(r2s[t2r], np.arange(ids.size))
    # inside a segment rows are in ascending token order
    k = cfg.top_k
    for l in range(cfg.E):
        seg = r2s[padded[l]:padded[l] + counts[l]]
        assert np.all(seg // k == np.sort(seg // k))
        assert np.all(ids.ravel()[seg] == l)
        assert np.all(r2s[padded[l] + counts[l]:padded[l + 1]] == -1)
    assert np.all(r2s[padded[-1]:] == -1)


def test_masking_ep_and_unrouted():
    cfg = mi.CONFIGS["relu2_ep"].with_(M=512)
    ids, _ = mi.routing(cfg)
    ids = mi.with_unrouted(ids, 0.1, 9, cfg.E)
    p = P.make_plan(ids, cfg.local_offset, cfg.El)
    t2r = p["token_to_row"]
    masked = (ids < 0) | (ids >= cfg.El)
    assert np.all((t2r == -1) == masked)
    assert p["counts"].sum() == (~masked).sum()


def test_offset_shifts_experts():
    ids = np.array([[5, 6], [6, 2]], dtype=np.int32)
    p = P.make_plan(ids, 5, 2)
    assert p["counts"].tolist() == [1, 2]
    assert p["token_to_row"].tolist() == [[0, 128], [129, -1]]


def test_empty_and_all_masked():
    ids = np.full((3, 2), -1, dtype=np.int32)
    p = P.make_plan(ids, 0, 4)
    assert p["num_rows"] == 0 and np.all(p["row_to_slot"] == -1)
    p0 = P.make_plan(np.zeros((0, 2), np.int32), 0, 4)
    assert p0["num_rows"] == 0 and p0["capacity"] == 0


def test_duplicates_rejected():
    ids = np.array([[1, 1]], dtype=np.int32)
    with pytest.raises(ValueError):
        P.make_plan(ids, 0, 4)
    p = P.make_plan(ids, 0, 4, allow_duplicates=True)
    assert p["duplicate"] and p["token_to_row"].tolist() == [[0, 1]]


def test_capacity_bound_is_tight():
    # every expert gets one row: E segments of 128 rows
    M, k, El = 64, 4, 256
    ids = np.arange(M * k, dtype=np.int32).reshape(M, k)
    p = P.make_plan(ids, 0, El)
    assert p["num_rows"] == 256 * 128 == P.plan_capacity(M, k, El)
