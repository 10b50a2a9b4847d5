"""The residency policy (host code of the library, no GPU): the most-used experts
become resident, residents that stay keep their slots, unused experts are never
promoted, and the answer is deterministic."""
import numpy as np
import pytest

import latent_sparse_moe_router_b300 as ext


def _brute(use, n_slots):
    order = sorted(range(len(use)), key=lambda e: (-use[e], e))
    return {e for e in order[:n_slots] if use[e] > 0}


@pytest.mark.parametrize("seed", range(6))
def test_plan_chooses_the_most_used_and_keeps_stayers_in_place(seed):
    rng = np.random.default_rng(seed)
    E, S = 64, 12
    use = rng.integers(0, 50, E).astype(np.uint32)
    use[rng.choice(E, 5, replace=False)] = 0
    cur = np.full(S, -1, np.int32)
    cur[: S // 2] = rng.choice(E, S // 2, replace=False)
    nxt, changed = ext.edge0_tier_plan(use, S, cur)
    want = _brute(use.tolist(), S)
    got = {int(e) for e in nxt if e >= 0}
    assert want <= got                                   # every chosen expert is resident
    assert len(got) == int(np.sum(nxt >= 0))             # no expert twice
    for k in range(S):                                   # a chosen resident keeps its slot
        if cur[k] >= 0 and cur[k] in want:
            assert nxt[k] == cur[k]
    for e in got - want:                                 # extra residents are only leftovers
        assert e in set(cur.tolist())
    assert changed == int(np.sum(nxt != cur))
    again, _ = ext.edge0_tier_plan(use, S, cur)
    assert np.array_equal(nxt, again)


def test_ties_rank_by_lower_index_and_unused_experts_stay_out():
    use = np.array([3, 5, 5, 0, 5, 0], np.uint32)
    nxt, n = ext.edge0_tier_plan(use, 3, np.full(3, -1, np.int32))
    assert sorted(nxt.tolist()) == [1, 2, 4]             # the three 5s beat the 3
    nxt, _ = ext.edge0_tier_plan(np.array([0, 7, 0, 0], np.uint32), 3, np.full(3, -1, np.int32))
    assert sorted(nxt.tolist()) == [-1, -1, 1]           # nothing promoted without a use


def test_bad_arguments_are_rejected():
    with pytest.raises(ext.Edge0Error):
        ext.edge0_tier_plan(np.zeros(4, np.uint32), 5, np.full(5, -1, np.int32))
