"""The split plan (host mirror of the device computation) against a brute-force
enumeration of segments: every block is owned by exactly one CTA, a unit's
first/last CTA are right, and partial-state slots never collide."""
import numpy as np
import pytest

import paged_gqa_decode_05_gb300 as pda
from paged_gqa_decode_05_gb300 import _build


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()


def brute_segments(nb, Hkv, P, cost=0):
    """(unit, cta) pairs where a CTA's range holds some of a unit's blocks, from
    explicit ranges: a unit of n > 0 blocks spans n + cost positions, blocks
    first."""
    units = []
    start = 0
    for b, n in enumerate(nb):
        for g in range(Hkv):
            units.append((start, start + n))
            start += n + cost if n > 0 else 0
    W = start
    ctas = [(c * W // P, (c + 1) * W // P) for c in range(P)]
    segs = {}
    for u, (us, ue) in enumerate(units):
        segs[u] = [c for c, (cs, ce) in enumerate(ctas) if max(us, cs) < min(ue, ce)]
    return segs, W, units, ctas


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("cost", [0, 1, 4, 8])
def test_plan_matches_brute_force(seed, cost):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    bs = int(rng.choice([8, 16, 32, 64]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    lens = rng.integers(0, 3000, size=B)
    lens[rng.random(B) < 0.2] = 0
    P = int(rng.choice([1, 3, 152, 304, 456]))
    first, last, W = pda.plan_units(lens, block_size=bs, num_kv_heads=Hkv, split_ctas=P,
                                    unit_cost=cost)
    nb = [-(-int(x) // bs) for x in lens]
    segs, W_ref, _, _ = brute_segments(nb, Hkv, P, cost)
    assert W == W_ref
    slots = set()
    for u, cs in segs.items():
        if not cs:
            assert first[u] == -1 and last[u] == -1
            continue
        assert first[u] == cs[0] and last[u] == cs[-1]
        assert cs == list(range(cs[0], cs[-1] + 1))  # the owners are consecutive CTAs
        for c in cs:
            slot = u + c
            assert slot not in slots  # one partial state per segment, never shared
            assert slot < len(segs) + P
            slots.add(slot)


def test_unit_cost_evens_segment_load():
    """Count a segment as its blocks plus the unit cost c.  With c in the plan a
    CTA's range of R positions holds its blocks, the cost tails of its
    segments but the last, possibly part of the last one's and of the tail of
    a unit ending in the CTA before; so the CTA's load stays within c of R,
    and the loads of all CTAs within 2c + 1 of each other.  A plan without
    the cost gives the CTAs that cover many short units more load."""
    rng = np.random.default_rng(7)
    Hkv, P, bs, cost = 8, 304, 32, 2
    lens = np.exp(rng.uniform(np.log(128), np.log(32768), size=64)).astype(np.int64)
    nb = [-(-int(x) // bs) for x in lens]

    def loads(c_plan):
        segs, W, units, ctas = brute_segments(nb, Hkv, P, c_plan)
        load = np.zeros(P, dtype=np.int64)
        for u, cs in segs.items():
            us, ue = units[u]
            for c in cs:
                lo, hi = ctas[c]
                load[c] += min(ue, hi) - max(us, lo) + cost
        return load

    plain, costed = loads(0), loads(cost)
    assert costed.max() - costed.min() <= 2 * cost + 1
    assert plain.max() - plain.min() > 2 * cost + 1


def test_block_counts_mode():
    first, last, W = pda.plan_units([3, 0, 5], block_size=16, num_kv_heads=2, split_ctas=4,
                                    blocks_given=True)
    assert W == 16
    assert list(first[2:4]) == [-1, -1]


def test_small_batches_are_planned_by_unit():
    """No more units than CTAs and every unit at most 4 stages of rows: CTA u
    processes unit u whole (no unit is split, so nothing merges); a unit one
    block longer than that, or more units than CTAs, takes the even split."""
    st, bs, Hkv = 64, 16, 2
    lens = [37, 0, 4 * st, 1]
    first, last, _ = pda.plan_units(lens, block_size=bs, num_kv_heads=Hkv, split_ctas=304,
                                    unit_cost=8, stage_tokens=st)
    for u in range(len(lens) * Hkv):
        if lens[u // Hkv] == 0:
            assert first[u] == last[u] == -1
        else:
            assert first[u] == last[u] == u
    # one block longer than four stages: the even split, units spread over CTAs
    first, last, _ = pda.plan_units([37, 4 * st + bs], block_size=bs, num_kv_heads=Hkv,
                                    split_ctas=304, unit_cost=8, stage_tokens=st)
    assert last[2] > first[2]
    # more units than CTAs: the even split
    first, last, W = pda.plan_units([5] * 4, block_size=bs, num_kv_heads=Hkv, split_ctas=7,
                                    unit_cost=8, stage_tokens=st)
    ref, ref_last, ref_W = pda.plan_units([5] * 4, block_size=bs, num_kv_heads=Hkv, split_ctas=7,
                                          unit_cost=8)
    assert W == ref_W and list(first) == list(ref) and list(last) == list(ref_last)
