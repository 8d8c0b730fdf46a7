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


def brute_segments(nb, Hkv, P):
    """(unit, cta) pairs whose ranges intersect, from explicit ranges."""
    units = []
    start = 0
    for b, n in enumerate(nb):
        for g in range(Hkv):
            units.append((start, start + n))
            start += n
    W = start
    ctas = [(c * W // P, (c + 1) * W // P) for c in range(P)]
    segs = {}
    for u, (us, ue) in enumerate(units):
        segs[u] = [c for c, (cs, ce) in enumerate(ctas) if max(us, cs) < min(ue, ce)]
    return segs, W


@pytest.mark.parametrize("seed", range(12))
def test_plan_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 40))
    bs = int(rng.choice([8, 16, 32, 64]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    lens = rng.integers(0, 3000, size=B)
    lens[rng.random(B) < 0.2] = 0
    P = int(rng.choice([1, 3, 152, 304, 456]))
    first, last, W = pda.plan_units(lens, block_size=bs, num_kv_heads=Hkv, split_ctas=P)
    nb = [-(-int(x) // bs) for x in lens]
    segs, W_ref = brute_segments(nb, Hkv, P)
    assert W == W_ref
    slots = set()
    for u, cs in segs.items():
        if not cs:
            assert first[u] == -1 and last[u] == -1
            continue
        assert first[u] == cs[0] and last[u] == cs[-1]
        for c in cs:
            slot = u + c
            assert slot not in slots  # one partial state per segment, never shared
            assert slot < len(segs) + P
            slots.add(slot)


def test_block_counts_mode():
    first, last, W = pda.plan_units([3, 0, 5], block_size=16, num_kv_heads=2, split_ctas=4,
                                    blocks_given=True)
    assert W == 16
    assert list(first[2:4]) == [-1, -1]
