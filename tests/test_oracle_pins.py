"""The oracle against its pins (CPU only): every pin of ``oracle_pins`` must hold."""
import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("name", sorted(oracle_pins.PINS))
def test_pin(orc, name):
    oracle_pins.PINS[name](orc)


def test_bf16_widening_exact(orc):
    # 0x3F80 = 1.0, 0xC000 = -2.0, 0x0001 = smallest subnormal 2^-133, 0x7F7F = bf16 max
    assert orc.bf16_to_double(0x3F80) == 1.0
    assert orc.bf16_to_double(0xC000) == -2.0
    assert orc.bf16_to_double(0x0001) == 2.0 ** -133
    assert orc.bf16_to_double(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127


def test_threads_do_not_change_result(orc):
    from paged_gqa_decode_05_gb300.workloads import make_workload
    w = make_workload("t", B=3, Hq=8, Hkv=2, D=16, block_size=4, seq_lens=[5, 33, 17], seed=9)
    args = (w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens)
    kw = dict(Hq=8, Hkv=2, D=16, block_size=4)
    one = orc.decode(*args, **kw, n_threads=1)
    many = orc.decode(*args, **kw, n_threads=5)
    import numpy as np
    assert np.array_equal(one, many)
    pairs = np.array([[2, 7], [0, 0], [1, 3]], dtype=np.int32)
    sub = orc.decode(*args, **kw, pairs=pairs, n_threads=2)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(sub[i], one[b, h])


def test_rejects_bad_table(orc):
    import numpy as np
    from paged_gqa_decode_05_gb300.workloads import make_workload
    w = make_workload("t", B=1, Hq=2, Hkv=1, D=8, block_size=4, seq_lens=[6], seed=3)
    w.block_table[0, 1] = w.num_blocks
    with pytest.raises(ValueError):
        orc.decode(w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hq=2, Hkv=1, D=8,
                   block_size=4)
