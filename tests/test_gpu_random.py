"""Seeded random shapes through every decode path, each against the oracle:
head size, block size, group size, batch, ragged lengths (including 0, 1 and
block boundaries), pool size and scale are drawn per case."""
import numpy as np
import pytest

import oracle
from gpu_util import TILED_VS_ONESHOT, assert_close_to_oracle, context_for, dev, host_f64, upload
from paged_gqa_decode_05_gb300 import workloads

pytestmark = pytest.mark.gpu

N_CASES = 40


def draw_case(i):
    rng = np.random.default_rng(20_000 + i)
    D = int(rng.choice([64, 128, 256]))
    bs = int(rng.choice([1, 2, 4, 8, 16, 32, 64]))
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 3])) if G < 8 else 1
    B = int(rng.integers(1, 9))
    special = [0, 1, bs - 1, bs, bs + 1, 64, 65, 2 * bs]
    lens = [int(rng.choice(special)) if rng.random() < 0.4 else int(rng.integers(0, 1500))
            for _ in range(B)]
    lens = [max(0, x) for x in lens]
    pool_extra = int(rng.integers(0, 40))
    needed = sum(-(-x // bs) for x in lens)
    scale = None if rng.random() < 0.6 else float(rng.uniform(-0.3, 0.3))
    w = workloads.make_workload(f"rand{i}", B=B, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs,
                                seq_lens=lens, seed=30_000 + i,
                                pool_blocks=max(1, needed + pool_extra))
    return w, scale, rng


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_one_shot(orc, i):
    import torch
    w, scale, _ = draw_case(i)
    ctx = context_for(w)
    t = upload(w)
    got = host_f64(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                              scale=scale))
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    ref = orc.decode(w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hq=w.Hq, Hkv=w.Hkv,
                     D=w.D, block_size=w.block_size, scale=scale)
    assert_close_to_oracle(got, ref, f"case {i}")
    for b in range(w.B):
        if w.seq_lens[b] == 0:
            assert np.all(got[b] == 0.0)


@pytest.mark.parametrize("i", range(0, N_CASES, 4))
def test_random_tiled(orc, i):
    """The same case folded in random tiles: equal to one-shot within 1e-3 (fp32)."""
    import torch
    from test_gpu_tiled import make_tiles
    w, scale, rng = draw_case(i)
    cap = int(rng.integers(1, 40))
    ctx = context_for(w, tile_capacity=cap)
    t = upload(w)
    ctx.begin_step(w.B)
    for blocks, counts, last in make_tiles(w, cap, rng):
        ctx.step_tile(t["q"], t["k_pool"], t["v_pool"], dev(blocks), dev(counts), dev(last),
                      scale=scale)
    f32 = host_f64(ctx.finalize(w.B, out_dtype=torch.float32))
    one = host_f64(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                              scale=scale, out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    assert np.max(np.abs(f32 - one)) <= TILED_VS_ONESHOT


@pytest.mark.parametrize("i", range(1, N_CASES, 4))
def test_random_multi(orc, i):
    import torch
    w, scale, rng = draw_case(i)
    q_len = int(rng.integers(2, 10))
    qm = workloads.multi_queries(w, q_len)
    ctx = context_for(w, max_seqs=w.B * q_len)
    t = upload(w)
    got = host_f64(ctx.decode_multi(dev(qm), t["k_pool"], t["v_pool"], t["block_table"],
                                    t["seq_lens"], scale=scale))
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    ref = orc.decode_multi(qm, w.k_pool, w.v_pool, w.block_table, w.seq_lens, q_len=q_len,
                           Hq=w.Hq, Hkv=w.Hkv, D=w.D, block_size=w.block_size, scale=scale)
    assert_close_to_oracle(got, ref, f"multi case {i}, q_len {q_len}")
