"""Batches that stress the split plan's unit cost: most plan positions are the
cost placeholders of short units, so many CTA ranges start or end inside one,
or hold no block at all.  Every path against the oracle."""
import numpy as np
import pytest

import oracle
from gpu_util import TILED_VS_ONESHOT, assert_close_to_oracle, context_for, dev, host_f64, upload
from paged_gqa_decode_05_gb300 import workloads

pytestmark = pytest.mark.gpu


def _short_batch(B, D, bs, G, Hkv, seed, long_every=0):
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(0, 3 * bs, size=B)]
    if long_every:
        for b in range(0, B, long_every):
            lens[b] = int(rng.integers(1000, 4000))
    return workloads.make_workload(f"short{seed}", B=B, Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs,
                                   seq_lens=lens, seed=seed)


CASES = [  # B, D, bs, G, Hkv, long_every
    (600, 128, 16, 4, 2, 0),
    (300, 64, 32, 8, 1, 37),
    (200, 256, 16, 2, 2, 0),
    (250, 128, 4, 4, 2, 50),   # row-gather loader
]


@pytest.mark.parametrize("case", CASES)
def test_short_units_one_shot(case):
    import torch
    B, D, bs, G, Hkv, long_every = case
    w = _short_batch(B, D, bs, G, Hkv, seed=B + D + bs, long_every=long_every)
    ctx = context_for(w)
    assert ctx.launch_info()["unit_cost"] >= 1
    t = upload(w)
    got = host_f64(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"]))
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    ref = oracle.load().decode(w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hq=w.Hq,
                               Hkv=w.Hkv, D=w.D, block_size=w.block_size,
                               n_threads=oracle.host_threads())
    assert_close_to_oracle(got, ref, f"B={B} D={D} bs={bs}")
    for b in range(w.B):
        if w.seq_lens[b] == 0:
            assert np.all(got[b] == 0.0)


@pytest.mark.parametrize("case", CASES[:2])
def test_short_units_tiled(case):
    """Folded in tiles of at most 3 blocks: the plan counts the unit cost on
    block counts too; equal to one-shot within the fp32 bar."""
    import torch
    from test_gpu_tiled import make_tiles
    B, D, bs, G, Hkv, long_every = case
    w = _short_batch(B, D, bs, G, Hkv, seed=B + D + bs, long_every=long_every)
    ctx = context_for(w, tile_capacity=3)
    t = upload(w)
    ctx.begin_step(w.B)
    for blocks, counts, last in make_tiles(w, 3, np.random.default_rng(3)):
        ctx.step_tile(t["q"], t["k_pool"], t["v_pool"], dev(blocks), dev(counts), dev(last))
    f32 = host_f64(ctx.finalize(w.B, out_dtype=torch.float32))
    one = host_f64(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                              out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    assert np.max(np.abs(f32 - one)) <= TILED_VS_ONESHOT


@pytest.mark.parametrize("case,q_len", [(CASES[0], 3), (CASES[1], 2)])
def test_short_units_multi(case, q_len):
    import torch
    B, D, bs, G, Hkv, long_every = case
    w = _short_batch(B // q_len, D, bs, G, Hkv, seed=B + D + bs, long_every=long_every)
    qm = workloads.multi_queries(w, q_len)
    ctx = context_for(w, max_seqs=w.B * q_len)
    t = upload(w)
    got = host_f64(ctx.decode_multi(dev(qm), t["k_pool"], t["v_pool"], t["block_table"],
                                    t["seq_lens"]))
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    ref = oracle.load().decode_multi(qm, w.k_pool, w.v_pool, w.block_table, w.seq_lens,
                                     q_len=q_len, Hq=w.Hq, Hkv=w.Hkv, D=w.D,
                                     block_size=w.block_size, n_threads=oracle.host_threads())
    assert_close_to_oracle(got, ref, f"q_len={q_len}")
