"""Large block pools: block ids spread over a pool of millions of blocks, so the
loaders' id arithmetic (TMA box coordinates; gather4 row indices = id times
the block's row stride) runs far from small values."""
import time

import numpy as np
import pytest

import oracle
from gpu_util import assert_close_to_oracle, context_for, host_f64, upload
from paged_gqa_decode_05_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs,pool,D,Hkv", [(1, 1_500_000, 64, 2), (16, 400_000, 64, 1)])
def test_block_ids_across_a_large_pool(bs, pool, D, Hkv):
    import torch
    t0 = time.time()
    lens = [3001, 1, 2 * bs + 3, 2500]
    w = workloads.make_workload("pool", B=len(lens), Hq=4 * Hkv, Hkv=Hkv, D=D, block_size=bs,
                                seq_lens=lens, seed=77 + bs, pool_blocks=pool)
    used = np.concatenate([w.block_table[b, :-(-n // bs)] for b, n in enumerate(lens)])
    assert used.max() > 0.9 * pool  # the table reaches the top of the pool
    ctx = context_for(w)
    t = upload(w)
    got = host_f64(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"]))
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    ref = oracle.load().decode(w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hq=w.Hq,
                               Hkv=w.Hkv, D=w.D, block_size=w.block_size)
    assert_close_to_oracle(got, ref, f"pool of {pool} blocks, block size {bs}")
    assert time.time() - t0 < 300
