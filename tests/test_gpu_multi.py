"""Causal multi-query decode (pda_decode_multi) against the oracle."""
import numpy as np
import pytest

import oracle
from gpu_util import assert_close_to_oracle, dev, host_f64, upload
from paged_gqa_decode_05_gb300 import workloads

pytestmark = pytest.mark.gpu


def _ctx(w, q_len):
    import paged_gqa_decode_05_gb300 as pda
    return pda.Context(max_seqs=w.B * q_len, num_q_heads=w.Hq, num_kv_heads=w.Hkv, head_dim=w.D,
                       block_size=w.block_size)


@pytest.mark.parametrize("D,bs,G,q_len", [(128, 16, 4, 4), (64, 32, 8, 2), (256, 8, 2, 7),
                                          (128, 1, 4, 3), (128, 16, 1, 16), (256, 4, 2, 5),
                                          (256, 2, 8, 3), (64, 16, 2, 9), (128, 32, 8, 5)])
def test_multi_matches_oracle(D, bs, G, q_len):
    import torch
    lens = [q_len, 1, q_len + bs, 900, 2 * 64 + 5, 3000]
    w = workloads.make_workload("multi", B=len(lens), Hq=G * 2, Hkv=2, D=D, block_size=bs,
                                seq_lens=lens, seed=D + bs + G + q_len)
    q = workloads.multi_queries(w, q_len)
    ctx = _ctx(w, q_len)
    t = upload(w)
    out = ctx.decode_multi(dev(q), t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    ref = oracle.load().decode_multi(q, w.k_pool, w.v_pool, w.block_table, w.seq_lens,
                                     q_len=q_len, Hq=w.Hq, Hkv=w.Hkv, D=D, block_size=bs,
                                     n_threads=oracle.host_threads())
    assert_close_to_oracle(host_f64(out), ref, f"q_len={q_len}")


def test_single_query_is_decode_bit_for_bit():
    import torch
    w = workloads.make_workload("multi1", B=4, Hq=8, Hkv=2, D=128, block_size=16,
                                seq_lens=[100, 3, 4096, 17], seed=5)
    ctx = _ctx(w, 1)
    t = upload(w)
    a = ctx.decode_multi(t["q"][:, None].contiguous(), t["k_pool"], t["v_pool"], t["block_table"],
                         t["seq_lens"])
    b = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    assert np.array_equal(a[:, 0].float().cpu().numpy(), b.float().cpu().numpy())


def test_eight_b_speculative_verify():
    """The 8B-style cache with 4 verified tokens per sequence."""
    import torch
    w = workloads.eight_b()
    q = workloads.multi_queries(w, 4)
    ctx = _ctx(w, 4)
    t = upload(w)
    out = ctx.decode_multi(dev(q), t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    ref = oracle.load().decode_multi(q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, q_len=4,
                                     Hq=w.Hq, Hkv=w.Hkv, D=w.D, block_size=w.block_size,
                                     n_threads=oracle.host_threads())
    assert_close_to_oracle(host_f64(out), ref, "8b q_len=4")
