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


@pytest.mark.parametrize("D,bs,G,q_len", [
    # n8 form (q_len * G <= 8, or head size 256)
    (128, 16, 4, 2), (64, 16, 2, 3), (256, 8, 2, 7), (256, 4, 2, 5), (256, 2, 8, 3),
    # row form, one q tile (9..16 q rows per walk)
    (128, 16, 4, 4), (64, 32, 8, 2), (128, 1, 4, 3), (128, 16, 1, 16), (64, 1, 4, 4),
    # row form, two q tiles (17..32 q rows per walk), several walks per sequence
    (64, 16, 2, 9), (128, 32, 8, 5), (128, 16, 4, 8), (64, 16, 8, 4), (128, 4, 4, 8),
    (64, 2, 2, 9), (128, 8, 3, 7), (128, 16, 8, 8), (128, 2, 1, 33)])
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


@pytest.mark.parametrize("D,G,q_len,form,qp,walks", [
    (128, 4, 2, 0, 2, 1), (128, 4, 3, 1, 3, 1), (128, 4, 4, 1, 4, 1), (128, 4, 8, 1, 8, 1),
    (128, 4, 9, 1, 8, 2), (128, 8, 2, 1, 2, 1), (128, 8, 5, 1, 4, 2), (64, 1, 8, 0, 8, 1),
    (64, 1, 9, 1, 9, 1), (64, 2, 16, 1, 16, 1), (256, 4, 4, 0, 2, 2), (256, 8, 3, 0, 1, 3)])
def test_multi_launch_shape(D, G, q_len, form, qp, walks):
    """The form a q_len takes: up to 8 q rows per sequence (and every head size
    256 call) the n8 form; more, the row form with up to 32 q rows per walk,
    one q tile (two CTAs per SM) up to 16 rows and two (one CTA per SM) above."""
    import paged_gqa_decode_05_gb300 as pda
    ctx = pda.Context(max_seqs=64, num_q_heads=2 * G, num_kv_heads=2, head_dim=D, block_size=16)
    info = ctx.multi_info(q_len)
    launch = ctx.launch_info()
    assert (info["form"], info["queries_per_walk"], info["walks_per_seq"]) == (form, qp, walks)
    assert info["rows_per_walk"] == qp * G
    if form == 0:
        assert info["split_ctas"] == launch["split_ctas"]
    else:
        per_sm = 2 if qp * G <= 16 else 1
        assert info["split_ctas"] == per_sm * launch["num_sms"]
    ctx.close()


@pytest.mark.parametrize("q_len", [2, 4, 8])
def test_multi_garbage_outside_valid_rows_ignored(q_len):
    """NaN bits in unused blocks, unused table entries and the slots past each
    sequence's length leave every form's output unchanged, bit for bit."""
    import torch
    lens = [37, 80, 1, 130, 2000]
    w = workloads.make_workload("multi_nan", B=len(lens), Hq=8, Hkv=2, D=128, block_size=16,
                                seq_lens=lens, seed=61, pool_blocks=200, max_blocks=140)
    q = workloads.multi_queries(w, q_len)
    ctx = _ctx(w, q_len)

    def run():
        t = upload(w)
        o = ctx.decode_multi(dev(q), t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
        torch.cuda.synchronize()
        return o.float().cpu().numpy()
    base = run()
    nan = np.uint16(0x7FC1)
    used = set()
    for b in range(w.B):
        n = int(w.seq_lens[b]); nb = -(-n // w.block_size)
        used.update(int(x) for x in w.block_table[b, :nb])
        last = w.block_table[b, nb - 1]
        w.k_pool[last, n - (nb - 1) * w.block_size:] = nan
        w.v_pool[last, n - (nb - 1) * w.block_size:] = nan
    unused = [i for i in range(w.num_blocks) if i not in used]
    w.k_pool[unused] = nan
    w.v_pool[unused] = nan
    for b in range(w.B):
        nb = -(-int(w.seq_lens[b]) // w.block_size)
        w.block_table[b, nb:] = unused[b % len(unused)]
    got = run()
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, base)
    assert ctx.read_device_errors() == 0


@pytest.mark.parametrize("q_len", [4, 8])
def test_multi_later_tokens_do_not_reach_earlier_queries(q_len):
    """Causality: new K/V values at a sequence's last token change only its
    last query's output; the earlier queries' outputs stay bit-identical."""
    import torch
    lens = [300, 4096, 77]
    w = workloads.make_workload("multi_causal", B=len(lens), Hq=16, Hkv=4, D=128, block_size=16,
                                seq_lens=lens, seed=62)
    q = workloads.multi_queries(w, q_len)
    ctx = _ctx(w, q_len)

    def run():
        t = upload(w)
        o = ctx.decode_multi(dev(q), t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
        torch.cuda.synchronize()
        return o.float().cpu().numpy()
    base = run()
    rng = np.random.default_rng(7)
    for b in range(w.B):
        n = int(w.seq_lens[b])
        blk, slot = w.block_table[b, (n - 1) // w.block_size], (n - 1) % w.block_size
        for pool in (w.k_pool, w.v_pool):
            vals = rng.standard_normal(pool[blk, slot].shape).astype(np.float32) * 3
            pool[blk, slot] = (vals.view(np.uint32) >> 16).astype(np.uint16)
    got = run()
    assert np.array_equal(got[:, :q_len - 1], base[:, :q_len - 1])
    assert not np.array_equal(got[:, q_len - 1], base[:, q_len - 1])
    assert ctx.read_device_errors() == 0


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


@pytest.mark.parametrize("q_len", [4, 8])
def test_eight_b_speculative_verify(q_len):
    """The 8B-style cache with 4 or 8 verified tokens per sequence (16 or 32 q
    rows per kv head: the row form with one or two q tiles)."""
    import torch
    w = workloads.eight_b()
    q = workloads.multi_queries(w, q_len)
    ctx = _ctx(w, q_len)
    t = upload(w)
    out = ctx.decode_multi(dev(q), t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    ref = oracle.load().decode_multi(q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, q_len=q_len,
                                     Hq=w.Hq, Hkv=w.Hkv, D=w.D, block_size=w.block_size,
                                     n_threads=oracle.host_threads())
    assert_close_to_oracle(host_f64(out), ref, f"8b q_len={q_len}")
