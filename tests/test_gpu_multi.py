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


TWO_TILE_CASES = [(64, 16, 2, 9), (128, 32, 8, 5), (128, 16, 4, 8), (64, 16, 8, 4), (128, 4, 4, 8),
                  (64, 2, 2, 9), (128, 8, 3, 7), (128, 16, 8, 8), (128, 2, 1, 33), (64, 8, 4, 6),
                  (128, 64, 2, 11), (128, 1, 8, 4)]


@pytest.mark.parametrize("D,bs,G,q_len,tc", [
    # n8 form (q_len * G <= 8, or head size 256)
    (128, 16, 4, 2, True), (64, 16, 2, 3, True), (256, 8, 2, 7, True), (256, 4, 2, 5, True),
    (256, 2, 8, 3, True),
    # row form, one q tile (9..16 q rows per walk)
    (128, 16, 4, 4, True), (64, 32, 8, 2, True), (128, 1, 4, 3, True), (128, 16, 1, 16, True),
    (64, 1, 4, 4, True)] +
    # 17..32 q rows per walk, several walks per sequence: the tcgen05 row form
    # (where the block layout allows it) and the mma.sync row form with two q tiles
    [c + (tc,) for c in TWO_TILE_CASES for tc in (True, False)])
def test_multi_matches_oracle(D, bs, G, q_len, tc):
    import torch
    lens = [q_len, 1, q_len + bs, 900, 2 * 64 + 5, 3000]
    w = workloads.make_workload("multi", B=len(lens), Hq=G * 2, Hkv=2, D=D, block_size=bs,
                                seq_lens=lens, seed=D + bs + G + q_len)
    q = workloads.multi_queries(w, q_len)
    ctx = _ctx(w, q_len)
    ctx.set_multi_tc(tc)
    t = upload(w)
    out = ctx.decode_multi(dev(q), t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    ref = oracle.load().decode_multi(q, w.k_pool, w.v_pool, w.block_table, w.seq_lens,
                                     q_len=q_len, Hq=w.Hq, Hkv=w.Hkv, D=D, block_size=bs,
                                     n_threads=oracle.host_threads())
    assert_close_to_oracle(host_f64(out), ref, f"q_len={q_len}")
    info = ctx.multi_info(q_len)
    rows = info["rows_per_walk"]
    tc_layout = bs >= 8 or (bs * D * 2) % 1024 != 0  # whole 1024-byte boxes, or gathered rows
    tc_form = tc and rows > 16 and D == 128 and tc_layout
    assert info["form"] == (2 if tc_form else 1 if rows > 8 and D <= 128 else 0)


@pytest.mark.parametrize("D,G,q_len,form,qp,walks,tc", [
    (128, 4, 2, 0, 2, 1, True), (128, 4, 3, 1, 3, 1, True), (128, 4, 4, 1, 4, 1, True),
    (128, 4, 8, 2, 8, 1, True), (128, 4, 8, 1, 8, 1, False), (128, 4, 9, 2, 8, 2, True),
    (128, 8, 2, 1, 2, 1, True), (128, 8, 5, 2, 4, 2, True), (128, 8, 5, 1, 4, 2, False),
    (64, 1, 8, 0, 8, 1, True), (64, 1, 9, 1, 9, 1, True), (64, 2, 16, 1, 16, 1, True),
    (64, 2, 16, 1, 16, 1, False), (256, 4, 4, 0, 2, 2, True), (256, 8, 3, 0, 1, 3, True)])
def test_multi_launch_shape(D, G, q_len, form, qp, walks, tc):
    """The form a q_len takes: up to 8 q rows per sequence (and every head size
    256 call) the n8 form; more, the row form with up to 32 q rows per walk:
    one q tile on mma.sync (two CTAs per SM) up to 16 rows, and above that two
    q tiles on mma.sync, or at head size 128 the tcgen05 form where it is
    switched on (one CTA per SM either way)."""
    import paged_gqa_decode_05_gb300 as pda
    ctx = pda.Context(max_seqs=64, num_q_heads=2 * G, num_kv_heads=2, head_dim=D, block_size=16)
    ctx.set_multi_tc(tc)
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


@pytest.mark.parametrize("q_len,tc", [(2, True), (4, True), (8, True), (8, False)])
def test_multi_garbage_outside_valid_rows_ignored(q_len, tc):
    """NaN bits in unused blocks, unused table entries and the slots past each
    sequence's length leave every form's output unchanged, bit for bit."""
    import torch
    lens = [37, 80, 1, 130, 2000]
    w = workloads.make_workload("multi_nan", B=len(lens), Hq=8, Hkv=2, D=128, block_size=16,
                                seq_lens=lens, seed=61, pool_blocks=200, max_blocks=140)
    q = workloads.multi_queries(w, q_len)
    ctx = _ctx(w, q_len)
    ctx.set_multi_tc(tc)

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


@pytest.mark.parametrize("q_len,tc", [(4, True), (8, True), (8, False)])
def test_multi_later_tokens_do_not_reach_earlier_queries(q_len, tc):
    """Causality: new K/V values at a sequence's last token change only its
    last query's output; the earlier queries' outputs stay bit-identical."""
    import torch
    lens = [300, 4096, 77]
    w = workloads.make_workload("multi_causal", B=len(lens), Hq=16, Hkv=4, D=128, block_size=16,
                                seq_lens=lens, seed=62)
    q = workloads.multi_queries(w, q_len)
    ctx = _ctx(w, q_len)
    ctx.set_multi_tc(tc)

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
    rows per kv head: the mma.sync row form with one or two q tiles; at 32 rows
    also the tcgen05 form, which agrees with it to fp32 rounding)."""
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
    ctx.set_multi_tc(True)
    if ctx.multi_info(q_len)["form"] == 2:
        out2 = ctx.decode_multi(dev(q), t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
        torch.cuda.synchronize()
        assert ctx.read_device_errors() == 0
        assert_close_to_oracle(host_f64(out2), ref, f"8b q_len={q_len} tcgen05")
        # the two forms differ only in fp32 summation order (and then the bf16 rounding of o)
        a, b = out.float(), out2.float()
        assert float((a - b).abs().max()) <= 2 ** -6 * max(1.0, float(b.abs().max()))


def test_tc_form_back_to_back_with_plain_decodes_in_a_graph():
    """The tcgen05 form holds all 512 tensor-memory columns of an SM per CTA.
    Replayed from one graph, tcgen05 multi-query calls interleaved with plain
    decodes (each launch overlapping the previous one's tail) give, every
    call, the output of the same call run alone, bit for bit."""
    import torch
    q_len = 8
    ws = [workloads.make_workload("tc_b2b", B=8, Hq=32, Hkv=8, D=128, block_size=16,
                                  seq_lens=lens, seed=70 + k, pool_blocks=1100)
          for k, lens in enumerate([[4096, 17, 2000, 9, 3000, 512, 8, 4096],
                                    [2048] * 8])]
    qs = [dev(workloads.multi_queries(w, q_len)) for w in ws]
    ctx = _ctx(ws[0], q_len)
    ctx.set_multi_tc(True)
    assert ctx.multi_info(q_len)["form"] == 2
    ts = [upload(w) for w in ws]

    def calls(outs_m, outs_d):
        for t, q, om, od in zip(ts, qs, outs_m, outs_d):
            ctx.decode_multi(q, t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], out=om)
            ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], out=od)
    alone_m, alone_d = [], []
    for t, q in zip(ts, qs):
        alone_m.append(ctx.decode_multi(q, t["k_pool"], t["v_pool"], t["block_table"],
                                        t["seq_lens"]).clone())
        torch.cuda.synchronize()
        alone_d.append(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                  t["seq_lens"]).clone())
        torch.cuda.synchronize()
    outs_m = [torch.empty_like(a) for a in alone_m]
    outs_d = [torch.empty_like(a) for a in alone_d]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        calls(outs_m, outs_d)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            calls(outs_m, outs_d)
    for o in outs_m + outs_d:
        o.zero_()
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    for o, a in zip(outs_m + outs_d, alone_m + alone_d):
        assert torch.equal(o, a)


@pytest.mark.parametrize("tc", [True, False])
def test_multi_more_launch_rows_than_one_launch(tc):
    """640 sequences of 8 queries: the tcgen05 form launches at most 512 launch
    rows (two chunks here), the mma.sync form 1024 (one); both against the
    oracle."""
    import torch
    rng = np.random.default_rng(71)
    lens = [int(x) for x in rng.integers(8, 200, size=640)]
    q_len = 8
    w = workloads.make_workload("multi_chunks", B=len(lens), Hq=8, Hkv=2, D=128, block_size=16,
                                seq_lens=lens, seed=72)
    q = workloads.multi_queries(w, q_len)
    ctx = _ctx(w, q_len)
    ctx.set_multi_tc(tc)
    assert ctx.multi_info(q_len)["form"] == (2 if tc else 1)
    t = upload(w)
    out = ctx.decode_multi(dev(q), t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    ref = oracle.load().decode_multi(q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, q_len=q_len,
                                     Hq=w.Hq, Hkv=w.Hkv, D=w.D, block_size=w.block_size,
                                     n_threads=oracle.host_threads())
    assert_close_to_oracle(host_f64(out), ref, "multi chunks")
