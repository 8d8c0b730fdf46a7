"""Runtime properties on the GPU: CUDA-graph capture of a decode, the bounded
waits' failure path, and streams."""
import numpy as np
import pytest

from gpu_util import context_for, upload
from paged_gqa_decode_05_gb300 import workloads

pytestmark = pytest.mark.gpu


def _w():
    return workloads.make_workload("rt", B=6, Hq=16, Hkv=4, D=128, block_size=16,
                                   seq_lens=[1000, 5, 0, 333, 4096, 77], seed=21)


def test_decode_captured_in_cuda_graph():
    import torch
    w = _w()
    ctx = context_for(w)
    t = upload(w)
    eager = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"]).clone()
    out = torch.zeros_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up on the capture stream
        ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], out=out)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(out.float().cpu().numpy(), eager.float().cpu().numpy())
    # replay reads the current contents of the captured buffers
    t["q"].mul_(-1)
    g.replay()
    flipped = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    assert np.array_equal(out.float().cpu().numpy(), flipped.float().cpu().numpy())


def test_bounded_wait_reports_timeout_and_context_stays_usable():
    import torch
    import paged_gqa_decode_05_gb300 as pda
    w = _w()
    ctx = context_for(w)
    assert ctx.read_device_errors() == 0
    flags = ctx.check_wait_timeout(limit_ns=20_000_000)  # a wait nothing completes, 20 ms
    assert flags & pda.DEVERR_TIMEOUT
    assert ctx.read_device_errors() == 0  # cleared by the previous read
    t = upload(w)
    out = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    assert torch.isfinite(out.float()).all()


def test_two_contexts_on_two_streams():
    import torch
    w = _w()
    t = upload(w)
    a_ctx, b_ctx = context_for(w), context_for(w)
    ref = a_ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"]).clone()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    outs = []
    for ctx, s in ((a_ctx, sa), (b_ctx, sb)):
        with torch.cuda.stream(s):
            outs.append(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                   t["seq_lens"]))
    torch.cuda.synchronize()
    for o in outs:
        assert np.array_equal(o.float().cpu().numpy(), ref.float().cpu().numpy())


@pytest.mark.parametrize("D,bs,rows,per_sm", [(128, 16, 64, 2), (64, 16, 64, 2), (256, 16, 64, 1),
                                              (256, 64, 64, 1), (256, 4, 64, 1), (256, 2, 64, 1),
                                              (256, 1, 32, 2), (128, 4, 64, 2), (128, 1, 64, 2)])
def test_split_kernel_shape(D, bs, rows, per_sm):
    """Stage rows and CTAs per SM as designed: two CTAs per SM at head size
    <= 128; at 256 one, or two with 32-row stages where rows are gathered one
    by one (block size 1: blocks of 2 and 4 rows load as one box each)."""
    import paged_gqa_decode_05_gb300 as pda
    ctx = pda.Context(max_seqs=32, num_q_heads=32, num_kv_heads=8, head_dim=D, block_size=bs)
    info = ctx.launch_info()
    assert info["stage_tokens"] == rows
    assert info["ctas_per_sm"] == per_sm
    assert info["split_ctas"] == per_sm * info["num_sms"]
    ctx.close()


def test_bound_decode_matches_decode_and_tracks_contents():
    """A decode bound once reruns on the same buffers: it follows their current
    contents, matches decode bit for bit, and refuses to run after close."""
    import torch
    import paged_gqa_decode_05_gb300 as pda
    w = _w()
    ctx = context_for(w)
    t = upload(w)
    out = torch.empty((w.B, w.Hq, w.D), device="cuda", dtype=torch.bfloat16)
    run = ctx.bind_decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], out)
    run()
    ref = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    t["q"].mul_(-1.0)  # new contents, same buffer
    run()
    ref2 = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    assert torch.equal(out, ref2) and not torch.equal(ref, ref2)
    ctx.close()
    with pytest.raises(pda.PdaError):
        run()


def test_back_to_back_decodes_with_changing_tables_in_a_graph():
    """Consecutive decodes replayed from one graph overlap their starts (the
    next call's prefetch warp reads lengths and block ids before the previous
    call ends); with a different table, lengths and q in every call, each
    output still equals its own decode run alone."""
    import torch
    ws = [workloads.make_workload("b2b", B=8, Hq=32, Hkv=8, D=128, block_size=16,
                                  seq_lens=lens, seed=40 + k, pool_blocks=1100)
          for k, lens in enumerate([[4096, 17, 2000, 1, 3000, 512, 0, 4096],
                                    [1, 4096, 33, 2500, 64, 4096, 1500, 7],
                                    [2048] * 8])]
    ctx = context_for(ws[0])
    ts = [upload(w) for w in ws]
    alone = []
    for t in ts:
        alone.append(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                t["seq_lens"]).clone())
        torch.cuda.synchronize()
    outs = [torch.empty_like(a) for a in alone]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for t, o in zip(ts, outs):
            ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], out=o)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            for t, o in zip(ts, outs):
                ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], out=o)
    for o in outs:
        o.zero_()
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    for o, a in zip(outs, alone):
        assert torch.equal(o, a)
