"""The tiled lifecycle (begin_step / step_tile / finalize) against the one-shot
path (fp32, before rounding, within 1e-3) and against the oracle."""
import numpy as np
import pytest

import oracle
from gpu_util import TILED_VS_ONESHOT, assert_close_to_oracle, context_for, dev, host_f64, upload
from paged_gqa_decode_05_gb300 import workloads

pytestmark = pytest.mark.gpu


def make_tiles(w, tile_capacity, rng):
    """Splits every sequence's block list into random consecutive tiles."""
    nb = -(-w.seq_lens.astype(np.int64) // w.block_size)
    cuts = []
    for b in range(w.B):
        c = [0]
        while c[-1] < nb[b]:
            c.append(min(int(nb[b]), c[-1] + int(rng.integers(1, tile_capacity + 1))))
        cuts.append(c)
    T = max(len(c) - 1 for c in cuts)
    tiles = []
    for i in range(T):
        blocks = np.zeros((w.B, tile_capacity), dtype=np.int32)
        counts = np.zeros(w.B, dtype=np.int32)
        last = np.full(w.B, w.block_size, dtype=np.int32)
        for b in range(w.B):
            if i + 1 < len(cuts[b]):
                lo, hi = cuts[b][i], cuts[b][i + 1]
                blocks[b, :hi - lo] = w.block_table[b, lo:hi]
                counts[b] = hi - lo
                if hi == nb[b]:
                    last[b] = int(w.seq_lens[b]) - (hi - 1) * w.block_size
        tiles.append((blocks, counts, last))
    return tiles


def run_tiled(ctx, w, tiles, t, scale=None):
    import torch
    ctx.begin_step(w.B)
    for blocks, counts, last in tiles:
        ctx.step_tile(t["q"], t["k_pool"], t["v_pool"], dev(blocks), dev(counts), dev(last),
                      scale=scale)
    f32 = ctx.finalize(w.B, out_dtype=torch.float32)
    b16 = ctx.finalize(w.B)
    torch.cuda.synchronize()
    return host_f64(f32), host_f64(b16)


@pytest.mark.parametrize("D,bs,G,cap", [(128, 16, 4, 8), (64, 32, 8, 3), (256, 16, 2, 16),
                                        (128, 8, 1, 64), (128, 1, 4, 200), (64, 4, 8, 33),
                                        (256, 4, 4, 40), (256, 1, 8, 100)])
def test_tiled_matches_oneshot_and_oracle(D, bs, G, cap):
    import torch
    rng = np.random.default_rng(D + bs + G)
    lens = [1, bs, 3 * bs + 1, 900, 0, 2500]
    w = workloads.make_workload("tiled", B=len(lens), Hq=G * 2, Hkv=2, D=D, block_size=bs,
                                seq_lens=lens, seed=D * bs + G)
    ctx = context_for(w, tile_capacity=cap)
    t = upload(w)
    tiles = make_tiles(w, cap, rng)
    f32, b16 = run_tiled(ctx, w, tiles, t)
    one = host_f64(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                              out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    assert np.max(np.abs(f32 - one)) <= TILED_VS_ONESHOT
    ref = oracle.load().decode(w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hq=w.Hq,
                               Hkv=w.Hkv, D=w.D, block_size=w.block_size)
    assert_close_to_oracle(b16, ref, "tiled bf16")


def test_tile_order_does_not_matter():
    """Tiles folded in reverse order give the same result within fp32 rounding."""
    import torch
    w = workloads.make_workload("order", B=3, Hq=8, Hkv=2, D=128, block_size=16,
                                seq_lens=[777, 64, 1500], seed=3)
    ctx = context_for(w, tile_capacity=10)
    t = upload(w)
    tiles = make_tiles(w, 10, np.random.default_rng(1))
    fwd, _ = run_tiled(ctx, w, tiles, t)
    # reversed: a tile's last_valid applies to its own last block, wherever it comes
    rev, _ = run_tiled(ctx, w, tiles[::-1], t)
    assert np.max(np.abs(fwd - rev)) <= TILED_VS_ONESHOT


def test_begin_step_resets():
    import torch
    w = workloads.make_workload("reset", B=2, Hq=4, Hkv=2, D=64, block_size=16,
                                seq_lens=[100, 50], seed=4)
    ctx = context_for(w, tile_capacity=16)
    t = upload(w)
    tiles = make_tiles(w, 16, np.random.default_rng(2))
    a, _ = run_tiled(ctx, w, tiles, t)
    b, _ = run_tiled(ctx, w, tiles, t)  # a second step starts from (-inf, 0, 0) again
    assert np.array_equal(a, b)
    ctx.begin_step(w.B)
    empty = ctx.finalize(w.B, out_dtype=torch.float32)
    assert torch.count_nonzero(empty).item() == 0


def test_eight_b_tiled_full_size():
    """The 8B-style batch folded in 4 tiles of 64 blocks per sequence."""
    import torch
    w = workloads.eight_b()
    ctx = context_for(w, tile_capacity=64)
    t = upload(w)
    tiles = make_tiles(w, 64, np.random.default_rng(3))
    f32, b16 = run_tiled(ctx, w, tiles, t)
    one = host_f64(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                              out_dtype=torch.float32))
    assert np.max(np.abs(f32 - one)) <= TILED_VS_ONESHOT


def _steps(ctx, w, dev_tiles, t):
    """One step on the current stream: reset, the device-resident tiles, fp32 finalize."""
    import torch
    ctx.begin_step(w.B)
    for blocks, counts, last in dev_tiles:
        ctx.step_tile(t["q"], t["k_pool"], t["v_pool"], blocks, counts, last)
    return ctx.finalize(w.B, out_dtype=torch.float32)


@pytest.mark.parametrize("tiles_per_seq", [4, 16])
def test_overlapped_tile_steps_match_waiting_ones(tiles_per_seq):
    """Tile steps issued back to back (device-resident tile lists, so each
    starts streaming while the previous finishes) give the same state, bit for
    bit, as tile steps that each wait for the previous one."""
    import torch
    w = workloads.eight_b()
    cap = 256 // tiles_per_seq
    ctx = context_for(w, tile_capacity=cap)
    t = upload(w)
    tiles = [(dev(b), dev(c), dev(l)) for b, c, l in make_tiles(w, cap, np.random.default_rng(5))]
    torch.cuda.synchronize()
    over = _steps(ctx, w, tiles, t).clone()
    ctx.set_tile_overlap(False)
    wait = _steps(ctx, w, tiles, t).clone()
    ctx.set_tile_overlap(True)
    again = _steps(ctx, w, tiles, t)
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    assert torch.equal(over, wait) and torch.equal(over, again)
    one = host_f64(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                              out_dtype=torch.float32))
    assert np.max(np.abs(host_f64(over) - one)) <= TILED_VS_ONESHOT


def test_overlapped_tile_steps_replayed_from_a_graph():
    """A whole step (reset, overlapped tiles, finalize) captured once and
    replayed matches the eager step, and follows new q contents."""
    import torch
    w = workloads.make_workload("graph_tiles", B=6, Hq=16, Hkv=4, D=128, block_size=16,
                                seq_lens=[1000, 5, 0, 333, 4096, 77], seed=23)
    ctx = context_for(w, tile_capacity=12)
    t = upload(w)
    tiles = [(dev(b), dev(c), dev(l)) for b, c, l in make_tiles(w, 12, np.random.default_rng(6))]
    eager = _steps(ctx, w, tiles, t).clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _steps(ctx, w, tiles, t)  # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = _steps(ctx, w, tiles, t)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    t["q"].mul_(-1)
    g.replay()
    flipped = _steps(ctx, w, tiles, t)
    torch.cuda.synchronize()
    assert torch.equal(out, flipped) and not torch.equal(out, eager)
    assert ctx.read_device_errors() == 0


def test_tile_steps_on_alternating_streams():
    """Tile steps of one step on two streams (each ordered after the previous
    one by an event) wait for their predecessor and match one stream."""
    import torch
    w = workloads.make_workload("streams_tiles", B=4, Hq=8, Hkv=2, D=64, block_size=16,
                                seq_lens=[2000, 17, 640, 1], seed=24)
    ctx = context_for(w, tile_capacity=9)
    t = upload(w)
    tiles = [(dev(b), dev(c), dev(l)) for b, c, l in make_tiles(w, 9, np.random.default_rng(7))]
    ref = _steps(ctx, w, tiles, t).clone()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    main = torch.cuda.current_stream()
    for st in streams:
        st.wait_stream(main)
    ctx.begin_step(w.B, stream=streams[0])
    prev = streams[0]
    for i, (blocks, counts, last) in enumerate(tiles):
        st = streams[i % 2]
        st.wait_stream(prev)
        with torch.cuda.stream(st):
            ctx.step_tile(t["q"], t["k_pool"], t["v_pool"], blocks, counts, last, stream=st)
        prev = st
    main.wait_stream(prev)
    got = ctx.finalize(w.B, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    assert ctx.read_device_errors() == 0
