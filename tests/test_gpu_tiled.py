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
