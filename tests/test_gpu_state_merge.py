"""Partial states across contexts (context-parallel decode): each emulated rank
is its own context folding a shard of every sequence's blocks; the exported
states, merged, equal the one-shot decode (fp32, within 1e-3) and the oracle.
The ranks run one after another on one GPU: no kernel waits on another."""
import math

import numpy as np
import pytest

import oracle
from gpu_util import TILED_VS_ONESHOT, assert_close_to_oracle, context_for, dev, host_f64, upload
from paged_gqa_decode_05_gb300 import workloads
from paged_gqa_decode_05_gb300.workloads import bf16_to_f32

pytestmark = pytest.mark.gpu


def shard_tiles(w, n_parts, rng):
    """Per part: (tile_blocks, counts, last_valid) covering a contiguous slice
    of every sequence's blocks (slices may be empty), and the tile width."""
    nb = -(-w.seq_lens.astype(np.int64) // w.block_size)
    cuts = [np.sort(rng.integers(0, int(n) + 1, size=n_parts - 1)) for n in nb]
    bounds = [np.concatenate([[0], c, [n]]).astype(int) for c, n in zip(cuts, nb)]
    cap = max(1, max(int(np.max(np.diff(b))) for b in bounds))
    parts = []
    for p in range(n_parts):
        blocks = np.zeros((w.B, cap), dtype=np.int32)
        counts = np.zeros(w.B, dtype=np.int32)
        last = np.full(w.B, w.block_size, dtype=np.int32)
        for b in range(w.B):
            lo, hi = bounds[b][p], bounds[b][p + 1]
            blocks[b, :hi - lo] = w.block_table[b, lo:hi]
            counts[b] = hi - lo
            if hi == nb[b] and hi > lo:
                last[b] = int(w.seq_lens[b]) - (hi - 1) * w.block_size
        parts.append((blocks, counts, last))
    return parts, cap


def rank_states(w, parts, cap, t):
    """Each part folded by its own context; the exported (m, l, o) stacked."""
    import torch
    ms, ls, os_ = [], [], []
    for blocks, counts, last in parts:
        ctx = context_for(w, tile_capacity=cap)
        ctx.begin_step(w.B)
        ctx.step_tile(t["q"], t["k_pool"], t["v_pool"], dev(blocks), dev(counts), dev(last))
        m, l, o = ctx.export_state(w.B)
        torch.cuda.synchronize()
        assert ctx.read_device_errors() == 0
        ms.append(m); ls.append(l); os_.append(o)
        ctx.close()
    return torch.stack(ms), torch.stack(ls), torch.stack(os_)


@pytest.mark.parametrize("D,bs,G,n_parts", [(128, 16, 4, 2), (64, 32, 8, 3), (256, 16, 2, 4),
                                            (128, 1, 4, 3), (256, 4, 8, 2)])
def test_sharded_states_merge_to_decode(D, bs, G, n_parts):
    import torch
    lens = [1, 3 * bs + 1, 900, 0, 2500, bs]
    w = workloads.make_workload("cp", B=len(lens), Hq=G * 2, Hkv=2, D=D, block_size=bs,
                                seq_lens=lens, seed=D + bs + n_parts)
    t = upload(w)
    parts, cap = shard_tiles(w, n_parts, np.random.default_rng(D * bs + n_parts))
    m, l, o = rank_states(w, parts, cap, t)
    ctx = context_for(w)
    f32 = host_f64(ctx.merge_states(m, l, o, out_dtype=torch.float32))
    b16 = host_f64(ctx.merge_states(m, l, o))
    one = host_f64(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                              out_dtype=torch.float32))
    torch.cuda.synchronize()
    assert np.max(np.abs(f32 - one)) <= TILED_VS_ONESHOT
    ref = oracle.load().decode(w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hq=w.Hq,
                               Hkv=w.Hkv, D=w.D, block_size=w.block_size)
    assert_close_to_oracle(b16, ref, f"merged {n_parts} parts")
    assert np.all(b16[3] == 0.0)  # the empty sequence


def test_single_part_merge_is_finalize():
    """One part: M = m, so O / L is the finalize quotient o / l exactly."""
    import torch
    w = workloads.make_workload("cp1", B=3, Hq=8, Hkv=2, D=128, block_size=16,
                                seq_lens=[700, 33, 1], seed=5)
    t = upload(w)
    parts, cap = shard_tiles(w, 1, np.random.default_rng(0))
    ctx = context_for(w, tile_capacity=cap)
    blocks, counts, last = parts[0]
    ctx.begin_step(w.B)
    ctx.step_tile(t["q"], t["k_pool"], t["v_pool"], dev(blocks), dev(counts), dev(last))
    m, l, o = ctx.export_state(w.B)
    fin32 = ctx.finalize(w.B, out_dtype=torch.float32).cpu().numpy()
    fin16 = ctx.finalize(w.B).float().cpu().numpy()
    mer32 = ctx.merge_states(m[None], l[None], o[None], out_dtype=torch.float32).cpu().numpy()
    mer16 = ctx.merge_states(m[None], l[None], o[None]).float().cpu().numpy()
    assert np.array_equal(mer32, fin32)
    assert np.array_equal(mer16, fin16)


def test_empty_states_merge_to_zero():
    import torch
    w = workloads.make_workload("cp0", B=2, Hq=4, Hkv=2, D=64, block_size=16, seq_lens=[5, 6], seed=6)
    ctx = context_for(w)
    m = torch.full((3, 2, 4), float("-inf"), device="cuda")
    l = torch.zeros((3, 2, 4), device="cuda")
    o = torch.zeros((3, 2, 4, 64), device="cuda")
    out = ctx.merge_states(m, l, o, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_export_state_is_in_natural_units():
    """A one-token sequence: m = scale * q.k (natural log units), l = 1, o = v."""
    import torch
    w = workloads.make_workload("cpu1", B=2, Hq=4, Hkv=2, D=64, block_size=16, seq_lens=[1, 1],
                                seed=7)
    t = upload(w)
    parts, cap = shard_tiles(w, 1, np.random.default_rng(1))
    ctx = context_for(w, tile_capacity=cap)
    blocks, counts, last = parts[0]
    ctx.begin_step(w.B)
    ctx.step_tile(t["q"], t["k_pool"], t["v_pool"], dev(blocks), dev(counts), dev(last))
    m, l, o = (x.double().cpu().numpy() for x in ctx.export_state(w.B))
    scale = 1.0 / math.sqrt(w.D)
    for b in range(w.B):
        blk = w.block_table[b, 0]
        for h in range(w.Hq):
            k = bf16_to_f32(w.k_pool[blk, 0, h // w.G]).astype(np.float64)
            v = bf16_to_f32(w.v_pool[blk, 0, h // w.G]).astype(np.float64)
            q = bf16_to_f32(w.q[b, h]).astype(np.float64)
            assert abs(m[b, h] - scale * float(q @ k)) <= 1e-4 * (1 + abs(m[b, h]))
            assert abs(l[b, h] - 1.0) <= 1e-6
            assert np.max(np.abs(o[b, h] - v)) <= 1e-6 * (1 + np.max(np.abs(v)))
