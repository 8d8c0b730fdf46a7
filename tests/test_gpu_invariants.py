"""GPU checks that need no tolerance: bit-exact gather, invariants that leave
the kernel's arithmetic unchanged, determinism, closed forms and device flags."""
import numpy as np
import pytest

import oracle
from gpu_util import context_for, dev, host_f64, upload
from paged_gqa_decode_05_gb300 import workloads
from paged_gqa_decode_05_gb300.workloads import bf16_bits, bf16_to_f32, make_workload

pytestmark = pytest.mark.gpu


def _decode(ctx, w, **kw):
    import torch
    t = upload(w)
    out = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], **kw)
    torch.cuda.synchronize()
    return out


def _w(seed=1, D=128, bs=16, G=4, Hkv=2, lens=(300, 1, 0, 129, 64), pool=None, width=None):
    return make_workload("inv", B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs,
                         seq_lens=list(lens), seed=seed, pool_blocks=pool, max_blocks=width)


@pytest.mark.parametrize("D,bs", [(64, 16), (128, 32), (256, 8), (128, 64), (128, 1), (64, 2),
                                  (256, 4)])
def test_gather_bit_exact(D, bs):
    """The loader's staged rows equal the oracle's gather, byte for byte."""
    import torch
    w = _w(seed=D + bs, D=D, bs=bs, lens=(5, 200, 0, 3 * bs, 1000), pool=200 if bs >= 8 else None)
    ctx = context_for(w)
    t = upload(w)
    k_rows, v_rows = ctx.debug_gather(t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    k_rows = k_rows.view(torch.int16).cpu().numpy().view(np.uint16)
    v_rows = v_rows.view(torch.int16).cpu().numpy().view(np.uint16)
    orc = oracle.load()
    for b in range(w.B):
        n = int(w.seq_lens[b])
        for g in range(w.Hkv):
            k, v = orc.gather(w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hkv=w.Hkv, D=w.D,
                              block_size=w.block_size, b=b, kvh=g)
            assert np.array_equal(k_rows[b, g, :n], k), (b, g)
            assert np.array_equal(v_rows[b, g, :n], v), (b, g)


def test_block_permutation_bit_identical():
    w = _w(seed=3, pool=90)
    ctx = context_for(w)
    base = _decode(ctx, w).clone()
    perm = np.random.default_rng(4).permutation(w.num_blocks)
    k2 = np.empty_like(w.k_pool); v2 = np.empty_like(w.v_pool)
    k2[perm] = w.k_pool; v2[perm] = w.v_pool
    w.k_pool, w.v_pool, w.block_table = k2, v2, perm[w.block_table].astype(np.int32)
    again = _decode(ctx, w)
    assert np.array_equal(base.cpu().float().numpy(), again.cpu().float().numpy())


def test_deterministic():
    w = _w(seed=5, lens=(4096, 333, 17, 2049))
    ctx = context_for(w)
    a = _decode(ctx, w).clone()
    b = _decode(ctx, w)
    assert np.array_equal(a.cpu().float().numpy(), b.cpu().float().numpy())


def test_garbage_outside_valid_rows_ignored():
    """NaN bits in unused blocks, unused table entries and masked tail slots."""
    w = _w(seed=6, lens=(37, 80, 1, 130), pool=60, width=12)
    ctx = context_for(w)
    base = host_f64(_decode(ctx, w))
    used = set()
    nan = np.uint16(0x7FC1)
    for b in range(w.B):
        n = int(w.seq_lens[b]); nb = -(-n // w.block_size)
        used.update(int(x) for x in w.block_table[b, :nb])
        last = w.block_table[b, nb - 1]
        w.k_pool[last, n - (nb - 1) * w.block_size:] = nan
        w.v_pool[last, n - (nb - 1) * w.block_size:] = nan
    unused = [i for i in range(w.num_blocks) if i not in used]
    w.k_pool[unused] = nan; w.v_pool[unused] = nan
    for b in range(w.B):
        nb = -(-int(w.seq_lens[b]) // w.block_size)
        w.block_table[b, nb:] = unused[b % len(unused)]
    got = host_f64(_decode(ctx, w))
    assert np.all(np.isfinite(got))
    assert np.array_equal(got, base)
    assert ctx.read_device_errors() == 0


@pytest.mark.parametrize("bs", [16, 2])
def test_slot_layout_strides_identical(bs):
    """The same cache in the slot layout [slot, K|V, kv_head, block, D]."""
    import torch
    import paged_gqa_decode_05_gb300 as pda
    w = _w(seed=7, bs=bs, lens=(100, 257, 3))
    ctx = context_for(w)
    base = _decode(ctx, w).cpu().float().numpy()
    nb, bs, Hkv, D = w.k_pool.shape
    slab = np.empty((nb, 2, Hkv, bs, D), dtype=np.uint16)
    slab[:, 0] = w.k_pool.transpose(0, 2, 1, 3)
    slab[:, 1] = w.v_pool.transpose(0, 2, 1, 3)
    flat = dev(slab.ravel())
    strides = pda.slot_strides(num_q_heads=w.Hq, num_kv_heads=w.Hkv, head_dim=w.D,
                               block_size=w.block_size)
    t = upload(w)
    out = ctx.decode(t["q"], flat, flat[Hkv * bs * D:], t["block_table"], t["seq_lens"],
                     strides=strides, num_blocks=nb)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().float().numpy(), base)


def test_constant_values_exact():
    w = _w(seed=8, lens=(500, 17, 64))
    c = bf16_bits(np.linspace(-3, 3, w.D).astype(np.float32) // 0.125 * 0.125)
    w.v_pool[...] = c
    ctx = context_for(w)
    got = host_f64(_decode(ctx, w))
    want = np.broadcast_to(bf16_to_f32(c).astype(np.float64), got.shape)
    assert np.array_equal(got, want)


def test_single_token_returns_value_row():
    w = _w(seed=9, lens=(1, 1, 1))
    ctx = context_for(w)
    got = host_f64(_decode(ctx, w))
    for b in range(w.B):
        blk = w.block_table[b, 0]
        for h in range(w.Hq):
            assert np.array_equal(got[b, h], bf16_to_f32(w.v_pool[blk, 0, h // w.G]).astype(np.float64))


def test_bad_block_id_is_flagged_not_faulted():
    w = _w(seed=10, lens=(40, 40))
    w.block_table[1, 1] = w.num_blocks + 5
    ctx = context_for(w)
    _decode(ctx, w)
    import paged_gqa_decode_05_gb300 as pda
    assert ctx.read_device_errors() & pda.DEVERR_BAD_BLOCK_ID
    assert ctx.read_device_errors() == 0  # cleared by the previous read


def test_length_beyond_table_is_flagged():
    w = _w(seed=11, lens=(40, 40), width=3)
    w.seq_lens[0] = 200  # needs 13 blocks; the table row has 3
    ctx = context_for(w)
    _decode(ctx, w)
    import paged_gqa_decode_05_gb300 as pda
    assert ctx.read_device_errors() & pda.DEVERR_BAD_LENGTH


def test_invalid_arguments_rejected():
    import torch
    import paged_gqa_decode_05_gb300 as pda
    w = _w(seed=12, lens=(10, 20))
    ctx = context_for(w)
    t = upload(w)
    with pytest.raises(pda.PdaError):
        ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                   scale=float("inf"))
    with pytest.raises(pda.PdaError):
        ctx.begin_step(w.B + 1)
    big = workloads.make_workload("big", B=3, Hq=w.Hq, Hkv=w.Hkv, D=w.D, block_size=w.block_size,
                                  seq_lens=[1, 1, 1], seed=1)
    tb = upload(big)
    with pytest.raises(pda.PdaError):  # batch > max_seqs
        ctx.decode(tb["q"], tb["k_pool"], tb["v_pool"], tb["block_table"], tb["seq_lens"])
    torch.cuda.synchronize()


def test_table_too_wide_for_int32_plan_rejected():
    """A launch's plan-block prefix is int32: a table width that could overflow
    it for the batch is refused on the host, before anything is launched (the
    table pointer is never read)."""
    import torch
    import paged_gqa_decode_05_gb300 as pda
    w = _w(seed=13, lens=(10, 20))
    ctx = pda.Context(max_seqs=1024, num_q_heads=w.Hq, num_kv_heads=w.Hkv, head_dim=w.D,
                      block_size=w.block_size)
    t = upload(w)
    q = torch.zeros((1024, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lens = torch.ones(1024, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    L = pda.lib()
    width = 1 << 21  # 1024 rows x (2^21 + unit cost) plan blocks > 2^31 - 1
    st = L.pda_decode(ctx._ctx, q.data_ptr(), t["k_pool"].data_ptr(), t["v_pool"].data_ptr(),
                      int(w.k_pool.shape[0]), t["block_table"].data_ptr(), width, lens.data_ptr(),
                      1024, float("nan"), out.data_ptr(), None)
    assert st == pda.ERR_INVALID_ARG
    assert b"too large" in L.pda_last_error()
    torch.cuda.synchronize()


@pytest.mark.parametrize("bs", [2, 16])
def test_padded_token_stride_identical(bs):
    """Token rows padded by 8 elements (strides not multiples of D): block size
    2 takes the 16-byte copy loader, 16 the TMA boxes; both match the dense pool."""
    import torch
    w = _w(seed=13, bs=bs, lens=(77, 300, 2))
    ctx = context_for(w)
    base = _decode(ctx, w).cpu().float().numpy()
    nb, _, Hkv, D = w.k_pool.shape
    row = Hkv * D + 8
    def padded(pool):
        a = np.zeros((nb, bs, row), dtype=np.uint16)
        a[:, :, :Hkv * D] = pool.reshape(nb, bs, Hkv * D)
        return dev(a.ravel())
    t = upload(w)
    out = ctx.decode(t["q"], padded(w.k_pool), padded(w.v_pool), t["block_table"], t["seq_lens"],
                     strides=(bs * row, row, D), num_blocks=nb)
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    assert np.array_equal(out.cpu().float().numpy(), base)


@pytest.mark.parametrize("D,bs", [(128, 16), (64, 1), (256, 32)])
def test_token_permutation_within_tolerance(D, bs):
    """Moving every token's K and V rows together to another position of the
    same sequence changes only the order of the softmax sums: the fp32 results
    agree to the kernel's own rounding, and both meet the oracle bar."""
    import torch
    from gpu_util import assert_close_to_oracle
    w = _w(seed=30 + D + bs, D=D, bs=bs, lens=(1000, 3, 0, 257, 64 * 5 + 7))
    ctx = context_for(w)
    t = upload(w)
    base = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                      out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(31)
    k2, v2 = w.k_pool.copy(), w.v_pool.copy()
    for b in range(w.B):
        n = int(w.seq_lens[b])
        tok = np.arange(n)
        src = (w.block_table[b, tok // w.block_size], tok % w.block_size)
        pt = rng.permutation(n)
        dst = (w.block_table[b, pt // w.block_size], pt % w.block_size)
        k2[dst] = w.k_pool[src]
        v2[dst] = w.v_pool[src]
    w.k_pool, w.v_pool = k2, v2
    t = upload(w)
    perm = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"],
                      out_dtype=torch.float32).cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    assert np.abs(perm - base).max() <= 2e-4  # twice the fp32 error budget of one decode
    ref = oracle.load().decode(w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hq=w.Hq,
                               Hkv=w.Hkv, D=w.D, block_size=w.block_size)
    assert_close_to_oracle(perm, ref, "token permutation", rounded=False)


def test_split_units_merge_identically_call_after_call():
    """The pieces of a unit split across CTAs find the piece that merges them
    through per-unit counters that every launch leaves at zero: repeated calls,
    and calls alternating between batches whose units split differently, give
    the same bits each time."""
    import torch
    a = _w(seed=40, lens=(4096, 5000, 17, 2049, 3333, 1, 0, 1024), G=4, Hkv=2)
    b = _w(seed=41, lens=(64 * 300 + 5, 3, 700), G=8, Hkv=1)
    ctx_a = context_for(a, max_seqs=8)
    ta = upload(a)
    first = ctx_a.decode(ta["q"], ta["k_pool"], ta["v_pool"], ta["block_table"], ta["seq_lens"]).clone()
    ctx_b = context_for(b)
    tb = upload(b)
    first_b = ctx_b.decode(tb["q"], tb["k_pool"], tb["v_pool"], tb["block_table"], tb["seq_lens"]).clone()
    for _ in range(4):
        again = ctx_a.decode(ta["q"], ta["k_pool"], ta["v_pool"], ta["block_table"], ta["seq_lens"])
        again_b = ctx_b.decode(tb["q"], tb["k_pool"], tb["v_pool"], tb["block_table"], tb["seq_lens"])
        torch.cuda.synchronize()
        assert torch.equal(again, first) and torch.equal(again_b, first_b)
    # the same context on a batch with another split, then the first batch again
    c = _w(seed=42, lens=(100, 9000, 64, 65), G=4, Hkv=2)
    tc = upload(c)
    ctx_a.decode(tc["q"], tc["k_pool"], tc["v_pool"], tc["block_table"], tc["seq_lens"])
    again = ctx_a.decode(ta["q"], ta["k_pool"], ta["v_pool"], ta["block_table"], ta["seq_lens"])
    torch.cuda.synchronize()
    assert torch.equal(again, first)
    assert ctx_a.read_device_errors() == 0 and ctx_b.read_device_errors() == 0
    ref = oracle.load().decode(a.q, a.k_pool, a.v_pool, a.block_table, a.seq_lens, Hq=a.Hq,
                               Hkv=a.Hkv, D=a.D, block_size=a.block_size)
    from gpu_util import assert_close_to_oracle
    assert_close_to_oracle(host_f64(first), ref, "split-unit merge")
