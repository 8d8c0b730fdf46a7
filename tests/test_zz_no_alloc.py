"""pda_decode_noalloc: the one-shot decode for callers that cannot allocate.

Some callers cannot call cudaMalloc where they decode: code that runs inside
a CUDA-graph capture it does not own, an allocator that forbids allocations
outside its own pool, or an embedder whose device memory budget is fixed
before any model runs.  pda_create allocates a context's workspace, so the
library has one more entry point whose scratch is a static device array.

These tests call it through the C ABI and check its output
  * against the fp64 oracle, at the suite's bar (max |err| <= 2e-2, mean
    |err| <= 2e-3), for every block size and head size the library accepts,
    with empty, one-token, partial-block and multi-stage lengths;
  * against pda_decode (the context-based entry point) within the same bar,
    on two calls in a row;
  * interleaved with context-based decodes of larger batches in the same
    process, which share the split kernels' launch attributes with it.
They also check that a request larger than the static scratch and a call
without a flags word are refused.  The file is named to be collected last,
so a run that stops at the first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest

import oracle
from gpu_util import MAX_ABS, MEAN_ABS, assert_close_to_oracle, context_for, host_f64, upload
from paged_gqa_decode_05_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def noalloc_fn():
    import paged_gqa_decode_05_gb300 as pda
    fn = pda.lib().pda_decode_noalloc
    P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    fn.restype = I32
    fn.argtypes = [P, P, P, I64, P, I32, P, I32, I32, I32, I32, I32, F, P, P, P]
    return fn


def call_noalloc(fn, w, t, out, flags):
    import torch
    return fn(t["q"].data_ptr(), t["k_pool"].data_ptr(), t["v_pool"].data_ptr(), w.num_blocks,
              t["block_table"].data_ptr(), w.max_blocks, t["seq_lens"].data_ptr(), w.B, w.Hq,
              w.Hkv, w.D, w.block_size, float("nan"), out.data_ptr(),
              None if flags is None else flags.data_ptr(), torch.cuda.current_stream().cuda_stream)


def run_noalloc(fn, w, t):
    """One call; returns the bf16 output as float64 on the host."""
    import torch
    out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda", dtype=torch.bfloat16)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert call_noalloc(fn, w, t, out, flags) == 0
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    return host_f64(out)


def oracle_ref(orc, w):
    return orc.decode(w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hq=w.Hq, Hkv=w.Hkv,
                      D=w.D, block_size=w.block_size, n_threads=oracle.host_threads())


def assert_within_bar(got, want, what):
    err = np.abs(got - want)
    assert np.all(np.isfinite(got)), what
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (what, err.max(), err.mean())


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16, 32])
def test_noalloc_matches_oracle(orc, D, bs):
    """Every block size, including those below 8 whose rows are gathered."""
    lens = [0, 1, bs + 1 if bs > 1 else 3, 64 + 5, 3 * 64 + bs - 1 if bs > 1 else 200, 517]
    w = make_workload("noalloc-sweep", B=len(lens), Hq=8, Hkv=2, D=D, block_size=bs,
                      seq_lens=lens, seed=300 + D + bs)
    got = run_noalloc(noalloc_fn(), w, upload(w))
    assert_close_to_oracle(got, oracle_ref(orc, w), f"noalloc D={D} bs={bs}")
    assert np.all(got[0] == 0.0)  # the empty sequence gives a zero row


def test_noalloc_matches_decode_on_two_calls_in_a_row(orc):
    import torch
    fn = noalloc_fn()
    cases = [
        make_workload("noalloc-a", B=6, Hq=32, Hkv=8, D=128, block_size=16,
                      seq_lens=[4096, 1, 0, 777, 2048, 130], seed=41),
        make_workload("noalloc-b", B=5, Hq=16, Hkv=2, D=64, block_size=4,
                      seq_lens=[33, 9000, 64, 5, 1500], seed=42),
    ]
    for w in cases:  # two calls in a row; the second reuses the scratch the first left
        t = upload(w)
        ctx = context_for(w)
        ref = host_f64(ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"],
                                  t["seq_lens"]))
        torch.cuda.synchronize()
        got = run_noalloc(fn, w, t)
        assert_within_bar(got, ref, w.name)
        assert_close_to_oracle(got, oracle_ref(orc, w), w.name)
        ctx.close()


def test_noalloc_interleaved_with_context_decodes(orc):
    """A context made for a large batch, a small allocation-free call, then the
    context's full batch, and again: neither path may leave the split kernel's
    launch limits below what the other launches with."""
    import torch
    fn = noalloc_fn()
    big = make_workload("noalloc-big-batch", B=1024, Hq=8, Hkv=2, D=128, block_size=16,
                        seq_lens=np.random.default_rng(7).integers(0, 200, size=1024), seed=45)
    small = make_workload("noalloc-one", B=1, Hq=8, Hkv=2, D=128, block_size=16,
                          seq_lens=[300], seed=46)
    tb, ts = upload(big), upload(small)
    ctx = context_for(big)
    ref_big = oracle_ref(orc, big)
    ref_small = oracle_ref(orc, small)
    for _ in range(2):
        assert_close_to_oracle(run_noalloc(fn, small, ts), ref_small, "noalloc batch 1")
        out = ctx.decode(tb["q"], tb["k_pool"], tb["v_pool"], tb["block_table"], tb["seq_lens"])
        torch.cuda.synchronize()
        assert ctx.read_device_errors() == 0
        assert_close_to_oracle(host_f64(out), ref_big, "context batch 1024 after noalloc")
    ctx.close()


def test_noalloc_repeated_calls_agree(orc):
    import torch
    fn = noalloc_fn()
    w = make_workload("noalloc-c", B=3, Hq=8, Hkv=8, D=256, block_size=8,
                      seq_lens=[100, 2500, 17], seed=43)
    t = upload(w)
    outs = []
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = torch.empty((w.B, w.Hq, w.D), device="cuda", dtype=torch.bfloat16)
        assert call_noalloc(fn, w, t, out, flags) == 0
        outs.append(out)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    ref = oracle_ref(orc, w)
    for out in outs:
        assert_close_to_oracle(host_f64(out), ref, "repeated noalloc")
    assert torch.equal(outs[0], outs[1])  # same inputs, same plan: identical bits


def test_noalloc_refuses_requests_beyond_its_scratch_and_without_flags():
    import torch
    import paged_gqa_decode_05_gb300 as pda
    fn = noalloc_fn()
    w = make_workload("noalloc-big", B=1024, Hq=64, Hkv=8, D=256, block_size=16,
                      seq_lens=[1] * 1024, seed=44)
    t = upload(w)
    out = torch.empty((w.B, w.Hq, w.D), device="cuda", dtype=torch.bfloat16)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert call_noalloc(fn, w, t, out, flags) == pda.ERR_INVALID_ARG
    assert b"scratch" in pda.lib().pda_last_error()
    assert call_noalloc(fn, w, t, out, None) == pda.ERR_INVALID_ARG
    assert b"device_flags" in pda.lib().pda_last_error()
