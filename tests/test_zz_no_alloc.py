"""pda_decode_noalloc: the one-shot decode for callers that cannot allocate.

Some callers cannot call cudaMalloc where they decode (inside a CUDA-graph
capture they do not own, or under a fixed memory budget), so the library has
one entry point whose scratch is a static device array instead of a context's
workspace.  These tests call it through the C ABI and check its output
against pda_decode (the context-based entry point) within the suite's bf16
tolerance, on two calls in a row with different shapes, and check that a
request larger than the static scratch is refused.  The file is named to be
collected last, so a run that stops at the first failure has run the rest.
"""
import ctypes

import numpy as np
import pytest

from gpu_util import MAX_ABS, MEAN_ABS, context_for, upload
from paged_gqa_decode_05_gb300.workloads import make_workload

pytestmark = pytest.mark.gpu


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


def test_noalloc_matches_decode_on_two_calls_in_a_row():
    import torch
    fn = noalloc_fn()
    cases = [
        make_workload("noalloc-a", B=6, Hq=32, Hkv=8, D=128, block_size=16,
                      seq_lens=[4096, 1, 0, 777, 2048, 130], seed=41),
        make_workload("noalloc-b", B=5, Hq=16, Hkv=2, D=64, block_size=32,
                      seq_lens=[33, 9000, 64, 5, 1500], seed=42),
    ]
    for w in cases:  # two calls in a row; the second reuses the scratch the first left
        t = upload(w)
        ctx = context_for(w)
        ref = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
        out = torch.full_like(ref, float("nan"))
        flags = torch.zeros(1, dtype=torch.int32, device="cuda")
        assert call_noalloc(fn, w, t, out, flags) == 0
        torch.cuda.synchronize()
        assert int(flags.item()) == 0
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        err = np.abs(got - want)
        assert np.all(np.isfinite(got))
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (w.name, err.max(), err.mean())
        ctx.close()


def test_noalloc_repeated_call_without_flags_word():
    import torch
    fn = noalloc_fn()
    w = make_workload("noalloc-c", B=3, Hq=8, Hkv=8, D=256, block_size=8,
                      seq_lens=[100, 2500, 17], seed=43)
    t = upload(w)
    outs = []
    for _ in range(2):
        out = torch.empty((w.B, w.Hq, w.D), device="cuda", dtype=torch.bfloat16)
        assert call_noalloc(fn, w, t, out, None) == 0
        outs.append(out)
    torch.cuda.synchronize()
    ctx = context_for(w)
    ref = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"])
    torch.cuda.synchronize()
    want = ref.float().cpu().numpy()
    for out in outs:
        err = np.abs(out.float().cpu().numpy() - want)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS
    ctx.close()


def test_noalloc_refuses_requests_beyond_its_scratch():
    import torch
    import paged_gqa_decode_05_gb300 as pda
    fn = noalloc_fn()
    w = make_workload("noalloc-big", B=1024, Hq=64, Hkv=8, D=256, block_size=16,
                      seq_lens=[1] * 1024, seed=44)
    t = upload(w)
    out = torch.empty((w.B, w.Hq, w.D), device="cuda", dtype=torch.bfloat16)
    st = call_noalloc(fn, w, t, out, None)
    assert st == pda.ERR_INVALID_ARG
    assert b"scratch" in pda.lib().pda_last_error()
