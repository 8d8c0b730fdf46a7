"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerance (bf16 outputs vs the fp64 oracle, over all B*Hq*D elements):
max |err| <= 2e-2 and mean |err| <= 2e-3.
"""
import numpy as np
import pytest

import oracle
from gpu_util import assert_close_to_oracle, context_for, host_f64, upload
from paged_gqa_decode_05_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.load()


def run_both(orc, w, scale=None, ctx=None):
    import torch
    ctx = ctx or context_for(w)
    t = upload(w)
    out = ctx.decode(t["q"], t["k_pool"], t["v_pool"], t["block_table"], t["seq_lens"], scale=scale)
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    ref = orc.decode(w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hq=w.Hq, Hkv=w.Hkv,
                     D=w.D, block_size=w.block_size, scale=scale,
                     n_threads=oracle.host_threads())
    return host_f64(out), ref


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
def test_named_workload(orc, name):
    """The five decode workloads at full size, every output element compared."""
    w = workloads.WORKLOADS[name]()
    got, ref = run_both(orc, w)
    assert_close_to_oracle(got, ref, name)


def _lens(bs, extra=()):
    # empty, one token, a partial block, exactly full blocks, several stages with a ragged tail
    return [0, 1, bs - 1, bs, 2 * bs, 64 * 3 + bs + 3, 700, *extra]


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_shape_sweep(orc, D, bs, G):
    Hkv = 2 if G < 8 else 1
    lens = _lens(bs)
    w = workloads.make_workload("sweep", B=len(lens), Hq=G * Hkv, Hkv=Hkv, D=D, block_size=bs,
                                seq_lens=lens, seed=D * 100 + bs * 10 + G,
                                pool_blocks=None, max_blocks=None)
    got, ref = run_both(orc, w)
    assert_close_to_oracle(got, ref, f"D={D} bs={bs} G={G}")
    # an empty sequence yields an exactly zero row
    assert np.all(got[0] == 0.0)


def test_custom_scale(orc):
    w = workloads.make_workload("scale", B=3, Hq=8, Hkv=2, D=128, block_size=16,
                                seq_lens=[100, 513, 77], seed=5)
    for scale in (0.0, 0.02, -0.1, 0.3):
        got, ref = run_both(orc, w, scale=scale)
        assert_close_to_oracle(got, ref, f"scale={scale}")


def test_long_single_sequence(orc):
    """One sequence spread over every CTA: many partial states merged."""
    w = workloads.make_workload("long", B=1, Hq=8, Hkv=1, D=128, block_size=32,
                                seq_lens=[32768 - 5], seed=6)
    got, ref = run_both(orc, w)
    assert_close_to_oracle(got, ref, "long")


def test_batch_over_launch_chunk(orc):
    """More sequences than one launch carries (1024): the batch is chunked."""
    rng = np.random.default_rng(8)
    lens = rng.integers(0, 90, size=1100)
    w = workloads.make_workload("chunks", B=1100, Hq=4, Hkv=2, D=64, block_size=16,
                                seq_lens=lens, seed=9)
    got, ref = run_both(orc, w)
    assert_close_to_oracle(got, ref, "chunked")


def test_peaky_softmax(orc):
    """Large scores (K spikes x3 on 1% of tokens, scale 1): one token dominates."""
    w = workloads.make_workload("peaky", B=4, Hq=16, Hkv=4, D=128, block_size=16,
                                seq_lens=[4000, 37, 1025, 2048], seed=10, spike_frac=0.01)
    got, ref = run_both(orc, w, scale=1.0)
    assert_close_to_oracle(got, ref, "peaky")
