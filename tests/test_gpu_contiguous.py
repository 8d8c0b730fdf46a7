"""Contiguous-KV decode (blhd layout, identity block table) against the oracle
and against the paged path with an explicit identity table (bit-identical)."""
import numpy as np
import pytest

import oracle
from gpu_util import assert_close_to_oracle, context_for, dev, host_f64, upload
from paged_gqa_decode_05_gb300 import workloads

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D,bs,G", [(128, 16, 4), (64, 32, 8), (256, 8, 2), (128, 64, 1),
                                    (256, 2, 4)])
def test_contiguous_matches_oracle_and_identity_table(D, bs, G):
    import torch
    lens = [0, 1, bs + 3, 900, 4 * 64 + 1, 2048]
    w = workloads.make_workload("contig", B=len(lens), Hq=G * 2, Hkv=2, D=D, block_size=bs,
                                seq_lens=lens, seed=D + bs + G)
    k, v = workloads.contiguous_kv(w)
    S = k.shape[1]
    ctx = context_for(w)
    t = upload(w)
    out = ctx.decode_contiguous(t["q"], dev(k), dev(v), t["seq_lens"])
    # the same cache as a paged pool with the identity table
    ident = (np.arange(w.B)[:, None] * (S // bs) + np.arange(S // bs)[None, :]).astype(np.int32)
    k_pool = k.reshape(w.B * S // bs, bs, w.Hkv, D)
    v_pool = v.reshape(w.B * S // bs, bs, w.Hkv, D)
    paged = ctx.decode(t["q"], dev(k_pool), dev(v_pool), dev(ident), t["seq_lens"])
    torch.cuda.synchronize()
    assert ctx.read_device_errors() == 0
    assert np.array_equal(out.cpu().float().numpy(), paged.cpu().float().numpy())
    ref = oracle.load().decode(w.q, k_pool, v_pool, ident, w.seq_lens, Hq=w.Hq, Hkv=w.Hkv, D=D,
                               block_size=bs, n_threads=oracle.host_threads())
    assert_close_to_oracle(host_f64(out), ref, "contiguous")


def test_contiguous_rejects_bad_length():
    import paged_gqa_decode_05_gb300 as pda
    w = workloads.make_workload("c", B=2, Hq=4, Hkv=2, D=64, block_size=16, seq_lens=[5, 9], seed=1)
    ctx = context_for(w)
    t = upload(w)
    k = dev(np.zeros((2, 24, 2, 64), np.uint16))
    with pytest.raises(pda.PdaError):  # 24 is not a multiple of the block size
        ctx.decode_contiguous(t["q"], k, k, t["seq_lens"])
