"""Pins for the fp64 oracle: checks against facts fixed outside the oracle.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with:
  * the hand-worked examples in ``golden/worked_examples.json``;
  * closed forms (constant V, one token, equal keys, zero scale, a dominant key,
    an empty sequence);
  * a library routine (``torch.nn.functional.scaled_dot_product_attention`` in
    float64 on a densely gathered copy, with the GQA heads repeated);
  * a second, pure-Python formulation (``oracle.brute``) on tiny inputs;
  * invariants (pool-block permutation, token permutation, garbage outside
    the valid rows, a score shift, linearity in V, convexity);
  * an independent numpy gather (bit-exact) and an alternative stride layout.

``tests/test_oracle_pins.py`` runs every pin on the oracle; the mutant test runs
them on deliberately broken copies and requires each copy to fail at least one.
"""
from __future__ import annotations

import json
import math
import os
from typing import Callable, Dict, List

import numpy as np

from oracle import brute
from paged_gqa_decode_05_gb300.workloads import bf16_bits, bf16_to_f32, make_workload

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "worked_examples.json")


def _bits(values) -> np.ndarray:
    a = np.asarray(values, dtype=np.float32)
    bits = bf16_bits(a)
    assert np.array_equal(bf16_to_f32(bits), a), "fixture value not exact in bf16"
    return bits


def _small(seed, B=2, Hq=4, Hkv=2, D=8, bs=4, lens=(7, 13), pool=None, width=None):
    return make_workload("pin", B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=bs, seq_lens=list(lens),
                         seed=seed, pool_blocks=pool, max_blocks=width)


def _run(orc, w, **kw):
    return orc.decode(w.q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hq=w.Hq, Hkv=w.Hkv,
                      D=w.D, block_size=w.block_size, **kw)


def _dense_kv(w, b):
    """numpy fancy-index gather of sequence b: float64 [n, Hkv, D] for K and V."""
    n = int(w.seq_lens[b])
    t = np.arange(n)
    blk = w.block_table[b, t // w.block_size]
    k = bf16_to_f32(w.k_pool[blk, t % w.block_size]).astype(np.float64)
    v = bf16_to_f32(w.v_pool[blk, t % w.block_size]).astype(np.float64)
    return k, v


# --------------------------------------------------------------------------- golden

def pin_worked_examples(orc):
    with open(GOLDEN) as f:
        data = json.load(f)
    for ex in data["examples"]:
        scale = math.log(3.0) if ex["scale"] == "ln3" else float(ex["scale"])
        out = orc.decode(_bits(ex["q"]), _bits(ex["k_pool"]), _bits(ex["v_pool"]),
                         np.asarray(ex["block_table"], np.int32),
                         np.asarray(ex["seq_lens"], np.int32), Hq=ex["Hq"], Hkv=ex["Hkv"],
                         D=ex["D"], block_size=ex["block_size"], scale=scale)
        np.testing.assert_allclose(out, np.asarray(ex["expected"]), rtol=0, atol=1e-13,
                                   err_msg=ex["name"])


# --------------------------------------------------------------------------- closed forms

def pin_constant_v(orc):
    w = _small(11, D=8, lens=(9, 30))
    c = _bits(np.linspace(-2, 2, w.D) // 0.25 * 0.25)
    w.v_pool[...] = c
    out = _run(orc, w)
    np.testing.assert_allclose(out, np.broadcast_to(bf16_to_f32(c), out.shape), rtol=0, atol=1e-14)


def pin_single_token(orc):
    w = _small(12, lens=(1, 1))
    out = _run(orc, w)
    for b in range(w.B):
        blk = w.block_table[b, 0]
        for h in range(w.Hq):
            row = bf16_to_f32(w.v_pool[blk, 0, h // w.G]).astype(np.float64)
            np.testing.assert_array_equal(out[b, h], row)


def pin_equal_keys_mean(orc):
    w = _small(13, lens=(10, 17))
    w.k_pool[...] = w.k_pool[0, 0, 0]          # one key everywhere
    out = _run(orc, w)
    for b in range(w.B):
        _, v = _dense_kv(w, b)
        for h in range(w.Hq):
            np.testing.assert_allclose(out[b, h], v[:, h // w.G].mean(axis=0), rtol=0, atol=1e-13)


def pin_zero_scale_mean(orc):
    w = _small(14, lens=(6, 21))
    out = _run(orc, w, scale=0.0)
    for b in range(w.B):
        _, v = _dense_kv(w, b)
        for h in range(w.Hq):
            np.testing.assert_allclose(out[b, h], v[:, h // w.G].mean(axis=0), rtol=0, atol=1e-13)


def pin_dominant_key(orc):
    """q.k of one token beats every other by far more than 50 nats."""
    w = _small(15, D=4, lens=(12, 5))
    w.q[...] = _bits([1.0, 0.0, 0.0, 0.0])
    w.k_pool[...] = _bits([0.0, 1.0, 1.0, 1.0])
    hot = {0: 7, 1: 4}
    for b, t in hot.items():
        w.k_pool[w.block_table[b, t // w.block_size], t % w.block_size, :] = _bits([256.0, 0, 0, 0])
    out = _run(orc, w, scale=1.0)
    for b, t in hot.items():
        blk = w.block_table[b, t // w.block_size]
        for h in range(w.Hq):
            row = bf16_to_f32(w.v_pool[blk, t % w.block_size, h // w.G]).astype(np.float64)
            np.testing.assert_allclose(out[b, h], row, rtol=0, atol=1e-12)


def pin_huge_scores(orc):
    """Scores in the thousands: the result must stay finite and exact."""
    w = _small(16, D=8, lens=(9, 14))
    ref = brute.decode(w.q.tolist(), w.k_pool.ravel().tolist(), w.v_pool.ravel().tolist(),
                       w.block_table.tolist(), w.seq_lens.tolist(), Hq=w.Hq, Hkv=w.Hkv, D=w.D,
                       block_size=w.block_size, scale=500.0)
    out = _run(orc, w, scale=500.0)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out, np.asarray(ref), rtol=0, atol=1e-10)


def pin_empty_sequence(orc):
    w = _small(17, lens=(0, 5))
    out = _run(orc, w)
    assert np.array_equal(out[0], np.zeros_like(out[0]))
    assert np.all(np.abs(out[1]) > 0)


# --------------------------------------------------------------------------- library / brute force

def pin_sdpa_library(orc):
    """fp64 SDPA (a library routine) on a numpy-gathered dense copy."""
    import torch
    import torch.nn.functional as F
    for seed, (Hq, Hkv, bs, lens) in enumerate([(4, 2, 4, (7, 13)), (6, 3, 1, (5, 11)),
                                               (8, 8, 16, (40, 3)), (8, 1, 2, (9, 1))]):
        w = _small(100 + seed, Hq=Hq, Hkv=Hkv, D=16, bs=bs, lens=lens)
        out = _run(orc, w)
        for b in range(w.B):
            k, v = _dense_kv(w, b)
            q = torch.from_numpy(bf16_to_f32(w.q[b]).astype(np.float64))[None, :, None, :]
            kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(w.G, dim=0)[None]
            vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(w.G, dim=0)[None]
            ref = F.scaled_dot_product_attention(q, kt, vt, scale=1.0 / math.sqrt(w.D))
            np.testing.assert_allclose(out[b], ref[0, :, 0].numpy(), rtol=0, atol=1e-12)


def pin_brute_force(orc):
    cases = [dict(Hq=4, Hkv=2, D=8, bs=4, lens=(7, 13)),
             dict(Hq=2, Hkv=2, D=4, bs=1, lens=(5, 9)),
             dict(Hq=8, Hkv=2, D=8, bs=16, lens=(40, 17), pool=9),
             dict(Hq=3, Hkv=1, D=6, bs=3, lens=(1, 12))]
    for i, c in enumerate(cases):
        w = _small(200 + i, Hq=c["Hq"], Hkv=c["Hkv"], D=c["D"], bs=c["bs"], lens=c["lens"],
                   pool=c.get("pool"))
        ref = brute.decode(w.q.tolist(), w.k_pool.ravel().tolist(), w.v_pool.ravel().tolist(),
                           w.block_table.tolist(), w.seq_lens.tolist(), Hq=w.Hq, Hkv=w.Hkv,
                           D=w.D, block_size=w.block_size)
        np.testing.assert_allclose(_run(orc, w), np.asarray(ref), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- invariants

def pin_block_permutation(orc):
    w = _small(21, lens=(15, 26), pool=20)
    base = _run(orc, w)
    perm = np.random.default_rng(5).permutation(w.num_blocks)      # new position of block i
    k2 = np.empty_like(w.k_pool); v2 = np.empty_like(w.v_pool)
    k2[perm] = w.k_pool; v2[perm] = w.v_pool
    w.k_pool, w.v_pool, w.block_table = k2, v2, perm[w.block_table].astype(np.int32)
    assert np.array_equal(_run(orc, w), base)


def pin_token_permutation(orc):
    w = _small(22, lens=(11, 19))
    base = _run(orc, w)
    rng = np.random.default_rng(6)
    k2, v2 = w.k_pool.copy(), w.v_pool.copy()
    for b in range(w.B):
        n = int(w.seq_lens[b])
        t = np.arange(n)
        src = (w.block_table[b, t // w.block_size], t % w.block_size)
        pt = rng.permutation(n)
        dst = (w.block_table[b, pt // w.block_size], pt % w.block_size)
        k2[dst] = w.k_pool[src]; v2[dst] = w.v_pool[src]
    w.k_pool, w.v_pool = k2, v2
    np.testing.assert_allclose(_run(orc, w), base, rtol=0, atol=1e-13)


def pin_garbage_outside(orc):
    """NaN bits in unused blocks, unused table slots and masked tail slots."""
    w = _small(23, lens=(6, 9), pool=12, width=5)
    base = _run(orc, w)
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
        w.block_table[b, nb:] = unused[0]
    out = _run(orc, w)
    assert np.array_equal(out, base)


def pin_score_shift(orc):
    """An extra dimension with q=1 and the same k=c on every token shifts all
    scores of a head equally; softmax does not move."""
    w = _small(24, D=8, lens=(8, 12))
    base = _run(orc, w)
    D2 = w.D + 1
    q2 = np.concatenate([w.q, np.full(w.q.shape[:-1] + (1,), bf16_bits(np.float32(1.0)))], -1)
    c = bf16_bits(np.float32(24.0))
    k2 = np.concatenate([w.k_pool, np.full(w.k_pool.shape[:-1] + (1,), c)], -1)
    v2 = np.concatenate([w.v_pool, np.zeros(w.v_pool.shape[:-1] + (1,), np.uint16)], -1)
    out = orc.decode(q2, k2, v2, w.block_table, w.seq_lens, Hq=w.Hq, Hkv=w.Hkv, D=D2,
                     block_size=w.block_size, scale=1.0 / math.sqrt(w.D))
    np.testing.assert_allclose(out[..., :w.D], base, rtol=0, atol=1e-12)
    assert np.all(out[..., w.D] == 0)


def pin_linear_in_v(orc):
    w = _small(25, lens=(14, 3))
    base = _run(orc, w)
    v = bf16_to_f32(w.v_pool)
    w.v_pool = bf16_bits(v * np.float32(-2.0))          # exact in bf16
    np.testing.assert_allclose(_run(orc, w), -2.0 * base, rtol=0, atol=1e-13)


def pin_convex_combination(orc):
    w = _small(26, lens=(16, 29))
    out = _run(orc, w)
    for b in range(w.B):
        _, v = _dense_kv(w, b)
        for h in range(w.Hq):
            lo, hi = v[:, h // w.G].min(0), v[:, h // w.G].max(0)
            assert np.all(out[b, h] >= lo - 1e-12) and np.all(out[b, h] <= hi + 1e-12)


# --------------------------------------------------------------------------- gather / layout

def pin_gather_bits(orc):
    w = _small(27, Hq=4, Hkv=2, D=8, bs=4, lens=(10, 7), pool=9)
    for b in range(w.B):
        n = int(w.seq_lens[b]); t = np.arange(n)
        blk = w.block_table[b, t // w.block_size]
        for kvh in range(w.Hkv):
            k, v = orc.gather(w.k_pool, w.v_pool, w.block_table, w.seq_lens, Hkv=w.Hkv, D=w.D,
                              block_size=w.block_size, b=b, kvh=kvh)
            assert np.array_equal(k, w.k_pool[blk, t % w.block_size, kvh])
            assert np.array_equal(v, w.v_pool[blk, t % w.block_size, kvh])


def pin_slot_layout_strides(orc):
    """The same logical cache in the slot layout [slot, K|V, kv_head, block, D]
    (stride triple (2*Hkv*bs*D, D, bs*D)) gives the identical result."""
    w = _small(28, lens=(13, 6))
    base = _run(orc, w)
    nb, bs, Hkv, D = w.k_pool.shape
    slab = np.empty((nb, 2, Hkv, bs, D), dtype=np.uint16)
    slab[:, 0] = w.k_pool.transpose(0, 2, 1, 3)
    slab[:, 1] = w.v_pool.transpose(0, 2, 1, 3)
    flat = slab.ravel()
    strides = (2 * Hkv * bs * D, D, bs * D)
    k_view = flat
    v_view = flat[Hkv * bs * D:]
    out = orc.decode(w.q, k_view, np.concatenate([v_view, np.zeros(Hkv * bs * D, np.uint16)]),
                     w.block_table, w.seq_lens, Hq=w.Hq, Hkv=w.Hkv, D=w.D,
                     block_size=w.block_size, strides=strides)
    assert np.array_equal(out, base)


# --------------------------------------------------------------------------- multi-query (causal)

def _multi(seed, q_len, B=2, Hq=4, Hkv=2, D=8, bs=4, lens=(9, 14)):
    w = _small(seed, B=B, Hq=Hq, Hkv=Hkv, D=D, bs=bs, lens=lens)
    rng = np.random.default_rng(seed)
    q = bf16_bits(rng.standard_normal((B, q_len, Hq, D)).astype(np.float32))
    return w, q


def _run_multi(orc, w, q, q_len, **kw):
    return orc.decode_multi(q, w.k_pool, w.v_pool, w.block_table, w.seq_lens, q_len=q_len,
                            Hq=w.Hq, Hkv=w.Hkv, D=w.D, block_size=w.block_size, **kw)


def pin_multi_worked_example(orc):
    with open(GOLDEN) as f:
        data = json.load(f)
    for ex in data["multi_query_examples"]:
        scale = math.log(3.0) if ex["scale"] == "ln3" else float(ex["scale"])
        out = orc.decode_multi(_bits(ex["q"]), _bits(ex["k_pool"]), _bits(ex["v_pool"]),
                               np.asarray(ex["block_table"], np.int32),
                               np.asarray(ex["seq_lens"], np.int32), q_len=ex["q_len"],
                               Hq=ex["Hq"], Hkv=ex["Hkv"], D=ex["D"], block_size=ex["block_size"],
                               scale=scale)
        np.testing.assert_allclose(out, np.asarray(ex["expected"]), rtol=0, atol=1e-13,
                                   err_msg=ex["name"])


def pin_multi_sdpa_causal(orc):
    """fp64 SDPA with an explicit end-aligned causal mask on a gathered copy."""
    import torch
    import torch.nn.functional as F
    for seed, (q_len, Hq, Hkv, bs, lens) in enumerate([(3, 4, 2, 4, (7, 13)), (5, 8, 1, 2, (5, 9)),
                                                       (2, 6, 3, 16, (40, 2))]):
        w, q = _multi(300 + seed, q_len, Hq=Hq, Hkv=Hkv, D=16, bs=bs, lens=lens)
        out = _run_multi(orc, w, q, q_len)
        for b in range(w.B):
            k, v = _dense_kv(w, b)
            L = int(w.seq_lens[b])
            qq = torch.from_numpy(bf16_to_f32(q[b]).astype(np.float64)).permute(1, 0, 2)[None]
            kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(w.G, dim=0)[None]
            vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(w.G, dim=0)[None]
            pos = L - q_len + np.arange(q_len)
            mask = torch.from_numpy(np.arange(L)[None, :] <= pos[:, None])
            ref = F.scaled_dot_product_attention(qq, kt, vt, attn_mask=mask,
                                                 scale=1.0 / math.sqrt(w.D))
            np.testing.assert_allclose(out[b], ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def pin_multi_brute_force(orc):
    w, q = _multi(310, 3, Hq=4, Hkv=2, D=6, bs=3, lens=(8, 2))
    ref = brute.decode_multi(q.tolist(), w.k_pool.ravel().tolist(), w.v_pool.ravel().tolist(),
                             w.block_table.tolist(), w.seq_lens.tolist(), q_len=3, Hq=w.Hq,
                             Hkv=w.Hkv, D=w.D, block_size=w.block_size)
    np.testing.assert_allclose(_run_multi(orc, w, q, 3), np.asarray(ref), rtol=0, atol=1e-12)


def pin_multi_single_query_is_decode(orc):
    w, q = _multi(320, 1, lens=(11, 5))
    out = _run_multi(orc, w, q, 1)
    w.q = q[:, 0]
    assert np.array_equal(out[:, 0], _run(orc, w))


PINS: Dict[str, Callable] = {name: fn for name, fn in globals().items() if name.startswith("pin_")}


def failing_pins(orc) -> List[str]:
    """Names of the pins the given oracle fails (an exception counts as a failure)."""
    bad = []
    for name, fn in PINS.items():
        try:
            fn(orc)
        except Exception:  # noqa: BLE001 - any failure of a pin counts
            bad.append(name)
    return bad
