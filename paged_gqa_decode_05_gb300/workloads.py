"""Seeded synthetic inputs for paged GQA decode attention.

This module only draws inputs; it holds none of the attention arithmetic.  The
CUDA path, the CPU oracle, the tests and the benchmark all consume the same
bf16 bit patterns produced here, so both sides see identical inputs.

Recipe (every workload):
  * one ``numpy.random.Generator(PCG64)`` per stream, spawned from
    ``SeedSequence(seed)``: q, K, V, lengths, table, spike positions;
  * q, K and V drawn N(0, 1) in float32 and rounded to bf16 (round to nearest,
    ties to even) -- the pools are filled completely, unused blocks included;
  * the block table maps each sequence's logical blocks to distinct pool
    blocks chosen by a seeded permutation; table entries past a sequence's
    last block hold valid but unrelated block ids, so an over-read would
    return wrong data rather than fault;
  * optional "spikes": K rows of a seeded fraction of (sequence, token)
    positions are multiplied by a factor before rounding (all KV heads of the
    token), which makes the softmax peaky.

The five named workloads follow the decode shapes used to evaluate the
method: a tiny case, a 1B-style, an 8B-style, a wide-head and a ragged
long-context batch (see ``WORKLOADS``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, Dict, Optional, Sequence

import numpy as np

_CHUNK_ELEMS = 1 << 24


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Inputs are finite draws (|x| far below the float32 maximum), so the
    integer rounding below never carries into the exponent's all-ones range.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + r) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Workload:
    """One decode batch: q, the paged K/V pools, the block table and lengths."""

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    block_size: int
    q: np.ndarray            # uint16 [B, Hq, D]
    k_pool: np.ndarray       # uint16 [num_blocks, block_size, Hkv, D]
    v_pool: np.ndarray       # uint16 [num_blocks, block_size, Hkv, D]
    block_table: np.ndarray  # int32  [B, max_blocks]
    seq_lens: np.ndarray     # int32  [B]
    seed: int
    scale: float = field(default=0.0)
    notes: str = ""

    def __post_init__(self):
        if self.scale == 0.0:
            self.scale = 1.0 / math.sqrt(self.D)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def num_blocks(self) -> int:
        return int(self.k_pool.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    def blocks_per_seq(self) -> np.ndarray:
        return (self.seq_lens.astype(np.int64) + self.block_size - 1) // self.block_size

    def algorithmic_bytes(self) -> int:
        """Bytes the method must move: valid K+V rows, q in, out (bf16)."""
        kv = int(self.seq_lens.astype(np.int64).sum()) * self.Hkv * self.D * 2 * 2
        return kv + 2 * self.B * self.Hq * self.D * 2

    def describe(self) -> dict:
        return {"workload": self.name, "B": self.B, "Hq": self.Hq, "Hkv": self.Hkv,
                "D": self.D, "block_size": self.block_size, "num_blocks": self.num_blocks,
                "max_blocks": self.max_blocks, "seed": self.seed,
                "tokens": int(self.seq_lens.astype(np.int64).sum()),
                "mean_seq_len": float(self.seq_lens.mean()) if self.B else 0.0}


def _normal_bits(rng: np.random.Generator, shape, spike: Optional[np.ndarray] = None) -> np.ndarray:
    """N(0,1) float32 draws rounded to bf16, generated in chunks along axis 0.

    ``spike`` (float32, shape[:2]) multiplies whole rows before rounding.
    """
    out = np.empty(shape, dtype=np.uint16)
    if out.size == 0:
        return out
    row = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    step = max(1, _CHUNK_ELEMS // max(row, 1))
    for i in range(0, shape[0], step):
        j = min(shape[0], i + step)
        x = rng.standard_normal((j - i,) + tuple(shape[1:]), dtype=np.float32)
        if spike is not None:
            x *= spike[i:j].reshape(spike[i:j].shape + (1,) * (len(shape) - 2))
        out[i:j] = bf16_bits(x)
    return out


def make_workload(name: str, *, B: int, Hq: int, Hkv: int, D: int, block_size: int,
                  seq_lens: Sequence[int], seed: int, pool_blocks: Optional[int] = None,
                  max_blocks: Optional[int] = None, spike_frac: float = 0.0,
                  spike_factor: float = 3.0, table_perm: Optional[np.ndarray] = None,
                  notes: str = "") -> Workload:
    """Builds a workload from explicit lengths (see the module docstring)."""
    ss = np.random.SeedSequence(seed)
    r_q, r_k, r_v, r_table, r_spike, r_fill = (np.random.Generator(np.random.PCG64(s))
                                               for s in ss.spawn(6))
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    assert seq_lens.shape == (B,)
    nb = (seq_lens.astype(np.int64) + block_size - 1) // block_size
    needed = int(nb.sum())
    pool = needed if pool_blocks is None else int(pool_blocks)
    assert pool >= needed and pool >= 1
    width = max(1, int(nb.max()) if B else 1) if max_blocks is None else int(max_blocks)
    assert width >= (int(nb.max()) if B else 0)

    perm = r_table.permutation(pool).astype(np.int32) if table_perm is None else \
        np.asarray(table_perm, dtype=np.int32)
    table = r_fill.integers(0, pool, size=(B, width), dtype=np.int32)
    cursor = 0
    for b in range(B):
        table[b, :nb[b]] = perm[cursor:cursor + nb[b]]
        cursor += int(nb[b])

    spike = None
    if spike_frac > 0.0:
        spike = np.ones((pool, block_size), dtype=np.float32)
        total = int(seq_lens.astype(np.int64).sum())
        count = int(round(spike_frac * total))
        starts = np.concatenate([[0], np.cumsum(seq_lens.astype(np.int64))])
        for flat in r_spike.choice(total, size=count, replace=False):
            b = int(np.searchsorted(starts, flat, side="right") - 1)
            t = int(flat - starts[b])
            spike[table[b, t // block_size], t % block_size] = spike_factor

    q = _normal_bits(r_q, (B, Hq, D))
    k_pool = _normal_bits(r_k, (pool, block_size, Hkv, D), spike)
    v_pool = _normal_bits(r_v, (pool, block_size, Hkv, D))
    return Workload(name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, block_size=block_size, q=q,
                    k_pool=k_pool, v_pool=v_pool, block_table=table, seq_lens=seq_lens,
                    seed=seed, notes=notes)


def tiny(seed: int = 1000) -> Workload:
    """B=2, Hq=4, Hkv=2, D=64, block 16, lengths {37, 80}, pool of 16 blocks;
    the table rows take the first 3 + 5 entries of a seeded permutation of 0..15."""
    return make_workload("tiny B2 Hq4 Hkv2 D64 bs16 len{37,80}", B=2, Hq=4, Hkv=2, D=64,
                         block_size=16, seq_lens=[37, 80], seed=seed, pool_blocks=16)


def one_b(seed: int = 1001) -> Workload:
    """1B-style: B=8, Hq=32, Hkv=8, D=64, block 16, lengths U[512, 2048],
    pool twice the needed blocks, injective table."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    lens = rng.integers(512, 2048, size=8, endpoint=True)
    needed = int(((lens + 15) // 16).sum())
    return make_workload("1B-style B8 Hq32 Hkv8 D64 bs16 len U[512,2048]", B=8, Hq=32, Hkv=8,
                         D=64, block_size=16, seq_lens=lens, seed=seed, pool_blocks=2 * needed)


def eight_b(seed: int = 1002) -> Workload:
    """8B-style: B=32, Hq=32, Hkv=8, D=128, block 16, every length 4096,
    shuffled table over 8192 blocks, K x3 on a seeded 1% of tokens."""
    return make_workload("8B-style B32 Hq32 Hkv8 D128 bs16 len4096", B=32, Hq=32, Hkv=8, D=128,
                         block_size=16, seq_lens=[4096] * 32, seed=seed, spike_frac=0.01)


def wide(seed: int = 1003) -> Workload:
    """Wide head: B=16, Hq=16, Hkv=4, D=256, block 16, lengths U[1024, 8192]."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    lens = rng.integers(1024, 8192, size=16, endpoint=True)
    return make_workload("wide-head B16 Hq16 Hkv4 D256 bs16 len U[1024,8192]", B=16, Hq=16,
                         Hkv=4, D=256, block_size=16, seq_lens=lens, seed=seed)


def ragged_lengths(rng: np.random.Generator, B: int, lo: int, hi: int, block_size: int) -> np.ndarray:
    """Log-uniform lengths in [lo, hi], none a multiple of the block size."""
    lens = np.exp(rng.uniform(np.log(lo), np.log(hi), size=B)).astype(np.int64)
    lens = np.clip(lens, lo, hi)
    full = lens % block_size == 0
    lens[full & (lens > lo)] -= 1
    lens[full & (lens == lo)] += 1
    return lens


def ragged(seed: int = 1004) -> Workload:
    """Ragged long context: B=64, Hq=64, Hkv=8, D=128, block 32, lengths
    log-uniform in [128, 32768] with every last block partially filled;
    table width 1024 blocks."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    lens = ragged_lengths(rng, 64, 128, 32768, 32)
    return make_workload("ragged B64 Hq64 Hkv8 D128 bs32 len logU[128,32768]", B=64, Hq=64,
                         Hkv=8, D=128, block_size=32, seq_lens=lens, seed=seed, max_blocks=1024)


def with_block_size(w: Workload, block_size: int) -> Workload:
    """The same batch shape and lengths drawn afresh with another block size
    (the pool holds exactly the needed blocks, shuffled)."""
    return make_workload(f"{w.name} (block {block_size})", B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D,
                         block_size=block_size, seq_lens=w.seq_lens, seed=w.seed)


def multi_queries(w: Workload, q_len: int) -> np.ndarray:
    """Seeded N(0,1) bf16 queries [B, q_len, Hq, D] for a causal multi-query
    decode over the workload's cache (the cache is unchanged)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 13, q_len])))
    return _normal_bits(rng, (w.B, q_len, w.Hq, w.D))


def contiguous_kv(w: Workload, max_seq_len: Optional[int] = None):
    """The workload's cache copied to the contiguous layout [B, S, Hkv, D]
    (S = max_seq_len, default the longest sequence rounded up to a block),
    rows past a sequence's length filled with N(0,1) bf16 draws.  Returns
    (k, v) as uint16 arrays; a pure copy of the inputs."""
    bs = w.block_size
    S = max_seq_len or int(-(-int(w.seq_lens.max()) // bs) * bs) if w.B else bs
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 11])))
    k = _normal_bits(rng, (w.B, S, w.Hkv, w.D))
    v = _normal_bits(rng, (w.B, S, w.Hkv, w.D))
    for b in range(w.B):
        n = int(w.seq_lens[b])
        t = np.arange(n)
        blk = w.block_table[b, t // bs]
        k[b, :n] = w.k_pool[blk, t % bs]
        v[b, :n] = w.v_pool[blk, t % bs]
    return k, v


WORKLOADS: Dict[str, Callable[[], Workload]] = {
    "tiny": tiny,
    "1b": one_b,
    "8b": eight_b,
    "wide": wide,
    "ragged": ragged,
}
