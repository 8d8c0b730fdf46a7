"""TEST INFRASTRUCTURE ONLY: a second, pure-Python statement of the oracle.

It is written differently from ``pda_oracle.c`` on purpose, so that the two
pin each other on tiny inputs:

  * the gather walks the block table into an explicit dense list of
    (K row, V row) pairs first, then forgets the pool;
  * every sum is ``math.fsum`` (exactly rounded), not a running double sum;
  * bf16 bits are widened with ``struct`` rather than a bit cast in C;
  * the q-head -> kv-head map is written as "kv head g serves q heads
    g*G .. g*G+G-1" (a loop over groups), not as a division.

Only small cases are practical (pure-Python loops).
"""
from __future__ import annotations

import math
import struct
from typing import List, Optional, Sequence


def bf16_value(bits: int) -> float:
    """The value of a bf16 bit pattern (the upper half of a float32)."""
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def gather_rows(k_pool, v_pool, table_row: Sequence[int], n: int, kvh: int, block_size: int,
                strides: Sequence[int], D: int):
    """Dense lists of the first n K and V rows of one sequence for one kv head.

    ``k_pool`` / ``v_pool`` are flat sequences of bf16 bits; ``strides`` is the
    (block, token, kv-head) element-stride triple.
    """
    blk_s, tok_s, kvh_s = strides
    ks: List[List[float]] = []
    vs: List[List[float]] = []
    for blk_index in range(0, (n + block_size - 1) // block_size):
        blk = int(table_row[blk_index])
        first = blk_index * block_size
        for slot in range(block_size):
            if first + slot >= n:
                break
            base = blk * blk_s + slot * tok_s + kvh * kvh_s
            ks.append([bf16_value(k_pool[base + d]) for d in range(D)])
            vs.append([bf16_value(v_pool[base + d]) for d in range(D)])
    return ks, vs


def decode(q, k_pool, v_pool, block_table, seq_lens, *, Hq: int, Hkv: int, D: int,
           block_size: int, scale: Optional[float] = None,
           strides: Optional[Sequence[int]] = None) -> List[List[List[float]]]:
    """out[b][h][d] for nested-list / flat inputs (q as [B][Hq][D] bits)."""
    if strides is None:
        strides = (block_size * Hkv * D, Hkv * D, D)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    G = Hq // Hkv
    B = len(seq_lens)
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(B)]
    for b in range(B):
        n = int(seq_lens[b])
        for g in range(Hkv):
            ks, vs = gather_rows(k_pool, v_pool, block_table[b], n, g, block_size, strides, D)
            for h in range(g * G, g * G + G):
                if n == 0:
                    continue
                qv = [bf16_value(q[b][h][d]) for d in range(D)]
                scores = [scale * math.fsum(qv[d] * k[d] for d in range(D)) for k in ks]
                top = max(scores)
                w = [math.exp(s - top) for s in scores]
                z = math.fsum(w)
                for d in range(D):
                    out[b][h][d] = math.fsum(w[t] * vs[t][d] for t in range(n)) / z
    return out


def decode_multi(q, k_pool, v_pool, block_table, seq_lens, *, q_len: int, Hq: int, Hkv: int,
                 D: int, block_size: int, scale: Optional[float] = None,
                 strides: Optional[Sequence[int]] = None) -> List[List[List[List[float]]]]:
    """out[b][i][h][d] for q as [B][q_len][Hq][D] bits: query i is token
    seq_lens[b] - q_len + i and sees every token up to and including itself."""
    if strides is None:
        strides = (block_size * Hkv * D, Hkv * D, D)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    G = Hq // Hkv
    out = []
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        rows = []
        for i in range(q_len):
            visible = max(0, L - q_len + 1 + i)
            heads = []
            for g in range(Hkv):
                ks, vs = gather_rows(k_pool, v_pool, block_table[b], visible, g, block_size,
                                     strides, D)
                for h in range(g * G, g * G + G):
                    if visible == 0:
                        heads.append([0.0] * D)
                        continue
                    qv = [bf16_value(q[b][i][h][d]) for d in range(D)]
                    scores = [scale * math.fsum(qv[d] * k[d] for d in range(D)) for k in ks]
                    top = max(scores)
                    w = [math.exp(x - top) for x in scores]
                    z = math.fsum(w)
                    heads.append([math.fsum(w[t] * vs[t][d] for t in range(visible)) / z
                                  for d in range(D)])
            rows.append(heads)
        out.append(rows)
    return out
