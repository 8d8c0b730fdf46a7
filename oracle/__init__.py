"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle for paged GQA decode attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it, and
it shares no code with the CUDA path: the two meet only at the seeded inputs.

``pda_oracle.c`` holds the plain definition (see its header for the passages
it follows); ``brute.py`` is a second, independent pure-Python formulation used
to pin the C code on tiny inputs.  Every function of the oracle is pinned by
``tests/test_oracle_pins.py`` (closed forms, invariants, a library routine,
brute force and hand-worked examples) and by ``tests/test_oracle_mutants.py``,
which checks that planted mistakes fail at least one pin.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pda_oracle.c")
LIBPATH = os.path.join(_HERE, "libpda_oracle.so")

_OK = 0
_ERRORS = {1: "bad argument", 2: "block id out of range", 3: "bad seq_len", 4: "out of memory"}


def build(source: str = SOURCE, libpath: str = LIBPATH, extra_flags: Sequence[str] = ()) -> str:
    """Compiles the oracle with gcc (plain C, -O2, no fast-math) into ``libpath``."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-I", os.path.dirname(os.path.abspath(source)), *extra_flags,
           source, "-o", libpath, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    return libpath


def _needs_build(libpath: str) -> bool:
    if not os.path.exists(libpath):
        return True
    return os.path.getmtime(libpath) < max(os.path.getmtime(SOURCE),
                                           os.path.getmtime(os.path.join(_HERE, "pda_oracle.h")))


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, libpath: str = LIBPATH):
        self.libpath = libpath
        lib = ctypes.CDLL(libpath)
        p = ctypes.c_void_p
        i32, i64 = ctypes.c_int32, ctypes.c_int64
        lib.pdo_decode.restype = ctypes.c_int
        lib.pdo_decode.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i64, i32,
                                   i64, i64, i64, ctypes.c_double, p, i64, i32, p]
        lib.pdo_decode_multi.restype = ctypes.c_int
        lib.pdo_decode_multi.argtypes = [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i64, i32,
                                         i64, i64, i64, ctypes.c_double, i32, p]
        lib.pdo_gather.restype = ctypes.c_int
        lib.pdo_gather.argtypes = [p, p, p, p, i32, i32, i32, i32, i64, i32,
                                   i64, i64, i64, i32, i32, p, p]
        lib.pdo_bf16_to_double.restype = ctypes.c_double
        lib.pdo_bf16_to_double.argtypes = [ctypes.c_uint16]
        self.lib = lib

    @staticmethod
    def _ptr(a: np.ndarray) -> int:
        return a.ctypes.data

    def bf16_to_double(self, bits: int) -> float:
        return self.lib.pdo_bf16_to_double(bits)

    def decode(self, q, k_pool, v_pool, block_table, seq_lens, *, Hq: int, Hkv: int, D: int,
               block_size: int, scale: Optional[float] = None,
               strides: Optional[Sequence[int]] = None,
               pairs: Optional[np.ndarray] = None, n_threads: int = 1) -> np.ndarray:
        """fp64 outputs: [B, Hq, D], or [len(pairs), D] when (b, h) pairs are given.

        ``q`` is [B, Hq, D] and the pools are flat or shaped uint16 bf16 bits; the
        pools' element strides default to the layout [blocks, block_size, Hkv, D].
        """
        q = np.ascontiguousarray(q, dtype=np.uint16)
        k_pool = np.ascontiguousarray(k_pool, dtype=np.uint16)
        v_pool = np.ascontiguousarray(v_pool, dtype=np.uint16)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B = seq_lens.shape[0]
        max_blocks = block_table.shape[1] if block_table.ndim == 2 else 0
        if strides is None:
            strides = (block_size * Hkv * D, Hkv * D, D)
        blk_s, tok_s, kvh_s = (int(x) for x in strides)
        num_blocks = k_pool.size // blk_s if blk_s > 0 else 0
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        if pairs is not None:
            pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
            out = np.zeros((pairs.shape[0], D), dtype=np.float64)
            pp, npairs = self._ptr(pairs), pairs.shape[0]
        else:
            out = np.zeros((B, Hq, D), dtype=np.float64)
            pp, npairs = None, 0
        st = self.lib.pdo_decode(self._ptr(q), self._ptr(k_pool), self._ptr(v_pool),
                                 self._ptr(block_table), self._ptr(seq_lens),
                                 B, Hq, Hkv, D, block_size, num_blocks, max_blocks,
                                 blk_s, tok_s, kvh_s, float(scale), pp, npairs,
                                 int(max(1, n_threads)), self._ptr(out))
        if st != _OK:
            raise ValueError(f"oracle decode failed: {_ERRORS.get(st, st)}")
        return out

    def decode_multi(self, q, k_pool, v_pool, block_table, seq_lens, *, q_len: int, Hq: int,
                     Hkv: int, D: int, block_size: int, scale: Optional[float] = None,
                     strides: Optional[Sequence[int]] = None, n_threads: int = 1) -> np.ndarray:
        """Causal multi-query outputs [B, q_len, Hq, D] (q is [B, q_len, Hq, D])."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        k_pool = np.ascontiguousarray(k_pool, dtype=np.uint16)
        v_pool = np.ascontiguousarray(v_pool, dtype=np.uint16)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B = seq_lens.shape[0]
        if strides is None:
            strides = (block_size * Hkv * D, Hkv * D, D)
        blk_s, tok_s, kvh_s = (int(x) for x in strides)
        if scale is None:
            scale = 1.0 / np.sqrt(D)
        out = np.zeros((B, q_len, Hq, D), dtype=np.float64)
        st = self.lib.pdo_decode_multi(self._ptr(q), self._ptr(k_pool), self._ptr(v_pool),
                                       self._ptr(block_table), self._ptr(seq_lens), B, q_len, Hq,
                                       Hkv, D, block_size, k_pool.size // blk_s,
                                       block_table.shape[1], blk_s, tok_s, kvh_s, float(scale),
                                       int(max(1, n_threads)), self._ptr(out))
        if st != _OK:
            raise ValueError(f"oracle multi-query decode failed: {_ERRORS.get(st, st)}")
        return out

    def gather(self, k_pool, v_pool, block_table, seq_lens, *, Hkv: int, D: int,
               block_size: int, b: int, kvh: int,
               strides: Optional[Sequence[int]] = None):
        """The gathered K and V rows (uint16 bf16 bits, [seq_lens[b], D] each)."""
        k_pool = np.ascontiguousarray(k_pool, dtype=np.uint16)
        v_pool = np.ascontiguousarray(v_pool, dtype=np.uint16)
        block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
        if strides is None:
            strides = (block_size * Hkv * D, Hkv * D, D)
        blk_s, tok_s, kvh_s = (int(x) for x in strides)
        n = int(seq_lens[b])
        k_rows = np.zeros((max(n, 0), D), dtype=np.uint16)
        v_rows = np.zeros((max(n, 0), D), dtype=np.uint16)
        st = self.lib.pdo_gather(self._ptr(k_pool), self._ptr(v_pool), self._ptr(block_table),
                                 self._ptr(seq_lens), seq_lens.shape[0], Hkv, D, block_size,
                                 k_pool.size // blk_s, block_table.shape[1], blk_s, tok_s,
                                 kvh_s, b, kvh, self._ptr(k_rows), self._ptr(v_rows))
        if st != _OK:
            raise ValueError(f"oracle gather failed: {_ERRORS.get(st, st)}")
        return k_rows, v_rows


_DEFAULT: Optional[Oracle] = None


def load(rebuild: bool = False) -> Oracle:
    """The oracle built from ``pda_oracle.c`` (compiled on first use)."""
    global _DEFAULT
    if rebuild or _needs_build(LIBPATH):
        build()
        _DEFAULT = None
    if _DEFAULT is None:
        _DEFAULT = Oracle(LIBPATH)
    return _DEFAULT


def host_threads() -> int:
    """Threads the oracle may use: the cores this process is allowed to run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
