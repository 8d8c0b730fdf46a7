"""Paged grouped-query decode attention for GB300 (sm_103a).

A thin ctypes binding of ``libpda.so`` (C ABI in ``include/pda.h``).  Every
step of the computation runs in the library's CUDA kernels; this module only
checks tensor shapes/dtypes and passes pointers, sizes and the current torch
stream.  PyTorch supplies device memory and streams.  There is no CPU
fallback: if the library is missing, every call raises ``RuntimeError``.

Typical use::

    import paged_gqa_decode_05_gb300 as pda
    ctx = pda.Context(max_seqs=32, num_q_heads=32, num_kv_heads=8, head_dim=128,
                      block_size=16)
    out = ctx.decode(q, k_pool, v_pool, block_table, seq_lens)   # bf16 [B, Hq, D]

Tiled lifecycle (tiled_attention.rs: begin_step / step_tile / finalize)::

    ctx.begin_step(B)
    for tile_blocks, counts, last_valid in tiles:
        ctx.step_tile(q, k_pool, v_pool, tile_blocks, counts, last_valid)
    out = ctx.finalize(B)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

__all__ = ["Context", "PdaError", "lib", "library_path", "check_dims", "paged_strides",
           "slot_strides", "plan_units", "gather_states", "DEVERR_BAD_BLOCK_ID",
           "DEVERR_BAD_LENGTH", "DEVERR_TIMEOUT"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBPATH = os.path.join(_HERE, "libpda.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_NO_DEVICE, ERR_DEVICE_DATA = range(6)
DEVERR_BAD_BLOCK_ID, DEVERR_BAD_LENGTH, DEVERR_TIMEOUT = 0x1, 0x2, 0x4


class PdaError(RuntimeError):
    """A libpda call returned a non-zero status."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


class Dims(ctypes.Structure):
    _fields_ = [("max_seqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("tile_capacity", ctypes.c_int32)]


class LaunchInfo(ctypes.Structure):
    _fields_ = [("split_ctas", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("stage_tokens", ctypes.c_int32),
                ("partial_slots", ctypes.c_int64), ("unit_cost", ctypes.c_int32)]


class MultiInfo(ctypes.Structure):
    _fields_ = [("form", ctypes.c_int32), ("queries_per_walk", ctypes.c_int32),
                ("rows_per_walk", ctypes.c_int32), ("walks_per_seq", ctypes.c_int32),
                ("split_ctas", ctypes.c_int32), ("stages", ctypes.c_int32)]


_LIB: Optional[ctypes.CDLL] = None
ABI_VERSION = 5  # PDA_ABI_VERSION of include/pda.h that these signatures follow


def library_path() -> str:
    return _LIBPATH


def lib() -> ctypes.CDLL:
    """The loaded libpda.so (raises RuntimeError if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(_LIBPATH):
        raise RuntimeError(f"{_LIBPATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(_LIBPATH)
    P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    sig = {
        "pda_abi_version": (I32, []),
        "pda_status_string": (ctypes.c_char_p, [I32]),
        "pda_last_error": (ctypes.c_char_p, []),
        "pda_check_dims": (I32, [ctypes.POINTER(Dims)]),
        "pda_paged_strides": (I32, [ctypes.POINTER(Dims), ctypes.POINTER(I64)]),
        "pda_slot_strides": (I32, [ctypes.POINTER(Dims), ctypes.POINTER(I64)]),
        "pda_create": (I32, [ctypes.POINTER(Dims), ctypes.POINTER(P)]),
        "pda_destroy": (None, [P]),
        "pda_decode": (I32, [P, P, P, P, I64, P, I32, P, I32, F, P, P]),
        "pda_decode_strided": (I32, [P, P, P, P, I64, I64, I64, I64, P, I32, P, I32, F, P, P]),
        "pda_decode_f32": (I32, [P, P, P, P, I64, I64, I64, I64, P, I32, P, I32, F, P, P]),
        "pda_decode_contiguous": (I32, [P, P, P, P, I32, P, I32, F, P, P]),
        "pda_decode_multi": (I32, [P, P, P, P, I64, P, I32, P, I32, I32, F, P, P]),
        "pda_begin_step": (I32, [P, I32, P]),
        "pda_step_tile": (I32, [P, P, P, P, I64, P, P, P, I32, I64, I64, I64, F, P]),
        "pda_finalize": (I32, [P, P, I32, P]),
        "pda_finalize_f32": (I32, [P, P, I32, P]),
        "pda_export_state": (I32, [P, I32, P, P, P, P]),
        "pda_merge_states": (I32, [P, I32, I32, P, P, P, P, P]),
        "pda_merge_states_f32": (I32, [P, I32, I32, P, P, P, P, P]),
        "pda_debug_gather": (I32, [P, P, P, I64, I64, I64, I64, P, I32, P, I32, P, P, P]),
        "pda_read_device_errors": (I32, [P, ctypes.POINTER(ctypes.c_uint32), I32, P]),
        "pda_set_timing_events": (I32, [P, P, P, P]),
        "pda_check_wait_timeout": (I32, [P, I64, P]),
        "pda_get_launch_info": (I32, [P, ctypes.POINTER(LaunchInfo)]),
        "pda_get_multi_info": (I32, [P, I32, ctypes.POINTER(MultiInfo)]),
        "pda_set_tile_overlap": (I32, [P, I32]),
        "pda_set_multi_tc": (I32, [P, I32]),
        "pda_plan_units": (I32, [P, I32, I32, I32, I32, I32, I32, I32, P, P, ctypes.POINTER(I64)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    if L.pda_abi_version() != ABI_VERSION:
        raise RuntimeError(f"{_LIBPATH} has ABI version {L.pda_abi_version()}, this binding "
                           f"expects {ABI_VERSION}: rebuild it")
    _LIB = L
    return L


def _check(status: int) -> None:
    if status != OK:
        L = lib()
        raise PdaError(status, f"{L.pda_status_string(status).decode()}: "
                               f"{L.pda_last_error().decode()}")


def _dims(max_seqs, num_q_heads, num_kv_heads, head_dim, block_size, tile_capacity) -> Dims:
    return Dims(int(max_seqs), int(num_q_heads), int(num_kv_heads), int(head_dim),
                int(block_size), int(tile_capacity))


def check_dims(**kw) -> int:
    """Status of pda_check_dims for the given dims (host only, no GPU)."""
    d = _dims(kw.get("max_seqs", 1), kw["num_q_heads"], kw["num_kv_heads"], kw["head_dim"],
              kw["block_size"], kw.get("tile_capacity", 1))
    return lib().pda_check_dims(ctypes.byref(d))


def _strides(fn, **kw) -> Tuple[int, int, int]:
    d = _dims(1, kw["num_q_heads"], kw["num_kv_heads"], kw["head_dim"], kw["block_size"], 1)
    out = (ctypes.c_int64 * 3)()
    _check(fn(ctypes.byref(d), out))
    return int(out[0]), int(out[1]), int(out[2])


def paged_strides(**kw) -> Tuple[int, int, int]:
    """(block, token, kv-head) element strides of [num_blocks, bs, Hkv, D]."""
    return _strides(lib().pda_paged_strides, **kw)


def slot_strides(**kw) -> Tuple[int, int, int]:
    """(block, token, kv-head) element strides of the slot layout [slot, K|V, Hkv, bs, D]."""
    return _strides(lib().pda_slot_strides, **kw)


def plan_units(lens: Sequence[int], *, block_size: int, num_kv_heads: int, split_ctas: int,
               blocks_given: bool = False, unit_cost: int = 0, stage_tokens: int = 0):
    """(first_cta, last_cta, total_blocks) of the split plan (host only); a
    context's unit_cost and stage_tokens are in its launch_info() (stage_tokens
    0: the even split for every batch, without the small-batch unit plan)."""
    import numpy as np
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    n = lens.shape[0] * num_kv_heads
    first = np.zeros(max(n, 1), dtype=np.int32)
    last = np.zeros(max(n, 1), dtype=np.int32)
    total = ctypes.c_int64()
    _check(lib().pda_plan_units(lens.ctypes.data, lens.shape[0], int(blocks_given), block_size,
                                num_kv_heads, split_ctas, unit_cost, stage_tokens, first.ctypes.data,
                                last.ctypes.data, ctypes.byref(total)))
    return first[:n], last[:n], int(total.value)


def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Context:
    """Owns the running (m, l, o) state and split workspace on one device
    (tiled_attention.rs: TiledAttention)."""

    def __init__(self, max_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 block_size: int, tile_capacity: int = 64, device=None):
        torch = _torch()
        self.dims = _dims(max_seqs, num_q_heads, num_kv_heads, head_dim, block_size, tile_capacity)
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None
                                   else torch.device(device).index or 0)
        self._ctx = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(lib().pda_create(ctypes.byref(self.dims), ctypes.byref(self._ctx)))
        self.G = num_q_heads // num_kv_heads

    # -- properties
    @property
    def num_q_heads(self) -> int:
        return self.dims.num_q_heads

    @property
    def num_kv_heads(self) -> int:
        return self.dims.num_kv_heads

    @property
    def head_dim(self) -> int:
        return self.dims.head_dim

    @property
    def block_size(self) -> int:
        return self.dims.block_size

    def close(self) -> None:
        if self._ctx:
            lib().pda_destroy(self._ctx)
            self._ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass

    def launch_info(self) -> dict:
        info = LaunchInfo()
        _check(lib().pda_get_launch_info(self._ctx, ctypes.byref(info)))
        return {f: getattr(info, f) for f, _ in LaunchInfo._fields_}

    def multi_info(self, q_len: int) -> dict:
        """The launch decode_multi makes for q_len queries per sequence (pda_get_multi_info);
        form 0: n8, 1: row form on mma.sync, 2: row form on tcgen05."""
        info = MultiInfo()
        _check(lib().pda_get_multi_info(self._ctx, int(q_len), ctypes.byref(info)))
        return {f: getattr(info, f) for f, _ in MultiInfo._fields_}

    def set_multi_tc(self, enable: bool) -> None:
        """decode_multi takes the tcgen05 row form where it applies, or the mma.sync row form
        (the default) (pda_set_multi_tc)."""
        _check(lib().pda_set_multi_tc(self._ctx, int(bool(enable))))

    # -- argument checks (marshalling only)
    def _bf16(self, t, name, shape=None):
        torch = _torch()
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")
        if shape is not None and tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
        return t

    def _i32(self, t, name, ndim):
        torch = _torch()
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() or t.dim() != ndim:
            raise ValueError(f"{name} must be a contiguous {ndim}-D int32 CUDA tensor")
        return t

    def _pool(self, k_pool, v_pool, strides, num_blocks):
        d = self.dims
        if strides is None:
            shape = (k_pool.shape[0], d.block_size, d.num_kv_heads, d.head_dim)
            self._bf16(k_pool, "k_pool", shape)
            self._bf16(v_pool, "v_pool", shape)
            strides = paged_strides(num_q_heads=d.num_q_heads, num_kv_heads=d.num_kv_heads,
                                    head_dim=d.head_dim, block_size=d.block_size)
            num_blocks = k_pool.shape[0]
        else:
            if k_pool.dtype != _torch().bfloat16 or v_pool.dtype != _torch().bfloat16:
                raise ValueError("k_pool / v_pool must be bfloat16")
            if num_blocks is None:
                raise ValueError("num_blocks is required with explicit strides")
        return tuple(int(s) for s in strides), int(num_blocks)

    def _scale(self, scale) -> float:
        return float("nan") if scale is None else float(scale)

    # -- one-shot decode
    def decode(self, q, k_pool, v_pool, block_table, seq_lens, scale: Optional[float] = None,
               out=None, strides: Optional[Sequence[int]] = None, num_blocks: Optional[int] = None,
               stream=None, out_dtype=None):
        """softmax(scale * q K^T) V over each sequence's paged KV -> [B, Hq, D].

        ``out_dtype=torch.float32`` returns the fp32 quotient o / l (no bf16 rounding).
        """
        torch = _torch()
        d = self.dims
        B = int(seq_lens.shape[0])
        self._bf16(q, "q", (B, d.num_q_heads, d.head_dim))
        self._i32(block_table, "block_table", 2)
        self._i32(seq_lens, "seq_lens", 1)
        if block_table.shape[0] != B:
            raise ValueError("block_table must have one row per sequence")
        (bs_, ts_, hs_), nblk = self._pool(k_pool, v_pool, strides, num_blocks)
        f32 = out_dtype == torch.float32
        if out is None:
            out = torch.empty((B, d.num_q_heads, d.head_dim), device=q.device,
                              dtype=torch.float32 if f32 else torch.bfloat16)
        L = lib()
        if f32:
            _check(L.pda_decode_f32(self._ctx, _ptr(q), _ptr(k_pool), _ptr(v_pool), nblk, bs_, ts_,
                                    hs_, _ptr(block_table), int(block_table.shape[1]),
                                    _ptr(seq_lens), B, self._scale(scale), _ptr(out),
                                    _stream(stream)))
        else:
            self._bf16(out, "out", (B, d.num_q_heads, d.head_dim))
            _check(L.pda_decode_strided(self._ctx, _ptr(q), _ptr(k_pool), _ptr(v_pool), nblk, bs_,
                                        ts_, hs_, _ptr(block_table), int(block_table.shape[1]),
                                        _ptr(seq_lens), B, self._scale(scale), _ptr(out),
                                        _stream(stream)))
        return out

    def bind_decode(self, q, k_pool, v_pool, block_table, seq_lens, out,
                    scale: Optional[float] = None, strides: Optional[Sequence[int]] = None,
                    num_blocks: Optional[int] = None, stream=None):
        """Validates one decode's tensors once and returns a zero-argument callable
        that reruns it (the same buffers, their contents free to change between
        calls) with only the C call: for decode loops over persistent buffers
        that do not use CUDA graphs.  The callable keeps the tensors and this
        context alive, launches on the stream current at binding (or `stream`),
        and raises once the context is closed."""
        d = self.dims
        B = int(seq_lens.shape[0])
        self._bf16(q, "q", (B, d.num_q_heads, d.head_dim))
        self._i32(block_table, "block_table", 2)
        self._i32(seq_lens, "seq_lens", 1)
        if block_table.shape[0] != B:
            raise ValueError("block_table must have one row per sequence")
        self._bf16(out, "out", (B, d.num_q_heads, d.head_dim))
        (bs_, ts_, hs_), nblk = self._pool(k_pool, v_pool, strides, num_blocks)
        args = (_ptr(q), _ptr(k_pool), _ptr(v_pool), nblk, bs_, ts_, hs_, _ptr(block_table),
                int(block_table.shape[1]), _ptr(seq_lens), B, self._scale(scale), _ptr(out),
                _stream(stream))
        return _Bound(self, lib().pda_decode_strided, args,
                      (q, k_pool, v_pool, block_table, seq_lens, out))

    def decode_multi(self, q, k_pool, v_pool, block_table, seq_lens, scale: Optional[float] = None,
                     out=None, stream=None):
        """Causal multi-query decode: q [B, q_len, Hq, D] are each sequence's last q_len
        tokens; query i sees tokens up to seq_lens[b] - q_len + i.  Returns [B, q_len, Hq, D]."""
        torch = _torch()
        d = self.dims
        B = int(seq_lens.shape[0])
        if q.dim() != 4 or q.shape[0] != B or q.shape[2:] != (d.num_q_heads, d.head_dim):
            raise ValueError("q must be [B, q_len, Hq, D]")
        self._bf16(q, "q")
        self._i32(block_table, "block_table", 2)
        self._i32(seq_lens, "seq_lens", 1)
        (bs_, ts_, hs_), nblk = self._pool(k_pool, v_pool, None, None)
        if out is None:
            out = torch.empty_like(q)
        self._bf16(out, "out", tuple(q.shape))
        _check(lib().pda_decode_multi(self._ctx, _ptr(q), _ptr(k_pool), _ptr(v_pool), nblk,
                                      _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
                                      B, int(q.shape[1]), self._scale(scale), _ptr(out),
                                      _stream(stream)))
        return out

    def decode_contiguous(self, q, k, v, seq_lens, scale: Optional[float] = None, out=None,
                          stream=None):
        """Decode over a contiguous cache k, v [B, S, Hkv, D] (S a multiple of block_size)."""
        torch = _torch()
        d = self.dims
        B = int(seq_lens.shape[0])
        self._bf16(q, "q", (B, d.num_q_heads, d.head_dim))
        self._i32(seq_lens, "seq_lens", 1)
        if k.dim() != 4 or k.shape[0] != B or k.shape[2:] != (d.num_kv_heads, d.head_dim):
            raise ValueError("k must be [B, S, Hkv, D]")
        self._bf16(k, "k")
        self._bf16(v, "v", tuple(k.shape))
        if out is None:
            out = torch.empty((B, d.num_q_heads, d.head_dim), device=q.device, dtype=torch.bfloat16)
        self._bf16(out, "out", (B, d.num_q_heads, d.head_dim))
        _check(lib().pda_decode_contiguous(self._ctx, _ptr(q), _ptr(k), _ptr(v), int(k.shape[1]),
                                           _ptr(seq_lens), B, self._scale(scale), _ptr(out),
                                           _stream(stream)))
        return out

    # -- tiled lifecycle
    def set_tile_overlap(self, enable: bool) -> None:
        """Tile steps of one step on one stream overlap (default) or each waits (pda_set_tile_overlap)."""
        _check(lib().pda_set_tile_overlap(self._ctx, int(bool(enable))))

    def begin_step(self, num_seqs: int, stream=None) -> None:
        _check(lib().pda_begin_step(self._ctx, int(num_seqs), _stream(stream)))

    def step_tile(self, q, k_pool, v_pool, tile_blocks, tile_block_counts, tile_last_valid=None,
                  scale: Optional[float] = None, strides: Optional[Sequence[int]] = None,
                  num_blocks: Optional[int] = None, stream=None) -> None:
        d = self.dims
        S = int(tile_block_counts.shape[0])
        self._bf16(q, "q")
        if q.dim() != 3 or q.shape[0] < S or q.shape[1:] != (d.num_q_heads, d.head_dim):
            raise ValueError("q must be [>=num_seqs, Hq, D]")
        self._i32(tile_blocks, "tile_blocks", 2)
        self._i32(tile_block_counts, "tile_block_counts", 1)
        if tile_blocks.shape[0] < S or tile_blocks.shape[1] != d.tile_capacity:
            raise ValueError(f"tile_blocks must be [num_seqs, tile_capacity={d.tile_capacity}]")
        if tile_last_valid is not None:
            self._i32(tile_last_valid, "tile_last_valid", 1)
        (bs_, ts_, hs_), nblk = self._pool(k_pool, v_pool, strides, num_blocks)
        _check(lib().pda_step_tile(self._ctx, _ptr(q), _ptr(k_pool), _ptr(v_pool), nblk,
                                   _ptr(tile_blocks), _ptr(tile_block_counts), _ptr(tile_last_valid),
                                   S, bs_, ts_, hs_, self._scale(scale), _stream(stream)))

    def finalize(self, num_seqs: int, out=None, out_dtype=None, stream=None):
        torch = _torch()
        d = self.dims
        f32 = out_dtype == torch.float32
        if out is None:
            out = torch.empty((num_seqs, d.num_q_heads, d.head_dim), device=self.device,
                              dtype=torch.float32 if f32 else torch.bfloat16)
        fn = lib().pda_finalize_f32 if f32 else lib().pda_finalize
        _check(fn(self._ctx, _ptr(out), int(num_seqs), _stream(stream)))
        return out

    # -- partial states across contexts (context-parallel decode)
    def export_state(self, num_seqs: int, stream=None):
        """The running (m, l, o) of sequences [0, num_seqs) as fp32 tensors
        [num_seqs, Hq], [num_seqs, Hq], [num_seqs, Hq, D]: m the reference (natural-log
        units of the scaled scores; the running max or up to 8 ln 2 below it),
        l = sum exp(s - m), o = sum exp(s - m) v."""
        torch = _torch()
        d = self.dims
        m = torch.empty((num_seqs, d.num_q_heads), device=self.device, dtype=torch.float32)
        l = torch.empty_like(m)
        o = torch.empty((num_seqs, d.num_q_heads, d.head_dim), device=self.device,
                        dtype=torch.float32)
        _check(lib().pda_export_state(self._ctx, int(num_seqs), _ptr(m), _ptr(l), _ptr(o),
                                      _stream(stream)))
        return m, l, o

    def merge_states(self, m_parts, l_parts, o_parts, out=None, out_dtype=None, stream=None):
        """o / l of P exported states per (sequence, q head): m_parts, l_parts
        [P, S, Hq], o_parts [P, S, Hq, D] (fp32, CUDA) -> [S, Hq, D]."""
        torch = _torch()
        d = self.dims
        P_, S = int(m_parts.shape[0]), int(m_parts.shape[1])
        for t, name, shape in ((m_parts, "m_parts", (P_, S, d.num_q_heads)),
                               (l_parts, "l_parts", (P_, S, d.num_q_heads)),
                               (o_parts, "o_parts", (P_, S, d.num_q_heads, d.head_dim))):
            if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous() or \
                    tuple(t.shape) != shape:
                raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape {shape}")
        f32 = out_dtype == torch.float32
        if out is None:
            out = torch.empty((S, d.num_q_heads, d.head_dim), device=self.device,
                              dtype=torch.float32 if f32 else torch.bfloat16)
        fn = lib().pda_merge_states_f32 if f32 else lib().pda_merge_states
        _check(fn(self._ctx, P_, S, _ptr(m_parts), _ptr(l_parts), _ptr(o_parts), _ptr(out),
                  _stream(stream)))
        return out

    # -- checks and hooks
    def debug_gather(self, k_pool, v_pool, block_table, seq_lens, strides=None, num_blocks=None,
                     stream=None):
        """The K/V rows the decode kernel's loader staged, [B, Hkv, max_blocks*bs, D] each."""
        torch = _torch()
        d = self.dims
        B = int(seq_lens.shape[0])
        self._i32(block_table, "block_table", 2)
        self._i32(seq_lens, "seq_lens", 1)
        (bs_, ts_, hs_), nblk = self._pool(k_pool, v_pool, strides, num_blocks)
        rows = int(block_table.shape[1]) * d.block_size
        k_rows = torch.zeros((B, d.num_kv_heads, rows, d.head_dim), device=self.device,
                             dtype=torch.bfloat16)
        v_rows = torch.zeros_like(k_rows)
        _check(lib().pda_debug_gather(self._ctx, _ptr(k_pool), _ptr(v_pool), nblk, bs_, ts_, hs_,
                                      _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
                                      B, _ptr(k_rows), _ptr(v_rows), _stream(stream)))
        return k_rows, v_rows

    def read_device_errors(self, clear: bool = True, stream=None) -> int:
        """PDA_DEVERR_* flags raised by kernels since the last clear (synchronises)."""
        flags = ctypes.c_uint32()
        st = lib().pda_read_device_errors(self._ctx, ctypes.byref(flags), int(clear),
                                          _stream(stream))
        if st not in (OK, ERR_DEVICE_DATA):
            _check(st)
        return int(flags.value)

    def check_wait_timeout(self, limit_ns: int = 20_000_000, stream=None) -> int:
        """Runs a bounded wait that cannot complete; returns the device flags after it."""
        _check(lib().pda_check_wait_timeout(self._ctx, int(limit_ns), _stream(stream)))
        return self.read_device_errors(stream=stream)

    def set_timing_events(self, ev_begin=None, ev_split=None, ev_end=None) -> None:
        h = [None if e is None else e.cuda_event for e in (ev_begin, ev_split, ev_end)]
        _check(lib().pda_set_timing_events(self._ctx, *h))


class _Bound:
    """A decode with its arguments marshalled once (Context.bind_decode)."""

    __slots__ = ("_owner", "_fn", "_args", "_keep")

    def __init__(self, owner, fn, args, keep):
        self._owner, self._fn, self._args, self._keep = owner, fn, args, keep

    def __call__(self) -> None:
        ctx = self._owner._ctx
        if not ctx:
            raise PdaError(ERR_INVALID_ARG, "the context of this bound decode is closed")
        _check(self._fn(ctx, *self._args))


def gather_states(m, l, o, group=None):
    """All-gathers one exported state (m, l, o) per rank over a torch.distributed
    process group into part-major stacks [world, ...] (rank order), ready for
    Context.merge_states.  Tensors stay on their device (NCCL for CUDA tensors)."""
    torch = _torch()
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = []
    for t in (m, l, o):
        t = t.contiguous()
        parts = [torch.empty_like(t) for _ in range(world)]
        dist.all_gather(parts, t, group=group)
        out.append(torch.stack(parts))
    return tuple(out)

