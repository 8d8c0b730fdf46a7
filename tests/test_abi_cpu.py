"""The C-ABI library on a machine without a GPU: it builds, loads, exports
every entry point include/pda.h declares, and its host-only calls behave."""
import ctypes
import os
import re

import pytest

import paged_gqa_decode_05_gb300 as pda
from paged_gqa_decode_05_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pda.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pda.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pda_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 18
    for name in names:
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.pda_abi_version() == 5
    hdr = open(HEADER).read()
    assert int(re.search(r"#define PDA_ABI_VERSION (\d+)", hdr).group(1)) == pda.ABI_VERSION == 5
    assert lib.pda_status_string(0) == b"ok"
    assert b"invalid" in lib.pda_status_string(1)


@pytest.mark.parametrize("dims,status", [
    (dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16), 0),
    (dict(num_q_heads=64, num_kv_heads=8, head_dim=64, block_size=32), 0),
    (dict(num_q_heads=16, num_kv_heads=4, head_dim=256, block_size=8), 0),
    (dict(num_q_heads=32, num_kv_heads=7, head_dim=128, block_size=16), pda.ERR_INVALID_ARG),
    (dict(num_q_heads=32, num_kv_heads=8, head_dim=512, block_size=16), pda.ERR_INVALID_ARG),
    (dict(num_q_heads=32, num_kv_heads=8, head_dim=96, block_size=16), pda.ERR_UNSUPPORTED),
    (dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=1), 0),
    (dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=3), pda.ERR_UNSUPPORTED),
    (dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=128), pda.ERR_UNSUPPORTED),
    (dict(num_q_heads=32, num_kv_heads=2, head_dim=128, block_size=16), pda.ERR_UNSUPPORTED),
    (dict(num_q_heads=0, num_kv_heads=8, head_dim=128, block_size=16), pda.ERR_INVALID_ARG),
])
def test_check_dims(lib, dims, status):
    assert pda.check_dims(**dims) == status
    if status:
        assert lib.pda_last_error()  # a message explains the failure


def test_stride_triples(lib):
    kw = dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16)
    assert pda.paged_strides(**kw) == (16 * 8 * 128, 8 * 128, 128)
    assert pda.slot_strides(**kw) == (2 * 8 * 16 * 128, 128, 16 * 128)


def test_create_without_gpu_fails_cleanly(lib):
    d = pda.Dims(4, 8, 2, 128, 16, 8)
    ctx = ctypes.c_void_p()
    st = lib.pda_create(ctypes.byref(d), ctypes.byref(ctx))
    assert st in (pda.ERR_NO_DEVICE, pda.ERR_CUDA)
    assert not ctx.value


def test_calls_on_null_context_are_rejected(lib):
    assert lib.pda_begin_step(None, 1, None) == pda.ERR_INVALID_ARG
    assert lib.pda_finalize(None, None, 1, None) == pda.ERR_INVALID_ARG
    assert lib.pda_decode(None, None, None, None, 1, None, 1, None, 1, 0.0, None, None) == \
        pda.ERR_INVALID_ARG
    flags = ctypes.c_uint32()
    assert lib.pda_read_device_errors(None, ctypes.byref(flags), 1, None) == pda.ERR_INVALID_ARG


def _noalloc(lib):
    fn = lib.pda_decode_noalloc
    P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    fn.restype = I32
    fn.argtypes = [P, P, P, I64, P, I32, P, I32, I32, I32, I32, I32, F, P, P, P]
    return fn


def test_noalloc_host_checks(lib):
    """The allocation-free decode refuses, before touching a device, a missing
    flags word (a failure would otherwise go unreported), unsupported dims and
    an oversized batch."""
    fn = _noalloc(lib)
    buf = ctypes.create_string_buffer(64)
    addr = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    args = dict(q=addr, k=addr, v=addr, nb=1, table=addr, mb=1, lens=addr, batch=1, hq=8, hkv=2,
                d=128, bs=16, scale=float("nan"), out=addr, flags=addr, stream=None)

    def call(**kw):
        a = {**args, **kw}
        return fn(a["q"], a["k"], a["v"], a["nb"], a["table"], a["mb"], a["lens"], a["batch"],
                  a["hq"], a["hkv"], a["d"], a["bs"], a["scale"], a["out"], a["flags"], a["stream"])

    assert call(flags=None) == pda.ERR_INVALID_ARG
    assert b"device_flags" in lib.pda_last_error()
    assert call(flags=addr + 2) == pda.ERR_INVALID_ARG
    assert call(d=96) == pda.ERR_UNSUPPORTED
    assert call(bs=3) == pda.ERR_UNSUPPORTED
    assert call(hkv=3) == pda.ERR_INVALID_ARG
    assert call(batch=1025) == pda.ERR_INVALID_ARG
    assert call(batch=-1) == pda.ERR_INVALID_ARG
    assert call(batch=0) == pda.OK  # nothing to do, nothing launched
