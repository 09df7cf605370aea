"""CPU-only checks of the C-ABI library: it loads, exports every symbol the
public header declares, and rejects bad arguments on the host before any CUDA
call (these calls never reach the GPU)."""
import ctypes
import os
import re

import pytest

from lse_merge_gb300 import _lib
from lse_merge_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "skv.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return _lib.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SKV_API\s+[\w\s\*]+?\b(skv_\w+)\s*\(", text)))


def test_header_declares_the_path():
    syms = declared_symbols()
    for name in ("skv_chunk_costs", "skv_lpt_order", "skv_attn_fwd", "skv_lse_merge", "skv_attn_bwd",
                 "skv_workspace_bytes", "skv_stream_status", "skv_status_str"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name


def test_struct_layout():
    # int32 x4, int64, int32 x3, (pad), 2 pointers, enum, float, int32, (pad)
    assert ctypes.sizeof(_lib.SkvProblem) == 72
    assert _lib.SkvProblem.S.offset == 16
    assert _lib.SkvProblem.s.offset == 40
    assert _lib.SkvProblem.dtype.offset == 56
    assert _lib.SkvProblem.n_kv_heads.offset == 64


def prob(**kw):
    base = dict(B=16, n_blocks=8, n_heads=4, head_dim=64, S=2048, m=512, P=4, J=1, s=0x1000, a=0x2000,
                dtype=0, scale=0.0, n_kv_heads=0)
    base.update(kw)
    return _lib.SkvProblem(*[base[f] for f, _ in _lib.SkvProblem._fields_])


def test_status_strings(lib):
    for code in range(7):
        assert lib.skv_status_str(code).decode()
    assert lib.skv_status_str(99).decode() == "unknown status"


def test_workspace_bytes_host_logic(lib):
    ok = prob()
    fwd = lib.skv_workspace_bytes(ctypes.byref(ok), 0)
    bwd = lib.skv_workspace_bytes(ctypes.byref(ok), 1)
    assert fwd > 0 and fwd % 256 == 0
    assert bwd > fwd
    assert lib.skv_workspace_bytes(ctypes.byref(ok), 7) == 0
    for bad in (dict(head_dim=96), dict(P=3), dict(m=100, S=400, P=4, J=1), dict(B=0), dict(n_heads=0),
                dict(scale=-1.0), dict(dtype=5), dict(s=None)):
        p = prob(**bad)
        assert lib.skv_workspace_bytes(ctypes.byref(p), 0) == 0, bad


def test_host_validation_rejects_before_launch(lib):
    E = _lib
    bad = prob(P=3)                    # P*J*m != S
    assert lib.skv_chunk_costs(ctypes.byref(bad), ctypes.c_void_p(0x1000), None) == E.SKV_ERR_INVALID_ARG
    assert lib.skv_chunk_costs(None, ctypes.c_void_p(0x1000), None) == E.SKV_ERR_INVALID_ARG
    assert lib.skv_chunk_costs(ctypes.byref(prob()), None, None) == E.SKV_ERR_INVALID_ARG
    assert lib.skv_lpt_order(ctypes.c_void_p(0x1000), 12, 4, 2, None, None, None, None) == E.SKV_ERR_INVALID_ARG
    assert lib.skv_lpt_order(ctypes.c_void_p(0x1000), 32768, 2, 16384, ctypes.c_void_p(0x1000),
                             ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), None) == E.SKV_ERR_UNSUPPORTED
    assert lib.skv_lse_merge(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), 0, 10, 64, ctypes.c_void_p(0x1000),
                             0, None, None) == E.SKV_ERR_INVALID_ARG
    assert lib.skv_lse_merge(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), 2, 10, 96, ctypes.c_void_p(0x1000),
                             0, None, None) == E.SKV_ERR_UNSUPPORTED
    assert lib.skv_lse_merge(ctypes.c_void_p(0x1004), ctypes.c_void_p(0x1000), 2, 10, 64, ctypes.c_void_p(0x1000),
                             0, None, None) == E.SKV_ERR_INVALID_ARG
    # rows == 0 is a valid no-op
    assert lib.skv_lse_merge(None, None, 2, 0, 64, None, 0, None, None) == E.SKV_OK
    p = prob(dtype=1)
    assert lib.skv_attn_fwd(ctypes.byref(p), None, None, None, None, None, None, ctypes.c_void_p(0x1000), 0,
                            None) == E.SKV_ERR_WORKSPACE
    ws = lib.skv_workspace_bytes(ctypes.byref(p), 0)
    assert lib.skv_attn_fwd(ctypes.byref(p), None, None, None, None, None, None, ctypes.c_void_p(0x1000), ws,
                            None) == E.SKV_ERR_INVALID_ARG
    assert lib.skv_attn_fwd(ctypes.byref(prob(head_dim=32)), None, None, None, None, None, None, None, 0,
                            None) == E.SKV_ERR_UNSUPPORTED
    # grouped-query layouts: Hkv must divide H (0 selects H)
    for hkv in (-1, 3, 5, 8):
        assert lib.skv_chunk_costs(ctypes.byref(prob(n_kv_heads=hkv)), ctypes.c_void_p(0x1000),
                                   None) == E.SKV_ERR_INVALID_ARG
    for hkv in (1, 2, 4):
        assert lib.skv_attn_fwd(ctypes.byref(prob(dtype=1, n_kv_heads=hkv)), None, None, None, None, None, None,
                                ctypes.c_void_p(0x1000), 0, None) == E.SKV_ERR_WORKSPACE
    # merge backward: the same argument checks as the merge
    assert lib.skv_lse_merge_bwd(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), 0, 10, 64, ctypes.c_void_p(0x1000),
                                 0, None, None, ctypes.c_void_p(0x1000), None) == E.SKV_ERR_INVALID_ARG
    assert lib.skv_lse_merge_bwd(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), 2, 10, 96, ctypes.c_void_p(0x1000),
                                 0, None, None, ctypes.c_void_p(0x1000), None) == E.SKV_ERR_UNSUPPORTED
    assert lib.skv_lse_merge_bwd(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x1000), 2, 10, 64, ctypes.c_void_p(0x1000),
                                 0, None, None, None, None) == E.SKV_ERR_INVALID_ARG
    assert lib.skv_lse_merge_bwd(None, None, 2, 0, 64, None, 0, None, None, None, None) == E.SKV_OK
    assert lib.skv_set_wait_limit(5) == E.SKV_OK
    assert lib.skv_set_wait_limit(0) == E.SKV_OK


def test_python_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load.__wrapped__ if hasattr(_lib.load, "__wrapped__") else None
        saved = _lib._lib
        _lib._lib = None
        try:
            _lib.load(str(tmp_path / "libskv.so"))
        finally:
            _lib._lib = saved


def test_merge_oproj_rejects_bad_shapes_on_the_host(lib):
    f = lib.skv_lse_merge_oproj
    args = dict(o_part=0x1000, lse_part=0x2000, P=4, Q=128, H=4, d=128, w=0x3000, d_model=256, o=0x4000, lse=0x5000,
                y=0x6000)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["o_part"], a["lse_part"], a["P"], a["Q"], a["H"], a["d"], a["w"], a["d_model"], a["o"], a["lse"],
                 a["y"], None)

    assert call(d_model=100) == _lib.SKV_ERR_INVALID_ARG        # not a multiple of 16
    assert call(d_model=0) == _lib.SKV_ERR_INVALID_ARG
    assert call(P=0) == _lib.SKV_ERR_INVALID_ARG
    assert call(d=96) == _lib.SKV_ERR_UNSUPPORTED
    assert call(w=0x3008) == _lib.SKV_ERR_INVALID_ARG           # misaligned weight
    assert call(y=0) == _lib.SKV_ERR_INVALID_ARG
    assert call(Q=0) == _lib.SKV_OK                             # nothing to do
