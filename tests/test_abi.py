"""The C-ABI library without a GPU: it builds, loads, exports every function
include/engram.h declares, and its host-side checks refuse bad configurations
before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from hashed_gram_embedding_engram_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib._lib()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(engram_\w+)\s*\(", src, flags=re.M))
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("engram_plan_create", "engram_plan_destroy", "engram_plan_workspace_bytes", "engram_hash",
              "engram_gather", "engram_stage_a", "engram_kv_projection", "engram_stage_b", "engram_forward",
              "engram_get_error", "engram_cache_create", "engram_cache_observe", "engram_cache_build",
              "engram_stage_a_cached", "engram_cache_stats", "engram_cache_destroy",
              "engram_status_string", "engram_plan_set_fused_stage_b", "engram_plan_set_cta_pairs", "engram_plan_set_fused_decode", "engram_cache_set_dedup", "engram_quantize_fp8"):
        assert n in names


def test_library_exports_every_declared_function(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_binding_return_types_match_the_header(lib):
    """A function the header declares returning a pointer gets a pointer restype,
    one returning engram_status_t or int an int (a truncated pointer would pass
    unnoticed until an address above 2^31)."""
    for f in os.listdir(os.path.join(ROOT, "include")):
        if not f.endswith(".h"):
            continue
        src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", f)).read(), flags=re.S)
        for ret, name in re.findall(r"^\s*((?:const\s+)?\w+\s*\**)\s*(engram_\w+)\s*\(", src, flags=re.M):
            rt = getattr(lib, name).restype
            if "*" in ret:
                assert rt in (ctypes.c_void_p, ctypes.c_char_p), (name, ret, rt)
            elif ret.strip() in ("engram_status_t", "int"):
                assert rt is ctypes.c_int, (name, ret, rt)


def test_status_strings(lib):
    from hashed_gram_embedding_engram_gb300 import _lib
    for s in range(8):
        assert lib.engram_status_string(s)
    assert _lib.STATUS_NAMES[_lib.ERR_NOT_MAPPED] == "NOT_MAPPED"


def _cfg(**kw):
    from hashed_gram_embedding_engram_gb300 import _lib
    base = dict(N=3, K=2, row_dim=16, d=64, M=1, conv_w=4, conv_dilation=3, table_dtype=_lib.F32,
                act_dtype=_lib.F32, eps=1e-6)
    base.update(kw)
    R = (base["N"] - 1) * base["K"]
    primes = (ctypes.c_uint32 * max(R, 1))(*([1009] * max(R, 1)))
    mults = (ctypes.c_uint64 * 600)(*([1] * 600))
    c = _lib.Config(base["N"], base["K"], base["row_dim"], base["d"], base["M"], base["conv_w"],
                    base["conv_dilation"], base["table_dtype"], base["act_dtype"], base["eps"], primes, mults)
    return c, (primes, mults)


@pytest.mark.parametrize("bad", [dict(N=1), dict(N=9), dict(K=0), dict(N=3, K=40), dict(M=0), dict(M=9),
                                 dict(d=12), dict(conv_w=0), dict(conv_w=9), dict(conv_dilation=0),
                                 dict(eps=0.0), dict(eps=float("nan")), dict(row_dim=3)])
def test_plan_rejects_bad_configs_before_cuda(lib, bad):
    from hashed_gram_embedding_engram_gb300 import _lib
    c, keep = _cfg(**bad)
    h = ctypes.c_void_p()
    assert lib.engram_plan_create(ctypes.byref(c), 100, ctypes.byref(h)) == _lib.ERR_INVALID_ARG
    assert not h.value


def test_plan_rejects_mismatched_dtypes(lib):
    from hashed_gram_embedding_engram_gb300 import _lib
    c, keep = _cfg(table_dtype=_lib.BF16, act_dtype=_lib.F32, row_dim=64)
    h = ctypes.c_void_p()
    assert lib.engram_plan_create(ctypes.byref(c), 100, ctypes.byref(h)) == _lib.ERR_UNSUPPORTED


def test_plan_rejects_bad_token_budget_and_null(lib):
    from hashed_gram_embedding_engram_gb300 import _lib
    c, keep = _cfg()
    h = ctypes.c_void_p()
    assert lib.engram_plan_create(ctypes.byref(c), 0, ctypes.byref(h)) == _lib.ERR_INVALID_ARG
    assert lib.engram_plan_create(None, 10, ctypes.byref(h)) == _lib.ERR_INVALID_ARG
    assert lib.engram_plan_destroy(None) == _lib.OK


def test_null_plan_is_refused_everywhere(lib):
    from hashed_gram_embedding_engram_gb300 import _lib
    n = ctypes.c_size_t()
    assert lib.engram_plan_workspace_bytes(None, 10, ctypes.byref(n)) == _lib.ERR_INVALID_ARG
    assert lib.engram_hash(None, None, 1, 1, None, 1, None, None, None) == _lib.ERR_INVALID_ARG
    assert lib.engram_gather(None, None, 1, None, None, None, None) == _lib.ERR_INVALID_ARG
    assert lib.engram_kv_projection(None, None, 1, None, None, None) == _lib.ERR_INVALID_ARG
    assert lib.engram_stage_b(None, None, 1, 1, None, 1, None, None, None, None, None, 0, None) == _lib.ERR_INVALID_ARG
    assert lib.engram_forward(None, None, 1, 1, None, 1, None, None, None, None, 0, None) == _lib.ERR_INVALID_ARG
    assert lib.engram_get_error(None, None, None) == _lib.ERR_INVALID_ARG


def test_newer_entry_points_refuse_null_and_bad_sizes_before_cuda(lib):
    """The several-layer, FP8, split and option entry points check their handles
    and sizes on the host: no CUDA call is needed to refuse these."""
    from hashed_gram_embedding_engram_gb300 import _lib
    bad = _lib.ERR_INVALID_ARG
    assert lib.engram_stage_a(None, None, 1, 1, None, 1, None, None, None, None, None) == bad
    assert lib.engram_stage_a_layers(0, None, None, 1, 1, None, 1, None, None, None, None, None) == bad
    assert lib.engram_stage_a_layers(9, None, None, 1, 1, None, 1, None, None, None, None, None) == bad
    assert lib.engram_stage_a_e4m3(None, None, 1, 1, None, 1, None, None, None, None, None) == bad
    assert lib.engram_stage_a_layers_e4m3(0, None, None, 1, 1, None, 1, None, None, None, None, None) == bad
    assert lib.engram_stage_b_e4m3(None, None, 1, 1, None, 1, None, None, None, None, None, None, 0, None) == bad
    assert lib.engram_forward_split(None, None, 1, None, None, 1, 1, None, 1, None, None, None, None, 0,
                                    None) == bad
    assert lib.engram_plan_set_sm_limit(None, 1) == bad
    assert lib.engram_plan_set_host_gather_sms(None, 1) == bad
    assert lib.engram_plan_host_gather_sms(None) == 0
    out = ctypes.c_void_p()
    for n in (0, -1):
        assert lib.engram_sm_split_create(0, n, ctypes.byref(out)) == bad
        assert not out.value
    assert lib.engram_sm_split_create(0, 8, None) == bad
    assert lib.engram_sm_split_sms(None, 0) == 0
    assert lib.engram_sm_split_stream(None, 1) is None
    assert lib.engram_sm_split_destroy(None) == _lib.OK


def test_front_end_fails_loudly_without_library(monkeypatch, tmp_path):
    from hashed_gram_embedding_engram_gb300 import _lib
    monkeypatch.setattr(_lib, "_LIB", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _lib._lib()
