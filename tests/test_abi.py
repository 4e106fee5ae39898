"""The C-ABI library builds, loads and exports every entry point of include/kvc.h.

CPU only: no compute call is made; only host-side argument checks that
return before touching a device are exercised.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvc.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    names = re.findall(r"\b(kvc_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from budgeted_kv_cache_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_four_calls():
    names = declared_functions()
    for n in ("kvc_score", "kvc_select", "kvc_compact_rerotate_quant", "kvc_decode_attn"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    f = lib.kvc_status_string
    f.restype = ctypes.c_char_p
    f.argtypes = [ctypes.c_int]
    assert f(0) == b"ok"
    assert f(1) == b"invalid argument"
    assert f(3) == b"workspace missing or too small"


def test_reference_store_call_checks_its_arguments(lib):
    import budgeted_kv_cache_gb300 as kvc
    kvc.library()
    shape = kvc.make_shape(1, 1, 4, 2, 64, 100)
    pol = kvc.Policy(budget_tokens=10, capacity=10, renumber=True).c()
    rs = kvc.kvc_ref_store(None, None, None, None, None)
    # no caches and an empty reference store: rejected before any launch
    assert kvc.library().kvc_compact_rerotate_quant_ref(
        ctypes.byref(shape), ctypes.byref(pol), None, None, None, None, None, None, None, 0,
        ctypes.byref(rs), None, None, None) == 1


def test_argument_errors_return_before_any_launch(lib):
    import budgeted_kv_cache_gb300 as kvc
    kvc.library()
    # null shape
    assert lib.kvc_score(None, None, None, 0, ctypes.c_float(0), None, None, 1, 0, None, None,
                         None, None, ctypes.c_size_t(0), None) == 1
    bad = kvc.make_shape(1, 1, 4, 2, 96, 100)       # head_dim 96 is not supported
    assert kvc.library().kvc_score(ctypes.byref(bad), None, None, 8, 0.0, None, None, 1, 0, None,
                                   None, None, None, 0, None) == 2
    shape = kvc.make_shape(1, 1, 4, 3, 64, 100)     # H_q not a multiple of H_kv
    pol = kvc.Policy(budget_tokens=10, capacity=10).c()
    assert kvc.library().kvc_select(ctypes.byref(shape), ctypes.byref(pol), None, None, None, None,
                                    None, None, 0, None) == 1
    shape = kvc.make_shape(1, 1, 4, 2, 64, 100)
    both = kvc.Policy(budget_tokens=10, budget_bytes=100, capacity=100).c()   # two budgets
    assert kvc.library().kvc_select(ctypes.byref(shape), ctypes.byref(both), None, None, None,
                                    None, None, None, 0, None) == 1
    small = kvc.Policy(budget_tokens=10, capacity=5).c()                       # capacity < budget
    assert kvc.library().kvc_select(ctypes.byref(shape), ctypes.byref(small), None, None, None,
                                    None, None, None, 0, None) == 1
    page = kvc.Policy(budget_tokens=24, capacity=24, page_size=16).c()        # budget % P
    assert kvc.library().kvc_select(ctypes.byref(shape), ctypes.byref(page), None, None, None,
                                    None, None, None, 0, None) == 1


def test_compaction_decode_and_variant_arguments_are_checked_first(lib):
    """Null, misaligned and out-of-range arguments of the compaction, decode and
    score-pooling calls return KVC_ERR_INVALID_ARG (or KVC_ERR_UNSUPPORTED)
    before the library looks for a device.  Every call below is refused by a
    host check, so the stand-in pointers are never dereferenced and no kernel
    is launched, on a machine with or without a GPU."""
    import budgeted_kv_cache_gb300 as kvc
    L = kvc.library()
    A = 1 << 20                                       # a 16-byte aligned stand-in pointer
    shape = kvc.make_shape(1, 1, 4, 2, 64, 100)
    ren = kvc.Policy(budget_tokens=10, capacity=10, renumber=True).c()
    pools = kvc.kvc_pools(A, A, None, None, None, None, None, None, None, None, A, None)
    SH, PO, PL = ctypes.byref(shape), ctypes.byref(ren), ctypes.byref(pools)

    def compact(k=A, v=A, pos=A, idx=A, cnt=A, cos=A, sin=A, max_pos=100, pol=PO, pl=PL):
        return L.kvc_compact_rerotate_quant(SH, pol, k, v, pos, idx, cnt, cos, sin, max_pos, pl,
                                            None, None)
    assert compact(k=None) == 1 and compact(idx=None) == 1 and compact(cnt=None) == 1
    assert compact(k=A + 8) == 1                                # caches 16-byte aligned
    assert compact(cos=None) == 1 and compact(sin=A + 4) == 1   # renumbering needs the tables
    assert compact(max_pos=5) == 1                              # tables shorter than the capacity
    no_pos = kvc.kvc_pools(A, A, None, None, None, None, None, None, None, None, None, None)
    assert compact(pl=ctypes.byref(no_pos)) == 1                # positions out are required
    byte = kvc.Policy(budget_bytes=4096, capacity=100).c()
    assert compact(pol=ctypes.byref(byte)) == 1                 # byte mode needs every pool

    def decode(q=A, pl=PL, cnt=A, out=A):
        return L.kvc_decode_attn(SH, PO, q, pl, cnt, 0.0, out, None, 0, None)
    assert decode(q=None) == 1 and decode(cnt=None) == 1 and decode(out=None) == 1
    wide = kvc.make_shape(1, 1, 32, 2, 64, 100)                 # 16 query heads per KV head
    assert L.kvc_decode_attn(ctypes.byref(wide), PO, A, PL, A, 0.0, A, None, 0, None) == 2

    B2 = 2 * A
    assert L.kvc_pool_scores(4, 100, A, B2, 4, 0, None) == 1    # kernel sizes 1, 3, 5, 7
    assert L.kvc_pool_scores(4, 100, A, B2, 3, 9, None) == 1    # average or maximum
    assert L.kvc_pool_scores(4, 100, A, A, 3, 0, None) == 1     # not in place
    assert L.kvc_pool_scores(65536, 100, A, B2, 3, 0, None) == 1  # rows within a grid dimension


def test_overrides_check_their_ranges(lib):
    """kvc_set_overrides is host-only: out-of-range fields are refused and change nothing."""
    import budgeted_kv_cache_gb300 as kvc
    kvc.library()
    bad = [kvc.kvc_overrides(-1, 0, 0, -1, -1), kvc.kvc_overrides(0, 33, 0, -1, -1),
           kvc.kvc_overrides(0, 0, -1, -1, -1), kvc.kvc_overrides(0, 0, 0, -2, -1),
           kvc.kvc_overrides(0, 0, 0, -1, -2)]
    for o in bad:
        assert kvc.library().kvc_set_overrides(ctypes.byref(o)) == 1
    ok = kvc.kvc_overrides(0, 8, 0, -1, 3)
    try:
        assert kvc.library().kvc_set_overrides(ctypes.byref(ok)) == 0
    finally:
        assert kvc.library().kvc_set_overrides(None) == 0   # defaults for every later call


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import budgeted_kv_cache_gb300 as kvc
    monkeypatch.setattr(kvc, "_LIB", None)
    monkeypatch.setattr(kvc, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(kvc.KvcError):
        kvc.library()
