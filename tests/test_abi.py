"""CPU checks of the native library: it loads and exports every entry point the
public header declares, with matching binding signatures. No compute call is
made (there may be no GPU)."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "sparse_attn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sa_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from sparse_paged_kv_page_gb300 import build as B
    B.build()
    from sparse_paged_kv_page_gb300 import _lib
    return _lib.load()


def test_header_declares_the_five_steps():
    names = _declared()
    for n in ("sa_append_kv", "sa_score_pages", "sa_select_topk", "sa_sparse_decode",
              "sa_h2o_update"):
        assert n in names


def test_every_declared_symbol_is_exported_and_bound(lib):
    from sparse_paged_kv_page_gb300 import _lib
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name


def test_host_only_calls(lib):
    import sparse_paged_kv_page_gb300 as S
    assert S.sa_version() == "0.1.0"
    assert S.sa_status_string(0) == "SA_OK" and S.sa_status_string(3) == "SA_ERR_WORKSPACE"
    assert S.sa_decode_workspace_size(0, 8, 64, 128, 16, 256) == 0
    assert S.sa_decode_workspace_size(4, 8, 64, 128, 16, 256) > 4 * 8 * 4
    # argument checks run on the host before any launch
    assert lib.sa_decode_step(None, None, None, None, None, 0, None, 8, 1.0, 0.25, None, 16, 4,
                              0, 1, None, None, 0.0, None, None, None, 0, None, None) == 1


def test_wait_selftest_rejects_bad_arguments_on_the_host(lib):
    import ctypes
    st, res = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000)
    for arrivals, limit in ((3, 1000), (-1, 1000), (1, 0), (1, 200_000_000)):
        assert lib.sa_wait_selftest(arrivals, limit, st, res, None) == 1
    assert lib.sa_wait_selftest(1, 1000, None, res, None) == 1


def test_misaligned_pointers_are_rejected_on_the_host(lib):
    """Pools and q must start on 16-byte boundaries; the check runs before any
    launch (the pointer values are never dereferenced on the host)."""
    import ctypes
    from sparse_paged_kv_page_gb300 import _lib
    lens = ctypes.c_void_p(0x10000)
    bt = ctypes.c_void_p(0x20000)
    batch = _lib.SaBatch(block_table=bt, seq_lens=lens, batch=1, bt_stride=4)
    good = dict(k=ctypes.c_void_p(0x100000), v=ctypes.c_void_p(0x200000), meta=ctypes.c_void_p(0x300000),
                dtype=0, num_blocks=4, num_kv_heads=1, page_size=16, head_dim=128, kstd=None)
    q = ctypes.c_void_p(0x400000)
    scores = ctypes.c_void_p(0x500000)
    for field in ("k", "v", "meta", "q"):
        kw = dict(good)
        qq = q
        if field == "q":
            qq = ctypes.c_void_p(0x400008)
        else:
            kw[field] = ctypes.c_void_p(kw[field].value + 8)
        cache = _lib.SaCache(**kw)
        st = lib.sa_score_pages(ctypes.byref(cache), ctypes.byref(batch), qq, 1, 1.0, 0.25, scores, 4,
                                None, None)
        assert st == 1, field
    # q read in 16-byte units by the decode, entmax and Gaussian entry points too
    kw = dict(good)
    kw["kstd"] = ctypes.c_void_p(0x600000)
    cache = _lib.SaCache(**kw)
    bad_q = ctypes.c_void_p(0x400004)
    P = ctypes.c_void_p
    sel, cnt, out = P(0x700000), P(0x710000), P(0x720000)
    assert lib.sa_sparse_decode(ctypes.byref(cache), ctypes.byref(batch), bad_q, 1, sel, cnt, 4, 0.0, out,
                                None, None, 0, P(0x730000), 1 << 20, None, None) == 1
    assert lib.sa_sparse_decode_entmax(ctypes.byref(cache), ctypes.byref(batch), bad_q, 1, sel, cnt, 4, 1.5,
                                       0.0, out, None, None, 0, P(0x730000), 1 << 20, None, None) == 1
    assert lib.sa_gauss_select(ctypes.byref(cache), ctypes.byref(batch), bad_q, 1, 1.5, 0.0, scores, 4, sel,
                               cnt, 4, None, None, None) == 1


def test_struct_layouts_match_the_binding(lib):
    import ctypes
    import sparse_paged_kv_page_gb300 as S
    from sparse_paged_kv_page_gb300 import _lib
    assert S.sa_struct_size(0) == ctypes.sizeof(_lib.SaCache)
    assert S.sa_struct_size(1) == ctypes.sizeof(_lib.SaBatch)
    assert _lib.SaCache.kstd.offset == ctypes.sizeof(_lib.SaCache) - ctypes.sizeof(ctypes.c_void_p)


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "sparse_paged_kv_page_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", txt, re.M), f
                assert "sa_synth" not in txt, f
