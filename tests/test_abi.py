"""C-ABI boundary checks that need no GPU: the library loads, exports every declared symbol,
and rejects invalid configurations on the host before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libdt():
    import __graft_entry__

    __graft_entry__._load_builder().build()
    from dynamic_draft_tree_gb300 import _lib

    return _lib


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dt.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dt_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("dt_expand_layer", "dt_cast_prune", "dt_rerank", "dt_build_tree_meta", "dt_verify",
              "dt_graft_retrieve", "dt_adj_update"):
        assert n in names


def test_library_exports_every_declared_symbol(libdt):
    out = subprocess.check_output(["nm", "-D", "--defined-only", libdt.LIB_PATH]).decode()
    exported = set(re.findall(r"\bT (dt_[a-z_]+)\b", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    assert sorted(libdt.EXPORTS) == sorted(declared_functions())


def test_invalid_config_rejected_on_host(libdt):
    lib = libdt.lib
    h = ctypes.c_void_p()
    good = dict(B_max=8, V=1000, K=10, W=10, D_max=6, P_max=61, dtype=0, flags=0)
    bad = [dict(V=1), dict(K=0), dict(K=33), dict(K=20, V=10), dict(W=0), dict(W=33),
           dict(D_max=0), dict(D_max=17), dict(P_max=0), dict(P_max=513),
           dict(B_max=0), dict(B_max=5000), dict(dtype=7)]
    for b in bad:
        c = dict(good, **b)
        cfg = libdt.DtConfig(*[c[f] for f, _ in libdt.DtConfig._fields_])
        rc = lib.dt_create(ctypes.byref(cfg), ctypes.byref(h))
        assert rc == libdt.DT_ERR_ARG, (b, rc)
        assert lib.dt_last_error_string()
    assert lib.dt_create(None, ctypes.byref(h)) == libdt.DT_ERR_ARG


def test_null_handle_rejected(libdt):
    lib = libdt.lib
    assert lib.dt_destroy(None) == libdt.DT_ERR_ARG
    assert lib.dt_tree_reset(None, 1, None, None) == libdt.DT_ERR_ARG
    assert lib.dt_expand_layer(None, None, 0, 1, None) == libdt.DT_ERR_ARG
    assert lib.dt_rerank(None, None, 0, 1, None, None) == libdt.DT_ERR_ARG
    assert lib.dt_verify(None, None, None, 0, 0, 0, 0, None, None, None, None, None) == libdt.DT_ERR_ARG
    msg = lib.dt_last_error_string().decode()
    assert "null" in msg


def test_python_binding_names_match_abi(libdt):
    import dynamic_draft_tree_gb300 as pkg

    for name in libdt.EXPORTS:
        if name == "dt_last_error_string":
            continue
        assert hasattr(pkg, name), name


def test_static_topk_arguments_rejected_on_host(libdt):
    """dt_row_topk_static checks its sizes before any CUDA call; the pointers are never touched."""
    lib = libdt.lib
    fake = 256  # 256-byte aligned, never dereferenced: every call below fails the host check
    assert lib.dt_row_topk_static(None, 1000, 4, 1000, 4, 0, fake, fake, None, None) == libdt.DT_ERR_ARG
    assert lib.dt_row_topk_static(fake, 1000, 1025, 1000, 4, 0, fake, fake, None, None) == libdt.DT_ERR_ARG
    assert "static scratch" in lib.dt_last_error_string().decode()
    for rows, V, K, dtype, ld in [(0, 1000, 4, 0, 1000), (4, 1, 1, 0, 1000), (4, 1000, 33, 0, 1000),
                                  (4, 10, 11, 0, 10), (4, 1000, 4, 5, 1000), (4, 1000, 4, 0, 999)]:
        assert lib.dt_row_topk_static(fake, ld, rows, V, K, dtype, fake, fake, None, None) == libdt.DT_ERR_ARG


def test_fused_cast_calls_reject_bad_arguments(libdt):
    """The fused CAST entry points check their arguments on the host (no GPU needed)."""
    lib = libdt.lib
    assert lib.dt_cast_prune_select(None, None, None, None, None) == libdt.DT_ERR_ARG
    assert lib.dt_cast_verify_rerank(None, None, None, None, None) == libdt.DT_ERR_ARG
    assert "null" in lib.dt_last_error_string().decode()
