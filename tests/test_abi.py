"""The C-ABI library loads here (no GPU) and exports what include/si.h declares;
host-side validation answers without touching CUDA."""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "si.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M)
    return sorted({n for n in names if n not in ("defined",)})


@pytest.fixture(scope="module")
def si():
    import activation_sparse_gb300 as si
    return si


def test_header_parses():
    names = header_functions()
    assert "si_sparse_ffn_decode" in names and "spax_tiered_down" in names
    assert len(names) >= 20


def test_library_exports_every_declared_symbol(si):
    lib = si.load()
    out = subprocess.run(["nm", "-D", "--defined-only", si.lib_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (\w+)$", out, flags=re.M))
    for name in header_functions():
        assert name in exported, name
        assert hasattr(lib, name)
        assert name in si.SIGNATURES, name


def test_counts_host_side(si):
    assert si.si_count(0.2, 1024) == 205
    assert si.si_counts(1024, 0.7, 0.2, 0.4) == (717, 205, 410, 205)
    assert si.si_counts(8192, 0.7, 0.2, 0.4) == (5734, 1638, 3277, 1639)
    assert si.si_counts(8192, 0.7, 0.25, 0.5) == (5734, 2048, 4096, 2048)
    assert si.si_counts(11008, 0.8, 0.25, 0.5) == (8806, 2752, 5504, 2752)
    assert si.si_packed_bytes(2048, 5734) == 3 * 2048 * 5734 * 2


@pytest.mark.parametrize("args", [(1024, 0.4, 0.2, 0.5), (1024, 1.1, 0.2, 0.4), (0, 0.7, 0.2, 0.4),
                                  (1024, 0.7, -0.1, 0.4), (1024, float("nan"), 0.2, 0.4)])
def test_counts_rejects_bad_ratios(si, args):
    with pytest.raises(si.SIError) as e:
        si.si_counts(*args)
    assert e.value.code == si.SI_ERR_INVALID_ARG


def test_validation_before_cuda(si):
    lib = si.load()
    h = C.c_void_p()
    # NULL weights / bad shapes are rejected without any CUDA call
    assert lib.si_pack_loaded(None, None, None, 64, 10, None, None, 0.5, 0.1, C.byref(h), None) == si.SI_ERR_INVALID_ARG
    assert b"NULL" in lib.si_last_error_string()
    p = C.c_void_p(16)
    assert lib.si_pack_loaded(p, p, p, 60, 10, p, p, 0.5, 0.1, C.byref(h), None) == si.SI_ERR_INVALID_ARG
    assert lib.si_pack_loaded(p, p, p, 64, 10, p, p, 0.5, 0.6, C.byref(h), None) == si.SI_ERR_INVALID_ARG
    assert lib.si_sparse_ffn_decode(None, p, 1, 1, p, p, None) == si.SI_ERR_INVALID_ARG
    assert lib.si_select_from_absact(None, p, 8, 1, 1, 1, 0.4, p, None, None, None) == si.SI_ERR_INVALID_ARG
    assert lib.spax_encode(p, 256, 10, 5, 128, C.byref(h), None) == si.SI_ERR_UNSUPPORTED
    # 3-bit records are whole 16-byte units only when d % 128 == 0
    assert lib.spax_encode(p, 192, 10, 3, 64, C.byref(h), None) == si.SI_ERR_INVALID_ARG
    assert lib.spax_encode(p, 256, 10, 4, 100, C.byref(h), None) == si.SI_ERR_INVALID_ARG
    assert lib.si_merge_scores(None, None, 1, 4, p, None) == si.SI_ERR_INVALID_ARG
    assert lib.si_layer_destroy(None) == si.SI_OK
    # the GEMM tile override only takes the widths the kernel is built for
    for bad in (-1, 1, 48, 72, 129, 256):
        assert lib.si_set_gemm_tile(bad) == si.SI_ERR_INVALID_ARG
    for good in (64, 80, 96, 112, 128, 0):
        assert lib.si_set_gemm_tile(good) == si.SI_OK
    assert lib.si_gemm_tile_for(512, 5734, None) == si.SI_ERR_INVALID_ARG
    # the extensions' entry points validate on the host too
    assert lib.si_layer_set_salience(None, 1) == si.SI_ERR_INVALID_ARG
    assert lib.si_layer_norms(None, C.byref(C.c_void_p())) == si.SI_ERR_INVALID_ARG
    assert lib.spax_select_decode(None, p, p, p, 1, p, 0.3, 0.3, p, None, None) == si.SI_ERR_INVALID_ARG
    n = C.c_int(0)
    assert lib.si_expand_clusters(None, p, 1, 32, p, C.byref(n), None) == si.SI_ERR_INVALID_ARG
    # |A| goes out by TMA: a misaligned output is refused before any launch
    odd = C.c_void_p(16 * 1024 + 4)
    assert lib.si_prefill_absact(p, p, 4, 1, odd, None) == si.SI_ERR_INVALID_ARG
    assert b"aligned" in lib.si_last_error_string()
    assert lib.si_select_dynamic(p, p, 4, 1, 1, 0.4, p, odd, None) == si.SI_ERR_INVALID_ARG


def test_sparse_layers_match_oracle(si):
    """Host-side layer range: the library's mask equals the oracle's for
    Table 1's range at the pages' depths and for other slices."""
    import oracle
    for L in (0, 1, 6, 7, 8, 16, 28, 36):
        for first, last in ((5, -2), (0, 0), (0, -1), (3, 10), (2, 40), (9, -9)):
            got = si.si_sparse_layers(L, first, last)
            ref = oracle.sparse_layers(L, first, last)
            assert np.array_equal(got, ref), (L, first, last)
    lib = si.load()
    assert lib.si_sparse_layers(4, -1, -2, None, None) == si.SI_ERR_INVALID_ARG
    assert lib.si_sparse_layers(4, 1, -2, None, None) == si.SI_ERR_INVALID_ARG
