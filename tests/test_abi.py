"""C-ABI library: build, exported symbols, host-side validation (no GPU calls)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from tests.helpers import ensure_built

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    from lattice_he_database_gb300 import pir
    return pir.lib()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(pir_\w+)\s*\(", src, flags=re.M))
    return names


def test_header_declares_the_boundary():
    names = declared_symbols()
    for must in ["pir_ctx_create", "pir_ctx_destroy", "pir_ntt_fwd", "pir_ntt_inv", "pir_db_encode",
                 "pir_db_bytes", "pir_rowsel", "pir_scalar_scan", "pir_status", "pir_strerror"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in sorted(declared_symbols()):
        assert hasattr(lib, name), name


def test_synth_device_library_builds_and_exports():
    import synth.device as sd
    sd.build()
    L = ctypes.CDLL(sd.LIB)
    assert hasattr(L, "synth_fill") and hasattr(L, "synth_fill_bytes")


def test_params_check(lib):
    from lattice_he_database_gb300 import pir
    qs = oracle.primes(4096, 3)
    assert pir.pir_params_check(4096, qs) == 0
    assert pir.pir_params_check(4096, qs[:1]) == 0
    bad = [
        (4096, []),                                  # L = 0
        (4096, qs + oracle.primes(4096, 5)[3:5]),    # L = 5
        (4097, qs),                                  # N not a power of two
        (8, oracle.primes(8, 1)),                    # N too small
        (8192, oracle.primes(8192, 1)),              # N too large
        (4096, [qs[0], qs[0]]),                      # duplicate prime
        (4096, [qs[0] + 8192 * 2]),                  # = 1 mod 2N but not prime (or above bound)
        (4096, [536813569 + 2]),                     # not = 1 mod 2N
        (4096, [oracle.primes(4096, 1, 1 << 30)[0]]),  # prime = 1 mod 2N but >= 2^29
    ]
    for N, q in bad:
        assert pir.pir_params_check(N, q) == pir.PIR_ERR_ARG, (N, q)
    # small rings used by the tests
    for N in (16, 64, 256):
        assert pir.pir_params_check(N, oracle.primes(N, 2)) == 0


def test_error_strings_and_null_ctx(lib):
    from lattice_he_database_gb300 import pir
    assert pir.pir_strerror(0) == "ok"
    assert "invalid" in pir.pir_strerror(pir.PIR_ERR_ARG)
    assert lib.pir_db_bytes(None, 4, 4) == 0
    assert lib.pir_rowsel(None, None, 1, 1, None, 1, None, None, 0, None) == pir.PIR_ERR_ARG
    assert lib.pir_rowsel_workspace_bytes(None, 4, 4, 1) == 0
    assert lib.pir_ntt_fwd(None, None, None, 1, None) == pir.PIR_ERR_ARG
    assert lib.pir_scalar_workspace_bytes(0, 64) == 0
    assert lib.pir_coltor_workspace_bytes(None, 4, 5) == 0
    assert lib.pir_coltor_stage(None, None, 5, 18, None, 4, None, None, 0, None) == pir.PIR_ERR_ARG
    assert lib.pir_coltor(None, None, 5, 18, None, 4, None, None, 0, None) == pir.PIR_ERR_ARG
    assert lib.pir_expand_workspace_bytes(None, 4, 5) == 0
    assert lib.pir_expand_stage(None, None, 5, 18, 0, None, 1, None, None, 0, None) == pir.PIR_ERR_ARG
    assert lib.pir_expand(None, None, 5, 18, 3, None, None, None, 0, None) == pir.PIR_ERR_ARG
    assert lib.pir_coltor_batch_workspace_bytes(None, 4, 2, 5) == 0
    assert lib.pir_coltor_batch(None, None, 5, 18, None, 4, 2, None, None, 0, None) == pir.PIR_ERR_ARG
    assert lib.pir_expand_batch(None, None, 5, 18, 3, None, 2, None, None, 0, None) == pir.PIR_ERR_ARG
    h = ctypes.c_void_p()
    assert lib.pir_server_create(ctypes.byref(h), None, None, 1, 1, 1) == pir.PIR_ERR_ARG and not h.value
    assert lib.pir_server_submit(None, None, None, None) == pir.PIR_ERR_ARG
    assert lib.pir_server_wait(None, 0) == pir.PIR_ERR_ARG
    lib.pir_server_destroy(None)


@pytest.mark.parametrize("N,L,D0,D1", [(16, 2, 3, 5), (16, 1, 2, 128), (16, 3, 4, 130), (4096, 3, 2, 1365)])
def test_db_layout_is_a_bijection(N, L, D0, D1):
    """Every (p, k, n) with n < D1 has its own word; padding columns fill the rest."""
    from lattice_he_database_gb300 import pir
    P = L * N
    D1p = (D1 + 3) // 4 * 4
    p, k, n = np.meshgrid(np.arange(P), np.arange(D0), np.arange(D1p), indexing="ij")
    off = pir.db_layout_offset(N, L, D0, D1, p, k, n).reshape(-1)
    assert off.min() == 0 and off.max() == P * D0 * D1p - 1
    assert np.unique(off).size == off.size
    # (p, slab) blocks are contiguous: within a slab, consecutive k are W_s apart
    if D1 > 128:
        o = pir.db_layout_offset(N, L, D0, D1, 0, np.arange(D0), 0)
        assert (np.diff(o) == 128).all()
