"""The C-ABI library builds, loads and exports what include/fa.h declares;
host-side validation (CPU only: no call here reaches a device)."""
import ctypes
import os
import re

import pytest

from io_aware_exact_10_gb300 import build as fab

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    fab.build()
    import io_aware_exact_10_gb300 as fa
    return fa.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("fa_fwd", "fa_bwd", "fa_fwd_gqa", "fa_bwd_gqa", "fa_fwd_ex", "fa_bwd_ex",
                     "fa_bwd_workspace_size", "fa_last_device_error", "fa_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in fa.h but not exported"


def test_strerror_and_version(L):
    import io_aware_exact_10_gb300 as fa
    for s in range(0, 7):
        assert len(fa.fa_strerror(s)) > 3
    assert "unknown" in fa.fa_strerror(99)
    assert "sm_103a" in fa.fa_version()


def test_workspace_size(L):
    import io_aware_exact_10_gb300 as fa
    r256 = lambda x: (x + 255) // 256 * 256
    for B, H, N, d in ((1, 1, 128, 64), (2, 3, 200, 128), (64, 16, 1024, 64), (1, 1, 1, 64)):
        rows = B * H * N
        stats = B * H * ((N + 127) // 128) * 256  # two floats per row, heads padded to 128 rows
        assert fa.fa_bwd_workspace_size(B, H, N, d) == r256(stats * 4) + r256(rows * d * 4)
    assert fa.fa_bwd_workspace_size(0, 1, 128, 64) == 0
    assert fa.fa_bwd_workspace_size(1, 1, 128, 96) == 0
    assert fa.fa_bwd_workspace_size(-1, 1, 128, 64) == 0


A = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


def fwd(L, q=A, k=A, v=A, o=A, lse=A, B=1, H=1, N=128, d=64, scale=0.125, causal=0):
    return L.fa_fwd(q, k, v, o, lse, B, H, N, d, ctypes.c_float(scale), causal, None)


def bwd(L, ws=A, ws_bytes=1 << 30, N=128, d=64, scale=0.125, causal=0, dq=A):
    return L.fa_bwd(A, A, A, A, A, A, dq, A, A, 1, 1, N, d, ctypes.c_float(scale), causal,
                    ws, ws_bytes, None)


def test_fwd_argument_errors(L):
    import io_aware_exact_10_gb300 as fa
    INV, UNS = fa.FA_ERR_INVALID_ARG, fa.FA_ERR_UNSUPPORTED
    assert fwd(L, q=None) == INV
    assert fwd(L, o=A + 8) == INV                  # not 16-byte aligned
    assert fwd(L, lse=A + 4) == INV
    assert fwd(L, B=-1) == INV
    assert fwd(L, N=-5) == INV
    assert fwd(L, scale=0.0) == INV
    assert fwd(L, scale=-0.1) == INV
    assert fwd(L, scale=float("nan")) == INV
    assert fwd(L, scale=float("inf")) == INV
    assert fwd(L, causal=2) == INV
    assert fwd(L, d=96) == UNS
    assert fwd(L, d=256) == UNS
    # empty problems succeed without touching a device
    assert fwd(L, N=0) == fa.FA_OK
    assert fwd(L, B=0, q=None) == fa.FA_OK


def test_bwd_argument_errors(L):
    import io_aware_exact_10_gb300 as fa
    INV = fa.FA_ERR_INVALID_ARG
    need = fa.fa_bwd_workspace_size(1, 1, 128, 64)
    assert bwd(L, ws=None) == INV
    assert bwd(L, ws=A + 16) == INV                # workspace must be 256-byte aligned
    assert bwd(L, ws_bytes=need - 1) == INV
    assert bwd(L, dq=A + 2) == INV
    assert bwd(L, scale=-1.0) == INV
    assert bwd(L, d=32) == fa.FA_ERR_UNSUPPORTED
    assert bwd(L, N=0) == fa.FA_OK


def test_gqa_argument_errors(L):
    """Grouped key/value heads: H_kv must lie in 1 ... H and divide H."""
    import io_aware_exact_10_gb300 as fa
    INV = fa.FA_ERR_INVALID_ARG
    f = lambda H, Hkv, B=1: L.fa_fwd_gqa(A, A, A, A, A, B, H, Hkv, 128, 64, ctypes.c_float(0.125),
                                         0, None)
    b = lambda H, Hkv: L.fa_bwd_gqa(A, A, A, A, A, A, A, A, A, 1, H, Hkv, 128, 64,
                                    ctypes.c_float(0.125), 0, A, 1 << 30, None)
    for H, Hkv in ((4, 0), (4, 3), (4, 5), (4, -2), (6, 4)):
        assert f(H, Hkv) == INV, (H, Hkv)
        assert b(H, Hkv) == INV, (H, Hkv)
    # valid groupings pass validation (and stop later, at the device)
    for H, Hkv in ((4, 4), (4, 2), (4, 1), (6, 3)):
        assert f(H, Hkv) != INV, (H, Hkv)
        assert b(H, Hkv) != INV, (H, Hkv)
    # an empty problem succeeds whatever H_kv is
    assert f(4, 0, B=0) == fa.FA_OK


def test_cross_length_argument_errors(L):
    """Query and key lengths that differ: causal needs N_k >= N_q; N_k = 0
    with query rows, negative or oversized lengths are refused; N_q = 0 is
    an empty problem for the forward, while the backward still owes zero
    dk, dv (so it goes on to the device)."""
    import io_aware_exact_10_gb300 as fa
    INV, OK, NODEV = fa.FA_ERR_INVALID_ARG, fa.FA_OK, fa.FA_ERR_NO_DEVICE
    sc = ctypes.c_float(0.125)
    f = lambda Nq, Nk, causal, B=1: L.fa_fwd_ex(A, A, A, A, A, B, 4, 2, Nq, Nk, 64, sc, causal,
                                                None)
    b = lambda Nq, Nk, causal, B=1: L.fa_bwd_ex(A, A, A, A, A, A, A, A, A, B, 4, 2, Nq, Nk, 64,
                                                sc, causal, A, 1 << 30, None)
    for Nq, Nk, causal in ((256, 128, 1), (2, 1, 1), (5, 0, 0), (5, 0, 1), (-1, 8, 0),
                           (8, -1, 0), ((1 << 30) + 1, 8, 0), (8, (1 << 30) + 1, 0)):
        assert f(Nq, Nk, causal) == INV, (Nq, Nk, causal)
        assert b(Nq, Nk, causal) == INV, (Nq, Nk, causal)
    for Nq, Nk, causal in ((128, 256, 1), (1, 4096, 1), (300, 7, 0), (7, 300, 0), (64, 64, 1)):
        assert f(Nq, Nk, causal) == NODEV, (Nq, Nk, causal)
        assert b(Nq, Nk, causal) == NODEV, (Nq, Nk, causal)
    assert f(0, 100, 1) == OK and f(0, 0, 0) == OK and f(8, 8, 1, B=0) == OK
    assert b(0, 0, 0) == OK and b(8, 8, 1, B=0) == OK
    assert b(0, 100, 1) == NODEV  # zeroes dk, dv on the device
    assert L.fa_bwd_ex(A, A, A, A, A, A, A, A, None, 1, 4, 2, 0, 100, 64, sc, 0, A, 0,
                       None) == INV  # ... which must then be valid pointers


def test_key_tile_argument(L):
    """fa_fwd_tiled takes 64- or 128-key tiles; other sizes are refused before
    any device work, valid ones pass validation (and stop at the device)."""
    import io_aware_exact_10_gb300 as fa
    sc = ctypes.c_float(0.125)
    f = lambda kt, d=64: L.fa_fwd_tiled(A, A, A, A, A, 1, 2, 2, 256, 256, d, sc, 1, kt, None)
    for kt in (0, 32, 96, 127, 256, -64):
        assert f(kt) == fa.FA_ERR_UNSUPPORTED, kt
    for kt in (64, 128):
        assert f(kt) == fa.FA_ERR_NO_DEVICE, kt
        assert f(kt, d=128) == fa.FA_ERR_NO_DEVICE, kt
    assert f(64, d=96) == fa.FA_ERR_UNSUPPORTED
