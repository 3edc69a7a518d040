"""Host-memory entry points (fa_fwd_host, fa_fwd_bwd_host): the staging-area
size rule and the argument checks, which run before anything touches a device
(CPU only)."""
import ctypes

import pytest

from io_aware_exact_10_gb300 import build as fab


@pytest.fixture(scope="module")
def L():
    fab.build()
    import io_aware_exact_10_gb300 as fa
    return fa.lib()


def r256(x):
    return (x + 255) // 256 * 256


def staging_bytes(B, H, H_kv, N_q, N_k, d, chunks, backward):
    """The layout the header documents, restated: device copies of every
    tensor (each region rounded to 256 bytes; lse with 16 bytes of slack per
    possible group) and one backward workspace for the largest group."""
    qb, kb, lb = B * H * N_q * d * 2, B * H_kv * N_k * d * 2, B * H * N_q * 4
    total = r256(qb) + 2 * r256(kb) + r256(qb) + r256(lb + 16 * 64)
    if backward:
        n_kv = B * H_kv
        n = min(chunks if chunks > 0 else 8, 64, n_kv)
        per = -(-n_kv // n) * (H // H_kv)  # query heads of the largest group
        stats = per * (-(-N_q // 128)) * 256 * 4
        ws = r256(stats) + r256(per * N_q * d * 4)
        total += 2 * r256(qb) + 2 * r256(kb) + r256(ws)
    return total


@pytest.mark.parametrize("shape", [(2, 4, 2, 200, 200, 64), (1, 6, 3, 77, 301, 128),
                                   (64, 16, 16, 1024, 1024, 64), (3, 8, 1, 5, 9000, 128)])
@pytest.mark.parametrize("chunks", [0, 1, 3, 100])
def test_staging_bytes(L, shape, chunks):
    B, H, H_kv, N_q, N_k, d = shape
    assert L.fa_fwd_host_device_bytes(*shape) == staging_bytes(*shape, chunks, False)
    assert L.fa_fwd_bwd_host_device_bytes(*shape, chunks) == staging_bytes(*shape, chunks, True)


def test_staging_bytes_invalid_and_empty(L):
    assert L.fa_fwd_host_device_bytes(1, 4, 3, 128, 128, 64) == 0   # H_kv does not divide H
    assert L.fa_fwd_host_device_bytes(1, 4, 4, 128, 128, 96) == 0   # unsupported d
    assert L.fa_fwd_bwd_host_device_bytes(0, 4, 4, 128, 128, 64, 0) == 0
    assert L.fa_fwd_bwd_host_device_bytes(1, 4, 4, -1, 128, 64, 0) == 0


def test_argument_errors_before_any_device_call(L):
    import io_aware_exact_10_gb300 as fa
    INV, OK, NODEV = fa.FA_ERR_INVALID_ARG, fa.FA_OK, fa.FA_ERR_NO_DEVICE
    host = ctypes.create_string_buffer(64)
    H_ = ctypes.addressof(host)
    DEV = 1 << 20  # a 256-byte aligned address; nothing dereferences it here
    sc = ctypes.c_float(0.125)

    def fb(B=1, H=4, H_kv=2, Nq=128, Nk=128, d=64, causal=0, scale=sc, dev=DEV, nbytes=1 << 40,
           ptr=H_, dq=None, mask=None):
        dq = ptr if dq is None else dq
        return L.fa_fwd_bwd_host(ptr, ptr, ptr, ptr, ptr, ptr, dq, ptr, ptr, B, H, H_kv, Nq, Nk, d,
                                 scale, causal, mask, dev, nbytes, 0, None)

    def ff(B=1, H=4, H_kv=2, Nq=128, Nk=128, d=64, causal=0, dev=DEV, nbytes=1 << 40, ptr=H_,
           mask=None):
        return L.fa_fwd_host(ptr, ptr, ptr, ptr, ptr, B, H, H_kv, Nq, Nk, d, sc, causal, mask, dev,
                             nbytes, 0, None)

    # valid arguments reach the device lookup (none here)
    assert fb() == NODEV and ff() == NODEV
    # sizes, flags and scale, as for fa_fwd_ex
    for kw in (dict(H_kv=3), dict(d=96), dict(causal=2), dict(Nq=256, Nk=128, causal=1),
               dict(Nq=5, Nk=0), dict(Nq=-1), dict(scale=ctypes.c_float(0.0)),
               dict(scale=ctypes.c_float(float("nan")))):
        assert fb(**kw) == INV, kw
    for kw in (dict(H_kv=3), dict(d=96), dict(causal=2), dict(Nq=256, Nk=128, causal=1)):
        assert ff(**kw) == INV, kw
    # the staging area: null, misaligned or short
    assert fb(dev=None) == INV and fb(dev=DEV + 16) == INV
    assert fb(nbytes=L.fa_fwd_bwd_host_device_bytes(1, 4, 2, 128, 128, 64, 0) - 1) == INV
    assert ff(nbytes=L.fa_fwd_host_device_bytes(1, 4, 2, 128, 128, 64) - 1) == INV
    # a null host pointer for a tensor that has elements
    assert fb(ptr=None) == INV and ff(ptr=None) == INV
    assert fb(dq=0) == INV
    # a block mask is limited to 4096 blocks per side, as for fa_fwd_sparse
    big = 4096 * 128 + 1
    assert fb(Nq=big, Nk=big, mask=DEV) == INV and ff(Nq=128, Nk=big, mask=DEV) == INV
    assert fb(Nq=big, Nk=big) == NODEV and fb(mask=DEV) == NODEV
    # empty problems: nothing to do
    assert fb(B=0) == OK and fb(H=0) == OK and ff(B=0) == OK
