"""ctypes wrapper around the fp64 C oracle (``attention_oracle.c``).

Test infrastructure only: see the package docstring.  Arrays are numpy fp64,
shaped [..., rows, d] (flattened to heads): q, o, dO, dq have Nq rows, k, v,
dk, dv Nk rows; lse is [..., Nq].  With causal masking and Nq != Nk the last
query row is aligned with the last key (key j visible to query i iff
j <= i + Nk - Nq), which needs Nk >= Nq.  An optional block mask
[ceil(Nq/bq), ceil(Nk/bk)] (nonzero = kept, shared by every head) hides the
keys of the blocks it zeroes; a row left with no key gets o = 0, lse = -inf.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "attention_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")


def compile_c(src: str, out: str) -> str:
    """gcc -O2 (with OpenMP when the compiler has it) into a shared object."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so``."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_c(SOURCE, _LIB_PATH)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _heads(a: np.ndarray):
    N, d = a.shape[-2], a.shape[-1]
    return a.reshape(-1, N, d), N, d


def _kv_rows(Nq: int, kh: np.ndarray, vh: np.ndarray, d: int, causal: bool) -> int:
    """Key count Nk of k, v (equal shapes, same d as q; Nk >= Nq when causal)."""
    if kh.shape != vh.shape or kh.shape[-1] != d:
        raise ValueError(f"k {kh.shape} and v {vh.shape} must match and have d={d}")
    Nk = kh.shape[1]
    if causal and Nk < Nq:
        raise ValueError(f"causal attention needs Nk >= Nq (Nq={Nq}, Nk={Nk})")
    return Nk


def _block_mask(block_mask, block, Nq: int, Nk: int):
    """(pointer, bq, bk, keep-alive array) for the C call; NULL when no mask."""
    if block_mask is None:
        return None, 1, 1, None
    bq, bk = (int(x) for x in block)
    if bq < 1 or bk < 1:
        raise ValueError(f"block sizes must be >= 1, got {block}")
    m = np.ascontiguousarray(np.asarray(block_mask) != 0, dtype=np.uint8)
    want = (-(-Nq // bq), -(-Nk // bk))
    if m.shape != want:
        raise ValueError(f"block mask shape {m.shape} != {want} for Nq={Nq}, Nk={Nk}, block={block}")
    return m.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)), bq, bk, m


def _group(BH: int, BHk: int, BHv: int) -> int:
    """Query heads per key/value head (1 for standard multi-head)."""
    if BHk != BHv or BHk < 1 or BH % BHk != 0:
        raise ValueError(f"k, v heads ({BHk}, {BHv}) must be equal and divide q heads ({BH})")
    return BH // BHk


class OracleLib:
    """The oracle's entry points, bound to one compiled shared object."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int)
        ci, cd = ctypes.c_int, ctypes.c_double
        bp = ctypes.POINTER(ctypes.c_ubyte)
        lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, ci, ci, ci, ci, cd, ci, ci, bp, ci, ci]
        lib.oracle_attn_fwd.restype = None
        lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp,
                                        ci, ci, ci, ci, cd, ci, ci, bp, ci, ci]
        lib.oracle_attn_bwd.restype = None
        lib.oracle_attn_fwd_rows.argtypes = [dp, dp, dp, ip, ci, dp, dp,
                                             ci, ci, ci, cd, ci]
        lib.oracle_attn_fwd_rows.restype = None
        lib.oracle_attn_bwd_rows.argtypes = [dp, dp, dp, dp, ip, ci, ip, ci, dp, dp, dp,
                                             ci, ci, ci, cd, ci]
        lib.oracle_attn_bwd_rows.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ci
        self._lib = lib

    def num_threads(self) -> int:
        return int(self._lib.oracle_num_threads())

    def attn_fwd(self, q, k, v, scale: float, causal: bool, block_mask=None, block=(128, 128)):
        """o = softmax(scale * q k^T [causal]) v and lse (natural log), fp64.

        q: [..., Nq, d]; k, v: [..., Nk, d] with the same or a dividing
        number of heads (grouped key/value heads: query head h uses key/value
        head h // G over the flattened head axis).  block_mask: optional
        [ceil(Nq/bq), ceil(Nk/bk)] array, block = (bq, bk).  Returns (o
        shaped like q, lse shaped [..., Nq] like q's heads).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        lead = q.shape[:-2]
        qh, N, d = _heads(q)
        kh, _, _ = _heads(k)
        vh, _, _ = _heads(v)
        Nk = _kv_rows(N, kh, vh, d, causal)
        BH = qh.shape[0]
        group = _group(BH, kh.shape[0], vh.shape[0])
        bm, bq, bk, _keep = _block_mask(block_mask, block, N, Nk)
        o = np.empty_like(qh)
        lse = np.empty((BH, N), dtype=np.float64)
        self._lib.oracle_attn_fwd(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(o),
                                  _ptr(lse), BH, N, Nk, d, float(scale),
                                  int(bool(causal)), group, bm, bq, bk)
        return o.reshape(*lead, N, d), lse.reshape(*lead, N)

    def attn_bwd(self, q, k, v, dO, scale: float, causal: bool,
                 return_D: bool = False, block_mask=None, block=(128, 128)):
        """Gradients (dq, dk, dv) of L with dL/dO = dO, fp64.

        With ``return_D`` also returns D = rowsum(P * dP) shaped [..., Nq].
        k, v may have fewer heads and another length than q (see attn_fwd);
        dk, dv are shaped like k and sum over each key/value head's query
        heads.  block_mask, block: as for attn_fwd.
        """
        q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
        if dO.shape != q.shape:
            raise ValueError(f"dO {dO.shape} must be shaped like q {q.shape}")
        lead = q.shape[:-2]
        lead_kv = k.shape[:-2]
        qh, N, d = _heads(q)
        kh, _, _ = _heads(k)
        vh, _, _ = _heads(v)
        dOh, _, _ = _heads(dO)
        Nk = _kv_rows(N, kh, vh, d, causal)
        BH = qh.shape[0]
        group = _group(BH, kh.shape[0], vh.shape[0])
        dq = np.empty_like(qh)
        dk = np.empty_like(kh)
        dv = np.empty_like(kh)
        D = np.empty((BH, N), dtype=np.float64)
        bm, bq, bk, _keep = _block_mask(block_mask, block, N, Nk)
        self._lib.oracle_attn_bwd(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(dOh),
                                  _ptr(dq), _ptr(dk), _ptr(dv), _ptr(D),
                                  BH, N, Nk, d, float(scale), int(bool(causal)), group,
                                  bm, bq, bk)
        out = (dq.reshape(*lead, N, d), dk.reshape(*lead_kv, Nk, d),
               dv.reshape(*lead_kv, Nk, d))
        if return_D:
            return out + (D.reshape(*lead, N),)
        return out

    def attn_fwd_rows(self, q, k, v, rows, scale: float, causal: bool):
        """Forward for selected query rows of ONE head: q is [Nq, d], k, v
        are [Nk, d].

        Returns (o [R, d], lse [R]) for the rows listed in ``rows``.
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        N, d = q.shape
        Nk = _kv_rows(N, k[None], v[None], d, causal)
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        R = rows.shape[0]
        o = np.empty((R, d), dtype=np.float64)
        lse = np.empty((R,), dtype=np.float64)
        self._lib.oracle_attn_fwd_rows(
            _ptr(q), _ptr(k), _ptr(v),
            rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), R,
            _ptr(o), _ptr(lse), N, Nk, d, float(scale), int(bool(causal)))
        return o, lse

    def attn_bwd_rows(self, q, k, v, dO, qrows, krows, scale: float, causal: bool):
        """Backward for selected rows of ONE head: q, dO are [Nq, d], k, v
        are [Nk, d].

        Returns (dq [Rq, d] for the query rows ``qrows``, dk [Rk, d] and
        dv [Rk, d] for the key rows ``krows``), equal to those rows of
        attn_bwd's outputs.
        """
        q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
        N, d = q.shape
        if dO.shape != q.shape:
            raise ValueError(f"dO {dO.shape} must be shaped like q {q.shape}")
        Nk = _kv_rows(N, k[None], v[None], d, causal)
        qr = np.ascontiguousarray(np.asarray(qrows, dtype=np.int32))
        kr = np.ascontiguousarray(np.asarray(krows, dtype=np.int32))
        if qr.size and (qr.min() < 0 or qr.max() >= N):
            raise ValueError("query row out of range")
        if kr.size and (kr.min() < 0 or kr.max() >= Nk):
            raise ValueError("key row out of range")
        dq = np.empty((qr.shape[0], d), dtype=np.float64)
        dk = np.empty((kr.shape[0], d), dtype=np.float64)
        dv = np.empty((kr.shape[0], d), dtype=np.float64)
        ip = ctypes.POINTER(ctypes.c_int)
        self._lib.oracle_attn_bwd_rows(
            _ptr(q), _ptr(k), _ptr(v), _ptr(dO), qr.ctypes.data_as(ip), qr.shape[0],
            kr.ctypes.data_as(ip), kr.shape[0], _ptr(dq), _ptr(dk), _ptr(dv),
            N, Nk, d, float(scale), int(bool(causal)))
        return dq, dk, dv


_default = None


def default() -> OracleLib:
    global _default
    if _default is None:
        _default = OracleLib(build())
    return _default


def num_threads() -> int:
    return default().num_threads()


def attn_fwd(q, k, v, scale, causal, block_mask=None, block=(128, 128)):
    return default().attn_fwd(q, k, v, scale, causal, block_mask, block)


def attn_bwd(q, k, v, dO, scale, causal, return_D=False, block_mask=None, block=(128, 128)):
    return default().attn_bwd(q, k, v, dO, scale, causal, return_D, block_mask, block)


def attn_fwd_rows(q, k, v, rows, scale, causal):
    return default().attn_fwd_rows(q, k, v, rows, scale, causal)


def attn_bwd_rows(q, k, v, dO, qrows, krows, scale, causal):
    return default().attn_bwd_rows(q, k, v, dO, qrows, krows, scale, causal)
