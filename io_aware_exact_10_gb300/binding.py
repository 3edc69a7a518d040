"""Thin ctypes binding of the C ABI in ``include/fa.h``.

Argument marshalling only: every step of the attention path runs in the CUDA
kernels of ``libfa_gb300.so``.  The functions keep the C names.  Tensor
arguments may be torch tensors (their ``data_ptr()`` is passed) or raw device
addresses (ints).  There is no fallback: if the library has not been built,
loading it raises.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_LAUNCH = 3
FA_ERR_TIMEOUT = 4
FA_ERR_NO_DEVICE = 5
FA_ERR_DEVICE = 6

_lib = None


class FAError(RuntimeError):
    """A non-zero fa_status returned by the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({fa_strerror(status)})")


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -m io_aware_exact_10_gb300.build` "
                "(the library has no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_fwd.restype = i
        L.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_fwd_gqa.restype = i
        L.fa_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        L.fa_fwd_ex.restype = i
        L.fa_bwd_workspace_size.argtypes = [i, i, i, i]
        L.fa_bwd_workspace_size.restype = sz
        L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
        L.fa_bwd.restype = i
        L.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz,
                                 vp]
        L.fa_bwd_gqa.restype = i
        L.fa_bwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz,
                                vp]
        L.fa_bwd_ex.restype = i
        L.fa_fwd_sparse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp]
        L.fa_fwd_sparse.restype = i
        L.fa_fwd_tiled.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
        L.fa_fwd_tiled.restype = i
        L.fa_bwd_sparse.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i,
                                    vp, vp, sz, vp]
        L.fa_bwd_sparse.restype = i
        L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_bwd_noalloc.restype = i
        L.fa_fwd_host_device_bytes.argtypes = [i, i, i, i, i, i]
        L.fa_fwd_host_device_bytes.restype = sz
        L.fa_fwd_bwd_host_device_bytes.argtypes = [i, i, i, i, i, i, i]
        L.fa_fwd_bwd_host_device_bytes.restype = sz
        L.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp, sz, i, vp]
        L.fa_fwd_host.restype = i
        L.fa_fwd_bwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i,
                                      vp, vp, sz, i, vp]
        L.fa_fwd_bwd_host.restype = i
        L.fa_last_device_error.argtypes = [vp]
        L.fa_last_device_error.restype = i
        L.fa_device_error_word.argtypes = [vp]
        L.fa_device_error_word.restype = ctypes.c_ulonglong
        L.fa_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
        L.fa_set_wait_timeout_ns.restype = None
        L.fa_strerror.argtypes = [i]
        L.fa_strerror.restype = ctypes.c_char_p
        L.fa_version.argtypes = []
        L.fa_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    """A torch stream, a raw cudaStream_t (int) or None (torch's current stream)."""
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != FA_OK:
        raise FAError(status, where)


def fa_strerror(status: int) -> str:
    return lib().fa_strerror(int(status)).decode()


def fa_version() -> str:
    return lib().fa_version().decode()


def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream=None, check=True) -> int:
    """fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> status."""
    s = lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H), int(N),
                     int(d), float(scale), int(causal), _stream(stream))
    if check:
        _check(s, "fa_fwd")
    return s


def fa_fwd_gqa(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, stream=None,
               check=True) -> int:
    """fa_fwd_gqa(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal, stream) -> status:
    k, v have H_kv heads; query head h uses key/value head h // (H // H_kv)."""
    s = lib().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                         int(H_kv), int(N), int(d), float(scale), int(causal), _stream(stream))
    if check:
        _check(s, "fa_fwd_gqa")
    return s


def fa_fwd_ex(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, scale, causal, stream=None,
              check=True) -> int:
    """fa_fwd_ex(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, scale, causal, stream) -> status:
    q, o have N_q rows, k, v N_k; causal aligns the last query with the last key."""
    s = lib().fa_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                        int(H_kv), int(N_q), int(N_k), int(d), float(scale), int(causal),
                        _stream(stream))
    if check:
        _check(s, "fa_fwd_ex")
    return s


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(lib().fa_bwd_workspace_size(int(B), int(H), int(N), int(d)))


def fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, workspace,
           workspace_bytes, stream=None, check=True) -> int:
    """fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal,
    workspace, workspace_bytes, stream) -> status."""
    s = lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                     _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d), float(scale),
                     int(causal), _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check:
        _check(s, "fa_bwd")
    return s


def fa_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N, d, scale, causal, workspace,
               workspace_bytes, stream=None, check=True) -> int:
    """fa_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N, d, scale, causal,
    workspace, workspace_bytes, stream) -> status: dk, dv (H_kv heads) sum
    over each key/value head's query heads."""
    s = lib().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                         _ptr(dk), _ptr(dv), int(B), int(H), int(H_kv), int(N), int(d),
                         float(scale), int(causal), _ptr(workspace), int(workspace_bytes),
                         _stream(stream))
    if check:
        _check(s, "fa_bwd_gqa")
    return s


def fa_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N_q, N_k, d, scale, causal,
              workspace, workspace_bytes, stream=None, check=True) -> int:
    """fa_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N_q, N_k, d, scale, causal,
    workspace, workspace_bytes, stream) -> status: the counterpart of fa_fwd_ex;
    the workspace is fa_bwd_workspace_size(B, H, N_q, d) bytes."""
    s = lib().fa_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                        _ptr(dk), _ptr(dv), int(B), int(H), int(H_kv), int(N_q), int(N_k),
                        int(d), float(scale), int(causal), _ptr(workspace),
                        int(workspace_bytes), _stream(stream))
    if check:
        _check(s, "fa_bwd_ex")
    return s


def fa_fwd_sparse(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, scale, causal, block_mask,
                  stream=None, check=True) -> int:
    """fa_fwd_sparse(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, scale, causal, block_mask,
    stream) -> status: block_mask is a device uint8 [ceil(N_q/128), ceil(N_k/128)]."""
    s = lib().fa_fwd_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                            int(H_kv), int(N_q), int(N_k), int(d), float(scale), int(causal),
                            _ptr(block_mask), _stream(stream))
    if check:
        _check(s, "fa_fwd_sparse")
    return s


def fa_fwd_tiled(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, scale, causal, key_tile,
                 stream=None, check=True) -> int:
    """fa_fwd_tiled(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, scale, causal, key_tile,
    stream) -> status: fa_fwd_ex with K/V tiles of key_tile (64 or 128) keys."""
    s = lib().fa_fwd_tiled(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                           int(H_kv), int(N_q), int(N_k), int(d), float(scale), int(causal),
                           int(key_tile), _stream(stream))
    if check:
        _check(s, "fa_fwd_tiled")
    return s


def fa_bwd_sparse(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N_q, N_k, d, scale, causal,
                  block_mask, workspace, workspace_bytes, stream=None, check=True) -> int:
    """fa_bwd_sparse(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N_q, N_k, d, scale, causal,
    block_mask, workspace, workspace_bytes, stream) -> status."""
    s = lib().fa_bwd_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                            _ptr(dk), _ptr(dv), int(B), int(H), int(H_kv), int(N_q), int(N_k),
                            int(d), float(scale), int(causal), _ptr(block_mask),
                            _ptr(workspace), int(workspace_bytes), _stream(stream))
    if check:
        _check(s, "fa_bwd_sparse")
    return s


def fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, stream=None,
                   check=True) -> int:
    """fa_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal,
    stream) -> status: the backward for callers that cannot allocate a
    workspace; its scratch is a fixed 64 MiB array inside the library."""
    s = lib().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq),
                             _ptr(dk), _ptr(dv), int(B), int(H), int(N), int(d), float(scale),
                             int(causal), _stream(stream))
    if check:
        _check(s, "fa_bwd_noalloc")
    return s


def fa_fwd_host_device_bytes(B, H, H_kv, N_q, N_k, d) -> int:
    return int(lib().fa_fwd_host_device_bytes(int(B), int(H), int(H_kv), int(N_q), int(N_k),
                                              int(d)))


def fa_fwd_bwd_host_device_bytes(B, H, H_kv, N_q, N_k, d, chunks=0) -> int:
    return int(lib().fa_fwd_bwd_host_device_bytes(int(B), int(H), int(H_kv), int(N_q), int(N_k),
                                                  int(d), int(chunks)))


def fa_fwd_host(q, k, v, o, lse, B, H, H_kv, N_q, N_k, d, scale, causal, dev, dev_bytes,
                chunks=0, stream=None, check=True, block_mask=None) -> int:
    """fa_fwd_host(...) -> status: q, k, v, o, lse are HOST buffers (torch CPU
    tensors, ideally pinned, or raw addresses); dev is the device staging area;
    block_mask an optional DEVICE block mask (as for fa_fwd_sparse)."""
    s = lib().fa_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(H),
                          int(H_kv), int(N_q), int(N_k), int(d), float(scale), int(causal),
                          _ptr(block_mask), _ptr(dev), int(dev_bytes), int(chunks),
                          _stream(stream))
    if check:
        _check(s, "fa_fwd_host")
    return s


def fa_fwd_bwd_host(q, k, v, dO, o, lse, dq, dk, dv, B, H, H_kv, N_q, N_k, d, scale, causal,
                    dev, dev_bytes, chunks=0, stream=None, check=True, block_mask=None) -> int:
    """fa_fwd_bwd_host(...) -> status: forward and backward with every tensor in
    HOST memory; copies of one head group overlap the kernels of the others.
    block_mask: optional DEVICE block mask (as for fa_fwd_sparse)."""
    s = lib().fa_fwd_bwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(o), _ptr(lse),
                              _ptr(dq), _ptr(dk), _ptr(dv), int(B), int(H), int(H_kv), int(N_q),
                              int(N_k), int(d), float(scale), int(causal), _ptr(block_mask),
                              _ptr(dev), int(dev_bytes), int(chunks), _stream(stream))
    if check:
        _check(s, "fa_fwd_bwd_host")
    return s


def fa_last_device_error(stream=None) -> int:
    return int(lib().fa_last_device_error(_stream(stream)))


def fa_device_error_word(stream=None) -> int:
    return int(lib().fa_device_error_word(_stream(stream)))


def fa_set_wait_timeout_ns(ns: int) -> None:
    lib().fa_set_wait_timeout_ns(int(ns))
