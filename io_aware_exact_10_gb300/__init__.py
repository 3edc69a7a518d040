"""GB300 (sm_103a) exact softmax attention, computed FlashAttention-style.

The compute path is the C-ABI library ``libfa_gb300.so`` (hand-written CUDA
for sm_103a: TMA, mbarriers, tcgen05 MMA with TMEM accumulators).  This
package holds the ctypes binding (``binding``, same names as ``include/fa.h``),
the in-tree build step (``build``) and the seeded input generators
(``workloads``).  PyTorch is used only to allocate device memory and to name
streams.

``forward`` and ``backward`` are conveniences that allocate the outputs with
torch on the inputs' device and call ``fa_fwd_ex`` / ``fa_bwd_ex`` (which equal
``fa_fwd`` / ``fa_bwd`` when k and v have as many heads and rows as q).
"""
from __future__ import annotations

import math

from .binding import (  # noqa: F401
    FA_ERR_DEVICE,
    FA_ERR_INVALID_ARG,
    FA_ERR_LAUNCH,
    FA_ERR_NO_DEVICE,
    FA_ERR_TIMEOUT,
    FA_ERR_UNSUPPORTED,
    FA_OK,
    FAError,
    fa_bwd,
    fa_bwd_ex,
    fa_bwd_gqa,
    fa_bwd_noalloc,
    fa_bwd_workspace_size,
    fa_device_error_word,
    fa_fwd,
    fa_fwd_ex,
    fa_fwd_gqa,
    fa_last_device_error,
    fa_set_wait_timeout_ns,
    fa_strerror,
    fa_version,
    lib,
)


def _shape(q):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(int(x) for x in q.shape)


def forward(q, k, v, scale=None, causal=False, stream=None):
    """O, LSE for bf16 [B, H, N_q, d] q and [B, H_kv, N_k, d] k, v CUDA tensors
    (outputs allocated with torch).  H_kv < H: grouped key/value heads;
    N_k != N_q: causal aligns the last query with the last key."""
    import torch
    B, H, N, d = _shape(q)
    _, H_kv, N_k, _ = _shape(k)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fwd_ex(q, k, v, o, lse, B, H, H_kv, N, N_k, d, scale, causal, stream)
    return o, lse


def backward(q, k, v, o, lse, dO, scale=None, causal=False, stream=None, workspace=None):
    """dQ, dK, dV for the forward that produced (o, lse)."""
    import torch
    B, H, N, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _, H_kv, N_k, _ = _shape(k)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    fa_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N, N_k, d, scale, causal, workspace,
              workspace.numel() * workspace.element_size(), stream)
    return dq, dk, dv
