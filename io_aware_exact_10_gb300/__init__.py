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
    fa_bwd_sparse,
    fa_bwd_workspace_size,
    fa_device_error_word,
    fa_fwd,
    fa_fwd_bwd_host,
    fa_fwd_bwd_host_device_bytes,
    fa_fwd_ex,
    fa_fwd_gqa,
    fa_fwd_host,
    fa_fwd_host_device_bytes,
    fa_fwd_sparse,
    fa_fwd_tiled,
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


def _mask_arg(block_mask, N_q, N_k, device):
    """A contiguous device uint8 [ceil(N_q/128), ceil(N_k/128)] copy of block_mask."""
    import torch
    want = ((N_q + 127) // 128, (N_k + 127) // 128)
    if tuple(block_mask.shape) != want:
        raise ValueError(f"block mask shape {tuple(block_mask.shape)} != {want}")
    return (block_mask != 0).to(device=device, dtype=torch.uint8).contiguous()


def forward(q, k, v, scale=None, causal=False, stream=None, block_mask=None):
    """O, LSE for bf16 [B, H, N_q, d] q and [B, H_kv, N_k, d] k, v CUDA tensors
    (outputs allocated with torch).  H_kv < H: grouped key/value heads;
    N_k != N_q: causal aligns the last query with the last key; block_mask:
    [ceil(N_q/128), ceil(N_k/128)] tensor, nonzero keeps a 128 x 128 block."""
    import torch
    B, H, N, d = _shape(q)
    _, H_kv, N_k, _ = _shape(k)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if block_mask is None:
        fa_fwd_ex(q, k, v, o, lse, B, H, H_kv, N, N_k, d, scale, causal, stream)
    else:
        m = _mask_arg(block_mask, N, N_k, q.device)
        fa_fwd_sparse(q, k, v, o, lse, B, H, H_kv, N, N_k, d, scale, causal, m, stream)
    return o, lse


def backward(q, k, v, o, lse, dO, scale=None, causal=False, stream=None, workspace=None,
             block_mask=None):
    """dQ, dK, dV for the forward that produced (o, lse) (with the same
    block_mask, if any)."""
    import torch
    B, H, N, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _, H_kv, N_k, _ = _shape(k)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    wsb = workspace.numel() * workspace.element_size()
    if block_mask is None:
        fa_bwd_ex(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N, N_k, d, scale, causal, workspace,
                  wsb, stream)
    else:
        m = _mask_arg(block_mask, N, N_k, q.device)
        fa_bwd_sparse(q, k, v, o, lse, dO, dq, dk, dv, B, H, H_kv, N, N_k, d, scale, causal, m,
                      workspace, wsb, stream)
    return dq, dk, dv
