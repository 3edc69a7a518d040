"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no attention arithmetic: it only draws random tensors.  Both
the CUDA path and the fp64 oracle are fed from it, so the oracle never sees a
value produced by the GPU.

Recipe (the same for every workload): one CPU ``torch.Generator`` seeded with
``seed`` draws Q, K, V and dO, in that order, as fp32 N(0, 1) tensors of shape
[B, H, N, d] (K and V with ``H_kv`` heads when the workload groups key/value
heads, and ``N_k`` rows when the keys outnumber or undercount the queries);
Q and K are multiplied by ``qk_std``; when ``boost_every`` is set,
key rows j with (j + 1) % boost_every == 0 (the 97th, 194th, ... row of each
head, counting from one) are multiplied by ``boost``; then every tensor is
rounded to bf16 (round to nearest even).  The default scale is 1/sqrt(d).

Block-sparse workloads add a block mask over 128 x 128 (query, key) blocks,
built by ``block_mask`` from the pattern string "localW_globalG_randomP":
block (i, j) is kept when |i - j| <= W (a local band), or i < G or j < G
(global blocks that see and are seen by all), or a uniform draw from a
numpy generator seeded with ``seed`` falls below P (random blocks).
"""
from __future__ import annotations

import math
import re
from dataclasses import dataclass

import numpy as np
import torch

BLOCK = 128  # rows and keys per block of a block mask


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    qk_std: float = 1.0
    boost_every: int = 0
    boost: float = 1.0
    seed: int = 0
    H_kv: int = 0  # key/value heads (0: one per query head)
    N_k: int = 0   # keys per head (0: N, as many as query rows)
    block_pattern: str = ""  # block-sparse pattern (see the module docstring); "" = dense

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    @property
    def kv_len(self) -> int:
        return self.N_k or self.N

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def fwd_flops(self) -> float:
        """Two contractions over the (query, key) pairs, 2 flop/MAC: 4*B*H*N*N_k*d,
        with N*N_k - N^2/2 pairs when causal (N^2/2 for N_k = N).  Block-sparse:
        the exact number of visible pairs in the kept blocks."""
        if self.block_pattern:
            pairs = visible_pairs(block_mask(self), self.N, self.kv_len, self.causal)
        else:
            pairs = self.N * self.kv_len - (self.N * self.N / 2 if self.causal else 0)
        return 4.0 * self.B * self.H * pairs * self.d

    def bwd_flops(self) -> float:
        """Five N^2 d contractions in the backward: 2.5x the forward."""
        return 2.5 * self.fwd_flops()


# The workloads the library is measured and checked on.
SINGLE_HEAD = Workload("single_head_N128_d64", 1, 1, 128, 64, causal=False)
GPT2_MEDIUM = Workload("gpt2_medium_B64_H16_N1024_d64", 64, 16, 1024, 64, causal=False)
GPT2_MEDIUM_CAUSAL = Workload("gpt2_medium_B64_H16_N1024_d64_causal", 64, 16, 1024, 64,
                              causal=True)
LONG_CAUSAL = Workload("long_causal_B4_H32_N8192_d128", 4, 32, 8192, 128, causal=True)
STRESS_CAUSAL = Workload("stress_B8_H16_N4096_d128_causal", 8, 16, 4096, 128, causal=True,
                         qk_std=4.0, boost_every=97, boost=8.0)
STRESS = Workload("stress_B8_H16_N4096_d128", 8, 16, 4096, 128, causal=False,
                  qk_std=4.0, boost_every=97, boost=8.0)
# grouped-query attention of current decoder models: 32 query heads on 8
# key/value heads
GQA_CAUSAL = Workload("gqa_B2_H32_Hkv8_N4096_d128_causal", 2, 32, 4096, 128, causal=True, H_kv=8)
# a prefill chunk: 1024 new queries after 7168 earlier positions (8192 keys),
# grouped heads as above
PREFILL_CHUNK = Workload("prefill_B4_H32_Hkv8_Nq1024_Nk8192_d128_causal", 4, 32, 1024, 128,
                         causal=True, H_kv=8, N_k=8192)

# block-sparse: local band of 3 blocks each side, one global block row and
# column, 5 % random blocks (BigBird-like; about 12 % of the blocks kept)
SPARSE_LOCAL_GLOBAL = Workload("sparse_B4_H16_N16384_d128_local3_global1_random5pct", 4, 16, 16384,
                               128, causal=False, block_pattern="local3_global1_random0.05")

SWEEP_N = (512, 1024, 2048, 4096, 8192, 16384, 32768)
SWEEP_D = (64, 128)


def sweep(N: int, d: int, causal: bool = True) -> Workload:
    """Sequence-length sweep point: H=16, B*N = 65536 tokens."""
    return Workload(f"sweep_N{N}_d{d}" + ("_causal" if causal else ""),
                    65536 // N, 16, N, d, causal=causal)


def block_mask(w: Workload) -> np.ndarray:
    """uint8 [ceil(N/128), ceil(N_k/128)] block mask of a block-sparse workload."""
    m = re.fullmatch(r"local(\d+)_global(\d+)_random([0-9.]+)", w.block_pattern)
    if not m:
        raise ValueError(f"unknown block pattern {w.block_pattern!r}")
    W, G, P = int(m.group(1)), int(m.group(2)), float(m.group(3))
    nbq, nbk = -(-w.N // BLOCK), -(-w.kv_len // BLOCK)
    i, j = np.meshgrid(np.arange(nbq), np.arange(nbk), indexing="ij")
    keep = (np.abs(i - j) <= W) | (i < G) | (j < G)
    keep |= np.random.default_rng(w.seed).random((nbq, nbk)) < P
    return keep.astype(np.uint8)


def visible_pairs(bm: np.ndarray, Nq: int, Nk: int, causal: bool) -> int:
    """Number of (query, key) pairs a query sees under the block mask bm and,
    when causal, the rule key <= query + Nk - Nq."""
    total = 0
    off = Nk - Nq
    for bi, bj in zip(*np.nonzero(bm)):
        r0, r1 = bi * BLOCK, min((bi + 1) * BLOCK, Nq)
        c0, c1 = bj * BLOCK, min((bj + 1) * BLOCK, Nk)
        if not causal:
            total += (r1 - r0) * (c1 - c0)
        else:
            rows = np.arange(r0, r1)
            total += int(np.clip(rows + off + 1 - c0, 0, c1 - c0).sum())
    return int(total)


def make_inputs(w: Workload, device: str = "cpu", with_grad: bool = True):
    """Draw (q, k, v, dO) as bf16 [B, H, N, d] tensors following the recipe
    (k, v: [B, H_kv, N_k, d])."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    out = []
    names = ("q", "k", "v", "dO") if with_grad else ("q", "k", "v")
    for name in names:
        heads, rows_n = (w.kv_heads, w.kv_len) if name in ("k", "v") else (w.H, w.N)
        t = torch.randn((w.B, heads, rows_n, w.d), generator=g, dtype=torch.float32)
        if name in ("q", "k") and w.qk_std != 1.0:
            t.mul_(w.qk_std)
        if name == "k" and w.boost_every:
            rows = torch.arange(rows_n)
            sel = ((rows + 1) % w.boost_every) == 0
            t[:, :, sel, :] *= w.boost
        out.append(t.to(torch.bfloat16).to(device))
    return tuple(out)


WORKLOADS = {w.name: w for w in (SINGLE_HEAD, GPT2_MEDIUM, GPT2_MEDIUM_CAUSAL, LONG_CAUSAL,
                                  STRESS_CAUSAL, STRESS, GQA_CAUSAL, PREFILL_CHUNK,
                                  SPARSE_LOCAL_GLOBAL)}
WORKLOADS.update({sweep(N, d).name: sweep(N, d) for N in SWEEP_N for d in SWEEP_D})
# short aliases
WORKLOADS.update({"gpt2_medium": GPT2_MEDIUM, "gpt2_medium_causal": GPT2_MEDIUM_CAUSAL,
                  "long_causal": LONG_CAUSAL, "stress": STRESS, "stress_causal": STRESS_CAUSAL,
                  "single_head": SINGLE_HEAD, "gqa_causal": GQA_CAUSAL,
                  "prefill_chunk": PREFILL_CHUNK, "sparse_local_global": SPARSE_LOCAL_GLOBAL})


def make_inputs_on_device(w: Workload, device, with_grad: bool = True):
    """The same recipe drawn by a seeded generator on `device` (a different
    random stream than make_inputs; used where only timing matters and the
    host-side draw of a large workload would dominate)."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    out = []
    for name in (("q", "k", "v", "dO") if with_grad else ("q", "k", "v")):
        heads, rows_n = (w.kv_heads, w.kv_len) if name in ("k", "v") else (w.H, w.N)
        t = torch.randn((w.B, heads, rows_n, w.d), generator=g, dtype=torch.float32,
                        device=device)
        if name in ("q", "k") and w.qk_std != 1.0:
            t.mul_(w.qk_std)
        if name == "k" and w.boost_every:
            rows = torch.arange(rows_n, device=device)
            t[:, :, ((rows + 1) % w.boost_every) == 0, :] *= w.boost
        out.append(t.to(torch.bfloat16))
    return tuple(out)


def random_bf16(shape, seed: int, std: float = 1.0, device: str = "cpu"):
    """One bf16 tensor drawn N(0, std^2) from its own seeded CPU generator."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, dtype=torch.float32) * std
    return t.to(torch.bfloat16).to(device)
