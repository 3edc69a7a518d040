"""Plain fp64 CPU oracle for exact softmax attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library's product path never does, and the
two share no code: the oracle is plain C (``attention_oracle.c``) loaded with
ctypes, and the CUDA path is a separate shared library.

Parity status of each function (what pins it, in ``tests/test_oracle_pins.py``):

* ``attn_fwd`` / ``attn_fwd_rows`` -- pinned: hand-computed four-score example,
  closed forms (identical keys, causal row 0, Q = 0, dominant key), rows of P
  summing to one, an independent blocked online-softmax recomputation, and
  torch's CPU ``scaled_dot_product_attention`` in fp64.
* ``attn_bwd`` -- pinned: central finite differences of the forward on tiny
  shapes, exact gradient invariants, and torch autograd in fp64.
* ``attn_bwd_rows`` (dq of chosen query rows, dk and dv of chosen key rows of
  one head) -- pinned: the full ``attn_bwd`` on those rows, and torch
  autograd in fp64 on those rows, with equal and unequal lengths.

Planted mistakes (``tests/test_oracle_mutants.py``) check that the pins catch
a dropped term, a wrong sign, a wrong index or a transposed operand.
"""
from .oracle import (  # noqa: F401
    OracleLib,
    attn_bwd,
    attn_bwd_rows,
    attn_fwd,
    attn_fwd_rows,
    build,
    compile_c,
    default,
    num_threads,
    SOURCE,
)
