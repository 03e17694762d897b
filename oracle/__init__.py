"""fp64 CPU oracle for RLA-2 / RAPT causal ReLU linear attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links
this package: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference arm may use it. It shares no code with the CUDA path
(``relu_linear_attention_gb300``); the two meet only in the seeded input
generator, which holds none of the method's arithmetic.

The oracle is the plain quadratic definition of the method, in float64, with a
library matmul as its only building block. Sources (titles of the pages):

* "线性注意力家族：RLA / RAPT / RLA-2 与 GPU 落地" (neuralnet.cpp,
  docs/development/08-rapt-algorithm.md): §1 (no 1/sqrt(d) scale, per-head
  RMSNorm on Q and K, RoPE before ReLU), §2.1 (original RLA with the L2
  denominator, eps 1e-6), §2.2 (non-negative score, causal state reset at
  document boundaries), §3 (RLA-2 core formula, eps 1e-4), §4.1 (inclusive
  prefix i <= t within the same document), §4.2 (forward_step: features,
  update the state first, then read out).
  §4.1 also fixes the non-causal (bidirectional) mode: the same sums taken over the
  whole document, one constant for every query.
* ruDNN README (docs.rs ruDNN 0.1.93), §7: RMSNorm statistics in fp32 over the
  last axis, gamma an fp32 vector, epsilon finite and positive; §8: fp32
  initial/final state per sequence, never overwritten in place.
* candle "05-nn/layers" notes, normalisation section (RMSNorm is LayerNorm
  without mean subtraction and without bias) and rotary_emb section (pairing
  of dimensions 2i and 2i+1 for the interleaved variant).

Pins. Every function here is checked, in tests marked ``not gpu``, against
facts fixed by the pages and by mathematics rather than against itself:
quadratic form == recurrence, exact zeros for disjoint positive supports,
weights in [0, 1) with v == 1, convex-hull bounds, RoPE norm preservation and
relative-position property, RMSNorm scale invariance and norm identity, the
L = 1 and constant-v closed forms, linearity in v, the L2 identity
sum(s^2) = q'^T (K'^T K') q', varlen == per-document dense runs, decode ==
last prefill row, bidirectional == causal on the last row and invariant under
any reordering of the keys, and an independent pure-Python brute force on L <= 16.
The causal L2 form (rla_l2_causal*) is pinned by brute force, the recurrence
with the A = sum k'k'^T state, the last row = the non-causal L2 row, homogeneity
of degree 0 in q' (up to eps), the v == 1 bound sqrt(t+1) and per-document runs.
The layer (rapt_layer: projections, attention, output projection) is pinned by
its special cases: identity projections give the attention itself, zero W_v or
W_q give exact zeros (which fixes the q | k | v row order), and a permutation
W_o permutes the output columns.
The backward (rla2_bwd.py, gradients of sum dout . out) is pinned by central
finite differences of the forward oracle and of the brute force, Euler's
identity in v, the RMSNorm scale identity, the RoPE adjoint, shared gains =
sum over heads, and varlen == per-document dense runs.
The RoPE frequency schedule theta_j = base^(-2j/d) is the textbook one; the
pages name the base and the pairing but print no frequency formula, so the
schedule is pinned only through its properties (pair 0 turns by exactly p
radians, the ratio between neighbouring frequencies is constant).
"""

from .rla2 import (  # noqa: F401
    rmsnorm,
    rope_adjacent,
    relu,
    features,
    rla2_causal_doc,
    rla2_recurrent_doc,
    rla2_prefill,
    rla2_varlen,
    rla2_decode_step,
    rla2_decode_from_history,
    rla2_bidir_doc,
    rla2_bidir,
    rla2_bidir_varlen,
    rla_l2,
    rla_l2_causal_doc,
    rla_l2_causal_recurrent_doc,
    rla_l2_causal,
    rla_l2_causal_varlen,
    linear,
    rapt_layer,
    relative_error,
)
from .rla2_bwd import (  # noqa: F401
    relu_bwd,
    rope_adjacent_bwd,
    rmsnorm_bwd,
    features_bwd,
    rla2_causal_doc_bwd,
    rla2_prefill_bwd,
    rla2_varlen_bwd,
)
