"""CPU oracle of the DeepSeek-style Mixture-of-Experts decode layer.

TEST INFRASTRUCTURE.  Only the tests, the smoke check in __graft_entry__ and
the CPU-baseline / reference leg of bench.py may import or run anything in
this package.  The product path (moe_expert_layer_07_gb300) never does, and
this package imports nothing from it: the two share no code.

Each step is written from its definition, plainly and slowly: numpy in
fp64 (fp32 where a quantisation or selection decision is taken, in the
precision the decision is defined in), with three C loops in moe_oracle.c
for the sizes numpy cannot reach.  Every function cites the passage of the
pages it follows; readings taken where the pages are silent are listed in
each module's docstring.

Parity pinning: each function is pinned by tests/test_oracle_*.py against
something other than itself (closed forms, brute force, library routines
used as checks, invariants).  Absolute layer outputs have no worked example
on the pages; they are pinned through the dense-FFN closed form of a
one-expert layer and the invariants listed in the tests.

Modules:
  quant    e4m3 and bf16 rounding, per-128 FP8 group quantisation
  routing  gate logits (fixed order), sigmoid/softmax group-limited top-k
  permute  slot -> per-expert row permutation and its offsets
  layer    expert SwiGLU FFN, grouped GEMM, combine, the whole layer
  balance  exhaustive balanced partition (tiny expert counts)
  affinity co-activation matrix, affinity-aware placement optimum (tiny E)
"""
from . import affinity, balance, layer, permute, quant, routing  # noqa: F401
from ._clib import build, num_threads, set_num_threads  # noqa: F401
