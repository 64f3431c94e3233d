"""CPU oracle for the sparse-KV decode step -- TEST INFRASTRUCTURE ONLY.

Plain, slow numpy code (fp64 wherever the pages leave the precision open)
that restates, stage by stage, what one layer of a predictive sparse-KV decode
step computes.  Only the test-suite, the package smoke check and the
benchmark's CPU-baseline leg may import it; the product path never does, and
it shares no code with the CUDA library.

Sources (web pages, cited by title and section / equation / figure):

* "DualDecoder: Accelerate Long Context LLM Inference by Predictive Prefetch"
  -- §2.2 (chunk landmarks), §4.1 (retrieval index from the token and the
  landmarks; speculative-token prediction), §5.2 (dual-token decoding),
  §5.4 and Fig. 11 (two-layer ping-pong buffer, GPU-side sparse assembly).
* "OasisKV" summary -- eqs. (1)-(3) (KV footprint, maximum batch, per-step
  byte budget); Methodology (top-K per KV head; normal and draft queries
  share one HBM working set).
* "Adaptive DHiSparse: Speculative Decoding over a Load-Adaptive KV
  Hierarchy" -- Fig. 2 (resolver: resident tiers first, host copy for
  misses), Fig. 3 (the selections of several queries resolved together so
  a chunk picked by several queries is fetched once; attention uses each query's own
  selection).

Every function is pinned by the tests in ``tests/test_oracle_pins.py``
against closed forms, library routines for special cases, brute force on
tiny inputs and the worked numbers printed on the pages.
"""
from .sparse_kv import *  # noqa: F401,F403
