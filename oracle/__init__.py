"""CPU oracle for speculative-decoding verify attention and speculative sampling.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU
baseline leg may import or run anything in this package.  The library under
``speculative_decoding_verify_attn_gb300`` never imports it, and this package imports nothing
from the library: the two share no code.  The only shared module is ``workloads`` (seeded
input generation, no arithmetic of the method).

Everything here is plain NumPy in float64, written from the definitions on the pages:

* "Guide to MagicDec: Fast Long-Context Speculative Decoding" (aifetchly) -- bounded
  circular-FIFO draft KV cache (Solution §1; Implementation Step 1), full-context verify
  (Solution §2), accept rule and residual (Solution §2 equations), verify flow (Step 3).
* "Speculative Decoding & Medusa Architecture" (zyekh) -- speculative sampling math (§2),
  expected accepted tokens per step (§1 formula block), tree attention with a 2D mask (§4).
* "Speculative Decoding in LLM Serving Systems" (elimelt, UW CSE 599K) -- the algorithm,
  accepting and rejecting (and the rollback of rejected tokens' K/V, ``commit.py``), 1 .. gamma+1
  tokens per round, tree attention over ancestors (Tree-based variants).

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms, invariants,
brute force and hand-worked fixtures (``tests/golden/``), not against itself.
"""

from . import attn, commit, lmhead, sample  # noqa: F401
