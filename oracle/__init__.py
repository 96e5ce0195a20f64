"""CPU oracle for the routed NVFP4 mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, calls or links
this package; only the tests, the smoke check and the CPU-baseline leg of the
benchmark do.  It shares no code with the CUDA path: it has its own NVFP4
encoder and decoder (``nvfp4``) and its own layer (``moe``), written in plain
numpy with fp64 arithmetic wherever the method does not fix a precision.

Sources (web pages; cited by title and section):

* PR #385 "feat(qwen4_exp): tensor parallelism for Qwen3.8-Flash-Next
  (offload backend)" -- section "What this adds": replicated router; NVFP4
  banks made of packed codes, 16-wide scale blocks and per-row globals;
  intermediate-axis bank slicing; ``routed + sigmoid(gate) * shared``
  combined before one reduce.  Section "Measurements / Correctness": the
  run-to-run divergence traced to bf16 atomics in the expert kernels.
* Issue #62 "Offloaded MoE ignores tensor parallelism: TP=2 is a regression,
  and the fix is not expert parallelism" -- section "What it touches":
  gate_up is [2I, H] with gate rows [0, I) and up rows [I, 2I), down is
  [H, I] and is sliced by columns; I/tp must stay a multiple of the block
  size.  Section "The fix that fits": sharding I makes the down projection
  produce partial sums.  First comment, "And the parts you predicted would be
  free were free": norm_topk_prob defaults to True and the router is
  replicated, so a plain SUM of the partials is exact.

Readings of points the pages leave open are listed in each function's
docstring.  Parity status: every function here is pinned by tests under
``tests/`` (closed forms, library routines, brute force, invariants and the
byte figures the pages print) except the activation-quantisation reading,
which is a stated design choice (parity unpinned by the pages).
"""

from . import nvfp4, moe  # noqa: F401
