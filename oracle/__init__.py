"""CPU oracle for the decoder-only transformer forward pass (test infrastructure).

This package is the plain, slow, obviously correct statement of what the
forward pass computes, in float64 numpy over the same bf16-rounded seeded
weights the CUDA library reads. It exists to check the CUDA library and is
test infrastructure only: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline arm may import it; the library never does, and the
library shares no code, table or helper with it.

Every function cites the passage of the pages it follows:

* "N7 · model/forward-parity" (fak proof ledger), Theorem 1 and Theorem 2 --
  the forward pass (embedding, decoder stack with RMSNorm, RoPE, causal GQA
  attention, SwiGLU, residuals, final norm, tied head), per-layer hidden
  slots, per-position argmax, cached-session prefill and greedy generation,
  and the family axes (QK-norm, sliding window, sandwich norm, llama3 RoPE
  scaling).
* "pegainfer issue #878" (Gemma3-style local/global tower), Description,
  Proposed Plan and Acceptance Criteria -- the scaled embedding, the layer
  map dispatch, the final-logit softcap and the window-edge gate.
* "N9 · metalgemm", Theorem 1 -- the GEMM Y = X·Wᵀ against a float64
  accumulated triple loop, and the op chain of a Llama decode.

Readings where the pages are silent (RoPE pairing, GELU form, Gemma's RoPE
bases, eps values, window boundary) are listed in the module docstring of
``oracle.forward``. Parity of the whole forward on full-size models is pinned
only by the per-op pins and by a brute-force re-derivation on tiny models; the
pages print no worked values reproducible without their trained checkpoints.
"""
from .forward import *  # noqa: F401,F403
