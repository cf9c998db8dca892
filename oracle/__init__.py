"""CPU oracle for the speculative-decoding verification path.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
float64 restatement of what the verification path computes.  Only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm
may import it.  The product path (the CUDA library and its Python binding)
never imports or calls anything here, and this package imports nothing from
the product path.

Modules
-------
decoder   Llama-style decoder (embedding, RMSNorm, rotate-half RoPE, GQA
          attention under an arbitrary visibility set, SwiGLU FFN, final norm,
          LM head) with a per-sequence KV cache.
spec      Layer-skip self-drafting, chain and tree verification, the round
          loop, plain greedy autoregressive decoding.
accept    Greedy chain / tree acceptance, rejection sampling with the integer
          inverse-CDF sampler, KV commit / rollback, confidence-scheduled k.
analytic  Closed-form speedup models printed on the pages.

Precision: all activations, attention and accumulations are float64.  Weights
are stored as the model's own values widened exactly to float32 and cast to
float64 at use.  The acceptance ratio test and the confidence score are exact
float64 expressions.  Integers (tokens, lengths, sampler weights) are exact.

Parity pins: every public function is pinned by a ``-m "not gpu"`` test
against a value the pages print, a closed form, an invariant, or brute force
on a tiny input (see tests/test_oracle_*.py).
"""
from . import decoder, accept, spec, analytic  # noqa: F401
