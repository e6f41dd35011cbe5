"""Oracle: a plain, slow, CPU restatement of what the rotated INT2 KV-cache path computes.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code, header, table or constant with the CUDA library under
``bit_rotated_kv_gb300/``; the only module both sides use is ``synth`` (seeded
inputs, which holds none of the method's arithmetic).

Sources (web pages on the method; cited by page title and section):
  [OSCAR]  "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
           Quantization" (paperlayer summary)
  [OScaR]  "OScaR：极端 KV 缓存量化的奥卡姆剃刀" (reading note on "OScaR: The Occam's
           Razor for Extreme KV Cache Quantization in LLMs and Beyond")
  [WUSH]   "WUSH-KV: KV Cache Quantization with Data-Adaptive Transforms" (digest)

Modules and what pins each one (tests/test_oracle_*.py, marked "not gpu"):
  fp         float64 -> bfloat16 / float16 rounding.  Pinned against exact
             rational rounding (Python ``fractions``) on random values and ties.
  transform  k' = T k, q' = T^{-T} q, normalised Walsh-Hadamard.  Pinned by the
             q^T k invariant for orthogonal and invertible T, H H^T = I, the fast
             transform == scipy's Sylvester Hadamard matrix, T^T T^{-T} = I.
  quant      kappa-quantile clipped affine INT2, QuEST RMS, l2 token scaling.
             Pinned by the worked example of [OScaR] (Delta = 2.0, bound 1.0), a
             hand-made group with a half-even tie, the |x - x_hat| <= Delta/2
             bound, numpy.quantile, brute force over all 4^G code vectors, the
             MSE-optimal Gaussian clip for QuEST's alpha, ||y|| = 1.
  cache      flush schedule (S_sink / S_keep / S_flush) and the mixed cache.
             Pinned by the closed form of eager flushing and its invariants.
  attention  float64 softmax decode attention over sink | INT2 | recent.
             Pinned against torch's scaled_dot_product_attention (float64),
             one-token, equal-score and g = 1 special cases, and the all-BF16
             case (context <= S_sink + S_keep).

Parity unpinned: the accuracy of INT2 attention relative to unquantized
attention (the pages' accuracy numbers need trained models); reported only.
"""

from . import fp, transform, quant, cache, attention, pipeline  # noqa: F401
