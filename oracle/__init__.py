"""CPU oracle for fused exact scaled-dot-product attention (forward + backward).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import, call, link or run it.
It shares no code, header, constant or helper with the CUDA library in
``attention_blackwell_gb300/``; the two meet only through the seeded input
generators in ``attention_blackwell_gb300.workloads``, which hold none of the
method's arithmetic.

Sources (cited by page title and section throughout):

* "FlashAttention-4 blog" -- the Together AI write-up of FlashAttention-4
  (read in its Chinese translation): sections "Forward pass: a new softmax
  pipeline with conditional rescaling", "Faster exponential: split 2^x between
  MUFU.EX2 and FMA", "Backward pass", "2-CTA backward", "Deterministic mode",
  "Scheduling".
* "FlashAttention-4 paper summary" -- the structured summary of arXiv
  2603.05451: §3.1.2 (pipeline), §3.1.3 (software exp2, Table 2),
  §3.1.4 (conditional rescaling), §3.2.3 (2-CTA MMA), the notation table.

Modules:

* ``attention``      -- the plain definition in float64: S, P, O, LSE and the
                        backward gradients, plus a pure-Python brute force.
* ``online_softmax`` -- a block-by-block float64 restatement of the forward
                        pipeline's online softmax with the conditional rescale
                        threshold tau, used to pin the rescale identity.
* ``exp2_poly``      -- Cody-Waite range reduction + degree-3 Horner exp2 in
                        float32 (C, ``exp2_poly.c``) and the minimax fit of its
                        coefficients.
"""
