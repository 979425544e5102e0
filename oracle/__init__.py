"""Plain, slow, obviously-correct CPU oracle for exact Gumbel-max sampling fused
into the LM head (FlashSampling: Fast and Memory-Efficient Exact Sampling).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call, link
or execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` use it.  It shares no code with the
CUDA path (``lm_head_exact_gb300``) and never imports it; both sides receive
their inputs from the seeded generators in ``lm_head_exact_gb300.synthetic``,
which hold none of the method's arithmetic.

Arithmetic is fp64 throughout.  Modules:

* ``philox``  -- Philox-4x32-10 counter-based generator (Salmon et al., SC'11).
* ``sampler`` -- logits, temperature, Gumbel noise, the total-order argmax,
  and the one-shot / partitioned / chunked / sharded samplers built on them;
  the early-finalization bound of the chunked sampler.
* ``topk``    -- Gumbel-top-k: the k best perturbed scores per row (k draws
  without replacement), and its partitioned form.

Pins (what ties each function to something other than itself) live in
``tests/test_oracle_*.py``; every function here is pinned, none is
"parity unpinned".
"""

from . import philox, sampler, topk  # noqa: F401
