"""Oracle: a plain, slow, fp64 CPU restatement of the batch-invariant forward step.

THIS PACKAGE IS TEST INFRASTRUCTURE.  Only the test suite, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it.  The
product path (``invariant_deterministic_gb300``) never imports, links or runs
anything here, and nothing here imports the product path: the two share no
kernels, helpers, tables or constants.  The seeded input generators live in
their own module (``invariant_deterministic_gb300.synth``), which holds none of
the method's arithmetic.

What is computed, and where the pages define it:

* ``gemm``       -- matrix multiplication C = A . W^T ("Deterministic and bit-exact
                    inference", *technical*: the matmul whose per-element
                    reduction order the invariant route fixes).
* ``rmsnorm``    -- RMSNorm (same passage).
* ``attention``  -- softmax attention, decode and causal prefill (same passage:
                    attention made batch-invariant with a fixed split size of
                    the key-value dimension; the split is a GPU scheduling
                    detail, so the oracle computes the unsplit softmax).
* ``rope``       -- rotate-half rotary embedding (layer glue, no reduction).
* ``glue``       -- embedding gather, residual add, SwiGLU.
* ``philox``     -- Philox4x32-10 (Salmon et al., SC'11).
* ``sampler``    -- the seeded sampler with the settings a Kinetic receipt
                    records (Kinetic "Receipts", *Making a receipt*: the
                    ``sampling`` object: temperature, top_k, top_p, min_p,
                    repeat_penalty, repeat_last_n, seed).
* ``model``      -- the pre-norm decoder layer and the full decode step built
                    from the pieces above.

Numbers: inputs are bf16 bit patterns (uint16 arrays) widened exactly to fp64;
every result is rounded to bf16 (round to nearest, ties to even) only where the
GPU path stores a bf16 tensor.  Where floating point decides an integer (the
sampler's ranking and thresholds), the decision is taken in the same precision
as the kernel, as each function documents.

Pins: every function is checked by ``tests/test_oracle_*.py`` against closed
forms, invariants, library routines or brute force; none is "parity unpinned"
except the end-to-end 36-layer decode, which is checked per kernel instead.
"""
