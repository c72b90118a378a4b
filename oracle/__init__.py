"""CPU oracle of one EAGLE-3 draft-and-verify round (float64, plain, slow).

TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA path: no kernels, headers, helpers, tables or constants; the only code
both sides use is the seeded input generator, which holds none of the method's
arithmetic.

Modules:
  layers  -- fp64 primitives of the one-layer draft decoder and the LM heads
  round   -- prefix cache, draft passes, confidence tree, verification
  philox  -- Philox4x64-10 and the verify step's uniforms / Gumbel noise

Parity pins (the pages print no worked example):
  * primitives against torch CPU fp64 functional ops (independent library);
  * RoPE by its relative-position invariant;
  * tree attention, positions and own-state feedback by a brute-force
    sequential causal forward over each root-to-node path;
  * orderings and the kept set by brute-force sorts and the tree invariants;
  * greedy verification by brute force over all root-to-node paths;
  * sampling verification by a chi-square test of the output marginals against
    the target distribution at V = 8;
  * Philox against numpy.random.Philox and the published Random123
    known-answer vectors;
  * the layer's composition, the decoder input, the log-sum-exp and the
    two-stage rescoring by closed-form special cases and scipy.
"""
