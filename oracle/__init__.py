"""CPU oracle for the FreeToken expert-cache MoE layer.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
restatement of what the layer computes: exact Python integers for the cache
control and float64 numpy for the expert arithmetic.  Only the tests, the
smoke check (``__graft_entry__.smoke``) and the benchmark's CPU-baseline /
reference arm may import it.  The product path (the CUDA library and its
Python binding) never imports, calls or links anything here, and nothing here
imports the product path: the two share only the seeded input generators in
``synth``.

Modules:
  control  -- routing, dedup, hit/miss, q, fill/CPU sets, LRU victims, map and
              stamp updates, slot rewrite, cache resize, prefill invalidation.
  numerics -- expert SwiGLU FFN, gated merge with the CPU-set partial sum,
              dense masked brute force.
  nvfp4    -- e2m1 / e4m3 decoding of NVFP4 records and the block-16
              activation quantiser.
  mxfp4    -- e2m1 / E8M0 decoding of MXFP4 records and the block-32 MX
              conversion.
  fp8      -- E4M3 decoding of block-FP8 records (fp32 scale per 128 x 128
              block) and the block quantiser.

Readings of the pages that these modules take where the pages are silent are
listed in each function's docstring.  Parity unpinned: none of the functions
here is left without a pin; the pins live in tests/test_oracle_*.py.
"""
