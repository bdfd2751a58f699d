"""CPU oracle for the Q4_K x q8 prefill GEMM -- TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct numpy implementation of what the CUDA path
computes, written from the pages' prose and the plain reading of the open
points.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may import it.  The library
(``quantized_prefill_gemm_gb300``) never imports it, and it imports nothing
from the library: the two share no code.

Modules
  q8          activation quantization into 32-element q8 blocks (qa, d_a, ssum)
  q4k_blocks  the 144-byte Q4_K super-block: decode to fields, encode fields
  gemm        the blockwise GEMM with the two-term rescale, the dense fp64
              brute force, the per-element error scale S = sum_k |w_k a_k|,
              and the per-chunk integer dot products

Pins (tests/test_oracle_*.py, ``-m "not gpu"``): exhaustive f16 decode vs the
IEEE definition, f16 round-to-nearest-even on ties, a hand-worked q8 block, the
q8 round-trip bound, exact integer blocks, a hand-worked Q4_K block, the
blockwise result vs the dense fp64 brute force, an exact integer GEMM special
case, and the degenerate cases (X = 0, q = 0, sc = m = 0).

Parity unpinned: the Q4_K byte layout is the public GGUF arrangement as this
project reads it; no GGUF file is available to check interop against.
"""
