"""CPU oracle for interval-masked / block-sparse attention (TEST INFRASTRUCTURE).

This package is the plain, slow, obviously-correct reference that the CUDA
path is checked against.  It is test infrastructure only: the library's
product path never imports it.  Only the tests, the smoke check and the
benchmark's CPU-baseline / reference arm use it.

It shares no code with the CUDA path.  The only thing both sides use is the
seeded input generator module, which draws inputs and does none of the
method's arithmetic.

Modules
  mask       endpoint validation and dense boolean expansion of a mask
             (interval endpoints per "Flex Attention Mask Plan Design" §2, §3;
             logical block masks per "Decoupling Logical Masks from GPU
             Execution..." §2, the effective set E(M)).
  plan       brute-force MaskPlan: tile classification, independent partial
             and full CSR lists, packed predicate payload, sequence and work
             descriptors, allocation header ("Flex Attention Mask Plan
             Design" §4.3, §4.5, §4.6, §4.8, §5).
  attention  fp64 masked attention with score_mods: softmax(mod(QK^T*scale))V
             and its log-sum-exp (FlexAttention Eq. 1; "Flex Attention Mask
             Plan Design" §6.1 for rows without visible keys).
  backward   fp64 gradients dQ, dK, dV and the K2Q backward view.
  decode     fp64 decoding rows over a paged KV cache: logical keys gathered
             through the page table, the mask evaluated at the query's
             absolute position (FlexAttention summary, §3.4 Paged Attention
             Integration and Modification Conversion for Inference).

Every function is pinned by tests under ``tests/test_oracle_*.py`` against
the pages' worked example, closed forms, library routines on special cases,
invariants and brute force.
"""
from . import mask, plan, attention, decode  # noqa: F401
