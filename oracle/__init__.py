"""Float64 CPU oracle for packed-THD context-parallel attention.

TEST INFRASTRUCTURE ONLY. This package is the independent, slow, obviously
correct statement of what the CUDA library computes. Only the tests, the
smoke check and the benchmark's CPU-baseline leg may import it; the library
itself never does, and it shares no code with the CUDA path.

Sources (TransformerEngine PR #3221 "[PyTorch] Add no-load-balance THD
all-gather CP"; torchtitan PR #2144 "[CP] Refactor Context Parallel to use new
PyTorch CP APIs"):

* ``partition``  -- DualChunkSwap (per-document, 2*cp_size chunks, rank r owns
  chunks r and 2*cp_size-1-r) and NO_LOAD_BALANCE (cp_size contiguous chunks of
  the physical buffer), section "Why" and "What changed" of the TE PR.
* ``reorder``    -- the gather of THD tensors into a rank's token order
  (TE PR "How to use": get_batch_on_this_cp_rank of input_ids, labels,
  position_ids).
* ``attention``  -- causal THD attention with documents isolated by
  cu_seqlens / cu_seqlens_padded (TE PR "Scope and constraints": causal, no
  sliding window; "What changed": logical document boundaries kept through
  THD metadata).

Every function here is pinned by tests/test_oracle_*.py against hand-worked
examples, brute force, closed forms and library routines. No function is
"parity unpinned".
"""
