"""CPU oracle of the hybrid-batch attention step (test infrastructure only).

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline and
reference legs import this package; the CUDA library and its Python binding
never do, and nothing here imports them.

  paged_attention  fp64 numpy: KV append into pages, attention through the
                   block table, split-softmax merge
  brute            pure-Python loops of the same attention (tiny shapes)
  stall_free       the stall-free batch builder, step by step
  linear           fp64 linear layers of the block (projection, gated MLP,
                   residual) around the attention step
"""
