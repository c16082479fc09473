"""Hybrid-batch paged attention for GB300 (sm_103a).

The product is the C-ABI library libhb.so (include/hb.h) built from csrc/;
`hb` is its thin ctypes binding and `device` moves a batch descriptor onto the
GPU for it.  `workloads` builds seeded synthetic inputs and is shared with the
tests.  Importing this package loads nothing; hb.load() loads the library.
"""
