"""CPU oracle for the paged KV-cache hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import anything here.  The
product package never imports it and shares no code, header, table or
constant with it.

Modules:
  attention  -- fp64 paged attention (C, OpenMP), gather-then-dense-softmax
  cache_ops  -- slot write and block copy as plain loops
  allocator  -- block pool / tables / refcounts / copy-on-write as dictionaries
  kv_math    -- block-count and KV-byte arithmetic
"""
