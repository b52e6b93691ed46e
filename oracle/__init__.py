"""fp64 CPU oracle for exact attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call, link
or execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` use it.  It shares no code with
the CUDA path (``exact_attention_66_gb300``); the only common module is
``attn_inputs`` (seeded input draws, no attention arithmetic).

Modules
-------
attn64    plain definition of masked/modded softmax attention in fp64 numpy,
          forward and backward, the decode step over a paged K/V cache, the
          128x128 block-sparsity map by brute force, the signed Hadamard
          rotation, RoPE and e4m3 quantisation.
brute     scalar triple loops for tiny shapes, written independently of
          attn64, used only to pin it.

Parity status: every function in attn64 is pinned by ``tests/test_oracle.py``
(closed forms, library special cases, brute force, finite differences).  The
one quantity without an absolute pin is the FP8 error ratio with versus
without the Hadamard rotation: parity unpinned (it is reported, not gated).
"""
