"""CPU oracle for sample packing and document-masked causal attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call, link or
execute anything in this package: only ``tests/``, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.
It shares no code, header, table or helper with the CUDA path under
``sample_packing_document_gb300/``; the two meet only through the seeded input
generators, which hold none of the method's arithmetic.

Contents
--------
``pack``       literal build_pack / build_unpack over Python lists, plus the
               batch fields derived from them (cu_seqlens, indexes, max_seqlen)
               and the global flat forms the C-ABI emits.
``pack_ref.c`` the same rules as sequential C, for timing on host cores.
``attn_ref.c`` fp64 attention with an explicit block-diagonal causal mask test
               and its exact gradient (OpenMP over independent rows).
``attention``  ctypes wrappers around ``attn_ref.c`` / ``pack_ref.c``.
``brute``      dense numpy fp64 attention over a materialised N x N mask, for
               tiny inputs; the independent cross-check of ``attn_ref.c``.
``tiles``      the tile classification of the block-diagonal causal mask
               (skip / partial / full) and the visited-tile count.
``rope``       rotary position embedding with per-document positions (fp64).
``loss``       masked token cross-entropy over packed labels, its gradient and the
               sequence-parallel token-weighted reduction (fp64).
"""
