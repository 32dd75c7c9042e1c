"""Tile classes of the block-diagonal causal mask. TEST INFRASTRUCTURE ONLY.

Page "Sample Packing: attention problems of long-sequence LLM training",
section 5.1 "FlashAttention": cut the mask into BM x BN tiles; a tile whose
mask is all zero is skipped, a tile that is partly zero needs the mask
applied, a tile that is all one is computed without a mask. Varlen attention
(same section) splits the block-diagonal mask into one causal attention per
document, so the tiles it visits are those of each document's own causal
triangle, with tiles starting at the document's first token.

Written by brute force over the explicit mask, so it can be checked by eye.
"""
import numpy as np


def classify(mask, bm, bn):
    """Counts (skip, partial, full) over the tiles of a dense bool mask. Edge
    tiles are clipped to the matrix."""
    n_r, n_c = mask.shape
    skip = partial = full = 0
    for r0 in range(0, n_r, bm):
        for c0 in range(0, n_c, bn):
            t = mask[r0:r0 + bm, c0:c0 + bn]
            if not t.any():
                skip += 1
            elif t.all():
                full += 1
            else:
                partial += 1
    return skip, partial, full


def visited_tiles_per_doc(doc_lens, bm, bn):
    """Tiles a varlen kernel visits: for every document on its own, the tiles
    of its causal triangle that hold at least one unmasked entry."""
    total = 0
    for n in doc_lens:
        skip, partial, full = classify(np.tril(np.ones((n, n), dtype=bool)), bm, bn)
        total += partial + full
    return total


def unmasked_pairs(doc_lens):
    """Entries of the block-diagonal causal mask that are one."""
    return sum(n * (n + 1) // 2 for n in doc_lens)
