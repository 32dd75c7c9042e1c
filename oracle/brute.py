"""Dense fp64 attention over a materialised N x N mask, for tiny inputs only.
TEST INFRASTRUCTURE ONLY: the independent cross-check of attn_ref.c.

The mask is built the way the page "Sample Packing: attention problems of
long-sequence LLM training" describes Megatron's reset_attention_mask (section
4.2 "Performance problems"): start from the full causal (lower-triangular)
matrix over the whole row, then for every document after the first zero the
block of its rows against all columns before it (for documents 3, 4, 5, 4 in
16 tokens the zeroed regions are 4x3, 5x(3+4) and 4x(3+4+5)). What remains is
one causal block per document (section 3, "Attention Mask").
"""
import numpy as np


def causal_mask(n):
    return np.tril(np.ones((n, n), dtype=bool))


def reset_attention_mask(cu_seqlens):
    """Block-diagonal causal mask from segment boundaries, Megatron style."""
    cu = [int(x) for x in cu_seqlens]
    n = cu[-1]
    m = causal_mask(n)
    for s in range(1, len(cu) - 1):
        start, end = cu[s], cu[s + 1]
        m[start:end, :start] = False
    return m


def bf16_bits_to_f64(a):
    a = np.asarray(a, dtype=np.uint16)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def attention(q, k, v, mask, scale):
    """q [N, Hq, d], k / v [N, Hkv, d] float64; mask [N, N] bool.
    Returns O [Hq, N, d] and LSE [Hq, N]."""
    N, Hq, d = q.shape
    Hkv = k.shape[1]
    group = Hq // Hkv
    out = np.zeros((Hq, N, d))
    lse = np.zeros((Hq, N))
    for h in range(Hq):
        g = h // group
        s = scale * q[:, h, :] @ k[:, g, :].T
        s = np.where(mask, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        out[h] = (e / l) @ v[:, g, :]
        lse[h] = (m + np.log(l))[:, 0]
    return out, lse
