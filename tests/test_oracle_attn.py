"""Pins for the attention oracle (CPU only).

attn_ref.c is checked against things other than itself:
* the dense Megatron-style mask construction (brute.py) and the counts the page
  "Sample Packing: attention problems of long-sequence LLM training" prints
  (section 4.2: zeroed regions 4x3, 5x(3+4), 4x(3+4+5) for documents 3, 4, 5, 4;
  section 5.1: 16x16 causal mask in 4x4 tiles; section 5.3: 74.80% sparsity of
  two 16K documents in a 32K sample; the sum-of-squares bound);
* torch's causal scaled_dot_product_attention in fp64 (one document is plain
  causal attention) and torch autograd in fp64 (the backward);
* the equivalence the page states in section 3: a packed row equals its
  documents attended separately;
* exact special cases: length-1 documents give O = V; GQA equals MHA with
  repeated K/V, and dK/dV are the group sums of the MHA gradients.
"""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import brute, tiles


def _bf16(shape, gen, scale=1.0):
    x = (torch.randn(*shape, generator=gen, dtype=torch.float32) * scale).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16).copy()


def _f64(u16):
    return brute.bf16_bits_to_f64(u16)


def _problem(lens, Hq, Hkv, d, seed):
    gen = torch.Generator().manual_seed(seed)
    T = sum(lens)
    q, k, v, do = (_bf16((T, H, d), gen) for H in (Hq, Hkv, Hkv, Hq))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q, k, v, do, cu


# --- mask counts printed on the page ---------------------------------------------------

def test_megatron_zeroed_regions_docs_3_4_5_4():
    cu = [0, 3, 7, 12, 16]
    causal = brute.causal_mask(16)
    m = brute.reset_attention_mask(cu)
    assert causal.sum() == 136
    assert (causal & ~m).sum() == 4 * 3 + 5 * 7 + 4 * 12 == 95
    assert m.sum() == 41 == tiles.unmasked_pairs([3, 4, 5, 4])
    # one causal block per document, nothing across documents
    for a, b in zip(cu[:-1], cu[1:]):
        assert (m[a:b, a:b] == np.tril(np.ones((b - a, b - a), bool))).all()
        assert not m[a:b, :a].any() and not m[a:b, b:].any()


def test_tile_classes_16x16_causal_4x4():
    assert tiles.classify(brute.causal_mask(16), 4, 4) == (6, 4, 6)


def test_two_16k_docs_tile_sparsity():
    visited = tiles.visited_tiles_per_doc([16384, 16384], 128, 128)
    assert visited == 16512
    assert round(100 * (1 - visited / (256 * 256)), 2) == 74.80


def test_sum_of_squares_bound():
    rng = np.random.default_rng(7)
    for _ in range(2000):
        S = int(rng.integers(2, 5000))
        lens = []
        while sum(lens) < S:
            lens.append(int(rng.integers(1, S // 2 + 1)))
        lens[-1] -= sum(lens) - S
        lens = [x for x in lens if x > 0]
        assert max(lens) <= S / 2
        assert sum(x * x for x in lens) <= S * S / 2


# --- forward ---------------------------------------------------------------------------

@pytest.mark.parametrize("lens,Hq,Hkv,d", [([3, 4, 5, 4], 2, 2, 16), ([1, 7, 2, 9, 13], 4, 2, 32),
                                           ([40], 3, 1, 8), ([5, 1, 1, 30, 2], 6, 3, 64)])
def test_fwd_matches_dense_megatron_mask(lens, Hq, Hkv, d):
    q, k, v, _, cu = _problem(lens, Hq, Hkv, d, seed=sum(lens) + Hq)
    o, lse = OA.attn_fwd(q, k, v, cu)
    ob, lseb = brute.attention(_f64(q), _f64(k), _f64(v), brute.reset_attention_mask(cu),
                               1.0 / np.sqrt(d))
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lseb, rtol=0, atol=1e-12)


def test_single_document_is_torch_causal_sdpa():
    q, k, v, _, cu = _problem([57], 4, 4, 32, seed=3)
    o, _ = OA.attn_fwd(q, k, v, cu, scale=0.3)
    t = lambda a: torch.from_numpy(_f64(a)).permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(t(q), t(k), t(v), is_causal=True,
                                                           scale=0.3)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def test_packed_row_equals_documents_alone():
    lens = [5, 17, 1, 9, 30]
    q, k, v, _, cu = _problem(lens, 4, 2, 16, seed=11)
    o, lse = OA.attn_fwd(q, k, v, cu)
    for a, b in zip(cu[:-1], cu[1:]):
        oa, la = OA.attn_fwd(q[a:b], k[a:b], v[a:b], [0, b - a])
        np.testing.assert_array_equal(o[:, a:b], oa)
        np.testing.assert_array_equal(lse[:, a:b], la)


def test_length_one_documents_give_v_exactly():
    q, k, v, _, cu = _problem([1] * 12, 4, 2, 16, seed=5)
    o, _ = OA.attn_fwd(q, k, v, cu)
    vv = _f64(v)
    for h in range(4):
        np.testing.assert_array_equal(o[h], vv[:, h // 2, :])


def test_gqa_equals_mha_with_repeated_kv():
    q, k, v, _, cu = _problem([6, 11, 3], 6, 2, 16, seed=8)
    o, lse = OA.attn_fwd(q, k, v, cu)
    o2, lse2 = OA.attn_fwd(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), cu)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_fwd_item_subset_matches_full():
    q, k, v, _, cu = _problem([6, 11, 3, 20], 4, 4, 16, seed=9)
    T = q.shape[0]
    o, lse = OA.attn_fwd(q, k, v, cu)
    items = np.array([0, 5, T + 7, 3 * T + 39, 2 * T + 21])
    os_, ls = OA.attn_fwd(q, k, v, cu, items=items)
    for n, it in enumerate(items):
        np.testing.assert_array_equal(os_[n], o[it // T, it % T])
        assert ls[n] == lse[it // T, it % T]


# --- backward --------------------------------------------------------------------------

def _torch_dense_grads(q, k, v, do, cu, scale):
    """Autograd through the dense masked formula, fp64."""
    Hq, Hkv = q.shape[1], k.shape[1]
    t = lambda a: torch.from_numpy(_f64(a)).requires_grad_(True)
    tq, tk, tv = t(q), t(k), t(v)
    mask = torch.from_numpy(brute.reset_attention_mask(cu))
    kk = tk.repeat_interleave(Hq // Hkv, dim=1)
    vv = tv.repeat_interleave(Hq // Hkv, dim=1)
    s = torch.einsum("ihc,jhc->hij", tq, kk) * scale
    s = s.masked_fill(~mask, float("-inf"))
    o = torch.einsum("hij,jhc->ihc", torch.softmax(s, dim=-1), vv)
    o.backward(torch.from_numpy(_f64(do)))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("lens,Hq,Hkv,d", [([3, 4, 5, 4], 2, 2, 16), ([9, 1, 14, 2], 4, 2, 32),
                                           ([25], 3, 1, 8), ([2, 1, 1, 19, 7], 6, 3, 16)])
def test_bwd_matches_autograd(lens, Hq, Hkv, d):
    q, k, v, do, cu = _problem(lens, Hq, Hkv, d, seed=31 + d)
    scale = 1.0 / np.sqrt(d)
    dq, dk, dv, rows = OA.attn_bwd(q, k, v, do, cu)
    gq, gk, gv = _torch_dense_grads(q, k, v, do, cu, scale)
    np.testing.assert_allclose(dq, gq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, gk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, gv, rtol=0, atol=1e-11)


def test_bwd_length_one_documents():
    q, k, v, do, cu = _problem([1] * 10, 4, 2, 16, seed=2)
    dq, dk, dv, _ = OA.attn_bwd(q, k, v, do, cu)
    assert (dq == 0).all() and (dk == 0).all()
    dof = _f64(do)
    np.testing.assert_array_equal(dv[:, 0], dof[:, 0] + dof[:, 1])
    np.testing.assert_array_equal(dv[:, 1], dof[:, 2] + dof[:, 3])


def test_bwd_gqa_is_group_sum_of_mha():
    q, k, v, do, cu = _problem([6, 13, 2], 6, 2, 16, seed=4)
    dq, dk, dv, _ = OA.attn_bwd(q, k, v, do, cu)
    dq2, dk2, dv2, _ = OA.attn_bwd(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), do, cu)
    np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, dk2.reshape(dk2.shape[0], 2, 3, -1).sum(2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, dv2.reshape(dv2.shape[0], 2, 3, -1).sum(2), rtol=0, atol=1e-12)


def test_bwd_segment_subset_and_dq_rows():
    lens = [7, 30, 4, 12]
    q, k, v, do, cu = _problem(lens, 4, 2, 16, seed=6)
    T = q.shape[0]
    dq, dk, dv, rows = OA.attn_bwd(q, k, v, do, cu)
    sdq, sdk, sdv, srows = OA.attn_bwd(q, k, v, do, cu, segs=[3, 1])
    np.testing.assert_array_equal(srows, np.concatenate([np.arange(41, 53), np.arange(7, 37)]))
    np.testing.assert_array_equal(sdq, dq[srows])
    np.testing.assert_array_equal(sdk, dk[srows])
    items = np.array([2 * T + 10, 0, 3 * T + 52])
    r = OA.attn_dq_rows(q, k, v, do, cu, items)
    for n, it in enumerate(items):
        np.testing.assert_allclose(r[n], dq[it % T, it // T], rtol=0, atol=1e-13)


def test_oracle_rejects_bad_seqlens():
    q, k, v, do, cu = _problem([4, 4], 2, 2, 8, seed=1)
    with pytest.raises(ValueError):
        OA.attn_fwd(q, k, v, [0, 4, 4, 8])
    with pytest.raises(ValueError):
        OA.attn_fwd(q, k, v, [0, 4, 7])
