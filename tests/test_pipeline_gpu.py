"""The library's calls composed as a training step uses them, each stage
checked against the oracle fed the previous stage's own inputs: pack the
documents; rotate q and k by the pack's indexes; attention over the pack's
cu_seqlens; the masked loss over the pack's labels (and its gradient); the
backward; the inverse rotation of dq and dk. The stages are pinned one by one
elsewhere; this checks that their layouts and conventions fit together."""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import loss as L
from oracle import pack as P
from oracle import rope as R

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _close_bf16(got, want):
    """bf16 storage of the result (half an ulp, 2^-9 relative) plus fp32 work."""
    got = got.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-5 * max(1.0, np.abs(want).max()))


def test_pack_rope_attention_loss_backward():
    from sample_packing_document_gb300 import build, ops
    build.build()
    rng = np.random.default_rng(2718)
    mb, sl, H, d, V = 2, 1024, 4, 128, 1000
    docs = [rng.integers(1, V, size=int(n)).tolist() for n in rng.integers(1, 700, size=9)]   # token ids are labels < V
    toks = torch.tensor([t for doc in docs for t in doc], dtype=torch.int32, device="cuda")
    lens = torch.tensor([len(doc) for doc in docs], dtype=torch.int32, device="cuda")
    packed = ops.pack_tokens(toks, lens, mb, sl)
    ns = ops.pack_num_segs([len(doc) for doc in docs], mb, sl)
    assert ops.read_status(packed["ws"]) == 0 and int(packed["num_segs"].item()) == ns
    ref = P.pack_flat(docs, mb, sl, True)
    assert packed["input_ids"].cpu().tolist() == ref["input_ids"]
    assert packed["labels"].cpu().tolist() == ref["labels"]
    assert packed["indexes"].cpu().tolist() == ref["indexes"]
    cu = np.asarray(ref["cu_seqlens"], np.int32)
    assert packed["cu_seqlens"][:ns + 1].cpu().numpy().tolist() == cu.tolist()
    T = packed["input_ids"].numel()

    g = torch.Generator(device="cuda").manual_seed(31)
    q, k, v, do = (torch.randn(T, H, d, generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    q0, k0 = _u16(q), _u16(k)
    ops.rope(q, k, packed["indexes"])
    pos = np.asarray(ref["indexes"], np.int64)
    _close_bf16(q, R.rope(_f64(q0), pos))
    _close_bf16(k, R.rope(_f64(k0), pos))

    out, lse = ops.varlen_attn_fwd(q, k, v, packed["cu_seqlens"], ns)
    o_ref, lse_ref = OA.attn_fwd(_u16(q), _u16(k), _u16(v), cu)
    assert np.abs(out.float().cpu().numpy().transpose(1, 0, 2) - o_ref).max() <= 2e-2
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3

    logits = (torch.randn(T, V, generator=g, device="cuda") * 2).to(torch.bfloat16)
    dlogits = torch.empty_like(logits)
    labels = packed["labels"]
    tok, loss_sum, n_tok = ops.masked_token_loss(logits, labels, dlogits=dlogits, grad_scale=1.0 / T)
    x = logits.float().cpu().numpy().astype(np.float64)
    lab = np.asarray(ref["labels"], np.int32)
    s, n, _ = L.masked_loss(x, lab)
    assert int(n_tok.item()) == n == int(np.sum(lab != -100))
    assert float(loss_sum.item()) == pytest.approx(s, rel=1e-5, abs=1e-3)
    want_g = L.logits_grad(x, lab, 1.0 / T)
    assert np.all(np.abs(dlogits.float().cpu().numpy() - want_g) <= 2.0 ** -8 * np.abs(want_g) + 1e-6 / T)

    dq, dk, dv = ops.varlen_attn_bwd(q, k, v, out, do, lse, packed["cu_seqlens"], ns, grad_dtype=torch.float32)
    gq, gk, gv, _ = OA.attn_bwd(_u16(q), _u16(k), _u16(v), _u16(do), cu)
    for got, want in ((dq, gq), (dk, gk), (dv, gv)):
        assert np.abs(got.cpu().numpy() - want).max() <= 5e-2
    dq16, dk16 = dq.to(torch.bfloat16), dk.to(torch.bfloat16)
    dq_b, dk_b = _u16(dq16), _u16(dk16)
    ops.rope(dq16, dk16, packed["indexes"], inverse=True)
    _close_bf16(dq16, R.rope(_f64(dq_b), pos, inverse=True))
    _close_bf16(dk16, R.rope(_f64(dk_b), pos, inverse=True))
