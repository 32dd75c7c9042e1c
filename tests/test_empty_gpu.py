"""Empty inputs through the GPU entry points: no documents, no tokens, no rows.

Each call returns SPD_OK and writes what an empty result has (the pack: no
rows, num_segs 0, cu_seqlens = row_seg_ptr = {0}, as the oracle's build_pack /
build_unpack give for an empty document list; attention, RoPE and the loss:
nothing, a zero sum and count), and nothing outside its buffers: the pack's
segment fields are placed inside a larger buffer whose other words must keep
their sentinel value.
"""
import numpy as np
import pytest
import torch

from oracle import pack as P

pytestmark = pytest.mark.gpu

SENTINEL = 777


@pytest.fixture(scope="module")
def ops():
    from sample_packing_document_gb300 import build, ops as _ops
    build.build()
    _ops.load()
    return _ops


@pytest.mark.parametrize("packed", [True, False])
def test_pack_no_documents(ops, packed):
    ref = P.pack_flat([], 2, 8, packed)
    out = ops.alloc_pack_outputs(0, 0, 2, 8, packed)
    assert out["rows"] == ref["rows"] == 0
    guard = torch.full((16,), SENTINEL, dtype=torch.int32, device="cuda")
    out["cu_seqlens"], out["row_seg_ptr"], out["num_segs"] = guard[4:5], guard[8:9], guard[12:13]
    empty = torch.empty(0, dtype=torch.int32, device="cuda")
    ops.pack_tokens(empty, empty, 2, 8, packed, out=out)
    assert ops.read_status(out["ws"]) == 0
    g = guard.cpu().tolist()
    assert [g[4], g[8], g[12]] == [ref["cu_seqlens"][0], ref["row_seg_ptr"][0], ref["num_segs"]] == [0, 0, 0]
    assert all(x == SENTINEL for i, x in enumerate(g) if i not in (4, 8, 12))


def test_attention_no_tokens(ops):
    for d in (64, 128):
        q = torch.empty(0, 4, d, dtype=torch.bfloat16, device="cuda")
        k = torch.empty(0, 2, d, dtype=torch.bfloat16, device="cuda")
        cu = torch.zeros(1, dtype=torch.int32, device="cuda")
        ws_f = ops.workspace(ops.attn_workspace_size(0, 0, 4, 2, d, False))
        out, lse = ops.varlen_attn_fwd(q, k, k, cu, 0, ws=ws_f)
        assert ops.read_status(ws_f) == 0
        assert out.shape == (0, 4, d) and lse.shape == (4, 0)
        ws_b = ops.workspace(ops.attn_workspace_size(0, 0, 4, 2, d, True))
        dq, dk, dv = ops.varlen_attn_bwd(q, k, k, out, out, lse, cu, 0, ws=ws_b)
        assert ops.read_status(ws_b) == 0
        assert dq.shape == (0, 4, d) and dk.shape == (0, 2, d) and dv.shape == (0, 2, d)
        out_r, lse_r = ops.varlen_attn_fwd_rope(q, k, k, cu, 0, ws=ws_f)
        assert ops.read_status(ws_f) == 0 and out_r.numel() == 0 and lse_r.numel() == 0


def test_rope_and_loss_no_tokens(ops):
    q = torch.empty(0, 4, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.empty(0, 2, 128, dtype=torch.bfloat16, device="cuda")
    pos = torch.empty(0, dtype=torch.int32, device="cuda")
    ops.rope(q, k, pos)
    logits = torch.empty(0, 1000, dtype=torch.bfloat16, device="cuda")
    labels = torch.empty(0, dtype=torch.int32, device="cuda")
    token_loss, loss_sum, num_tokens = ops.masked_token_loss(logits, labels)
    torch.cuda.synchronize()
    assert token_loss.numel() == 0
    assert float(loss_sum.item()) == 0.0 and int(num_tokens.item()) == 0
    assert np.isfinite(float(loss_sum.item()))
