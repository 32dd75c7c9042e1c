"""Failure detection on the GPU without a fault.

spd_debug_skip_arrive makes the TMA producer of the next forward / backward
call leave out its first Q (forward) or K / V (backward) load, so the barrier
the MMA issuer waits on never completes. Every wait in the kernels is bounded
(2 s of the global timer): the issuer's wait runs out, raises the CTA's abort
flag, the other roles leave at their next bounded wait, the producer lets its
own copies land, tensor memory is freed, and SPD_ERR_DEVICE_TIMEOUT lands in the
status word. Nothing traps, faults or hangs; the same CUDA context then runs a
clean call whose results equal those of a call before the failure, bit for bit.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

TIMEOUT = -5   # SPD_ERR_DEVICE_TIMEOUT


def _setup():
    from sample_packing_document_gb300 import build, ops, workloads as W
    build.build()
    lens = [300, 17, 500, 1]
    T, ns, Hq, Hkv, d = sum(lens), len(lens), 4, 2, 128
    cu = torch.tensor([0, 300, 317, 817, 818], dtype=torch.int32, device="cuda")
    q, k, v, do = W.qkv(T, Hq, Hkv, d, seed=7, device="cuda")
    return ops, cu, ns, q, k, v, do


def test_forward_bounded_wait_reports_timeout_and_context_survives():
    ops, cu, ns, q, k, v, _ = _setup()
    T, Hq, d = q.shape
    ws = ops.workspace(ops.attn_workspace_size(T, ns, Hq, k.shape[1], d, False))
    o_ref, lse_ref = ops.varlen_attn_fwd(q, k, v, cu, ns, ws=ws)
    assert ops.read_status(ws) == 0
    ops.debug_skip_arrive(ops.DEBUG_SKIP_FWD_Q)
    ops.varlen_attn_fwd(q, k, v, cu, ns, ws=ws)
    assert ops.read_status(ws) == TIMEOUT
    o, lse = ops.varlen_attn_fwd(q, k, v, cu, ns, ws=ws)   # the hook is consumed
    assert ops.read_status(ws) == 0
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


def test_backward_bounded_wait_reports_timeout_and_context_survives():
    ops, cu, ns, q, k, v, do = _setup()
    T, Hq, d = q.shape
    o, lse = ops.varlen_attn_fwd(q, k, v, cu, ns)
    ws = ops.workspace(ops.attn_workspace_size(T, ns, Hq, k.shape[1], d, True))
    ref = ops.varlen_attn_bwd(q, k, v, o, do, lse, cu, ns, ws=ws)
    assert ops.read_status(ws) == 0
    ops.debug_skip_arrive(ops.DEBUG_SKIP_BWD_KV)
    ops.varlen_attn_bwd(q, k, v, o, do, lse, cu, ns, ws=ws)
    assert ops.read_status(ws) == TIMEOUT
    got = ops.varlen_attn_bwd(q, k, v, o, do, lse, cu, ns, ws=ws)
    assert ops.read_status(ws) == 0
    for g, r in zip(got, ref):
        assert torch.equal(g, r)
