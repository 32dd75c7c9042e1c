"""The library on several streams and host threads at once.

Every call keeps its state in the caller's workspace (status word, tile
schedule, work counter, dQ accumulator) and the host side keeps none beyond a
cached driver entry point and per-thread test hooks, so two problems in
flight together on two streams, or issued from two host threads, must give
what they give alone. The forward output, the LSE and dK / dV are produced in
a fixed order (one CTA per q-tile unit, one per kv-tile unit) and must match
the sequential run bit for bit; dQ is summed by fp32 reduce-adds whose order
varies between runs, so it is compared with the fp64 oracle at the usual bar.
"""
import threading

import numpy as np
import pytest
import torch

from oracle import attention as OA

pytestmark = pytest.mark.gpu

TOL_G = 5e-2

# (lengths, Hq, Hkv, head_dim, gradient dtype)
PROBLEMS = [
    ([700, 33, 1290, 1, 2000], 4, 2, 128, torch.bfloat16),
    ([128, 5, 900, 2000, 64, 3], 6, 6, 64, torch.float32),
]


@pytest.fixture(scope="module")
def ops():
    from sample_packing_document_gb300 import build, ops as _ops
    build.build()
    _ops.load()
    return _ops


def _problem(i, device="cuda"):
    from sample_packing_document_gb300 import workloads as W
    lens, Hq, Hkv, d, gdt = PROBLEMS[i]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, do = W.qkv(int(cu[-1]), Hq, Hkv, d, 70 + i, device=device)
    return dict(q=q, k=k, v=v, do=do, cu_h=cu, cu=torch.tensor(cu, device=device), ns=len(lens), gdt=gdt)


def _step(ops, p, stream):
    """Forward then backward of problem p on `stream`, with workspaces and outputs
    allocated on that stream."""
    with torch.cuda.stream(stream):
        T, Hq, d = p["q"].shape
        Hkv = p["k"].shape[1]
        ws_f = ops.workspace(ops.attn_workspace_size(T, p["ns"], Hq, Hkv, d, False))
        ws_b = ops.workspace(ops.attn_workspace_size(T, p["ns"], Hq, Hkv, d, True))
        out, lse = ops.varlen_attn_fwd(p["q"], p["k"], p["v"], p["cu"], p["ns"], ws=ws_f, stream=stream)
        dq, dk, dv = ops.varlen_attn_bwd(p["q"], p["k"], p["v"], out, p["do"], lse, p["cu"], p["ns"],
                                         grad_dtype=p["gdt"], ws=ws_b, stream=stream)
    return dict(out=out, lse=lse, dq=dq, dk=dk, dv=dv, ws_f=ws_f, ws_b=ws_b, stream=stream)


def _statuses_ok(ops, r):
    return ops.read_status(r["ws_f"], r["stream"]) == 0 and ops.read_status(r["ws_b"], r["stream"]) == 0


def _same_fixed_order_outputs(a, b):
    for key in ("out", "lse", "dk", "dv"):
        assert torch.equal(a[key], b[key]), key


def _dq_matches_oracle(p, dq):
    u16 = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    gq, _, _, _ = OA.attn_bwd(u16(p["q"]), u16(p["k"]), u16(p["v"]), u16(p["do"]), p["cu_h"])
    err = float(np.max(np.abs(dq.float().cpu().numpy().astype(np.float64) - gq)))
    assert err <= TOL_G, err


def test_two_streams_in_flight_together(ops):
    probs = [_problem(0), _problem(1)]
    torch.cuda.synchronize()
    alone = []
    for p in probs:
        r = _step(ops, p, torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert _statuses_ok(ops, r)
        alone.append(r)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    # both problems issued before either is waited for, three rounds each
    together = [[_step(ops, p, s) for p, s in zip(probs, streams)] for _ in range(3)]
    torch.cuda.synchronize()
    for rnd in together:
        for i, r in enumerate(rnd):
            assert _statuses_ok(ops, r)
            _same_fixed_order_outputs(r, alone[i])
    for i, p in enumerate(probs):
        _dq_matches_oracle(p, together[-1][i]["dq"])


def test_two_host_threads(ops):
    probs = [_problem(0), _problem(1)]
    torch.cuda.synchronize()
    alone = []
    for p in probs:
        r = _step(ops, p, torch.cuda.current_stream())
        torch.cuda.synchronize()
        alone.append(r)
    results, errors = [None, None], []

    def worker(i, stream):
        try:
            torch.cuda.set_device(probs[i]["q"].device)
            rs = [_step(ops, probs[i], stream) for _ in range(4)]
            stream.synchronize()
            results[i] = rs
        except Exception as e:      # reported by the main thread
            errors.append(e)

    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    threads = [threading.Thread(target=worker, args=(i, streams[i])) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    assert all(not t.is_alive() for t in threads)
    torch.cuda.synchronize()
    for i in range(2):
        for r in results[i]:
            assert _statuses_ok(ops, r)
            _same_fixed_order_outputs(r, alone[i])
        _dq_matches_oracle(probs[i], results[i][-1]["dq"])
