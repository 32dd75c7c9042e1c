"""spd_varlen_attn_fwd_noalloc: the forward pass for callers that cannot
allocate device memory (a plugin inside a framework that owns all device
memory, or a path that must not call cudaMalloc / cudaFree). It keeps its
scratch in a fixed array of the library's device image instead of a caller
workspace, so its result must equal spd_varlen_attn_fwd's.

Called through the C ABI (ctypes) twice in a row with different documents,
so the second call runs on scratch the first one left behind. Collected last
so a stop-at-first-failure run has run everything else before it.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 2e-2, 1e-3


def _lib():
    from sample_packing_document_gb300 import build, ops
    build.build()
    return ops.load(), ops


def _call_noalloc(lib, q, k, v, cu, ns, out, lse, status):
    P = ctypes.c_void_p
    T, Hq, d = q.shape
    return lib.spd_varlen_attn_fwd_noalloc(
        P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(cu.data_ptr()), ns, T, 0, Hq, k.shape[1], d,
        ctypes.c_float(0.0), P(out.data_ptr()), P(lse.data_ptr()), P(status.data_ptr()),
        P(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("lens_list", [[[700, 33, 1290, 1], [128, 5, 900, 2000, 64, 3]]])
def test_noalloc_matches_workspace_entry_point(lens_list):
    from sample_packing_document_gb300 import workloads as W
    lib, ops = _lib()
    for n, lens in enumerate(lens_list):
        cu_h = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T, ns = int(cu_h[-1]), len(lens)
        q, k, v, _ = W.qkv(T, 6, 2, 128, seed=40 + n, device="cuda")
        cu = torch.tensor(cu_h, device="cuda")
        out_ref, lse_ref = ops.varlen_attn_fwd(q, k, v, cu, ns)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((6, T), float("nan"), device="cuda")
        status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
        assert _call_noalloc(lib, q, k, v, cu, ns, out, lse, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert float((out.float() - out_ref.float()).abs().max()) <= TOL_O
        assert float((lse - lse_ref).abs().max()) <= TOL_LSE
        assert torch.equal(out, out_ref)           # same kernels, same inputs


def test_noalloc_rejects_oversize_and_reports_bad_seqlens():
    lib, ops = _lib()
    q = torch.zeros(256, 2, 128, dtype=torch.bfloat16, device="cuda")
    out, lse = torch.empty_like(q), torch.empty(2, 256, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # scratch of (2^24 + 2^17) tokens in 2^17 segments exceeds the fixed array: refused on the host
    P = ctypes.c_void_p
    rc = lib.spd_varlen_attn_fwd_noalloc(P(q.data_ptr()), P(q.data_ptr()), P(q.data_ptr()), P(q.data_ptr()),
                                         1 << 17, (1 << 24) + (1 << 17), 0, 2, 2, 128, ctypes.c_float(0.0),
                                         P(out.data_ptr()), P(lse.data_ptr()), None,
                                         P(torch.cuda.current_stream().cuda_stream))
    assert rc == -8 and "no-allocation" in ops.status_string(rc)
    # a null q is a bad argument, reported before the size check
    rc = lib.spd_varlen_attn_fwd_noalloc(None, P(q.data_ptr()), P(q.data_ptr()), P(q.data_ptr()),
                                         1 << 17, (1 << 24) + (1 << 17), 0, 2, 2, 128, ctypes.c_float(0.0),
                                         P(out.data_ptr()), P(lse.data_ptr()), None,
                                         P(torch.cuda.current_stream().cuda_stream))
    assert rc == -1
    cu = torch.tensor([0, 200, 100, 256], dtype=torch.int32, device="cuda")
    assert _call_noalloc(lib, q, q, q, cu, 3, out, lse, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == -4


def test_noalloc_random_problems_equal_the_workspace_entry_point():
    """A seeded sweep of problems on the shared fixed scratch, back to back:
    the output equals the workspace entry point's bit for bit every time."""
    from sample_packing_document_gb300 import workloads as W
    lib, ops = _lib()
    rng = np.random.default_rng(4242)
    for case in range(30):
        nseg = int(rng.integers(1, 12))
        lens = rng.integers(1, 2000, size=nseg).tolist()
        Hq, Hkv = [(1, 1), (4, 2), (7, 1), (4, 4)][int(rng.integers(4))]
        d = 64 if rng.random() < 0.4 else 128
        cu_h = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu_h[-1])
        q, k, v, _ = W.qkv(T, Hq, Hkv, d, seed=600 + case, device="cuda")
        cu = torch.tensor(cu_h, device="cuda")
        out_ref, lse_ref = ops.varlen_attn_fwd(q, k, v, cu, nseg)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((Hq, T), float("nan"), device="cuda")
        status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
        assert _call_noalloc(lib, q, k, v, cu, nseg, out, lse, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(out, out_ref) and torch.equal(lse, lse_ref), (case, lens, Hq, Hkv, d)
