"""spd_rope on the GPU against the fp64 oracle: per-document positions from a
packed batch (documents up to 20K tokens long), both head dims, GQA head
counts, the inverse rotation; position 0 must leave a row bit for bit."""
import numpy as np
import pytest
import torch

from oracle import rope as R

pytestmark = pytest.mark.gpu


def _ops():
    from sample_packing_document_gb300 import build, ops
    build.build()
    return ops


def _bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _positions(T, seed):
    """indexes of a packed row: positions restart at every document start."""
    rng = np.random.default_rng(seed)
    pos, n = [], 0
    while n < T:
        L = int(min(rng.integers(1, 20000), T - n))
        pos.extend(range(L))
        n += L
    return np.array(pos, dtype=np.int32)


def _check(got, want):
    """bf16 rounding of the result (half an ulp = 2^-8 relative) plus fp32 work."""
    got = got.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - want)
    assert np.all(err <= 2.0 ** -8 * np.abs(want) + 1e-5 * np.abs(want).max()), float(err.max())


@pytest.mark.parametrize("T,Hq,Hkv,d,theta", [(3000, 4, 2, 128, 10000.0), (40000, 7, 1, 128, 1.0e6),
                                              (5000, 2, 2, 64, 10000.0), (257, 1, 1, 64, 500.0)])
def test_rope_matches_oracle(T, Hq, Hkv, d, theta):
    ops = _ops()
    q0, k0 = _bf16((T, Hq, d), 1), _bf16((T, Hkv, d), 2)
    pos = _positions(T, T)
    q, k = q0.cuda(), k0.cuda()
    p = torch.tensor(pos, device="cuda")
    ops.rope(q, k, p, rope_theta=theta)
    torch.cuda.synchronize()
    _check(q, R.rope(q0.float().numpy(), pos, theta))
    _check(k, R.rope(k0.float().numpy(), pos, theta))
    # the inverse rotation of the rotated (bf16) tensors, against the oracle's inverse of the same bits
    q1, k1 = q.clone(), k.clone()
    ops.rope(q, k, p, rope_theta=theta, inverse=True)
    torch.cuda.synchronize()
    _check(q, R.rope(q1.float().cpu().numpy(), pos, theta, inverse=True))
    _check(k, R.rope(k1.float().cpu().numpy(), pos, theta, inverse=True))


def test_rope_position_zero_is_exact_and_q_only():
    ops = _ops()
    T, H, d = 512, 3, 128
    x0 = _bf16((T, H, d), 5)
    x = x0.cuda()
    ops.rope(x, None, torch.zeros(T, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(x.cpu(), x0)


def test_rope_host_checks():
    ops = _ops()
    lib = ops.load()
    x = torch.zeros((4, 2, 128), dtype=torch.bfloat16, device="cuda")
    p = torch.zeros(4, dtype=torch.int32, device="cuda")
    import ctypes
    P = ctypes.c_void_p
    assert lib.spd_rope(P(x.data_ptr()), None, P(p.data_ptr()), 4, 2, 0, 96, ctypes.c_float(0), 0, None) == -2
    assert lib.spd_rope(P(x.data_ptr() + 2), None, P(p.data_ptr()), 4, 2, 0, 128, ctypes.c_float(0), 0, None) == -1
    assert lib.spd_rope(P(x.data_ptr()), None, None, 4, 2, 0, 128, ctypes.c_float(0), 0, None) == -1
