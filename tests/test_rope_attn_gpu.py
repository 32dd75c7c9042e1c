"""spd_varlen_attn_fwd_rope (RoPE fused into the attention prologue) against
the oracle's composition: the fp64 rotation of q and k by per-document
positions (oracle/rope.py), rounded to bf16 as every attention input is, then
the fp64 attention oracle. Bars as for the plain forward: max |O - O_ref| <=
2e-2, max |LSE - LSE_ref| <= 1e-3.

Positions are each token's offset inside its segment of cu_seqlens; for a
batch from spd_pack_tokens they equal its `indexes` (checked here). The fused
call is also compared with the unfused GPU path (spd_rope on copies of q and k,
then spd_varlen_attn_fwd)."""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import pack as P
from oracle import rope as R

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 2e-2, 1e-3


@pytest.fixture(scope="module")
def ops():
    from sample_packing_document_gb300 import build, ops as _ops
    build.build()
    _ops.load()
    return _ops


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bf16_bits(x):
    """Round to bf16 (round to nearest even), as bit patterns."""
    u = np.asarray(x, np.float64).astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _positions(cu):
    T = int(cu[-1])
    seg = np.repeat(np.arange(len(cu) - 1), np.diff(cu))
    return (np.arange(T) - np.asarray(cu)[seg]).astype(np.int64)


def _reference(q, k, v, cu, theta, items=None):
    pos = _positions(cu)
    qr = _bf16_bits(R.rope(_f64(_u16(q)), pos, theta))
    kr = _bf16_bits(R.rope(_f64(_u16(k)), pos, theta))
    return OA.attn_fwd(qr, kr, _u16(v), np.asarray(cu, np.int32), items=items)


def _run(ops, lens, Hq, Hkv, d, theta, seed):
    from sample_packing_document_gb300 import workloads as W
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, _ = W.qkv(T, Hq, Hkv, d, seed, device="cuda")
    cu_t = torch.tensor(cu, device="cuda")
    ws = ops.workspace(ops.attn_workspace_size(T, len(lens), Hq, Hkv, d, False))
    q_in, k_in = q.clone(), k.clone()
    out, lse = ops.varlen_attn_fwd_rope(q, k, v, cu_t, len(lens), rope_theta=theta, ws=ws)
    assert ops.read_status(ws) == 0
    assert torch.equal(q, q_in) and torch.equal(k, k_in)      # inputs are read, not rotated in place
    return cu, q, k, v, out, lse


@pytest.mark.parametrize("lens,Hq,Hkv,d,theta", [
    ([300, 1, 129, 517, 2, 128, 1000], 4, 2, 128, 10000.0),   # ragged tails, 1 / 2 / 128 / 129 tokens
    ([1, 250, 127, 384, 64], 6, 2, 64, 500000.0),             # head_dim 64, group 3
    ([700, 33, 1290], 7, 1, 128, 1.0e6),                       # group 7
    ([20000, 700, 33], 2, 1, 128, 10000.0),                    # positions up to 20K: 157 tiles of one document
])
def test_fused_rope_forward_matches_oracle(ops, lens, Hq, Hkv, d, theta):
    cu, q, k, v, out, lse = _run(ops, lens, Hq, Hkv, d, theta, seed=sum(lens) % 89)
    o_ref, lse_ref = _reference(q, k, v, cu, theta)
    e_o = float(np.abs(out.float().cpu().numpy().transpose(1, 0, 2) - o_ref).max())
    e_l = float(np.abs(lse.cpu().numpy() - lse_ref).max())
    print("fused rope lens=%s Hq=%d Hkv=%d d=%d theta=%g: |dO| %.3g |dLSE| %.3g" % (lens, Hq, Hkv, d, theta, e_o, e_l))
    assert e_o <= TOL_O and e_l <= TOL_LSE


def test_fused_rope_equals_rope_then_attention_on_gpu(ops):
    """The unfused GPU path (spd_rope on copies of q and k with the pack's
    indexes, then the plain forward) gives the same attention."""
    rng = np.random.default_rng(31)
    lens = rng.integers(20, 3000, size=9).astype(np.int32)
    toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
    mb, sl = 2, 4096
    po = ops.pack_tokens(torch.tensor(toks, device="cuda"), torch.tensor(lens, device="cuda"), mb, sl, True)
    ns = int(po["num_segs"].item())
    cu_t = po["cu_seqlens"][:ns + 1].contiguous()
    cu = cu_t.cpu().numpy()
    idx = po["indexes"].cpu().numpy()
    np.testing.assert_array_equal(idx, _positions(cu))         # positions from cu_seqlens = the pack's indexes
    ref = P.pack_flat([toks[a:b].tolist() for a, b in zip(np.r_[0, np.cumsum(lens)[:-1]], np.cumsum(lens))],
                      mb, sl, True)
    np.testing.assert_array_equal(idx, ref["indexes"])
    from sample_packing_document_gb300 import workloads as W
    T = int(cu[-1])
    q, k, v, _ = W.qkv(T, 4, 2, 128, 5, device="cuda")
    out_f, lse_f = ops.varlen_attn_fwd_rope(q, k, v, cu_t, ns, rope_theta=10000.0)
    qr, kr = q.clone(), k.clone()
    ops.rope(qr, kr, po["indexes"], rope_theta=10000.0)
    out_u, lse_u = ops.varlen_attn_fwd(qr, kr, v, cu_t, ns)
    torch.cuda.synchronize()
    assert float((out_f.float() - out_u.float()).abs().max()) <= TOL_O
    assert float((lse_f - lse_u).abs().max()) <= TOL_LSE
    o_ref, lse_ref = _reference(q, k, v, cu, 10000.0)
    assert float(np.abs(out_f.float().cpu().numpy().transpose(1, 0, 2) - o_ref).max()) <= TOL_O


def test_fused_rope_position_zero_is_identity(ops):
    """Length-1 documents sit at position 0, where the rotation is the identity:
    O equals V bit for bit, as without RoPE."""
    cu, q, k, v, out, lse = _run(ops, [1] * 300, 4, 2, 128, 10000.0, seed=3)
    o = out.cpu()
    vv = v.cpu()
    for h in range(4):
        assert torch.equal(o[:, h, :], vv[:, h // 2, :])


def test_fused_rope_full_size_sampled(ops):
    """The 131K-token sequence-parallel rank shape (7 q / 1 kv heads, documents
    up to 19725 tokens) on sampled rows, including the longest document's last
    rows (positions near 20K)."""
    from sample_packing_document_gb300 import workloads as W
    w = W.WORKLOADS["c4"]
    lens, toks = W.documents(w)
    flat = OA.pack(toks, lens, w.micro_bsz, w.seq_len, w.use_packed_dataset)
    cu = flat["cu_seqlens"]
    T = int(cu[-1])
    q, k, v, _ = W.qkv(T, w.Hq, w.Hkv, w.head_dim, w.seed, device="cuda")
    cu_t = torch.tensor(cu, device="cuda")
    out, lse = ops.varlen_attn_fwd_rope(q, k, v, cu_t, len(cu) - 1, rope_theta=10000.0)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    s = int(np.argmax(np.diff(cu)))
    rows = list(rng.integers(0, T, size=40)) + [int(cu[s + 1]) - 1, int(cu[s + 1]) - 200]
    items = np.array([int(rng.integers(0, w.Hq)) * T + r for r in rows], np.int64)
    pos = _positions(cu)
    # the oracle needs only the rows' own segments rotated: rotate everything once
    qr = _bf16_bits(R.rope(_f64(_u16(q)), pos, 10000.0))
    kr = _bf16_bits(R.rope(_f64(_u16(k)), pos, 10000.0))
    o_ref, lse_ref = OA.attn_fwd(qr, kr, _u16(v), cu, items=items)
    o = out.float().cpu().numpy()
    l = lse.cpu().numpy()
    for n, it in enumerate(items):
        h, i = divmod(int(it), T)
        assert float(np.abs(o[i, h] - o_ref[n]).max()) <= TOL_O
        assert abs(float(l[h, i]) - lse_ref[n]) <= TOL_LSE


@pytest.mark.parametrize("block", range(4))
def test_fused_rope_random_problems(ops, block):
    """A seeded sweep: 1-8 segments with lengths at the tile edges or uniform
    below 1500, GQA groups 1, 2, 3, 7, head_dim 64 / 128, rope_theta from 10^2
    to 10^6; every output against the oracle's rotation then attention."""
    rng = np.random.default_rng(7100 + block)
    edges = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257]
    heads = [(1, 1), (2, 2), (2, 1), (6, 2), (7, 1)]
    for case in range(10):
        nseg = int(rng.integers(1, 9))
        lens = [int(rng.choice(edges)) if rng.random() < 0.5 else int(rng.integers(1, 1500)) for _ in range(nseg)]
        Hq, Hkv = heads[int(rng.integers(len(heads)))]
        d = 64 if rng.random() < 0.4 else 128
        theta = float(10.0 ** rng.uniform(2, 6))
        cu, q, k, v, out, lse = _run(ops, lens, Hq, Hkv, d, theta, seed=300 + 10 * block + case)
        o_ref, lse_ref = _reference(q, k, v, cu, theta)
        what = (block, case, lens, Hq, Hkv, d, theta)
        assert float(np.abs(out.float().cpu().numpy().transpose(1, 0, 2) - o_ref).max()) <= TOL_O, what
        assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= TOL_LSE, what
