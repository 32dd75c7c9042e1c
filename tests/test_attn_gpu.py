"""GPU parity of spd_varlen_attn_fwd / spd_varlen_attn_bwd against the fp64
oracle on the same bf16 inputs.

Bars (stated for this library): max |O - O_ref| <= 2e-2, max |LSE - LSE_ref|
<= 1e-3, and max |g - g_ref| <= 5e-2 for dQ, dK, dV, whether the gradients
are written as fp32 or as bf16 (the benchmarked form).

Small cases (several tiles, ragged tails, every segment-length class around
the 128-token tile, GQA groups 1 / 2 / 3 / 7, head_dim 64 and 128) are
compared element by element over all outputs. The five workloads at full size
run with bf16 and with fp32 gradient outputs and are compared on sampled rows
(forward and dQ: any segment, including the longest; dK / dV: whole short
segments) plus finiteness everywhere; on the 32K and 131K workloads one long
segment is compared whole for one kv head's group (dK / dV summed over
hundreds of q-tile steps), and a 33000-token document is compared whole.
The tile schedules the kernels run are read back and checked against the
tile counts the pages give.
"""
import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import pack as P

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE, TOL_G = 2e-2, 1e-3, 5e-2


@pytest.fixture(scope="module")
def ops():
    from sample_packing_document_gb300 import build, ops as _ops
    build.build()
    _ops.load()
    return _ops


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _inputs(T, Hq, Hkv, d, seed, q_scale=1.0, device="cuda"):
    from sample_packing_document_gb300 import workloads as W
    return W.qkv(T, Hq, Hkv, d, seed, device=device, q_scale=q_scale)


def _run(ops, q, k, v, do, cu, scale=None, grad_dtype=torch.float32):
    cu_t = torch.tensor(np.asarray(cu, np.int32), device="cuda")
    ns = len(cu) - 1
    ws_f = ops.workspace(ops.attn_workspace_size(q.shape[0], ns, q.shape[1], k.shape[1], q.shape[2], False))
    out, lse = ops.varlen_attn_fwd(q, k, v, cu_t, ns, softmax_scale=scale, ws=ws_f)
    assert ops.read_status(ws_f) == 0
    ws_b = ops.workspace(ops.attn_workspace_size(q.shape[0], ns, q.shape[1], k.shape[1], q.shape[2], True))
    dq, dk, dv = ops.varlen_attn_bwd(q, k, v, out, do, lse, cu_t, ns, softmax_scale=scale, grad_dtype=grad_dtype,
                                     ws=ws_b)
    assert ops.read_status(ws_b) == 0
    torch.cuda.synchronize()
    return out, lse, dq, dk, dv


def _maxerr(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def _check_full(ops, lens, Hq, Hkv, d, seed, scale=None, grad_dtype=torch.float32, q_scale=1.0):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, do = _inputs(T, Hq, Hkv, d, seed, q_scale=q_scale)
    out, lse, dq, dk, dv = _run(ops, q, k, v, do, cu, scale, grad_dtype)
    qn, kn, vn, don = _u16(q), _u16(k), _u16(v), _u16(do)
    o_ref, lse_ref = OA.attn_fwd(qn, kn, vn, cu, scale=scale)
    o_gpu = out.float().cpu().numpy().transpose(1, 0, 2)
    assert _maxerr(o_gpu, o_ref) <= TOL_O
    assert _maxerr(lse.cpu().numpy(), lse_ref) <= TOL_LSE
    gq, gk, gv, _ = OA.attn_bwd(qn, kn, vn, don, cu, scale=scale)
    print("parity lens=%s Hq=%d Hkv=%d d=%d: |dO| %.3g |dLSE| %.3g |ddq| %.3g |ddk| %.3g |ddv| %.3g "
          "(max |dq| %.3g |dk| %.3g |dv| %.3g)" % (
              lens[:8], Hq, Hkv, d, _maxerr(o_gpu, o_ref), _maxerr(lse.cpu().numpy(), lse_ref),
              _maxerr(dq.float().cpu().numpy(), gq), _maxerr(dk.float().cpu().numpy(), gk),
              _maxerr(dv.float().cpu().numpy(), gv), np.abs(gq).max(), np.abs(gk).max(), np.abs(gv).max()))
    for g, ref in ((dq, gq), (dk, gk), (dv, gv)):
        assert _maxerr(g.float().cpu().numpy(), ref) <= TOL_G
    return out, lse, dq, dk, dv, (qn, kn, vn, don, cu)


@pytest.mark.parametrize("lens,Hq,Hkv,d", [
    ([3, 4, 5, 4], 2, 2, 64),                       # the page's documents 3, 4, 5, 4
    ([300, 1, 129, 517, 2, 128, 1000], 4, 2, 128),  # tiles, ragged tails, 1 / 2 / 128 / 129
    ([1, 250, 127, 384, 64], 6, 2, 64),             # head_dim 64, group 3
    ([1100], 1, 1, 128),                            # one document, 9 tiles
    ([700, 33, 1290], 7, 1, 128),                   # group 7 (one sequence-parallel rank of 56 / 8)
    ([256, 255, 257], 2, 2, 128),
])
def test_small_cases_full_compare(ops, lens, Hq, Hkv, d):
    _check_full(ops, lens, Hq, Hkv, d, seed=sum(lens) % 97)


@pytest.mark.parametrize("lens,Hq,Hkv,d", [
    ([400, 77, 900], 4, 4, 128),
    ([1, 250, 127, 384, 64], 6, 2, 64),             # head_dim 64 (no TMA-box store of dK / dV), group 3
    ([700, 33, 1290], 7, 1, 128),                   # group 7
])
def test_bf16_gradient_output(ops, lens, Hq, Hkv, d):
    _check_full(ops, lens, Hq, Hkv, d, seed=3, grad_dtype=torch.bfloat16)


def test_custom_scale_and_scaled_q(ops):
    """softmax_scale other than 1/sqrt(d), and q drawn as N(0, 1) / sqrt(128).
    The bars are absolute, so the cases keep the gradients at the magnitude of
    the workloads: dQ = scale * sum_j dS_ij k_j grows with the scale, and its
    error (the bf16 rounding of dS, relative 2^-9) grows with it."""
    _check_full(ops, [333, 555], 4, 2, 128, seed=4, scale=0.06)
    _check_full(ops, [333, 555], 4, 2, 128, seed=5, q_scale=1.0 / np.sqrt(128.0))
    _check_full(ops, [100, 901], 2, 1, 64, seed=6, scale=0.2)


def test_length_one_documents(ops):
    """P = 1 for every row: O equals V bit for bit; dQ, dK vanish; dV is the
    group sum of dO."""
    out, lse, dq, dk, dv, (qn, kn, vn, don, cu) = _check_full(ops, [1] * 200, 4, 2, 128, seed=6)
    o = out.cpu()
    vv = torch.from_numpy(vn.view(np.int16)).view(torch.bfloat16)
    for h in range(4):
        assert torch.equal(o[:, h, :], vv[:, h // 2, :])
    assert float(dq.abs().max()) < 1e-4 and float(dk.abs().max()) < 1e-4


def test_many_segments(ops):
    """Thousands of segments (4500 one-token documents, then two longer ones):
    the scheduler's per-segment offsets and search at that count."""
    _check_full(ops, [1] * 4500 + [300, 129], 2, 2, 64, seed=9)


def test_packed_row_from_pack_kernel(ops):
    """The pipeline: pack_tokens' cu_seqlens (documents split across rows and a
    padding tail) feed the attention calls directly."""
    rng = np.random.default_rng(12)
    lens = rng.integers(20, 700, size=17).astype(np.int32)
    toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
    mb, sl = 2, 1024
    po = ops.pack_tokens(torch.tensor(toks, device="cuda"), torch.tensor(lens, device="cuda"), mb, sl, True)
    ns = int(po["num_segs"].item())
    cu_gpu = po["cu_seqlens"][:ns + 1].cpu().numpy()
    ref = P.pack_flat([toks[a:b].tolist() for a, b in zip(np.r_[0, np.cumsum(lens)[:-1]], np.cumsum(lens))],
                      mb, sl, True)
    np.testing.assert_array_equal(cu_gpu, ref["cu_seqlens"])
    lens_seg = np.diff(cu_gpu)
    _check_full(ops, lens_seg.tolist(), 4, 2, 128, seed=7)


def test_mid_size_full_compare(ops):
    rng = np.random.default_rng(21)
    lens = rng.integers(1, 1500, size=9).tolist() + [3000]
    _check_full(ops, lens, 4, 2, 128, seed=8)


def test_backward_workspace_reuse(ops):
    """One backward workspace used again and again: repeated calls, a call of
    another shape (the workspace regions move), the first shape again, and a
    workspace full of garbage must all match the oracle (nothing a call leaves
    behind in the workspace may leak into the next)."""
    Hq, Hkv, d = 4, 2, 128
    shapes = ([300, 1, 129, 517], [700, 260])
    size = max(ops.attn_workspace_size(sum(l), len(l), Hq, Hkv, d, True) for l in shapes)
    ws_b = ops.workspace(size)
    cases = []
    for n, lens in enumerate(shapes):
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        T = int(cu[-1])
        q, k, v, do = _inputs(T, Hq, Hkv, d, 30 + n)
        cu_t = torch.tensor(cu, device="cuda")
        ws_f = ops.workspace(ops.attn_workspace_size(T, len(lens), Hq, Hkv, d, False))
        out, lse = ops.varlen_attn_fwd(q, k, v, cu_t, len(lens), ws=ws_f)
        ref = OA.attn_bwd(_u16(q), _u16(k), _u16(v), _u16(do), cu)[:3]
        cases.append((q, k, v, do, out, lse, cu_t, len(lens), ref))

    def check(c):
        q, k, v, do, out, lse, cu_t, ns, ref = c
        g = ops.varlen_attn_bwd(q, k, v, out, do, lse, cu_t, ns, grad_dtype=torch.float32, ws=ws_b)
        assert ops.read_status(ws_b) == 0
        for x, r in zip(g, ref):
            assert _maxerr(x.float().cpu().numpy(), r) <= TOL_G

    for c in (cases[0], cases[0], cases[0], cases[1], cases[1], cases[0]):
        check(c)
    ws_b.fill_(0x7f)           # memory used for something else in between
    check(cases[1])
    check(cases[1])


def test_bad_seqlens_set_status(ops):
    q, k, v, do = _inputs(512, 2, 2, 128, 1)
    for cu in ([0, 300, 200, 512], [0, 300, 511], [1, 300, 512], [0, 300, 300, 512]):
        cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
        ws = ops.workspace(ops.attn_workspace_size(512, len(cu) - 1, 2, 2, 128, True))
        ops.varlen_attn_fwd(q, k, v, cu_t, len(cu) - 1, ws=ws)
        assert ops.read_status(ws) == -4
        out = torch.zeros_like(q)
        lse = torch.zeros(2, 512, device="cuda")
        ops.varlen_attn_bwd(q, k, v, out, do, lse, cu_t, len(cu) - 1, ws=ws)
        assert ops.read_status(ws) == -4
    cu_t = torch.tensor([0, 200, 512], dtype=torch.int32, device="cuda")   # the context is still good
    ws = ops.workspace(ops.attn_workspace_size(512, 2, 2, 2, 128, False))
    ops.varlen_attn_fwd(q, k, v, cu_t, 2, ws=ws)
    assert ops.read_status(ws) == 0


# ----------------------------------------------------------------------------- full size

def _workload_inputs(name):
    from sample_packing_document_gb300 import workloads as W
    w = W.WORKLOADS[name]
    lens, toks = W.documents(w)
    flat = OA.pack(toks, lens, w.micro_bsz, w.seq_len, w.use_packed_dataset)
    cu = flat["cu_seqlens"]
    T = int(cu[-1])
    q, k, v, do = _inputs(T, w.Hq, w.Hkv, w.head_dim, w.seed, q_scale=w.q_scale)
    return w, cu, q, k, v, do


def _segment_group_compare(qn, kn, vn, don, cu, s, g, group, grads, label):
    """Whole-segment gradient check for kv head g of segment s: the oracle on
    that segment alone with the q heads of g's group (segments and kv groups
    never interact, the equivalence the pages state), against the slice of the
    full-size GPU result."""
    a, b = int(cu[s]), int(cu[s + 1])
    hs = slice(g * group, (g + 1) * group)
    sub = lambda x, h: np.ascontiguousarray(x[a:b, h])
    gq, gk, gv, _ = OA.attn_bwd(sub(qn, hs), sub(kn, slice(g, g + 1)), sub(vn, slice(g, g + 1)), sub(don, hs),
                                np.array([0, b - a], np.int32))
    for gdt, (dq, dk, dv) in grads.items():
        e = (_maxerr(dq.float().cpu().numpy()[a:b, hs], gq), _maxerr(dk.float().cpu().numpy()[a:b, g:g + 1], gk),
             _maxerr(dv.float().cpu().numpy()[a:b, g:g + 1], gv))
        print("%s segment %d (%d tokens), kv head %d, %s grads: |ddq| %.3g |ddk| %.3g |ddv| %.3g "
              "(max |dq| %.3g |dk| %.3g |dv| %.3g)" % (label, s, b - a, g, gdt, *e, np.abs(gq).max(),
                                                      np.abs(gk).max(), np.abs(gv).max()))
        assert max(e) <= TOL_G, (gdt, e)


@pytest.mark.parametrize("name", ["tiny", "c2", "c3", "c4", "c5"])
def test_workload_full_size_sampled(ops, name):
    """Full-size workload, forward once, backward with bf16 gradients (what
    the bench times) and with fp32 gradients, both against the fp64 oracle at
    the same bars."""
    w, cu, q, k, v, do = _workload_inputs(name)
    T, Hq = q.shape[0], q.shape[1]
    out, lse, dq, dk, dv = _run(ops, q, k, v, do, cu, grad_dtype=torch.bfloat16)
    grads = {"bf16": (dq, dk, dv)}
    cu_t = torch.tensor(np.asarray(cu, np.int32), device="cuda")
    ws_b = ops.workspace(ops.attn_workspace_size(T, len(cu) - 1, Hq, k.shape[1], q.shape[2], True))
    grads["fp32"] = ops.varlen_attn_bwd(q, k, v, out, do, lse, cu_t, len(cu) - 1, grad_dtype=torch.float32, ws=ws_b)
    assert ops.read_status(ws_b) == 0
    for t in (out, lse) + grads["bf16"] + grads["fp32"]:
        assert bool(torch.isfinite(t).all())
    qn, kn, vn, don = _u16(q), _u16(k), _u16(v), _u16(do)
    rng = np.random.default_rng(77)
    lens = np.diff(cu)
    longest = int(np.argmax(lens))
    rows = list(rng.integers(0, T, size=96))
    rows += [int(cu[longest]), int(cu[longest + 1]) - 1, int(cu[longest + 1]) - 129, int(cu[1]) - 1]
    rows = [r for r in rows if 0 <= r < T]
    items = np.array([(int(rng.integers(0, Hq)) * T + r) for r in rows], np.int64)
    o_ref, lse_ref = OA.attn_fwd(qn, kn, vn, cu, items=items)
    o_gpu = out.float().cpu().numpy().reshape(T, Hq, -1)
    lse_gpu = lse.cpu().numpy()
    for n, it in enumerate(items):
        h, i = divmod(int(it), T)
        assert _maxerr(o_gpu[i, h], o_ref[n]) <= TOL_O
        assert abs(float(lse_gpu[h, i]) - lse_ref[n]) <= TOL_LSE
    dq_items = items[:48]
    dq_ref = OA.attn_dq_rows(qn, kn, vn, don, cu, dq_items)
    for gdt, (dq_, _, _) in grads.items():
        dq_gpu = dq_.float().cpu().numpy()
        for n, it in enumerate(dq_items):
            h, i = divmod(int(it), T)
            assert _maxerr(dq_gpu[i, h], dq_ref[n]) <= TOL_G, gdt
    # dK / dV: whole segments, the shortest ones and one of up to 2048 tokens
    order = np.argsort(lens, kind="stable")
    segs = [int(s) for s in order[:3]]
    mid = [int(s) for s in order if lens[s] <= 2048]
    if mid and mid[-1] not in segs:
        segs.append(mid[-1])
    gq, gk, gv, srows = OA.attn_bwd(qn, kn, vn, don, cu, segs=segs)
    print("%s: max |ref| over the compared segments: dq %.3g dk %.3g dv %.3g" % (
        name, np.abs(gq).max(), np.abs(gk).max(), np.abs(gv).max()))
    for gdt, (dq_, dk_, dv_) in grads.items():
        assert _maxerr(dk_.float().cpu().numpy()[srows], gk) <= TOL_G, gdt
        assert _maxerr(dv_.float().cpu().numpy()[srows], gv) <= TOL_G, gdt
        assert _maxerr(dq_.float().cpu().numpy()[srows], gq) <= TOL_G, gdt
    # one long segment whole, for the q heads of one kv head: c3's longest
    # (11470 tokens, 4 q heads), c4's fourth longest (11809 tokens, 7 q heads)
    pick = {"c3": 0, "c4": 3}
    if name in pick:
        s = int(np.argsort(-lens, kind="stable")[pick[name]])
        _segment_group_compare(qn, kn, vn, don, cu, s, 0, Hq // k.shape[1], grads, name)


def test_long_document_whole_compare(ops):
    """A 33000-token document (258 tiles: kv tile 0 sums dK / dV over 516 q-tile
    steps of two q heads) plus short ones, every gradient element compared,
    bf16 gradient outputs (the benchmarked form)."""
    _check_full(ops, [33000, 700, 5, 1], 2, 1, 128, seed=13, grad_dtype=torch.bfloat16)


SINGLE = 1 << 30     # backward schedule: the unit is one kv tile, not a pair


def _blocks_of_schedule(units, bwd):
    """(segment start, q tile, kv tile) blocks the schedule visits, from the
    unit meaning spd_attn_read_schedule documents."""
    blocks = []
    for a, b, t, cost in units.tolist():
        n = -(-(b - a) // 128)
        if bwd:
            kvs = [t & ~SINGLE] if t & SINGLE else sorted({t, n - 1 - t})
            got = [(a, i, kv) for kv in kvs for i in range(kv, n)]
        else:
            got = [(a, i, j) for i in (t, t + 1) if i < n for j in range(i + 1)]
        assert cost == len(got), (a, b, t, cost)
        blocks += got
    return blocks


def _unmasked_pairs(a, b, qi, kj):
    """Entries (i, j) of block (q tile qi, kv tile kj) of segment [a, b) with
    a <= j <= i < b."""
    n = 0
    for i in range(a + 128 * qi, min(b, a + 128 * qi + 128)):
        lo, hi = a + 128 * kj, min(b, a + 128 * kj + 128, i + 1)
        n += max(0, hi - lo)
    return n


@pytest.mark.parametrize("lens,blocks_per_head,pairs", [
    ([3, 4, 5, 4], 4, 41),               # the page's documents 3, 4, 5, 4: 41 kept entries of 136
    ([16384, 16384], 16512, None),       # two 16K documents in 32K: 16512 tiles of 65536 (74.80% skipped)
    ([300, 1, 129, 517, 2, 128, 1000], None, None),
    ([20000, 2048, 2100, 4000, 77, 3000], None, None),   # long and short: the backward pairs kv tiles
])
def test_schedule_visits_exactly_the_unmasked_tiles(ops, lens, blocks_per_head, pairs):
    """The work lists the forward and backward kernels run, read back from the
    workspace: every (q tile, kv tile) block with an unmasked entry is visited
    once per head, no other block is, the lists are longest first, and the
    totals are the page's (section 5.1 tile classes and its sparsity figure)."""
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, do = _inputs(T, 2, 1, 128, 3)
    cu_t = torch.tensor(cu, device="cuda")
    ws_f = ops.workspace(ops.attn_workspace_size(T, len(lens), 2, 1, 128, False))
    ws_b = ops.workspace(ops.attn_workspace_size(T, len(lens), 2, 1, 128, True))
    out, lse = ops.varlen_attn_fwd(q, k, v, cu_t, len(lens), ws=ws_f)
    ops.varlen_attn_bwd(q, k, v, out, do, lse, cu_t, len(lens), ws=ws_b)
    want = set()
    for a, b in zip(cu[:-1], cu[1:]):
        n = -(-(int(b) - int(a)) // 128)
        want |= {(int(a), i, j) for i in range(n) for j in range(i + 1)}
    for ws, bwd in ((ws_f, False), (ws_b, True)):
        units = ops.read_schedule(ws)
        assert np.all(np.diff(units[:, 3]) <= 0)              # longest first
        if bwd:                                                # a segment's pairs in consecutive slots, in order
            pair = (units[:, 2] & SINGLE) == 0
            if lens[0] == 20000:
                assert pair.sum() > 0
            for a in np.unique(units[pair, 0]):
                ts = units[pair & (units[:, 0] == a), 2]
                assert ts.tolist() == list(range(len(ts)))
                assert np.all(np.diff(np.flatnonzero(pair & (units[:, 0] == a))) == 1)
        blocks = _blocks_of_schedule(units, bwd)
        assert len(blocks) == len(set(blocks))                 # each block once
        assert set(blocks) == want                             # exactly the blocks with unmasked entries
        seg_end = {int(a): int(b) for a, b in zip(cu[:-1], cu[1:])}
        kept = [_unmasked_pairs(a, seg_end[a], i, j) for a, i, j in blocks]
        assert min(kept) > 0
        if blocks_per_head is not None:
            assert len(blocks) == blocks_per_head
        if pairs is not None:
            assert sum(kept) == pairs
        assert sum(kept) == sum(L * (L + 1) // 2 for L in lens)


def test_paired_backward_units_full_compare(ops):
    """Random document lengths of 2100-2900 tokens (17-23 kv tiles) with enough
    heads that the backward schedule pairs their kv tiles p and n - 1 - p into
    one unit (the second walking its q tiles downward): the schedule read back
    holds pairs, and every output element of the forward and of both gradient
    forms (bf16 and fp32) meets the bars against the oracle."""
    rng = np.random.default_rng(808)
    lens = rng.integers(2100, 2901, size=3).tolist()
    Hq = Hkv = 48
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k, v, do = _inputs(T, Hq, Hkv, 64, 12)
    cu_t = torch.tensor(cu, device="cuda")
    ws_b = ops.workspace(ops.attn_workspace_size(T, len(lens), Hq, Hkv, 64, True))
    out, lse = ops.varlen_attn_fwd(q, k, v, cu_t, len(lens))
    g32 = ops.varlen_attn_bwd(q, k, v, out, do, lse, cu_t, len(lens), grad_dtype=torch.float32, ws=ws_b)
    assert ops.read_status(ws_b) == 0
    units = ops.read_schedule(ws_b)
    assert ((units[:, 2] & SINGLE) == 0).sum() > 0            # paired units were scheduled
    g16 = ops.varlen_attn_bwd(q, k, v, out, do, lse, cu_t, len(lens), grad_dtype=torch.bfloat16, ws=ws_b)
    assert ops.read_status(ws_b) == 0
    qn, kn, vn, don = _u16(q), _u16(k), _u16(v), _u16(do)
    o_ref, lse_ref = OA.attn_fwd(qn, kn, vn, cu)
    assert _maxerr(out.float().cpu().numpy().transpose(1, 0, 2), o_ref) <= TOL_O
    assert _maxerr(lse.cpu().numpy(), lse_ref) <= TOL_LSE
    refs = OA.attn_bwd(qn, kn, vn, don, cu)[:3]
    for g, ref in zip(g32, refs):
        assert _maxerr(g.cpu().numpy(), ref) <= TOL_G
    for g, ref in zip(g16, refs):
        assert _maxerr(g.float().cpu().numpy(), ref) <= TOL_G
