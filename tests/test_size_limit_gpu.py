"""The pack and the data steps at the largest size the ABI accepts: rows x
row length just below 2^31 - 65537 positions (positions are 32-bit in the
kernels, which step up to one chunk past the last position before their
bounds checks). The pack on each of its four paths: build_pack in one launch
(few documents) and in two (more than 1024 documents), build_unpack in one
launch and in two; then the sequence split (three tensors, 16-byte and
scalar paths), the sequence-parallel padding (a filled and a counting kind)
and unpack_data.

The outputs (25.8 GB) are far too large for the oracle's Python loops, so
they are checked against closed forms that hold at any size: the tokens are
t[i] = i mod 49999 + 1, and every output position is described by the
segment it falls in (its first position, the input position of that first
token, and the output position where its document's kept tokens end). The
segment list is built here from the document lengths alone (build_pack: the
documents end to end, cut at every row start, the padding tail its own
segment; build_unpack: micro_bsz documents per row, each cut to seq_len, then
the row's padding), and `test_segment_model_matches_oracle` pins that builder
to the oracle's build_pack / build_unpack on small random cases, element by
element.
"""
import random

import numpy as np
import pytest
import torch

from oracle import pack as P

LIMIT = 2 ** 31 - 65537
TOKEN_MOD = 49999


def segments(lens, mb, sl, packed):
    """(first position, end, input position of the first token or None for
    padding, output end of the document's kept tokens) for every segment, in
    order, plus the row count and row length."""
    plen = mb * sl
    nd = len(lens)
    total = int(sum(lens))
    out = []
    if packed:
        rows = -(-total // plen)
        start = 0
        for n in lens:
            end = start + int(n)
            a = start
            while a < end:                       # cut at every row start inside the document
                b = min(end, (a // plen + 1) * plen)
                out.append((a, b, a, end))
                a = b
            start = end
        if total < rows * plen:
            out.append((total, rows * plen, None, None))
    else:
        rows = -(-nd // mb)
        in_start = np.concatenate([[0], np.cumsum(np.asarray(lens, np.int64))]).astype(np.int64)
        for r in range(rows):
            o = r * plen
            for d in range(r * mb, min(nd, r * mb + mb)):
                keep = min(int(lens[d]), sl)
                out.append((o, o + keep, int(in_start[d]), o + keep))
                o += keep
            if o < (r + 1) * plen:
                out.append((o, (r + 1) * plen, None, None))
    return out, rows, plen


def segment_fields(segs, rows, plen):
    cu = [a for a, _, _, _ in segs] + [rows * plen]
    rsp, mx = [], [0] * rows
    i = 0
    for r in range(rows):
        while i < len(segs) and segs[i][0] < r * plen:
            i += 1
        rsp.append(i)
    rsp.append(len(segs))
    for a, b, _, _ in segs:
        mx[a // plen] = max(mx[a // plen], b - a)
    return cu, rsp, mx


def expected_small(toks, lens, mb, sl, packed):
    """Every output from the segment model (small cases only)."""
    segs, rows, plen = segments(lens, mb, sl, packed)
    n = rows * plen
    ids, lab, idx = [0] * n, [-100] * n, [0] * n
    for a, b, src, dend in segs:
        for p in range(a, b):
            idx[p] = p - a
            if src is not None:
                t = src + (p - a)
                ids[p] = toks[t]
                lab[p] = toks[t + 1] if p + 1 < dend else -100
    cu, rsp, mx = segment_fields(segs, rows, plen)
    return {"input_ids": ids, "labels": lab, "indexes": idx, "cu_seqlens": cu, "row_seg_ptr": rsp,
            "max_seqlen": mx, "num_segs": len(segs), "rows": rows}


def test_segment_model_matches_oracle():
    rng = random.Random(271)
    for packed in (True, False):
        for _ in range(400):
            mb, sl = rng.randint(1, 4), rng.randint(1, 12)
            docs = [[rng.randint(1, 49999) for _ in range(rng.randint(1, 3 * mb * sl))]
                    for _ in range(rng.randint(1, 9))]
            toks = [t for d in docs for t in d]
            got = expected_small(toks, [len(d) for d in docs], mb, sl, packed)
            ref = P.pack_flat(docs, mb, sl, packed)
            for key in ("input_ids", "labels", "indexes", "cu_seqlens", "row_seg_ptr", "max_seqlen", "num_segs",
                        "rows"):
                assert list(np.atleast_1d(got[key])) == list(np.atleast_1d(ref[key])), (packed, key)


# ------------------------------------------------------------------ GPU, at the size limit

def _tokens(n, device):
    t = torch.empty(n, dtype=torch.int32, device=device)
    step = 1 << 26
    for c0 in range(0, n, step):
        c1 = min(n, c0 + step)
        t[c0:c1] = (torch.arange(c0, c1, dtype=torch.int64, device=device) % TOKEN_MOD + 1).to(torch.int32)
    return t


def _check_outputs(out, segs, rows, plen):
    dev = out["input_ids"].device
    step = 1 << 26
    for a, b, src, dend in segs:
        for c0 in range(a, b, step):
            c1 = min(b, c0 + step)
            rel = torch.arange(c0 - a, c1 - a, dtype=torch.int64, device=dev)
            if src is None:
                ids = torch.zeros_like(rel)
                lab = torch.full_like(rel, -100)
            else:
                t = rel + src
                ids = t % TOKEN_MOD + 1
                lab = (t + 1) % TOKEN_MOD + 1
                if c0 <= dend - 1 < c1:           # the document's last kept token
                    lab[dend - 1 - c0] = -100
            assert torch.equal(out["input_ids"][c0:c1], ids.to(torch.int32)), ("input_ids", a, c0)
            assert torch.equal(out["labels"][c0:c1], lab.to(torch.int32)), ("labels", a, c0)
            assert torch.equal(out["indexes"][c0:c1], rel.to(torch.int32)), ("indexes", a, c0)
    cu, rsp, mx = segment_fields(segs, rows, plen)
    ns = int(out["num_segs"].item())
    assert ns == len(segs)
    assert out["cu_seqlens"][:ns + 1].cpu().tolist() == cu
    assert out["row_seg_ptr"][:rows + 1].cpu().tolist() == rsp
    assert out["max_seqlen"][:rows].cpu().tolist() == mx


def _case(name):
    rng = np.random.default_rng(1234)
    if name == "pack_one_launch":
        mb, sl, packed = 1, LIMIT // 2, True
        total = 2 * sl - 5                                  # a 5-token padding tail
        lens = [1, sl - 1, 123456789, 1]                    # the third document starts on row 1's start
        lens.append(total - sum(lens))
    elif name == "pack_two_launches":
        mb, sl, packed = 1, LIMIT // 2, True
        total = 2 * sl - 3
        lens = rng.integers(1, 2_000_000, size=1499).tolist()
        lens.append(total - sum(lens))
    elif name == "unpack_one_launch":
        mb, sl, packed = 2, LIMIT // 4, False
        lens = [sl + 7, 3, sl, 100]                         # cut, short, exact, short (padded row)
    else:                                                   # unpack_two_launches
        mb, packed = 1024, False
        sl = LIMIT // (2 * mb)
        lens = rng.integers(1, sl + sl // 4, size=2048).tolist()
    assert mb * sl * (-(-sum(lens) // (mb * sl)) if packed else -(-len(lens) // mb)) <= LIMIT
    return lens, mb, sl, packed


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["pack_one_launch", "pack_two_launches", "unpack_one_launch",
                                  "unpack_two_launches"])
def test_pack_at_the_position_limit(name):
    from sample_packing_document_gb300 import build, ops
    build.build()
    ops.load()
    lens, mb, sl, packed = _case(name)
    segs, rows, plen = segments(lens, mb, sl, packed)
    assert rows * plen > LIMIT - 4 * mb * sl // 1000     # within a fraction of a row of the limit
    dev = "cuda"
    toks = _tokens(int(sum(lens)), dev)
    lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
    out = ops.alloc_pack_outputs(len(lens), toks.numel(), mb, sl, packed, dev)
    assert out["rows"] == rows
    ops.pack_tokens(toks, lens_d, mb, sl, packed, out=out)
    assert ops.read_status(out["ws"]) == 0
    del toks
    _check_outputs(out, segs, rows, plen)
    del out
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ data steps at the size limit

def _closed(lo, hi, device, plus=1):
    """t[i] = i mod 49999 + plus for i in [lo, hi) (int32)."""
    return (torch.arange(lo, hi, dtype=torch.int64, device=device) % TOKEN_MOD + plus).to(torch.int32)


def _filled(shape, device, plus=1):
    t = torch.empty(shape, dtype=torch.int32, device=device)
    flat, step = t.view(-1), 1 << 26
    for c0 in range(0, flat.numel(), step):
        c1 = min(flat.numel(), c0 + step)
        flat[c0:c1] = _closed(c0, c1, device, plus)
    return t


def _ops():
    from sample_packing_document_gb300 import build, ops
    build.build()
    ops.load()
    return ops


@pytest.mark.gpu
@pytest.mark.parametrize("vec", [True, False])
def test_split_at_the_position_limit(vec):
    ops, dev, sp, rank, rows = _ops(), "cuda", 8, 5, 2
    n = (LIMIT // rows) // 32 * 32 - (0 if vec else 8)   # chunk n / 8: a multiple of 4 (16-byte path) or odd
    assert ((n // sp) % 4 == 0) == vec and rows * n <= LIMIT
    src = _filled((rows, n), dev)
    outs = ops.split_sequence_parallel([src, src, src], sp, rank)
    c = n // sp
    for o in outs:
        for r in range(rows):
            for c0 in range(0, c, 1 << 26):
                c1 = min(c, c0 + (1 << 26))
                lo = r * n + rank * c
                assert torch.equal(o[r, c0:c1], _closed(lo + c0, lo + c1, dev)), (r, c0)
    del src, outs
    torch.cuda.empty_cache()


@pytest.mark.gpu
def test_pad_at_the_position_limit():
    ops, dev, sp, rows = _ops(), "cuda", 8, 2
    n = LIMIT // rows - 13
    padded = -(-n // sp) * sp
    assert rows * padded <= LIMIT and padded > n
    src = _filled((rows, n), dev)
    _, lab, pos, _ = ops.pad_for_sequence_parallel(sp, labels=src, position_ids=src)
    for r in range(rows):
        for c0 in range(0, n, 1 << 26):
            c1 = min(n, c0 + (1 << 26))
            want = _closed(r * n + c0, r * n + c1, dev)
            assert torch.equal(lab[r, c0:c1], want) and torch.equal(pos[r, c0:c1], want), (r, c0)
        extra = padded - n
        assert lab[r, n:].tolist() == [-100] * extra
        assert pos[r, n:].tolist() == list(range(extra))
    del src, lab, pos
    torch.cuda.empty_cache()


@pytest.mark.gpu
def test_unpack_data_at_the_position_limit():
    """Packed rows of 2 x seq_len: row 0 holds a 1000-token document, one of
    seq_len + 3 (cut to seq_len) and padding; row 1 one seq_len document and a
    padding segment of seq_len. Output row (r, m) is segment m of row r cut to
    seq_len, then 0 / -100 (the oracle's unpack_data rule)."""
    ops, dev, mb = _ops(), "cuda", 2
    sl = LIMIT // 4
    plen, rows = mb * sl, 2
    cu = [0, 1000, 1000 + sl + 3, plen, plen + sl, 2 * plen]
    rsp = [0, 3, 5]
    ids = _filled((rows * plen,), dev)
    lab = _filled((rows * plen,), dev, plus=2)
    o_ids, o_lab = ops.unpack_data(ids, lab, torch.tensor(cu, dtype=torch.int32, device=dev),
                                   torch.tensor(rsp, dtype=torch.int32, device=dev), rows, mb, sl)
    del ids, lab
    for r in range(rows):
        for m in range(mb):
            s_ = rsp[r] + m
            a, n = (cu[s_], min(cu[s_ + 1] - cu[s_], sl)) if s_ < rsp[r + 1] else (0, 0)
            for c0 in range(0, sl, 1 << 26):
                c1 = min(sl, c0 + (1 << 26))
                k = max(0, min(c1, n) - c0)               # copied positions in [c0, c1)
                want_i = torch.zeros(c1 - c0, dtype=torch.int32, device=dev)
                want_l = torch.full((c1 - c0,), -100, dtype=torch.int32, device=dev)
                if k:
                    want_i[:k] = _closed(a + c0, a + c0 + k, dev)
                    want_l[:k] = _closed(a + c0, a + c0 + k, dev, plus=2)
                assert torch.equal(o_ids[r, m, c0:c1], want_i), (r, m, c0)
                assert torch.equal(o_lab[r, m, c0:c1], want_l), (r, m, c0)
    del o_ids, o_lab
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ attention past 2^31 elements

def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.gpu
def test_attention_past_2_31_elements():
    """q / out / dO / dQ of 2 heads and k / v / dK / dV of 1 head over
    2^24 + 2^16 tokens: more than 2^31 elements per tensor, so every element
    offset needs 64 bits (q's pass 2^31 at token 2^23, k's at token 2^24).
    Documents of 96-160 tokens keep the work small; bf16 gradients (the
    benchmarked form). The segments at the start, across both 2^31-element
    offsets and at the end are compared whole with the fp64 oracle at the
    attention bars, and every output is finite."""
    from oracle import attention as OA
    from sample_packing_document_gb300 import workloads as W
    ops = _ops()
    Hq, Hkv, d = 2, 1, 128
    T = (1 << 24) + (1 << 16)
    rng = np.random.default_rng(2024)
    lens = rng.integers(96, 161, size=T // 96 + 1)
    cu = np.concatenate([[0], np.cumsum(lens)])
    cu = cu[cu < T]
    cu = np.append(cu, T).astype(np.int64)
    assert T * Hq * d > 2 ** 32 and T * Hkv * d > 2 ** 31
    ns = len(cu) - 1
    q, k, v, do = W.qkv(T, Hq, Hkv, d, 77, device="cuda")
    cu_d = torch.tensor(cu.astype(np.int32), device="cuda")
    ws_f = ops.workspace(ops.attn_workspace_size(T, ns, Hq, Hkv, d, False))
    out, lse = ops.varlen_attn_fwd(q, k, v, cu_d, ns, ws=ws_f)
    assert ops.read_status(ws_f) == 0
    del ws_f
    ws_b = ops.workspace(ops.attn_workspace_size(T, ns, Hq, Hkv, d, True))
    dq, dk, dv = ops.varlen_attn_bwd(q, k, v, out, do, lse, cu_d, ns, grad_dtype=torch.bfloat16, ws=ws_b)
    assert ops.read_status(ws_b) == 0
    del ws_b
    for t in (out, dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    assert bool(torch.isfinite(lse).all())
    pick = {0, 1, ns - 2, ns - 1}
    for tok in (1 << 23, 1 << 24):                    # the segments around each 2^31-element offset
        s = int(np.searchsorted(cu, tok, side="right")) - 1
        pick |= {s - 1, s, s + 1}
    for s in sorted(pick):
        a, b = int(cu[s]), int(cu[s + 1])
        sub = [np.asarray([0, b - a], np.int32)]
        qs, ks, vs, ds = _u16(q[a:b]), _u16(k[a:b]), _u16(v[a:b]), _u16(do[a:b])
        o_ref, lse_ref = OA.attn_fwd(qs, ks, vs, sub[0])
        gq, gk, gv, _ = OA.attn_bwd(qs, ks, vs, ds, sub[0])
        o_gpu = out[a:b].float().cpu().numpy().transpose(1, 0, 2)
        assert np.max(np.abs(o_gpu - o_ref)) <= 2e-2, s
        assert np.max(np.abs(lse[:, a:b].cpu().numpy() - lse_ref)) <= 1e-3, s
        for g, ref in ((dq, gq), (dk, gk), (dv, gv)):
            assert np.max(np.abs(g[a:b].float().cpu().numpy() - ref)) <= 5e-2, s
    del q, k, v, do, out, lse, dq, dk, dv
    torch.cuda.empty_cache()
