"""GPU parity of spd_pack_tokens: bit-exact against the oracle.

Cases: the worked examples of the InternEvo page "Data loading and flow";
thousands of random tiny cases (carry-over across rows, padding, length-1
documents, documents longer than a row, both modes); the five workloads at
full size; unaligned outputs (scalar store path); bad document lengths
(status word, no fault).
"""
import json
import os
import random

import numpy as np
import pytest
import torch

from oracle import attention as OA
from oracle import pack as P

pytestmark = pytest.mark.gpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pack_examples.json")))


@pytest.fixture(scope="module")
def ops():
    from sample_packing_document_gb300 import build, ops as _ops
    build.build()
    _ops.load()
    return _ops


def _gpu_pack(ops, toks, lens, mb, sl, packed):
    t = torch.tensor(np.asarray(toks, np.int32), device="cuda")
    l = torch.tensor(np.asarray(lens, np.int32), device="cuda")
    out = ops.pack_tokens(t, l, mb, sl, packed)
    st = ops.read_status(out["ws"])
    ns = int(out["num_segs"].item())
    rows = out["rows"]
    return st, {
        "input_ids": out["input_ids"].cpu().numpy(), "labels": out["labels"].cpu().numpy(),
        "indexes": out["indexes"].cpu().numpy(), "cu_seqlens": out["cu_seqlens"][:ns + 1].cpu().numpy(),
        "row_seg_ptr": out["row_seg_ptr"].cpu().numpy(), "max_seqlen": out["max_seqlen"][:rows].cpu().numpy(),
        "num_segs": ns, "rows": rows}


def _assert_same(g, ref):
    assert g["rows"] == ref["rows"]
    assert g["num_segs"] == ref["num_segs"]
    for key in ("input_ids", "labels", "indexes", "cu_seqlens", "row_seg_ptr", "max_seqlen"):
        np.testing.assert_array_equal(np.asarray(g[key]), np.asarray(ref[key], dtype=np.int32), err_msg=key)


def test_worked_examples(ops):
    for key in ("build_pack", "build_unpack"):
        gd = GOLDEN[key]
        docs = gd["docs"]
        st, g = _gpu_pack(ops, [t for d in docs for t in d], [len(d) for d in docs], gd["micro_bsz"],
                          gd["seq_len"], gd["use_packed_dataset"])
        assert st == 0
        rows = len(gd["input_ids"])
        assert g["input_ids"].reshape(rows, -1).tolist() == gd["input_ids"]
        assert g["labels"].reshape(rows, -1).tolist() == gd["labels"]
        _assert_same(g, P.pack_flat(docs, gd["micro_bsz"], gd["seq_len"], gd["use_packed_dataset"]))
    st, g = _gpu_pack(ops, [t for d in GOLDEN["build_pack"]["docs"] for t in d],
                      [len(d) for d in GOLDEN["build_pack"]["docs"]], 2, 8, True)
    assert g["indexes"].reshape(2, -1).tolist() == GOLDEN["batch_fields"]["indexes"]
    assert g["cu_seqlens"].tolist() == [0, 4, 11, 16, 19, 24, 32]
    assert g["max_seqlen"][0] == GOLDEN["batch_fields"]["max_seqlen_row0"]


@pytest.mark.parametrize("packed", [True, False])
def test_random_tiny_cases(ops, packed):
    rng = random.Random(4242 + packed)
    for _ in range(5000):
        mb, sl = rng.randint(1, 4), rng.randint(1, 16)
        plen = mb * sl
        n = rng.randint(1, 10)
        docs = [[rng.randint(1, 49999) for _ in range(rng.randint(1, 3 * plen))] for _ in range(n)]
        st, g = _gpu_pack(ops, [t for d in docs for t in d], [len(d) for d in docs], mb, sl, packed)
        assert st == 0
        _assert_same(g, P.pack_flat(docs, mb, sl, packed))


@pytest.mark.parametrize("packed", [True, False])
def test_many_docs_multi_pass_scan(ops, packed):
    """More documents than one pass of the scan covers (4096 per pass)."""
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 9, size=20000).astype(np.int32)
    toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
    for mb, sl in ((3, 7), (1, 64), (8, 1)):
        st, g = _gpu_pack(ops, toks, lens, mb, sl, packed)
        assert st == 0
        _assert_same(g, OA.pack(toks, lens, mb, sl, packed))


@pytest.mark.parametrize("name", ["tiny", "c2", "c3", "c3_unpack", "c4", "c5"])
def test_workloads_full_size(ops, name):
    from sample_packing_document_gb300 import workloads as W
    w = W.WORKLOADS[name]
    lens, toks = W.documents(w)
    st, g = _gpu_pack(ops, toks, lens, w.micro_bsz, w.seq_len, w.use_packed_dataset)
    assert st == 0
    _assert_same(g, OA.pack(toks, lens, w.micro_bsz, w.seq_len, w.use_packed_dataset))


def test_unaligned_outputs_take_scalar_path(ops):
    rng = np.random.default_rng(9)
    lens = rng.integers(1, 40, size=300).astype(np.int32)
    toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
    mb, sl = 2, 33
    ref = OA.pack(toks, lens, mb, sl, True)
    n = ref["rows"] * mb * sl
    base = torch.zeros(3 * n + 8, dtype=torch.int32, device="cuda")
    out = ops.alloc_pack_outputs(len(lens), len(toks), mb, sl, True)
    out["input_ids"], out["labels"], out["indexes"] = base[1:1 + n], base[2 + n:2 + 2 * n], base[3 + 2 * n:3 + 3 * n]
    tb = torch.zeros(len(toks) + 1, dtype=torch.int32, device="cuda")
    tb[1:] = torch.tensor(toks, device="cuda")
    t = tb[1:]                                           # unaligned tokens too
    ops.pack_tokens(t, torch.tensor(lens, device="cuda"), mb, sl, True, out=out)
    assert ops.read_status(out["ws"]) == 0
    np.testing.assert_array_equal(out["input_ids"].cpu().numpy(), ref["input_ids"])
    np.testing.assert_array_equal(out["labels"].cpu().numpy(), ref["labels"])
    np.testing.assert_array_equal(out["indexes"].cpu().numpy(), ref["indexes"])


def test_random_two_launch_cases(ops):
    """Random build_pack cases past the fused path's limits (more than 1024
    documents or more than 512 rows): row starts on and inside documents,
    documents longer than a row, padding, both kernel lookup paths."""
    rng = np.random.default_rng(31)
    for _ in range(40):
        nd = int(rng.integers(1025, 2600)) if rng.random() < 0.7 else int(rng.integers(1, 200))
        mb, sl = int(rng.integers(1, 4)), int(rng.integers(1, 40))
        plen = mb * sl
        hi = int(rng.choice([3, 3 * plen + 1, 600]))
        lens = rng.integers(1, max(2, hi), size=nd).astype(np.int32)
        toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
        ref = OA.pack(toks, lens, mb, sl, True)
        if nd <= 1024 and ref["rows"] <= 512:
            continue
        st, g = _gpu_pack(ops, toks, lens, mb, sl, True)
        assert st == 0
        _assert_same(g, ref)


@pytest.mark.parametrize("case", ["long_docs_16_rows", "tiny_docs_window_overflow", "many_rows_few_docs",
                                  "unaligned_many_docs"])
def test_two_launch_build_pack(ops, case):
    """build_pack through the scan and token-stream launches (more than 1024
    documents or 512 rows): documents spanning many 4096-position chunks, chunks
    overlapping more documents than the 1024 starts a CTA stages (the global
    lookup path), many rows, and unaligned tokens / outputs (scalar paths)."""
    rng = np.random.default_rng({"long_docs_16_rows": 21, "tiny_docs_window_overflow": 22,
                                 "many_rows_few_docs": 23, "unaligned_many_docs": 24}[case])
    if case == "long_docs_16_rows":
        from sample_packing_document_gb300 import workloads as W
        w = W.WORKLOADS["c5"]
        lens, toks = W.documents(w)
        lens, toks = np.tile(np.asarray(lens, np.int32), 16), np.tile(np.asarray(toks, np.int32), 16)
        mb, sl = w.micro_bsz, w.seq_len
    elif case == "tiny_docs_window_overflow":
        lens = rng.integers(1, 3, size=30000).astype(np.int32)      # ~2700 documents per 4096 positions
        toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
        mb, sl = 1, 10000
    elif case == "many_rows_few_docs":
        lens = rng.integers(1, 200, size=300).astype(np.int32)
        toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
        mb, sl = 2, 4                                               # > 512 rows of 8
    else:
        lens = rng.integers(1, 700, size=3000).astype(np.int32)
        toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
        mb, sl = 3, 5000
    ref = OA.pack(toks, lens, mb, sl, True)
    if case != "unaligned_many_docs":
        st, g = _gpu_pack(ops, toks, lens, mb, sl, True)
        assert st == 0
        _assert_same(g, ref)
        return
    n = ref["rows"] * mb * sl
    base = torch.zeros(3 * n + 8, dtype=torch.int32, device="cuda")
    out = ops.alloc_pack_outputs(len(lens), len(toks), mb, sl, True)
    out["input_ids"], out["labels"], out["indexes"] = base[1:1 + n], base[2 + n:2 + 2 * n], base[3 + 2 * n:3 + 3 * n]
    tb = torch.zeros(len(toks) + 1, dtype=torch.int32, device="cuda")
    tb[1:] = torch.tensor(toks, device="cuda")
    ops.pack_tokens(tb[1:], torch.tensor(lens, device="cuda"), mb, sl, True, out=out)
    assert ops.read_status(out["ws"]) == 0
    np.testing.assert_array_equal(out["input_ids"].cpu().numpy(), ref["input_ids"])
    np.testing.assert_array_equal(out["labels"].cpu().numpy(), ref["labels"])
    np.testing.assert_array_equal(out["indexes"].cpu().numpy(), ref["indexes"])
    ns = int(out["num_segs"].item())
    np.testing.assert_array_equal(out["cu_seqlens"][:ns + 1].cpu().numpy(), ref["cu_seqlens"])


def test_bad_doc_lengths_set_status(ops):
    toks = torch.arange(1, 11, dtype=torch.int32, device="cuda")
    st, _ = _gpu_pack(ops, toks.cpu().numpy(), [4, 0, 6], 2, 4, True)
    assert st == -7
    st, _ = _gpu_pack(ops, toks.cpu().numpy(), [4, 5, 2], 2, 4, True)   # sums to 11, not 10
    assert st == -7
    st, g = _gpu_pack(ops, toks.cpu().numpy(), [4, 6], 2, 4, True)      # and the next call is clean
    assert st == 0 and g["num_segs"] == 4 and g["cu_seqlens"].tolist() == [0, 4, 8, 10, 16]


@pytest.mark.parametrize("nd_lo,nd_hi", [(1, 1024), (1025, 3000)])
def test_random_unpack_cases(ops, nd_lo, nd_hi):
    """build_unpack (use_packed_dataset=False) on both sides of the one-launch
    limit (1024 documents): documents shorter and longer than SEQ_LEN, a
    partial last row, row lengths that are not a multiple of four."""
    rng = np.random.default_rng(77 + nd_lo)
    for _ in range(30):
        nd = int(rng.integers(nd_lo, nd_hi + 1))
        mb, sl = int(rng.integers(1, 6)), int(rng.integers(1, 40))
        lens = rng.integers(1, 3 * sl + 1, size=nd).astype(np.int32)
        toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
        st, g = _gpu_pack(ops, toks, lens, mb, sl, False)
        assert st == 0
        _assert_same(g, OA.pack(toks, lens, mb, sl, False))


@pytest.mark.parametrize("nd", [3, 2000])
def test_bad_doc_lengths_set_status_unpack(ops, nd):
    """build_unpack with a zero-length document or lengths that do not sum to
    num_tokens reports SPD_ERR_BAD_DOCS (one-launch and two-launch paths)."""
    rng = np.random.default_rng(nd)
    lens = rng.integers(1, 9, size=nd).astype(np.int32)
    toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
    bad = lens.copy()
    bad[nd // 2] = 0
    st, _ = _gpu_pack(ops, toks[:int(bad.sum())], bad, 2, 8, False)
    assert st == -7
    st, _ = _gpu_pack(ops, toks[:-1], lens, 2, 8, False)
    assert st == -7
    st, g = _gpu_pack(ops, toks, lens, 2, 8, False)
    assert st == 0
    _assert_same(g, OA.pack(toks, lens, 2, 8, False))


@pytest.mark.parametrize("n_docs,len_hi,mb,sl", [
    (40000, 8, 1, 65536),        # 10 prefix CTAs chained by the look-back
    (300000, 8, 4, 8192),        # 74 prefix CTAs, many rows, documents split across rows
    (9000, 3000, 2, 4096),       # 3 prefix CTAs, long documents over many rows, a padding tail
])
def test_many_documents_multi_cta_prefix(ops, n_docs, len_hi, mb, sl):
    """build_pack with more than 4096 documents: the document-start prefix and
    the aligned-start counts are chained across CTAs (decoupled look-back); the
    segment fields come from the stream kernel. Bit-exact against the C oracle
    twin (itself pinned to the literal oracle)."""
    rng = np.random.default_rng(n_docs)
    lens = rng.integers(1, len_hi + 1, size=n_docs).astype(np.int32)
    toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
    st, g = _gpu_pack(ops, toks, lens, mb, sl, True)
    assert st == 0
    _assert_same(g, OA.pack(toks, lens, mb, sl, True))


def test_many_documents_bad_length_sets_status(ops):
    """A zero-length document in a late prefix CTA and a wrong total are both
    reported, and the next call on a fresh workspace is clean."""
    rng = np.random.default_rng(3)
    lens = rng.integers(1, 9, size=20000).astype(np.int32)
    toks = rng.integers(1, 50000, size=int(lens.sum())).astype(np.int32)
    bad = lens.copy()
    bad[9000] = 0                                              # in the third of five prefix CTAs
    st, _ = _gpu_pack(ops, toks[:int(bad.sum())], bad, 2, 4096, True)
    assert st == -7
    st, _ = _gpu_pack(ops, toks[:-1], lens, 2, 4096, True)          # lengths sum past num_tokens
    assert st == -7
    st, g = _gpu_pack(ops, toks, lens, 2, 4096, True)
    assert st == 0
    _assert_same(g, OA.pack(toks, lens, 2, 4096, True))
