"""spd_unpack_data and spd_split_sequence_parallel on the GPU against the
oracle (bit-exact): the pages' worked examples, then seeded random batches
covering truncated documents, rows with fewer documents than micro_bsz,
sequence lengths that are not multiples of four and every rank."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import pack as P

pytestmark = pytest.mark.gpu

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pack_examples.json")))


def _ops():
    from sample_packing_document_gb300 import build, ops
    build.build()
    return ops


def _dev(x):
    return torch.tensor(np.asarray(x, dtype=np.int32).reshape(-1), device="cuda")


def _unpack_gpu(ops, docs, micro_bsz, seq_len):
    """Pack the documents with the oracle (use_packed_dataset=False) and unpack
    the rows on the GPU."""
    f = P.pack_flat(docs, micro_bsz, seq_len, False)
    ids, labs = ops.unpack_data(_dev(f["input_ids"]), _dev(f["labels"]), _dev(f["cu_seqlens"]),
                                _dev(f["row_seg_ptr"]), f["rows"], micro_bsz, seq_len)
    torch.cuda.synchronize()
    return f, ids.cpu().numpy(), labs.cpu().numpy()


def _unpack_oracle(docs, micro_bsz, seq_len):
    b = P.pack_batch(docs, micro_bsz, seq_len, False)
    out_i, out_l = [], []
    for r in range(len(b["input_ids"])):
        i, l = P.unpack_data(b["input_ids"][r], b["labels"][r], b["cu_seqlens"][r], micro_bsz, seq_len)
        out_i.append(i)
        out_l.append(l)
    return np.array(out_i, dtype=np.int32), np.array(out_l, dtype=np.int32)


def test_unpack_worked_example():
    ops = _ops()
    g = GOLDEN["unpack_data"]
    f, ids, labs = _unpack_gpu(ops, g["docs"], g["micro_bsz"], g["seq_len"])
    assert f["input_ids"] == g["packed_input_ids"] and f["labels"] == g["packed_labels"]
    assert ids[0].tolist() == g["unpacked_input_ids"]
    assert labs[0].tolist() == g["unpacked_labels"]


def test_split_worked_examples():
    ops = _ops()
    g, s = GOLDEN["build_pack"], GOLDEN["split_sequence_parallel_packed"]
    b = P.pack_batch(g["docs"], g["micro_bsz"], g["seq_len"], True)
    row = [_dev(b["input_ids"][0]), _dev(b["indexes"][0]), _dev(b["labels"][0])]
    for r in range(s["sp_size"]):
        got = [x.cpu().tolist() for x in ops.split_sequence_parallel(row, s["sp_size"], r)]
        want = s["rank%d" % r]
        assert got == [want["input_ids"], want["indexes"], want["labels"]]
    u, s = GOLDEN["unpack_data"], GOLDEN["split_sequence_parallel_unpacked"]
    t = [torch.tensor(u["unpacked_input_ids"], dtype=torch.int32, device="cuda"),
         torch.tensor(u["unpacked_labels"], dtype=torch.int32, device="cuda")]
    for r in range(s["sp_size"]):
        got = [x.cpu().tolist() for x in ops.split_sequence_parallel(t, s["sp_size"], r)]
        want = s["rank%d" % r]
        assert got == [want["input_ids"], want["labels"]]


@pytest.mark.parametrize("micro_bsz,seq_len,seed", [(1, 5, 0), (2, 8, 1), (3, 13, 2), (4, 64, 3), (2, 256, 4)])
def test_unpack_random_matches_oracle(micro_bsz, seq_len, seed):
    ops = _ops()
    rng = np.random.default_rng(seed)
    n_docs = int(rng.integers(1, 12))
    docs = [rng.integers(1, 50000, size=int(rng.integers(1, 2 * seq_len + 3))).tolist() for _ in range(n_docs)]
    _, ids, labs = _unpack_gpu(ops, docs, micro_bsz, seq_len)
    want_i, want_l = _unpack_oracle(docs, micro_bsz, seq_len)
    assert np.array_equal(ids, want_i) and np.array_equal(labs, want_l)


@pytest.mark.parametrize("rows,length,sp", [(1, 16, 2), (3, 24, 8), (5, 1000, 4), (2, 4096, 8), (7, 30, 1)])
def test_split_random_matches_oracle(rows, length, sp):
    ops = _ops()
    rng = np.random.default_rng(rows * 100 + sp)
    src = [rng.integers(-100, 50000, size=(rows, length)).astype(np.int32) for _ in range(3)]
    dev = [torch.tensor(x, device="cuda") for x in src]
    for r in range(sp):
        got = ops.split_sequence_parallel(dev, sp, r)
        for g, x in zip(got, src):
            want = np.array([P.split_sequence_parallel(list(row), sp, r) for row in x], dtype=np.int32)
            assert np.array_equal(g.cpu().numpy(), want)


@pytest.mark.parametrize("rows,length,sp", [(1, 13, 8), (3, 24, 8), (5, 1001, 4), (2, 4093, 8), (7, 30, 1),
                                             (1, 1, 5), (4, 0, 3), (2, 15, 16),
                                             (9, 4099, 8), (6, 70001, 16), (5, 256, 8)])   # every source shift of a row
def test_pad_for_sequence_parallel_matches_oracle(rows, length, sp):
    """Every tensor kind, ragged and already-divisible lengths, the empty row,
    sp_size larger than the row; then the page's purpose: the padded rows split
    evenly (split of the pad = split of the oracle's pad on every rank)."""
    ops = _ops()
    rng = np.random.default_rng(rows * 1000 + length + sp)
    src = {k: rng.integers(-100, 50000, size=(rows, length)).astype(np.int32)
           for k in ("input_ids", "labels", "position_ids", "attention_mask")}
    got = ops.pad_for_sequence_parallel(sp, **{k: torch.tensor(v, device="cuda") for k, v in src.items()})
    wants = []
    for g, (k, x) in zip(got, src.items()):
        want = np.array([P.pad_for_sequence_parallel(list(row), sp, k) for row in x], dtype=np.int32).reshape(rows, -(-length // sp) * sp)
        assert np.array_equal(g.cpu().numpy(), want), k
        wants.append(want)
    if length > 0:
        for r in range(sp):
            parts = ops.split_sequence_parallel(list(got[:3]), sp, r)
            for part, want in zip(parts, wants[:3]):
                assert np.array_equal(part.cpu().numpy(),
                                      np.array([P.split_sequence_parallel(list(row), sp, r) for row in want]))


def test_pad_full_size_row():
    """The timed case: one 1048573-token row padded to sp_size 8 (1048576), every
    tensor kind, compared in full with the oracle."""
    ops = _ops()
    T, sp = (1 << 20) - 3, 8
    rng = np.random.default_rng(11)
    src = rng.integers(-100, 50000, size=(1, T)).astype(np.int32)
    x = torch.tensor(src, device="cuda")
    got = ops.pad_for_sequence_parallel(sp, input_ids=x, labels=x, position_ids=x, attention_mask=x)
    for g, kind in zip(got, ("input_ids", "labels", "position_ids", "attention_mask")):
        want = np.array(P.pad_for_sequence_parallel(src[0].tolist(), sp, kind), dtype=np.int32)
        assert g.shape == (1, 1 << 20)
        assert np.array_equal(g.cpu().numpy()[0], want), kind


def test_pad_1d_and_unaligned_output():
    """A [len] tensor, and an output view that is not 16-byte aligned (the
    scalar store path); a source view that is not 16-byte aligned (the scalar
    load path) over rows long enough for the vector path otherwise."""
    ops = _ops()
    x = torch.arange(1, 11, dtype=torch.int32, device="cuda")
    (y,) = [t for t in ops.pad_for_sequence_parallel(4, labels=x) if t is not None]
    assert y.cpu().tolist() == list(range(1, 11)) + [-100, -100]
    lib = ops.load()
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    rc = lib.spd_pad_for_sequence_parallel(ops._ptr(x), ops._ptr(buf[1:]), 1, 10, 4, 0, 1, ops._stream(None))
    assert rc == 0
    torch.cuda.synchronize()
    assert buf[1:13].cpu().tolist() == list(range(1, 11)) + [0, 1] and int(buf[0]) == 0 and int(buf[13]) == 0
    rows, n, sp = 3, 1001, 8
    base = torch.arange(rows * n + 1, dtype=torch.int32, device="cuda")
    src = base[1:].view(rows, n)                           # 4 bytes past an aligned start
    (z,) = [t for t in ops.pad_for_sequence_parallel(sp, labels=src) if t is not None]
    want = np.array([P.pad_for_sequence_parallel(row.tolist(), sp, "labels") for row in src.cpu().numpy()])
    assert np.array_equal(z.cpu().numpy(), want)


def test_split_rejects_a_length_that_does_not_divide():
    ops = _ops()
    x = torch.zeros((2, 10), dtype=torch.int32, device="cuda")
    lib = ops.load()
    import ctypes
    P_ = ctypes.c_void_p
    assert lib.spd_split_sequence_parallel(P_(x.data_ptr()), None, None, 2, 10, 4, 0, P_(x.data_ptr()), None, None,
                                           None) == -1
