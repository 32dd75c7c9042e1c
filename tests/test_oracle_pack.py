"""Pins for the packing oracle (CPU only).

The literal Python oracle is pinned to the worked examples printed on the
InternEvo page "Data loading and flow" (tests/golden/pack_examples.json) and
to invariants that any correct packing satisfies; the C restatement is pinned
to the Python one on thousands of random tiny cases.
"""
import json
import os
import random

import numpy as np
import pytest

from oracle import pack as P
from oracle import attention as OA

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pack_examples.json")))


def test_build_pack_worked_example():
    g = GOLDEN["build_pack"]
    ids, labels, _ = P.build_pack(g["docs"], g["micro_bsz"], g["seq_len"])
    assert ids == g["input_ids"]
    assert labels == g["labels"]


def test_batch_fields_worked_example():
    g, f = GOLDEN["build_pack"], GOLDEN["batch_fields"]
    b = P.pack_batch(g["docs"], f["micro_bsz"], f["seq_len"], True)
    assert len(b["input_ids"]) == f["micro_num"]
    assert b["cu_seqlens"] == f["cu_seqlens"]
    assert b["indexes"] == f["indexes"]
    assert b["max_seqlen"][0] == f["max_seqlen_row0"]


def test_build_unpack_worked_example():
    g = GOLDEN["build_unpack"]
    ids, labels, _ = P.build_unpack(g["docs"], g["micro_bsz"], g["seq_len"])
    assert ids == g["input_ids"]
    assert labels == g["labels"]


def test_unpack_data_worked_example():
    g = GOLDEN["unpack_data"]
    b = P.pack_batch(g["docs"], g["micro_bsz"], g["seq_len"], False)
    assert b["input_ids"][0] == g["packed_input_ids"]
    assert b["labels"][0] == g["packed_labels"]
    ids, labs = P.unpack_data(b["input_ids"][0], b["labels"][0], b["cu_seqlens"][0],
                              g["micro_bsz"], g["seq_len"])
    assert ids == g["unpacked_input_ids"]
    assert labs == g["unpacked_labels"]


def test_split_sequence_parallel_worked_example():
    g, s = GOLDEN["build_pack"], GOLDEN["split_sequence_parallel_packed"]
    b = P.pack_batch(g["docs"], g["micro_bsz"], g["seq_len"], True)
    for r in range(s["sp_size"]):
        want = s["rank%d" % r]
        assert P.split_sequence_parallel(b["input_ids"][0], s["sp_size"], r) == want["input_ids"]
        assert P.split_sequence_parallel(b["indexes"][0], s["sp_size"], r) == want["indexes"]
        assert P.split_sequence_parallel(b["labels"][0], s["sp_size"], r) == want["labels"]


def test_split_after_unpack_worked_example():
    """The page's second split example: tp size 2 over the unpacked batch."""
    g, s = GOLDEN["unpack_data"], GOLDEN["split_sequence_parallel_unpacked"]
    for r in range(s["sp_size"]):
        want = s["rank%d" % r]
        assert [P.split_sequence_parallel(row, s["sp_size"], r) for row in g["unpacked_input_ids"]] == want["input_ids"]
        assert [P.split_sequence_parallel(row, s["sp_size"], r) for row in g["unpacked_labels"]] == want["labels"]


def test_pad_for_sequence_parallel_pins():
    """No worked example on the page: pinned by what it states (the padded
    length divides by the sequence-parallel size so the row splits evenly) and
    by the packing page's own rules for the values read for the pad."""
    import numpy as np
    from oracle import loss as L
    rng = np.random.default_rng(3)
    for _ in range(40):
        n, sp = int(rng.integers(1, 60)), int(rng.integers(1, 9))
        seq = rng.integers(-100, 50000, size=n).tolist()
        for kind in ("input_ids", "labels", "position_ids", "attention_mask"):
            out = P.pad_for_sequence_parallel(seq, sp, kind)
            assert len(out) % sp == 0 and len(out) - len(seq) < sp and out[:n] == seq
            if n % sp == 0:
                assert out == seq
            # the page's purpose: the padded row splits into equal chunks that rebuild it
            chunks = [P.split_sequence_parallel(out, sp, r) for r in range(sp)]
            assert all(len(c) == len(out) // sp for c in chunks) and sum(chunks, []) == out
    # labels: the added tokens are ignored by the masked loss (same loss, same count)
    logits_rng = np.random.default_rng(4)
    labels = logits_rng.integers(0, 11, size=13).tolist()
    labels[5] = P.IGNORE_INDEX
    padded = P.pad_for_sequence_parallel(labels, 8, "labels")
    lg = logits_rng.normal(size=(len(padded), 11))
    a = L.masked_loss(lg[:13], np.array(labels))
    b = L.masked_loss(lg, np.array(padded))
    assert a[0] == b[0] and a[1] == b[1]
    # input ids: the pad id of the packing rules
    assert P.pad_for_sequence_parallel([7, 8, 9], 4, "input_ids") == [7, 8, 9, P.PAD_ID]
    # position ids: the added positions are indexed like a padding segment of
    # their own (row_indexes of the row with one more boundary at the old end)
    g = GOLDEN["build_pack"]
    b = P.pack_batch(g["docs"], g["micro_bsz"], g["seq_len"], True)
    idx, cu = b["indexes"][1], b["cu_seqlens"][1]
    for sp in (3, 5, 7):
        padded = P.pad_for_sequence_parallel(idx, sp, "position_ids")
        assert padded == P.row_indexes(cu + [len(padded)])[:len(padded)]


def test_flat_layout_worked_example():
    g = GOLDEN["build_pack"]
    f = P.pack_flat(g["docs"], g["micro_bsz"], g["seq_len"], True)
    assert f["cu_seqlens"] == [0, 4, 11, 16, 19, 24, 32]
    assert f["row_seg_ptr"] == [0, 3, 6]
    assert f["num_segs"] == 6 and f["rows"] == 2


def test_rejects_empty_docs_and_bad_sizes():
    with pytest.raises(ValueError):
        P.build_pack([[1, 2], []], 2, 4)
    with pytest.raises(ValueError):
        P.build_unpack([[1]], 0, 4)
    b = P.pack_flat([], 2, 4, True)
    assert b["rows"] == 0 and b["num_segs"] == 0 and b["cu_seqlens"] == [0]


def _random_docs(rng, max_len, n_max):
    n = rng.randint(0, n_max)
    return [[rng.randint(1, 49999) for _ in range(rng.randint(1, max_len))] for _ in range(n)]


@pytest.mark.parametrize("packed", [True, False])
def test_invariants_random(packed):
    rng = random.Random(1234 + packed)
    for _ in range(1500):
        mb, sl = rng.randint(1, 4), rng.randint(1, 16)
        plen = mb * sl
        docs = _random_docs(rng, 3 * plen, 9)
        b = P.pack_batch(docs, mb, sl, packed)
        for r in range(len(b["input_ids"])):
            cu = b["cu_seqlens"][r]
            assert cu[0] == 0 and cu[-1] == plen                      # lengths sum to plen
            assert all(cu[s + 1] > cu[s] for s in range(len(cu) - 1))
            for p in range(plen):                                      # indexes definition
                s = max(i for i in range(len(cu) - 1) if cu[i] <= p)
                assert b["indexes"][r][p] == p - cu[s]
            assert b["max_seqlen"][r] == max(np.diff(cu))
        flat_ids = [x for row in b["input_ids"] for x in row]
        flat_lab = [x for row in b["labels"] for x in row]
        if packed:
            stream = [t for d in docs for t in d]
            n = len(stream)
            assert flat_ids[:n] == stream                              # non-pad prefix
            assert all(x == 0 for x in flat_ids[n:])
            npad = len(flat_ids) - n
            assert flat_lab.count(-100) == len(docs) + npad            # one -100 per doc
            ends = set(np.cumsum([len(d) for d in docs]).tolist())
            for p in range(n - 1):                                     # label = next token
                if p + 1 not in ends:
                    assert flat_lab[p] == flat_ids[p + 1]
            assert len(b["input_ids"]) == -(-n // plen)
        else:
            assert len(b["input_ids"]) == -(-len(docs) // mb)
            for r in range(len(b["input_ids"])):
                kept = [d[:sl] for d in docs[r * mb:(r + 1) * mb]]
                row = [t for d in kept for t in d]
                assert b["input_ids"][r][:len(row)] == row
                assert b["labels"][r].count(-100) == len(kept) + plen - len(row)


def _flat_equal(f, c):
    assert c["rows"] == f["rows"]
    assert c["num_segs"] == f["num_segs"]
    for key in ("input_ids", "labels", "indexes", "cu_seqlens", "row_seg_ptr", "max_seqlen"):
        assert list(c[key]) == list(f[key]), key


def test_c_twin_worked_examples():
    for key in ("build_pack", "build_unpack"):
        g = GOLDEN[key]
        docs = g["docs"]
        c = OA.pack([t for d in docs for t in d], [len(d) for d in docs], g["micro_bsz"],
                    g["seq_len"], g["use_packed_dataset"])
        rows = len(g["input_ids"])
        assert c["input_ids"].reshape(rows, -1).tolist() == g["input_ids"]
        assert c["labels"].reshape(rows, -1).tolist() == g["labels"]
    c = OA.pack([t for d in GOLDEN["build_pack"]["docs"] for t in d],
                [len(d) for d in GOLDEN["build_pack"]["docs"]], 2, 8, True)
    assert c["indexes"].reshape(2, -1).tolist() == GOLDEN["batch_fields"]["indexes"]
    assert c["cu_seqlens"].tolist() == [0, 4, 11, 16, 19, 24, 32]


@pytest.mark.parametrize("packed", [True, False])
def test_c_twin_matches_literal_random(packed):
    rng = random.Random(99 + packed)
    for _ in range(5000):
        mb, sl = rng.randint(1, 4), rng.randint(1, 16)
        docs = _random_docs(rng, 3 * mb * sl, 10)
        f = P.pack_flat(docs, mb, sl, packed)
        c = OA.pack([t for d in docs for t in d], [len(d) for d in docs], mb, sl, packed)
        _flat_equal(f, c)
