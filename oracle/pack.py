"""Literal packing oracle (pure Python lists). TEST INFRASTRUCTURE ONLY.

Follows the InternEvo page "Data loading and flow" (internevo.readthedocs.io,
data_flow.html):

* section "Dataloader loading data": build_pack (use_packed_dataset=True) and
  build_unpack (use_packed_dataset=False), pad id 0, label rule "tokens 2..n of
  the input, then -100";
* section "Fetching data from the Dataloader": the batch fields input_ids,
  cu_seqlens (segment boundaries, padding tail as its own segment), indexes
  (position inside the current segment, restarting at 0) and label;
* section "Processing data": max_seqlen (largest segment of the row),
  unpack_data, split_data_sequence_parallel.

Readings where the page is silent (each one is listed in the design notes):

* a document longer than a packed row keeps being cut at every row end; each
  piece is its own segment and its indexes restart at 0;
* the padding tail of the last row is one segment whose indexes count 0, 1, ...
  (the printed example shows this);
* in build_unpack, labels are taken from the truncated document, so the last
  kept token of a truncated document gets -100 (the printed example shows
  this); cu_seqlens / indexes follow the same convention as build_pack:
  one segment per (truncated) document, then one padding segment;
* zero-length documents are rejected; token id 0 inside a document is copied
  as is; an empty document list gives zero rows.

Everything here is written as plain loops over Python lists so it can be read
against the page.
"""

PAD_ID = 0
IGNORE_INDEX = -100


def _check(docs, micro_bsz, seq_len):
    if micro_bsz <= 0 or seq_len <= 0:
        raise ValueError("micro_bsz and SEQ_LEN must be positive")
    for doc in docs:
        if len(doc) == 0:
            raise ValueError("zero-length documents are not accepted")


def build_pack(docs, micro_bsz, seq_len):
    """use_packed_dataset=True.

    All documents are laid end to end; the stream is cut every
    packed_length = micro_bsz * SEQ_LEN tokens, the part of a document that
    does not fit continues at the start of the next row, and the last row is
    filled up with 0. Each document's labels are its tokens from the second
    on followed by -100, computed before the cut, so a row's last label can be
    the first token of the next row. Padding positions get -100.

    Returns (rows_ids, rows_labels, rows_owner) where rows_owner[r][c] is the
    index of the document that position c of row r came from, or -1 for
    padding. The owner lists are what the segment fields are derived from.
    """
    _check(docs, micro_bsz, seq_len)
    plen = micro_bsz * seq_len
    stream, lstream, owner = [], [], []
    for d, doc in enumerate(docs):
        stream.extend(doc)
        lstream.extend(list(doc[1:]) + [IGNORE_INDEX])
        owner.extend([d] * len(doc))
    rows_ids, rows_labels, rows_owner = [], [], []
    start = 0
    while start < len(stream):
        ids = stream[start:start + plen]
        labs = lstream[start:start + plen]
        own = owner[start:start + plen]
        npad = plen - len(ids)
        rows_ids.append(ids + [PAD_ID] * npad)
        rows_labels.append(labs + [IGNORE_INDEX] * npad)
        rows_owner.append(own + [-1] * npad)
        start += plen
    return rows_ids, rows_labels, rows_owner


def build_unpack(docs, micro_bsz, seq_len):
    """use_packed_dataset=False.

    Rule 1: at most micro_bsz documents go into one row; the rest of the row
    is filled with 0 even if the next document would fit. Rule 2: a document
    longer than SEQ_LEN is cut to SEQ_LEN and the excess is thrown away.
    Rule 3 (cut a row that overflows micro_bsz * SEQ_LEN) can never apply
    once rules 1 and 2 hold. Labels come from the truncated document.
    """
    _check(docs, micro_bsz, seq_len)
    plen = micro_bsz * seq_len
    rows_ids, rows_labels, rows_owner = [], [], []
    for first in range(0, len(docs), micro_bsz):
        ids, labs, own = [], [], []
        for d in range(first, min(first + micro_bsz, len(docs))):
            kept = list(docs[d][:seq_len])
            ids.extend(kept)
            labs.extend(kept[1:] + [IGNORE_INDEX])
            own.extend([d] * len(kept))
        assert len(ids) <= plen  # rule 3 is implied by rules 1 and 2
        npad = plen - len(ids)
        rows_ids.append(ids + [PAD_ID] * npad)
        rows_labels.append(labs + [IGNORE_INDEX] * npad)
        rows_owner.append(own + [-1] * npad)
    return rows_ids, rows_labels, rows_owner


def row_segments(owner_row):
    """Segments of one row: maximal runs of positions with the same owner
    (one document's tokens, or the padding tail). Returns cu_seqlens for the
    row (boundaries from 0 to packed_length)."""
    cu = [0]
    for c in range(1, len(owner_row)):
        if owner_row[c] != owner_row[c - 1]:
            cu.append(c)
    cu.append(len(owner_row))
    return cu


def row_indexes(cu_row):
    """Position of each token inside its segment, counting from 0."""
    idx = []
    for s in range(len(cu_row) - 1):
        idx.extend(range(cu_row[s + 1] - cu_row[s]))
    return idx


def row_max_seqlen(cu_row):
    """Largest segment length of the row (the padding segment counts)."""
    return max(cu_row[s + 1] - cu_row[s] for s in range(len(cu_row) - 1))


def pack_batch(docs, micro_bsz, seq_len, use_packed_dataset=True):
    """All batch fields, per row, as the page prints them.

    Returns a dict with lists of rows: input_ids, labels, cu_seqlens (ragged),
    indexes, max_seqlen.
    """
    build = build_pack if use_packed_dataset else build_unpack
    ids, labels, owner = build(docs, micro_bsz, seq_len)
    cu = [row_segments(o) for o in owner]
    return {
        "input_ids": ids,
        "labels": labels,
        "cu_seqlens": cu,
        "indexes": [row_indexes(c) for c in cu],
        "max_seqlen": [row_max_seqlen(c) for c in cu],
    }


def pack_flat(docs, micro_bsz, seq_len, use_packed_dataset=True):
    """The same fields in the flat layout the C-ABI writes.

    input_ids / labels / indexes: rows concatenated. cu_seqlens: one global
    list, row r's boundaries shifted by r * packed_length, shared row ends
    written once. row_seg_ptr[r] is where row r's segments start in that list.
    """
    b = pack_batch(docs, micro_bsz, seq_len, use_packed_dataset)
    plen = micro_bsz * seq_len
    flat = {"input_ids": [], "labels": [], "indexes": [], "cu_seqlens": [0],
            "row_seg_ptr": [0], "max_seqlen": list(b["max_seqlen"])}
    for r in range(len(b["input_ids"])):
        flat["input_ids"].extend(b["input_ids"][r])
        flat["labels"].extend(b["labels"][r])
        flat["indexes"].extend(b["indexes"][r])
        flat["cu_seqlens"].extend(r * plen + c for c in b["cu_seqlens"][r][1:])
        flat["row_seg_ptr"].append(len(flat["cu_seqlens"]) - 1)
    flat["num_segs"] = len(flat["cu_seqlens"]) - 1
    flat["rows"] = len(b["input_ids"])
    return flat


def unpack_data(packed_ids, packed_labels, cu_row, micro_bsz, seq_len):
    """section "Processing data", unpack_data: turn one packed row back into
    micro_bsz rows of SEQ_LEN, one document per row, padded with 0 / -100;
    cu_seqlens and indexes are dropped. Only document segments are unpacked:
    a trailing padding segment holds nothing but 0 / -100."""
    out_ids = [[PAD_ID] * seq_len for _ in range(micro_bsz)]
    out_lab = [[IGNORE_INDEX] * seq_len for _ in range(micro_bsz)]
    for s in range(min(micro_bsz, len(cu_row) - 1)):
        a, b = cu_row[s], cu_row[s + 1]
        n = min(b - a, seq_len)
        out_ids[s][:n] = packed_ids[a:a + n]
        out_lab[s][:n] = packed_labels[a:a + n]
    return out_ids, out_lab


# Pad values of pad_for_sequence_parallel (XTuner page, "Sequence parallel API",
# data pad and split): the page names the tensors (input_ids, labels,
# position_ids, attention_mask) but not the values; read as the pad id 0 and
# the ignore index -100 of the packing page, position ids that count 0, 1, 2, ...
# over the added positions (the packing page's padding tail is a segment of its
# own whose indexes count from 0), and attention mask 0 (padding attends to
# nothing and is attended by nothing).
SP_PAD = {"input_ids": ("value", PAD_ID), "labels": ("value", IGNORE_INDEX),
          "position_ids": ("count", 0), "attention_mask": ("value", 0)}


def sp_padded_length(n, sp_size):
    """Smallest multiple of sp_size that is >= n."""
    if sp_size < 1:
        raise ValueError("sp_size must be >= 1")
    return -(-n // sp_size) * sp_size


def pad_for_sequence_parallel(seq, sp_size, kind):
    """Pad one row of `kind` (a key of SP_PAD) so that its length divides by
    sp_size; the original positions are kept as they are."""
    mode, v = SP_PAD[kind]
    n = len(seq)
    extra = sp_padded_length(n, sp_size) - n
    fill = [v] * extra if mode == "value" else list(range(extra))
    return list(seq) + fill


def split_sequence_parallel(seq, sp_size, rank):
    """section "Processing data", split_data_sequence_parallel: contiguous
    equal chunks of the sequence dimension, one per rank."""
    n = len(seq)
    if n % sp_size:
        raise ValueError("sequence length must divide by sp_size")
    c = n // sp_size
    return seq[rank * c:(rank + 1) * c]
