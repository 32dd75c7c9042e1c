"""The C-ABI library builds, loads and exports every entry point include/spd.h
declares; host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sample_packing_document_gb300 import build, ops
    build.build()
    return ops.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "spd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spd_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    from sample_packing_document_gb300 import ops
    names = _declared()
    assert "spd_pack_tokens" in names and "spd_varlen_attn_fwd" in names and "spd_varlen_attn_bwd" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ops.SIGNATURES)


def _prototypes():
    """name -> (return type, [parameter types]) of every declaration in spd.h."""
    text = open(os.path.join(ROOT, "include", "spd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    out = {}
    for ret, name, params in re.findall(r"([A-Za-z_][\w\s\*]*?)\s*\b(spd_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", text):
        ps = [] if params.strip() in ("", "void") else [p.strip() for p in params.split(",")]
        types = []
        for p_ in ps:
            p_ = re.sub(r"\bconst\b", "", p_)
            if "*" in p_:
                types.append("*")
            else:
                types.append(p_.split()[0])            # the type; the name follows it
        out[name] = (" ".join(ret.replace("const", "").split()), types)
    return out


def test_binding_signatures_match_the_header():
    """The ctypes argument and return types of every entry point follow its C
    prototype: pointers (and spd_stream_t) as pointers, int64_t / int32_t /
    int / float / size_t as the same widths."""
    from sample_packing_document_gb300 import ops
    width = {"int64_t": ctypes.c_int64, "int32_t": ctypes.c_int32, "int": ctypes.c_int, "float": ctypes.c_float,
             "size_t": ctypes.c_size_t}
    protos = _prototypes()
    assert set(protos) == set(ops.SIGNATURES)
    for name, (ret, params) in protos.items():
        res, args = ops.SIGNATURES[name]
        assert len(args) == len(params), name
        for i, (c_type, py_type) in enumerate(zip(params, args)):
            if c_type in ("*", "spd_stream_t"):
                assert py_type is ctypes.c_void_p or issubclass(py_type, ctypes._Pointer), (name, i)
            else:
                assert ctypes.sizeof(py_type) == ctypes.sizeof(width[c_type]) and \
                    (py_type is ctypes.c_float) == (c_type == "float"), (name, i, c_type, py_type)
        if ret.endswith("*"):
            assert res is ctypes.c_char_p, name
        else:
            assert ctypes.sizeof(res) == ctypes.sizeof(width[ret]), name


def test_read_schedule_host_checks(lib):
    """spd_attn_read_schedule refuses null pointers before touching a GPU."""
    n = ctypes.c_int32(0)
    assert lib.spd_attn_read_schedule(None, None, ctypes.byref(n), None, 0) == -1
    assert lib.spd_attn_read_schedule(ctypes.c_void_p(256), None, None, None, 0) == -1
    assert lib.spd_attn_read_schedule(ctypes.c_void_p(256), None, ctypes.byref(n), None, 4) == -1
    assert lib.spd_attn_read_schedule(ctypes.c_void_p(256), None, ctypes.byref(n), None, -1) == -1


def test_status_strings_and_version(lib):
    from sample_packing_document_gb300 import ops
    assert lib.spd_version() >= 100
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert ops.status_string(code) != "unknown status"


def test_pack_num_segs_matches_the_oracle(lib):
    """The host segment count equals the number of segments the oracle's
    packing rules produce (which the GPU pack is pinned to bit for bit), in
    both modes, with documents split across rows, exact row fits and
    truncation."""
    import numpy as np
    from oracle import pack as P
    from sample_packing_document_gb300 import ops
    rng = np.random.default_rng(5)
    cases = [([3, 4, 5, 4], 2, 4), ([8, 8], 2, 4), ([1], 1, 1), ([16], 2, 8), ([17, 1, 30, 2], 2, 8)]
    for _ in range(60):
        n = int(rng.integers(1, 30))
        cases.append((rng.integers(1, 40, size=n).tolist(), int(rng.integers(1, 4)), int(rng.integers(1, 24))))
    for lens, mb, sl in cases:
        docs = [[1] * L for L in lens]
        for packed in (True, False):
            want = P.pack_flat(docs, mb, sl, packed)["num_segs"]
            assert ops.pack_num_segs(lens, mb, sl, packed) == want, (lens, mb, sl, packed)
    assert ops.pack_num_segs([], 2, 8, True) == 0
    with pytest.raises(ops.SpdError):
        ops.pack_num_segs([3, 0, 2], 2, 8, True)


def test_position_limit_leaves_a_margin(lib):
    """Packing and data steps accept at most 2^31 - 65537 positions: the
    kernels' 32-bit position arithmetic steps up to one chunk past the end."""
    import ctypes as C
    from sample_packing_document_gb300 import ops
    L = ops.load()
    rows, ms = C.c_int64(0), C.c_int64(0)
    limit = 2 ** 31 - 65537
    assert L.spd_pack_rows(1, limit, 1, limit, 1, C.byref(rows), C.byref(ms)) == 0 and rows.value == 1
    assert L.spd_pack_rows(1, limit + 1, 1, limit + 1, 1, C.byref(rows), C.byref(ms)) == -1
    fake = C.c_void_p(4096)
    assert L.spd_pad_for_sequence_parallel(fake, fake, 1, limit + 1, 1, 0, 0, None) == -1
    assert L.spd_split_sequence_parallel(fake, None, None, 1, limit + 1, 1, 0, fake, None, None, None) == -1
    assert L.spd_unpack_data(fake, fake, fake, fake, 1, 1, limit + 1, fake, fake, None) == -1


def test_pad_for_sequence_parallel_host_checks(lib):
    """Argument checks answered on the host, before any GPU work."""
    import ctypes as C
    from sample_packing_document_gb300 import ops
    L = ops.load()
    fake = C.c_void_p(4096)
    assert L.spd_pad_for_sequence_parallel(fake, fake, 1, 10, 0, 0, 0, None) == -1      # sp_size < 1
    assert L.spd_pad_for_sequence_parallel(fake, fake, -1, 10, 4, 0, 0, None) == -1     # rows < 0
    assert L.spd_pad_for_sequence_parallel(fake, fake, 4, 2 ** 30, 3, 0, 0, None) == -1  # rows * padded > 2^31 - 1
    assert L.spd_pad_for_sequence_parallel(fake, None, 1, 10, 4, 0, 0, None) == -1      # no output
    assert L.spd_pad_for_sequence_parallel(fake, C.c_void_p(4098), 1, 10, 4, 0, 0, None) == -1   # unaligned
    assert L.spd_pad_for_sequence_parallel(None, None, 0, 10, 4, 0, 0, None) == 0       # nothing to do


def test_pack_rows_host_logic(lib):
    from sample_packing_document_gb300 import ops
    assert ops.pack_rows(4, 24, 2, 8, True) == (2, 8)        # the page's example: 2 rows
    assert ops.pack_rows(6, 44, 2, 8, False) == (3, 12)      # build_unpack example: 3 rows
    assert ops.pack_rows(0, 0, 2, 8, True) == (0, 0)
    with pytest.raises(ops.SpdError):
        ops.pack_rows(1, 1, 0, 8, True)
    with pytest.raises(ops.SpdError):
        ops.pack_rows(1, 2 ** 31, 1, 8, True)
    with pytest.raises(ops.SpdError):
        ops.pack_rows(1, 0, 1, 8, True)


def test_attn_workspace_and_rejections_without_gpu(lib):
    from sample_packing_document_gb300 import ops
    assert ops.attn_workspace_size(1000, 3, 4, 2, 128, False) > 0
    bwd = ops.attn_workspace_size(1000, 3, 4, 2, 128, True)
    assert bwd >= 4 * 1000 * 128 * 4                         # holds the fp32 dQ accumulator
    assert lib.spd_attn_workspace_size(1000, 3, 4, 2, 96, 0) == 0    # head_dim 96 unsupported
    assert lib.spd_attn_workspace_size(1000, 3, 6, 4, 128, 0) == 0   # Hq % Hkv != 0
    # host checks come before any CUDA call
    rc = lib.spd_varlen_attn_fwd(None, None, None, None, 3, 1000, 0, 4, 2, 96, 0.0, None, None, None, 0, None)
    assert rc == -2
    rc = lib.spd_varlen_attn_fwd(None, None, None, None, 3, 1000, 0, 4, 2, 128, 0.0, None, None, None, 0, None)
    assert rc == -6
    rc = lib.spd_varlen_attn_fwd(None, None, None, None, 0, 1000, 0, 4, 2, 128, 0.0, None, None, None, 0, None)
    assert rc == -1
    rc = lib.spd_varlen_attn_bwd(None, None, None, None, None, None, None, 3, 1000, 0, 4, 2, 128, 0.0, 2,
                                 None, None, None, None, 0, None)
    assert rc == -1
    rc = lib.spd_pack_tokens(None, None, 2, 5, 2, 8, 1, None, None, None, None, None, None, None, None, 0, None)
    assert rc == -6


def test_oracle_does_not_leak_into_product():
    """The product package never imports the oracle."""
    pkg = os.path.join(ROOT, "sample_packing_document_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", text, re.M), f
                assert "oracle/" not in text and "liboracle" not in text, f


def test_debug_skip_hook_validates_its_argument():
    """The failure-detection test hook accepts only its three codes (host only)."""
    from sample_packing_document_gb300 import build, ops
    build.build()
    lib = ops.load()
    assert lib.spd_debug_skip_arrive(3) == -1
    assert lib.spd_debug_skip_arrive(-1) == -1
    assert lib.spd_debug_skip_arrive(ops.DEBUG_SKIP_FWD_Q) == 0
    assert lib.spd_debug_skip_arrive(ops.DEBUG_SKIP_NONE) == 0   # cleared again


def test_data_steps_host_checks_without_gpu(lib):
    """Argument checks of the data-step entry points run before any GPU call."""
    import ctypes
    P = ctypes.c_void_p
    one = P(16)
    # unpack: micro_bsz / seq_len must be >= 1; rows == 0 is a no-op
    assert lib.spd_unpack_data(one, one, one, one, 1, 0, 8, one, one, None) == -1
    assert lib.spd_unpack_data(one, one, one, one, 1, 2, 0, one, one, None) == -1
    assert lib.spd_unpack_data(one, one, one, one, 0, 2, 8, one, one, None) == 0
    # split: len must divide by sp_size, rank in range, src / dst paired
    assert lib.spd_split_sequence_parallel(one, None, None, 2, 10, 4, 0, one, None, None, None) == -1
    assert lib.spd_split_sequence_parallel(one, None, None, 2, 8, 4, 4, one, None, None, None) == -1
    assert lib.spd_split_sequence_parallel(one, one, None, 2, 8, 4, 0, one, None, None, None) == -1
    assert lib.spd_split_sequence_parallel(one, None, None, 0, 8, 4, 0, one, None, None, None) == 0


def test_rope_host_checks_without_gpu(lib):
    """spd_rope's argument checks run before any GPU call."""
    import ctypes
    P = ctypes.c_void_p
    assert lib.spd_rope(P(16), None, P(16), 4, 2, 0, 96, ctypes.c_float(0), 0, None) == -2   # head_dim
    assert lib.spd_rope(P(18), None, P(16), 4, 2, 0, 128, ctypes.c_float(0), 0, None) == -1  # alignment
    assert lib.spd_rope(P(16), None, None, 4, 2, 0, 128, ctypes.c_float(0), 0, None) == -1   # positions
    assert lib.spd_rope(P(16), None, P(16), 0, 2, 0, 128, ctypes.c_float(0), 0, None) == 0   # T = 0


def test_loss_host_checks_without_gpu(lib):
    """spd_masked_token_loss's argument checks run before any GPU call."""
    import ctypes
    P = ctypes.c_void_p
    assert lib.spd_masked_token_loss(P(16), P(16), 4, 0, P(16), P(16), P(16), None, ctypes.c_float(0), None,
                                     None) == -1   # V < 1
    assert lib.spd_masked_token_loss(P(16), P(16), 4, 8, P(16), None, P(16), None, ctypes.c_float(0), None,
                                     None) == -1   # no loss_sum
    assert lib.spd_masked_token_loss(P(16), P(16), 4, 8, P(16), P(12), P(16), None, ctypes.c_float(0), None,
                                     None) == -1   # loss_sum not 8-byte aligned
