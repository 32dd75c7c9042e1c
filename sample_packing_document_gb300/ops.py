"""Python binding of libspd.so: argument marshalling only.

Every step runs in the library's CUDA kernels; torch supplies device memory
and the current stream. There is no CPU fallback: if the library or a GB300
is missing, the first call raises.

Names follow the C ABI in include/spd.h.
"""
import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libspd.so")
_lib = None

SPD_OK = 0
_P = ctypes.c_void_p
_I32, _I64, _INT, _F32, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

# name -> (restype, argtypes); the full exported surface of include/spd.h
SIGNATURES = {
    "spd_status_string": (ctypes.c_char_p, [_INT]),
    "spd_version": (_INT, []),
    "spd_read_status": (_INT, [_P, _P, ctypes.POINTER(_INT)]),
    "spd_attn_read_schedule": (_INT, [_P, _P, ctypes.POINTER(_I32), _P, _I64]),
    "spd_set_profile_events": (_INT, [_P, _P, _INT]),
    "spd_debug_skip_arrive": (_INT, [_INT]),
    "spd_pack_rows": (_INT, [_I64, _I64, _INT, _INT, _INT, ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "spd_pack_workspace_size": (_SZ, [_I64]),
    "spd_pack_tokens": (_INT, [_P, _P, _I64, _I64, _INT, _INT, _INT, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "spd_attn_workspace_size": (_SZ, [_I64, _I32, _INT, _INT, _INT, _INT]),
    "spd_pack_num_segs": (_INT, [_P, _I64, _INT, _INT, _INT, ctypes.POINTER(_I64)]),
    "spd_varlen_attn_fwd": (_INT, [_P, _P, _P, _P, _I32, _I64, _I32, _INT, _INT, _INT, _F32, _P, _P, _P, _SZ, _P]),
    "spd_varlen_attn_bwd": (_INT, [_P, _P, _P, _P, _P, _P, _P, _I32, _I64, _I32, _INT, _INT, _INT, _F32, _INT,
                                   _P, _P, _P, _P, _SZ, _P]),
    "spd_varlen_attn_fwd_rope": (_INT, [_P, _P, _P, _P, _I32, _I64, _I32, _INT, _INT, _INT, _F32, _F32, _P, _P, _P,
                                        _SZ, _P]),
    "spd_varlen_attn_fwd_noalloc": (_INT, [_P, _P, _P, _P, _I32, _I64, _I32, _INT, _INT, _INT, _F32, _P, _P, _P,
                                           _P]),
    "spd_unpack_data": (_INT, [_P, _P, _P, _P, _I64, _INT, _INT, _P, _P, _P]),
    "spd_split_sequence_parallel": (_INT, [_P, _P, _P, _I64, _I64, _INT, _INT, _P, _P, _P, _P]),
    "spd_pad_for_sequence_parallel": (_INT, [_P, _P, _I64, _I64, _INT, _I32, _INT, _P]),
    "spd_rope": (_INT, [_P, _P, _P, _I64, _INT, _INT, _INT, _F32, _INT, _P]),
    "spd_masked_token_loss": (_INT, [_P, _P, _I64, _I64, _P, _P, _P, _P, _F32, _P, _P]),
}


class SpdError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__("%s: %s (%d)" % (fn, status_string(status), status))


def load(path=_LIB_PATH):
    """Load libspd.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError("libspd.so is not built (run __graft_entry__.build()); there is no CPU fallback")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def status_string(status):
    return load().spd_status_string(int(status)).decode()


def _check(fn, rc):
    if rc != SPD_OK:
        raise SpdError(fn, rc)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need_cuda(*ts):
    if not torch.cuda.is_available():
        raise RuntimeError("spd needs a CUDA GPU (GB300); there is no CPU fallback")
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("inputs must be contiguous CUDA tensors")


def workspace(nbytes, device=None):
    """A 256-byte aligned byte buffer (torch allocations are)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def read_status(ws, stream=None):
    """Synchronise and return the device status word of the last call on ws."""
    v = _INT(0)
    _check("spd_read_status", load().spd_read_status(_ptr(ws), _stream(stream), ctypes.byref(v)))
    return v.value


def read_schedule(ws, stream=None):
    """Synchronise and return the tile schedule of the last attention call on
    ws as an int32 array [units, 4] of {segment start, segment end, tile, cost}
    (see spd_attn_read_schedule)."""
    import numpy as np
    n = _I32(0)
    _check("spd_attn_read_schedule", load().spd_attn_read_schedule(_ptr(ws), _stream(stream), ctypes.byref(n),
                                                                   None, 0))
    units = np.zeros((max(n.value, 0), 4), np.int32)
    if n.value > 0:
        _check("spd_attn_read_schedule",
               load().spd_attn_read_schedule(_ptr(ws), _stream(stream), ctypes.byref(n),
                                             units.ctypes.data_as(ctypes.c_void_p), units.shape[0]))
    return units


(PROFILE_NONE, PROFILE_PACK_STREAM, PROFILE_ATTN_FWD, PROFILE_ATTN_BWD, PROFILE_UNPACK, PROFILE_SPLIT,
 PROFILE_ROPE, PROFILE_LOSS, PROFILE_PAD) = 0, 1, 2, 3, 4, 5, 6, 7, 8

# Pad of each tensor pad_for_sequence_parallel pads: (value, count): the pad id,
# the ignore index, position ids counting 0, 1, 2, ... and attention mask 0.
SP_PAD = {"input_ids": (0, False), "labels": (-100, False), "position_ids": (0, True), "attention_mask": (0, False)}


def set_profile_events(begin, end, kernel):
    """Record torch.cuda.Event pair (begin, end) around one library kernel of
    the following calls on this thread (see spd_set_profile_events)."""
    b = ctypes.c_void_p(begin.cuda_event) if begin is not None else None
    e = ctypes.c_void_p(end.cuda_event) if end is not None else None
    _check("spd_set_profile_events", load().spd_set_profile_events(b, e, int(kernel)))


DEBUG_SKIP_NONE, DEBUG_SKIP_FWD_Q, DEBUG_SKIP_BWD_KV = 0, 1, 2


def debug_skip_arrive(which):
    """Failure-detection test hook (see spd_debug_skip_arrive): the next
    forward (DEBUG_SKIP_FWD_Q) or backward (DEBUG_SKIP_BWD_KV) call on this
    thread leaves one producer arrive out and reports a device timeout."""
    _check("spd_debug_skip_arrive", load().spd_debug_skip_arrive(int(which)))


# ----------------------------------------------------------------------------- packing

def pack_rows(num_docs, num_tokens, micro_bsz, seq_len, use_packed_dataset=True):
    rows, max_segs = _I64(0), _I64(0)
    _check("spd_pack_rows", load().spd_pack_rows(int(num_docs), int(num_tokens), int(micro_bsz), int(seq_len),
                                                 int(bool(use_packed_dataset)), ctypes.byref(rows),
                                                 ctypes.byref(max_segs)))
    return rows.value, max_segs.value


def pack_workspace_size(num_docs):
    return load().spd_pack_workspace_size(int(num_docs))


def pack_num_segs(doc_lens, micro_bsz, seq_len, use_packed_dataset=True):
    """spd_pack_num_segs on host document lengths (any int sequence): the
    segment count spd_pack_tokens will produce, without touching the GPU."""
    import numpy as np
    lens = np.ascontiguousarray(np.asarray(doc_lens, dtype=np.int32))
    n = _I64(0)
    _check("spd_pack_num_segs", load().spd_pack_num_segs(lens.ctypes.data_as(ctypes.c_void_p), int(lens.shape[0]),
                                                         int(micro_bsz), int(seq_len), int(bool(use_packed_dataset)),
                                                         ctypes.byref(n)))
    return int(n.value)


def alloc_pack_outputs(num_docs, num_tokens, micro_bsz, seq_len, use_packed_dataset=True, device="cuda"):
    rows, max_segs = pack_rows(num_docs, num_tokens, micro_bsz, seq_len, use_packed_dataset)
    n = rows * micro_bsz * seq_len
    i32 = dict(dtype=torch.int32, device=device)
    return {
        "rows": rows, "max_segs": max_segs,
        "input_ids": torch.empty(n, **i32), "labels": torch.empty(n, **i32), "indexes": torch.empty(n, **i32),
        "cu_seqlens": torch.empty(max_segs + 1, **i32), "row_seg_ptr": torch.empty(rows + 1, **i32),
        "max_seqlen": torch.empty(max(rows, 1), **i32), "num_segs": torch.empty(1, **i32),
        "ws": workspace(pack_workspace_size(num_docs), device),
    }


def pack_tokens(tokens, doc_lens, micro_bsz, seq_len, use_packed_dataset=True, out=None, stream=None):
    """spd_pack_tokens. tokens / doc_lens: int32 CUDA tensors. Returns the
    output dict (see alloc_pack_outputs); its num_segs stays on the device."""
    _need_cuda(tokens, doc_lens)
    assert tokens.dtype == torch.int32 and doc_lens.dtype == torch.int32
    nd, nt = doc_lens.numel(), tokens.numel()
    if out is None:
        out = alloc_pack_outputs(nd, nt, micro_bsz, seq_len, use_packed_dataset, tokens.device)
    ws = out["ws"]
    _check("spd_pack_tokens", load().spd_pack_tokens(
        _ptr(tokens), _ptr(doc_lens), nd, nt, int(micro_bsz), int(seq_len), int(bool(use_packed_dataset)),
        _ptr(out["input_ids"]), _ptr(out["labels"]), _ptr(out["indexes"]), _ptr(out["cu_seqlens"]),
        _ptr(out["row_seg_ptr"]), _ptr(out["max_seqlen"]), _ptr(out["num_segs"]), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def unpack_data(input_ids, labels, cu_seqlens, row_seg_ptr, rows, micro_bsz, seq_len, out_ids=None,
                out_labels=None, stream=None):
    """spd_unpack_data: packed rows (as pack_tokens wrote them, use_packed_dataset
    False) -> (ids, labels) int32 [rows, micro_bsz, seq_len]."""
    _need_cuda(input_ids, labels, cu_seqlens, row_seg_ptr)
    shape = (int(rows), int(micro_bsz), int(seq_len))
    if out_ids is None:
        out_ids = torch.empty(shape, dtype=torch.int32, device=input_ids.device)
    if out_labels is None:
        out_labels = torch.empty(shape, dtype=torch.int32, device=input_ids.device)
    _check("spd_unpack_data", load().spd_unpack_data(
        _ptr(input_ids), _ptr(labels), _ptr(cu_seqlens), _ptr(row_seg_ptr), int(rows), int(micro_bsz),
        int(seq_len), _ptr(out_ids), _ptr(out_labels), _stream(stream)))
    return out_ids, out_labels


def split_sequence_parallel(tensors, sp_size, rank, out=None, stream=None):
    """spd_split_sequence_parallel: up to three int32 CUDA tensors [rows, len]
    (or [len]) -> this rank's [rows, len / sp_size] chunks."""
    tensors = list(tensors)
    if not 1 <= len(tensors) <= 3:
        raise ValueError("one to three tensors")
    _need_cuda(*tensors)
    shp = tensors[0].shape
    rows, n = (1, shp[0]) if len(shp) == 1 else (shp[0], shp[1])
    if out is None:
        oshape = (n // sp_size,) if len(shp) == 1 else (rows, n // sp_size)
        out = [torch.empty(oshape, dtype=torch.int32, device=tensors[0].device) for _ in tensors]
    src = [_ptr(x) for x in tensors] + [None] * (3 - len(tensors))
    dst = [_ptr(x) for x in out] + [None] * (3 - len(out))
    _check("spd_split_sequence_parallel", load().spd_split_sequence_parallel(
        src[0], src[1], src[2], int(rows), int(n), int(sp_size), int(rank), dst[0], dst[1], dst[2],
        _stream(stream)))
    return out


def pad_for_sequence_parallel(sp_size, input_ids=None, labels=None, position_ids=None, attention_mask=None,
                              stream=None):
    """spd_pad_for_sequence_parallel on each given int32 CUDA tensor [rows, len]
    (or [len]): padded to the smallest multiple of sp_size along the sequence
    with the pad of its kind (SP_PAD). Returns the four results in order (None
    for tensors not given)."""
    out = []
    for kind, x in (("input_ids", input_ids), ("labels", labels), ("position_ids", position_ids),
                    ("attention_mask", attention_mask)):
        if x is None:
            out.append(None)
            continue
        _need_cuda(x)
        rows, n = (1, x.shape[0]) if x.dim() == 1 else (x.shape[0], x.shape[1])
        padded = -(-n // sp_size) * sp_size if sp_size >= 1 else n
        y = torch.empty((padded,) if x.dim() == 1 else (rows, padded), dtype=torch.int32, device=x.device)
        value, count = SP_PAD[kind]
        _check("spd_pad_for_sequence_parallel", load().spd_pad_for_sequence_parallel(
            _ptr(x), _ptr(y), int(rows), int(n), int(sp_size), int(value), int(count), _stream(stream)))
        out.append(y)
    return tuple(out)


def rope(q, k, positions, rope_theta=None, inverse=False, stream=None):
    """spd_rope: rotate q [T, Hq, d] and / or k [T, Hkv, d] (bf16 CUDA tensors,
    either may be None) in place by the per-token positions (int32 [T], e.g.
    the pack's indexes). inverse=True applies the transposed rotation (the
    gradient map). Returns (q, k)."""
    _need_cuda(q, k, positions)
    ref = q if q is not None else k
    T, _, d = ref.shape
    Hq = q.shape[1] if q is not None else 0
    Hkv = k.shape[1] if k is not None else 0
    _check("spd_rope", load().spd_rope(_ptr(q), _ptr(k), _ptr(positions), int(T), int(Hq), int(Hkv), int(d),
                                       float(rope_theta or 0.0), int(bool(inverse)), _stream(stream)))
    return q, k


def masked_token_loss(logits, labels, dlogits=None, grad_scale=0.0, token_loss=None, device_status=None,
                      stream=None):
    """spd_masked_token_loss: logits bf16 [T, V], labels int32 [T] CUDA tensors.
    Returns (token_loss fp32 [T], loss_sum fp64 [1], num_tokens int32 [1]) on the
    device; dlogits (bf16 [T, V]) is filled when given."""
    _need_cuda(logits, labels, dlogits, device_status)
    T, V = logits.shape
    if token_loss is None:
        token_loss = torch.empty(T, dtype=torch.float32, device=logits.device)
    loss_sum = torch.empty(1, dtype=torch.float64, device=logits.device)
    num_tokens = torch.empty(1, dtype=torch.int32, device=logits.device)
    _check("spd_masked_token_loss", load().spd_masked_token_loss(
        _ptr(logits), _ptr(labels), int(T), int(V), _ptr(token_loss), _ptr(loss_sum), _ptr(num_tokens),
        _ptr(dlogits), float(grad_scale), _ptr(device_status), _stream(stream)))
    return token_loss, loss_sum, num_tokens


# ----------------------------------------------------------------------------- attention

def attn_workspace_size(total_tokens, num_segs, Hq, Hkv, head_dim, bwd):
    n = load().spd_attn_workspace_size(int(total_tokens), int(num_segs), int(Hq), int(Hkv), int(head_dim),
                                       int(bool(bwd)))
    if n == 0:
        raise ValueError("unsupported attention shape")
    return n


def _as_u16(t):
    assert t.dtype == torch.bfloat16
    return t


def varlen_attn_fwd(q, k, v, cu_seqlens, num_segs, max_seqlen=0, softmax_scale=None, out=None, lse=None,
                    ws=None, stream=None):
    """spd_varlen_attn_fwd. q [T, Hq, d], k / v [T, Hkv, d] bf16 CUDA tensors,
    cu_seqlens int32 [num_segs + 1] CUDA tensor, num_segs a host int.
    Returns (out bf16 [T, Hq, d], lse fp32 [Hq, T])."""
    _need_cuda(q, k, v, cu_seqlens)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, T, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(attn_workspace_size(T, num_segs, Hq, Hkv, d, False), q.device)
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check("spd_varlen_attn_fwd", load().spd_varlen_attn_fwd(
        _ptr(_as_u16(q)), _ptr(_as_u16(k)), _ptr(_as_u16(v)), _ptr(cu_seqlens), int(num_segs), T, int(max_seqlen),
        Hq, Hkv, d, scale, _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))
    return out, lse


def varlen_attn_fwd_rope(q, k, v, cu_seqlens, num_segs, rope_theta=10000.0, max_seqlen=0, softmax_scale=None,
                         out=None, lse=None, ws=None, stream=None):
    """spd_varlen_attn_fwd_rope: the forward pass on RoPE-rotated q and k, the
    rotation (per-document positions from cu_seqlens) done inside the kernel.
    Returns (out bf16 [T, Hq, d], lse fp32 [Hq, T])."""
    _need_cuda(q, k, v, cu_seqlens)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, T, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(attn_workspace_size(T, num_segs, Hq, Hkv, d, False), q.device)
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check("spd_varlen_attn_fwd_rope", load().spd_varlen_attn_fwd_rope(
        _ptr(_as_u16(q)), _ptr(_as_u16(k)), _ptr(_as_u16(v)), _ptr(cu_seqlens), int(num_segs), T, int(max_seqlen),
        Hq, Hkv, d, scale, float(rope_theta), _ptr(out), _ptr(lse), _ptr(ws), ws.numel(), _stream(stream)))
    return out, lse


def varlen_attn_bwd(q, k, v, out, dout, lse, cu_seqlens, num_segs, max_seqlen=0, softmax_scale=None,
                    grad_dtype=torch.bfloat16, dq=None, dk=None, dv=None, ws=None, stream=None):
    """spd_varlen_attn_bwd. Returns (dq, dk, dv) in grad_dtype (bf16 or fp32)."""
    _need_cuda(q, k, v, out, dout, lse, cu_seqlens)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    assert grad_dtype in (torch.bfloat16, torch.float32)
    if dq is None:
        dq = torch.empty(T, Hq, d, dtype=grad_dtype, device=q.device)
    if dk is None:
        dk = torch.empty(T, Hkv, d, dtype=grad_dtype, device=q.device)
    if dv is None:
        dv = torch.empty(T, Hkv, d, dtype=grad_dtype, device=q.device)
    if ws is None:
        ws = workspace(attn_workspace_size(T, num_segs, Hq, Hkv, d, True), q.device)
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check("spd_varlen_attn_bwd", load().spd_varlen_attn_bwd(
        _ptr(_as_u16(q)), _ptr(_as_u16(k)), _ptr(_as_u16(v)), _ptr(_as_u16(out)), _ptr(_as_u16(dout)), _ptr(lse),
        _ptr(cu_seqlens), int(num_segs), T, int(max_seqlen), Hq, Hkv, d, scale,
        1 if grad_dtype == torch.float32 else 0, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
        _stream(stream)))
    return dq, dk, dv


def default_scale(head_dim):
    return 1.0 / math.sqrt(head_dim)


def varlen_attn_fwd_noalloc(q, k, v, cu_seqlens, num_segs, out, lse, device_status=None, max_seqlen=0,
                            softmax_scale=None, stream=None):
    """spd_varlen_attn_fwd_noalloc: the forward pass for callers that cannot
    allocate. The caller passes every tensor (out, lse, and optionally a
    one-element int32 device_status); the library uses its fixed scratch."""
    _need_cuda(q, k, v, cu_seqlens, out, lse)
    T, Hq, d = q.shape
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check("spd_varlen_attn_fwd_noalloc", load().spd_varlen_attn_fwd_noalloc(
        _ptr(_as_u16(q)), _ptr(_as_u16(k)), _ptr(_as_u16(v)), _ptr(cu_seqlens), int(num_segs), T, int(max_seqlen),
        Hq, k.shape[1], d, scale, _ptr(out), _ptr(lse), _ptr(device_status), _stream(stream)))
    return out, lse
