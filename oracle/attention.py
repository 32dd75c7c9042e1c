"""ctypes wrappers around the C oracle (attn_ref.c, pack_ref.c).
TEST INFRASTRUCTURE ONLY.

Arrays in: numpy. Attention inputs are bf16 bit patterns as uint16 arrays
(q [T, Hq, d], k / v [T, Hkv, d]); the C side widens them exactly to double.
Outputs are float64 (attention) or int32 (packing).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        L.spd_oracle_attn_fwd.argtypes = [P, P, P, P, i32, i64, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, dbl, i64, P, P, P, ctypes.c_int]
        L.spd_oracle_attn_dq_rows.argtypes = [P, P, P, P, P, i32, i64, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, dbl, i64, P, P,
                                              ctypes.c_int]
        L.spd_oracle_attn_bwd.argtypes = [P, P, P, P, P, i32, i64, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, dbl, i32, P, P, P, P, ctypes.c_int]
        L.spd_oracle_pack_rows.argtypes = [i64, i64, P, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, P, P]
        L.spd_oracle_pack.argtypes = [P, P, i64, i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      P, P, P, P, P, P, P]
        for f in (L.spd_oracle_attn_fwd, L.spd_oracle_attn_dq_rows, L.spd_oracle_attn_bwd,
                  L.spd_oracle_pack_rows, L.spd_oracle_pack):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "attention oracle takes bf16 bit patterns (uint16)"
    return a


def _cu(cu):
    return np.ascontiguousarray(np.asarray(cu, dtype=np.int32))


def default_threads():
    return len(os.sched_getaffinity(0))


def attn_fwd(q, k, v, cu_seqlens, scale=None, items=None, nthreads=0):
    """O and LSE. items: None (every row, returned as out [Hq, T, d],
    lse [Hq, T]) or an int64 array of h * T + i (returned as [n, d], [n])."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    cu = _cu(cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if items is None:
        n = Hq * T
        it = None
    else:
        it = np.ascontiguousarray(np.asarray(items, dtype=np.int64))
        n = it.shape[0]
    out = np.empty((n, d), np.float64)
    lse = np.empty((n,), np.float64)
    rc = lib().spd_oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, T, Hq,
                                   Hkv, d, float(scale), n, _ptr(it), _ptr(out), _ptr(lse),
                                   nthreads)
    if rc != 0:
        raise ValueError("oracle attn_fwd rejected its arguments")
    if items is None:
        return out.reshape(Hq, T, d), lse.reshape(Hq, T)
    return out, lse


def attn_dq_rows(q, k, v, dout, cu_seqlens, items, scale=None, nthreads=0):
    """dQ for the (head, row) items h * T + i; returns [n, d]."""
    q, k, v, dout = _u16(q), _u16(k), _u16(v), _u16(dout)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    cu = _cu(cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    it = np.ascontiguousarray(np.asarray(items, dtype=np.int64))
    dq = np.empty((it.shape[0], d), np.float64)
    rc = lib().spd_oracle_attn_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(cu),
                                       len(cu) - 1, T, Hq, Hkv, d, float(scale), it.shape[0],
                                       _ptr(it), _ptr(dq), nthreads)
    if rc != 0:
        raise ValueError("oracle attn_dq_rows rejected its arguments")
    return dq


def attn_bwd(q, k, v, dout, cu_seqlens, segs=None, scale=None, nthreads=0):
    """Exact gradient over whole segments. segs: None (all) or a list of
    segment ids. Returns (dq, dk, dv, rows) where rows are the token indices
    the compact outputs cover, in order: dq [len(rows), Hq, d],
    dk / dv [len(rows), Hkv, d]."""
    q, k, v, dout = _u16(q), _u16(k), _u16(v), _u16(dout)
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    cu = _cu(cu_seqlens)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if segs is None:
        sel = None
        rows = np.arange(T)
    else:
        sel = np.ascontiguousarray(np.asarray(segs, dtype=np.int32))
        rows = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in sel]) if len(sel) else \
            np.zeros((0,), np.int64)
    n = rows.shape[0]
    dq = np.empty((n, Hq, d), np.float64)
    dk = np.empty((n, Hkv, d), np.float64)
    dv = np.empty((n, Hkv, d), np.float64)
    nsel = len(cu) - 1 if sel is None else sel.shape[0]
    rc = lib().spd_oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(cu), len(cu) - 1,
                                   T, Hq, Hkv, d, float(scale), nsel, _ptr(sel), _ptr(dq),
                                   _ptr(dk), _ptr(dv), nthreads)
    if rc != 0:
        raise ValueError("oracle attn_bwd rejected its arguments")
    return dq, dk, dv, rows


def pack(tokens, doc_lens, micro_bsz, seq_len, use_packed_dataset=True):
    """The C restatement of the packing rules; flat outputs as numpy int32."""
    tokens = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
    doc_lens = np.ascontiguousarray(np.asarray(doc_lens, dtype=np.int32))
    rows = ctypes.c_int64()
    max_segs = ctypes.c_int64()
    L = lib()
    rc = L.spd_oracle_pack_rows(doc_lens.shape[0], tokens.shape[0], _ptr(doc_lens), micro_bsz,
                                seq_len, int(bool(use_packed_dataset)), ctypes.byref(rows),
                                ctypes.byref(max_segs))
    if rc != 0:
        raise ValueError("oracle pack rejected its arguments")
    n = rows.value * micro_bsz * seq_len
    ids = np.empty(n, np.int32)
    labels = np.empty(n, np.int32)
    indexes = np.empty(n, np.int32)
    cu = np.empty(max_segs.value + 1, np.int32)
    rsp = np.empty(rows.value + 1, np.int32)
    mx = np.empty(max(rows.value, 1), np.int32)
    ns = np.empty(1, np.int32)
    rc = L.spd_oracle_pack(_ptr(tokens), _ptr(doc_lens), doc_lens.shape[0], tokens.shape[0],
                           micro_bsz, seq_len, int(bool(use_packed_dataset)), _ptr(ids),
                           _ptr(labels), _ptr(indexes), _ptr(cu), _ptr(rsp), _ptr(mx), _ptr(ns))
    if rc != 0:
        raise ValueError("oracle pack rejected its arguments")
    return {"input_ids": ids, "labels": labels, "indexes": indexes,
            "cu_seqlens": cu[:ns[0] + 1].copy(), "row_seg_ptr": rsp,
            "max_seqlen": mx[:rows.value].copy(), "num_segs": int(ns[0]), "rows": rows.value}
