"""Thin ctypes binding of libcpattn's C ABI (include/cpattn.h).

The ``cpattn_*`` functions here have the C names and arguments (device
pointers as Python ints, sizes, a stream handle) and do nothing but
marshalling. ``shard``, ``fwd``, ``bwd`` ... below them only read pointers and
sizes off torch tensors and call those functions; every step of the
computation runs in the library's CUDA kernels. There is no fallback: if the
shared library is missing or a call fails, a ``CpattnError`` is raised.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcpattn.so")

OK, ERR_ARG, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED = range(8)
F32, BF16 = 0, 1

# Every symbol the header declares.
EXPORTS = ("cpattn_shard", "cpattn_unshard", "cpattn_shard_rope", "cpattn_unshard_rope",
           "cpattn_shard_index", "cpattn_fwd",
           "cpattn_bwd_workspace_bytes", "cpattn_bwd", "cpattn_merge", "cpattn_last_error",
           "cpattn_sync_status", "cpattn_version", "cpattn_set_trace_events", "cpattn_bwd_noalloc",
           "cpattn_fwd_gqa", "cpattn_bwd_gqa", "cpattn_shard_rope_cfg", "cpattn_unshard_rope_cfg",
           "cpattn_doc_bounds", "cpattn_fwd_varlen", "cpattn_bwd_varlen", "cpattn_ulysses_a2a",
           "cpattn_ulysses_a2a_rope", "cpattn_fwd_rope_cfg", "cpattn_bwd_rope_cfg",
           "cpattn_check_wait_timeout", "cpattn_fwd_rope_save", "cpattn_bwd_rotated", "cpattn_shard_batch",
           "cpattn_unshard_batch")


class CpattnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"cpattn status {status}: {msg}")
        self.status = status


_lib = None
_c = ctypes
_vp, _i, _sz = _c.c_void_p, _c.c_int, _c.c_size_t


class RopeCfg(ctypes.Structure):
    """cpattn_rope_cfg: RoPE base and the YaRN extension (factor 1 = standard)."""
    _fields_ = [("base", ctypes.c_double), ("factor", ctypes.c_double),
                ("original_max_position", ctypes.c_int), ("beta_fast", ctypes.c_double),
                ("beta_slow", ctypes.c_double), ("attention_factor", ctypes.c_double)]

    def __init__(self, factor=1.0, original_max_position=0, base=10000.0, beta_fast=32.0,
                 beta_slow=1.0, attention_factor=0.0):
        super().__init__(base, factor, original_max_position, beta_fast, beta_slow, attention_factor)


def _declare(lib):
    sig = {
        "cpattn_shard": [_vp, _vp, _i, _i, _i, _i, _i, _i, _vp],
        "cpattn_unshard": [_vp, _vp, _i, _i, _i, _i, _i, _i, _vp],
        "cpattn_shard_rope": [_vp, _vp, _i, _i, _i, _i, _i, _i, _vp],
        "cpattn_unshard_rope": [_vp, _vp, _i, _i, _i, _i, _i, _i, _vp],
        "cpattn_shard_index": [_i, _i, _c.POINTER(_c.c_int32)],
        "cpattn_fwd": [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i, _vp],
        "cpattn_bwd": [_vp] * 10 + [_i] * 9 + [_vp],
        "cpattn_bwd_noalloc": [_vp] * 9 + [_i] * 9 + [_vp],
        "cpattn_fwd_gqa": [_vp] * 5 + [_i] * 10 + [_vp],
        "cpattn_doc_bounds": [_vp, _i, _i, _vp, _vp, _vp],
        "cpattn_ulysses_a2a": [_vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp],
        "cpattn_ulysses_a2a_rope": [_vp, _vp, _i, _i, _i, _i, _i, _i, _c.POINTER(RopeCfg), _i, _vp],
        "cpattn_fwd_varlen": [_vp] * 5 + [_i] * 8 + [_vp, _vp, _i, _vp],
        "cpattn_bwd_varlen": [_vp] * 10 + [_i] * 8 + [_vp, _vp, _i, _vp],
        "cpattn_shard_rope_cfg": [_vp, _vp, _i, _i, _i, _i, _i, _i, _c.POINTER(RopeCfg), _vp],
        "cpattn_unshard_rope_cfg": [_vp, _vp, _i, _i, _i, _i, _i, _i, _c.POINTER(RopeCfg), _vp],
        "cpattn_bwd_gqa": [_vp] * 10 + [_i] * 10 + [_vp],
        "cpattn_fwd_rope_cfg": [_vp] * 5 + [_i] * 8 + [_c.POINTER(RopeCfg), _i, _vp],
        "cpattn_bwd_rope_cfg": [_vp] * 10 + [_i] * 8 + [_c.POINTER(RopeCfg), _i, _vp],
        "cpattn_merge": [_c.POINTER(_vp), _c.POINTER(_vp), _i, _vp, _vp, _i, _i, _i, _i, _i, _vp],
        "cpattn_sync_status": [_vp],
        "cpattn_check_wait_timeout": [_c.c_ulonglong, _vp],
        "cpattn_shard_batch": [_c.POINTER(_vp), _c.POINTER(_vp), _c.POINTER(_i), _c.POINTER(_i), _i, _i, _i, _i, _i,
                               _c.POINTER(RopeCfg), _i, _vp],
        "cpattn_unshard_batch": [_c.POINTER(_vp), _c.POINTER(_vp), _c.POINTER(_i), _c.POINTER(_i), _i, _i, _i, _i, _i,
                                 _c.POINTER(RopeCfg), _i, _vp],
        "cpattn_fwd_rope_save": [_vp] * 7 + [_i] * 8 + [_vp, _vp, _c.POINTER(RopeCfg), _i, _vp],
        "cpattn_bwd_rotated": [_vp] * 10 + [_i] * 8 + [_vp, _vp, _c.POINTER(RopeCfg), _i, _vp],
        "cpattn_set_trace_events": [_c.POINTER(_vp), _i],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _i
    lib.cpattn_bwd_workspace_bytes.argtypes = [_i, _i, _i, _i]
    lib.cpattn_bwd_workspace_bytes.restype = _sz
    lib.cpattn_last_error.argtypes = []
    lib.cpattn_last_error.restype = _c.c_char_p
    lib.cpattn_version.argtypes = []
    lib.cpattn_version.restype = _c.c_char_p


def lib():
    """The loaded shared library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise CpattnError(ERR_UNSUPPORTED, f"{LIB_PATH} is not built; run __graft_entry__.build()")
        handle = ctypes.CDLL(LIB_PATH)
        _declare(handle)
        _lib = handle
    return _lib


def _check(status: int) -> None:
    if status != OK:
        raise CpattnError(status, lib().cpattn_last_error().decode(errors="replace"))


# ------------------------------------------------------- C-named entry points

def cpattn_shard(src, dst, B, H, T, d, cp, dt, stream=None):
    _check(lib().cpattn_shard(src, dst, B, H, T, d, cp, dt, stream))


def cpattn_unshard(src, dst, B, H, T, d, cp, dt, stream=None):
    _check(lib().cpattn_unshard(src, dst, B, H, T, d, cp, dt, stream))


def cpattn_shard_rope(src, dst, B, H, T, d, cp, dt, stream=None):
    _check(lib().cpattn_shard_rope(src, dst, B, H, T, d, cp, dt, stream))


def cpattn_unshard_rope(src, dst, B, H, T, d, cp, dt, stream=None):
    _check(lib().cpattn_unshard_rope(src, dst, B, H, T, d, cp, dt, stream))


def cpattn_shard_rope_cfg(src, dst, B, H, T, d, cp, dt, cfg, stream=None):
    _check(lib().cpattn_shard_rope_cfg(src, dst, B, H, T, d, cp, dt,
                                       None if cfg is None else ctypes.byref(cfg), stream))


def cpattn_unshard_rope_cfg(src, dst, B, H, T, d, cp, dt, cfg, stream=None):
    _check(lib().cpattn_unshard_rope_cfg(src, dst, B, H, T, d, cp, dt,
                                         None if cfg is None else ctypes.byref(cfg), stream))


def cpattn_ulysses_a2a(src, dst, B, H, T, d, P, inverse, dt, stream=None):
    _check(lib().cpattn_ulysses_a2a(src, dst, B, H, T, d, P, inverse, dt, stream))


def cpattn_ulysses_a2a_rope(src, dst, B, H, T, d, P, inverse, cfg, dt, stream=None):
    _check(lib().cpattn_ulysses_a2a_rope(src, dst, B, H, T, d, P, inverse,
                                         None if cfg is None else ctypes.byref(cfg), dt, stream))


def cpattn_shard_index(T, cp):
    buf = (ctypes.c_int32 * T)()
    _check(lib().cpattn_shard_index(T, cp, buf))
    return list(buf)


def cpattn_fwd(q, k, v, o, lse, B, T, T_valid, H, d, cp, causal, rope, dt, stream=None):
    _check(lib().cpattn_fwd(q, k, v, o, lse, B, T, T_valid, H, d, cp, causal, rope, dt, stream))


def cpattn_fwd_gqa(q, k, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal, rope, dt, stream=None):
    _check(lib().cpattn_fwd_gqa(q, k, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal, rope, dt,
                                stream))


def cpattn_fwd_varlen(q, k, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal, doc_lo, doc_hi, dt,
                      stream=None):
    _check(lib().cpattn_fwd_varlen(q, k, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal, doc_lo,
                                   doc_hi, dt, stream))


def cpattn_fwd_rope_cfg(q, k, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal, cfg, dt, stream=None):
    _check(lib().cpattn_fwd_rope_cfg(q, k, v, o, lse, B, T, T_valid, H, H_kv, d, cp, causal,
                                     None if cfg is None else ctypes.byref(cfg), dt, stream))


def cpattn_bwd_rope_cfg(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d, cp,
                        causal, cfg, dt, stream=None):
    _check(lib().cpattn_bwd_rope_cfg(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv,
                                     d, cp, causal, None if cfg is None else ctypes.byref(cfg), dt,
                                     stream))


def cpattn_fwd_rope_save(q, k, v, o, lse, q_rot, k_rot, B, T, T_valid, H, H_kv, d, cp, causal, doc_lo, doc_hi,
                         cfg, dt, stream=None):
    _check(lib().cpattn_fwd_rope_save(q, k, v, o, lse, q_rot, k_rot, B, T, T_valid, H, H_kv, d, cp, causal,
                                      doc_lo, doc_hi, None if cfg is None else ctypes.byref(cfg), dt, stream))


def cpattn_bwd_rotated(q_rot, k_rot, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d, cp, causal,
                       doc_lo, doc_hi, cfg, dt, stream=None):
    _check(lib().cpattn_bwd_rotated(q_rot, k_rot, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d,
                                    cp, causal, doc_lo, doc_hi, None if cfg is None else ctypes.byref(cfg), dt,
                                    stream))


def _batch_args(src, dst, heads, rope):
    n = len(src)
    return ((_vp * n)(*src), (_vp * n)(*dst), (_i * n)(*heads), (_i * n)(*rope), n)


def cpattn_shard_batch(src, dst, heads, rope, B, T, d, cp, cfg, dt, stream=None):
    s_, d_, h_, r_, n = _batch_args(src, dst, heads, rope)
    _check(lib().cpattn_shard_batch(s_, d_, h_, r_, n, B, T, d, cp, None if cfg is None else ctypes.byref(cfg),
                                    dt, stream))


def cpattn_unshard_batch(src, dst, heads, rope, B, T, d, cp, cfg, dt, stream=None):
    s_, d_, h_, r_, n = _batch_args(src, dst, heads, rope)
    _check(lib().cpattn_unshard_batch(s_, d_, h_, r_, n, B, T, d, cp, None if cfg is None else ctypes.byref(cfg),
                                      dt, stream))


def cpattn_doc_bounds(cu_seqlens, n_docs, T, doc_lo, doc_hi, stream=None):
    _check(lib().cpattn_doc_bounds(cu_seqlens, n_docs, T, doc_lo, doc_hi, stream))


def cpattn_bwd_workspace_bytes(B, T, H, d):
    return int(lib().cpattn_bwd_workspace_bytes(B, T, H, d))


def cpattn_bwd(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, d, cp, causal, rope,
               dt, stream=None):
    _check(lib().cpattn_bwd(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, d, cp,
                            causal, rope, dt, stream))


def cpattn_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d, cp, causal,
                   rope, dt, stream=None):
    _check(lib().cpattn_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d,
                                cp, causal, rope, dt, stream))


def cpattn_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv, d, cp,
                      causal, doc_lo, doc_hi, dt, stream=None):
    _check(lib().cpattn_bwd_varlen(q, k, v, o, lse, dO, dq, dk, dv, workspace, B, T, T_valid, H, H_kv,
                                   d, cp, causal, doc_lo, doc_hi, dt, stream))


def cpattn_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, T, T_valid, H, d, cp, causal, rope, dt,
                       stream=None):
    _check(lib().cpattn_bwd_noalloc(q, k, v, o, lse, dO, dq, dk, dv, B, T, T_valid, H, d, cp,
                                    causal, rope, dt, stream))


def cpattn_merge(o_parts, lse_parts, o, lse, B, H, T, d, dt, stream=None):
    n = len(o_parts)
    po = (ctypes.c_void_p * n)(*o_parts)
    pl = (ctypes.c_void_p * n)(*lse_parts)
    _check(lib().cpattn_merge(po, pl, n, o, lse, B, H, T, d, dt, stream))


def cpattn_sync_status(stream=None):
    _check(lib().cpattn_sync_status(stream))


def cpattn_check_wait_timeout(limit_ns, stream=None):
    _check(lib().cpattn_check_wait_timeout(limit_ns, stream))


def cpattn_set_trace_events(events):
    """events: list of raw cudaEvent_t handles (ints), or [] to turn tracing off."""
    n = len(events)
    arr = (ctypes.c_void_p * max(n, 1))(*events) if n else None
    _check(lib().cpattn_set_trace_events(arr, n))


def cpattn_last_error():
    return lib().cpattn_last_error().decode(errors="replace")


def cpattn_version():
    return lib().cpattn_version().decode()


# ------------------------------------------------------ tensor conveniences

def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise CpattnError(ERR_DTYPE, f"unsupported dtype {t.dtype}")


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ptr(t):
    if not t.is_cuda or not t.is_contiguous():
        raise CpattnError(ERR_ARG, "tensors must be contiguous CUDA tensors")
    return t.data_ptr()


def shard(src, dst, cp, stream=None):
    B, H, T, d = src.shape
    cpattn_shard(_ptr(src), _ptr(dst), B, H, T, d, cp, _dtype_code(src), _stream(stream))


def unshard(src, dst, cp, stream=None):
    B, H, T, d = src.shape
    cpattn_unshard(_ptr(src), _ptr(dst), B, H, T, d, cp, _dtype_code(src), _stream(stream))


def shard_rope(src, dst, cp, stream=None, cfg: RopeCfg | None = None):
    """dst = HeadTail shard of m R(p) src; cfg selects YaRN (None: standard RoPE)."""
    B, H, T, d = src.shape
    if cfg is None:
        cpattn_shard_rope(_ptr(src), _ptr(dst), B, H, T, d, cp, _dtype_code(src), _stream(stream))
    else:
        cpattn_shard_rope_cfg(_ptr(src), _ptr(dst), B, H, T, d, cp, _dtype_code(src), cfg,
                              _stream(stream))


def unshard_rope(src, dst, cp, stream=None, cfg: RopeCfg | None = None):
    """dst = unshard of (m R(p))^T src, the adjoint of shard_rope with the same cfg."""
    B, H, T, d = src.shape
    if cfg is None:
        cpattn_unshard_rope(_ptr(src), _ptr(dst), B, H, T, d, cp, _dtype_code(src), _stream(stream))
    else:
        cpattn_unshard_rope_cfg(_ptr(src), _ptr(dst), B, H, T, d, cp, _dtype_code(src), cfg,
                                _stream(stream))


def _kv_heads(q, *kv):
    """K/V head count of [B,H_kv,T,d] tensors that go with q [B,H,T,d]."""
    B, H, T, d = q.shape
    H_kv = kv[0].shape[1]
    for t in kv:
        if tuple(t.shape) != (B, H_kv, T, d):
            raise CpattnError(ERR_SHAPE, f"K/V-side tensor of shape {tuple(t.shape)} does not match "
                                         f"q {tuple(q.shape)} with {H_kv} K/V heads")
    return H_kv


def ulysses_a2a(src, dst, P, inverse=False, rope=False, cfg: RopeCfg | None = None, stream=None):
    """Sequence shards [P*B, H, T/P, d] <-> head shards [P*B, max(H/P, 1), T, d]
    (both rank-major). With H < P each head goes to P/H ranks and the inverse
    sums the replicas. rope=True also rotates rows at their natural positions,
    with cfg (YaRN) when given; cfg is not used when rope is False."""
    seq = dst if inverse else src
    PB, H, Tl, d = seq.shape
    B, T = PB // P, Tl * P
    head = (PB, max(H // P, 1), T, d)
    if tuple((src if inverse else dst).shape) != head:
        raise CpattnError(ERR_SHAPE, f"head shards must be {head}")
    if rope:
        cpattn_ulysses_a2a_rope(_ptr(src), _ptr(dst), B, H, T, d, P, int(inverse), cfg, _dtype_code(src),
                                _stream(stream))
    else:
        cpattn_ulysses_a2a(_ptr(src), _ptr(dst), B, H, T, d, P, int(inverse), _dtype_code(src),
                           _stream(stream))


def doc_bounds(cu_seqlens, T, doc_lo, doc_hi, stream=None):
    """doc_lo, doc_hi [T] int32 (device) from cu_seqlens [n_docs + 1] int32 (device)."""
    for t in (cu_seqlens, doc_lo, doc_hi):
        if t.dtype != _torch().int32:
            raise CpattnError(ERR_DTYPE, "cu_seqlens, doc_lo and doc_hi must be int32")
    cpattn_doc_bounds(_ptr(cu_seqlens), cu_seqlens.numel() - 1, T, _ptr(doc_lo), _ptr(doc_hi),
                      _stream(stream))


def _torch():
    import torch
    return torch


def fwd(q, k, v, o, lse, cp, T_valid=None, causal=True, rope=False, stream=None, docs=None,
        rope_cfg: RopeCfg | None = None):
    """o, lse = attention(q, k, v); k, v may have fewer heads than q (grouped K/V);
    docs = (doc_lo, doc_hi) from doc_bounds restricts attention to documents;
    rope=True rotates q, k inside the kernels, with rope_cfg (YaRN) when given."""
    B, H, T, d = q.shape
    H_kv = _kv_heads(q, k, v)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, T, T if T_valid is None else T_valid)
    if docs is not None:
        if rope:
            raise CpattnError(ERR_ARG, "packed documents take RoPE from shard_rope (rope=False)")
        cpattn_fwd_varlen(*args, H, H_kv, d, cp, int(causal), _ptr(docs[0]), _ptr(docs[1]),
                          _dtype_code(q), _stream(stream))
        return
    if rope and rope_cfg is not None:
        cpattn_fwd_rope_cfg(*args, H, H_kv, d, cp, int(causal), rope_cfg, _dtype_code(q), _stream(stream))
        return
    tail = (d, cp, int(causal), int(rope), _dtype_code(q), _stream(stream))
    if H_kv == H:
        cpattn_fwd(*args, H, *tail)
    else:
        cpattn_fwd_gqa(*args, H, H_kv, *tail)


def bwd(q, k, v, o, lse, dO, dq, dk, dv, workspace, cp, T_valid=None, causal=True, rope=False,
        stream=None, docs=None, rope_cfg: RopeCfg | None = None):
    """dq, dk, dv of sum(dO * o); k, v, dk, dv may have fewer heads than q;
    docs, rope and rope_cfg as for fwd."""
    B, H, T, d = q.shape
    H_kv = _kv_heads(q, k, v, dk, dv)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
            _ptr(workspace), B, T, T if T_valid is None else T_valid)
    if docs is not None:
        if rope:
            raise CpattnError(ERR_ARG, "packed documents take RoPE from shard_rope (rope=False)")
        cpattn_bwd_varlen(*args, H, H_kv, d, cp, int(causal), _ptr(docs[0]), _ptr(docs[1]),
                          _dtype_code(q), _stream(stream))
        return
    if rope and rope_cfg is not None:
        cpattn_bwd_rope_cfg(*args, H, H_kv, d, cp, int(causal), rope_cfg, _dtype_code(q), _stream(stream))
        return
    tail = (d, cp, int(causal), int(rope), _dtype_code(q), _stream(stream))
    if H_kv == H:
        cpattn_bwd(*args, H, *tail)
    else:
        cpattn_bwd_gqa(*args, H, H_kv, *tail)


def fwd_rope_save(q, k, v, o, lse, q_rot, k_rot, cp, T_valid=None, causal=True, stream=None, docs=None,
                  rope_cfg: RopeCfg | None = None):
    """fwd with in-kernel RoPE that also stores the rotated q_rot, k_rot for bwd_rotated."""
    B, H, T, d = q.shape
    H_kv = _kv_heads(q, k, v, k_rot)
    cpattn_fwd_rope_save(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(q_rot), _ptr(k_rot), B, T,
                         T if T_valid is None else T_valid, H, H_kv, d, cp, int(causal),
                         None if docs is None else _ptr(docs[0]), None if docs is None else _ptr(docs[1]),
                         rope_cfg, _dtype_code(q), _stream(stream))


def bwd_rotated(q_rot, k_rot, v, o, lse, dO, dq, dk, dv, workspace, cp, T_valid=None, causal=True, stream=None,
                docs=None, rope_cfg: RopeCfg | None = None):
    """dq, dk, dv with respect to the unrotated q, k, from the rotated copies that fwd_rope_save stored."""
    B, H, T, d = q_rot.shape
    H_kv = _kv_heads(q_rot, k_rot, v, dk, dv)
    cpattn_bwd_rotated(_ptr(q_rot), _ptr(k_rot), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk),
                       _ptr(dv), _ptr(workspace), B, T, T if T_valid is None else T_valid, H, H_kv, d, cp,
                       int(causal), None if docs is None else _ptr(docs[0]), None if docs is None else _ptr(docs[1]),
                       rope_cfg, _dtype_code(q_rot), _stream(stream))


def shard_batch(srcs, dsts, cp, rope=None, stream=None, cfg: RopeCfg | None = None, inverse=False):
    """HeadTail shard (inverse: unshard) of several [B, H_i, T, d] tensors in one launch;
    rope[i] rotates tensor i (R in, R^T out)."""
    B, _, T, d = srcs[0].shape
    heads = [t.shape[1] for t in srcs]
    for a, b_ in zip(srcs, dsts):
        if tuple(a.shape) != tuple(b_.shape) or a.shape[0] != B or a.shape[2] != T or a.shape[3] != d:
            raise CpattnError(ERR_SHAPE, "batched tensors must share B, T and d, and dst the shape of src")
    rope = [0] * len(srcs) if rope is None else [int(bool(r)) for r in rope]
    fn = cpattn_unshard_batch if inverse else cpattn_shard_batch
    fn([_ptr(t) for t in srcs], [_ptr(t) for t in dsts], heads, rope, B, T, d, cp, cfg, _dtype_code(srcs[0]),
       _stream(stream))


def merge(o_parts, lse_parts, o, lse, stream=None):
    B, H, T, d = o.shape
    cpattn_merge([_ptr(x) for x in o_parts], [_ptr(x) for x in lse_parts], _ptr(o), _ptr(lse),
                 B, H, T, d, _dtype_code(o), _stream(stream))
