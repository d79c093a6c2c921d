"""Host-side checks of the C-ABI library: it loads, exports every symbol its
header declares, and validates arguments without touching a GPU."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from context_causal_attention_headtail_gb300 import cpattn
from oracle import headtail as HT

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(cpattn.LIB_PATH):
        from context_causal_attention_headtail_gb300 import build
        build.build_library()
    return cpattn.lib()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "cpattn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpattn_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(cpattn.EXPORTS) == names
    assert "sm_103a" in cpattn.cpattn_version()


def test_shard_index_host_only(lib):
    for T, cp in [(8, 2), (48, 3), (4096, 4), (12296, 4)]:
        assert cpattn.cpattn_shard_index(T, cp) == HT.shard_index(T, cp).tolist()
    with pytest.raises(cpattn.CpattnError) as e:
        cpattn.cpattn_shard_index(10, 2)
    assert e.value.status == cpattn.ERR_SHAPE


# Fake, aligned, non-null addresses: validation must reject before any device access.
P = [0x100000 * (i + 1) for i in range(10)]


@pytest.mark.parametrize("args,status", [
    (dict(T=1000, cp=3), cpattn.ERR_SHAPE),          # T % (2 cp) != 0
    (dict(d=96), cpattn.ERR_SHAPE),                  # unsupported head dim
    (dict(T_valid=0), cpattn.ERR_SHAPE),
    (dict(T_valid=1025), cpattn.ERR_SHAPE),
    (dict(causal=2), cpattn.ERR_ARG),
    (dict(dt=5), cpattn.ERR_DTYPE),
    (dict(misalign=True), cpattn.ERR_ALIGN),
    (dict(null=True), cpattn.ERR_ARG),
    (dict(B=0), cpattn.ERR_SHAPE),
])
def test_fwd_validation(lib, args, status):
    a = dict(B=1, T=1024, T_valid=1024, H=2, d=128, cp=2, causal=1, rope=1, dt=cpattn.BF16)
    a.update({k: v for k, v in args.items() if k in a})
    ptrs = list(P[:5])
    if args.get("misalign"):
        ptrs[1] += 8
    if args.get("null"):
        ptrs[2] = None
    st = lib.cpattn_fwd(*ptrs, a["B"], a["T"], a["T_valid"], a["H"], a["d"], a["cp"], a["causal"],
                        a["rope"], a["dt"], None)
    assert st == status
    assert cpattn.cpattn_last_error() != ""


def test_rope_save_and_rotated_validation(lib):
    st = lib.cpattn_fwd_rope_save(*P[:5], None, P[6], 1, 1024, 1024, 2, 2, 128, 2, 1, None, None, None,
                                  cpattn.BF16, None)
    assert st == cpattn.ERR_ARG
    st = lib.cpattn_fwd_rope_save(*P[:5], P[0], P[6], 1, 1024, 1024, 2, 2, 128, 2, 1, None, None, None,
                                  cpattn.BF16, None)            # q_rot aliases q
    assert st == cpattn.ERR_ARG and "overlap" in cpattn.cpattn_last_error()
    st = lib.cpattn_fwd_rope_save(*P[:7], 1, 1024, 1024, 2, 2, 96, 2, 1, None, None, None, cpattn.BF16, None)
    assert st == cpattn.ERR_SHAPE
    st = lib.cpattn_bwd_rotated(*P, 1, 1024, 1024, 2, 2, 128, 2, 1, P[0], None, None, cpattn.BF16, None)
    assert st == cpattn.ERR_ARG and "document" in cpattn.cpattn_last_error()
    st = lib.cpattn_bwd_rotated(*P, 1, 1000, 1000, 2, 2, 128, 3, 1, None, None, None, cpattn.BF16, None)
    assert st == cpattn.ERR_SHAPE


def test_shard_batch_validation(lib):
    def call(src, dst, heads, rope, n=None, d=128, T=1024, cp=2):
        n = len(src) if n is None else n
        k = max(len(src), 1)
        return lib.cpattn_shard_batch((ctypes.c_void_p * k)(*src), (ctypes.c_void_p * k)(*dst),
                                      (ctypes.c_int * k)(*heads), (ctypes.c_int * k)(*rope), n, 1, T, d, cp,
                                      None, cpattn.BF16, None)
    assert call(P[:2], P[2:4], [2, 2], [1, 0], n=0) == cpattn.ERR_ARG
    assert call(P[:2], P[2:4], [2, 2], [1, 0], n=9) == cpattn.ERR_ARG
    assert call(P[:2], P[2:4], [2, 2], [2, 0]) == cpattn.ERR_ARG                       # rope flag
    assert call(P[:2], [P[2], P[1]], [2, 2], [1, 0]) == cpattn.ERR_ARG                 # dst 1 is src 1
    assert "overlaps" in cpattn.cpattn_last_error()
    assert call(P[:2], P[2:4], [2, 2], [1, 0], d=96) == cpattn.ERR_SHAPE
    assert call(P[:2], P[2:4], [2, 2], [1, 0], T=1000, cp=3) == cpattn.ERR_SHAPE
    assert call(P[:2], [P[2] + 8, P[3]], [2, 2], [1, 0]) == cpattn.ERR_ALIGN


def test_wait_probe_limit_is_validated(lib):
    for bad in (0, 999, 10 ** 9 + 1):
        assert lib.cpattn_check_wait_timeout(bad, None) == cpattn.ERR_ARG
        assert "limit_ns" in cpattn.cpattn_last_error()


def test_bwd_and_merge_validation(lib):
    ws = cpattn.cpattn_bwd_workspace_bytes(2, 4096, 12, 64)
    assert ws >= 2 * 4096 * 12 * 4 and ws % 256 == 0
    st = lib.cpattn_bwd(*P, 1, 1000, 1000, 2, 128, 3, 1, 1, cpattn.BF16, None)
    assert st == cpattn.ERR_SHAPE
    # gradient output aliasing an input is rejected
    st = lib.cpattn_bwd(*(P[:6] + [P[0]] + P[7:]), 1, 1024, 1024, 2, 128, 2, 1, 1, cpattn.BF16, None)
    assert st == cpattn.ERR_ARG
    arr = (ctypes.c_void_p * 17)(*([P[0]] * 17))
    st = lib.cpattn_merge(arr, arr, 17, P[1], P[2], 1, 1, 8, 64, cpattn.F32, None)
    assert st == cpattn.ERR_ARG
    st = lib.cpattn_shard(P[0], P[0] + 8, 1, 1, 8, 64, 2, cpattn.BF16, None)
    assert st == cpattn.ERR_ALIGN
    st = lib.cpattn_shard(P[0], P[0] + 16, 1, 1, 8, 64, 2, cpattn.BF16, None)
    assert st == cpattn.ERR_ARG                    # overlapping src and dst


@pytest.mark.parametrize("H,H_kv,status", [(8, 3, cpattn.ERR_SHAPE), (4, 0, cpattn.ERR_SHAPE),
                                           (2, 4, cpattn.ERR_SHAPE)])
def test_gqa_head_counts_are_validated(lib, H, H_kv, status):
    st = lib.cpattn_fwd_gqa(*P[:5], 1, 1024, 1024, H, H_kv, 128, 2, 1, 1, cpattn.BF16, None)
    assert st == status and "H_kv" in cpattn.cpattn_last_error()
    st = lib.cpattn_bwd_gqa(*P, 1, 1024, 1024, H, H_kv, 128, 2, 1, 1, cpattn.BF16, None)
    assert st == status


def test_gqa_overlap_uses_kv_sizes(lib):
    # k is [1,1,1024,128] bf16 (256 KiB): a dk starting inside it is rejected
    kv_bytes = 1024 * 128 * 2
    base = 0x40000000
    q, k, v, o, lse, do, dq, dv, ws = (base + i * 0x1000000 for i in range(9))
    st = lib.cpattn_bwd_gqa(q, k, v, o, lse, do, dq, k + kv_bytes // 2, dv, ws, 1, 1024, 1024, 4, 1,
                            128, 2, 1, 1, cpattn.BF16, None)
    assert st == cpattn.ERR_ARG


@pytest.mark.parametrize("kw", [dict(base=1.0), dict(factor=0.5), dict(factor=2.0),
                                dict(factor=2.0, original_max_position=4096, beta_fast=1.0,
                                     beta_slow=32.0),
                                dict(factor=float("nan"))])
def test_rope_cfg_is_validated(lib, kw):
    args = dict(factor=1.0, original_max_position=0)
    args.update(kw)
    cfg = cpattn.RopeCfg(**args)
    for fn in (lib.cpattn_shard_rope_cfg, lib.cpattn_unshard_rope_cfg):
        st = fn(P[0], P[1], 1, 1, 1024, 128, 2, cpattn.BF16, ctypes.byref(cfg), None)
        assert st == cpattn.ERR_ARG
    assert lib.cpattn_shard_rope_cfg(P[0], P[1], 1, 1, 1024, 128, 2, cpattn.BF16, None, None) == cpattn.ERR_ARG
    # the in-kernel RoPE entry points validate the same configuration, and need one
    for c in (ctypes.byref(cfg), None):
        assert lib.cpattn_fwd_rope_cfg(*P[:5], 1, 1024, 1024, 2, 2, 128, 2, 1, c, cpattn.BF16, None) == cpattn.ERR_ARG
        assert lib.cpattn_bwd_rope_cfg(*P, 1, 1024, 1024, 2, 2, 128, 2, 1, c, cpattn.BF16, None) == cpattn.ERR_ARG


def test_rope_cfg_layout_matches_header():
    # double, double, int (+4 bytes padding), double, double, double
    assert ctypes.sizeof(cpattn.RopeCfg) == 48
    assert cpattn.RopeCfg.beta_fast.offset == 24 and cpattn.RopeCfg.attention_factor.offset == 40


def test_varlen_and_doc_bounds_validation(lib):
    assert lib.cpattn_doc_bounds(None, 4, 64, P[1], P[2], None) == cpattn.ERR_ARG
    assert lib.cpattn_doc_bounds(P[0], 0, 64, P[1], P[2], None) == cpattn.ERR_SHAPE
    assert lib.cpattn_doc_bounds(P[0], 4, 64, P[1] + 4, P[2], None) == cpattn.ERR_ALIGN
    assert lib.cpattn_doc_bounds(P[0], 4, 64, P[1], P[1] + 128, None) == cpattn.ERR_ARG   # lo, hi overlap
    st = lib.cpattn_fwd_varlen(*P[:5], 1, 1024, 1024, 2, 2, 128, 2, 1, None, P[6], cpattn.BF16, None)
    assert st == cpattn.ERR_ARG
    st = lib.cpattn_bwd_varlen(*P, 1, 1024, 1024, 2, 2, 128, 2, 1, P[0], None, cpattn.BF16, None)
    assert st == cpattn.ERR_ARG
    st = lib.cpattn_fwd_varlen(*P[:5], 1, 1000, 1000, 2, 2, 128, 3, 1, P[5], P[6], cpattn.BF16, None)
    assert st == cpattn.ERR_SHAPE


def test_ulysses_binding_rotates_only_when_asked(monkeypatch):
    """The wrapper picks the rotating entry point from rope alone; a YaRN cfg
    handed along for V / dO must not rotate them."""
    import torch
    calls = []
    monkeypatch.setattr(cpattn, "_ptr", lambda t: 16)
    monkeypatch.setattr(cpattn, "_stream", lambda s: None)
    monkeypatch.setattr(cpattn, "cpattn_ulysses_a2a", lambda *a, **k: calls.append("plain"))
    monkeypatch.setattr(cpattn, "cpattn_ulysses_a2a_rope", lambda *a, **k: calls.append("rope"))
    x = torch.zeros(2, 4, 8, 64, dtype=torch.bfloat16)
    y = torch.zeros(2, 2, 16, 64, dtype=torch.bfloat16)
    cfg = cpattn.RopeCfg(factor=2.0, original_max_position=8)
    cpattn.ulysses_a2a(x, y, 2, rope=False, cfg=cfg)
    cpattn.ulysses_a2a(x, y, 2, rope=True, cfg=cfg)
    cpattn.ulysses_a2a(y, x, 2, inverse=True, rope=False, cfg=cfg)
    assert calls == ["plain", "rope", "plain"]
