"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Small cases are compared element by element over the whole output; they span
several 128-row tiles per chunk, ragged last tiles (c not a multiple of 128,
c < 128), cp in {1, 2, 3, 4}, d in {64, 128}, non-causal attention and tail
padding. The five benchmark workloads run at full size and are compared on
sampled rows (O, LSE, dQ over several heads; dK, dV over one head, which needs
that head's full forward in the oracle), plus properties that hold at any size
(pad-row gradients exactly zero, bitwise determinism).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from context_causal_attention_headtail_gb300 import cpattn
from context_causal_attention_headtail_gb300.synth import SEEDS, WORKLOADS, make_inputs, make_workload
from oracle import attention as A
from oracle import headtail as HT

from harness import (TOL, compare, oracle_docs, oracle_rope, run_gpu, run_gpu_ulysses,
                     sample_rows, to_seq_shards)
from oracle import ulysses as U

pytestmark = pytest.mark.gpu


def _oracle_full(w, inp):
    q, k, v, do = (inp[n].double().numpy() for n in ("q", "k", "v", "do"))
    O, L = A.forward(q, k, v, w.causal, w.T_valid, oracle_rope(w), docs=oracle_docs(w))
    dq, dk, dv = A.backward(q, k, v, O, L, do, w.causal, w.T_valid, oracle_rope(w), docs=oracle_docs(w))
    return {"o": O, "lse": L, "dq": dq, "dk": dk, "dv": dv}


def _check_full(w, got, want):
    tol = TOL[w.dtype]
    reps = [compare("o", got["o"], want["o"], tol["o"], tol["cos"]),
            compare("lse", got["lse"], want["lse"], tol["lse"])]
    for g in ("dq", "dk", "dv"):
        reps.append(compare(g, got[g], want[g], tol["grad"], tol["cos"]))
    return reps


# ------------------------------------------------------------- shard ----

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,H,T,d,cp", [(1, 2, 8, 64, 2), (2, 3, 24, 128, 3), (1, 1, 512, 64, 1),
                                        (2, 2, 12296, 128, 4)])
def test_shard_unshard_bit_exact(dtype, B, H, T, d, cp):
    x = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(T + cp)).to(dtype)
    xs = x.cuda()
    ys, zs = torch.empty_like(xs), torch.empty_like(xs)
    cpattn.shard(xs, ys, cp)
    cpattn.unshard(ys, zs, cp)
    torch.cuda.synchronize()
    want = torch.from_numpy(HT.shard(x.float().numpy(), cp)).to(dtype)
    assert torch.equal(ys.cpu(), want)
    assert torch.equal(zs.cpu(), x)


@pytest.mark.parametrize("dtype,B,H,H_kv,T,d,cp,yarn", [(torch.bfloat16, 1, 4, 2, 1200, 128, 2, False),
                                                         (torch.float32, 2, 2, 1, 768, 64, 3, True),
                                                         (torch.bfloat16, 1, 16, 16, 32768, 128, 2, False)])
def test_shard_batch_equals_single_calls(dtype, B, H, H_kv, T, d, cp, yarn):
    """cpattn_shard_batch / cpattn_unshard_batch (q, k rotated, v, dO plain; GQA
    heads) give bit for bit what the single-tensor calls give."""
    g = torch.Generator().manual_seed(T + H)
    shapes = [(B, H, T, d), (B, H_kv, T, d), (B, H_kv, T, d), (B, H, T, d)]
    xs = [(torch.randn(sh, generator=g) * 0.5).to(dtype).cuda() for sh in shapes]
    rope = [1, 1, 0, 0]
    cfg = cpattn.RopeCfg(factor=2.0, original_max_position=T // 2) if yarn else None
    for inverse in (False, True):
        got = [torch.empty_like(x) for x in xs]
        cpattn.shard_batch(xs, got, cp, rope=rope, cfg=cfg, inverse=inverse)
        for x, y, r in zip(xs, got, rope):
            want = torch.empty_like(x)
            if r:
                (cpattn.unshard_rope if inverse else cpattn.shard_rope)(x, want, cp, cfg=cfg)
            else:
                (cpattn.unshard if inverse else cpattn.shard)(x, want, cp)
            torch.cuda.synchronize()
            assert torch.equal(y, want)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,H,T,d,cp", [(1, 2, 8, 64, 2), (2, 1, 1200, 128, 2), (1, 2, 32768, 128, 2),
                                        (1, 1, 12296, 64, 4)])
def test_shard_rope_against_oracle(dtype, B, H, T, d, cp):
    x = (torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(T + d)) * 0.5).to(dtype)
    xs = x.cuda()
    ys, zs = torch.empty_like(xs), torch.empty_like(xs)
    cpattn.shard_rope(xs, ys, cp)
    cpattn.unshard_rope(ys, zs, cp)
    torch.cuda.synchronize()
    xd = x.double().numpy()
    want = HT.shard(A.rope(xd, np.arange(T)), cp)
    # Bounds: the GPU rotates the same stored values with angles good to ~1e-6
    # rad and rounds once to the storage type (unit roundoff u); the round trip
    # adds a second rounding, which R^T spreads over each (i, i + d/2) pair.
    u = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -24
    pair = np.sqrt(xd[..., : d // 2] ** 2 + xd[..., d // 2:] ** 2)
    pair = np.concatenate([pair, pair], axis=-1)
    err = np.abs(ys.double().cpu().numpy() - want)
    bound = u * np.abs(want) + 4e-6 * HT.shard(pair, cp) + 1e-7
    worst = float((err / bound).max())
    assert worst <= 1.0, f"shard_rope: worst error/bound {worst:.3f}, max err {err.max():.3e}"
    back = zs.double().cpu().numpy()
    err = np.abs(back - xd)
    worst = float((err / (3 * u * pair + 8e-6 * pair + 1e-7)).max())
    assert worst <= 1.0, f"round trip: worst error/bound {worst:.3f}, max err {err.max():.3e}"


@pytest.mark.parametrize("dtype,B,H,T,d,cp,factor,L", [
    (torch.bfloat16, 1, 2, 32768, 128, 2, 2.0, 16384),     # the 32k extension run
    (torch.float32, 1, 1, 12296, 64, 4, 8.0, 2048),
    (torch.bfloat16, 2, 1, 1200, 128, 2, 4.0, 300),
])
def test_shard_rope_yarn_against_oracle(dtype, B, H, T, d, cp, factor, L):
    x = (torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(T + 7)) * 0.5).to(dtype)
    xs = x.cuda()
    ys, zs = torch.empty_like(xs), torch.empty_like(xs)
    cfg = cpattn.RopeCfg(factor=factor, original_max_position=L)
    cpattn.shard_rope(xs, ys, cp, cfg=cfg)
    cpattn.unshard_rope(ys, zs, cp, cfg=cfg)
    torch.cuda.synchronize()
    spec = A.RopeSpec(factor=factor, original_max_position=L)
    m = spec.mscale()
    xd = x.double().numpy()
    want = HT.shard(A.rope(xd, np.arange(T), spec), cp)
    # as for the standard rotation, with every magnitude scaled by m (m^2 after
    # the round trip); m is itself rounded to fp32 (relative 2^-24)
    u = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -24
    pair = np.sqrt(xd[..., : d // 2] ** 2 + xd[..., d // 2:] ** 2)
    pair = np.concatenate([pair, pair], axis=-1)
    err = np.abs(ys.double().cpu().numpy() - want)
    bound = u * np.abs(want) + 5e-6 * m * HT.shard(pair, cp) + 1e-7
    worst = float((err / bound).max())
    assert worst <= 1.0, f"shard_rope yarn: worst error/bound {worst:.3f}, max err {err.max():.3e}"
    back = zs.double().cpu().numpy()
    err = np.abs(back - m * m * xd)
    worst = float((err / (3 * u * m * m * pair + 1e-5 * m * m * pair + 1e-7)).max())
    assert worst <= 1.0, f"round trip: worst error/bound {worst:.3f}, max err {err.max():.3e}"


def test_shard_rope_cfg_factor_one_is_plain_rope():
    x = (torch.randn(1, 2, 4096, 128, generator=torch.Generator().manual_seed(3)) * 0.5).to(torch.bfloat16).cuda()
    a, b = torch.empty_like(x), torch.empty_like(x)
    cpattn.shard_rope(x, a, 2)
    cpattn.shard_rope(x, b, 2, cfg=cpattn.RopeCfg(factor=1.0))
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    cpattn.unshard_rope(a, b, 2)
    c = torch.empty_like(x)
    cpattn.unshard_rope(a, c, 2, cfg=cpattn.RopeCfg(factor=1.0))
    torch.cuda.synchronize()
    assert torch.equal(b, c)


@pytest.mark.parametrize("cu,T", [([0, 5, 6, 23, 40, 61], 64), ([0, 64], 64), ([0, 0, 3, 3, 10], 16),
                                  ([0, 1000, 1000, 4097, 8000, 12289], 12296)])
def test_doc_bounds_against_oracle(cu, T):
    cu_d = torch.tensor(cu, dtype=torch.int32, device="cuda")
    lo = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    hi = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    cpattn.doc_bounds(cu_d, T, lo, hi)
    cpattn.cpattn_sync_status(None)
    doc = A.document_of(np.arange(T), np.array(cu))
    cu_np = np.array(cu)
    want_lo = np.where(doc >= 0, cu_np[np.maximum(doc, 0)], cu[-1])
    want_hi = np.where(doc >= 0, cu_np[np.maximum(doc, 0) + 1], cu[-1])
    assert np.array_equal(lo.cpu().numpy(), want_lo)
    assert np.array_equal(hi.cpu().numpy(), want_hi)


def test_doc_bounds_rejects_a_bad_list():
    cu_d = torch.tensor([0, 9, 4, 16], dtype=torch.int32, device="cuda")    # not non-decreasing
    lo = torch.empty(16, dtype=torch.int32, device="cuda")
    hi = torch.empty(16, dtype=torch.int32, device="cuda")
    cpattn.doc_bounds(cu_d, 16, lo, hi)
    with pytest.raises(cpattn.CpattnError) as e:
        cpattn.cpattn_sync_status(None)
    assert e.value.status == cpattn.ERR_ARG
    cpattn.cpattn_sync_status(None)     # the flag is cleared once reported
    assert int(lo.min()) >= 0 and int(hi.max()) <= 16


def test_varlen_long_schedule_sampled():
    """Packed documents on a schedule past the tile table (2560 entries per CTA),
    which the one-tile kernels run: sampled rows of O, LSE and dQ against the
    oracle, dK and dV through per-document identities of the exact gradient."""
    w = make_workload("long_varlen", B=1, T=2 * 256 * 513, T_valid=2 * 256 * 513 - 3, H=2, H_kv=1, d=64,
                      cp=256, rope=False, doc_len=(100, 5000), doc_seed=8)
    assert 2 * w.cp * -(-w.chunk // 128) > 2048
    inp = make_inputs(w, seed=1)
    got = run_gpu(w, inp)
    for g in ("o", "dq", "dk", "dv"):
        assert torch.isfinite(got[g]).all(), g
    cu = w.cu_seqlens()
    tol = TOL[w.dtype]
    rng = np.random.default_rng(3)
    rows = np.array(sorted(set(rng.integers(0, w.T_valid, size=24).tolist()) |
                           {int(x) for x in cu[1:4]} | {int(cu[1]) - 1, w.T_valid - 1}))
    q, k, v, do = (inp[n] for n in ("q", "k", "v", "do"))
    for h in range(w.H):
        o_r, l_r = A.forward_rows(q, k, v, 0, h, rows, w.causal, w.T_valid, False, docs=oracle_docs(w))
        compare(f"o[{h}]", got["o"][0, h, rows], o_r, tol["o"], tol["cos"])
        compare(f"lse[{h}]", got["lse"][0, h, rows], l_r, tol["lse"])
        dq_r = A.backward_dq_rows(q, k, v, do, 0, h, rows, w.causal, w.T_valid, False, docs=oracle_docs(w))
        compare(f"dq[{h}]", got["dq"][0, h, rows], dq_r, tol["grad"], tol["cos"])
    # dK, dV through identities of the exact gradient inside each document:
    # rows of dS sum to zero and rows of P to one over the document's keys, so
    # over a document sum dK = 0 and sum dV = the sum of dO over its query rows
    # (both query heads read K/V head 0).
    dk = got["dk"][0, 0].double().numpy()
    dv = got["dv"][0, 0].double().numpy()
    dO = do[0].double().numpy().sum(axis=0)
    for i in range(min(6, len(cu) - 1)):
        lo, hi = int(cu[i]), min(int(cu[i + 1]), w.T_valid)
        if hi - lo < 2:
            continue
        assert np.linalg.norm(dk[lo:hi].sum(0)) <= 5e-2 * np.sqrt((dk[lo:hi] ** 2).sum()), ("sum dK", i)
        assert (np.linalg.norm(dv[lo:hi].sum(0) - dO[lo:hi].sum(0)) <=
                5e-2 * np.sqrt((dv[lo:hi] ** 2).sum())), ("sum dV", i)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,H,T,d,P", [(1, 4, 8, 64, 2), (2, 6, 24, 128, 3), (1, 16, 32768, 128, 2),
                                       (2, 8, 4096, 64, 4), (1, 3, 300, 128, 1)])
def test_ulysses_a2a_bit_exact(dtype, B, H, T, d, P):
    x = torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(T + P)).to(dtype)
    xs = to_seq_shards(x, P).cuda()
    head = torch.empty((B * P, H // P, T, d), dtype=dtype, device="cuda")
    back = torch.empty_like(xs)
    cpattn.ulysses_a2a(xs, head, P)
    cpattn.ulysses_a2a(head, back, P, inverse=True)
    torch.cuda.synchronize()
    want = U.all_to_all(U.seq_shards(x.float().numpy(), P))       # [P, B, Hl, T, d]
    assert torch.equal(head.cpu(), torch.from_numpy(want.reshape(B * P, H // P, T, d)).to(dtype))
    assert torch.equal(back.cpu(), xs.cpu())


@pytest.mark.parametrize("dtype,B,H,T,d,P,yarn", [(torch.bfloat16, 1, 4, 32768, 128, 2, False),
                                                  (torch.float32, 2, 6, 1200, 64, 3, True)])
def test_ulysses_a2a_rope_against_oracle(dtype, B, H, T, d, P, yarn):
    x = (torch.randn(B, H, T, d, generator=torch.Generator().manual_seed(T)) * 0.5).to(dtype)
    spec = A.RopeSpec(factor=4.0, original_max_position=T // 4) if yarn else A.STANDARD_ROPE
    cfg = cpattn.RopeCfg(factor=4.0, original_max_position=T // 4) if yarn else None
    xs = to_seq_shards(x, P).cuda()
    head = torch.empty((B * P, H // P, T, d), dtype=dtype, device="cuda")
    back = torch.empty_like(xs)
    cpattn.ulysses_a2a(xs, head, P, rope=True, cfg=cfg)
    cpattn.ulysses_a2a(head, back, P, inverse=True, rope=True, cfg=cfg)
    torch.cuda.synchronize()
    xd = x.double().numpy()
    m = spec.mscale()
    want = U.all_to_all(U.seq_shards(A.rope(xd, np.arange(T), spec), P)).reshape(B * P, H // P, T, d)
    pair = np.sqrt(xd[..., : d // 2] ** 2 + xd[..., d // 2:] ** 2)
    pair = np.concatenate([pair, pair], axis=-1)
    u = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -24
    pair_h = U.all_to_all(U.seq_shards(pair, P)).reshape(want.shape)
    err = np.abs(head.double().cpu().numpy() - want)
    worst = float((err / (u * np.abs(want) + 5e-6 * m * pair_h + 1e-7)).max())
    assert worst <= 1.0, f"a2a+rope: worst error/bound {worst:.3f}"
    err = np.abs(back.double().cpu().numpy() - m * m * to_seq_shards(x.double(), P).numpy())
    pair_s = to_seq_shards(torch.from_numpy(pair), P).numpy()
    worst = float((err / (3 * u * m * m * pair_s + 1e-5 * m * m * pair_s + 1e-7)).max())
    assert worst <= 1.0, f"round trip: worst error/bound {worst:.3f}"


@pytest.mark.parametrize("dtype,rope", [(torch.bfloat16, False), (torch.float32, True), (torch.bfloat16, True)])
@pytest.mark.parametrize("B,H,T,d,P", [(1, 2, 1024, 128, 4), (2, 1, 512, 64, 4), (1, 2, 768, 128, 8)])
def test_ulysses_kv_replication_against_oracle(dtype, rope, B, H, T, d, P):
    """Forward: each K/V head to its P/H ranks (bit-exact without RoPE). Inverse:
    the replicas summed (bit-exact for bf16: the fp32 sum of a few bf16 values
    is exact, then one rounding, as the oracle's sum rounded once)."""
    g = torch.Generator().manual_seed(T + H + P)
    x = (torch.randn(B, H, T, d, generator=g) * 0.5).to(dtype)
    xs = to_seq_shards(x, P).cuda()
    head = torch.empty((B * P, 1, T, d), dtype=dtype, device="cuda")
    cpattn.ulysses_a2a(xs, head, P, rope=rope)
    y = (torch.randn(B * P, 1, T, d, generator=g) * 0.5).to(dtype)
    back = torch.empty_like(xs)
    cpattn.ulysses_a2a(y.cuda(), back, P, inverse=True, rope=rope)
    torch.cuda.synchronize()
    xd = x.double().numpy()
    if rope:
        xd = A.rope(xd, np.arange(T))
    want = U.all_to_all_kv(U.seq_shards(xd, P)).reshape(B * P, 1, T, d)
    yd = y.double().numpy().reshape(P, B, 1, T, d)
    back_want = U.all_to_all_kv_adjoint(yd, H)          # [P, B, H, T/P, d]
    if rope:   # (R^T) of the sum, at the natural positions of each sequence shard
        Tl = T // P
        for r in range(P):
            back_want[r] = A.rope_transpose(back_want[r], np.arange(r * Tl, (r + 1) * Tl))
    back_want = back_want.reshape(B * P, H, T // P, d)
    if not rope:
        assert torch.equal(head.cpu(), torch.from_numpy(want).to(dtype))
        if dtype == torch.bfloat16:
            assert torch.equal(back.cpu(), torch.from_numpy(back_want).to(dtype))
    u = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -23
    compare("a2a_kv", head.cpu().double(), want, 4 * u * np.abs(want).max() + 1e-5)
    compare("a2a_kv_adjoint", back.cpu().double(), back_want, 4 * u * np.abs(back_want).max() + 1e-5)


ULYSSES_SMALL = [
    make_workload("ulysses2_rope", B=1, T=1024, T_valid=1021, H=4, d=128, cp=1, rope=True, ulysses=2),
    make_workload("ulysses4_gqa_d64", B=2, T=768, H=8, H_kv=4, d=64, cp=1, rope=True, ulysses=4),
    make_workload("ulysses2_f32", B=1, T=256, H=2, d=64, cp=1, rope=True, dtype="f32", qkv_std=1.0,
                  ulysses=2),
    make_workload("ulysses2_yarn_noncausal", B=1, T=640, H=4, d=128, cp=1, causal=False, rope=True,
                  yarn_factor=2.0, yarn_original=320, ulysses=2),
    # fewer K/V heads than ranks: K/V replicated to P / H_kv ranks, gradients summed
    make_workload("ulysses4_kv2_rep", B=1, T=1024, H=8, H_kv=2, d=128, cp=1, rope=True, ulysses=4),
    make_workload("ulysses4_mqa_d64", B=2, T=512, H=4, H_kv=1, d=64, cp=1, rope=True, ulysses=4),
]


@pytest.mark.parametrize("w", ULYSSES_SMALL, ids=lambda w: w.name)
def test_ulysses_path_full(w):
    inp = make_inputs(w, seed=11 + w.T)
    got = run_gpu_ulysses(w, inp)
    _check_full(w, got, _oracle_full(w, inp))


def test_ulysses_32k_sampled():
    w = WORKLOADS["ulysses_32k"]
    inp = make_inputs(w, SEEDS["ulysses_32k"])
    got = run_gpu_ulysses(w, inp)
    for g in ("o", "lse", "dq", "dk", "dv"):
        assert torch.isfinite(got[g]).all(), g
    _sampled_check(w, inp, got, [(0, 0), (0, 7), (0, 15)], kv_heads=[(0, 9), (0, 2)])


def test_shard_index_matches_oracle():
    for T, cp in [(8, 2), (24, 3), (32768, 2), (12296, 4)]:
        assert cpattn.cpattn_shard_index(T, cp) == HT.shard_index(T, cp).tolist()


# -------------------------------------------------- small, full compare ----

ROPE_MODES = ["kernel", "shard", "save"]

SMALL_F32 = [
    WORKLOADS["tiny_fp32"],
    make_workload("f32_rope_pad", B=1, T=384, T_valid=381, H=2, d=128, cp=3, rope=True, dtype="f32",
                  qkv_std=1.0),
    make_workload("f32_noncausal", B=2, T=256, H=1, d=64, cp=2, causal=False, rope=True, dtype="f32",
                  qkv_std=1.0),
]

SMALL_GQA_F32 = [
    make_workload("f32_gqa_rope", B=1, T=256, T_valid=253, H=4, H_kv=2, d=64, cp=2, rope=True,
                  dtype="f32", qkv_std=1.0),
    make_workload("f32_yarn", B=1, T=384, T_valid=381, H=2, d=128, cp=3, rope=True, dtype="f32",
                  qkv_std=1.0, yarn_factor=4.0, yarn_original=96),
    make_workload("f32_varlen", B=1, T=384, T_valid=379, H=2, H_kv=1, d=64, cp=2, rope=True,
                  dtype="f32", qkv_std=1.0, doc_len=(1, 120), doc_seed=1),
]

SMALL_BF16 = [
    make_workload("two_tiles_rope", B=1, T=1024, H=2, d=128, cp=2, rope=True),
    make_workload("ragged_d64_pad", B=2, T=800, T_valid=797, H=1, d=64, cp=2, rope=False),
    make_workload("cp1", B=1, T=512, H=1, d=128, cp=1, rope=True),
    make_workload("noncausal_cp3", B=1, T=768, H=2, d=64, cp=3, causal=False, rope=True),
    make_workload("small_chunks_cp4", B=1, T=512, T_valid=509, H=1, d=128, cp=4, rope=True),
    make_workload("ragged_c300", B=1, T=1200, T_valid=1195, H=2, d=128, cp=2, rope=True),
    make_workload("noncausal_pad_d128", B=1, T=640, T_valid=600, H=1, d=128, cp=2, causal=False,
                  rope=False),
    # 15 (b, h) problems: the launch order's last head group is partial in every kernel
    # (groups of 4 heads in the forward, of 2 K/V heads in dK/dV)
    make_workload("heads15_pad", B=3, T=768, T_valid=765, H=5, d=128, cp=2, rope=True),
    # grouped K/V heads: GQA with RoPE and padding, MQA, non-causal GQA, ragged chunks
    make_workload("gqa4x2_rope_pad", B=1, T=1024, T_valid=1021, H=4, H_kv=2, d=128, cp=2, rope=True),
    make_workload("mqa_d64_cp3", B=2, T=768, H=3, H_kv=1, d=64, cp=3, rope=False),
    make_workload("gqa6x3_noncausal", B=1, T=512, H=6, H_kv=3, d=128, cp=2, causal=False, rope=True),
    make_workload("gqa8x2_ragged", B=1, T=1200, T_valid=1195, H=8, H_kv=2, d=64, cp=2, rope=True),
    # YaRN RoPE (trained length a quarter / half of T, so the extension is used)
    make_workload("yarn4_pad", B=1, T=1024, T_valid=1019, H=2, d=128, cp=2, rope=True,
                  yarn_factor=4.0, yarn_original=256),
    make_workload("yarn2_gqa_d64", B=2, T=768, H=4, H_kv=2, d=64, cp=3, rope=True,
                  yarn_factor=2.0, yarn_original=384),
    # packed documents: short and long ones, boundaries inside tiles and chunks,
    # one-token documents, padding, GQA, non-causal, ragged chunks
    make_workload("varlen_short_docs", B=1, T=1024, T_valid=1019, H=2, d=128, cp=2, rope=True,
                  doc_len=(1, 90), doc_seed=2),
    make_workload("varlen_long_docs_gqa", B=2, T=2048, H=4, H_kv=2, d=128, cp=2, rope=True,
                  doc_len=(200, 900), doc_seed=3),
    make_workload("varlen_noncausal_d64", B=1, T=768, T_valid=760, H=2, d=64, cp=3, causal=False,
                  rope=False, doc_len=(30, 300), doc_seed=4),
    make_workload("varlen_ragged_c300", B=1, T=1200, T_valid=1195, H=2, d=128, cp=2, rope=True,
                  doc_len=(100, 500), doc_seed=5),
]


@pytest.mark.parametrize("mode", ROPE_MODES)
@pytest.mark.parametrize("w", SMALL_F32 + SMALL_GQA_F32, ids=lambda w: w.name)
def test_fp32_path_full(w, mode):
    if mode != "kernel" and not w.rope:
        pytest.skip("no RoPE: one path")
    if mode == "kernel" and w.packed and w.rope:
        pytest.skip("packed documents take RoPE from the shard passes or the save path")
    inp = make_inputs(w, seed=SEEDS.get(w.name, 99))
    _check_full(w, run_gpu(w, inp, rope_mode=mode), _oracle_full(w, inp))


@pytest.mark.parametrize("mode", ROPE_MODES)
@pytest.mark.parametrize("w", SMALL_BF16, ids=lambda w: w.name)
def test_bf16_path_full(w, mode):
    if mode != "kernel" and not w.rope:
        pytest.skip("no RoPE: one path")
    if mode == "kernel" and w.packed and w.rope:
        pytest.skip("packed documents take RoPE from the shard passes or the save path")
    inp = make_inputs(w, seed=7 + w.T + w.cp)
    got = run_gpu(w, inp, rope_mode=mode)
    want = _oracle_full(w, inp)
    _check_full(w, got, want)
    if w.T_valid < w.T:   # pad rows: dO = 0 there, so every gradient row is exactly zero
        for g in ("dq", "dk", "dv"):
            assert torch.count_nonzero(got[g][:, :, w.T_valid:]) == 0


@pytest.mark.parametrize("mode", ROPE_MODES)
def test_bf16_deterministic(mode):
    w = make_workload("det", B=1, T=1024, T_valid=1020, H=2, d=128, cp=2, rope=True)
    inp = make_inputs(w, seed=5)
    a, b = run_gpu(w, inp, rope_mode=mode), run_gpu(w, inp, rope_mode=mode)
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("w", [make_workload("save_gqa_yarn", B=1, T=1536, H=4, H_kv=2, d=128, cp=3, rope=True,
                                             yarn_factor=2.0, yarn_original=512),
                               make_workload("save_d64", B=2, T=1024, H=2, d=64, cp=2, rope=True)],
                         ids=lambda w: w.name)
def test_fwd_rope_save_stores_the_rotated_inputs(w):
    """cpattn_fwd_rope_save writes q_rot = m R q and k_rot = m R k at every
    sharded row (no padding here, so every key tile is read by the query tile
    at its own positions): bounded against the oracle's rotation."""
    from harness import gpu_rope_cfg
    inp = make_inputs(w, seed=21 + w.T)
    dev = torch.device("cuda:0")
    sh = {}
    for n_ in ("q", "k", "v"):
        x = inp[n_].to(dev)
        sh[n_] = torch.empty_like(x)
        cpattn.shard(x, sh[n_], w.cp)
    o = torch.empty_like(sh["q"])
    lse = torch.empty((w.B, w.H, w.T), dtype=torch.float32, device=dev)
    q_rot, k_rot = torch.full_like(sh["q"], float("nan")), torch.full_like(sh["k"], float("nan"))
    cpattn.fwd_rope_save(sh["q"], sh["k"], sh["v"], o, lse, q_rot, k_rot, w.cp, w.T_valid, w.causal,
                         docs=None, rope_cfg=gpu_rope_cfg(w))
    cpattn.cpattn_sync_status(None)
    spec = oracle_rope(w)
    spec = A.STANDARD_ROPE if spec is True else spec
    m = spec.mscale()
    for name, got in (("q", q_rot), ("k", k_rot)):
        xd = inp[name].double().numpy()
        want = HT.shard(A.rope(xd, np.arange(w.T), spec), w.cp)
        g = got.double().cpu().numpy()
        assert np.isfinite(g).all(), f"{name}_rot has rows that were not written"
        pair = np.sqrt(xd[..., : w.d // 2] ** 2 + xd[..., w.d // 2:] ** 2)
        pair = HT.shard(np.concatenate([pair, pair], axis=-1), w.cp)
        bound = 2.0 ** -8 * np.abs(want) + 1e-5 * m * pair + 1e-7
        worst = float((np.abs(g - want) / bound).max())
        assert worst <= 1.0, f"{name}_rot: worst error/bound {worst:.3f}"


# ------------------------------------------------------------- merge ----

@pytest.mark.parametrize("n,d,dtype", [(1, 64, torch.float32), (2, 128, torch.float32),
                                       (5, 128, torch.bfloat16), (16, 64, torch.float32)])
def test_merge_against_oracle(n, d, dtype):
    B, H, T = 2, 3, 257
    g = torch.Generator().manual_seed(n * 1000 + d)
    o_parts = [torch.randn(B, H, T, d, generator=g) for _ in range(n)]
    l_parts = [torch.randn(B, H, T, generator=g) * 3 for _ in range(n)]
    for i, l in enumerate(l_parts):          # empty partials, incl. rows empty in every part
        l[:, :, i::7] = -float("inf")
        o_parts[i][:, :, i::7] = 0.0
    l_parts[0][:, :, 5] = -float("inf")
    for i in range(n):
        l_parts[i][:, :, 5] = -float("inf")
        o_parts[i][:, :, 5] = 0.0
    o = torch.empty(B, H, T, d, dtype=dtype, device="cuda")
    lse = torch.empty(B, H, T, device="cuda")
    cpattn.merge([x.cuda() for x in o_parts], [x.cuda() for x in l_parts], o, lse)
    torch.cuda.synchronize()
    Ow, Lw = A.merge_many([x.double().numpy() for x in o_parts], [x.double().numpy() for x in l_parts])
    tol = 1e-5 if dtype == torch.float32 else 2e-2
    compare("merge_o", o.float().cpu(), Ow, tol)
    compare("merge_lse", lse.cpu(), Lw, 1e-5)


# ------------------------------------------------- full-size workloads ----

def _sampled_check(w, inp, got, heads, kv_heads, n_random=24):
    tol = TOL[w.dtype]
    q, k, v, do = (inp[n] for n in ("q", "k", "v", "do"))
    rows = sample_rows(w, n_random, seed=w.T)
    real = rows[rows < w.T_valid]
    for (b, h) in heads:
        o_r, l_r = A.forward_rows(q, k, v, b, h, rows, w.causal, w.T_valid, oracle_rope(w),
                                  docs=oracle_docs(w))
        compare(f"o[{b},{h}]", got["o"][b, h, rows], o_r, tol["o"], tol["cos"])
        compare(f"lse[{b},{h}]", got["lse"][b, h, rows], l_r, tol["lse"])
        dq_r = A.backward_dq_rows(q, k, v, do, b, h, real, w.causal, w.T_valid, oracle_rope(w),
                                  docs=oracle_docs(w))
        compare(f"dq[{b},{h}]", got["dq"][b, h, real], dq_r, tol["grad"], tol["cos"])
    for b, h in kv_heads:
        dk_c, dv_c = A.backward_dkdv_cols(q, k, v, do, b, h, rows, w.causal, w.T_valid, oracle_rope(w),
                                          docs=oracle_docs(w))
        compare(f"dk[{b},{h}]", got["dk"][b, h, rows], dk_c, tol["grad"], tol["cos"])
        compare(f"dv[{b},{h}]", got["dv"][b, h, rows], dv_c, tol["grad"], tol["cos"])


@pytest.mark.parametrize("name,mode", [("gpt2_small", "shard"), ("gpt2_small", "kernel"),
                                       ("long_16k", "shard"), ("long_16k", "kernel"),
                                       ("window_32k", "shard"), ("window_32k", "kernel"),
                                       ("padded_12289", "shard"), ("padded_12289", "kernel"),
                                       ("gqa_32k", "shard"), ("gqa_32k", "kernel"),
                                       ("yarn_32k", "shard"), ("yarn_32k", "kernel"),
                                       ("varlen_32k", "shard"), ("window_32k", "save"),
                                       ("gqa_32k", "save"), ("padded_12289", "save"),
                                       ("varlen_32k", "save"), ("gpt2_small", "save")])
def test_workload_full_size_sampled(name, mode):
    w = WORKLOADS[name]
    inp = make_inputs(w, SEEDS[name])
    got = run_gpu(w, inp, rope_mode=mode)
    for g in ("o", "lse", "dq", "dk", "dv"):
        assert torch.isfinite(got[g][:, :, : w.T_valid]).all(), g
    heads = [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 2)]
    _sampled_check(w, inp, got, heads, kv_heads=[(w.B - 1, w.kv_heads // 3), (0, w.kv_heads - 1)])
    if w.T_valid < w.T:
        for g in ("dq", "dk", "dv"):
            assert torch.count_nonzero(got[g][:, :, w.T_valid:]) == 0, g
        # gradient invariance: the padded run's real rows equal the unpadded oracle
        wu = make_workload("unpadded", B=w.B, T=w.T_valid, H=w.H, d=w.d, cp=1, rope=w.rope,
                           causal=w.causal, dtype=w.dtype, qkv_std=w.qkv_std)
        inp_u = {k_: t[:, :, : w.T_valid] for k_, t in inp.items()}
        rows = sample_rows(wu, 8, seed=3)
        b, h = 1, 5
        o_u, l_u = A.forward_rows(inp_u["q"], inp_u["k"], inp_u["v"], b, h, rows, True, w.T_valid, w.rope)
        compare("o_vs_unpadded", got["o"][b, h, rows], o_u, TOL["bf16"]["o"], TOL["bf16"]["cos"])
        dq_u = A.backward_dq_rows(inp_u["q"], inp_u["k"], inp_u["v"], inp_u["do"], b, h, rows, True,
                                  w.T_valid, w.rope)
        compare("dq_vs_unpadded", got["dq"][b, h, rows], dq_u, TOL["bf16"]["grad"], TOL["bf16"]["cos"])


# Schedules longer than the pipelined kernels' shared-memory tile table
# (2*cp*ceil(c/128) > 2048 entries) run on the one-tile kernels. cp=256 and
# c=513 give 2560 entries per CTA, and every chunk ends in a one-row tile.
LONG_SCHEDULE = dict(B=1, T=2 * 256 * 513, H=1, d=64, cp=256, rope=False)


def test_long_schedule_sampled_rows():
    w = make_workload("long_schedule", T_valid=LONG_SCHEDULE["T"] - 5, **LONG_SCHEDULE)
    inp = make_inputs(w, seed=77)
    got = run_gpu(w, inp)
    c = w.chunk
    kappas = [0, 1, 2, w.cp - 1, w.cp, w.cp + 1, 2 * w.cp - 2, 2 * w.cp - 1]
    rows = {0, w.T_valid - 1, w.T - 1}
    for kap in kappas:
        rows |= {kap * c, kap * c + 127, kap * c + 128, kap * c + c - 1}
    rows |= set(np.random.default_rng(5).integers(0, w.T, size=24).tolist())
    rows = np.array(sorted(rows))
    real = rows[rows < w.T_valid]
    tol = TOL[w.dtype]
    o_r, l_r = A.forward_rows(inp["q"], inp["k"], inp["v"], 0, 0, rows, w.causal, w.T_valid, w.rope)
    compare("o", got["o"][0, 0, rows], o_r, tol["o"], tol["cos"])
    compare("lse", got["lse"][0, 0, rows], l_r, tol["lse"])
    dq_r = A.backward_dq_rows(inp["q"], inp["k"], inp["v"], inp["do"], 0, 0, real, w.causal,
                              w.T_valid, w.rope)
    compare("dq", got["dq"][0, 0, real], dq_r, tol["grad"], tol["cos"])
    # dK, dV at this size through identities of the exact gradient (no RoPE):
    # each row of dS sums to zero, so sum_k dK_k = 0; each row of P sums to
    # one, so sum_k dV_k = sum_i dO_i over the real query rows.
    dk = got["dk"][0, 0].double().numpy()
    dv = got["dv"][0, 0].double().numpy()
    do = inp["do"][0, 0, : w.T_valid].double().numpy()
    assert np.linalg.norm(dk.sum(0)) <= 5e-2 * np.sqrt((dk ** 2).sum())
    assert np.linalg.norm(dv.sum(0) - do.sum(0)) <= 5e-2 * np.sqrt((dv ** 2).sum())
    for g in ("dq", "dk", "dv"):
        assert torch.count_nonzero(got[g][:, :, w.T_valid:]) == 0, g


@pytest.mark.parametrize("H,H_kv", [(1, 1), (2, 1)])
def test_long_schedule_padded_against_unpadded_oracle(H, H_kv):
    """Only the first 3000 tokens are real; the real rows must equal the oracle
    on those 3000 tokens alone, for every output and gradient."""
    w = make_workload("long_schedule_pad", T_valid=3000, **{**LONG_SCHEDULE, "H": H}, H_kv=H_kv)
    inp = make_inputs(w, seed=78)
    got = run_gpu(w, inp)
    wu = make_workload("unpadded", B=1, T=w.T_valid, H=H, H_kv=H_kv, d=w.d, cp=1, rope=False)
    want = _oracle_full(wu, {k: t[:, :, : w.T_valid] for k, t in inp.items()})
    _check_full(wu, {k: t[:, :, : w.T_valid] for k, t in got.items()}, want)
    for g in ("dq", "dk", "dv"):
        assert torch.count_nonzero(got[g][:, :, w.T_valid:]) == 0, g


def test_error_codes_on_device_buffers():
    x = torch.zeros(1, 1, 10, 64, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    with pytest.raises(cpattn.CpattnError) as e:
        cpattn.shard(x, y, 2)            # T=10 is not a multiple of 4
    assert e.value.status == cpattn.ERR_SHAPE
    lse = torch.empty(1, 1, 10, device="cuda")
    with pytest.raises(cpattn.CpattnError) as e:
        cpattn.fwd(x, x, x, y, lse, cp=1, T_valid=11)
    assert e.value.status == cpattn.ERR_SHAPE
    cpattn.cpattn_sync_status(None)


# ------------------------------------------------------------ edge cases ----

EDGE_SMALL = [
    # one row per chunk: every tile has a single valid row
    make_workload("c1_bf16", B=1, T=4, H=1, d=64, cp=2, rope=True),
    make_workload("c1_f32", B=1, T=8, H=2, d=128, cp=4, rope=True, dtype="f32", qkv_std=1.0),
    # a single real token followed by padding
    make_workload("one_valid_token", B=1, T=256, T_valid=1, H=2, d=128, cp=2, rope=True),
    # many (b, h) problems in one launch
    make_workload("many_heads", B=8, T=256, H=32, d=64, cp=2, rope=False),
]


@pytest.mark.parametrize("w", EDGE_SMALL, ids=lambda w: w.name)
def test_edge_cases_full(w):
    inp = make_inputs(w, seed=3 + w.T)
    got = run_gpu(w, inp, rope_mode="shard")
    _check_full(w, got, _oracle_full(w, inp))
    if w.T_valid < w.T:
        for g in ("dq", "dk", "dv"):
            assert torch.count_nonzero(got[g][:, :, w.T_valid:]) == 0, g


# Schedules above the pipelined kernels' 2048-entry tile table run on the
# one-tile kernels, which rotate Q and K themselves when asked to (rope=1).
# One- and two-row chunks at cp > 1024 exceed the table with few tokens, so the
# whole problem is compared with the oracle in both RoPE modes. Between 1024
# and 2048 entries (cp > 512 with one- and two-row chunks) the pipelined
# kernels run with slots above 1023, the top of the table's slot field.
ONE_TILE = [
    make_workload("one_tile_c1_pad", B=1, T=2050, T_valid=2047, H=2, d=128, cp=1025, rope=True),
    make_workload("one_tile_c2_gqa_d64", B=1, T=4160, H=2, H_kv=1, d=64, cp=1040, rope=True),
    make_workload("one_tile_c2_docs", B=1, T=4160, T_valid=4157, H=2, H_kv=1, d=128, cp=1040, rope=True,
                  doc_len=(1, 700), doc_seed=9),
]
WIDE_TABLE = [
    make_workload("wide_table_c1_pad", B=1, T=1026, T_valid=1023, H=2, d=128, cp=513, rope=True),
    make_workload("wide_table_c2_gqa_d64", B=1, T=2080, H=2, H_kv=1, d=64, cp=520, rope=True,
                  doc_len=(1, 300), doc_seed=6),
]


@pytest.mark.parametrize("mode", ROPE_MODES)
@pytest.mark.parametrize("w", WIDE_TABLE, ids=lambda w: w.name)
def test_wide_tile_tables_full(w, mode):
    assert 1024 < 2 * w.cp * -(-w.chunk // 128) <= 2048
    if mode == "kernel" and w.packed:
        pytest.skip("packed documents take RoPE from the shard passes or the save path")
    inp = make_inputs(w, seed=13 + w.cp)
    got = run_gpu(w, inp, rope_mode=mode)
    _check_full(w, got, _oracle_full(w, inp))


@pytest.mark.parametrize("mode", ROPE_MODES)
@pytest.mark.parametrize("w", ONE_TILE, ids=lambda w: w.name)
def test_one_tile_kernels_full(w, mode):
    assert 2 * w.cp * -(-w.chunk // 128) > 2048
    if mode == "kernel" and w.packed:
        pytest.skip("packed documents take RoPE from the shard passes or the save path")
    inp = make_inputs(w, seed=11 + w.cp)
    got = run_gpu(w, inp, rope_mode=mode)
    _check_full(w, got, _oracle_full(w, inp))
    if w.T_valid < w.T:
        for g in ("dq", "dk", "dv"):
            assert torch.count_nonzero(got[g][:, :, w.T_valid:]) == 0, g


def test_one_million_tokens_sampled():
    """T = 2^20 on one head (cp = 64, c = 8192: the one-tile kernels' schedule
    of 8192 tiles per CTA): sampled rows of O, LSE and dQ against the oracle,
    dK and dV through identities of the exact gradient (no RoPE): each row of
    dS sums to zero, so sum_k dK_k = 0; each row of P sums to one, so
    sum_k dV_k = sum_i dO_i."""
    w = make_workload("one_million", B=1, T=1 << 20, H=1, d=64, cp=64, rope=False)
    inp = make_inputs(w, seed=2024)
    got = run_gpu(w, inp)
    rows = np.array(sorted({0, 1, 8191, 8192, (1 << 19) - 1, 1 << 19, (1 << 20) - 1} |
                           set(np.random.default_rng(9).integers(0, w.T, size=12).tolist())))
    tol = TOL[w.dtype]
    o_r, l_r = A.forward_rows(inp["q"], inp["k"], inp["v"], 0, 0, rows, True, w.T_valid, False)
    compare("o", got["o"][0, 0, rows], o_r, tol["o"], tol["cos"])
    compare("lse", got["lse"][0, 0, rows], l_r, tol["lse"])
    dq_r = A.backward_dq_rows(inp["q"], inp["k"], inp["v"], inp["do"], 0, 0, rows, True, w.T_valid, False)
    compare("dq", got["dq"][0, 0, rows], dq_r, tol["grad"], tol["cos"])
    dk = got["dk"][0, 0].double().numpy()
    dv = got["dv"][0, 0].double().numpy()
    do = inp["do"][0, 0].double().numpy()
    assert np.linalg.norm(dk.sum(0)) <= 5e-2 * np.sqrt((dk ** 2).sum())
    # over 2^20 rows the sums carry the bf16 level of the path (P and dS are
    # bf16 MMA operands, 2^-9 relative each): bound the mismatch at 2^-7 of |sum dO|
    assert np.linalg.norm(dv.sum(0) - do.sum(0)) <= 2.0 ** -7 * np.linalg.norm(do.sum(0))
