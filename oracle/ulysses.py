"""Ulysses (DeepSpeed) sequence parallelism on P virtual ranks, float-free.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: "BluScriptCP -- docs/Claude Logs.md", entries 2026-06-30 (Ulysses
next to the ring: all-to-all layout swaps [B,H,Tl,D] <-> [B,Hl,T,D], a plain
rank-order gather, contiguous shards without the HeadTail permutation, and
one full attention per rank) and 2026-07-01 (GQA/MQA: the K/V all-to-all
carries only the K/V heads).

P virtual ranks; Tl = T / P tokens and Hl = H / P heads per rank. Rank r
holds the contiguous tokens [r*Tl, (r+1)*Tl) of every head (its sequence
shard). The all-to-all sends head block s (heads [s*Hl, (s+1)*Hl)) of rank
r's tokens to rank s, which lays what it receives out in rank order, so that
rank s ends up with all T tokens of its Hl heads (its head shard). Each rank
runs one attention over its heads; the inverse all-to-all brings the output
back to the sequence shards.

Layouts (the P ranks' buffers stacked rank-major):
    sequence shards  [P, B, H,  Tl, d]
    head shards      [P, B, Hl, T,  d]
"""
from __future__ import annotations

import numpy as np

from . import attention


def check_shape(T: int, H: int, P: int) -> tuple[int, int]:
    if P < 1 or T % P or H % P:
        raise ValueError(f"P={P} must divide T={T} and H={H}")
    return T // P, H // P


def seq_shards(x: np.ndarray, P: int) -> np.ndarray:
    """Natural [B, H, T, d] -> the P ranks' sequence shards [P, B, H, Tl, d]
    (only the token count must split evenly; the head count matters to the
    all-to-all)."""
    B, H, T, d = x.shape
    if P < 1 or T % P:
        raise ValueError(f"P={P} must divide T={T}")
    Tl = T // P
    return np.stack([x[:, :, r * Tl:(r + 1) * Tl] for r in range(P)])


def all_to_all(x_seq: np.ndarray) -> np.ndarray:
    """Sequence shards [P, B, H, Tl, d] -> head shards [P, B, Hl, T, d]."""
    P, B, H, Tl, d = x_seq.shape
    _, Hl = check_shape(Tl * P, H, P)
    out = np.empty((P, B, Hl, Tl * P, d), dtype=x_seq.dtype)
    for s in range(P):                  # receiving rank
        for r in range(P):              # sending rank: its tokens land in rank order
            out[s, :, :, r * Tl:(r + 1) * Tl] = x_seq[r, :, s * Hl:(s + 1) * Hl]
    return out


def all_to_all_inverse(x_head: np.ndarray) -> np.ndarray:
    """Head shards [P, B, Hl, T, d] -> sequence shards [P, B, H, Tl, d]."""
    P, B, Hl, T, d = x_head.shape
    Tl, _ = check_shape(T, Hl * P, P)
    out = np.empty((P, B, Hl * P, Tl, d), dtype=x_head.dtype)
    for r in range(P):                  # receiving rank: its own token block
        for s in range(P):              # sending rank: its heads
            out[r, :, s * Hl:(s + 1) * Hl] = x_head[s, :, :, r * Tl:(r + 1) * Tl]
    return out


def all_to_all_kv(x_seq: np.ndarray) -> np.ndarray:
    """The K/V all-to-all: sequence shards [P, B, H_kv, Tl, d] -> head shards.

    With H_kv >= P it is ``all_to_all``. With fewer K/V heads than ranks
    (P = rep * H_kv) every K/V head is replicated to the rep ranks whose query
    heads read it ("Claude Logs", 2026-07-01: partial replication by P / n_kv
    when n_kv < P): rank s receives K/V head s // rep, all T tokens, as
    [P, B, 1, T, d].
    """
    P, B, Hkv, Tl, d = x_seq.shape
    if Hkv >= P:
        return all_to_all(x_seq)
    if P % Hkv:
        raise ValueError(f"H_kv={Hkv} must divide P={P} when H_kv < P")
    rep = P // Hkv
    out = np.empty((P, B, 1, Tl * P, d), dtype=x_seq.dtype)
    for s in range(P):
        for r in range(P):
            out[s, :, 0, r * Tl:(r + 1) * Tl] = x_seq[r, :, s // rep]
    return out


def all_to_all_kv_adjoint(g_head: np.ndarray, H_kv: int) -> np.ndarray:
    """Adjoint of ``all_to_all_kv``: head-shard gradients back to sequence
    shards; the rep replicas of a K/V head add up (the group reduce that is the
    backward of a replication)."""
    P, B, Hl, T, d = g_head.shape
    if H_kv >= P:
        return all_to_all_inverse(g_head)
    rep = P // H_kv
    Tl = T // P
    out = np.zeros((P, B, H_kv, Tl, d), dtype=np.float64)
    for s in range(P):
        for r in range(P):
            out[r, :, s // rep] += g_head[s, :, 0, r * Tl:(r + 1) * Tl]
    return out


def ulysses_forward(q, k, v, P: int, causal: bool = True, T_valid: int | None = None,
                    rope_on=False, docs=None):
    """The Ulysses schedule stated rank by rank; returns natural-order O and LSE.

    q is [B, H, T, d]; k, v are [B, H_kv, T, d] with P dividing H_kv, or
    H_kv dividing P (the K/V all-to-all moves K/V heads only, replicating each
    to P / H_kv ranks when there are fewer than P). Rank s attends its Hl query
    heads over all T tokens with the K/V heads it received.
    """
    q, k, v = (attention.as_f64(x) for x in (q, k, v))
    B, H, T, d = q.shape
    Tl, Hl = check_shape(T, H, P)
    qh = all_to_all(seq_shards(q, P))
    kh, vh = (all_to_all_kv(seq_shards(x, P)) for x in (k, v))
    o_head = np.empty_like(qh)
    l_head = np.empty(qh.shape[:4])
    for s in range(P):
        o_head[s], l_head[s] = attention.forward(qh[s], kh[s], vh[s], causal, T_valid, rope_on, docs=docs)
    o_seq = all_to_all_inverse(o_head)
    l_seq = all_to_all_inverse(l_head[..., None])[..., 0]
    return np.concatenate(list(o_seq), axis=2), np.concatenate(list(l_seq), axis=2)
