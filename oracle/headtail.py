"""HeadTail (chunk-level) load-balanced sequence sharding, float-free.

Source: "BluScriptCP -- docs/Claude Logs.md", entries 2026-05-16 ("HeadTail
kernel rewritten to chunk-level (PyTorch parity)"), 2026-06-29 (Megatron's
``index_select [r, 2cp-1-r]`` cos/sin sharding, and the pure-CPU delta helper
whose worked example gives rank 0 the tokens {0, 1, 6, 7} for N=2); and
"fix(cp): preserve gradients when sharding VLM inputs - #2931" (round-robin
local indices matching torch's 2*cp head-tail chunk pairing).

The sequence of T tokens is cut into 2*cp chunks of c = T / (2*cp). Virtual
rank r owns chunk r (its "head") followed by chunk 2*cp-1-r (its "tail"), and
the sharded tensor lists the ranks in order, so the sharded row of natural
token t is

    kappa = t // c, o = t % c
    r     = kappa            if kappa < cp else 2*cp - 1 - kappa
    l     = o                if kappa < cp else c + o
    sigma(t) = 2*c*r + l
"""
from __future__ import annotations

import numpy as np


def check_shape(T: int, cp: int) -> int:
    if cp < 1 or T < 1 or T % (2 * cp) != 0:
        raise ValueError(f"T={T} must be a positive multiple of 2*cp={2 * cp}")
    return T // (2 * cp)


def shard_index(T: int, cp: int) -> np.ndarray:
    """sigma[t] = sharded row of natural token t (int64), by the closed form above."""
    c = check_shape(T, cp)
    sigma = np.empty(T, dtype=np.int64)
    for t in range(T):
        kappa, o = divmod(t, c)
        if kappa < cp:
            r, l = kappa, o
        else:
            r, l = 2 * cp - 1 - kappa, c + o
        sigma[t] = 2 * c * r + l
    return sigma


def rank_tokens(T: int, cp: int, r: int) -> np.ndarray:
    """Natural token positions held by virtual rank r, in its local row order."""
    c = check_shape(T, cp)
    head = np.arange(r * c, (r + 1) * c)
    tail = np.arange((2 * cp - 1 - r) * c, (2 * cp - r) * c)
    return np.concatenate([head, tail])


def positions_of_sharded_rows(T: int, cp: int) -> np.ndarray:
    """pos[i] = natural position of sharded row i (the inverse of sigma)."""
    sigma = shard_index(T, cp)
    pos = np.empty(T, dtype=np.int64)
    pos[sigma] = np.arange(T)
    return pos


def shard(x: np.ndarray, cp: int, axis: int = -2) -> np.ndarray:
    """Natural -> sharded order along ``axis`` (out of place)."""
    T = x.shape[axis]
    sigma = shard_index(T, cp)
    out = np.empty_like(x)
    idx_dst = [slice(None)] * x.ndim
    idx_dst[axis] = sigma
    out[tuple(idx_dst)] = x
    return out


def unshard(x: np.ndarray, cp: int, axis: int = -2) -> np.ndarray:
    """Sharded -> natural order along ``axis`` (out of place)."""
    T = x.shape[axis]
    sigma = shard_index(T, cp)
    return np.take(x, sigma, axis=axis)
