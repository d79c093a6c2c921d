"""Float64 single-pass causal attention, its gradients, the LSE merge and the ring.

TEST INFRASTRUCTURE ONLY (see the package docstring).

What the pages fix, and where:

* "BluScriptCP -- docs/Claude Logs.md", entry 2026-03-20 (ring attention with
  an SDPA per step and an SDPAMerger), 2026-04-20 (global causal mask through
  T_q / T_k / q_offset / k_offset), 2026-06-17 (the three step shapes of a
  HeadTail ring: the 2c x 2c causal diagonal and two dense rectangles),
  2026-03-24 (the backward's D correction), 2026-06-22 (dK/dV accumulate
  across ring steps and return to their owner), 2026-05-07 and 2026-06-05
  (a RoPE applied at local instead of global positions was a bug), 2026-06-29
  (standard RoPE under HeadTail needs each token's global position).
* "fix(cp): preserve gradients when sharding VLM inputs - #2931": sequences
  are padded at the tail to a multiple of 2*cp before sharding; pad tokens
  must not change the loss.

* "Claude Logs", 2026-07-09, and "HANDOFF_H200_32K": YaRN-extended RoPE
  (``RopeSpec``).

Readings taken where the pages are silent (each is listed in the design
notes): softmax scale 1/sqrt(d); LSE is the natural log of the sum of
exponentials of the *scaled* scores; RoPE is the rotate-half pairing
(i, i + d/2) with theta_i = 10000^(-2i/d) at the token's natural position;
keys at positions >= T_valid are masked; the backward differentiates the
loss sum(dO * O) of the single-pass result (final O and LSE).

Everything here is a direct transcription of those definitions. A row's
forward result depends on that row alone, so rows may be evaluated in groups
(``_ROW_BLOCK``) to bound memory; no other blocking or reordering is done.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import headtail

_ROW_BLOCK = 1024
ROPE_BASE = 10000.0


def as_f64(x) -> np.ndarray:
    """Accept numpy arrays or torch tensors (any float dtype) and return float64."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------- RoPE ----

@dataclasses.dataclass(frozen=True)
class RopeSpec:
    """Which rotary embedding: the standard one, or YaRN context extension.

    "Claude Logs", 2026-07-09 (YaRN in the RoPE cache: an NTK-by-parts blend of
    the frequencies over a dimension-index ramp set by the correction
    dimensions, and an attention temperature m = 0.1 ln(s) + 1 multiplied into
    cos and sin, so logits scale by m^2; scale 1 gives the standard RoPE), and
    "HANDOFF_H200_32K" (the 32k run: scale 2 over an original 16384 positions).
    The method is YaRN (Peng et al., 2023, sections 3.2 and 3.4).
    """
    base: float = ROPE_BASE
    factor: float = 1.0                  # s: context-extension factor
    original_max_position: int = 0       # L: length the weights were trained at
    beta_fast: float = 32.0              # rotations over L above which a pair keeps theta
    beta_slow: float = 1.0               # rotations over L below which a pair gets theta / s
    attention_factor: float = 0.0        # m; <= 0 selects 0.1 ln(s) + 1 (1 when s <= 1)

    def theta(self, d: int) -> np.ndarray:
        """Per-pair angular frequency theta_i, i in [0, d/2)."""
        i = np.arange(d // 2, dtype=np.float64)
        plain = self.base ** (-2.0 * i / d)
        if self.factor <= 1.0:
            return plain
        # Pair index at which a frequency makes n rotations over L:
        # L * base^(-2i/d) = 2 pi n  =>  i = d ln(L / (2 pi n)) / (2 ln base).
        def pair_index(n):
            return d * math.log(self.original_max_position / (2.0 * math.pi * n)) / (2.0 * math.log(self.base))
        lo = max(math.floor(pair_index(self.beta_fast)), 0)
        hi = min(math.ceil(pair_index(self.beta_slow)), d - 1)
        if hi == lo:
            hi += 0.001                  # keeps the ramp a step instead of 0/0
        ramp = np.clip((i - lo) / (hi - lo), 0.0, 1.0)   # 0: keep theta, 1: theta / s
        return plain * (1.0 - ramp) + (plain / self.factor) * ramp

    def mscale(self) -> float:
        if self.attention_factor > 0.0:
            return self.attention_factor
        return 0.1 * math.log(self.factor) + 1.0 if self.factor > 1.0 else 1.0


STANDARD_ROPE = RopeSpec()


def _spec(rope_on) -> RopeSpec | None:
    """rope_on may be False / True (standard RoPE) or a RopeSpec."""
    if isinstance(rope_on, RopeSpec):
        return rope_on
    return STANDARD_ROPE if rope_on else None


def rope_angles(positions: np.ndarray, d: int, spec: RopeSpec = STANDARD_ROPE) -> np.ndarray:
    """angle[p, i] = pos_p * theta_i; standard theta_i = base^(-2i/d), i in [0, d/2)."""
    return np.asarray(positions, dtype=np.float64)[:, None] * spec.theta(d)[None, :]


def rope(x: np.ndarray, positions: np.ndarray, spec: RopeSpec = STANDARD_ROPE) -> np.ndarray:
    """Rotate-half RoPE of x[..., T, d] at the given per-row positions, times m.

    x'_i = m (x_i cos - x_{i+d/2} sin) ;  x'_{i+d/2} = m (x_{i+d/2} cos + x_i sin),
    with m = 1 for the standard rotation.
    """
    d = x.shape[-1]
    ang = rope_angles(positions, d, spec)
    m = spec.mscale()
    c, s = m * np.cos(ang), m * np.sin(ang)
    x1, x2 = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def rope_transpose(g: np.ndarray, positions: np.ndarray, spec: RopeSpec = STANDARD_ROPE) -> np.ndarray:
    """(m R(p))^T g: the adjoint of ``rope``, which carries a gradient back through it."""
    d = g.shape[-1]
    ang = rope_angles(positions, d, spec)
    m = spec.mscale()
    c, s = m * np.cos(ang), m * np.sin(ang)
    g1, g2 = g[..., : d // 2], g[..., d // 2:]
    return np.concatenate([g1 * c + g2 * s, g2 * c - g1 * s], axis=-1)


# ------------------------------------------------------- masked softmax ----

def document_of(positions: np.ndarray, docs) -> np.ndarray:
    """Index of the packed document holding each natural position, -1 for none.

    ``docs`` is cu_seqlens: 0 = docs[0] < docs[1] < ... < docs[n]; document i
    holds positions [docs[i], docs[i+1]); positions >= docs[n] are padding and
    belong to no document.
    """
    docs = np.asarray(docs, dtype=np.int64)
    idx = np.searchsorted(docs, np.asarray(positions), side="right") - 1
    return np.where(np.asarray(positions) < docs[-1], idx, -1)


def allowed(q_pos: np.ndarray, k_pos: np.ndarray, causal: bool, T_valid: int,
            docs=None) -> np.ndarray:
    """allowed[a, b] = (not causal or k_pos[b] <= q_pos[a]) and k_pos[b] < T_valid
    and, for packed documents (``docs`` = cu_seqlens), both positions lie in the
    same document ("fix(cp): ... #2931": packed THD batches; "Claude Logs",
    2026-07-16 training on length-bucketed documents)."""
    ok = np.broadcast_to(k_pos[None, :] < T_valid, (len(q_pos), len(k_pos))).copy()
    if causal:
        ok &= k_pos[None, :] <= q_pos[:, None]
    if docs is not None:
        dq, dk = document_of(q_pos, docs), document_of(k_pos, docs)
        ok &= (dq[:, None] == dk[None, :]) & (dq[:, None] >= 0)
    return ok


def allowed_sum(W: np.ndarray, ok: np.ndarray, X: np.ndarray) -> np.ndarray:
    """out[t, :] = sum over the j with ok[t, j] of W[t, j] * X[j, :].

    The attention sums run over allowed pairs only: a pair the mask excludes
    contributes nothing, even where W or X holds an Inf or a NaN (which a dense
    product with zeros at masked pairs would turn into NaN, 0 * Inf). Finite
    entries of X go through one matrix product; each non-finite entry is then
    added on its own into the rows allowed to see it.
    """
    W = np.where(ok, W, 0.0)
    bad = ~np.isfinite(X)
    out = W @ np.where(bad, 0.0, X)
    for j, c in zip(*np.nonzero(bad)):
        out[:, c] += np.where(ok[:, j], W[:, j] * X[j, c], 0.0)
    return out


def partial_attention(qr: np.ndarray, kr: np.ndarray, vr: np.ndarray, q_pos: np.ndarray,
                      k_pos: np.ndarray, causal: bool, T_valid: int, docs=None):
    """Softmax attention of query rows over a key set, with the global mask.

    qr, kr are already rotated (if RoPE is on). Returns (O, LSE); a row with no
    allowed key gets the merge identity (O = 0, LSE = -inf). Only allowed pairs
    enter the max, the sums and the product with V, so a NaN or an Inf reaches
    exactly the rows whose allowed pairs hold it.
    """
    d = qr.shape[-1]
    S = (qr @ kr.T) / math.sqrt(d)
    ok = allowed(q_pos, k_pos, causal, T_valid, docs)
    has = ok.any(axis=1)                               # a row is empty iff no pair is allowed
    S = np.where(ok, S, -np.inf)
    m = np.where(has, np.max(S, axis=1, initial=-np.inf), 0.0)
    E = np.where(ok, np.exp(S - m[:, None]), 0.0)      # exp(-inf) = 0 on masked pairs
    ssum = E.sum(axis=1)
    lse = np.where(has, m + np.log(np.where(has, ssum, 1.0)), -np.inf)
    P = np.where(has[:, None], E / np.where(has, ssum, 1.0)[:, None], 0.0)
    return allowed_sum(P, ok, vr), lse


def _heads(x):
    x = as_f64(x)
    B, H = x.shape[0], x.shape[1]
    return x, B, H


def kv_head(h: int, H: int, H_kv: int) -> int:
    """K/V head read by query head h when H query heads share H_kv K/V heads.

    "Claude Logs", 2026-06-29 (keep GQA-grouped K/V in the ring) and
    2026-07-01 (GQA/MQA: K/V heads broadcast to their query heads by a
    repeat-interleave, whose adjoint is a sum over each group). Under a
    repeat-interleave, consecutive query heads share a K/V head: query head h
    reads K/V head h // (H / H_kv). H_kv = H is multi-head attention, H_kv = 1
    multi-query attention.
    """
    if H_kv < 1 or H % H_kv:
        raise ValueError(f"H_kv={H_kv} must divide H={H}")
    return h // (H // H_kv)


def _rotated(xh: np.ndarray, rope_on) -> np.ndarray:
    spec = _spec(rope_on)
    if spec is None:
        return xh
    return rope(xh, np.arange(xh.shape[0]), spec)


def forward(q, k, v, causal: bool = True, T_valid: int | None = None, rope_on: bool | RopeSpec = False, docs=None):
    """Single-pass attention over natural-order inputs: q [B, H, T, d], k and v
    [B, H_kv, T, d] (H_kv divides H; see ``kv_head``).

    Returns O [B, H, T, d] and LSE [B, H, T] (float64). RoPE, when on, is applied
    to q and k at their natural (global) positions.
    """
    q, B, H = _heads(q)
    k, v = as_f64(k), as_f64(v)
    T = q.shape[2]
    T_valid = T if T_valid is None else T_valid
    pos = np.arange(T)
    O = np.zeros_like(q)
    L = np.zeros(q.shape[:3])
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, k.shape[1])
            qh, kh = _rotated(q[b, h], rope_on), _rotated(k[b, hk], rope_on)
            for r0 in range(0, T, _ROW_BLOCK):
                rows = pos[r0:r0 + _ROW_BLOCK]
                O[b, h, rows], L[b, h, rows] = partial_attention(
                    qh[rows], kh, v[b, hk], rows, pos, causal, T_valid, docs)
    return O, L


def forward_rows(q, k, v, b: int, h: int, rows, causal: bool = True,
                 T_valid: int | None = None, rope_on: bool | RopeSpec = False, docs=None):
    """O and LSE of selected natural rows of one head (each row is independent)."""
    rows = np.asarray(rows, dtype=np.int64)
    hk = kv_head(h, q.shape[1], k.shape[1])
    qh, kh, vh = as_f64(q[b, h]), as_f64(k[b, hk]), as_f64(v[b, hk])
    T = kh.shape[0]
    T_valid = T if T_valid is None else T_valid
    qr = rope(qh[rows], rows, _spec(rope_on)) if rope_on else qh[rows]
    kr = _rotated(kh, rope_on)
    return partial_attention(qr, kr, vh, rows, np.arange(T), causal, T_valid, docs)


# ------------------------------------------------------------ backward ----

def _backward_head(qh, kh, vh, oh, lseh, doh, causal, T_valid, rope_on, docs=None):
    """Gradient of sum(dO * O) for one head, all rows (T x T matrices)."""
    T, d = qh.shape
    pos = np.arange(T)
    qr, kr = _rotated(qh, rope_on), _rotated(kh, rope_on)
    S = (qr @ kr.T) / math.sqrt(d)
    ok = allowed(pos, pos, causal, T_valid, docs)
    P = np.where(ok, np.exp(np.where(ok, S, 0.0) - lseh[:, None]), 0.0)
    dV = allowed_sum(P.T, ok.T, doh)
    dP = doh @ vh.T
    D = np.sum(doh * oh, axis=1)
    dS = np.where(ok, P * (dP - D[:, None]), 0.0)
    dQr = allowed_sum(dS, ok, kr) / math.sqrt(d)
    dKr = allowed_sum(dS.T, ok.T, qr) / math.sqrt(d)
    if rope_on:
        return rope_transpose(dQr, pos, _spec(rope_on)), rope_transpose(dKr, pos, _spec(rope_on)), dV
    return dQr, dKr, dV


def backward(q, k, v, o, lse, do, causal: bool = True, T_valid: int | None = None,
             rope_on: bool | RopeSpec = False, docs=None):
    """dq, dk, dv of the loss sum(dO * O), through RoPE if it is on.

    o and lse are the single-pass forward results (float64). With P = exp(S - LSE):
    dV = P^T dO;  dP = dO V^T;  D = rowsum(dO * O);  dS = P * (dP - D);
    dQ' = dS K' / sqrt(d);  dK' = dS^T Q' / sqrt(d);  dq = R^T dQ', dk = R^T dK'.
    """
    q, B, H = _heads(q)
    k, v, o, lse, do = (as_f64(x) for x in (k, v, o, lse, do))
    T = q.shape[2]
    T_valid = T if T_valid is None else T_valid
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, k.shape[1])
            dq[b, h], dk_h, dv_h = _backward_head(
                q[b, h], k[b, hk], v[b, hk], o[b, h], lse[b, h], do[b, h], causal, T_valid, rope_on,
                docs)
            dk[b, hk] += dk_h           # a shared K/V head gathers its group's gradients
            dv[b, hk] += dv_h
    return dq, dk, dv


def backward_dq_rows(q, k, v, do, b: int, h: int, rows, causal: bool = True,
                     T_valid: int | None = None, rope_on: bool | RopeSpec = False, docs=None):
    """dq of selected natural rows of one head; each needs only its own row of P."""
    rows = np.asarray(rows, dtype=np.int64)
    hk = kv_head(h, q.shape[1], k.shape[1])
    kh, vh, doh = as_f64(k[b, hk]), as_f64(v[b, hk]), as_f64(do[b, h])
    T, d = kh.shape
    T_valid = T if T_valid is None else T_valid
    o_r, lse_r = forward_rows(q, k, v, b, h, rows, causal, T_valid, rope_on, docs)
    qr = rope(as_f64(q[b, h])[rows], rows, _spec(rope_on)) if rope_on else as_f64(q[b, h])[rows]
    kr = _rotated(kh, rope_on)
    ok = allowed(rows, np.arange(T), causal, T_valid, docs)
    S = (qr @ kr.T) / math.sqrt(d)
    P = np.where(ok, np.exp(np.where(ok, S, 0.0) - lse_r[:, None]), 0.0)
    dP = doh[rows] @ vh.T
    D = np.sum(doh[rows] * o_r, axis=1)
    dQr = allowed_sum(np.where(ok, P * (dP - D[:, None]), 0.0), ok, kr) / math.sqrt(d)
    return rope_transpose(dQr, rows, _spec(rope_on)) if rope_on else dQr


def backward_dkdv_cols(q, k, v, do, b: int, h: int, cols, causal: bool = True,
                       T_valid: int | None = None, rope_on: bool | RopeSpec = False, docs=None):
    """dk, dv of selected natural key rows of K/V head h.

    For each query head that reads K/V head h (one head without grouping, see
    ``kv_head``): O and LSE of every query row of that head (computed here, row
    by row as in ``forward``), then one column of P, dP and dS per selected
    key; the group's contributions are summed.
    """
    cols = np.asarray(cols, dtype=np.int64)
    H, H_kv = q.shape[1], k.shape[1]
    kh, vh = as_f64(k[b, h]), as_f64(v[b, h])
    T, d = kh.shape
    T_valid = T if T_valid is None else T_valid
    pos = np.arange(T)
    kr = _rotated(kh, rope_on)
    dK = np.zeros((len(cols), d))
    dV = np.zeros((len(cols), d))
    for hq in (x for x in range(H) if kv_head(x, H, H_kv) == h):
        qh, doh = as_f64(q[b, hq]), as_f64(do[b, hq])
        qr = _rotated(qh, rope_on)
        O = np.zeros_like(qh)
        L = np.zeros(T)
        for r0 in range(0, T, _ROW_BLOCK):
            rows = pos[r0:r0 + _ROW_BLOCK]
            O[rows], L[rows] = partial_attention(qr[rows], kr, vh, rows, pos, causal, T_valid, docs)
        D = np.sum(doh * O, axis=1)
        ok = allowed(pos, cols, causal, T_valid, docs)      # [T, n_cols]
        S = (qr @ kr[cols].T) / math.sqrt(d)
        P = np.where(ok, np.exp(np.where(ok, S, 0.0) - L[:, None]), 0.0)
        dV += allowed_sum(P.T, ok.T, doh)
        dP = doh @ vh[cols].T
        dS = np.where(ok, P * (dP - D[:, None]), 0.0)
        dK += allowed_sum(dS.T, ok.T, qr) / math.sqrt(d)
    return (rope_transpose(dK, cols, _spec(rope_on)) if rope_on else dK), dV


# ---------------------------------------------------------- LSE merge ----

def merge(o_a: np.ndarray, l_a: np.ndarray, o_b: np.ndarray, l_b: np.ndarray):
    """SDPAMerger for two partials of the same rows.

    L = m + log(e^{L_a - m} + e^{L_b - m}) with m = max(L_a, L_b);
    O = e^{L_a - L} O_a + e^{L_b - L} O_b. (-inf, 0) is the identity, and two
    empty partials give (-inf, 0).
    """
    l_a, l_b = np.asarray(l_a, np.float64), np.asarray(l_b, np.float64)
    none_a, none_b = l_a == -np.inf, l_b == -np.inf     # partials that saw no key
    empty = none_a & none_b
    m = np.maximum(l_a, l_b)                           # a NaN LSE stays NaN
    m_safe = np.where(empty, 0.0, m)
    wa = np.where(none_a, 0.0, np.exp(l_a - m_safe))
    wb = np.where(none_b, 0.0, np.exp(l_b - m_safe))
    tot = wa + wb
    L = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, tot)))
    scale_a = np.where(empty, 0.0, wa / np.where(empty, 1.0, tot))
    scale_b = np.where(empty, 0.0, wb / np.where(empty, 1.0, tot))
    O = scale_a[..., None] * o_a + scale_b[..., None] * o_b
    return O, L


def merge_many(o_parts, l_parts):
    """Left fold of ``merge`` over a list of partials, starting from the identity."""
    O = np.zeros_like(np.asarray(o_parts[0], np.float64))
    L = np.full(np.asarray(l_parts[0]).shape, -np.inf)
    for o_s, l_s in zip(o_parts, l_parts):
        O, L = merge(O, L, o_s, l_s)
    return O, L


# ---------------------------------------------------------------- ring ----

def ring_forward(q, k, v, cp: int, causal: bool = True, T_valid: int | None = None,
                 rope_on: bool | RopeSpec = False, docs=None):
    """The ring schedule, stated step by step; returns natural-order O and LSE.

    Virtual rank r holds HeadTail chunks r and 2cp-1-r. At ring step s it
    holds the K/V of rank j = (r - s) mod cp (received from its predecessor),
    attends its queries to those keys under the global causal mask, and merges
    that partial into its running (O, LSE) with the SDPAMerger.
    """
    q, B, H = _heads(q)
    k, v = as_f64(k), as_f64(v)
    T = q.shape[2]
    T_valid = T if T_valid is None else T_valid
    O = np.zeros_like(q)
    L = np.zeros(q.shape[:3])
    for b in range(B):
        for h in range(H):
            hk = kv_head(h, H, k.shape[1])
            qh, kh = _rotated(q[b, h], rope_on), _rotated(k[b, hk], rope_on)
            for r in range(cp):
                rows = headtail.rank_tokens(T, cp, r)
                o_run = np.zeros((len(rows), q.shape[3]))
                l_run = np.full(len(rows), -np.inf)
                for s in range(cp):
                    j = (r - s) % cp
                    keys = headtail.rank_tokens(T, cp, j)
                    o_s, l_s = partial_attention(qh[rows], kh[keys], v[b, hk][keys], rows, keys,
                                                 causal, T_valid, docs)
                    o_run, l_run = merge(o_run, l_run, o_s, l_s)
                O[b, h, rows], L[b, h, rows] = o_run, l_run
    return O, L


def rank_causal_work(T: int, cp: int, causal: bool = True, T_valid: int | None = None) -> list[int]:
    """Number of allowed (query, key) pairs whose query sits on each virtual rank."""
    T_valid = T if T_valid is None else T_valid
    pos = np.arange(T)
    work = []
    for r in range(cp):
        rows = headtail.rank_tokens(T, cp, r)
        work.append(int(allowed(rows, pos, causal, T_valid).sum()))
    return work
