"""Pins for the CPU oracle: each checks it against something other than itself.

The pins are the pages' worked HeadTail example (tests/golden), brute-force
softmax written with plain Python loops and complex-number RoPE, closed forms,
scipy's softmax / logsumexp, the ring == single-pass invariant, the algebra of
the LSE merge, and central finite differences of the analytic gradients. The
"planted" tests feed deliberately wrong variants of oracle pieces to the same
checks and require them to fail, so a plausible slip (a dropped term, a wrong
sign, an off-by-one mask, a transposed operand) cannot pass unnoticed.
"""
from __future__ import annotations

import cmath
import math
import os

import numpy as np
import pytest
from scipy import special

from oracle import attention as A
from oracle import headtail as HT

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(20261202)


def rnd(*shape, std=1.0):
    return rng.standard_normal(shape) * std


# ------------------------------------------------------------ HeadTail ----

def test_headtail_worked_example():
    want = {}
    with open(os.path.join(GOLDEN, "headtail_T8_cp2.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            r, toks = line.split(":")
            want[int(r)] = [int(t) for t in toks.split()]
    assert set(want) == {0, 1}
    for r, toks in want.items():
        assert list(HT.rank_tokens(8, 2, r)) == toks
    pos = HT.positions_of_sharded_rows(8, 2)
    assert list(pos) == want[0] + want[1]


def _pairing_by_enumeration(T, cp):
    """Independent construction: list the 2cp chunks, give rank r chunks r and 2cp-1-r."""
    c = T // (2 * cp)
    chunks = [list(range(i * c, (i + 1) * c)) for i in range(2 * cp)]
    order = []
    for r in range(cp):
        order += chunks[r] + chunks[2 * cp - 1 - r]
    return order


@pytest.mark.parametrize("T,cp", [(8, 1), (8, 2), (24, 3), (64, 4), (48, 8), (30, 5)])
def test_headtail_closed_form_and_bijection(T, cp):
    sigma = HT.shard_index(T, cp)
    assert sorted(sigma.tolist()) == list(range(T))               # bijection
    assert HT.positions_of_sharded_rows(T, cp).tolist() == _pairing_by_enumeration(T, cp)
    x = rnd(2, 3, T, 5)
    assert np.array_equal(HT.unshard(HT.shard(x, cp), cp), x)     # round trip, bit-exact
    if cp == 1:
        assert np.array_equal(sigma, np.arange(T))                # cp=1 is the identity


@pytest.mark.parametrize("T,cp", [(16, 2), (64, 4), (96, 3), (128, 8)])
def test_headtail_balances_causal_work(T, cp):
    work = A.rank_causal_work(T, cp)
    assert len(set(work)) == 1, work
    # and contiguous sharding would not: rank 0 of a contiguous split does least
    c2 = T // cp
    contiguous = [sum(t + 1 for t in range(r * c2, (r + 1) * c2)) for r in range(cp)]
    assert cp == 1 or len(set(contiguous)) > 1


@pytest.mark.parametrize("T,cp,T_valid", [(8, 2, 8), (8, 2, 6), (24, 3, 20), (64, 4, 64), (60, 5, 41)])
def test_rank_causal_work_counts_pairs(T, cp, T_valid):
    """Independent count: a causal row t sees keys 0..min(t, T_valid - 1), i.e.
    min(t + 1, T_valid) of them; a non-causal row sees T_valid. Rows come from
    the enumerated pairing, not from the oracle's index map."""
    order = _pairing_by_enumeration(T, cp)
    per_rank = T // cp
    want_causal = [sum(min(t + 1, T_valid) for t in order[r * per_rank:(r + 1) * per_rank])
                   for r in range(cp)]
    assert A.rank_causal_work(T, cp, True, T_valid) == want_causal
    assert A.rank_causal_work(T, cp, False, T_valid) == [per_rank * T_valid] * cp
    if (T, cp) == (8, 2):
        # by hand: rank 0 = {0,1,6,7}, rank 1 = {2,3,4,5}
        assert want_causal == ([1 + 2 + 7 + 8, 3 + 4 + 5 + 6] if T_valid == 8
                               else [1 + 2 + 6 + 6, 3 + 4 + 5 + 6])


def test_headtail_rejects_bad_shapes():
    with pytest.raises(ValueError):
        HT.shard_index(10, 2)


# ---------------------------------------------------------------- RoPE ----

def _rope_complex(x, positions):
    """Textbook form: pair (x_i, x_{i+d/2}) as a complex number times e^{i p theta_i}."""
    T, d = x.shape
    out = np.empty_like(x)
    for t in range(T):
        for i in range(d // 2):
            theta = 10000.0 ** (-2.0 * i / d)
            z = complex(x[t, i], x[t, i + d // 2]) * cmath.exp(1j * positions[t] * theta)
            out[t, i], out[t, i + d // 2] = z.real, z.imag
    return out


def check_rope(rope_fn, rope_t_fn):
    x = rnd(9, 8)
    pos = np.array([0, 1, 2, 5, 17, 100, 1000, 4097, 32767])
    err = np.abs(rope_fn(x, pos) - _rope_complex(x, pos)).max()
    y = rnd(9, 8)
    # adjoint: <R x, y> == <x, R^T y>
    err = max(err, abs(np.sum(rope_fn(x, pos) * y) - np.sum(x * rope_t_fn(y, pos))))
    return err


def test_rope_against_complex_rotation():
    assert check_rope(A.rope, A.rope_transpose) < 1e-12


def test_rope_properties():
    x = rnd(6, 16)
    pos = np.arange(6) * 7
    assert np.allclose(np.linalg.norm(A.rope(x, pos), axis=1), np.linalg.norm(x, axis=1), atol=1e-12)
    assert np.array_equal(A.rope(x, np.zeros(6)), x)                  # p = 0 is the identity
    q, k = rnd(16), rnd(16)
    for m, n, delta in [(5, 2, 11), (100, 99, 1000), (3, 30, 7)]:
        a = A.rope(q[None], np.array([m])) @ A.rope(k[None], np.array([n])).T
        b = A.rope(q[None], np.array([m + delta])) @ A.rope(k[None], np.array([n + delta])).T
        assert abs(a - b).max() < 1e-10                              # relative position only
    assert np.allclose(A.rope_transpose(A.rope(x, pos), pos), x, atol=1e-12)


def test_planted_rope_sign_is_caught():
    def bad_rope(x, positions):
        d = x.shape[-1]
        ang = A.rope_angles(positions, d)
        c, s = np.cos(ang), np.sin(ang)
        x1, x2 = x[..., : d // 2], x[..., d // 2:]
        return np.concatenate([x1 * c + x2 * s, x2 * c - x1 * s], axis=-1)
    assert check_rope(bad_rope, A.rope_transpose) > 1e-3


# ------------------------------------------------------------- forward ----

def brute_force_forward(q, k, v, causal, T_valid, rope_on):
    """Plain Python loops, direct exp and sum with no max shift, complex RoPE."""
    T, d = q.shape
    if rope_on:
        q, k = _rope_complex(q, np.arange(T)), _rope_complex(k, np.arange(T))
    O = np.zeros((T, d))
    L = np.zeros(T)
    for t in range(T):
        w = []
        for j in range(T):
            if (causal and j > t) or j >= T_valid:
                w.append(0.0)
            else:
                w.append(math.exp(sum(q[t, i] * k[j, i] for i in range(d)) / math.sqrt(d)))
        tot = sum(w)
        L[t] = math.log(tot)
        for i in range(d):
            O[t, i] = sum(w[j] * v[j, i] for j in range(T)) / tot
    return O, L


def check_forward(fwd):
    err = 0.0
    for causal, T_valid, rope_on in [(True, 7, False), (False, 7, False), (True, 5, True),
                                     (False, 6, True), (True, 7, True)]:
        q, k, v = rnd(1, 1, 7, 6), rnd(1, 1, 7, 6), rnd(1, 1, 7, 6)
        O, L = fwd(q, k, v, causal=causal, T_valid=T_valid, rope_on=rope_on)
        Ob, Lb = brute_force_forward(q[0, 0], k[0, 0], v[0, 0], causal, T_valid, rope_on)
        err = max(err, np.abs(O[0, 0] - Ob).max(), np.abs(L[0, 0] - Lb).max())
    return err


def test_forward_against_brute_force():
    assert check_forward(A.forward) < 1e-12


def test_planted_forward_mistakes_are_caught(monkeypatch):
    real_allowed = A.allowed

    def strict_causal(q_pos, k_pos, causal, T_valid, docs=None):   # j < t instead of j <= t
        ok = real_allowed(q_pos, k_pos, causal, T_valid, docs)
        if causal:
            ok &= k_pos[None, :] != q_pos[:, None]
        return ok
    monkeypatch.setattr(A, "allowed", strict_causal)
    with np.errstate(all="ignore"):
        assert not check_forward(A.forward) < 1e-6
    monkeypatch.setattr(A, "allowed", real_allowed)

    def no_pad_mask(q_pos, k_pos, causal, T_valid, docs=None):
        return real_allowed(q_pos, k_pos, causal, 10 ** 9, docs)
    monkeypatch.setattr(A, "allowed", no_pad_mask)
    assert not check_forward(A.forward) < 1e-6
    monkeypatch.setattr(A, "allowed", real_allowed)

    real_pa = A.partial_attention

    def transposed_v(qr, kr, vr, q_pos, k_pos, causal, T_valid, docs=None):
        return real_pa(qr, kr, vr[::-1], q_pos, k_pos, causal, T_valid, docs)
    monkeypatch.setattr(A, "partial_attention", transposed_v)
    assert not check_forward(A.forward) < 1e-6


def test_forward_closed_forms():
    T, d = 12, 8
    q, k, v = rnd(1, 2, T, d), rnd(1, 2, T, d), rnd(1, 2, T, d)
    O, L = A.forward(q, k, v, causal=True)
    # row 0 sees only key 0
    assert np.allclose(O[:, :, 0], v[:, :, 0], atol=1e-14)
    assert np.allclose(L[:, :, 0], np.sum(q[:, :, 0] * k[:, :, 0], -1) / math.sqrt(d), atol=1e-14)
    # k == 0: uniform weights over the causal prefix
    O0, L0 = A.forward(q, np.zeros_like(k), v, causal=True)
    prefix_mean = np.cumsum(v, axis=2) / np.arange(1, T + 1)[None, None, :, None]
    assert np.allclose(O0, prefix_mean, atol=1e-13)
    assert np.allclose(L0, np.log(np.arange(1, T + 1))[None, None], atol=1e-13)
    # v constant: every row returns it
    u = rnd(d)
    Ou, _ = A.forward(q, k, np.broadcast_to(u, v.shape), causal=True)
    assert np.allclose(Ou, np.broadcast_to(u, v.shape), atol=1e-13)


def test_noncausal_matches_scipy_softmax():
    T, d = 33, 16
    q, k, v = rnd(2, 1, T, d), rnd(2, 1, T, d), rnd(2, 1, T, d)
    O, L = A.forward(q, k, v, causal=False)
    for b in range(2):
        S = q[b, 0] @ k[b, 0].T / math.sqrt(d)
        assert np.allclose(O[b, 0], special.softmax(S, axis=1) @ v[b, 0], atol=1e-13)
        assert np.allclose(L[b, 0], special.logsumexp(S, axis=1), atol=1e-13)


def test_forward_rows_matches_full():
    q, k, v = rnd(1, 2, 40, 8), rnd(1, 2, 40, 8), rnd(1, 2, 40, 8)
    O, L = A.forward(q, k, v, causal=True, T_valid=37, rope_on=True)
    rows = [0, 3, 17, 36, 39]
    o_r, l_r = A.forward_rows(q, k, v, 0, 1, rows, True, 37, True)
    assert np.allclose(o_r, O[0, 1, rows], atol=1e-13) and np.allclose(l_r, L[0, 1, rows], atol=1e-13)


# ---------------------------------------------------------- ring + merge ----

@pytest.mark.parametrize("cp", [1, 2, 4, 8])
@pytest.mark.parametrize("causal,T_valid,rope_on", [(True, 64, False), (True, 59, True),
                                                    (False, 64, True)])
def test_ring_equals_single_pass(cp, causal, T_valid, rope_on):
    T, d = 64, 8
    q, k, v = rnd(1, 2, T, d), rnd(1, 2, T, d), rnd(1, 2, T, d)
    O, L = A.forward(q, k, v, causal, T_valid, rope_on)
    Or, Lr = A.ring_forward(q, k, v, cp, causal, T_valid, rope_on)
    assert np.abs(O - Or).max() <= 1e-12 and np.abs(L - Lr).max() <= 1e-12


def test_merge_algebra():
    n, d = 10, 5
    parts = [(rnd(n, d), rnd(n)) for _ in range(3)]
    parts[1][1][2] = -np.inf                                  # one empty partial row
    (oa, la), (ob, lb), (oc, lc) = parts
    left = A.merge(*A.merge(oa, la, ob, lb), oc, lc)
    right = A.merge(oa, la, *A.merge(ob, lb, oc, lc))
    assert np.abs(left[0] - right[0]).max() <= 1e-13 and np.abs(left[1] - right[1]).max() <= 1e-13
    ab, ba = A.merge(oa, la, ob, lb), A.merge(ob, lb, oa, la)
    assert np.abs(ab[0] - ba[0]).max() <= 1e-13 and np.abs(ab[1] - ba[1]).max() <= 1e-13
    ident = A.merge(oa, la, np.zeros((n, d)), np.full(n, -np.inf))
    assert np.abs(ident[0] - oa).max() <= 1e-15 and np.abs(ident[1] - la).max() <= 1e-15
    empty = A.merge(np.zeros((n, d)), np.full(n, -np.inf), np.zeros((n, d)), np.full(n, -np.inf))
    assert np.all(empty[1] == -np.inf) and np.all(empty[0] == 0)
    # merge of two disjoint key sets == softmax over their union (scipy)
    d2 = 6
    q, k, v = rnd(4, d2), rnd(9, d2), rnd(9, d2)
    S = q @ k.T / math.sqrt(d2)
    pa = A.partial_attention(q, k[:4], v[:4], np.full(4, 100), np.arange(4), False, 100)
    pb = A.partial_attention(q, k[4:], v[4:], np.full(4, 100), np.arange(4, 9), False, 100)
    Om, Lm = A.merge(*pa, *pb)
    assert np.allclose(Om, special.softmax(S, axis=1) @ v, atol=1e-13)
    assert np.allclose(Lm, special.logsumexp(S, axis=1), atol=1e-13)


def check_merge_many(merge_many_fn):
    """Max error of an n-way SDPAMerger fold against scipy over the union of keys.

    "Claude Logs", 2026-03-20 (an SDPAMerger folds the per-step partials) and
    2026-05-20 (partials that see no key must not disturb the result). Each
    partial is built here directly with scipy from its own key subset, so the
    check rests on nothing else in the oracle. Keys are split into n disjoint,
    interleaved subsets; a causal mask leaves some rows empty in some partials
    and some rows (position -1) empty in all of them. An empty partial carries
    LSE = -inf and an arbitrary finite O, which must not leak into the result.
    """
    err = 0.0
    d = 6
    for n in (1, 2, 5, 16):
        Tk = 3 * n + 2
        nq = 9
        q, k, v = rnd(nq, d), rnd(Tk, d), rnd(Tk, d)
        q_pos = np.array([-1, 0, 1, 2, 5, Tk // 2, Tk - 2, Tk - 1, -1])
        k_pos = np.arange(Tk)
        S = np.where(k_pos[None, :] <= q_pos[:, None], q @ k.T / math.sqrt(d), -np.inf)
        subset = rng.permutation(Tk) % n                      # key j belongs to partial subset[j]
        o_parts, l_parts = [], []
        for i in range(n):
            Si = np.where(subset[None, :] == i, S, -np.inf)
            with np.errstate(invalid="ignore"):
                Pi = special.softmax(Si, axis=1)
            live = np.isfinite(Si).any(axis=1)
            o_parts.append(np.where(live[:, None], np.nan_to_num(Pi) @ v, rnd(nq, d)))
            l_parts.append(np.where(live, special.logsumexp(Si, axis=1), -np.inf))
        O, L = merge_many_fn(o_parts, l_parts)
        live = np.isfinite(S).any(axis=1)
        with np.errstate(invalid="ignore"):
            want_o = np.where(live[:, None], np.nan_to_num(special.softmax(S, axis=1)) @ v, 0.0)
        want_l = np.where(live, special.logsumexp(S, axis=1), -np.inf)
        if not (np.array_equal(np.isfinite(L), live) and np.all(L[~live] == -np.inf)
                and np.all(O[~live] == 0.0)):
            return np.inf
        err = max(err, np.abs(O - want_o).max(), np.abs(L[live] - want_l[live]).max())
    return err


def test_merge_many_against_scipy_union():
    assert check_merge_many(A.merge_many) < 1e-13


def test_planted_merge_many_mistakes_are_caught():
    def from_zero(o_parts, l_parts):                          # fold starts at L = 0, not -inf
        O, L = np.zeros_like(o_parts[0]), np.zeros(np.shape(l_parts[0]))
        for o_s, l_s in zip(o_parts, l_parts):
            O, L = A.merge(O, L, o_s, l_s)
        return O, L

    def first_twice(o_parts, l_parts):                        # partial 0 merged twice
        return A.merge_many([o_parts[0]] + list(o_parts), [l_parts[0]] + list(l_parts))

    def last_dropped(o_parts, l_parts):                       # loop stops one short
        n = max(len(o_parts) - 1, 1)
        return A.merge_many(o_parts[:n], l_parts[:n])

    def plain_average(o_parts, l_parts):                      # no LSE weights at all
        w = [np.isfinite(l).astype(float) for l in l_parts]
        tot = np.maximum(sum(w), 1.0)
        O = sum(wi[:, None] * o for wi, o in zip(w, o_parts)) / tot[:, None]
        return O, A.merge_many(o_parts, l_parts)[1]

    with np.errstate(all="ignore"):
        for bad in (from_zero, first_twice, last_dropped, plain_average):
            assert not check_merge_many(bad) < 1e-6, bad.__name__


# ------------------------------------------------- non-finite inputs ----
# The sums of attention run over allowed pairs only, so a NaN or an Inf in an
# input reaches exactly the outputs whose allowed pairs hold it: every other
# output equals the result on the same inputs with that value made finite.

def _poisoned(T=12, d=4, t0=5, j0=7):
    q, k, v, do = (rnd(1, 1, T, d) for _ in range(4))
    qn, vi = q.copy(), v.copy()
    qn[0, 0, t0, 1] = np.nan
    vi[0, 0, j0, 2] = np.inf
    return q, k, v, do, qn, vi, t0, j0


def check_nonfinite(forward, backward):
    """0 if NaN / Inf inputs reach exactly the outputs that see them, else 1."""
    q, k, v, do, qn, vi, t0, j0 = _poisoned()
    T = q.shape[2]
    with np.errstate(invalid="ignore", over="ignore"):
        O0, L0 = forward(q, k, v, True, T)
        g0 = backward(q, k, v, O0, L0, do, True, T)
        # NaN in q[t0]: O, LSE, dq of row t0; dk, dv of keys j <= t0
        O, L = forward(qn, k, v, True, T)
        dq, dk, dv = backward(qn, k, v, O, L, do, True, T)
        rows = np.arange(T) != t0
        ok = (np.all(~np.isfinite(O[0, 0, t0])) and np.isnan(L[0, 0, t0])
              and np.allclose(O[0, 0, rows], O0[0, 0, rows], rtol=0, atol=1e-13)
              and np.allclose(L[0, 0, rows], L0[0, 0, rows], rtol=0, atol=1e-13)
              and np.all(np.isnan(dq[0, 0, t0]))
              and np.allclose(dq[0, 0, rows], g0[0][0, 0, rows], rtol=0, atol=1e-12))
        for g, g_ref in ((dk, g0[1]), (dv, g0[2])):
            ok = ok and np.all(~np.isfinite(g[0, 0, :t0 + 1])) and np.allclose(
                g[0, 0, t0 + 1:], g_ref[0, 0, t0 + 1:], rtol=0, atol=1e-12)
        # +Inf in v[j0, 2]: column 2 of O for rows t >= j0; D, hence dq rows
        # t >= j0 and every dk row (the last query sees every key); dv untouched
        O, L = forward(q, k, vi, True, T)
        dq, dk, dv = backward(q, k, vi, O, L, do, True, T)
        fin = np.ones((T, q.shape[3]), bool)
        fin[j0:, 2] = False
        ok = ok and (np.array_equal(np.isfinite(O[0, 0]), fin) and np.all(O[0, 0, j0:, 2] == np.inf)
                     and np.allclose(O[0, 0][fin], O0[0, 0][fin], rtol=0, atol=1e-13)
                     and np.allclose(L, L0, rtol=0, atol=1e-13)
                     and np.all(~np.isfinite(dq[0, 0, j0:]))
                     and np.allclose(dq[0, 0, :j0], g0[0][0, 0, :j0], rtol=0, atol=1e-12)
                     and np.all(~np.isfinite(dk)) and np.allclose(dv, g0[2], rtol=0, atol=1e-12))
    return 0 if ok else 1


def test_nonfinite_inputs_reach_only_the_outputs_that_see_them():
    assert check_nonfinite(A.forward, A.backward) == 0


def test_planted_nonfinite_mistakes_are_caught(monkeypatch):
    def dense(W, ok, X):                                      # masked pairs as zeros of a dense product
        return np.where(ok, W, 0.0) @ X
    monkeypatch.setattr(A, "allowed_sum", dense)
    assert check_nonfinite(A.forward, A.backward) == 1
    monkeypatch.undo()
    real_pa = A.partial_attention

    def nan_row_is_empty(qr, kr, vr, q_pos, k_pos, causal, T_valid, docs=None):
        O, L = real_pa(qr, kr, vr, q_pos, k_pos, causal, T_valid, docs)
        bad = ~np.isfinite(L)
        return np.where(bad[:, None], 0.0, O), np.where(bad, -np.inf, L)
    monkeypatch.setattr(A, "partial_attention", nan_row_is_empty)
    assert check_nonfinite(A.forward, A.backward) == 1


def test_merge_keeps_nan_and_empty_apart():
    o, l = rnd(3, 2), np.array([0.5, np.nan, -np.inf])
    O, L = A.merge(o, l, np.zeros((3, 2)), np.full(3, -np.inf))
    assert L[0] == 0.5 and np.isnan(L[1]) and L[2] == -np.inf
    assert np.all(np.isnan(O[1])) and np.all(O[2] == 0.0)


# ------------------------------------------------------------ backward ----

def check_gradients_fd(bwd, causal, T_valid, rope_on, h=1e-6):
    """Max relative error of analytic grads against central finite differences."""
    T, d = 6, 4
    q, k, v, do = rnd(1, 1, T, d), rnd(1, 1, T, d), rnd(1, 1, T, d), rnd(1, 1, T, d)

    def loss(q_, k_, v_):
        O, _ = A.forward(q_, k_, v_, causal, T_valid, rope_on)
        return np.sum(do * O)

    O, L = A.forward(q, k, v, causal, T_valid, rope_on)
    grads = bwd(q, k, v, O, L, do, causal, T_valid, rope_on)
    worst = 0.0
    for which, g in enumerate(grads):
        fd = np.zeros_like(g)
        for idx in np.ndindex(g.shape):
            args_p = [q.copy(), k.copy(), v.copy()]
            args_m = [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        worst = max(worst, np.abs(g - fd).max() / max(np.abs(fd).max(), 1e-3))
    return worst


@pytest.mark.parametrize("causal,T_valid,rope_on", [(True, 6, False), (True, 6, True),
                                                    (False, 6, True), (True, 4, True)])
def test_backward_against_finite_differences(causal, T_valid, rope_on):
    assert check_gradients_fd(A.backward, causal, T_valid, rope_on) <= 1e-6


def test_planted_backward_mistakes_are_caught(monkeypatch):
    real = A._backward_head

    def no_D(qh, kh, vh, oh, lseh, doh, causal, T_valid, rope_on, docs=None):   # drops the D term
        return real(qh, kh, vh, np.zeros_like(oh), lseh, doh, causal, T_valid, rope_on, docs)
    monkeypatch.setattr(A, "_backward_head", no_D)
    assert check_gradients_fd(A.backward, True, 6, False) > 1e-3

    def no_rope_adjoint(qh, kh, vh, oh, lseh, doh, causal, T_valid, rope_on, docs=None):
        dq, dk, dv = real(qh, kh, vh, oh, lseh, doh, causal, T_valid, rope_on, docs)
        pos = np.arange(qh.shape[0])
        return A.rope(A.rope(dq, pos), pos), dk, dv                     # R instead of R^T
    monkeypatch.setattr(A, "_backward_head", no_rope_adjoint)
    assert check_gradients_fd(A.backward, True, 6, True) > 1e-3


def test_backward_invariants():
    T, d = 20, 8
    q, k, v, do = rnd(1, 2, T, d), rnd(1, 2, T, d), rnd(1, 2, T, d), rnd(1, 2, T, d)
    O, L = A.forward(q, k, v, True)
    dq, dk, dv = A.backward(q, k, v, O, L, do, True)
    # softmax rows sum to one: sum_j dV_j = sum_t dO_t
    assert np.allclose(dv.sum(axis=2), do.sum(axis=2), atol=1e-12)
    # sum_j dS_tj = 0 per row, so without RoPE sum_j dK_j = 0
    assert np.abs(dk.sum(axis=2)).max() < 1e-12


def test_sampled_backward_matches_full():
    T, d = 48, 8
    q, k, v, do = rnd(1, 2, T, d), rnd(1, 2, T, d), rnd(1, 2, T, d), rnd(1, 2, T, d)
    do[:, :, 45:] = 0
    O, L = A.forward(q, k, v, True, 45, True)
    dq, dk, dv = A.backward(q, k, v, O, L, do, True, 45, True)
    rows = [0, 1, 30, 44, 47]
    assert np.allclose(A.backward_dq_rows(q, k, v, do, 0, 1, rows, True, 45, True), dq[0, 1, rows],
                       atol=1e-12)
    dk_c, dv_c = A.backward_dkdv_cols(q, k, v, do, 0, 1, rows, True, 45, True)
    assert np.allclose(dk_c, dk[0, 1, rows], atol=1e-12)
    assert np.allclose(dv_c, dv[0, 1, rows], atol=1e-12)


# ------------------------------------------------------------- padding ----

def test_padding_is_invisible_to_real_rows():
    Tr, Tp, d = 13, 16, 8
    q, k, v, do = rnd(1, 2, Tp, d), rnd(1, 2, Tp, d), rnd(1, 2, Tp, d), rnd(1, 2, Tp, d)
    do[:, :, Tr:] = 0
    Op, Lp = A.forward(q, k, v, True, Tr, True)
    Ou, Lu = A.forward(q[:, :, :Tr], k[:, :, :Tr], v[:, :, :Tr], True, Tr, True)
    assert np.abs(Op[:, :, :Tr] - Ou).max() < 1e-13 and np.abs(Lp[:, :, :Tr] - Lu).max() < 1e-13
    gp = A.backward(q, k, v, Op, Lp, do, True, Tr, True)
    gu = A.backward(q[:, :, :Tr], k[:, :, :Tr], v[:, :, :Tr], Ou, Lu, do[:, :, :Tr], True, Tr, True)
    for a, b in zip(gp, gu):
        assert np.abs(a[:, :, :Tr] - b).max() < 1e-13
        assert np.all(a[:, :, Tr:] == 0.0)                 # pad-row grads are exactly zero


# --------------------------------------------- grouped K/V heads (GQA) ----

def test_kv_head_is_repeat_interleave():
    # repeat-interleave of K/V heads: query heads 0..g-1 read K/V head 0, ...
    assert [A.kv_head(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [A.kv_head(h, 6, 3) for h in range(6)] == [0, 0, 1, 1, 2, 2]
    assert [A.kv_head(h, 4, 4) for h in range(4)] == [0, 1, 2, 3]
    assert [A.kv_head(h, 4, 1) for h in range(4)] == [0, 0, 0, 0]
    with pytest.raises(ValueError):
        A.kv_head(0, 6, 4)


def _gqa_case(H=6, H_kv=2, T=24, d=8, T_valid=21):
    q, do = rnd(2, H, T, d), rnd(2, H, T, d)
    k, v = rnd(2, H_kv, T, d), rnd(2, H_kv, T, d)
    do[:, :, T_valid:] = 0
    return q, k, v, do, T_valid


def _check_gqa_equals_repeated_mha(rope_on):
    """GQA == multi-head attention on K/V repeated along heads (np.repeat is a
    repeat-interleave); the GQA gradient of a K/V head is the sum of the
    repeated copies' gradients."""
    q, k, v, do, Tv = _gqa_case()
    g = q.shape[1] // k.shape[1]
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    O, L = A.forward(q, k, v, True, Tv, rope_on)
    Om, Lm = A.forward(q, kr, vr, True, Tv, rope_on)
    err = max(np.abs(O - Om).max(), np.abs(L - Lm).max())
    dq, dk, dv = A.backward(q, k, v, O, L, do, True, Tv, rope_on)
    dqm, dkm, dvm = A.backward(q, kr, vr, Om, Lm, do, True, Tv, rope_on)
    B, H_kv, T, d = k.shape
    err = max(err, np.abs(dq - dqm).max(),
              np.abs(dk - dkm.reshape(B, H_kv, g, T, d).sum(2)).max(),
              np.abs(dv - dvm.reshape(B, H_kv, g, T, d).sum(2)).max())
    return err


@pytest.mark.parametrize("rope_on", [False, True])
def test_gqa_equals_mha_with_repeated_kv(rope_on):
    assert _check_gqa_equals_repeated_mha(rope_on) < 1e-12


def test_planted_gqa_head_map_is_caught(monkeypatch):
    # the other common grouping (query head h -> K/V head h mod H_kv) must fail
    monkeypatch.setattr(A, "kv_head", lambda h, H, H_kv: h % H_kv)
    assert _check_gqa_equals_repeated_mha(False) > 1e-3


def test_gqa_backward_against_finite_differences():
    H, H_kv, T, d, h = 4, 2, 5, 4, 1e-6
    q, do = rnd(1, H, T, d), rnd(1, H, T, d)
    k, v = rnd(1, H_kv, T, d), rnd(1, H_kv, T, d)

    def loss(q_, k_, v_):
        return np.sum(do * A.forward(q_, k_, v_, True, T, True)[0])

    O, L = A.forward(q, k, v, True, T, True)
    grads = A.backward(q, k, v, O, L, do, True, T, True)
    worst = 0.0
    for which, g in enumerate(grads):
        fd = np.zeros_like(g)
        for idx in np.ndindex(g.shape):
            args_p, args_m = [q.copy(), k.copy(), v.copy()], [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        worst = max(worst, np.abs(g - fd).max() / max(np.abs(fd).max(), 1e-3))
    assert worst <= 1e-6


def test_mqa_invariants_and_sampled_match_full():
    q, k, v, do, Tv = _gqa_case(H=4, H_kv=1)
    O, L = A.forward(q, k, v, True, Tv)
    dq, dk, dv = A.backward(q, k, v, O, L, do, True, Tv)
    # each softmax row sums to one and each row of dS to zero, over all 4 query heads
    assert np.allclose(dv.sum(axis=2)[:, 0], do.sum(axis=(1, 2)), atol=1e-12)
    assert np.abs(dk.sum(axis=2)).max() < 1e-12
    rows = [0, 5, 20, 23]
    for b, hq in [(0, 0), (1, 3)]:
        Or, Lr = A.forward_rows(q, k, v, b, hq, rows, True, Tv)
        assert np.abs(Or - O[b, hq, rows]).max() < 1e-13 and np.abs(Lr - L[b, hq, rows]).max() < 1e-13
        assert np.abs(A.backward_dq_rows(q, k, v, do, b, hq, rows, True, Tv) - dq[b, hq, rows]).max() < 1e-12
    q, k, v, do, Tv = _gqa_case()
    O, L = A.forward(q, k, v, True, Tv, True)
    dq, dk, dv = A.backward(q, k, v, O, L, do, True, Tv, True)
    dk_c, dv_c = A.backward_dkdv_cols(q, k, v, do, 1, 1, rows, True, Tv, True)
    assert np.abs(dk_c - dk[1, 1, rows]).max() < 1e-12 and np.abs(dv_c - dv[1, 1, rows]).max() < 1e-12


def test_gqa_ring_equals_single_pass():
    q, k, v, _, Tv = _gqa_case()
    O, L = A.forward(q, k, v, True, Tv, True)
    Or, Lr = A.ring_forward(q, k, v, 3, True, Tv, True)
    assert np.abs(O - Or).max() < 1e-12 and np.abs(L - Lr).max() < 1e-12


# ------------------------------------------------------------- YaRN RoPE ----

# The 32k extension run: scale 2 over the 16384 positions the weights saw.
YARN_32K = A.RopeSpec(factor=2.0, original_max_position=16384)


def test_yarn_scale_one_is_standard_rope():
    x = rnd(2, 40, 64)
    pos = np.arange(40) * 37
    plain = A.rope(x, pos)
    same = A.rope(x, pos, A.RopeSpec(factor=1.0, original_max_position=4096))
    assert np.array_equal(plain, same)
    assert A.RopeSpec(factor=1.0).mscale() == 1.0


def test_yarn_frequencies_closed_form_for_the_32k_run():
    # d = 128, base 1e4, L = 16384: a frequency makes n rotations over L at pair
    # index 128 ln(L / (2 pi n)) / (2 ln 1e4) = 30.58 for n = 32 and 54.66 for
    # n = 1, so the ramp runs from pair 30 (floor) to pair 55 (ceil).
    th = YARN_32K.theta(128)
    plain = 1e4 ** (-np.arange(64) / 64.0)
    assert np.array_equal(th[:31], plain[:31])               # pairs 0..30 keep theta
    assert np.allclose(th[55:], plain[55:] / 2, rtol=1e-15)  # pairs 55..63 get theta / 2
    for i in (31, 40, 54):                                    # linear in between
        w = (i - 30) / 25.0
        assert abs(th[i] - plain[i] * (1 - w / 2)) <= 1e-15 * plain[i]
    assert abs(YARN_32K.mscale() - (0.1 * math.log(2.0) + 1.0)) < 1e-15
    assert abs(YARN_32K.mscale() - 1.0693147180559945) < 1e-15


def test_yarn_keeps_fast_pairs_and_scales_slow_ones():
    """Stated in rotations over L (YaRN section 3.2): pairs that turn many times
    over the trained length keep their frequency, pairs that turn less than
    once are interpolated by the factor."""
    for d, L, s in [(128, 16384, 2.0), (64, 4096, 8.0), (128, 2048, 4.0)]:
        spec = A.RopeSpec(factor=s, original_max_position=L)
        plain = 1e4 ** (-np.arange(d // 2) * 2.0 / d)
        rot = L * plain / (2 * math.pi)
        step = 1e4 ** (2.0 / d)                              # ratio of adjacent frequencies
        fast, slow = rot >= 32 * step, rot <= 1 / step
        assert fast.any() and slow.any()
        assert np.array_equal(spec.theta(d)[fast], plain[fast])
        assert np.allclose(spec.theta(d)[slow], plain[slow] / s, rtol=1e-15)
        assert np.all(np.diff(spec.theta(d)) < 0)            # still strictly decreasing


def test_yarn_rotation_properties():
    x, y = rnd(3, 50, 128), rnd(3, 50, 128)
    pos = np.arange(50) * 601
    m = YARN_32K.mscale()
    r = A.rope(x, pos, YARN_32K)
    # each (i, i + d/2) pair is rotated and scaled by m
    n_in = np.hypot(x[..., :64], x[..., 64:])
    n_out = np.hypot(r[..., :64], r[..., 64:])
    assert np.allclose(n_out, m * n_in, rtol=1e-13)
    # the adjoint used by the backward
    assert abs(np.sum(r * y) - np.sum(x * A.rope_transpose(y, pos, YARN_32K))) < 1e-9
    # scores depend on the position difference only, and carry m^2
    q, k = rnd(1, 128), rnd(1, 128)
    s1 = A.rope(q, np.array([20000]), YARN_32K) @ A.rope(k, np.array([19000]), YARN_32K).T
    s2 = A.rope(q, np.array([1500]), YARN_32K) @ A.rope(k, np.array([500]), YARN_32K).T
    assert abs(s1 - s2).max() < 1e-10
    s0 = A.rope(q, np.array([0]), YARN_32K) @ A.rope(k, np.array([0]), YARN_32K).T
    assert abs(s0 - m * m * (q @ k.T)).max() < 1e-12


# small trained length so that the ramp is not trivial at d = 8: pairs 0..3 get
# weights 0, 1/2, 1, 1 towards theta / 4
YARN_TINY = A.RopeSpec(factor=4.0, original_max_position=64)


def test_yarn_tiny_spec_has_a_ramp():
    th = YARN_TINY.theta(8)
    plain = 1e4 ** (-np.arange(4) / 4.0)
    assert np.allclose(th, plain * (1 - np.array([0, 0.5, 1, 1]) * 0.75), rtol=1e-15)


def test_yarn_backward_against_finite_differences():
    T, d, h = 6, 8, 1e-6
    q, k, v, do = rnd(1, 2, T, d), rnd(1, 1, T, d), rnd(1, 1, T, d), rnd(1, 2, T, d)

    def loss(q_, k_, v_):
        return np.sum(do * A.forward(q_, k_, v_, True, T, YARN_TINY)[0])

    O, L = A.forward(q, k, v, True, T, YARN_TINY)
    grads = A.backward(q, k, v, O, L, do, True, T, YARN_TINY)
    worst = 0.0
    for which, g in enumerate(grads):
        fd = np.zeros_like(g)
        for idx in np.ndindex(g.shape):
            args_p, args_m = [q.copy(), k.copy(), v.copy()], [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        worst = max(worst, np.abs(g - fd).max() / max(np.abs(fd).max(), 1e-3))
    assert worst <= 1e-6


def test_planted_yarn_mistakes_are_caught():
    # beta_fast and beta_slow swapped: the ramp collapses and the closed form fails
    swapped = A.RopeSpec(factor=2.0, original_max_position=16384, beta_fast=1.0, beta_slow=32.0)
    plain = 1e4 ** (-np.arange(64) / 64.0)
    assert not np.allclose(swapped.theta(128)[55:], plain[55:] / 2)
    # temperature applied once instead of to both q and k: scores lose a factor m
    q, k = rnd(1, 128), rnd(1, 128)
    one_sided = A.rope(q, np.array([0]), YARN_32K) @ k.T
    assert abs(one_sided - YARN_32K.mscale() ** 2 * (q @ k.T)).max() > 1e-3


def test_yarn_ring_and_sampled_rows_match_full():
    T, d = 48, 16
    spec = A.RopeSpec(factor=4.0, original_max_position=12)
    q, k, v, do = rnd(1, 2, T, d), rnd(1, 2, T, d), rnd(1, 2, T, d), rnd(1, 2, T, d)
    O, L = A.forward(q, k, v, True, T, spec)
    Or, Lr = A.ring_forward(q, k, v, 4, True, T, spec)
    assert np.abs(O - Or).max() < 1e-12 and np.abs(L - Lr).max() < 1e-12
    dq, dk, dv = A.backward(q, k, v, O, L, do, True, T, spec)
    rows = [0, 7, 31, 47]
    assert np.abs(A.backward_dq_rows(q, k, v, do, 0, 1, rows, True, T, spec) - dq[0, 1, rows]).max() < 1e-12
    dk_c, dv_c = A.backward_dkdv_cols(q, k, v, do, 0, 0, rows, True, T, spec)
    assert np.abs(dk_c - dk[0, 0, rows]).max() < 1e-12 and np.abs(dv_c - dv[0, 0, rows]).max() < 1e-12


# ------------------------------------------------ packed documents (varlen) ----

# 64 positions: documents of 5, 1, 17, 17 and 21 tokens, then 3 pad positions.
DOCS = np.array([0, 5, 6, 23, 40, 61])


def test_document_of():
    pos = np.arange(64)
    want = [0] * 5 + [1] + [2] * 17 + [3] * 17 + [4] * 21 + [-1] * 3
    assert A.document_of(pos, DOCS).tolist() == want


def _varlen_vs_documents(causal, rope_on, H=4, H_kv=2):
    """Max difference between packed attention and each document run alone,
    with its positions restarting at 0 (RoPE scores depend on position
    differences only, so the packed run may keep global positions)."""
    T, d, Tv = 64, 8, int(DOCS[-1])
    q, do = rnd(2, H, T, d), rnd(2, H, T, d)
    k, v = rnd(2, H_kv, T, d), rnd(2, H_kv, T, d)
    O, L = A.forward(q, k, v, causal, Tv, rope_on, docs=DOCS)
    dq, dk, dv = A.backward(q, k, v, O, L, do, causal, Tv, rope_on, docs=DOCS)
    err = 0.0
    for a, b in zip(DOCS[:-1], DOCS[1:]):
        sl = slice(a, b)
        Od, Ld = A.forward(q[:, :, sl], k[:, :, sl], v[:, :, sl], causal, b - a, rope_on)
        g = A.backward(q[:, :, sl], k[:, :, sl], v[:, :, sl], Od, Ld, do[:, :, sl], causal, b - a, rope_on)
        err = max(err, np.abs(O[:, :, sl] - Od).max(), np.abs(L[:, :, sl] - Ld).max(),
                  *(np.abs(x[:, :, sl] - y).max() for x, y in zip((dq, dk, dv), g)))
    # pad rows attend nothing and receive nothing
    assert np.all(O[:, :, Tv:] == 0) and np.all(L[:, :, Tv:] == -np.inf)
    for x in (dq, dk, dv):
        assert np.all(x[:, :, Tv:] == 0)
    return err


@pytest.mark.parametrize("causal,rope_on", [(True, False), (True, True), (False, True),
                                            (True, A.RopeSpec(factor=4.0, original_max_position=8))])
def test_varlen_equals_documents_run_alone(causal, rope_on):
    assert _varlen_vs_documents(causal, rope_on) < 1e-12


def test_planted_document_boundary_is_caught(monkeypatch):
    real = A.document_of

    def off_by_one(positions, docs):      # first token of each document put in the previous one
        docs = np.asarray(docs)
        idx = np.searchsorted(docs, np.asarray(positions), side="left") - 1
        return np.where(np.asarray(positions) < docs[-1], np.maximum(idx, 0), -1)
    monkeypatch.setattr(A, "document_of", off_by_one)
    assert _varlen_vs_documents(True, False) > 1e-3
    monkeypatch.setattr(A, "document_of", real)


def test_single_document_is_plain_causal():
    T, d = 40, 8
    q, k, v, do = rnd(1, 2, T, d), rnd(1, 2, T, d), rnd(1, 2, T, d), rnd(1, 2, T, d)
    O, L = A.forward(q, k, v, True, 37, True)
    Od, Ld = A.forward(q, k, v, True, 37, True, docs=np.array([0, 37]))
    assert np.array_equal(O[:, :, :37], Od[:, :, :37]) and np.array_equal(L[:, :, :37], Ld[:, :, :37])


def test_varlen_backward_against_finite_differences():
    T, d, h = 7, 4, 1e-6
    docs = np.array([0, 3, 4, 7])
    q, k, v, do = rnd(1, 1, T, d), rnd(1, 1, T, d), rnd(1, 1, T, d), rnd(1, 1, T, d)

    def loss(q_, k_, v_):
        return np.sum(do * A.forward(q_, k_, v_, True, T, True, docs=docs)[0])

    O, L = A.forward(q, k, v, True, T, True, docs=docs)
    grads = A.backward(q, k, v, O, L, do, True, T, True, docs=docs)
    worst = 0.0
    for which, g in enumerate(grads):
        fd = np.zeros_like(g)
        for idx in np.ndindex(g.shape):
            args_p, args_m = [q.copy(), k.copy(), v.copy()], [q.copy(), k.copy(), v.copy()]
            args_p[which][idx] += h
            args_m[which][idx] -= h
            fd[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        worst = max(worst, np.abs(g - fd).max() / max(np.abs(fd).max(), 1e-3))
    assert worst <= 1e-6


def test_varlen_ring_and_sampled_match_full():
    T, d = 64, 8
    q, k, v, do = rnd(1, 2, T, d), rnd(1, 1, T, d), rnd(1, 1, T, d), rnd(1, 2, T, d)
    O, L = A.forward(q, k, v, True, 61, True, docs=DOCS)
    Or, Lr = A.ring_forward(q, k, v, 4, True, 61, True, docs=DOCS)
    assert np.abs(O - Or).max() < 1e-12 and np.array_equal(np.isinf(L), np.isinf(Lr))
    fin = np.isfinite(L)
    assert np.abs(L[fin] - Lr[fin]).max() < 1e-12
    dq, dk, dv = A.backward(q, k, v, O, L, do, True, 61, True, docs=DOCS)
    rows = [0, 4, 5, 6, 22, 23, 60, 62]
    assert np.abs(A.backward_dq_rows(q, k, v, do, 0, 1, rows, True, 61, True, docs=DOCS)
                  - dq[0, 1, rows]).max() < 1e-12
    dk_c, dv_c = A.backward_dkdv_cols(q, k, v, do, 0, 0, rows, True, 61, True, docs=DOCS)
    assert np.abs(dk_c - dk[0, 0, rows]).max() < 1e-12 and np.abs(dv_c - dv[0, 0, rows]).max() < 1e-12


# ---------------------------------------------------------------- Ulysses ----

from oracle import ulysses as U  # noqa: E402


@pytest.mark.parametrize("B,H,T,P", [(1, 4, 8, 2), (2, 6, 12, 3), (1, 8, 16, 4), (2, 3, 9, 1)])
def test_ulysses_all_to_all_gives_head_blocks(B, H, T, P):
    x = rnd(B, H, T, 5)
    xs = U.seq_shards(x, P)
    Tl, Hl = T // P, H // P
    for r in range(P):                                    # rank r holds its token block
        assert np.array_equal(xs[r], x[:, :, r * Tl:(r + 1) * Tl])
    xh = U.all_to_all(xs)
    for s in range(P):                                    # rank s holds its heads, all tokens
        assert np.array_equal(xh[s], x[:, s * Hl:(s + 1) * Hl])
    assert np.array_equal(U.all_to_all_inverse(xh), xs)


def test_ulysses_rejects_bad_shapes():
    with pytest.raises(ValueError):
        U.seq_shards(rnd(1, 4, 10, 2), 3)
    with pytest.raises(ValueError):
        U.all_to_all(U.seq_shards(rnd(1, 3, 8, 2), 2))       # 2 ranks cannot split 3 heads
    with pytest.raises(ValueError):
        U.all_to_all_kv(U.seq_shards(rnd(1, 3, 8, 2), 4))    # nor replicate 3 heads over 4 ranks
    with pytest.raises(ValueError):
        U.all_to_all(rnd(2, 1, 3, 5, 2))


@pytest.mark.parametrize("P,H_kv,rope_on,docs", [(2, 4, False, None), (4, 4, True, None),
                                                 (2, 2, True, None), (2, 4, True, np.array([0, 9, 30, 47]))])
def test_ulysses_equals_single_pass(P, H_kv, rope_on, docs):
    T, d = 48, 8
    q, k, v = rnd(2, 4, T, d), rnd(2, H_kv, T, d), rnd(2, H_kv, T, d)
    O, L = A.forward(q, k, v, True, 47, rope_on, docs=docs)
    Ou, Lu = U.ulysses_forward(q, k, v, P, True, 47, rope_on, docs=docs)
    assert np.abs(O - Ou).max() < 1e-13
    fin = np.isfinite(L)
    assert np.array_equal(fin, np.isfinite(Lu)) and np.abs(L[fin] - Lu[fin]).max() < 1e-13


@pytest.mark.parametrize("P,H,H_kv", [(4, 8, 2), (4, 4, 1), (8, 8, 2), (2, 4, 1)])
def test_ulysses_kv_replication_equals_single_pass_gqa(P, H, H_kv):
    T, d = 32, 8
    q, k, v = rnd(2, H, T, d), rnd(2, H_kv, T, d), rnd(2, H_kv, T, d)
    O, L = A.forward(q, k, v, True, T, True)
    Ou, Lu = U.ulysses_forward(q, k, v, P, True, T, True)
    assert np.abs(O - Ou).max() < 1e-13 and np.abs(L - Lu).max() < 1e-13


@pytest.mark.parametrize("P,H_kv", [(4, 2), (4, 1), (8, 2), (4, 4)])
def test_ulysses_kv_adjoint(P, H_kv):
    """<A x, y> = <x, A^T y> for the replicating all-to-all and its reduce."""
    T, d = 16, 5
    x = rnd(P, 2, H_kv, T // P, d)
    y = rnd(*U.all_to_all_kv(x).shape)
    lhs = np.sum(U.all_to_all_kv(x) * y)
    rhs = np.sum(x * U.all_to_all_kv_adjoint(y, H_kv))
    assert abs(lhs - rhs) < 1e-10
    if H_kv < P:   # replication: each K/V head reaches exactly P / H_kv ranks
        ones = np.ones_like(U.all_to_all_kv(x))
        assert np.all(U.all_to_all_kv_adjoint(ones, H_kv) == P // H_kv)
