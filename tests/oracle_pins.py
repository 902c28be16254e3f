"""Pins for the fp64 oracle: facts fixed by the pages or by mathematics, each written
so that a plausible mistake in the oracle (a dropped term, a wrong sign or index, a
transposed operand, a missing scale) fails at least one of them.

Every check takes an ``oracle.Oracle`` handle and raises ``AssertionError`` on failure.
``tests/test_oracle_pins.py`` runs them on the real oracle; ``tests/test_oracle_mutants.py``
runs them on builds with one planted mistake each and expects a failure.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def online_softmax_tiles(scores, values, cuts):
    """Test-only online-softmax recurrence (fp64) over one score row split at ``cuts``.

    Follows "15. FlashAttention" (inference.shantanugoel.com), section "Online softmax:
    normalize as you go": m_new = max(m_old, max(tile)), alpha = e^(m_old - m_new),
    p = e^(s - m_new), l = alpha*l + sum(p), a = alpha*a + p V, and O = a / l at the end.
    Returns O, the final (m, l) and the per-tile intermediates.
    """
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    if values.ndim == 1:
        values = values[:, None]
    bounds = [0] + list(cuts) + [len(scores)]
    m, l = -math.inf, 0.0
    a = np.zeros(values.shape[1])
    steps = []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        if hi <= lo:
            continue
        s = scores[lo:hi]
        m_new = max(m, float(s.max()))
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        p = np.exp(s - m_new)
        l = alpha * l + float(p.sum())
        a = alpha * a + p @ values[lo:hi]
        steps.append({"m": m_new, "alpha": alpha, "p": p.copy(), "l": l, "a": a.copy()})
        m = m_new
    return a / l, m, l, steps


def _score_row_case(scores, values, d=64):
    """Embed one raw score row and scalar values into [1,1,n,d] tensors with scale 1:
    query 0 = e_0, key j = s_j e_0, value j = v_j e_0 (exact in bf16 for small integers)."""
    n = len(scores)
    q = np.zeros((1, 1, n, d))
    k = np.zeros((1, 1, n, d))
    v = np.zeros((1, 1, n, d))
    q[0, 0, 0, 0] = 1.0
    k[0, 0, :, 0] = scores
    v[0, 0, :, 0] = values
    return q, k, v


# ---------------------------------------------------------------------------------------
# Page fixtures

def check_worked_example_oracle(orc):
    g = json.load(open(os.path.join(GOLDEN, "worked_example_online_softmax.json")))
    q, k, v = _score_row_case(g["scores"], g["values"])
    o, lse = orc.forward_f64(q, k, v, causal=False, scale=1.0)
    tol = 0.5 * 10 ** -g["printed_decimals"]
    assert abs(o[0, 0, 0, 0] - g["printed"]["O"]) <= tol, o[0, 0, 0, 0]
    # Not printed on the page: LSE = ln(e^0 + e^1 + e^2 + e^-1), from the tile-2 state
    # m = 2, l = 1.5530 (ln form m + ln l).
    assert abs(lse[0, 0, 0] - (2.0 + math.log(g["printed"]["final_l"]))) <= 1e-4
    # Same values through the bf16 entry point (all inputs are exact in bf16).
    bits = [_to_bf16_bits(x) for x in (q, k, v)]
    o2, lse2 = orc.forward_bf16(*bits, causal=False, scale=1.0)
    assert abs(o2[0, 0, 0, 0] - o[0, 0, 0, 0]) <= 1e-15
    assert abs(lse2[0, 0, 0] - lse[0, 0, 0]) <= 1e-15


def check_worked_example_two_tiles(orc):
    g = json.load(open(os.path.join(GOLDEN, "worked_example_online_softmax.json")))
    pr = g["printed"]
    tol = 0.5 * 10 ** -g["printed_decimals"] + 1e-12
    O, m, l, steps = online_softmax_tiles(g["scores"], g["values"], [g["tile"]])
    t1, t2 = steps
    assert abs(t1["m"] - pr["tile1_m"]) <= tol
    assert np.all(np.abs(t1["p"] - pr["tile1_p"]) <= tol)
    assert abs(t1["l"] - pr["tile1_l"]) <= tol
    assert abs(t1["a"][0] - pr["tile1_a"]) <= tol
    assert abs(t2["m"] - pr["tile2_m"]) <= tol
    assert abs(t2["alpha"] - pr["tile2_alpha"]) <= tol
    assert np.all(np.abs(t2["p"] - pr["tile2_p"]) <= tol)
    assert abs(t2["l"] - pr["final_l"]) <= tol
    # The page rounds alpha and l1 before multiplying; the exact a differs from 2.8915
    # by up to ~1e-4, so the final accumulator is held to the printed O instead.
    assert abs(t2["a"][0] - pr["final_a"]) <= 2e-4
    assert abs(O[0] - pr["O"]) <= tol
    # One pass (a single tile) and the oracle give the same number.
    O1, _, _, _ = online_softmax_tiles(g["scores"], g["values"], [])
    q, k, v = _score_row_case(g["scores"], g["values"])
    o, _ = orc.forward_f64(q, k, v, causal=False, scale=1.0)
    assert abs(O1[0] - O[0]) <= 1e-14
    assert abs(o[0, 0, 0, 0] - O[0]) <= 1e-14


def _to_bf16_bits(x):
    f = np.asarray(x, dtype=np.float32)
    assert np.all(f.astype(np.float64) == x), "value not exact in float32"
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------------------
# Recurrence invariants (exactness by induction)

def check_online_every_split(orc):
    """Every split of random rows (length <= 12) through the recurrence equals the
    materialised oracle row (blog.euler0525.cn, the three invariants after block j)."""
    r = _rng(11)
    for n in range(1, 13):
        d = 3
        q = r.standard_normal((1, 1, n, d))
        k = r.standard_normal((1, 1, n, d)) * 2.0
        v = r.standard_normal((1, 1, n, d))
        scale = 0.7
        o, lse = orc.forward_f64(q, k, v, causal=False, scale=scale)
        for i in range(n):
            s = scale * (k[0, 0] @ q[0, 0, i])
            for c1 in range(0, n + 1):
                for c2 in range(c1, n + 1):
                    O, m, l, _ = online_softmax_tiles(s, v[0, 0], [c1, c2])
                    assert np.max(np.abs(O - o[0, 0, i])) <= 1e-12
                    assert abs(m + math.log(l) - lse[0, 0, i]) <= 1e-12


def check_prob_rows(orc):
    r = _rng(12)
    for causal in (False, True):
        q = r.standard_normal((2, 2, 9, 4))
        k = r.standard_normal((2, 2, 9, 4))
        P = orc.probs_f64(q, k, causal=causal, scale=0.9)
        assert np.all(P >= 0.0)
        assert np.max(np.abs(P.sum(-1) - 1.0)) <= 1e-12
        if causal:
            assert np.all(np.triu(P, 1) == 0.0)
            assert np.all(np.diagonal(P, axis1=-2, axis2=-1) > 0.0)
        else:
            assert np.all(P > 0.0)


# ---------------------------------------------------------------------------------------
# Closed forms

def check_constant_v(orc):
    r = _rng(13)
    for causal in (False, True):
        q = r.standard_normal((1, 2, 7, 5)) * 3
        k = r.standard_normal((1, 2, 7, 5)) * 3
        row = r.standard_normal(5)
        v = np.broadcast_to(row, (1, 2, 7, 5)).copy()
        o, _ = orc.forward_f64(q, k, v, causal=causal, scale=0.5)
        assert np.max(np.abs(o - row)) <= 1e-13


def check_zero_q(orc):
    r = _rng(14)
    N = 10
    q = np.zeros((1, 1, N, 4))
    k = r.standard_normal((1, 1, N, 4))
    v = r.standard_normal((1, 1, N, 4))
    o, lse = orc.forward_f64(q, k, v, causal=False, scale=1.3)
    assert np.max(np.abs(lse - math.log(N))) <= 1e-13
    assert np.max(np.abs(o[0, 0] - v[0, 0].mean(0))) <= 1e-13
    o, lse = orc.forward_f64(q, k, v, causal=True, scale=1.3)
    for i in range(N):
        assert abs(lse[0, 0, i] - math.log(i + 1)) <= 1e-13
        assert np.max(np.abs(o[0, 0, i] - v[0, 0, : i + 1].mean(0))) <= 1e-13


def check_single_visible_key(orc):
    r = _rng(15)
    q = r.standard_normal((1, 1, 1, 6))
    k = r.standard_normal((1, 1, 1, 6))
    v = r.standard_normal((1, 1, 1, 6))
    for causal in (False, True):
        o, lse = orc.forward_f64(q, k, v, causal=causal, scale=0.4)
        assert np.max(np.abs(o - v)) <= 1e-15
        assert abs(lse[0, 0, 0] - 0.4 * float(q[0, 0, 0] @ k[0, 0, 0])) <= 1e-14
    # Causal row 0 sees key 0 only, whatever the other keys hold.
    q = r.standard_normal((1, 1, 5, 6))
    k = r.standard_normal((1, 1, 5, 6))
    v = r.standard_normal((1, 1, 5, 6))
    o, lse = orc.forward_f64(q, k, v, causal=True, scale=0.4)
    assert np.max(np.abs(o[0, 0, 0] - v[0, 0, 0])) <= 1e-15
    assert abs(lse[0, 0, 0] - 0.4 * float(q[0, 0, 0] @ k[0, 0, 0])) <= 1e-14


def check_causality(orc):
    """Changing keys/values after position i leaves causal rows <= i unchanged."""
    r = _rng(16)
    q = r.standard_normal((1, 1, 8, 4))
    k = r.standard_normal((1, 1, 8, 4))
    v = r.standard_normal((1, 1, 8, 4))
    o, lse = orc.forward_f64(q, k, v, causal=True, scale=0.8)
    for i in range(7):
        k2, v2 = k.copy(), v.copy()
        k2[0, 0, i + 1:] = r.standard_normal((7 - i, 4)) * 5
        v2[0, 0, i + 1:] = r.standard_normal((7 - i, 4)) * 5
        o2, lse2 = orc.forward_f64(q, k2, v2, causal=True, scale=0.8)
        assert np.max(np.abs(o2[0, 0, : i + 1] - o[0, 0, : i + 1])) <= 1e-15
        assert np.max(np.abs(lse2[0, 0, : i + 1] - lse[0, 0, : i + 1])) <= 1e-15
        # ... while the next row does change.
        assert np.max(np.abs(o2[0, 0, i + 1] - o[0, 0, i + 1])) > 1e-6


def check_permutation_invariance(orc):
    r = _rng(17)
    q = r.standard_normal((1, 1, 11, 5))
    k = r.standard_normal((1, 1, 11, 5))
    v = r.standard_normal((1, 1, 11, 5))
    o, lse = orc.forward_f64(q, k, v, causal=False, scale=0.6)
    perm = r.permutation(11)
    o2, lse2 = orc.forward_f64(q, k[:, :, perm], v[:, :, perm], causal=False, scale=0.6)
    assert np.max(np.abs(o2 - o)) <= 1e-13
    assert np.max(np.abs(lse2 - lse)) <= 1e-13


def check_scale_zero_is_mean(orc):
    r = _rng(18)
    q = r.standard_normal((1, 1, 6, 3)) * 10
    k = r.standard_normal((1, 1, 6, 3)) * 10
    v = r.standard_normal((1, 1, 6, 3))
    o, lse = orc.forward_f64(q, k, v, causal=False, scale=0.0)
    assert np.max(np.abs(o[0, 0] - v[0, 0].mean(0))) <= 1e-14
    assert np.max(np.abs(lse - math.log(6))) <= 1e-14


def check_library_softmax(orc):
    """Library routines: scipy's logsumexp and softmax on numpy's matmul."""
    from scipy.special import logsumexp, softmax
    r = _rng(19)
    q = r.standard_normal((2, 3, 13, 8))
    k = r.standard_normal((2, 3, 13, 8))
    v = r.standard_normal((2, 3, 13, 8))
    for causal in (False, True):
        o, lse = orc.forward_f64(q, k, v, causal=causal, scale=0.35)
        s = 0.35 * np.einsum("bhie,bhje->bhij", q, k)
        if causal:
            s = np.where(np.tril(np.ones((13, 13), dtype=bool)), s, -np.inf)
        assert np.max(np.abs(lse - logsumexp(s, axis=-1))) <= 1e-12
        assert np.max(np.abs(o - softmax(s, axis=-1) @ v)) <= 1e-12


def check_large_scores_stable(orc):
    """Scores of size ~1e3 (no overflow thanks to the max subtraction): O stays a convex
    combination of V rows and LSE stays finite and >= the row max."""
    r = _rng(20)
    q = r.standard_normal((1, 1, 6, 4)) * 30
    k = r.standard_normal((1, 1, 6, 4)) * 30
    v = r.standard_normal((1, 1, 6, 4))
    o, lse = orc.forward_f64(q, k, v, causal=False, scale=1.0)
    s = np.einsum("ie,je->ij", q[0, 0], k[0, 0])
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert np.all(lse[0, 0] >= s.max(-1) - 1e-9)
    assert np.all(lse[0, 0] <= s.max(-1) + math.log(6) + 1e-9)
    assert np.all(o[0, 0] <= v[0, 0].max(0) + 1e-12) and np.all(o[0, 0] >= v[0, 0].min(0) - 1e-12)


# ---------------------------------------------------------------------------------------
# Backward

def _loss(orc, q, k, v, dout, causal, scale):
    o, _ = orc.forward_f64(q, k, v, causal=causal, scale=scale)
    return float(np.sum(o * dout))


def check_backward_finite_differences(orc):
    """Central differences of L = sum(O * dO); pins every gradient including the scale."""
    r = _rng(21)
    h = 1e-5
    for (N, d, causal, scale) in ((5, 3, False, 0.8), (7, 4, True, 1.7), (9, 2, True, 0.45)):
        q = r.standard_normal((1, 1, N, d))
        k = r.standard_normal((1, 1, N, d))
        v = r.standard_normal((1, 1, N, d))
        dout = r.standard_normal((1, 1, N, d))
        dq, dk, dv = orc.backward_f64(q, k, v, dout, causal=causal, scale=scale)
        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp = x.copy()
                xm = x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": q, "k": k, "v": v}
                args_m = {"q": q, "k": k, "v": v}
                args_p[name] = xp
                args_m[name] = xm
                num[idx] = (_loss(orc, args_p["q"], args_p["k"], args_p["v"], dout, causal, scale)
                            - _loss(orc, args_m["q"], args_m["k"], args_m["v"], dout, causal,
                                    scale)) / (2 * h)
            err = np.max(np.abs(num - g)) / max(1.0, np.max(np.abs(g)))
            assert err <= 1e-6, (name, N, d, causal, err)


def check_backward_identities(orc):
    """D_i = O_i . dO_i makes every row of dS sum to zero, so the key-gradient rows sum to
    zero; rows of P summing to one make the value-gradient rows sum to sum_i dO_i."""
    r = _rng(22)
    for causal in (False, True):
        q = r.standard_normal((2, 2, 12, 5))
        k = r.standard_normal((2, 2, 12, 5))
        v = r.standard_normal((2, 2, 12, 5))
        dout = r.standard_normal((2, 2, 12, 5))
        dq, dk, dv = orc.backward_f64(q, k, v, dout, causal=causal, scale=0.7)
        assert np.max(np.abs(dk.sum(2))) <= 1e-12
        assert np.max(np.abs(dv.sum(2) - dout.sum(2))) <= 1e-12
        if causal:
            # The last key is seen by the last query only.
            P = orc.probs_f64(q, k, causal=True, scale=0.7)
            assert np.max(np.abs(dv[:, :, -1] - P[:, :, -1, -1, None] * dout[:, :, -1])) <= 1e-13


def check_backward_linear_in_dout(orc):
    r = _rng(23)
    q, k, v, d1, d2 = (r.standard_normal((1, 2, 6, 3)) for _ in range(5))
    g1 = orc.backward_f64(q, k, v, d1, causal=True, scale=0.9)
    g2 = orc.backward_f64(q, k, v, d2, causal=True, scale=0.9)
    g3 = orc.backward_f64(q, k, v, 2.0 * d1 - d2, causal=True, scale=0.9)
    for a, b, c in zip(g1, g2, g3):
        assert np.max(np.abs(c - (2.0 * a - b))) <= 1e-12


# ---------------------------------------------------------------------------------------
# Entry points agree with each other (bf16 widening, sampled rows)

def check_entry_points_agree(orc):
    from exact_io_aware_fa_gb300 import synthetic as syn
    B, H, N, d = 1, 2, 37, 8
    x = syn.attention_inputs(B, H, N, d, seed=99, with_dout=True)
    f = {kk: syn.bf16_bits_to_float64(vv) for kk, vv in x.items()}
    rows = np.array([0, 5, 17, 36])
    for causal in (False, True):
        o, lse = orc.forward_bf16(x["q"], x["k"], x["v"], causal=causal, scale=0.3)
        o64, lse64 = orc.forward_f64(f["q"], f["k"], f["v"], causal=causal, scale=0.3)
        assert np.array_equal(o, o64) and np.array_equal(lse, lse64)
        orow, lrow = orc.forward_rows_bf16(x["q"], x["k"], x["v"], causal, 0.3, rows)
        assert np.array_equal(orow, o[:, :, rows]) and np.array_equal(lrow, lse[:, :, rows])
        g = orc.backward_bf16(x["q"], x["k"], x["v"], x["do"], causal=causal, scale=0.3)
        g64 = orc.backward_f64(f["q"], f["k"], f["v"], f["do"], causal=causal, scale=0.3)
        for a, b in zip(g, g64):
            assert np.array_equal(a, b)
        sq, sk, sv = orc.backward_rows_bf16(x["q"], x["k"], x["v"], x["do"], causal, 0.3,
                                            rows, rows[::-1])
        assert np.max(np.abs(sq - g[0][:, :, rows])) <= 1e-12
        assert np.max(np.abs(sk - g[1][:, :, rows[::-1]])) <= 1e-12
        assert np.max(np.abs(sv - g[2][:, :, rows[::-1]])) <= 1e-12


# ---------------------------------------------------------------------------------------
# Extension: grouped KV heads, query offset (bottom-right alignment), sliding window

def check_ex_reduces_to_mha(orc):
    """Hq = Hkv, Tq = Tk, no window: the extended entry points equal the plain ones."""
    r = _rng(30)
    for causal in (False, True):
        q, k, v, dout = (r.standard_normal((2, 3, 10, 4)) for _ in range(4))
        o, lse = orc.forward_f64(q, k, v, causal=causal, scale=0.6)
        oe, lsee = orc.forward_ex(q, k, v, causal, 0.6)
        assert np.max(np.abs(oe - o)) <= 1e-14 and np.max(np.abs(lsee - lse)) <= 1e-14
        g = orc.backward_f64(q, k, v, dout, causal=causal, scale=0.6)
        ge = orc.backward_ex(q, k, v, dout, causal, 0.6)
        for a, b in zip(ge, g):
            assert np.max(np.abs(a - b)) <= 1e-13


def check_ex_gqa_equals_repeated_kv(orc):
    """Query head h reads KV head h // group: same as multi-head attention with every KV head
    repeated `group` times; its dK/dV are the sums over the group."""
    r = _rng(31)
    B, Hkv, group, T, d = 2, 2, 3, 9, 4
    q = r.standard_normal((B, Hkv * group, T, d))
    k = r.standard_normal((B, Hkv, T, d))
    v = r.standard_normal((B, Hkv, T, d))
    dout = r.standard_normal((B, Hkv * group, T, d))
    kr, vr = np.repeat(k, group, axis=1), np.repeat(v, group, axis=1)
    for causal in (False, True):
        o, lse = orc.forward_f64(q, kr, vr, causal=causal, scale=0.7)
        oe, lsee = orc.forward_ex(q, k, v, causal, 0.7)
        assert np.max(np.abs(oe - o)) <= 1e-13 and np.max(np.abs(lsee - lse)) <= 1e-13
        dq, dk, dv = orc.backward_f64(q, kr, vr, dout, causal=causal, scale=0.7)
        dqe, dke, dve = orc.backward_ex(q, k, v, dout, causal, 0.7)
        assert np.max(np.abs(dqe - dq)) <= 1e-12
        assert np.max(np.abs(dke - dk.reshape(B, Hkv, group, T, d).sum(2))) <= 1e-12
        assert np.max(np.abs(dve - dv.reshape(B, Hkv, group, T, d).sum(2))) <= 1e-12


def check_ex_query_offset_bottom_right(orc):
    """Tq < Tk, causal: query row i sits at key position Tk - Tq + i, so the rows equal the
    last Tq rows of a full causal attention whose last queries are these."""
    r = _rng(32)
    Tq, Tk, d = 5, 12, 3
    q = r.standard_normal((1, 2, Tq, d))
    k = r.standard_normal((1, 2, Tk, d))
    v = r.standard_normal((1, 2, Tk, d))
    qf = r.standard_normal((1, 2, Tk, d))
    qf[:, :, Tk - Tq:] = q
    of, lf = orc.forward_f64(qf, k, v, causal=True, scale=0.9)
    oe, le = orc.forward_ex(q, k, v, True, 0.9)
    assert np.max(np.abs(oe - of[:, :, Tk - Tq:])) <= 1e-14
    assert np.max(np.abs(le - lf[:, :, Tk - Tq:])) <= 1e-14
    # Non-causal rows do not depend on the offset: every key is visible.
    o2, l2 = orc.forward_ex(q, k, v, False, 0.9)
    s = 0.9 * np.einsum("bhie,bhje->bhij", q, k)
    from scipy.special import logsumexp, softmax
    assert np.max(np.abs(l2 - logsumexp(s, -1))) <= 1e-12
    assert np.max(np.abs(o2 - softmax(s, -1) @ v)) <= 1e-12
    # A query before the first key (Tq > Tk, causal) has nothing to attend to.
    try:
        orc.forward_ex(r.standard_normal((1, 1, 6, d)), k[:, :1, :4], v[:, :1, :4], True, 0.9)
    except ValueError:
        pass
    else:
        raise AssertionError("a row with no visible key was accepted")


def check_ex_sliding_window(orc):
    """Window w: key j visible iff pos - w <= j <= pos ("15. FlashAttention", stretch item 3:
    tiles wholly before q_pos - window are skipped)."""
    from scipy.special import logsumexp, softmax
    r = _rng(33)
    Tq, Tk, d = 7, 10, 3
    q = r.standard_normal((1, 2, Tq, d))
    k = r.standard_normal((1, 2, Tk, d))
    v = r.standard_normal((1, 2, Tk, d))
    # window 0: each row sees only the key at its own position
    o, lse = orc.forward_ex(q, k, v, True, 0.8, window=0)
    pos = np.arange(Tq) + (Tk - Tq)
    assert np.max(np.abs(o - v[:, :, pos])) <= 1e-15
    s_own = 0.8 * np.einsum("bhie,bhie->bhi", q, k[:, :, pos])
    assert np.max(np.abs(lse - s_own)) <= 1e-14
    # window >= Tk: plain causal
    o1, l1 = orc.forward_ex(q, k, v, True, 0.8, window=Tk)
    o2, l2 = orc.forward_ex(q, k, v, True, 0.8)
    assert np.max(np.abs(o1 - o2)) <= 1e-15 and np.max(np.abs(l1 - l2)) <= 1e-15
    # window 3 against scipy on the explicit mask
    w = 3
    s = 0.8 * np.einsum("bhie,bhje->bhij", q, k)
    j = np.arange(Tk)[None, :]
    vis = (j <= pos[:, None]) & (j >= pos[:, None] - w)
    s = np.where(vis, s, -np.inf)
    o3, l3 = orc.forward_ex(q, k, v, True, 0.8, window=w)
    assert np.max(np.abs(l3 - logsumexp(s, -1))) <= 1e-12
    assert np.max(np.abs(o3 - softmax(s, -1) @ v)) <= 1e-12
    # a window without the causal mask is not defined here
    try:
        orc.forward_ex(q, k, v, False, 0.8, window=2)
    except (ValueError, RuntimeError):
        pass
    else:
        raise AssertionError("window without causal accepted")


def check_ex_backward_finite_differences(orc):
    """Gradients of the extended forward (GQA + offset + window) by central differences."""
    r = _rng(34)
    h = 1e-5
    B, Hkv, group, Tq, Tk, d = 1, 1, 2, 4, 7, 2
    q = r.standard_normal((B, Hkv * group, Tq, d))
    k = r.standard_normal((B, Hkv, Tk, d))
    v = r.standard_normal((B, Hkv, Tk, d))
    dout = r.standard_normal((B, Hkv * group, Tq, d))
    for window in (-1, 2):
        dq, dk, dv = orc.backward_ex(q, k, v, dout, True, 1.3, window=window)

        def loss(qq, kk, vv):
            o, _ = orc.forward_ex(qq, kk, vv, True, 1.3, window=window)
            return float(np.sum(o * dout))

        for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                a = {"q": q, "k": k, "v": v}
                b = dict(a)
                a[name], b[name] = xp, xm
                num[idx] = (loss(a["q"], a["k"], a["v"]) - loss(b["q"], b["k"], b["v"])) / (2 * h)
            err = np.max(np.abs(num - g)) / max(1.0, np.max(np.abs(g)))
            assert err <= 1e-6, (name, window, err)


def check_ex_backward_sensitivities(orc):
    """The gradient sensitivities (the parity tests' bound for bf16 rounding of P and dS)
    against a brute-force numpy restatement of the definitions on a tiny GQA + offset + window
    case, the closed form sum_j sv_je = sum_i |dO_ie| (rows of P sum to 1), and the gradients
    returned beside them equal backward_ex's."""
    r = _rng(35)
    B, Hkv, group, Tq, Tk, d = 2, 2, 3, 5, 9, 4
    Hq = Hkv * group
    bits = {}
    vals = {}
    for name, shape in (("q", (B, Hq, Tq, d)), ("k", (B, Hkv, Tk, d)), ("v", (B, Hkv, Tk, d)),
                        ("do", (B, Hq, Tq, d))):
        x = np.round(r.standard_normal(shape) * 8) / 8  # exact in bf16
        vals[name], bits[name] = x, _to_bf16_bits(x)
    scale = 0.6
    for causal, window in ((False, -1), (True, -1), (True, 3)):
        (dq, dk, dv), (sq, sk, sv) = orc.backward_ex_sens(bits["q"], bits["k"], bits["v"],
                                                          bits["do"], causal, scale, window)
        ref = orc.backward_ex(bits["q"], bits["k"], bits["v"], bits["do"], causal, scale, window)
        for a, b in zip((dq, dk, dv), ref):
            assert np.array_equal(a, b), (causal, window)
        bq, bk, bv = np.zeros_like(sq), np.zeros_like(sk), np.zeros_like(sv)
        for b_ in range(B):
            for h in range(Hq):
                hk = h // group
                qh, kh, vh, doh = (vals["q"][b_, h], vals["k"][b_, hk], vals["v"][b_, hk],
                                   vals["do"][b_, h])
                pos = np.arange(Tq)[:, None] + (Tk - Tq)
                j = np.arange(Tk)[None, :]
                vis = np.ones((Tq, Tk), dtype=bool)
                if causal:
                    vis &= j <= pos
                if window >= 0:
                    vis &= j >= pos - window
                s = np.where(vis, scale * qh @ kh.T, -np.inf)
                P = np.exp(s - s.max(axis=1, keepdims=True))
                P /= P.sum(axis=1, keepdims=True)
                dP = doh @ vh.T
                dS = P * (dP - (P * dP).sum(axis=1, keepdims=True))
                bv[b_, hk] += P.T @ np.abs(doh)
                bk[b_, hk] += scale * np.abs(dS).T @ np.abs(qh)
                bq[b_, h] = scale * np.abs(dS) @ np.abs(kh)
        for name, a, b in (("sq", sq, bq), ("sk", sk, bk), ("sv", sv, bv)):
            assert np.allclose(a, b, rtol=1e-12, atol=1e-12), (name, causal, window)
        col = np.abs(vals["do"]).reshape(B, Hkv, group * Tq, d).sum(axis=2)
        assert np.allclose(sv.sum(axis=2), col, rtol=1e-12, atol=1e-12), (causal, window)


def check_split_merge_equals_unsplit(orc):
    """Flash-decoding: partials over any chunking of the keys (including empty chunks and
    chunks some rows cannot see) merge to the unsplit attention ("15. FlashAttention",
    section "Decode is different: flash-decoding")."""
    r = _rng(40)
    B, Hkv, group, Tq, Tk, d = 1, 2, 2, 6, 23, 3
    q = r.standard_normal((B, Hkv * group, Tq, d))
    k = r.standard_normal((B, Hkv, Tk, d))
    v = r.standard_normal((B, Hkv, Tk, d))
    for causal, window in ((False, -1), (True, -1), (True, 4)):
        o_ref, lse_ref = orc.forward_ex(q, k, v, causal, 0.7, window)
        for bounds in ([0, Tk], [0, 11, Tk], [0, 0, 5, 5, 17, Tk], [0, 1, 2, 3, 20, Tk],
                       list(range(0, Tk + 1))):
            m, l, a = oracle.partials_f64(q, k, v, causal, 0.7, window, bounds)
            _, _, _, o, lse = oracle.merge_partials(m, l, a)
            assert np.allclose(o, o_ref, rtol=0, atol=1e-12), (causal, window, bounds)
            assert np.allclose(lse, lse_ref, rtol=0, atol=1e-12), (causal, window, bounds)


def check_merge_is_associative(orc):
    """Merging partials in any grouping gives the same (m, l, a) (the page states the rule is
    associative); a merged triple is itself a partial."""
    r = _rng(41)
    q = r.standard_normal((1, 1, 4, 3))
    k = r.standard_normal((1, 1, 30, 3))
    v = r.standard_normal((1, 1, 30, 3))
    m, l, a = oracle.partials_f64(q, k, v, True, 1.3, -1, [0, 7, 9, 21, 30])
    whole = oracle.merge_partials(m, l, a)
    left = oracle.merge_partials(m[:2], l[:2], a[:2])
    right = oracle.merge_partials(m[2:], l[2:], a[2:])
    grouped = oracle.merge_partials(np.stack([left[0], right[0]]), np.stack([left[1], right[1]]),
                                    np.stack([left[2], right[2]]))
    for x, y in zip(whole, grouped):
        assert np.allclose(x, y, rtol=1e-13, atol=1e-13)
    # the merged max is the largest partial max; l >= the l of the chunk holding it
    assert np.array_equal(whole[0], m.max(axis=0))


ALL_CHECKS = [
    check_worked_example_oracle,
    check_worked_example_two_tiles,
    check_online_every_split,
    check_prob_rows,
    check_constant_v,
    check_zero_q,
    check_single_visible_key,
    check_causality,
    check_permutation_invariance,
    check_scale_zero_is_mean,
    check_library_softmax,
    check_large_scores_stable,
    check_backward_finite_differences,
    check_backward_identities,
    check_backward_linear_in_dout,
    check_entry_points_agree,
    check_ex_reduces_to_mha,
    check_ex_gqa_equals_repeated_kv,
    check_ex_query_offset_bottom_right,
    check_ex_sliding_window,
    check_ex_backward_finite_differences,
    check_ex_backward_sensitivities,
    check_split_merge_equals_unsplit,
    check_merge_is_associative,
]
