"""Pins for the Gated Delta Net oracle (oracle/gdn_ref.c), none of which re-types its recurrence.

* alpha = 1, beta = 0: the state never moves, o_t = scale * S0 q_t;
* beta = 0: pure decay, o_t = scale * (prod alpha) * S0 q_t;
* one token from a zero state: o = scale * beta * (k . q) * v;
* beta = 1 with a unit key: after the update the state maps k_t to v_t exactly, whatever it
  held before (the delta rule's defining property), and with orthonormal keys every earlier
  (k_s, v_s) pair stays recallable;
* the product form S_t = alpha S_{t-1} (I - beta k k^T) + beta v k^T, an algebraically different
  statement of the same recurrence, in exact rational arithmetic on tiny shapes;
* invariances: packing sequences equals running them one by one, and grouped value heads equal
  multi-head attention with the query/key heads repeated;
* planted mistakes in a numpy copy, each of which some pin must catch.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest

import oracle


def _rand(rng, T, h_qk, h_v, dk, dv):
    q = rng.standard_normal((T, h_qk, dk))
    k = rng.standard_normal((T, h_qk, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, h_v, dv))
    a = rng.uniform(0.8, 1.0, (T, h_v))
    b = rng.uniform(0.0, 1.0, (T, h_v))
    return q, k, v, a, b


def _oracle(q, k, v, a, b, cu, scale, s0=None):
    return oracle.gdn_f64(q, k, v, a, b, cu, scale, s0)


# ---- pins written as functions of a gdn(q, k, v, a, b, cu, scale, s0) callable -----------------

def pin_frozen_state(gdn):
    rng = np.random.default_rng(1)
    q, k, v, a, b = _rand(rng, 7, 2, 2, 5, 4)
    a[:] = 1.0
    b[:] = 0.0
    s0 = rng.standard_normal((1, 2, 4, 5))
    o, sf = gdn(q, k, v, a, b, [0, 7], 0.73, s0)
    want = 0.73 * np.einsum("hvk,thk->thv", s0[0], q)
    return int(not np.allclose(o, want, rtol=1e-14, atol=1e-14)) + \
        int(not np.array_equal(sf, s0))


def pin_pure_decay(gdn):
    rng = np.random.default_rng(2)
    q, k, v, a, b = _rand(rng, 6, 1, 1, 4, 4)
    b[:] = 0.0
    s0 = rng.standard_normal((1, 1, 4, 4))
    o, sf = gdn(q, k, v, a, b, [0, 6], 1.5, s0)
    g = np.cumprod(a[:, 0])
    want = 1.5 * g[:, None] * np.einsum("vk,tk->tv", s0[0, 0], q[:, 0])
    return int(not np.allclose(o[:, 0], want, rtol=1e-13, atol=1e-14)) + \
        int(not np.allclose(sf[0, 0], g[-1] * s0[0, 0], rtol=1e-13, atol=0))


def pin_single_token(gdn):
    rng = np.random.default_rng(3)
    q, k, v, a, b = _rand(rng, 1, 1, 1, 6, 3)
    o, sf = gdn(q, k, v, a, b, [0, 1], 0.5, None)
    want = 0.5 * b[0, 0] * float(k[0, 0] @ q[0, 0]) * v[0, 0]
    return int(not np.allclose(o[0, 0], want, rtol=1e-14, atol=1e-15)) + \
        int(not np.allclose(sf[0, 0], b[0, 0] * np.outer(v[0, 0], k[0, 0]), rtol=1e-14,
                            atol=1e-15))


def pin_delta_rule_writes_v_at_k(gdn):
    """beta = 1 and k = a basis vector: the prediction error is fully corrected, so with q = k the
    output is exactly scale * v, for any earlier state and decay."""
    rng = np.random.default_rng(4)
    T, d = 6, 5
    q, k, v, a, b = _rand(rng, T, 1, 1, d, d)
    b[:] = 1.0
    k[:] = 0.0
    for t in range(T):
        k[t, 0, t % d] = 1.0
    q[:] = k
    s0 = rng.standard_normal((1, 1, d, d))
    o, _ = gdn(q, k, v, a, b, [0, T], 0.73, s0)
    return int(not np.allclose(o[:, 0], 0.73 * v[:, 0], rtol=1e-13, atol=1e-13))


def pin_orthonormal_recall(gdn):
    """alpha = beta = 1, orthonormal keys e_0..e_{T-1}, zero start: at token t the state maps
    every earlier key e_s to v_s, so querying e_s returns scale * v_s exactly."""
    rng = np.random.default_rng(5)
    T, d = 5, 6
    q, k, v, a, b = _rand(rng, T, 1, 1, d, 3)
    a[:] = 1.0
    b[:] = 1.0
    k[:] = 0.0
    for t in range(T):
        k[t, 0, t] = 1.0
    fails = 0
    for s in range(T):
        q[:] = 0.0
        q[:, 0, s] = 1.0
        o, _ = gdn(q, k, v, a, b, [0, T], 2.0, None)
        for t in range(T):
            want = 2.0 * v[s, 0] if t >= s else np.zeros(3)
            fails += int(not np.array_equal(o[t, 0], want))
    return fails


def pin_product_form_exact(gdn):
    """S_t = alpha S_{t-1} (I - beta k k^T) + beta v k^T in rationals; o_t = scale S_t q_t."""
    rng = np.random.default_rng(6)
    fails = 0
    for (T, dk, dv) in ((3, 2, 2), (4, 3, 2), (2, 2, 3)):
        ints = lambda *shape: rng.integers(-4, 5, size=shape).astype(np.float64) / 4.0
        q, k, v = ints(T, 1, dk), ints(T, 1, dk), ints(T, 1, dv)
        a = rng.integers(2, 5, size=(T, 1)).astype(np.float64) / 4.0
        b = rng.integers(0, 5, size=(T, 1)).astype(np.float64) / 4.0
        s0 = ints(1, 1, dv, dk)
        o, sf = gdn(q, k, v, a, b, [0, T], 0.75, s0)
        S = [[Fraction(x) for x in row] for row in s0[0, 0]]
        for t in range(T):
            kt = [Fraction(x) for x in k[t, 0]]
            al, be = Fraction(a[t, 0]), Fraction(b[t, 0])
            P = [[(1 if i == j else 0) - be * kt[i] * kt[j] for j in range(dk)] for i in range(dk)]
            S = [[al * sum(S[r][m] * P[m][c] for m in range(dk)) + be * Fraction(v[t, 0, r]) * kt[c]
                  for c in range(dk)] for r in range(dv)]
            for r in range(dv):
                want = Fraction(3, 4) * sum(S[r][c] * Fraction(q[t, 0, c]) for c in range(dk))
                fails += int(abs(Fraction(o[t, 0, r]) - want) > Fraction(1, 2 ** 48))
        for r in range(dv):
            for c in range(dk):
                fails += int(abs(Fraction(sf[0, 0, r, c]) - S[r][c]) > Fraction(1, 2 ** 48))
    return fails


def pin_packing_is_independent_runs(gdn):
    rng = np.random.default_rng(7)
    lens = [3, 1, 5, 2]
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, a, b = _rand(rng, int(cu[-1]), 2, 2, 4, 3)
    s0 = rng.standard_normal((len(lens), 2, 3, 4))
    o, sf = gdn(q, k, v, a, b, cu, 0.9, s0)
    fails = 0
    for i in range(len(lens)):
        sl = slice(cu[i], cu[i + 1])
        oi, sfi = gdn(q[sl], k[sl], v[sl], a[sl], b[sl], [0, lens[i]], 0.9, s0[i:i + 1])
        fails += int(not np.allclose(o[sl], oi, rtol=1e-14, atol=1e-15))
        fails += int(not np.allclose(sf[i], sfi[0], rtol=1e-14, atol=1e-15))
    return fails


def pin_grouped_values_equal_repeated_heads(gdn):
    rng = np.random.default_rng(8)
    T, hqk, g = 6, 2, 3
    q, k, v, a, b = _rand(rng, T, hqk, hqk * g, 4, 3)
    o, sf = gdn(q, k, v, a, b, [0, T], 0.6, None)
    qr, kr = np.repeat(q, g, axis=1), np.repeat(k, g, axis=1)
    o2, sf2 = gdn(qr, kr, v, a, b, [0, T], 0.6, None)
    return int(not np.array_equal(o, o2)) + int(not np.array_equal(sf, sf2))


PINS = [pin_frozen_state, pin_pure_decay, pin_single_token, pin_delta_rule_writes_v_at_k,
        pin_orthonormal_recall, pin_product_form_exact, pin_packing_is_independent_runs,
        pin_grouped_values_equal_repeated_heads]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_passes_pin(pin):
    assert pin(_oracle) == 0


def test_shape_checks():
    q = np.zeros((4, 2, 3))
    v = np.zeros((4, 3, 3))
    ab = np.ones((4, 3))
    with pytest.raises(ValueError):      # h_v not a multiple of h_qk
        oracle.gdn_f64(q, q, v, ab, ab, [0, 4], 1.0)
    v = np.zeros((4, 2, 3))
    ab = np.ones((4, 2))
    with pytest.raises(ValueError):      # offsets must end at T
        oracle.gdn_f64(q, q, v, ab, ab, [0, 3], 1.0)
    with pytest.raises(ValueError):      # wrong initial-state shape
        oracle.gdn_f64(q, q, v, ab, ab, [0, 4], 1.0, np.zeros((1, 2, 3, 2)))
    o, sf = oracle.gdn_f64(q[:0], q[:0], v[:0], ab[:0], ab[:0], [0], 1.0)
    assert o.shape == (0, 2, 3) and sf.shape == (0, 2, 3, 3)


def test_empty_sequence_keeps_its_initial_state():
    rng = np.random.default_rng(9)
    q, k, v, a, b = _rand(rng, 3, 1, 1, 2, 2)
    s0 = rng.standard_normal((2, 1, 2, 2))
    _, sf = oracle.gdn_f64(q, k, v, a, b, [0, 0, 3], 1.0, s0)
    assert np.array_equal(sf[0], s0[0])


# ---- planted mistakes ------------------------------------------------------------------------------

def _np_gdn(mutant=None):
    def gdn(q, k, v, a, b, cu, scale, s0=None):
        q, k, v, a, b = (np.asarray(x, dtype=np.float64) for x in (q, k, v, a, b))
        T, hqk, dk = q.shape
        hv, dv = v.shape[1], v.shape[2]
        n = len(cu) - 1
        o = np.zeros((T, hv, dv))
        sf = np.zeros((n, hv, dv, dk))
        for i in range(n):
            for j in range(hv):
                H = np.zeros((dv, dk)) if s0 is None else np.array(s0[i, j], dtype=np.float64)
                jq = j // (hv // hqk)
                for t in range(cu[i], cu[i + 1]):
                    kt, qt, vt = k[t, jq], q[t, jq], v[t, j]
                    Hd = a[t, j] * H
                    pred = (H if mutant == "pred_from_undecayed" else Hd) @ kt
                    upd = (vt - pred) if mutant == "no_beta" else b[t, j] * (vt - pred)
                    if mutant == "outer_transposed" and dv == dk:   # only square states
                        Hn = Hd + np.outer(kt, upd)
                    elif mutant == "decay_after_update":
                        Hn = a[t, j] * (H + np.outer(b[t, j] * (vt - H @ kt), kt))
                    else:
                        Hn = Hd + np.outer(upd, kt)
                    Hout = Hd if mutant == "output_before_update" else Hn
                    o[t, j] = (1.0 if mutant == "no_scale" else scale) * (Hout @ qt)
                    H = Hn
                sf[i, j] = H
        return o, sf
    return gdn


MUTANTS = ["pred_from_undecayed", "no_beta", "outer_transposed", "decay_after_update",
           "output_before_update", "no_scale"]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_pins_catch_planted_mistakes(mutant):
    g = _np_gdn(mutant)
    assert sum(pin(g) for pin in PINS) >= 1, f"no pin caught {mutant}"


def test_unmutated_numpy_copy_passes_every_pin():
    g = _np_gdn(None)
    assert all(pin(g) == 0 for pin in PINS)


# ---- grouped queries (GQA) and mixed layouts ---------------------------------------------------
# q: [T, h_q, dk], k: [T, h_k, dk], v: [T, h_v, dv].  With h_q a multiple of h_v, query head m
# reads state m / (h_q / h_v) and has its own output.  Each pin reduces a grouped layout to
# single-head runs, which the pins above fix.

def _rand_heads(rng, T, h_q, h_k, h_v, dk, dv):
    q = rng.standard_normal((T, h_q, dk))
    k = rng.standard_normal((T, h_k, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, h_v, dv))
    a = rng.uniform(0.8, 1.0, (T, h_v))
    b = rng.uniform(0.0, 1.0, (T, h_v))
    return q, k, v, a, b


def _single_head_runs(gdn, q, k, v, a, b, cu, scale, s0, state_of, key_of):
    """Outputs and states of every query head m run alone with its state's key, value, decays."""
    h_q, h_v = q.shape[1], v.shape[1]
    outs = []
    for m in range(h_q):
        j = state_of(m)
        om, sm = gdn(q[:, m:m + 1], k[:, key_of(j):key_of(j) + 1], v[:, j:j + 1],
                     a[:, j:j + 1], b[:, j:j + 1], cu, scale,
                     None if s0 is None else s0[:, j:j + 1])
        outs.append((om[:, 0], sm[:, 0]))
    return outs


def pin_grouped_queries_are_single_head_runs(gdn):
    rng = np.random.default_rng(10)
    T, h_q, h_kv = 9, 6, 2
    q, k, v, a, b = _rand_heads(rng, T, h_q, h_kv, h_kv, 4, 3)
    cu = [0, 4, 9]
    s0 = rng.standard_normal((2, h_kv, 3, 4))
    o, sf = gdn(q, k, v, a, b, cu, 0.8, s0)
    r = h_q // h_kv
    fails = int(o.shape != (T, h_q, 3))
    for m, (om, sm) in enumerate(_single_head_runs(gdn, q, k, v, a, b, cu, 0.8, s0,
                                                  lambda m: m // r, lambda j: j)):
        fails += int(not np.array_equal(o[:, m], om))
        fails += int(not np.array_equal(sf[:, m // r], sm))
    return fails


def pin_mixed_layout_is_single_head_runs(gdn):
    """h_q = 4 query heads over h_v = 2 states that share h_k = 1 key head."""
    rng = np.random.default_rng(11)
    T = 7
    q, k, v, a, b = _rand_heads(rng, T, 4, 1, 2, 4, 4)
    o, sf = gdn(q, k, v, a, b, [0, T], 1.1, None)
    fails = int(o.shape != (T, 4, 4))
    for m, (om, sm) in enumerate(_single_head_runs(gdn, q, k, v, a, b, [0, T], 1.1, None,
                                                  lambda m: m // 2, lambda j: 0)):
        fails += int(not np.array_equal(o[:, m], om))
    return fails


GQA_PINS = [pin_grouped_queries_are_single_head_runs, pin_mixed_layout_is_single_head_runs]


@pytest.mark.parametrize("pin", GQA_PINS, ids=lambda p: p.__name__)
def test_oracle_passes_grouped_query_pin(pin):
    assert pin(_oracle) == 0


def test_head_layouts():
    assert oracle.gdn_out_heads(2, 2, 2) == 2      # MHA
    assert oracle.gdn_out_heads(2, 2, 6) == 6      # GVA
    assert oracle.gdn_out_heads(8, 2, 2) == 8      # GQA
    assert oracle.gdn_out_heads(4, 1, 2) == 4      # grouped queries over grouped values
    for bad in [(2, 4, 2), (3, 2, 2), (2, 1, 4), (6, 2, 4)]:
        with pytest.raises(ValueError):
            oracle.gdn_out_heads(*bad)


def _np_gdn_heads(mutant=None):
    """A numpy statement of the head layouts, with planted head-mapping mistakes."""
    def gdn(q, k, v, a, b, cu, scale, s0=None):
        q, k, v, a, b = (np.asarray(x, dtype=np.float64) for x in (q, k, v, a, b))
        T, hq, dk = q.shape
        hk, hv, dv = k.shape[1], v.shape[1], v.shape[2]
        ho = hv if hq == hk else hq
        r = 1 if ho == hv else hq // hv
        o = np.zeros((T, ho, dv))
        sf = np.zeros((len(cu) - 1, hv, dv, dk))
        for i in range(len(cu) - 1):
            for j in range(hv):
                H = np.zeros((dv, dk)) if s0 is None else np.array(s0[i, j], dtype=np.float64)
                jk = j // (hv // hk)
                for t in range(cu[i], cu[i + 1]):
                    kt, vt = k[t, jk], v[t, j]
                    Hd = a[t, j] * H
                    H = Hd + np.outer(b[t, j] * (vt - Hd @ kt), kt)
                    for g in range(r):
                        m = (j // (hv // hk)) if ho == hv else j * r + g
                        if mutant == "interleaved_queries" and ho != hv:
                            m = g * hv + j            # query m read from state m % h_v
                        if mutant == "first_query_only" and g > 0:
                            continue
                        o[t, (j if ho == hv else j * r + g)] = scale * (H @ q[t, m])
                sf[i, j] = H
        return o, sf
    return gdn


@pytest.mark.parametrize("mutant", ["interleaved_queries", "first_query_only"])
def test_grouped_query_pins_catch_planted_mistakes(mutant):
    g = _np_gdn_heads(mutant)
    assert sum(pin(g) for pin in GQA_PINS) >= 1, f"no pin caught {mutant}"


def test_unmutated_head_layout_copy_passes_the_grouped_query_pins():
    g = _np_gdn_heads(None)
    assert all(pin(g) == 0 for pin in GQA_PINS)
