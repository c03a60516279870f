"""Pins of the oracle's multilingual sampler ladder (CFG combine -> repetition
penalty -> temperature -> min_p -> top-p -> top-k -> draw in vocabulary order,
"Chatterbox -> ggml Port: Development Journal", the multilingual port's
sampling path): enumeration from the definitions on 16-entry vocabularies
(membership by counting comparisons, no sorting), reductions to the plain
sampler, and hand cases for each stage, including the repetition penalty's sign
rule that the journal records getting backwards."""

import math

import numpy as np

import oracle
from tests import test_oracle_ops as oo

F32 = np.float32


def _ladder_probs(zc, zu, w, seen, pen, T, min_p, top_p, k):
    """Selection probabilities of the ladder, straight from the definitions."""
    V = len(zc)
    w, pen, T, min_p, top_p = (float(F32(v)) for v in (w, pen, T, min_p, top_p))
    z = [float(zc[i]) for i in range(V)]
    if zu is not None and w != 0.0:
        z = [z[i] + w * (z[i] - float(zu[i])) for i in range(V)]
    if seen is not None and pen != 1.0:
        z = [(z[i] / pen if z[i] > 0 else z[i] * pen) if seen[i] else z[i] for i in range(V)]
    z = [v / T for v in z]
    m = max(z)
    p = [math.exp(v - m) for v in z]
    S = [True] * V
    if min_p > 0:
        S = [p[i] >= min(min_p, 1.0) for i in range(V)]
    if top_p < 1.0:
        mass = sum(p[i] for i in range(V) if S[i])
        S = [S[i] and sum(p[j] for j in range(V) if S[j] and (z[j] > z[i] or (z[j] == z[i] and j < i))) / mass < top_p
             for i in range(V)]
    n = sum(S)
    kk = n if k < 1 or k > n else k
    S = [S[i] and sum(1 for j in range(V) if S[j] and z[j] > z[i]) < kk for i in range(V)]
    q = np.array([p[i] if S[i] else 0.0 for i in range(V)])
    return q / q.sum()


def _check(zc, zu, w, seen, pen, T, min_p, top_p, k, n_grid=1 << 12):
    probs = _ladder_probs(zc, zu, w, seen, pen, T, min_p, top_p, k)
    cdf = np.cumsum(probs)
    counts = np.zeros(len(zc))
    for g in range(n_grid):
        u = g / n_grid
        tok, margin = oracle.sample_ladder(zc, zu, w, seen, pen, T, min_p, top_p, k, u)
        exp = min(int(np.searchsorted(cdf, u, side="right")), len(zc) - 1)
        while probs[exp] == 0:
            exp -= 1
        if tok != exp:
            assert margin < 1e-9, (w, pen, T, min_p, top_p, k, u, tok, exp)
        counts[tok] += 1
    assert np.all(np.abs(counts / n_grid - probs) <= 1.5 / n_grid + 1e-12)


def test_ladder_bruteforce_random_logits():
    rng = np.random.default_rng(21)
    combos = [(0.0, 1.0, 1.0, 0.0, 1.0, 0), (0.5, 1.3, 0.8, 0.05, 0.9, 8), (1.0, 1.05, 0.9, 0.0, 0.95, 50),
              (-0.5, 2.0, 1.2, 0.2, 0.7, 3), (0.0, 1.0, 0.7, 0.3, 1.0, 0), (2.0, 1.5, 1.0, 0.01, 0.8, 5)]
    for trial in range(5):
        zc = (rng.standard_normal(16) * 2).astype(F32)
        zu = (zc + rng.standard_normal(16)).astype(F32)
        seen = (rng.random(16) < 0.4).astype(np.uint8)
        for w, pen, T, min_p, top_p, k in combos:
            _check(zc, zu, w, seen, pen, T, min_p, top_p, k)


def test_ladder_without_its_extra_stages_is_the_plain_sampler():
    rng = np.random.default_rng(22)
    for trial in range(4):
        z = (rng.standard_normal(16) * 2).astype(F32)
        for T, k, p in [(0.8, 5, 1.0), (1.3, 16, 1.0), (0.9, 16, 0.9), (1.0, 16, 0.5)]:
            for g in range(1 << 10):
                u = g / (1 << 10)
                a, ma = oracle.sample_ladder(z, temperature=T, top_k=k, top_p=p, u=u)
                b, mb = oracle.sample(z, T, k, p, False, u)
                assert a == b or min(ma, mb) < 1e-12, (T, k, p, u, a, b)


def test_cfg_weight_minus_one_samples_the_unconditional_logits():
    rng = np.random.default_rng(23)
    zc = (rng.standard_normal(16) * 2).astype(F32)
    zu = (rng.standard_normal(16) * 2).astype(F32)
    for g in range(1 << 10):
        u = g / (1 << 10)
        a, ma = oracle.sample_ladder(zc, zu, cfg_weight=-1.0, temperature=0.9, top_p=0.9, u=u)
        b, mb = oracle.sample_ladder(zu, temperature=0.9, top_p=0.9, u=u)
        assert a == b or min(ma, mb) < 1e-9
    # w = 0 ignores the unconditional logits entirely
    assert oracle.sample_ladder(zc, zu, cfg_weight=0.0, temperature=0)[0] == int(np.argmax(zc))


def test_repetition_penalty_divides_positive_and_multiplies_negative_logits():
    seen = np.array([1, 1, 0, 0], np.uint8)
    # a seen positive leader is divided: 2.0 -> 1.0 falls below the unseen 1.5
    z = np.array([2.0, -2.0, 1.5, -1.0], F32)
    assert oracle.sample_ladder(z, seen=seen, rep_penalty=2.0, temperature=0)[0] == 2
    # a seen negative leader is multiplied: -1.0 -> -2.0 falls below the unseen -1.5
    z = np.array([-1.0, -3.0, -1.5, -4.0], F32)
    assert oracle.sample_ladder(z, seen=seen, rep_penalty=2.0, temperature=0)[0] == 2
    # penalty 1 and an empty history change nothing
    z = np.array([0.3, 2.0, -1.0, 1.0], F32)
    assert oracle.sample_ladder(z, seen=np.ones(4, np.uint8), rep_penalty=1.0, temperature=0)[0] == 1
    assert oracle.sample_ladder(z, seen=np.zeros(4, np.uint8), rep_penalty=3.0, temperature=0)[0] == 1


def test_min_p_one_keeps_only_the_largest():
    z = np.array([0.1, 2.0, -1.0, 2.0, 1.9], F32)   # two equal leaders
    toks = {oracle.sample_ladder(z, temperature=0.7, min_p=1.0, u=g / 64)[0] for g in range(64)}
    assert toks == {1, 3}
    # min_p = 0.5 keeps exactly the tokens within log 2 of the leader (at T = 1)
    z = np.array([0.0, -0.5, -0.69, -0.7, -3.0], F32)
    probs = _ladder_probs(z, None, 0, None, 1, 1.0, 0.5, 1.0, 0)
    assert list(probs > 0) == [True, True, True, False, False]
    _check(z, None, 0, None, 1, 1.0, 0.5, 1.0, 0)


def test_top_p_acts_before_top_k():
    # probabilities 0.4, 0.3, 0.2, 0.1: top-p 0.5 keeps {0, 1}; top-k 2 then keeps both.
    # The reverse order (top-k 2 -> {0, 1} renormalised to 4/7, 3/7, then top-p 0.5)
    # would keep token 0 alone.
    z = np.log(np.array([0.4, 0.3, 0.2, 0.1])).astype(F32)
    assert oracle.sample_ladder(z, temperature=1.0, top_p=0.5, top_k=2, u=0.9)[0] == 1
    _check(z, None, 0, None, 1, 1.0, 0.0, 0.5, 2)


def _ladder(T, min_p, top_p, k):
    return lambda z, u: oracle.sample_ladder(z, temperature=T, min_p=min_p, top_p=top_p, top_k=k, u=u)


def test_ladder_margin_bruteforce_changes_below_it_keep_the_token():
    """The ladder's margin means what the plain sampler's does (over the final
    scaled logits): moving u, or the scaled logits, by less than it keeps the
    token, and it never exceeds the draw's distance to its CDF edges."""
    rng = np.random.default_rng(24)
    for trial in range(16):
        z = (rng.standard_normal(16) * rng.choice([1.0, 2.0, 3.0])).astype(F32)
        if trial % 2:
            for i in rng.choice(16, size=4, replace=False):
                z[(i + 1) % 16] = z[i] - F32(rng.choice([1e-3, 1e-2]))
        T = float(F32(rng.choice([0.7, 1.0, 1.2])))
        min_p = float(F32(rng.choice([0.0, 0.02, 0.1, 0.3])))
        top_p = float(F32(rng.choice([1.0, 0.6, 0.9])))
        k = int(rng.choice([0, 3, 6]))
        probs = _ladder_probs(z, None, 0.0, None, 1.0, T, min_p, top_p, k)
        for u in rng.random(3):
            tok, M = oo._assert_margin_sound(_ladder(T, min_p, top_p, k), z, T, float(u))
            assert M <= oo._draw_distance(probs, tok, float(u)) * (1 + 1e-12) + 1e-15


def test_ladder_margin_at_a_min_p_boundary():
    # probabilities relative to the largest: 1 (id 4), 0.5 (id 9), 0.1 e^0.01 (id 2),
    # the rest below 0.1 / e: min_p = 0.1 keeps three, and id 2 drops once a change
    # of expm1(0.01) lets its ratio to the largest fall under min_p
    z = np.full(16, -4.0, F32) - 0.05 * np.arange(16, dtype=F32)
    z[4], z[9], z[2] = 0.0, math.log(0.5), math.log(0.1) + 0.01
    u = 0.03                                            # inside id 2's interval (first in vocabulary order)
    tok, M = oo._assert_margin_sound(_ladder(1.0, 0.1, 1.0, 0), z, 1.0, u)
    assert tok == 2
    delta = float(z[2]) - float(z[4]) - math.log(float(F32(0.1)))
    assert abs(M - math.expm1(delta)) <= 1e-9 * M, (M, math.expm1(delta))
    d = np.ones(16)
    d[2] = -1.0
    assert oo._flip_within(_ladder(1.0, 0.1, 1.0, 0), z, 1.0, u, tok, M, d)
