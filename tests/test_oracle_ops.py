"""Pins of the oracle's operations against things other than itself:
library routines (numpy fp16 conversion, torch float64 functional ops),
closed forms, hand-built blocks with known values, invariants and brute force."""

import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from synth.weights import quantize_q4_0, quantize_q8_0, quantize_a8g64, quantize_q5_0, quantize_a4

KQ8, KQ4, KA8, KQ5, KA4G32, KA4G64 = 1, 2, 3, 4, 5, 6
F32 = np.float32


# ----------------------------------------------------------------------------- fp16

def test_fp16_conversions_match_numpy():
    rng = np.random.default_rng(0)
    special = np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, 1e9, -1e9, 6.1035156e-05,
                        6.0975552e-05, 5.9604645e-08, 2.9802322e-08, 2.98023259e-08, 1e-10, 0.1, 1 / 3,
                        2049.0, 2051.0, 2050.0, 1.00048828125, 1.000732421875], np.float32)
    x = np.concatenate([special, rng.standard_normal(4000).astype(np.float32) * 3,
                        rng.standard_normal(2000).astype(np.float32) * 1e-5,
                        rng.standard_normal(500).astype(np.float32) * 3e4])
    got = oracle.float_to_half(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)
    allh = np.arange(0, 65536, dtype=np.uint16)
    allh = allh[~np.isnan(allh.view(np.float16))]
    back = oracle.half_to_float(allh)
    assert np.array_equal(back.view(np.uint32), allh.view(np.float16).astype(np.float32).view(np.uint32))


# ----------------------------------------------------------------------------- dequantisation

def test_q4_0_hand_block():
    """Block with d = 0.25 and byte j = j | (15-j) << 4: element j (j<16) is
    0.25*(j-8) and element 16+j is 0.25*(7-j) (nibble order of the Q4_0 block)."""
    blk = np.zeros(18, np.uint8)
    blk[0:2] = np.array([0.25], np.float16).view(np.uint8)
    for j in range(16):
        blk[2 + j] = j | ((15 - j) << 4)
    out = oracle.dequant(KQ4, blk, 1, 32)[0]
    exp = np.array([0.25 * (j - 8) for j in range(16)] + [0.25 * (7 - j) for j in range(16)], np.float32)
    assert np.array_equal(out, exp)


def test_q8_0_hand_block():
    blk = np.zeros(34, np.uint8)
    blk[0:2] = np.array([-0.5], np.float16).view(np.uint8)
    codes = np.arange(-16, 16, dtype=np.int8) * 4 + 3
    blk[2:] = codes.view(np.uint8)
    out = oracle.dequant(KQ8, blk, 1, 32)[0]
    assert np.array_equal(out, (-0.5 * codes.astype(np.float32)).astype(np.float32))


def test_a8g64_hand_group():
    q = np.arange(64, dtype=np.uint8) * 4
    scale = np.array([0.125], np.float16)
    bias = np.array([-3.0], np.float16)
    data = np.concatenate([q, scale.view(np.uint8), bias.view(np.uint8)])
    out = oracle.dequant(KA8, data, 1, 64)[0]
    assert np.array_equal(out, (0.125 * q.astype(np.float32) - 3.0).astype(np.float32))


def test_q5_0_hand_block():
    """Block with d = -0.5, fifth bits 0xF0F0F0F0 and byte j = j | (15-j) << 4:
    element j (j<16) has code j + 16*bit(j) and element 16+j has code (15-j) +
    16*bit(16+j); the value is d*(code - 16).  The two halves of the fifth-bit
    word are different (bits 4-7 and 12-15 of each half set), so a bit taken
    from the wrong element changes the result."""
    blk = np.zeros(22, np.uint8)
    blk[0:2] = np.array([-0.5], np.float16).view(np.uint8)
    qh = 0xF0F0F00F
    blk[2:6] = np.array([qh], "<u4").view(np.uint8)
    for j in range(16):
        blk[6 + j] = j | ((15 - j) << 4)
    out = oracle.dequant(KQ5, blk, 1, 32)[0]
    codes = [j + 16 * ((qh >> j) & 1) for j in range(16)] + [(15 - j) + 16 * ((qh >> (16 + j)) & 1) for j in range(16)]
    exp = np.array([-0.5 * (c - 16) for c in codes], np.float32)
    assert np.array_equal(out, exp)
    # the extremes: code 0 -> -16 d, code 31 -> 15 d
    blk[2:6] = np.array([0x0000FFFF], "<u4").view(np.uint8)
    blk[6:] = 0xF0   # low nibble 0 (elements 0..15), high nibble 15 (elements 16..31)
    out = oracle.dequant(KQ5, blk, 1, 32)[0]
    assert np.array_equal(out, np.array([-0.5 * 0] * 16 + [-0.5 * -1] * 16, np.float32))


@pytest.mark.parametrize("kind,gs", [(KA4G32, 32), (KA4G64, 64)])
def test_a4_hand_group(kind, gs):
    """Two groups per row, codes 0..15 repeated: element 2i sits in the low
    nibble of byte i, element 2i+1 in its high nibble; value scale*q + bias with
    each group's own scale and bias."""
    q = (np.arange(2 * gs) * 7 % 16).astype(np.uint8)
    packed = (q[0::2] | (q[1::2] << 4)).astype(np.uint8)
    scale = np.array([0.125, -0.25], np.float16)
    bias = np.array([-3.0, 0.5], np.float16)
    data = np.concatenate([packed, scale.view(np.uint8), bias.view(np.uint8)])
    out = oracle.dequant(kind, data, 1, 2 * gs)[0]
    g = np.arange(2 * gs) // gs
    exp = (scale.astype(np.float32)[g] * q.astype(np.float32) + bias.astype(np.float32)[g]).astype(np.float32)
    assert np.array_equal(out, exp)


def _roundtrip_case(kind, w):
    if kind == KQ8:
        q1 = quantize_q8_0(w)
        deq = oracle.dequant(KQ8, q1, *w.shape)
        q2 = quantize_q8_0(deq)
        assert np.array_equal(q1, q2)
        d = q1[..., 0:2].copy().view(np.float16).astype(np.float32)[..., 0]
        err = np.abs(deq - w).reshape(w.shape[0], -1, 32).max(-1)
        assert np.all(err <= np.abs(d) * (0.5 + 127 * 2 ** -11) + 1e-12)
    elif kind == KQ4:
        q1 = quantize_q4_0(w)
        deq = oracle.dequant(KQ4, q1, *w.shape)
        q2 = quantize_q4_0(deq)
        assert np.array_equal(q1, q2)
        d = q1[..., 0:2].copy().view(np.float16).astype(np.float32)[..., 0]
        err = np.abs(deq - w).reshape(w.shape[0], -1, 32).max(-1)
        assert np.all(err <= np.abs(d) * (1 + 8 * 2 ** -11) + 1e-12)
    elif kind == KQ5:
        q1 = quantize_q5_0(w)
        deq = oracle.dequant(KQ5, q1, *w.shape)
        q2 = quantize_q5_0(deq)
        assert np.array_equal(q1, q2)
        d = q1[..., 0:2].copy().view(np.float16).astype(np.float32)[..., 0]
        err = np.abs(deq - w).reshape(w.shape[0], -1, 32).max(-1)
        assert np.all(err <= np.abs(d) * (1 + 16 * 2 ** -11) + 1e-12)
    else:
        gs, steps = {KA8: (64, 255), KA4G32: (32, 15), KA4G64: (64, 15)}[kind]
        q, s, b = quantize_a8g64(w) if kind == KA8 else quantize_a4(w, gs)
        data = np.concatenate([q.ravel(), s.view(np.uint8).ravel(), b.view(np.uint8).ravel()])
        deq = oracle.dequant(kind, data, *w.shape)
        q2, s2, b2 = quantize_a8g64(deq) if kind == KA8 else quantize_a4(deq, gs)
        assert np.array_equal(q, q2)
        err = np.abs(deq - w).reshape(w.shape[0], -1, gs).max(-1)
        sc = s.astype(np.float32)
        # half a step, plus the fp16 rounding of bias and scale (up to `steps` steps)
        bound = 0.5 * sc + np.abs(b.astype(np.float32)) * 2 ** -11 + steps * sc * 2 ** -11 + 1e-7
        assert np.all(err <= bound)
    return deq


@pytest.mark.parametrize("kind", [KQ8, KQ4, KA8, KQ5, KA4G32, KA4G64])
def test_dequant_roundtrip_and_bounds(kind):
    rng = np.random.default_rng(kind)
    w = (rng.standard_normal((37, 256)) * 0.02).astype(np.float32)
    _roundtrip_case(kind, w)
    # special cases: an all-zero block/group, a constant group, an extreme element
    w2 = w.copy()
    w2[0, :64] = 0
    w2[1, :64] = 0.0123
    w2[2, 5] = 0.5
    w2[3, 40] = -0.5
    deq = _roundtrip_case(kind, w2)
    assert np.all(deq[0, :64] == 0)
    if kind == KQ8:
        assert abs(deq[2, 5] - 0.5) <= 0.5 * 2 ** -11      # code +127 hits the max exactly up to fp16 d
    if kind == KQ4:
        assert abs(deq[3, 40] + 0.5) <= 0.5 * 2 ** -11     # code 0 -> -8 d = m up to fp16 d
    if kind == KQ5:
        assert abs(deq[3, 40] + 0.5) <= 0.5 * 2 ** -11     # code 0 -> -16 d = m up to fp16 d
    if kind in (KA8, KA4G32, KA4G64):
        assert np.all(deq[1, :64] == deq[1, 0])


# ----------------------------------------------------------------------------- sampler with a repetition penalty

def test_penalised_sampler_follows_the_sign_rule():
    """A seen positive logit is divided (it can lose the argmax), a seen negative
    one multiplied (it moves further down); unseen tokens keep their logits."""
    z = np.array([2.0, 1.5, -0.5, -0.6], np.float32)
    seen = np.array([1, 0, 0, 0], np.uint8)
    assert oracle.sample(z, greedy=True, seen=seen, rep_penalty=2.0)[0] == 1      # 2.0 / 2 = 1.0 < 1.5
    assert oracle.sample(z, greedy=True, seen=seen, rep_penalty=1.2)[0] == 0      # 2.0 / 1.2 > 1.5
    z2 = np.array([-1.0, -0.9, -3.0], np.float32)
    seen2 = np.array([0, 1, 0], np.uint8)
    assert oracle.sample(z2, greedy=True, seen=seen2, rep_penalty=1.2)[0] == 0    # -0.9 * 1.2 = -1.08 < -1.0
    assert oracle.sample(z2, greedy=True, seen=seen2, rep_penalty=1.0)[0] == 1
    assert oracle.sample(z2, greedy=True, seen=None, rep_penalty=3.0)[0] == 1


def test_penalised_sampler_bruteforce():
    """Enumeration from the definitions on 16-entry vocabularies: the penalised
    logits (HF rule) through temperature, top-k (ties kept), top-p (shortest
    prefix in probability desc / index asc order) and the index-order draw."""
    rng = np.random.default_rng(44)
    for case in range(60):
        z = (rng.standard_normal(16) * 1.5).astype(np.float32)
        seen = (rng.random(16) < 0.4).astype(np.uint8)
        pen = float(rng.choice([1.1, 1.5, 2.0]))
        T = float(rng.choice([0.5, 0.9, 1.3]))
        k = int(rng.choice([3, 8, 16]))
        p = float(rng.choice([0.6, 0.9, 1.0]))
        zp = np.array([(v / pen if v > 0 else v * pen) if sn else v for v, sn in zip(z.astype(np.float64), seen)])
        zp = zp.astype(np.float32).astype(np.float64) / T
        order = sorted(range(16), key=lambda i: (-zp[i], i))
        kept = [i for i in range(16) if sum(zp[j] > zp[i] for j in range(16)) < k]
        w = {i: math.exp(zp[i] - zp[order[0]]) for i in kept}
        Z = sum(w.values())
        if p < 1.0:
            cum, keep2 = 0.0, []
            for i in sorted(kept, key=lambda i: (-zp[i], i)):
                keep2.append(i)
                cum += w[i] / Z
                if cum >= p:
                    break
            kept = keep2
        ZS = sum(w[i] for i in kept)
        for u in (0.03, 0.31, 0.58, 0.77, 0.96):
            acc, want = 0.0, None
            for i in sorted(kept):
                acc += w[i] / ZS
                if acc > u:
                    want = i
                    break
            got, margin = oracle.sample(z, temperature=T, top_k=k, top_p=p, greedy=False, u=u, seen=seen,
                                        rep_penalty=pen)
            if margin > 1e-9:
                assert got == want, (case, u, got, want, margin)


def test_penalty_of_one_or_no_history_is_the_plain_sampler():
    rng = np.random.default_rng(45)
    for _ in range(30):
        z = rng.standard_normal(300).astype(np.float32)
        u = float(rng.random())
        a = oracle.sample(z, temperature=0.9, top_k=50, top_p=0.95, greedy=False, u=u)
        b = oracle.sample(z, temperature=0.9, top_k=50, top_p=0.95, greedy=False, u=u,
                          seen=np.ones(300, np.uint8), rep_penalty=1.0)
        c = oracle.sample(z, temperature=0.9, top_k=50, top_p=0.95, greedy=False, u=u,
                          seen=np.zeros(300, np.uint8), rep_penalty=1.7)
        assert a == b == c


# ----------------------------------------------------------------------------- linear

def quant_data(kind, w):
    """The canonical stored bytes of w in format `kind` (affine: codes, scales, biases)."""
    if kind == KQ8:
        return quantize_q8_0(w)
    if kind == KQ4:
        return quantize_q4_0(w)
    if kind == KQ5:
        return quantize_q5_0(w)
    q, s, b = quantize_a8g64(w) if kind == KA8 else quantize_a4(w, 32 if kind == KA4G32 else 64)
    return np.concatenate([q.ravel(), s.view(np.uint8).ravel(), b.view(np.uint8).ravel()])


@pytest.mark.parametrize("kind", [KQ8, KQ4, KA8, KQ5, KA4G32, KA4G64])
def test_linear_against_float64_dot(kind):
    rng = np.random.default_rng(10 + kind)
    rows, cols = 70, 384
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    data = quant_data(kind, w)
    deq = oracle.dequant(kind, data, rows, cols).astype(np.float64)
    x = rng.standard_normal(cols).astype(np.float32)
    bias = rng.standard_normal(rows).astype(np.float32)
    y = oracle.linear(kind, data, rows, cols, x, bias)
    ref = deq @ x.astype(np.float64) + bias
    gamma = cols * 2.0 ** -53 / (1 - cols * 2.0 ** -53)
    bound = gamma * (np.abs(deq) @ np.abs(x.astype(np.float64)) + np.abs(bias)) + np.abs(ref) * 2.0 ** -24
    assert np.all(np.abs(y - ref) <= bound * 1.01 + 1e-30)
    # one-hot input selects a column exactly
    e = np.zeros(cols, np.float32)
    e[17] = 1.0
    assert np.array_equal(oracle.linear(kind, data, rows, cols, e), deq[:, 17].astype(np.float32))


def test_linear_f32_kind():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((5, 8)).astype(np.float32)
    x = rng.standard_normal(8).astype(np.float32)
    y = oracle.linear(0, w, 5, 8, x)
    assert np.allclose(y, w.astype(np.float64) @ x, rtol=1e-7, atol=0)


# ----------------------------------------------------------------------------- norms and activations

def test_layernorm_invariants_and_torch():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(1024) * 3 + 1.5).astype(np.float32)
    one, zero = np.ones(1024, np.float32), np.zeros(1024, np.float32)
    h = oracle.layernorm(x, one, zero, 1e-5).astype(np.float64)
    var = np.var(x.astype(np.float64))
    assert abs(h.mean()) < 1e-6
    assert abs(h.var() - var / (var + 1e-5)) < 1e-6
    g = (1 + 0.02 * rng.standard_normal(1024)).astype(np.float32)
    b = (0.02 * rng.standard_normal(1024)).astype(np.float32)
    h2 = oracle.layernorm(x, g, b, 1e-5)
    ref = F.layer_norm(torch.tensor(x, dtype=torch.float64), (1024,), torch.tensor(g, dtype=torch.float64),
                       torch.tensor(b, dtype=torch.float64), eps=1e-5).numpy()
    assert np.max(np.abs(h2 - ref)) <= 4 * 2.0 ** -24 * np.max(np.abs(ref))


def test_rmsnorm_invariants_and_torch():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(2048) * 2).astype(np.float32)
    one = np.ones(2048, np.float32)
    h = oracle.rmsnorm(x, one, 1e-5).astype(np.float64)
    ms = np.mean(x.astype(np.float64) ** 2)
    assert abs(np.mean(h ** 2) - ms / (ms + 1e-5)) < 1e-6
    g = (1 + 0.02 * rng.standard_normal(2048)).astype(np.float32)
    ref = F.rms_norm(torch.tensor(x, dtype=torch.float64), (2048,), torch.tensor(g, dtype=torch.float64),
                     eps=1e-5).numpy()
    assert np.max(np.abs(oracle.rmsnorm(x, g, 1e-5) - ref)) <= 4 * 2.0 ** -24 * np.max(np.abs(ref))


def test_activations_against_torch():
    t = np.concatenate([np.linspace(-12, 12, 2001), [0.0, 1e-8, -1e-8, 30.0, -30.0]]).astype(np.float32)
    tt = torch.tensor(t, dtype=torch.float64)
    g = oracle.gelu_tanh(t)
    # 1 + tanh(.) cancels for t below about -7: there only an absolute bound is meaningful
    assert np.allclose(g, F.gelu(tt, approximate="tanh").numpy(), rtol=2 ** -23, atol=1e-14)
    assert g[2001] == 0.0 and g[2004] == 30.0
    s = oracle.silu(t)
    assert np.allclose(s, F.silu(tt).numpy(), rtol=2 ** -23, atol=1e-37)


# ----------------------------------------------------------------------------- RoPE

def test_rope_identity_norms_and_complex_form():
    rng = np.random.default_rng(6)
    for hd in (64, 128):
        x = rng.standard_normal(hd).astype(np.float32)
        assert np.array_equal(oracle.rope(x, 0), x)              # pos 0 is the identity
        for pos in (1, 7, 399, 2047):
            y = oracle.rope(x, pos).astype(np.float64)
            half = hd // 2
            # rotation of each (i, i + hd/2) pair: norms preserved
            n0 = x[:half].astype(np.float64) ** 2 + x[half:].astype(np.float64) ** 2
            n1 = y[:half] ** 2 + y[half:] ** 2
            assert np.allclose(n0, n1, rtol=1e-6)
            # the half-split convention as a complex product (a + ib) e^{i phi}
            i = np.arange(half)
            phi = pos * 10000.0 ** (-2.0 * i / hd)
            z = (x[:half].astype(np.float64) + 1j * x[half:].astype(np.float64)) * np.exp(1j * phi)
            assert np.allclose(y[:half], z.real, rtol=0, atol=4e-7 * np.abs(z).max())
            assert np.allclose(y[half:], z.imag, rtol=0, atol=4e-7 * np.abs(z).max())


# ----------------------------------------------------------------------------- attention

def test_attention_closed_forms_and_sdpa():
    rng = np.random.default_rng(7)
    hd = 64
    k = rng.standard_normal((9, hd)).astype(np.float16).view(np.uint16)
    v = rng.standard_normal((9, hd)).astype(np.float16).view(np.uint16)
    q = rng.standard_normal(hd).astype(np.float32)
    vf = v.view(np.float16).astype(np.float64)
    # one cached position: the output is that value row exactly
    assert np.array_equal(oracle.attend(q, k[:1], v[:1]), vf[0].astype(np.float32))
    # zero query: uniform weights, the mean of V
    o = oracle.attend(np.zeros(hd, np.float32), k, v)
    assert np.allclose(o, vf.mean(0), rtol=0, atol=2e-7 * np.abs(vf).max())
    # against torch's float64 scaled-dot-product attention
    o = oracle.attend(q, k, v)
    kf = torch.tensor(k.view(np.float16).astype(np.float64))
    ref = F.scaled_dot_product_attention(torch.tensor(q, dtype=torch.float64)[None, None],
                                         kf[None], torch.tensor(vf)[None])[0, 0].numpy()
    assert np.allclose(o, ref, rtol=0, atol=2 ** -23 * np.abs(ref).max())


def test_attention_softmax_weights_sum_to_one():
    rng = np.random.default_rng(8)
    hd = 128
    n = 50
    k = (rng.standard_normal((n, hd)) * 3).astype(np.float16).view(np.uint16)
    ones = np.ones((n, hd), np.float16).view(np.uint16)
    q = rng.standard_normal(hd).astype(np.float32)
    # V = 1 everywhere: the output is the sum of the softmax weights
    o = oracle.attend(q, k, ones)
    assert np.all(np.abs(o.astype(np.float64) - 1.0) <= 2.0 ** -24)


# ----------------------------------------------------------------------------- sampler

def _enumerated_probs(z, T, k, p):
    """Selection probabilities straight from the definitions, without sorting."""
    V = len(z)
    zz = z.astype(np.float64) / T
    kept = [sum(zz[j] > zz[i] for j in range(V)) < k for i in range(V)]
    m = max(zz[i] for i in range(V) if kept[i])
    w = np.array([math.exp(zz[i] - m) if kept[i] else 0.0 for i in range(V)])
    Z = w.sum()
    if p < 1.0:
        S = []
        for i in range(V):
            if not kept[i]:
                S.append(False)
                continue
            before = sum(w[j] for j in range(V) if kept[j] and (w[j] > w[i] or (w[j] == w[i] and j < i)))
            S.append(before / Z < p)
    else:
        S = kept
    w = np.where(S, w, 0.0)
    return w / w.sum()


def _check_sampler(z, T, k, p, n_grid=1 << 16):
    probs = _enumerated_probs(z, T, k, p)
    cdf = np.cumsum(probs)
    counts = np.zeros(len(z))
    for g in range(n_grid):
        u = g / n_grid
        tok, margin = oracle.sample(z, T, k, p, False, u)
        exp = int(np.searchsorted(cdf, u, side="right"))
        exp = min(exp, len(z) - 1)
        while probs[exp] == 0:
            exp -= 1
        if tok != exp:
            assert margin < 1e-9, (z, T, k, p, u, tok, exp)
        counts[tok] += 1
    assert np.all(np.abs(counts / n_grid - probs) <= 1.5 / n_grid + 1e-12)


def test_sampler_bruteforce_random_logits():
    rng = np.random.default_rng(9)
    for trial in range(6):
        z = (rng.standard_normal(16) * 2).astype(np.float32)
        for T, k, p in [(0.8, 16, 1.0), (0.8, 5, 1.0), (1.3, 16, 0.7), (0.5, 7, 0.9), (1.0, 3, 0.95)]:
            _check_sampler(z, T, k, p, n_grid=1 << 12 if trial else 1 << 16)


def test_sampler_adversarial_ties_and_boundaries():
    # ties at the top-k threshold are all kept
    z = np.array([3, 1, 2, 2, 2, 0, -1, 2, 1, 1, 0, 0, -2, -3, 5, 2], np.float32)
    _check_sampler(z, 1.0, 3, 1.0, n_grid=1 << 13)
    probs = _enumerated_probs(z, 1.0, 3, 1.0)
    assert (probs > 0).sum() == 2 + 5           # 5 and 3, then every 2 tie
    # a top-p cut exactly on a boundary: two equal leaders with p = 1/2 each
    z2 = np.full(16, -80.0, np.float32)
    z2[4] = z2[9] = 10.0
    probs2 = _enumerated_probs(z2, 1.0, 16, 0.5)
    assert probs2[4] == 1.0                       # the lower index wins the tie
    for u in (0.0, 0.3, 0.99):
        assert oracle.sample(z2, 1.0, 16, 0.5, False, u)[0] == 4
    _check_sampler(z2, 1.0, 16, 0.5, n_grid=1 << 12)


def test_sampler_special_cases():
    rng = np.random.default_rng(11)
    z = rng.standard_normal(16).astype(np.float32)
    am = int(np.argmax(z))
    for u in (0.0, 0.5, 0.999):
        assert oracle.sample(z, 0.8, 1, 0.95, False, u)[0] == am            # top_k = 1 is argmax
        assert oracle.sample(z, 0.8, 1000, 0.95, True, u)[0] == am          # greedy flag
    # ties under greedy go to the lowest index
    zt = np.zeros(16, np.float32)
    zt[[3, 8, 12]] = 2.0
    tok, m = oracle.sample(zt, 1.0, 1, 1.0, True, 0.0)
    assert tok == 3 and m == 0.0
    # top_k >= V and top_p = 1 is plain softmax sampling (inverse CDF in index order)
    p = np.exp(z.astype(np.float64) / 0.7 - np.max(z) / 0.7)
    p /= p.sum()
    cdf = np.cumsum(p)
    for u in np.linspace(0, 0.999, 37):
        assert oracle.sample(z, 0.7, 16, 1.0, False, float(u))[0] == int(np.searchsorted(cdf, u, side="right"))


def test_sampler_margin_greedy():
    z = np.array([0.0, 1.5, 1.25, -2.0], np.float32)
    tok, m = oracle.sample(z, 1.0, 1, 1.0, True, 0.0)
    assert tok == 1 and m == 0.25


# ----------------------------------------------------------------------------- sampled decision margin
#
# The margin of a sampled draw is read as the smallest change that can change
# the token, in one unit r: u moved by r, or every unnormalised probability
# multiplied by its own factor within [(1+r)^-1/2, (1+r)^1/2] (every scaled
# logit moved by at most log1p(r)/2).  The pins below check it against brute
# force on 16-entry vocabularies: changes below the margin never change the
# token; where a CDF edge is nearest the margin is the enumerated distance to
# it; where a top-k or top-p membership flip is nearest, it is the size at which
# the flip first becomes possible, and a change just above it does flip the token.

def _draw_distance(probs, tok, u):
    """Distance of u to the token's interval edges on the enumerated CDF (vocabulary
    order), counting only edges shared with another kept entry."""
    kept = np.nonzero(probs > 0)[0]
    cdf = np.concatenate([[0.0], np.cumsum(probs)])
    lo, hi = cdf[tok], cdf[tok + 1]
    return min(u - lo if tok != kept[0] else math.inf, hi - u if tok != kept[-1] else math.inf)


def _directions(z, T):
    """Sign patterns of a change of the scaled logits: prefix/suffix splits of the
    (scaled logit desc, index asc) order and of the vocabulary order, one entry
    against all others, every ordered pair, and random signs."""
    V = len(z)
    order = sorted(range(V), key=lambda i: (-float(z[i]) / T, i))
    dirs = []
    for j in range(1, V):
        top = -np.ones(V)
        top[order[:j]] = 1.0
        voc = np.where(np.arange(V) < j, 1.0, -1.0)
        dirs += [top, -top, voc, -voc]
    for a in range(V):
        e = -np.ones(V)
        e[a] = 1.0
        dirs += [e, -e]
        for b in range(V):
            if a != b:
                d = np.zeros(V)
                d[a], d[b] = 1.0, -1.0
                dirs.append(d)
    dirs += list(np.random.default_rng(V).choice([-1.0, 1.0], size=(24, V)))
    return dirs


def _changed(z, T, d, r):
    """Logits after moving every scaled logit by d * log1p(r) / 2 (rounded to fp32),
    and the size of the change that the rounding actually made."""
    z64 = np.asarray(z, np.float64)
    zp = (z64 + T * d * math.log1p(r) / 2).astype(np.float32)
    dev = float(np.max(np.abs(zp.astype(np.float64) - z64))) / T
    return zp, math.expm1(2 * dev)


def _assert_margin_sound(draw, z, T, u, frac=0.999):
    """draw(z, u) -> (token, margin).  Moving u, or the scaled logits in any of the
    directions above, by less than the margin keeps the token."""
    tok, M = draw(z, u)
    assert M >= 0.0
    if math.isinf(M):
        for uu in np.linspace(0.0, 0.999, 41):
            assert draw(z, float(uu))[0] == tok
        return tok, M
    for f in (0.25, 0.5, 0.9, frac):
        for uu in (u - f * M, u + f * M):
            if 0.0 <= uu < 1.0:
                assert draw(z, uu)[0] == tok, ("u moved", u, uu, M)
    if M > 0.0:
        for d in _directions(z, T):
            zp, r = _changed(z, T, d, frac * M)
            if r < M:
                assert draw(zp, u)[0] == tok, ("logits moved", z, T, u, M, r, d)
    return tok, M


def _plain(T, k, p):
    return lambda z, u: oracle.sample(z, T, k, p, False, u)


def test_sampler_margin_bruteforce_changes_below_it_keep_the_token():
    rng = np.random.default_rng(21)
    n_bound = 0
    for trial in range(40):
        z = (rng.standard_normal(16) * rng.choice([0.5, 1.0, 2.0, 4.0])).astype(np.float32)
        if trial % 2:   # near-ties: pairs a small gap apart make boundary flips cheap
            for i in rng.choice(16, size=4, replace=False):
                z[(i + 1) % 16] = z[i] - F32(rng.choice([1e-3, 1e-2, 5e-2]))
        T = float(F32(rng.choice([0.5, 0.8, 1.3])))      # the values the oracle sees (fp32)
        k = int(rng.choice([2, 3, 5, 8, 16]))
        p = float(F32(rng.choice([1.0, 0.5, 0.7, 0.9, 0.95])))
        for u in rng.random(4):
            tok, M = _assert_margin_sound(_plain(T, k, p), z, T, float(u))
            probs = _enumerated_probs(z, T, k, p)
            dist = _draw_distance(probs, tok, float(u))
            assert M <= dist * (1 + 1e-12) + 1e-15           # never beyond the draw's own edges
            n_bound += M < dist * (1 - 1e-9)
    assert n_bound > 0     # some cases were decided by a membership flip, not the draw



def test_sampler_margin_is_the_draw_distance_when_no_flip_reaches():
    rng = np.random.default_rng(23)
    # no selection at all: only the draw decides
    for _ in range(6):
        z = (rng.standard_normal(16) * 1.5).astype(np.float32)
        T = float(F32(rng.choice([0.6, 1.0, 1.7])))
        probs = _enumerated_probs(z, T, 16, 1.0)
        for u in np.linspace(0.0, 0.999, 97):
            tok, M = oracle.sample(z, T, 16, 1.0, False, float(u))
            d = _draw_distance(probs, tok, float(u))
            assert (math.isinf(M) and math.isinf(d)) or abs(M - d) <= 1e-12, (u, tok, M, d)
    # a top-k boundary 4 apart and a top-p cut far from top_p: no flip within reach
    w = np.array([0.03, 0.0002, 0.0003, 0.3, 0.0004, 0.0005, 0.0006, 0.5, 0.0007, 0.0008, 0.0009, 0.15,
                  0.001, 0.0011, 0.0012, 0.0013])
    z = np.log(w).astype(np.float32)
    for k, p in [(16, float(F32(0.9))), (4, 1.0), (3, float(F32(0.9)))]:
        probs = _enumerated_probs(z, 1.0, k, p)
        for u in np.linspace(0.0, 0.999, 61):
            tok, M = oracle.sample(z, 1.0, k, p, False, float(u))
            d = _draw_distance(probs, tok, float(u))
            assert (math.isinf(M) and math.isinf(d)) or abs(M - d) <= 1e-12, (k, p, u, tok, M, d)


def _flip_within(draw, z, T, u, tok, M, d):
    """A change of 1.01 x the margin in direction d changes the token."""
    zp, r = _changed(z, T, d, 1.01 * M)
    assert r < 1.02 * M
    return draw(zp, u)[0] != tok


def test_sampler_margin_at_a_top_k_boundary():
    # scaled logits 2, 1.5, 1.0 | 0.98, rest <= -4 at T = 0.5: k = 3 keeps the first
    # three; the third and fourth are 0.02 apart, so they swap once a change of
    # expm1(0.02) is allowed; the draw sits inside the third's interval, which
    # then leaves the kept set
    z = np.array([-2.0 - 0.1 * i for i in range(16)], np.float32)
    z[5], z[9], z[2], z[12] = 1.0, 0.75, 0.5, 0.49
    T, k, p, u = 0.5, 3, 1.0, 0.09
    tok, M = _assert_margin_sound(_plain(T, k, p), z, T, u)
    assert tok == 2
    gap = (float(z[2]) - float(z[12])) / T
    assert abs(M - math.expm1(gap)) <= 1e-12 * M, (M, math.expm1(gap))
    d = np.zeros(16)
    d[2], d[12] = -1.0, 1.0
    assert _flip_within(_plain(T, k, p), z, T, u, tok, M, d)


def _cut_case():
    # probabilities 0.5 (id 7), 0.3 (id 3), 0.15 (id 11), 0.03 (id 0), 12 small ones
    w = np.zeros(16)
    w[7], w[3], w[11], w[0] = 0.5, 0.3, 0.15, 0.03
    small = [i for i in range(16) if w[i] == 0]
    w[small] = 0.02 * np.arange(1, 13) / 78.0
    z = np.log(w).astype(np.float32)
    q = np.exp(z.astype(np.float64) - float(np.max(z)))
    return z, q / q.sum()


def test_sampler_margin_at_a_top_p_cut_that_can_shrink():
    # top_p just above the mass of the first two: the third (id 11) is kept, and
    # a change that grows the first two against the rest by a factor 1 + r drops
    # it once prev (1+r) / (prev (1+r) + 1 - prev) reaches top_p
    z, q = _cut_case()
    top_p = 0.801
    tp = float(F32(top_p))
    prev = q[7] + q[3]
    r_prev = (tp - prev) / (prev * (1 - tp))
    u = 0.92                                       # inside id 11's interval
    tok, M = _assert_margin_sound(_plain(1.0, 16, top_p), z, 1.0, u)
    assert tok == 11
    assert abs(M - r_prev) <= 1e-9 * r_prev, (M, r_prev)
    d = -np.ones(16)
    d[[7, 3]] = 1.0
    assert _flip_within(_plain(1.0, 16, top_p), z, 1.0, u, tok, M, d)


def test_sampler_margin_at_a_top_p_cut_that_can_grow():
    # top_p just below the mass of the first three: the fourth (id 0, first in
    # vocabulary order) joins once cum / (cum + (1+r)(1 - cum)) falls below top_p,
    # which moves every edge of the kept CDF up past a draw close above one
    z, q = _cut_case()
    cum = q[7] + q[3] + q[11]
    top_p = float(F32(cum - 2e-4))
    r_cum = (cum - top_p) / (top_p * (1 - cum))
    kept = q[3] + q[7] + q[11]
    u = q[3] / kept + 0.01                         # 0.01 above the edge between id 3 and id 7
    tok, M = _assert_margin_sound(_plain(1.0, 16, top_p), z, 1.0, u)
    assert tok == 7
    assert abs(M - r_cum) <= 1e-9 * r_cum, (M, r_cum)
    d = np.ones(16)
    d[[7, 3, 11]] = -1.0
    assert _flip_within(_plain(1.0, 16, top_p), z, 1.0, u, tok, M, d)
