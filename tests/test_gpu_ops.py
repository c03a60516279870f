"""Kernel-level parity of libsd.so against the oracle, at the workloads' shapes
and at ragged sizes that leave partial tiles (through the C ABI of sd_ops.h)."""

import numpy as np
import pytest

import oracle
from synth import uniform_draws
from synth.weights import quantize_q4_0, quantize_q8_0, quantize_a8g64, quantize_q5_0, quantize_a4
from tests.conftest import golden_path

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

KQ8, KQ4, KA8, KQ5, KA4G32, KA4G64 = 1, 2, 3, 4, 5, 6
AFFINE = {KA8: (64, None), KA4G32: (32, 32), KA4G64: (64, 64)}
U = 2.0 ** -24


@pytest.fixture(scope="module")
def sd():
    import __graft_entry__
    __graft_entry__.build()
    import autoregressive_speech_token_gb300 as pkg
    assert torch.cuda.is_available()
    return pkg


def _affine(kind, w):
    return quantize_a8g64(w) if kind == KA8 else quantize_a4(w, AFFINE[kind][1])


def _canon(kind, w):
    if kind == KQ8:
        return quantize_q8_0(w).reshape(-1)
    if kind == KQ4:
        return quantize_q4_0(w).reshape(-1)
    if kind == KQ5:
        return quantize_q5_0(w).reshape(-1)
    q, s, b = _affine(kind, w)
    return np.concatenate([q.ravel(), s.view(np.uint8).ravel(), b.view(np.uint8).ravel()])


def _weights(rows, cols, seed):
    return (np.random.default_rng(seed).standard_normal((rows, cols)) * 0.02).astype(np.float32)


SHAPES = {
    KQ8: [(3072, 1024), (1024, 4096), (6563, 1024), (37, 96), (5, 1056), (1, 32)],
    KQ4: [(3072, 1024), (8192, 1024), (1024, 4096), (8194, 1024), (37, 96), (5, 1056)],
    KA8: [(4096, 2048), (2048, 6144), (12288, 2048), (1024, 3072), (2048, 1024), (37, 128), (5, 1088)],
    KQ5: [(3072, 1024), (1024, 4096), (6563, 1024), (37, 96), (5, 1056), (1, 32)],
    KA4G32: [(1024, 3072), (6144, 1024), (2048, 1024), (37, 96), (5, 1056)],
    KA4G64: [(1024, 3072), (6144, 1024), (2048, 1024), (37, 128), (5, 1088)],
}
CASES = [(k, s) for k, ss in SHAPES.items() for s in ss]


@pytest.mark.parametrize("kind,shape", CASES)
def test_dequant_bit_exact(sd, kind, shape):
    rows, cols = shape
    canon = _canon(kind, _weights(rows, cols, rows + cols + kind))
    h = sd.sd_qmat_create(kind, canon, rows, cols)
    try:
        out = torch.empty(rows, cols, dtype=torch.float32, device="cuda")
        sd.sd_qmat_dequant(h, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
    finally:
        sd.sd_qmat_destroy(h)
    ref = oracle.dequant(kind, canon, rows, cols)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("nb", [1, 2])
@pytest.mark.parametrize("kind,shape", CASES)
def test_gemv_against_oracle(sd, kind, shape, nb):
    rows, cols = shape
    rng = np.random.default_rng(rows * 7 + cols + nb)
    canon = _canon(kind, _weights(rows, cols, rows + cols + kind))
    x = rng.standard_normal((nb, cols)).astype(np.float32)
    bias = rng.standard_normal(rows).astype(np.float32) * 0.1
    h = sd.sd_qmat_create(kind, canon, rows, cols)
    try:
        xd = torch.from_numpy(x).cuda()
        bd = torch.from_numpy(bias).cuda()
        yd = torch.empty(nb, rows, dtype=torch.float32, device="cuda")
        sd.sd_qmat_gemv(h, xd, nb, bd, yd)
        torch.cuda.synchronize()
        y = yd.cpu().numpy()
    finally:
        sd.sd_qmat_destroy(h)
    deq = np.abs(oracle.dequant(kind, canon, rows, cols).astype(np.float64))
    for b in range(nb):
        ref = oracle.linear(kind, canon, rows, cols, x[b], bias).astype(np.float64)
        # fp32 accumulation in a reduction tree at most ~64 deep: |err| <= 64 u sum|w||x|
        # (affine: the factored form scale*sum(q x) + bias*sum(x) adds the |bias| sum|x| terms)
        mag = deq @ np.abs(x[b].astype(np.float64)) + np.abs(bias)
        if kind in AFFINE:
            q, s, bb = _affine(kind, _weights(rows, cols, rows + cols + kind))
            gsum = np.abs(x[b].astype(np.float64)).reshape(-1, AFFINE[kind][0]).sum(1)
            mag = mag + 2 * np.abs(bb.astype(np.float64)) @ gsum
        err = np.abs(y[b] - ref)
        bound = 64 * U * mag + 2 * U * np.abs(ref)
        assert np.all(err <= bound), (b, float(np.max(err / bound)))


SAMPLERS = [
    (1.0, 1, 1.0, 1),          # greedy
    (0.8, 1000, 0.95, 0),      # T3 defaults
    (0.9, 50, 0.95, 0),        # Talker / code predictor
    (1.0, 100000, 1.0, 0),     # plain softmax sampling over the whole vocabulary
    (0.7, 5, 1.0, 0),
    (1.3, 400, 0.5, 0),
]


@pytest.mark.parametrize("V", [16, 2048, 3072, 6563, 8194])
@pytest.mark.parametrize("samp", SAMPLERS)
def test_sampler_against_oracle(sd, V, samp):
    T, k, p, greedy = samp
    rows = 8
    rng = np.random.default_rng(V + k)
    z = (rng.standard_normal((rows, V)) * 0.64).astype(np.float32)
    z[3] *= 8.0                                     # a peaked row
    z[5, ::7] = z[5, 0]                             # ties
    u = uniform_draws(11, 1, rows)[0, :, 0]
    zd, ud = torch.from_numpy(z).cuda(), torch.from_numpy(u).cuda()
    out = torch.empty(rows, dtype=torch.int32, device="cuda")
    s = sd.Sampler(T, min(k, 1 << 30), p, greedy)
    sd.sd_sample_rows(zd, rows, V, s, ud, out)
    got = out.cpu().numpy()
    for b in range(rows):
        tok, margin = oracle.sample(z[b], T, k, p, bool(greedy), float(u[b]))
        if margin >= 1e-4:
            assert got[b] == tok, (b, got[b], tok, margin)
        else:
            assert 0 <= got[b] < V


def test_sampler_u_grid_16_entries(sd):
    """Sixteen-entry vocabulary: the token as a function of u matches the
    oracle on a 2^12 grid, except within 1e-5 of a CDF boundary."""
    rng = np.random.default_rng(5)
    z = (rng.standard_normal(16) * 2).astype(np.float32)
    n = 1 << 12
    for T, k, p in [(0.8, 16, 1.0), (0.8, 5, 1.0), (1.3, 16, 0.7), (0.5, 7, 0.9)]:
        u = (np.arange(n) / n).astype(np.float32)
        zz = np.repeat(z[None], n, 0)
        out = torch.empty(n, dtype=torch.int32, device="cuda")
        sd.sd_sample_rows(torch.from_numpy(zz).cuda(), n, 16, sd.Sampler(T, k, p, 0),
                          torch.from_numpy(u).cuda(), out)
        got = out.cpu().numpy()
        for g in range(n):
            tok, margin = oracle.sample(z, T, k, p, False, float(u[g]))
            if margin > 1e-5:
                assert got[g] == tok, (T, k, p, g)


@pytest.mark.parametrize("H,Hkv,hd", [(16, 16, 64), (16, 8, 128), (4, 4, 64), (8, 2, 64)])
@pytest.mark.parametrize("n,nsplit", [(1, 8), (2, 8), (37, 1), (150, 8), (399, 8), (400, 16), (2048, 8)])
def test_attention_against_oracle(sd, H, Hkv, hd, n, nsplit):
    B, n_ctx = 2, 2048
    rng = np.random.default_rng(n * 3 + hd + H)
    q = rng.standard_normal((B, H, hd)).astype(np.float32)
    k = (rng.standard_normal((B, Hkv, n_ctx, hd)) * 1.5).astype(np.float16)
    v = rng.standard_normal((B, Hkv, n_ctx, hd)).astype(np.float16)
    out = torch.empty(B, H, hd, dtype=torch.float32, device="cuda")
    sd.sd_attend_rows(torch.from_numpy(q).cuda(), torch.from_numpy(k.view(np.uint16)).cuda(),
                      torch.from_numpy(v.view(np.uint16)).cuda(), B, H, Hkv, hd, n_ctx, n, nsplit, out)
    got = out.cpu().numpy()
    G = H // Hkv
    for b in range(B):
        for h in range(H):
            g = h // G
            ref = oracle.attend(q[b, h], k[b, g, :n].view(np.uint16), v[b, g, :n].view(np.uint16))
            assert np.max(np.abs(got[b, h] - ref)) <= 2e-5 * np.max(np.abs(v[b, g, :n].astype(np.float32))), (b, h)
