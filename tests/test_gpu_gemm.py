"""Parity of the tensor-core GEMM (sd_qmat_gemm) with the oracle's
dequantisation followed by a float64 matrix product, for every weight format,
ragged row counts and output widths, and every epilogue."""

import numpy as np
import pytest

import oracle
from synth.weights import quantize_a8g64, quantize_q4_0, quantize_q8_0

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

KQ8, KQ4, KA8 = 1, 2, 3
U = 2.0 ** -24


@pytest.fixture(scope="module")
def sd():
    import __graft_entry__
    __graft_entry__.build()
    import autoregressive_speech_token_gb300 as pkg
    assert torch.cuda.is_available()
    return pkg


def _canon(kind, w):
    if kind == KQ8:
        return quantize_q8_0(w).reshape(-1), None
    if kind == KQ4:
        return quantize_q4_0(w).reshape(-1), None
    q, s, b = quantize_a8g64(w)
    return np.concatenate([q.ravel(), s.view(np.uint8).ravel(), b.view(np.uint8).ravel()]), b


def _gelu(t):
    return 0.5 * t * (1.0 + np.tanh(0.7978845608028654 * (t + 0.044715 * t ** 3)))


def _silu(t):
    return t / (1.0 + np.exp(-t))


def _run(sd, kind, rows, cols, M, epi, with_bias, with_resid, seed, tc=False, g16=False):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    canon, abias = _canon(kind, w)
    x = rng.standard_normal((M, cols)).astype(np.float32)
    x[:, ::5] *= 1e-3                                 # small activations exercise the fp16 low half
    out_cols = rows // 2 if epi == 2 else rows
    bias = (rng.standard_normal(rows) * 0.1).astype(np.float32) if with_bias else None
    resid = rng.standard_normal((M, out_cols)).astype(np.float32) if with_resid else None
    h = sd.sd_qmat_create(kind, canon, rows, cols)
    try:
        xd = torch.from_numpy(x).cuda()
        bd = torch.from_numpy(bias).cuda() if bias is not None else None
        yd = torch.from_numpy(resid).cuda() if resid is not None else torch.empty(M, out_cols, device="cuda")
        gemm = sd.sd_qmat_gemm_tc if tc else (sd.sd_qmat_gemm16 if g16 else sd.sd_qmat_gemm)
        y0 = yd.clone()
        gemm(h, xd, M, epi, bd, yd if resid is not None else None, yd)
        torch.cuda.synchronize()
        y = yd.cpu().numpy().astype(np.float64)
        if g16:
            # the split-K partial sums are added in a fixed order: a second call gives the same bits
            yd.copy_(y0)
            gemm(h, xd, M, epi, bd, yd if resid is not None else None, yd)
            torch.cuda.synchronize()
            assert np.array_equal(yd.cpu().numpy().astype(np.float64), y)
    finally:
        sd.sd_qmat_destroy(h)
    deq = oracle.dequant(kind, canon, rows, cols).astype(np.float64)
    x64 = x.astype(np.float64)
    t = x64 @ deq.T
    # error of t: fp16 hi/lo split of x (relative 2^-22, absolute 2^-25 below the fp16 normal
    # range), fp32 accumulation inside each quantisation block and across the K/BK blocks
    bk = 64 if kind == KA8 else 32
    mag = np.abs(x64) @ np.abs(deq).T
    if kind == KA8:
        gsum = np.abs(x64).reshape(M, -1, 64).sum(2)
        mag = mag + 2 * gsum @ np.abs(abias.astype(np.float64)).T
    et = (2 * (cols // bk) + 64) * U * mag + 2.0 ** -25 * np.abs(deq).sum(1)
    if tc:
        # fp32 accumulation over K/16 steps of three products; the low fp16 parts of
        # weights (|w - hi| < 2^-12 |w|) and activations may be subnormal: 2^-25 absolute each
        et = (3 * (cols // 16) + 64) * U * mag + 2.0 ** -25 * (np.abs(deq).sum(1) + np.abs(x64).sum(1)[:, None])
    if bias is not None:
        t = t + bias
        et = et + 2 * U * np.abs(t)
    if epi == 1:
        ref = _gelu(t)
        err_bound = 1.13 * et + 8 * U * (np.abs(ref) + 1e-6)
    elif epi == 2:
        g, u = t[:, 0::2], t[:, 1::2]
        ref = _silu(g) * u
        eg, eu = et[:, 0::2], et[:, 1::2]
        err_bound = 1.1 * eg * (np.abs(u) + eu) + np.abs(_silu(g)) * eu + 8 * U * (np.abs(ref) + 1e-6)
    else:
        ref = t
        err_bound = et
    if resid is not None:
        ref = ref + resid
        err_bound = err_bound + 2 * U * np.abs(ref)
    err = np.abs(y - ref)
    assert np.all(np.isfinite(y))
    worst = float(np.max(err / err_bound))
    assert worst <= 1.0, (worst, np.unravel_index(np.argmax(err / err_bound), err.shape))


SHAPES = {
    KQ8: [(3072, 1024), (1024, 4096), (200, 96), (64, 32)],
    KQ4: [(3072, 1024), (8192, 1024), (1024, 4096), (200, 96)],
    KA8: [(4096, 2048), (2048, 6144), (1024, 3072), (130, 128)],
}
CASES = [(k, s) for k, ss in SHAPES.items() for s in ss]


@pytest.mark.parametrize("M", [1, 37, 150, 300])
@pytest.mark.parametrize("kind,shape", CASES)
def test_gemm_linear_bias(sd, kind, shape, M):
    rows, cols = shape
    _run(sd, kind, rows, cols, M, 0, True, False, rows + cols + M + kind)


@pytest.mark.parametrize("kind", [KQ8, KQ4, KA8])
@pytest.mark.parametrize("M", [16, 150])
def test_gemm_gelu_and_residual(sd, kind, M):
    cols = 1024 if kind != KA8 else 2048
    _run(sd, kind, 4096, cols, M, 1, True, False, 11 + M + kind)
    _run(sd, kind, 1024, cols, M, 0, True, True, 12 + M + kind)


@pytest.mark.parametrize("kind", [KQ8, KQ4, KA8])
@pytest.mark.parametrize("M", [16, 200])
def test_gemm_swiglu(sd, kind, M):
    cols = 1024 if kind != KA8 else 2048
    _run(sd, kind, 8192 if kind != KA8 else 12288, cols, M, 2, False, False, 13 + M + kind)
    _run(sd, kind, 66, 64 if kind == KA8 else 96, M, 2, False, True, 14 + M + kind)


def test_gemm_rejects_bad_arguments(sd):
    w = (np.random.default_rng(0).standard_normal((64, 64)) * 0.02).astype(np.float32)
    canon, _ = _canon(KQ8, w)
    h = sd.sd_qmat_create(KQ8, canon, 64, 64)
    try:
        x = torch.zeros(4, 64, device="cuda")
        y = torch.zeros(4, 64, device="cuda")
        b = torch.zeros(64, device="cuda")
        for args in [(x, 0, 0, None, None, y), (x, 4, 3, None, None, y), (x, 4, 2, b, None, y)]:
            with pytest.raises(sd.SdError):
                sd.sd_qmat_gemm(h, *args)
    finally:
        sd.sd_qmat_destroy(h)


TC_SHAPES = [(KQ8, (3072, 1024)), (KQ8, (130, 128)), (KQ4, (3072, 1024)), (KQ4, (1024, 4096)), (KQ4, (200, 64)),
             (KA8, (4096, 2048)), (KA8, (2048, 6144)), (KA8, (130, 128))]


@pytest.mark.parametrize("M", [1, 37, 150, 300])
@pytest.mark.parametrize("kind,shape", TC_SHAPES)
def test_gemm_tc_linear_bias(sd, kind, shape, M):
    """The tcgen05 GEMM: ragged row counts (a partial 128-row tile), ragged
    output counts (a partial 128-column tile), one K step (cols 64) up to 96."""
    rows, cols = shape
    _run(sd, kind, rows, cols, M, 0, True, False, rows + cols + M + kind + 7, tc=True)


@pytest.mark.parametrize("kind", [KQ8, KQ4, KA8])
def test_gemm_tc_epilogues(sd, kind):
    cols = 1024 if kind != KA8 else 2048
    _run(sd, kind, 4096, cols, 150, 1, True, False, 21 + kind, tc=True)
    _run(sd, kind, 1024, cols, 150, 0, True, True, 22 + kind, tc=True)
    _run(sd, kind, 8192 if kind != KA8 else 12288, cols, 200, 2, False, False, 23 + kind, tc=True)
    _run(sd, kind, 66, 128, 16, 2, False, True, 24 + kind, tc=True)


def test_gemm_tc_rejects_unaligned_k(sd):
    w = (np.random.default_rng(0).standard_normal((64, 96)) * 0.02).astype(np.float32)
    canon, _ = _canon(KQ8, w)
    h = sd.sd_qmat_create(KQ8, canon, 64, 96)
    try:
        x = torch.zeros(4, 96, device="cuda")
        y = torch.zeros(4, 64, device="cuda")
        with pytest.raises(sd.SdError) as e:
            sd.sd_qmat_gemm_tc(h, x, 4, 0, None, None, y)
        assert e.value.code == -7
    finally:
        sd.sd_qmat_destroy(h)



G16_SHAPES = [(KQ8, (3072, 1024)), (KQ8, (200, 96)), (KQ8, (64, 32)), (KQ8, (1024, 4096)),
              (KQ4, (3072, 1024)), (KQ4, (200, 96)), (KQ4, (1024, 4096)), (KQ4, (130, 1088)),
              (KA8, (4096, 2048)), (KA8, (2048, 6144)), (KA8, (1024, 3072)), (KA8, (130, 128)), (KA8, (3072, 1024))]


@pytest.fixture(params=["tc", "skinny"])
def g16_path(request, monkeypatch):
    """The mma.sync skinny GEMM (default), and with SD_ROWS_GEMM=tc the tcgen05 one for
    8-bit affine weights (the other formats always take the mma.sync kernel)."""
    if request.param == "tc":
        monkeypatch.setenv("SD_ROWS_GEMM", "tc")
    else:
        monkeypatch.delenv("SD_ROWS_GEMM", raising=False)
    return request.param


@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
@pytest.mark.parametrize("kind,shape", G16_SHAPES)
def test_gemm16_linear_bias(sd, kind, shape, M, g16_path):
    """The skinny split-K GEMM: row counts up to 16 (one or both MMA row halves),
    ragged column tiles (200, 130 rows), K ranges that are and are not multiples
    of 64, one split (K = 32) up to many."""
    rows, cols = shape
    _run(sd, kind, rows, cols, M, 0, True, False, rows + cols + M + kind + 31, g16=True)


@pytest.mark.parametrize("kind", [KQ8, KQ4, KA8])
@pytest.mark.parametrize("M", [5, 16])
def test_gemm16_epilogues(sd, kind, M, g16_path):
    cols = 1024 if kind != KA8 else 2048
    _run(sd, kind, 4096, cols, M, 1, True, False, 41 + M + kind, g16=True)
    _run(sd, kind, 1024, cols, M, 0, True, True, 42 + M + kind, g16=True)
    _run(sd, kind, 8192 if kind != KA8 else 12288, cols, M, 2, False, False, 43 + M + kind, g16=True)
    _run(sd, kind, 66, 128, M, 2, False, True, 44 + M + kind, g16=True)


def test_gemm16_rejects_bad_arguments(sd):
    w = (np.random.default_rng(0).standard_normal((64, 64)) * 0.02).astype(np.float32)
    canon, _ = _canon(KQ8, w)
    h = sd.sd_qmat_create(KQ8, canon, 64, 64)
    try:
        x = torch.zeros(20, 64, device="cuda")
        y = torch.zeros(20, 64, device="cuda")
        b = torch.zeros(64, device="cuda")
        xm = torch.zeros(4 * 64 + 1, device="cuda")[1:]       # not 16-byte aligned
        for args in [(x, 17, 0, None, None, y), (x, 0, 0, None, None, y), (x, 4, 3, None, None, y),
                     (x, 4, 2, b, None, y), (xm, 4, 0, None, None, y)]:
            with pytest.raises(sd.SdError):
                sd.sd_qmat_gemm16(h, *args)
    finally:
        sd.sd_qmat_destroy(h)
