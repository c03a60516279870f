"""Parity of the device sampler ladder (sd_sample_rows_ladder) with the
oracle's ladder on the same logits: CFG combine, repetition penalty,
temperature, min_p, top-p, top-k and the index-order draw, over vocabulary
sizes from 16 to 16384, random histories and draws, the greedy path, ties at
the thresholds, and argument checks.  Both sides compute in double precision,
so tokens must agree except where the draw lies within 1e-9 of a CDF edge."""

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

F32 = np.float32


@pytest.fixture(scope="module")
def sd():
    import __graft_entry__
    __graft_entry__.build()
    import autoregressive_speech_token_gb300 as pkg
    assert torch.cuda.is_available()
    return pkg


def _run(sd, zc, zu, seen, params, us):
    rows, V = zc.shape
    w, pen, T, min_p, top_p, k = params
    s = sd.SamplerLadder(w, pen, T, min_p, top_p, k)
    zc_d = torch.from_numpy(zc).cuda()
    zu_d = torch.from_numpy(zu).cuda() if zu is not None else None
    sn_d = torch.from_numpy(seen).cuda() if seen is not None else None
    u_d = torch.from_numpy(np.asarray(us, F32)).cuda()
    out = torch.zeros(rows, dtype=torch.int32, device="cuda")
    sd.sd_sample_rows_ladder(zc_d, zu_d, rows, V, s, sn_d, u_d, out, torch.cuda.current_stream().cuda_stream)
    return out.cpu().numpy()


def _compare(sd, zc, zu, seen, params, n_u=48, seed=0):
    rng = np.random.default_rng(seed)
    rows = zc.shape[0]
    checked = 0
    for rep in range(n_u // rows + 1):
        us = rng.random(rows).astype(F32)
        got = _run(sd, zc, zu, seen, params, us)
        w, pen, T, min_p, top_p, k = params
        for b in range(rows):
            # both sides compute the ladder in double precision from the same inputs, so only a
            # draw within 1e-9 of a CDF edge may go either way (exact ties at a threshold do not:
            # both sides break them by the same rule)
            tok, _, dd = oracle.sample_ladder(zc[b], zu[b] if zu is not None else None, w,
                                              seen[b] if seen is not None else None, pen, T, min_p, top_p, k,
                                              float(us[b]), with_draw=True)
            if dd >= 1e-9:
                assert int(got[b]) == tok, (params, b, float(us[b]), int(got[b]), tok, dd)
                checked += 1
    assert checked > 0


COMBOS = [(0.0, 1.0, 1.0, 0.0, 1.0, 0), (0.5, 1.3, 0.8, 0.05, 0.9, 8), (1.0, 1.05, 0.9, 0.0, 0.95, 50),
          (-0.5, 2.0, 1.2, 0.2, 0.7, 3), (0.0, 1.0, 0.7, 0.3, 1.0, 0), (2.0, 1.5, 1.0, 0.01, 0.8, 1000)]


@pytest.mark.parametrize("V", [16, 2048, 3072, 6563, 8192, 8194, 16384])
def test_ladder_matches_oracle(sd, V):
    rng = np.random.default_rng(V)
    rows = 4
    zc = (rng.standard_normal((rows, V)) * 2).astype(F32)
    zu = (zc + rng.standard_normal((rows, V))).astype(F32)
    seen = (rng.random((rows, V)) < 0.1).astype(np.uint8)
    for i, params in enumerate(COMBOS):
        _compare(sd, zc, zu, seen, params, seed=V + i)
    # no unconditional logits and no history
    _compare(sd, zc, None, None, (0.0, 1.0, 0.9, 0.0, 0.95, 50), seed=V + 99)


def test_ladder_greedy_is_argmax_of_the_penalised_combination(sd):
    rng = np.random.default_rng(5)
    zc = (rng.standard_normal((3, 300)) * 2).astype(F32)
    zu = (rng.standard_normal((3, 300)) * 2).astype(F32)
    seen = (rng.random((3, 300)) < 0.3).astype(np.uint8)
    got = _run(sd, zc, zu, seen, (0.7, 1.8, 0.0, 0.0, 1.0, 0), [0.5] * 3)
    for b in range(3):
        assert int(got[b]) == oracle.sample_ladder(zc[b], zu[b], 0.7, seen[b], 1.8, 0.0)[0]


def test_ladder_threshold_ties(sd):
    # ties at the top-k threshold are kept; equal leaders under min_p = 1; an exact top-p boundary
    z = np.array([3, 1, 2, 2, 2, 0, -1, 2, 1, 1, 0, 0, -2, -3, 5, 2], F32)
    _compare(sd, np.stack([z] * 4), None, None, (0.0, 1.0, 1.0, 0.0, 1.0, 3), n_u=64)
    z2 = np.array([0.1, 2.0, -1.0, 2.0, 1.9, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0, 0.0], F32)
    _compare(sd, np.stack([z2] * 4), None, None, (0.0, 1.0, 0.7, 1.0, 1.0, 0), n_u=64)
    z3 = np.full(16, -80.0, F32)
    z3[4] = z3[9] = 10.0
    _compare(sd, np.stack([z3] * 4), None, None, (0.0, 1.0, 1.0, 0.0, 0.5, 0), n_u=64)


def test_ladder_rejects_bad_arguments(sd):
    z = torch.zeros(2, 16, device="cuda")
    u = torch.zeros(2, device="cuda")
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    big = torch.zeros(1, 16385, device="cuda")
    with pytest.raises(sd.SdError):
        sd.sd_sample_rows_ladder(big, None, 1, 16385, sd.SamplerLadder(0, 1, 1, 0, 1, 0), None, u, out, st)
    for bad in [sd.SamplerLadder(0, 1, 1, 0, 0.0, 0), sd.SamplerLadder(0, 0.0, 1, 0, 1, 0),
                sd.SamplerLadder(0, 1, 1, -0.5, 1, 0)]:
        with pytest.raises(sd.SdError):
            sd.sd_sample_rows_ladder(z, None, 2, 16, bad, None, u, out, st)
