"""sd_attend_rows_static -- the attention entry point for callers that may
not allocate device memory while they run (for example a host thread with a
hard latency budget, or a framework that owns all device memory in its own
pool).  It must return what sd_attend_rows returns, call after call, with
its scratch in a fixed device array instead of per-call allocations.

Kept in a file that pytest collects last, so that a run stopping at the first
failure has already run every other test."""

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-5   # the attention tests' bound, relative to max |V|


@pytest.fixture(scope="module")
def sd():
    import __graft_entry__
    __graft_entry__.build()
    import autoregressive_speech_token_gb300 as pkg
    assert torch.cuda.is_available()
    return pkg


def _inputs(seed, B, H, Hkv, hd, n_ctx):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, hd)).astype(np.float32)
    k = (rng.standard_normal((B, Hkv, n_ctx, hd)) * 1.5).astype(np.float16)
    v = rng.standard_normal((B, Hkv, n_ctx, hd)).astype(np.float16)
    return (torch.from_numpy(q).cuda(), torch.from_numpy(k.view(np.uint16)).cuda(),
            torch.from_numpy(v.view(np.uint16)).cuda(), float(np.abs(v.astype(np.float32)).max()))


@pytest.mark.parametrize("B,H,Hkv,hd,n_ctx,n,nsplit", [(1, 16, 16, 64, 2048, 275, 8), (2, 16, 8, 128, 512, 425, 16)])
def test_static_scratch_matches_allocating_entry(sd, B, H, Hkv, hd, n_ctx, n, nsplit):
    # two calls in a row with different inputs: the second must not see the first's scratch
    for call, seed in enumerate((1, 2)):
        q, k, v, vmax = _inputs(seed + 10 * hd, B, H, Hkv, hd, n_ctx)
        n_call = n if call == 0 else n // 3 + 1
        ref = torch.empty(B, H, hd, dtype=torch.float32, device="cuda")
        out = torch.full((B, H, hd), float("nan"), dtype=torch.float32, device="cuda")
        sd.sd_attend_rows(q, k, v, B, H, Hkv, hd, n_ctx, n_call, nsplit, ref)
        sd.sd_attend_rows_static(q, k, v, B, H, Hkv, hd, n_ctx, n_call, nsplit, out)
        torch.cuda.synchronize()
        diff = (out - ref).abs().max().item()
        assert diff <= TOL * vmax, (call, diff)


def test_static_scratch_rejects_oversized_requests(sd):
    q, k, v, _ = _inputs(3, 1, 16, 16, 64, 64)
    out = torch.empty(1, 16, 64, dtype=torch.float32, device="cuda")
    # 16 rows x 32 heads x 64 chunks x 132 floats > 1048576
    with pytest.raises(sd.SdError) as e:
        sd.sd_attend_rows_static(q, k, v, 16, 32, 32, 128, 64, 64, 64, out)
    assert e.value.code == -1 and "scratch" in str(e.value)


def test_static_scratch_at_its_capacity_edges(sd):
    """need = B * Hkv * (H / Hkv * nsplit * (hd + 4) + 1) floats always has an odd
    factor above 1, so neither 2^20 nor 2^20 + 1 (= 17 * 61681) is a reachable
    size: the closest requests on each side are checked instead."""
    # 13 * 79 * 15 * 68 + 13 * 79 = 1048567 floats: 9 under the capacity -- accepted and correct
    B, H, Hkv, hd, n_ctx, n, nsplit = 13, 79, 79, 64, 64, 60, 15
    assert B * H * nsplit * (hd + 4) + B * Hkv == (1 << 20) - 9
    q, k, v, vmax = _inputs(5, B, H, Hkv, hd, n_ctx)
    ref = torch.empty(B, H, hd, dtype=torch.float32, device="cuda")
    out = torch.full((B, H, hd), float("nan"), dtype=torch.float32, device="cuda")
    sd.sd_attend_rows(q, k, v, B, H, Hkv, hd, n_ctx, n, nsplit, ref)
    sd.sd_attend_rows_static(q, k, v, B, H, Hkv, hd, n_ctx, n, nsplit, out)
    torch.cuda.synchronize()
    assert (out - ref).abs().max().item() <= TOL * vmax
    # 8 * 107 * 18 * 68 + 8 * 107 = 1048600 floats: 24 over -- rejected before any work
    B, H, Hkv, nsplit = 8, 107, 107, 18
    assert B * H * nsplit * (hd + 4) + B * Hkv == (1 << 20) + 24
    q, k, v, _ = _inputs(6, B, H, Hkv, hd, n_ctx)
    out = torch.empty(B, H, hd, dtype=torch.float32, device="cuda")
    with pytest.raises(sd.SdError) as e:
        sd.sd_attend_rows_static(q, k, v, B, H, Hkv, hd, n_ctx, n, nsplit, out)
    assert e.value.code == -1 and "scratch" in str(e.value)


def test_static_call_allocates_nothing(sd):
    """After one warm-up call, a call captured into a CUDA graph in global capture
    mode (where any cudaMalloc or cudaFree, from any thread, breaks the capture)
    records only its memset and kernel, and replaying the graph gives the
    allocating entry's result; the device's free memory is unchanged by a loop of
    calls."""
    B, H, Hkv, hd, n_ctx, n, nsplit = 2, 16, 8, 128, 512, 333, 8
    q, k, v, vmax = _inputs(7, B, H, Hkv, hd, n_ctx)
    ref = torch.empty(B, H, hd, dtype=torch.float32, device="cuda")
    out = torch.full((B, H, hd), float("nan"), dtype=torch.float32, device="cuda")
    sd.sd_attend_rows(q, k, v, B, H, Hkv, hd, n_ctx, n, nsplit, ref)
    sd.sd_attend_rows_static(q, k, v, B, H, Hkv, hd, n_ctx, n, nsplit, out)   # warm-up: address lookup
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(50):
        sd.sd_attend_rows_static(q, k, v, B, H, Hkv, hd, n_ctx, n, nsplit, out)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="global"):
        sd.sd_attend_rows_static(q, k, v, B, H, Hkv, hd, n_ctx, n, nsplit, out,
                                 torch.cuda.current_stream().cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    assert (out - ref).abs().max().item() <= TOL * vmax


def test_static_entry_matches_the_oracle(sd):
    """The static entry against the oracle's attention (plain loops, fp64 sums) at
    one shape, per (row, head): no device path in between."""
    import oracle
    B, H, Hkv, hd, n_ctx, n, nsplit = 2, 8, 2, 64, 300, 277, 6
    q, k, v, vmax = _inputs(8, B, H, Hkv, hd, n_ctx)
    out = torch.empty(B, H, hd, dtype=torch.float32, device="cuda")
    sd.sd_attend_rows_static(q, k, v, B, H, Hkv, hd, n_ctx, n, nsplit, out)
    torch.cuda.synchronize()
    qh, kh, vh, got = q.cpu().numpy(), k.cpu().numpy(), v.cpu().numpy(), out.cpu().numpy()
    for b in range(B):
        for h in range(H):
            g = h // (H // Hkv)
            want = oracle.attend(qh[b, h], kh[b, g, :n], vh[b, g, :n])
            assert np.abs(got[b, h] - want).max() <= TOL * vmax, (b, h)
