"""Seeded input generators: Philox, quantised storage formats, byte model."""

import numpy as np
import pytest

from synth import get_preset, philox4x32_10, uniform_draws, PRESETS
from synth import presets as P
from synth.blob import read_table, KIND_Q4_0, KIND_Q8_0, KIND_A8G64
from synth.weights import build_model_blob, quantize_q4_0, quantize_q8_0, quantize_a8g64, prompt_tokens
from tests.conftest import golden_path, read_kv_golden


def test_philox_known_answers():
    rows = []
    with open(golden_path("philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append([int(t, 16) for t in line.split()])
    assert len(rows) == 3
    for r in rows:
        out = philox4x32_10(np.array(r[:4], np.uint32), (r[4], r[5]))
        assert [int(v) for v in out] == r[6:]


def test_uniform_draws_grid():
    u = uniform_draws(3, 50, 4, 16)
    assert u.shape == (50, 4, 16) and u.dtype == np.float32
    assert (u >= 0).all() and (u < 1).all()
    # every draw sits on the 2^-24 grid, so fp32 holds it exactly
    assert np.all((u.astype(np.float64) * 2 ** 24) == np.floor(u.astype(np.float64) * 2 ** 24))
    # counter-based: a window equals the corresponding slice of a longer run
    assert np.array_equal(uniform_draws(3, 5, 4, 16, step0=10), u[10:15])
    assert abs(u.mean() - 0.5) < 0.02


def test_q4_0_layout_matches_page():
    g = read_kv_golden("page_byte_counts.txt")
    w = np.random.default_rng(0).standard_normal((3, 1024)).astype(np.float32)
    q = quantize_q4_0(w)
    assert q.shape[-1] == g["q4_0_block_bytes"]
    assert q.reshape(3, -1).shape[1] == g["q4_0_row_bytes_k1024"]


def test_q4_0_nibble_order_and_scale():
    # block whose largest-magnitude element is negative: d = m / -8 is positive
    w = np.zeros((1, 32), np.float32)
    w[0, :] = np.linspace(-0.7, 0.5, 32, dtype=np.float32)
    w[0, 3] = -1.6
    q = quantize_q4_0(w)[0, 0]
    d = np.frombuffer(q[:2].tobytes(), np.float16)[0]
    assert float(d) == pytest.approx(0.2, rel=1e-3)
    codes = np.concatenate([q[2:] & 0xF, q[2:] >> 4])
    assert codes[3] == 0                     # the extreme element maps to code 0 exactly
    rec = float(d) * (codes.astype(np.float32) - 8)
    # codes are rounded with the fp32 scale, the stored scale is fp16: |d32 - d16| <= |d| 2^-11
    assert np.max(np.abs(rec - w[0])) <= float(d) / 2 + 8 * float(d) * 2 ** -11


def test_q8_0_basic():
    w = np.random.default_rng(1).standard_normal((4, 64)).astype(np.float32)
    q = quantize_q8_0(w)
    assert q.shape == (4, 2, 34)
    codes = q[..., 2:].view(np.int8)
    assert np.abs(codes).max() == 127


def test_affine_bits_per_weight_matches_page():
    g = read_kv_golden("page_byte_counts.txt")
    q, s, b = quantize_a8g64(np.random.default_rng(2).standard_normal((2, 128)).astype(np.float32))
    bits = 8 * (q.nbytes + s.nbytes + b.nbytes) / q.size
    assert bits == g["p3_affine_bits_per_weight"]
    assert P.BYTES_PER_WEIGHT[P.A8G64] * 8 == g["p3_affine_bits_per_weight"]


def test_param_model_matches_page_counts():
    """The byte model used for the roofline reproduces the blog's printed counts
    for its own 0.6B shapes (Talker hidden 1024, MLP 3072, 16/8 heads of 128)."""
    g = read_kv_golden("page_byte_counts.txt")
    m = P.ModelSpec(arch=P.ARCH_QWEN_TTS, n_layer=28, d_model=1024, n_head=16, n_kv_head=8, head_dim=128,
                    d_ff=3072, vocab=3072, max_ctx=512, batch=1, quant=P.A8G64,
                    cp_layer=5, cp_d_model=1024, cp_n_head=16, cp_n_kv_head=8, cp_head_dim=128,
                    cp_d_ff=3072, cp_vocab=2048, n_codebooks=16, cp_max_ctx=16)
    per_layer = (m.talker_params() - m.vocab * m.d_model) / m.n_layer
    assert round(per_layer / 1e6, 1) == g["p3_talker_params_per_layer_m"]
    assert round(m.talker_params() / 1e6, 1) == g["p3_talker_params_per_step_m"]
    assert round(m.cp_pass_params() / 1e6, 1) == g["p3_cp_params_per_pass_m"]
    assert m.kv_bytes_per_position() / 1024 == g["p3_kv_bytes_per_token_kib"]
    cp_frame = 15 * m.cp_pass_params() * P.BYTES_PER_WEIGHT[P.A8G64]
    assert round(cp_frame / 1e9, 2) == g["p3_cp_frame_gb_q8"]


def test_workload_param_counts():
    assert PRESETS["gpt2m_q4"].model.quantised_params_per_step() == 308_710_400
    llama = PRESETS["llama_q4"].model
    assert round(llama.quantised_params_per_step() / 1e6, 1) == 511.7
    q = PRESETS["qwen_a8"].model
    assert round(q.talker_params() / 1e9, 3) == 1.416
    assert round(q.cp_pass_params() / 1e6, 1) == 70.3


def test_blob_table_and_determinism():
    run = get_preset("tiny")
    b1, _ = build_model_blob(run.model)
    b2, _ = build_model_blob(run.model)
    assert np.array_equal(b1, b2)
    t = read_table(b1)
    assert t["l0.wqkv"][0] == KIND_Q8_0 and t["l0.wqkv"][1:3] == (768, 256)
    assert all(v[3] % 256 == 0 for v in t.values())
    q4 = run.with_model(quant=P.Q4_0)
    t4 = read_table(build_model_blob(q4.model)[0])
    assert t4["whead"][0] == KIND_Q4_0 and t4["whead"][4] == 6561 * 8 * 18


def test_prompt_tokens():
    run = get_preset("llama_q4")
    p = prompt_tokens(run)
    assert p.shape == (2, 200) and p.min() >= 0 and p.max() < 8192
    assert not np.array_equal(p[0], p[1])
    g = prompt_tokens(get_preset("qwen_a8_g16"))
    assert g.shape == (16, 300) and (g == g[0]).all()


def test_affine_blob_kind():
    run = get_preset("qwen_a8").with_model(n_layer=1, cp_layer=1, d_model=128, d_ff=256, n_head=2,
                                           n_kv_head=1, head_dim=64, vocab=64, cp_d_model=64,
                                           cp_d_ff=128, cp_n_head=1, cp_n_kv_head=1, cp_head_dim=64,
                                           cp_vocab=32, n_codebooks=4)
    t = read_table(build_model_blob(run.model)[0])
    assert t["t0.wqkv"][0] == KIND_A8G64
    kind, rows, cols, off, nb = t["cp.proj"]
    assert nb == rows * cols + 2 * 2 * rows * cols // 64


def test_with_batch_equals_a_blob_built_for_that_batch():
    import dataclasses
    from synth import get_preset
    from synth.blob import with_batch
    from synth.weights import build_model_blob
    run = get_preset("tiny")
    a = build_model_blob(run.model)[0]
    b = build_model_blob(dataclasses.replace(run.model, batch=3))[0]
    assert np.array_equal(with_batch(a, 3), b)
