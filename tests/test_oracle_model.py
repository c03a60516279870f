"""Whole-forward pins of the oracle: its incremental KV-cache decode against an
independent full causal recompute in torch float64 (tests/torch_ref.py), on
small GPT-2, Llama (with grouped KV heads) and Talker + code-predictor models,
plus closed-form special cases."""

import dataclasses

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from synth import get_preset, uniform_draws, prompt_tokens
from synth import presets as P
from synth.presets import SamplerSpec
from synth.weights import build_model_blob
from tests import torch_ref

TOL = 2e-5   # fp32 rounding noise, relative to the largest logit magnitude


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.max(np.abs(a - b)) / np.max(np.abs(b))


def _small_llama():
    return P.ModelSpec(arch=P.ARCH_LLAMA, n_layer=2, d_model=256, n_head=4, n_kv_head=2, head_dim=64,
                       d_ff=512, vocab=300, max_ctx=64, batch=2, quant=P.Q4_0)


def _small_qwen():
    return P.ModelSpec(arch=P.ARCH_QWEN_TTS, n_layer=2, d_model=256, n_head=4, n_kv_head=2, head_dim=64,
                       d_ff=512, vocab=128, max_ctx=64, batch=1, quant=P.A8G64,
                       cp_layer=2, cp_d_model=128, cp_n_head=2, cp_n_kv_head=2, cp_head_dim=64,
                       cp_d_ff=256, cp_vocab=64, n_codebooks=16, cp_max_ctx=16)


def test_tiny_gpt2_incremental_equals_full_recompute():
    run = get_preset("tiny")
    m = run.model
    blob, _ = build_model_blob(m)
    model = oracle.Model(blob)
    prompt = prompt_tokens(run)
    n = 16
    draws = uniform_draws(run.draw_seed, n + 1, 1)[..., 0]
    tr = oracle.run_t3(model, m, prompt, draws, n, run.sampler)[0]
    seq = list(prompt[0]) + tr.tokens[:n]
    ref = torch_ref.t3_logits(blob, m, seq)
    P_ = prompt.shape[1]
    for i in range(n + 1):
        assert _rel(tr.logits[i], ref[P_ - 1 + i]) < TOL, i
    # greedy tokens are the argmax of the recomputed logits wherever the margin is clear
    for i in range(n + 1):
        if tr.margins[i] > 1e-4:
            assert tr.tokens[i] == int(np.argmax(ref[P_ - 1 + i]))


@pytest.mark.parametrize("quant", [P.Q4_0, P.Q5_0])
def test_q4_gpt2_sampled_run_matches_recompute(quant):
    run = get_preset("tiny").with_model(quant=quant, n_layer=1)
    m = run.model
    blob, _ = build_model_blob(m)
    model = oracle.Model(blob)
    prompt = prompt_tokens(run)[:, :10]
    n = 8
    draws = uniform_draws(3, n + 1, 1)[..., 0]
    s = SamplerSpec(temperature=0.8, top_k=1000, top_p=0.95, greedy=False)
    tr = oracle.run_t3(model, m, prompt, draws, n, s)[0]
    ref = torch_ref.t3_logits(blob, m, list(prompt[0]) + tr.tokens[:n])
    for i in range(n + 1):
        assert _rel(tr.logits[i], ref[9 + i]) < TOL


def test_llama_gqa_rows_match_full_recompute():
    m = _small_llama()
    blob, _ = build_model_blob(m)
    model = oracle.Model(blob)
    rng = np.random.default_rng(5)
    prompt = rng.integers(0, m.vocab, size=(2, 12)).astype(np.int32)
    n = 10
    draws = uniform_draws(3, n + 1, 2)[..., 0]
    s = SamplerSpec(temperature=0.8, top_k=50, top_p=0.9, greedy=False)
    trs = oracle.run_t3(model, m, prompt, draws, n, s)
    for b in range(2):
        ref = torch_ref.t3_logits(blob, m, list(prompt[b]) + trs[b].tokens[:n])
        for i in range(n + 1):
            assert _rel(trs[b].logits[i], ref[11 + i]) < TOL, (b, i)


@pytest.mark.parametrize("arch", [P.ARCH_GPT2, P.ARCH_LLAMA])
def test_conditioning_prefix_matches_full_recompute(arch):
    """A prompt given as input vectors (a conditioning prefix) instead of token
    IDs: the logits equal a full recompute whose first positions take those
    vectors; and vectors equal to the tokens' embedding rows give the token
    prompt's run bit for bit."""
    if arch == P.ARCH_GPT2:
        m = dataclasses.replace(get_preset("tiny").model, n_layer=1, batch=2)
    else:
        m = _small_llama()
    blob, fp32 = build_model_blob(m, keep_fp32=True)
    rng = np.random.default_rng(8)
    P_, n = 10, 6
    emb = (rng.standard_normal((2, P_, m.d_model)) * 0.05).astype(np.float32)
    prompt = np.zeros((2, P_), np.int32)
    draws = uniform_draws(4, n + 1, 2)[..., 0]
    s = SamplerSpec(temperature=0.8, top_k=50, top_p=0.9, greedy=False)
    trs = oracle.run_t3(oracle.Model(blob), m, prompt, draws, n, s, prompt_embeds=emb)
    for b in range(2):
        ref = torch_ref.t3_logits(blob, m, [0] * P_ + trs[b].tokens[:n], prefix=emb[b])
        for i in range(n + 1):
            assert _rel(trs[b].logits[i], ref[P_ - 1 + i]) < TOL, (b, i)
    toks = rng.integers(0, m.vocab, size=(2, P_)).astype(np.int32)
    rows = fp32["wte"][toks]
    a = oracle.run_t3(oracle.Model(blob), m, toks, draws, n, s)
    e = oracle.run_t3(oracle.Model(blob), m, toks, draws, n, s, prompt_embeds=rows)
    for b in range(2):
        assert a[b].tokens == e[b].tokens
        assert all(np.array_equal(x, y) for x, y in zip(a[b].logits, e[b].logits))


def _cfg_run(ladder, n=10, seed=5):
    m = _small_llama()
    blob, _ = build_model_blob(m)
    rng = np.random.default_rng(seed)
    prompt = rng.integers(0, m.vocab, size=(2, 12)).astype(np.int32)
    draws = uniform_draws(3, n + 1, 1)[:, 0, 0]
    return m, blob, prompt, draws, oracle.run_t3_cfg(oracle.Model(blob), m, prompt, draws, n, ladder)


def test_cfg_rows_both_consume_the_ladder_token():
    """Both rows are fed the one picked token: each row's logits equal a full
    recompute of its own prompt followed by the picked tokens."""
    n = 10
    m, blob, prompt, draws, tr = _cfg_run(P.LadderSpec(), n)
    for b in range(2):
        ref = torch_ref.t3_logits(blob, m, list(prompt[b]) + tr.tokens[:n])
        for i in range(n + 1):
            assert _rel(tr.logits[i][b], ref[11 + i]) < TOL, (b, i)


def test_cfg_run_with_neutral_stages_is_the_plain_run_of_a_row():
    """Guidance weight 0 with no penalty, min_p or top-p samples the conditional
    row like the plain sampler; weight -1 samples the unconditional row."""
    n = 10
    for w, row in ((0.0, 0), (-1.0, 1)):
        lad = P.LadderSpec(cfg_weight=w, rep_penalty=1.0, temperature=0.8, min_p=0.0, top_p=1.0, top_k=50)
        m, blob, prompt, draws, tr = _cfg_run(lad, n)
        d2 = np.stack([draws, draws], axis=1)
        plain = oracle.run_t3(oracle.Model(blob), m, prompt, d2, n,
                              SamplerSpec(temperature=0.8, top_k=50, top_p=1.0, greedy=False))[row]
        assert tr.tokens == plain.tokens, (w, tr.tokens, plain.tokens)


def test_cfg_history_holds_the_fed_tokens_only():
    """Greedy with a huge repetition penalty: the first token is the plain
    argmax of the combined logits (the prompt is not in the history), and no
    fed token is picked again; without the penalty the same model repeats."""
    n = 24
    big = P.LadderSpec(cfg_weight=0.5, rep_penalty=1e6, temperature=0.0, min_p=0.0, top_p=1.0, top_k=1)
    m, blob, prompt, draws, tr = _cfg_run(big, n)
    zc, zu = (np.asarray(z, np.float64) for z in tr.logits[0])
    assert tr.tokens[0] == int(np.argmax(zc + 0.5 * (zc - zu)))
    assert len(set(tr.tokens)) == n + 1, tr.tokens
    none = dataclasses.replace(big, rep_penalty=1.0)
    _, _, _, _, tr0 = _cfg_run(none, n)
    assert len(set(tr0.tokens)) < n + 1, tr0.tokens


@pytest.mark.parametrize("cp_quant", [0, P.A4G32, P.A4G64])
def test_qwen_frames_match_full_recompute(cp_quant):
    """The Talker in 8-bit affine, the code predictor in its own format (4-bit
    group 32 / 64 included: the blob records each tensor's format)."""
    m = dataclasses.replace(_small_qwen(), cp_quant=cp_quant)
    blob, _ = build_model_blob(m)
    model = oracle.Model(blob)
    prompt = np.random.default_rng(6).integers(0, m.vocab, size=(1, 9)).astype(np.int32)
    nf = 3
    draws = uniform_draws(3, nf + 1, 1, 16)
    s = SamplerSpec(temperature=0.9, top_k=50, top_p=0.95, greedy=False)
    tr = oracle.run_qwen(model, m, prompt, draws, nf, s, s)[0]
    ref = torch_ref.qwen_frame_logits(blob, m, prompt[0], tr.tokens)
    for f in range(nf + 1):
        for j in range(16):
            assert _rel(tr.logits[f][j], ref[f][j]) < TOL, (f, j)


def test_qwen_talker_penalty_history_is_the_fed_codes():
    """Greedy Talker with a huge repetition penalty: frame 0's code 0 is the plain
    argmax (the prompt is not in the history) and no codebook-0 token fed forward
    is picked again."""
    m = _small_qwen()
    blob, _ = build_model_blob(m)
    prompt = np.random.default_rng(9).integers(0, m.vocab, size=(1, 6)).astype(np.int32)
    nf = 14
    draws = uniform_draws(5, nf + 1, 1, 16)
    talker = SamplerSpec(greedy=True, rep_penalty=1e6)
    cp = SamplerSpec(temperature=0.9, top_k=50, top_p=0.95, greedy=False)
    tr = oracle.run_qwen(oracle.Model(blob), m, prompt, draws, nf, talker, cp)[0]
    c0 = [f[0] for f in tr.tokens]
    assert c0[0] == int(np.argmax(tr.logits[0][0]))
    assert len(set(c0)) == nf + 1, c0


def test_qwen_rows_sharing_a_prompt_match_full_recompute():
    """Rows whose prompt equals an earlier row's start from a copy of that row's
    cache (run_qwen's shortcut for G rollouts of one prompt); every row's frames
    still match an independent full recompute of its own tokens."""
    import dataclasses
    m = dataclasses.replace(_small_qwen(), batch=3)
    blob, _ = build_model_blob(m)
    model = oracle.Model(blob)
    rng = np.random.default_rng(7)
    prompt = rng.integers(0, m.vocab, size=(3, 7)).astype(np.int32)
    prompt[2] = prompt[0]
    nf = 2
    draws = uniform_draws(5, nf + 1, 3, 16)
    s = SamplerSpec(temperature=0.9, top_k=50, top_p=0.95, greedy=False)
    trs = oracle.run_qwen(model, m, prompt, draws, nf, s, s)
    for b in range(3):
        ref = torch_ref.qwen_frame_logits(blob, m, prompt[b], trs[b].tokens)
        for f in range(nf + 1):
            for j in range(16):
                # 5 x TOL: over three frames an fp16 cache rounding may tip between the two
                # computations; a wrong or missing copy errs by the logits' own size
                assert _rel(trs[b].logits[f][j], ref[f][j]) < 5 * TOL, (b, f, j)
    assert np.array_equal(trs[0].logits[0][0], trs[2].logits[0][0])


def test_zero_layer_model_is_head_of_norm_of_embedding():
    m = P.ModelSpec(arch=P.ARCH_GPT2, n_layer=0, d_model=128, n_head=2, n_kv_head=2, head_dim=64,
                    d_ff=256, vocab=200, max_ctx=16, batch=1, quant=P.Q8_0)
    blob, _ = build_model_blob(m)
    model = oracle.Model(blob)
    W = torch_ref.Weights(blob)
    for pos, tok in enumerate([5, 199, 0]):
        z = model.token_forward(0, tok, m.vocab)
        x = (W.get("wte")[tok].float() + W.get("wpe")[pos].float()).double()
        h = F.layer_norm(x, (128,), W.vec("lnf.g"), W.vec("lnf.b"), eps=1e-5).float().double()
        ref = (h @ W.get("whead").T).numpy()
        assert _rel(z, ref) < 1e-6


def test_threads_do_not_change_results():
    run = get_preset("tiny")
    blob, _ = build_model_blob(run.model)
    prompt = prompt_tokens(run)[:, :6]
    out = []
    for th in (1, 4):
        model = oracle.Model(blob, threads=th)
        z = None
        for t in prompt[0]:
            z = model.token_forward(0, int(t), run.model.vocab)
        out.append(z)
    assert np.array_equal(out[0], out[1])


def test_context_full_and_bad_token_rejected():
    m = P.ModelSpec(arch=P.ARCH_GPT2, n_layer=1, d_model=64, n_head=1, n_kv_head=1, head_dim=64,
                    d_ff=128, vocab=50, max_ctx=3, batch=1, quant=P.Q8_0)
    blob, _ = build_model_blob(m)
    model = oracle.Model(blob)
    with pytest.raises(ValueError):
        model.token_forward(0, 50, 50)
    for t in range(3):
        model.token_forward(0, t, 50)
    with pytest.raises(ValueError):
        model.token_forward(0, 1, 50)
    model.reset()
    assert model.pos(0) == 0
