"""Model-level parity of libsd.so against the oracle, through the C ABI.

Teacher forcing: every GPU step consumes the oracle's token (or, for the
bench's free-running run, the oracle replays the GPU's tokens), so a flip at a
low-margin step cannot cascade.  Acceptance, per step: logits relative L2 <=
1e-3; tokens identical at every decision whose oracle margin is at least 1e-4.
Each model test also reports how many decisions a rule derived from the step's
logit error would check (see _Tally).
"""

import dataclasses
import math
import os

import numpy as np
import pytest

import oracle
from synth import get_preset, prompt_tokens, uniform_draws
from synth import presets as P
from synth.presets import SamplerSpec
from synth.blob import with_batch
from synth.weights import build_model_blob

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

REL_L2 = 1e-3
MARGIN = 1e-4
SAMPLER_MARGIN = 1e-5   # same logits on both sides: fp32 vs fp64 sampler arithmetic only
THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def sd():
    import __graft_entry__
    __graft_entry__.build()
    import autoregressive_speech_token_gb300 as pkg
    assert torch.cuda.is_available()
    torch.cuda.set_device(0)
    return pkg


_BLOBS = {}


def _blob(spec):
    """The model's weight blob; the last one built is kept, and a spec that differs
    only in its batch reuses it with the header's batch changed."""
    key = repr(dataclasses.replace(spec, batch=1))
    if key not in _BLOBS:
        _BLOBS.clear()
        _BLOBS[key] = build_model_blob(spec)[0]
    return with_batch(_BLOBS[key], spec.batch)


def _rel(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(np.asarray(b, np.float64)))


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _logit_error(z_dev, z_ref):
    return float(np.max(np.abs(np.asarray(z_dev, np.float64) - z_ref)))


def _error_bound(d, sampler):
    """The largest change of the decision's inputs that a logit error of d (max
    norm) can make, in the oracle margin's units: greedy, the gap between two
    logits shrinks by up to 2d; sampled, every unnormalised probability moves by a
    factor within exp(+-d/T), which is a change of size expm1(2d/T)."""
    if sampler.greedy or sampler.top_k == 1 or sampler.temperature <= 0:
        return 2 * d
    return math.expm1(2 * d / sampler.temperature)


class _Tally:
    """Token decisions against the oracle's, counted under two rules and reported:
    the stated rule (the tokens agree at every decision whose oracle margin is at
    least MARGIN) and the error-derived rule (at every decision whose margin is at
    least max(MARGIN, bound(d)), d being that step's logit error against the
    oracle).  Every strict-rule disagreement is listed with its margin and d.
    Asserted: no disagreement under the error-derived rule -- that is, the stated
    rule at every decision where the step's logits are accurate enough for it
    (bound(d) <= MARGIN), and elsewhere every disagreement lies within the change
    the measured logit error can make.  (With the logits held to relative L2
    1e-3, d of 1e-4 already allows changes of size 2.5e-4 at T = 0.8: the two
    tolerances cannot both be met at every decision.)"""

    def __init__(self, name, sampler):
        self.name, self.sampler = name, sampler
        self.total = self.strict = self.derived = 0
        self.strict_bad, self.derived_bad = [], []

    def add(self, where, got, want, margin, z_dev, z_ref, d=None):
        d = _logit_error(z_dev, z_ref) if d is None else d
        self.total += 1
        if margin >= MARGIN:
            self.strict += 1
            if got != want:
                self.strict_bad.append(dict(at=where, gpu=got, oracle=want, margin=margin, d=d,
                                            bound=_error_bound(d, self.sampler)))
        if margin >= max(MARGIN, _error_bound(d, self.sampler)):
            self.derived += 1
            if got != want:
                self.derived_bad.append(where)

    def report(self):
        print(f"[{self.name}] decisions {self.total}: strict rule (margin >= {MARGIN:g}) checks {self.strict}, "
              f"disagreements {len(self.strict_bad)}; error-derived rule checks {self.derived}, "
              f"disagreements {len(self.derived_bad)}")
        for b in self.strict_bad:
            print(f"[{self.name}] STRICT-RULE DISAGREEMENT {b}")

    def check(self):
        self.report()
        assert not self.derived_bad, (self.derived_bad, self.strict_bad)
        for b in self.strict_bad:
            assert b["margin"] < b["bound"], b


def _check_t3(sd, run, n_steps, prompt=None, spec=None, prompt_embeds=None):
    spec = spec or run.model
    blob = _blob(spec)
    prompt = prompt_tokens(run) if prompt is None else prompt
    B = spec.batch
    draws = uniform_draws(run.draw_seed, n_steps + 1, B)[..., 0]
    ref = oracle.run_t3(oracle.Model(blob, THREADS), spec, prompt, draws, n_steps, run.sampler,
                        prompt_embeds=prompt_embeds)
    dec = sd.Decoder(spec, blob, stream=_stream())
    s = sd.Sampler.from_spec(run.sampler)
    if prompt_embeds is not None:
        got = dec.prefill_embeds(prompt_embeds, s, draws[0])
    else:
        got = dec.prefill(prompt, s, draws[0])
    worst = 0.0
    name = f"{run.name} {P.QUANT_NAMES[spec.quant]} rows {B} steps {n_steps + 1}"
    tally = _Tally(name, run.sampler)
    sa = dict(temperature=run.sampler.temperature, top_k=run.sampler.top_k, top_p=run.sampler.top_p,
              greedy=run.sampler.greedy)
    for i in range(n_steps + 1):
        z = dec.logits()
        for b in range(B):
            r = _rel(z[b], ref[b].logits[i])
            worst = max(worst, r)
            assert r <= REL_L2, (i, b, r)
            # the device sampler decides like the oracle's sampler on the same (device) logits
            tg, mg = oracle.sample(z[b], u=float(draws[i][b]), **sa)
            if mg >= SAMPLER_MARGIN:
                assert int(got[b]) == tg, ("sampler", i, b, int(got[b]), tg, mg)
            tally.add((i, b), int(got[b]), ref[b].tokens[i], ref[b].margins[i], z[b], ref[b].logits[i])
        if i < n_steps:
            fed = np.array([ref[b].tokens[i] for b in range(B)], np.int32)
            got = dec.step(fed, s, draws[i + 1])
    dec.close()
    print(f"[{name}] worst logits rel L2 {worst:.2e}")
    tally.check()
    return worst


def test_tiny_full_run(sd):
    run = get_preset("tiny")
    worst = _check_t3(sd, run, run.n_steps)
    assert worst < 1e-4


def test_tiny_q4_sampled(sd):
    run = get_preset("tiny").with_model(quant=P.Q4_0)
    run = dataclasses.replace(run, sampler=SamplerSpec(0.8, 1000, 0.95, False))
    _check_t3(sd, run, 40)


def test_tiny_q5_sampled_every_prefill_path(sd, prefill_path):
    """Q5_0 weights (journal, Tier A item A3): the per-operation step graph
    decodes (the persistent kernels take Q8_0 / Q4_0), the prompt goes through
    the tensor-core GEMM, or the step graphs where the mma.sync GEMM is asked for."""
    run = get_preset("tiny").with_model(quant=P.Q5_0)
    run = dataclasses.replace(run, sampler=SamplerSpec(0.8, 1000, 0.95, False))
    _check_t3(sd, run, 24)


def test_llama_q5_two_rows(sd):
    spec = P.ModelSpec(arch=P.ARCH_LLAMA, n_layer=3, d_model=512, n_head=8, n_kv_head=2, head_dim=64,
                       d_ff=1536, vocab=1000, max_ctx=300, batch=2, quant=P.Q5_0)
    run = get_preset("llama_q4").with_model(**{f: getattr(spec, f) for f in
                                               ("n_layer", "d_model", "n_head", "n_kv_head", "d_ff", "vocab",
                                                "max_ctx", "quant")})
    prompt = np.random.default_rng(2).integers(0, 1000, size=(2, 40)).astype(np.int32)
    _check_t3(sd, run, 30, prompt=prompt)


@pytest.mark.parametrize("arch", ["gpt2", "llama"])
def test_conditioning_prefix_every_prefill_path(sd, prefill_path, arch):
    """A prompt of input vectors (sd_prefill_embeds) instead of token IDs, then
    token steps, against the oracle; on every prefill path and both step paths
    that run by default (GPT-2: the cluster kernel at one row; Llama: two rows)."""
    if arch == "gpt2":
        run = get_preset("tiny").with_model(quant=P.Q4_0)
        run = dataclasses.replace(run, sampler=SamplerSpec(0.8, 1000, 0.95, False))
        prompt = np.zeros((1, 24), np.int32)
    else:
        spec = P.ModelSpec(arch=P.ARCH_LLAMA, n_layer=3, d_model=512, n_head=8, n_kv_head=2, head_dim=64,
                           d_ff=1536, vocab=1000, max_ctx=300, batch=2, quant=P.Q4_0)
        run = get_preset("llama_q4").with_model(**{f: getattr(spec, f) for f in
                                                   ("n_layer", "d_model", "n_head", "n_kv_head", "d_ff", "vocab",
                                                    "max_ctx", "quant")})
        prompt = np.zeros((2, 40), np.int32)
    B, n = prompt.shape
    emb = (np.random.default_rng(11).standard_normal((B, n, run.model.d_model)) * 0.05).astype(np.float32)
    _check_t3(sd, run, 12, prompt=prompt, prompt_embeds=emb)


def test_prefix_of_embedding_rows_equals_token_prompt(sd):
    """Prompt vectors equal to the tokens' embedding rows decode bit for bit like
    the token prompt (GPT-2: the learned positions are added to both)."""
    run = get_preset("tiny").with_model(quant=P.Q4_0)
    spec = run.model
    blob, fp32 = build_model_blob(spec, keep_fp32=True)
    prompt = prompt_tokens(run)
    draws = uniform_draws(5, 9, 1)[..., 0]
    s = sd.Sampler.from_spec(P.T3_SAMPLED)
    outs = []
    for use_embeds in (False, True):
        dec = sd.Decoder(spec, blob, stream=_stream())
        t = dec.prefill_embeds(fp32["wte"][prompt], s, draws[0]) if use_embeds else dec.prefill(prompt, s, draws[0])
        toks, zs = [int(t[0])], [dec.logits()]
        for i in range(8):
            t = dec.step(np.array([toks[-1]], np.int32), s, draws[i + 1])
            toks.append(int(t[0]))
            zs.append(dec.logits())
        outs.append((toks, zs))
        dec.close()
    assert outs[0][0] == outs[1][0]
    for a, b in zip(outs[0][1], outs[1][1]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_talker_prefix_of_embedding_rows_equals_token_prompt(sd):
    """The Talker's prompt as input vectors equal to the codebook-0 embedding rows
    of a token prompt gives the token prompt's frames bit for bit."""
    spec = P.ModelSpec(arch=P.ARCH_QWEN_TTS, n_layer=2, d_model=512, n_head=4, n_kv_head=2, head_dim=128,
                       d_ff=1024, vocab=300, max_ctx=64, batch=2, quant=P.A8G64,
                       cp_layer=2, cp_d_model=256, cp_n_head=4, cp_n_kv_head=4, cp_head_dim=64,
                       cp_d_ff=512, cp_vocab=128, n_codebooks=16, cp_max_ctx=16)
    blob, fp32 = build_model_blob(spec, keep_fp32=True)
    prompt = np.random.default_rng(14).integers(0, 300, size=(2, 10)).astype(np.int32)
    draws = uniform_draws(6, 3, 2, 16)
    s = sd.Sampler.from_spec(P.QWEN_SAMPLED)
    outs = []
    for use_embeds in (False, True):
        dec = sd.Decoder(spec, blob, stream=_stream())
        c = dec.prefill_embeds(fp32["emb.0"][prompt], s, draws[0]) if use_embeds else dec.prefill(prompt, s, draws[0])
        res = [(np.array(c), dec.logits())]
        for f in range(2):
            c = dec.frame(np.asarray(c, np.int32), s, s, draws[f + 1])
            res.append((np.array(c), dec.logits()))
        outs.append(res)
        dec.close()
    for (ca, za), (cb, zb) in zip(*outs):
        assert np.array_equal(ca, cb)
        assert np.array_equal(za.view(np.uint32), zb.view(np.uint32))


def _prefill_both_ways(sd, spec, prompt1, u, sampler, steps_fn):
    """(codes or tokens, logits, later-step logits) after sd_prefill with the prompt
    replicated to every row and after sd_prefill_shared with it once."""
    blob = _blob(spec)
    res = []
    for shared in (False, True):
        dec = sd.Decoder(spec, blob, stream=_stream())
        if shared:
            t = dec.prefill_shared(prompt1, sampler, u)
        else:
            t = dec.prefill(np.repeat(prompt1[None, :], spec.batch, axis=0), sampler, u)
        res.append((np.array(t), dec.logits(), steps_fn(dec, t)))
        dec.close()
    return res


def test_shared_prompt_equals_replicated_prompt_t3(sd, prefill_path):
    """sd_prefill_shared (row 0's prompt KV computed once and copied) gives the
    replicated prompt's tokens and logits bit for bit, then and after steps."""
    spec = P.ModelSpec(arch=P.ARCH_LLAMA, n_layer=3, d_model=512, n_head=8, n_kv_head=2, head_dim=64,
                       d_ff=1536, vocab=1000, max_ctx=300, batch=2, quant=P.Q4_0)
    prompt1 = np.random.default_rng(12).integers(0, 1000, size=40).astype(np.int32)
    draws = uniform_draws(6, 7, 2)[..., 0]
    s = sd.Sampler.from_spec(P.T3_SAMPLED)

    def steps(dec, t):
        zs = []
        for i in range(6):
            t = dec.step(np.asarray(t, np.int32), s, draws[i + 1])
            zs.append(dec.logits())
        return zs

    (ta, za, sa), (tb, zb, sb) = _prefill_both_ways(sd, spec, prompt1, draws[0], s, steps)
    assert np.array_equal(ta, tb)
    assert np.array_equal(za.view(np.uint32), zb.view(np.uint32))
    for a, b in zip(sa, sb):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_shared_prompt_g16_rollouts(sd):
    """Sixteen rollouts of one prompt (Talker + code predictor, G = 16): the shared
    prefill equals the replicated one bit for bit and matches the oracle."""
    spec = P.ModelSpec(arch=P.ARCH_QWEN_TTS, n_layer=2, d_model=512, n_head=4, n_kv_head=2, head_dim=128,
                       d_ff=1024, vocab=300, max_ctx=64, batch=16, quant=P.A8G64,
                       cp_layer=2, cp_d_model=256, cp_n_head=4, cp_n_kv_head=4, cp_head_dim=64,
                       cp_d_ff=512, cp_vocab=128, n_codebooks=16, cp_max_ctx=16)
    prompt1 = np.random.default_rng(13).integers(0, 300, size=20).astype(np.int32)
    draws = uniform_draws(3, 3, 16, 16)
    s = sd.Sampler.from_spec(P.QWEN_SAMPLED)

    def frames(dec, codes):
        zs = []
        for f in range(2):
            codes = dec.frame(np.asarray(codes, np.int32), s, s, draws[f + 1])
            zs.append(dec.logits())
        return zs

    (ta, za, fa), (tb, zb, fb) = _prefill_both_ways(sd, spec, prompt1, draws[0], s, frames)
    assert np.array_equal(ta, tb)
    assert np.array_equal(za.view(np.uint32), zb.view(np.uint32))
    for a, b in zip(fa, fb):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # and the shared prompt's first frame against the oracle (rows started from one prompt state)
    ref = oracle.run_qwen(oracle.Model(_blob(spec), THREADS), spec, np.repeat(prompt1[None, :], 16, axis=0),
                          draws, 0, P.QWEN_SAMPLED, P.QWEN_SAMPLED)
    for b in range(16):
        assert _rel(zb[b, 0, :spec.vocab], ref[b].logits[0][0]) <= REL_L2


def test_gpt2m_q8_greedy(sd):
    """GPT-2-Medium Q8_0 at its configured length: 150-token prompt, 250 greedy steps."""
    run = get_preset("gpt2m_q8")
    _check_t3(sd, run, run.n_steps)


def test_gpt2m_q4_sampled(sd):
    _check_t3(sd, get_preset("gpt2m_q4"), 6)


def test_llama_q4_two_rows(sd):
    """Llama-style T3 Q4_0 at its configured length: two 200-token prompt rows,
    400 sampled steps on both."""
    run = get_preset("llama_q4")
    _check_t3(sd, run, run.n_steps)


def test_llama_gqa_small(sd):
    spec = P.ModelSpec(arch=P.ARCH_LLAMA, n_layer=3, d_model=512, n_head=8, n_kv_head=2, head_dim=64,
                       d_ff=1536, vocab=1000, max_ctx=300, batch=2, quant=P.Q8_0)
    run = get_preset("llama_q4").with_model(**{f: getattr(spec, f) for f in
                                               ("n_layer", "d_model", "n_head", "n_kv_head", "d_ff", "vocab",
                                                "max_ctx", "quant")})
    prompt = np.random.default_rng(1).integers(0, 1000, size=(2, 40)).astype(np.int32)
    _check_t3(sd, run, 30, prompt=prompt)


def test_bench_configuration_gpt2m_q4(sd):
    """The benchmark's configuration: GPT-2-Medium Q4_0, a 150-token prompt, then
    250 sampled steps with device-side feedback (sd_decode_n, draws resident on
    the device).  The oracle replays the GPU's token stream.  The same steps as a
    chain of sd_step calls give every step's logits: the chain's tokens and final
    logits equal decode_n's bit for bit, and every step's logits are compared with
    the oracle's."""
    run = get_preset("gpt2m_q4")
    spec = run.model
    blob = _blob(spec)
    prompt = prompt_tokens(run)
    n = run.n_steps
    draws = uniform_draws(run.draw_seed, n + 1, 1)[..., 0]
    dec = sd.Decoder(spec, blob, stream=_stream())
    s = sd.Sampler.from_spec(run.sampler)
    first = dec.prefill(prompt, s, draws[0])
    u_dev = torch.from_numpy(np.ascontiguousarray(draws[1:])).cuda()
    out_dev = torch.zeros(n, 1, dtype=torch.int32, device="cuda")
    dec.decode_n(n, s, u_dev, out_dev)
    toks = [int(first[0])] + [int(t) for t in out_dev.cpu().numpy()[:, 0]]
    z_last = dec.logits()[0]
    dec.reset()
    t = dec.prefill(prompt, s, draws[0])
    assert int(t[0]) == toks[0]
    zs = [dec.logits()[0]]
    for i in range(n):
        t = dec.step(np.array([toks[i]], np.int32), s, draws[i + 1])
        assert int(t[0]) == toks[i + 1], i
        zs.append(dec.logits()[0])
    assert np.array_equal(zs[-1].view(np.uint32), z_last.view(np.uint32))
    dec.close()
    ref = oracle.run_t3(oracle.Model(blob, THREADS), spec, prompt, draws, n, run.sampler, forced=[toks[:n]])[0]
    name = f"bench config gpt2m_q4 steps {n + 1}"
    tally = _Tally(name, run.sampler)
    worst = 0.0
    for i in range(n + 1):
        r = _rel(zs[i], ref.logits[i])
        worst = max(worst, r)
        assert r <= REL_L2, (i, r)
        tally.add((i, 0), toks[i], ref.tokens[i], ref.margins[i], zs[i], ref.logits[i])
    print(f"[{name}] worst logits rel L2 {worst:.2e}")
    tally.check()


def _ladder_input(zc, zu, lad, seen):
    """The ladder's input to its temperature stage, in float64: the guided
    combination of the two rows, then the repetition penalty on the history (a
    measure of how far the two sides' inputs to the sampling stages differ)."""
    zc, zu = np.asarray(zc, np.float64), np.asarray(zu, np.float64)
    z = zc + lad.cfg_weight * (zc - zu)
    pen = seen.astype(bool)
    z[pen] = np.where(z[pen] > 0, z[pen] / lad.rep_penalty, z[pen] * lad.rep_penalty)
    return z


def _check_cfg(sd, spec, prompt, n_steps, lad, name, draw_seed=3):
    """The multilingual T3 with guidance through sd_set_ladder: row 0 conditional,
    row 1 unconditional, one token per step fed to both rows, teacher-forced with
    the oracle's tokens.  Per step: both rows' logits within REL_L2 of the
    oracle's; the device ladder picks what the oracle's ladder picks on the
    device's own logits (same history, margin >= SAMPLER_MARGIN); the token
    against the oracle's under _Tally's rules, d being the largest difference
    between the two sides' inputs to the ladder's temperature stage (guided
    combination, then repetition penalty)."""
    blob = _blob(spec)
    draws = uniform_draws(draw_seed, n_steps + 1, 2)[..., 0]
    ref = oracle.run_t3_cfg(oracle.Model(blob, THREADS), spec, prompt, draws[:, 0], n_steps, lad)
    dec = sd.Decoder(spec, blob, stream=_stream())
    dec.set_ladder(sd.SamplerLadder.from_spec(lad))
    s = sd.Sampler.from_spec(P.T3_SAMPLED)     # per-row sampler: not used while the ladder is set
    got = dec.prefill(prompt, s, draws[0])
    as_sampler = SamplerSpec(temperature=lad.temperature, top_k=lad.top_k, top_p=lad.top_p,
                             greedy=lad.temperature <= 0)
    tally = _Tally(name, as_sampler)
    seen = np.zeros(spec.vocab, np.uint8)
    worst = 0.0
    for i in range(n_steps + 1):
        z = dec.logits()
        assert int(got[0]) == int(got[1]), (i, got)
        for b in range(2):
            r = _rel(z[b], ref.logits[i][b])
            worst = max(worst, r)
            assert r <= REL_L2, (i, b, r)
        tg, mg = oracle.sample_ladder(z[0], z[1], lad.cfg_weight, seen, lad.rep_penalty, lad.temperature,
                                      lad.min_p, lad.top_p, lad.top_k, u=float(draws[i][0]))
        if mg >= SAMPLER_MARGIN:
            assert int(got[0]) == tg, ("ladder", i, int(got[0]), tg, mg)
        d = _logit_error(_ladder_input(z[0], z[1], lad, seen), _ladder_input(*ref.logits[i], lad, seen))
        tally.add(i, int(got[0]), ref.tokens[i], ref.margins[i], None, None, d=d)
        if i < n_steps:
            t = ref.tokens[i]
            seen[t] = 1
            got = dec.step(np.array([t, t], np.int32), s, draws[i + 1])
    dec.close()
    print(f"[{name}] worst logits rel L2 {worst:.2e}")
    tally.check()


def test_cfg_ladder_small_llama(sd):
    spec = P.ModelSpec(arch=P.ARCH_LLAMA, n_layer=3, d_model=512, n_head=8, n_kv_head=2, head_dim=64,
                       d_ff=1536, vocab=1000, max_ctx=300, batch=2, quant=P.Q4_0)
    prompt = np.random.default_rng(4).integers(0, 1000, size=(2, 40)).astype(np.int32)
    _check_cfg(sd, spec, prompt, 80, P.MTL_LADDER, "cfg ladder llama-small q4")
    greedy = dataclasses.replace(P.MTL_LADDER, temperature=0.0, top_k=1)
    _check_cfg(sd, spec, prompt, 40, greedy, "cfg ladder llama-small q4 greedy")


def test_cfg_ladder_llama_q4(sd):
    """The multilingual T3's shape (Llama-style, Q4_0, two rows: conditional and
    unconditional, 200-token prompts) with the ladder, 100 steps."""
    run = get_preset("llama_q4")
    _check_cfg(sd, run.model, prompt_tokens(run), 100, P.MTL_LADDER, "cfg ladder llama_q4")


def test_cfg_ladder_decode_n_equals_step_chain(sd):
    """decode_n with the ladder (device-side feedback and history) gives the
    step chain's tokens and final logits bit for bit."""
    spec = P.ModelSpec(arch=P.ARCH_LLAMA, n_layer=2, d_model=512, n_head=8, n_kv_head=2, head_dim=64,
                       d_ff=1536, vocab=1000, max_ctx=300, batch=2, quant=P.Q8_0)
    blob = _blob(spec)
    prompt = np.random.default_rng(6).integers(0, 1000, size=(2, 24)).astype(np.int32)
    n = 30
    draws = uniform_draws(8, n + 1, 2)[..., 0]
    s = sd.Sampler.from_spec(P.T3_SAMPLED)
    a = sd.Decoder(spec, blob, stream=_stream())
    a.set_ladder(sd.SamplerLadder.from_spec(P.MTL_LADDER))
    t = a.prefill(prompt, s, draws[0])
    chain = [int(t[0])]
    for i in range(n):
        t = a.step(np.array([chain[-1]] * 2, np.int32), s, draws[i + 1])
        assert int(t[0]) == int(t[1])
        chain.append(int(t[0]))
    za = a.logits()
    a.reset()
    t = a.prefill(prompt, s, draws[0])
    assert int(t[0]) == chain[0]
    out = torch.zeros(n, 2, dtype=torch.int32, device="cuda")
    a.decode_n(n, s, torch.from_numpy(np.ascontiguousarray(draws[1:])).cuda(), out)
    o = out.cpu().numpy()
    assert [int(x) for x in o[:, 0]] == chain[1:]
    assert np.array_equal(o[:, 0], o[:, 1])
    assert np.array_equal(a.logits().view(np.uint32), za.view(np.uint32))
    # the ladder off again: the per-row sampler, rows independent
    a.reset()
    a.set_ladder(None)
    t = a.prefill(prompt, s, draws[0])
    z = a.logits()
    for b in range(2):
        tg, mg = oracle.sample(z[b], u=float(draws[0][b]), temperature=0.8, top_k=1000, top_p=0.95, greedy=False)
        if mg >= SAMPLER_MARGIN:
            assert int(t[b]) == tg, (b, int(t[b]), tg, mg)
    a.close()


def test_set_ladder_rejects(sd):
    spec = P.ModelSpec(arch=P.ARCH_LLAMA, n_layer=1, d_model=256, n_head=4, n_kv_head=4, head_dim=64,
                       d_ff=512, vocab=300, max_ctx=40, batch=1, quant=P.Q8_0)
    dec = sd.Decoder(spec, _blob(spec), stream=_stream())
    with pytest.raises(sd.SdError):
        dec.set_ladder(sd.SamplerLadder.from_spec(P.MTL_LADDER))     # one row
    dec.close()
    spec2 = dataclasses.replace(spec, batch=2)
    dec = sd.Decoder(spec2, _blob(spec2), stream=_stream())
    for bad in (dict(rep_penalty=0.0), dict(top_p=0.0), dict(top_p=1.5), dict(min_p=-0.1)):
        with pytest.raises(sd.SdError):
            dec.set_ladder(sd.SamplerLadder.from_spec(dataclasses.replace(P.MTL_LADDER, **bad)))
    s = sd.Sampler.from_spec(P.T3_SAMPLED)
    dec.prefill(np.zeros((2, 4), np.int32), s, np.zeros(2, np.float32))
    with pytest.raises(sd.SdError):
        dec.set_ladder(sd.SamplerLadder.from_spec(P.MTL_LADDER))     # not reset
    dec.close()


@pytest.fixture(params=["graph", "flat", "cluster"])
def step_path(request, monkeypatch):
    """Run a test on the per-operation graph, the flat persistent step kernel and
    the cluster persistent step kernel."""
    monkeypatch.setenv("SD_PERSISTENT", {"graph": "0", "flat": "flat", "cluster": "cluster"}[request.param])
    return request.param


def test_gpt2m_q4_both_step_paths(sd, step_path):
    _check_t3(sd, get_preset("gpt2m_q4"), 4)


def test_llama_q4_both_step_paths(sd, step_path):
    _check_t3(sd, get_preset("llama_q4"), 4)


@pytest.fixture(params=["tcgen05", "mma", "steps"])
def prefill_path(request, monkeypatch):
    """Run a test with the tcgen05 GEMM prefill, the mma.sync GEMM prefill and
    the per-position step graphs."""
    monkeypatch.setenv("SD_PREFILL", request.param)
    return request.param


@pytest.mark.parametrize("name,want", [("gpt2m_q4", 2), ("llama_q4", 2), ("qwen_a8", 2), ("tiny", 2)])
def test_prefill_uses_tensor_cores(sd, monkeypatch, name, want):
    monkeypatch.delenv("SD_PREFILL", raising=False)
    run = get_preset(name)
    dec = sd.Decoder(run.model, _blob(run.model), stream=_stream())
    assert dec.info().prefill == want
    dec.close()


def test_gpt2m_q4_both_prefill_paths(sd, prefill_path):
    _check_t3(sd, get_preset("gpt2m_q4"), 3)


def test_llama_gqa_prompt_spanning_chunks(sd, prefill_path):
    """Two batch rows, 8 query / 2 KV heads, a 290-token prompt: the GEMM
    prefill runs it as two chunks (256 positions, then 33)."""
    spec = P.ModelSpec(arch=P.ARCH_LLAMA, n_layer=2, d_model=512, n_head=8, n_kv_head=2, head_dim=64,
                       d_ff=1536, vocab=1000, max_ctx=300, batch=2, quant=P.Q4_0)
    run = get_preset("llama_q4").with_model(**{f: getattr(spec, f) for f in
                                               ("n_layer", "d_model", "n_head", "n_kv_head", "d_ff", "vocab",
                                                "max_ctx", "quant")})
    prompt = np.random.default_rng(5).integers(0, 1000, size=(2, 290)).astype(np.int32)
    _check_t3(sd, run, 6, prompt=prompt)


def test_one_token_prompt(sd, prefill_path):
    run = get_preset("tiny")
    _check_t3(sd, run, 3, prompt=np.array([[17]], np.int32))


@pytest.mark.parametrize("name", ["tiny", "gpt2m_q4", "gpt2m_q8", "llama_q4"])
@pytest.mark.parametrize("kind", ["flat", "cluster"])
def test_persistent_kernel_is_used(sd, monkeypatch, name, kind):
    """Both persistent step kernels' plans accept every GPT-2 / Llama workload
    (so the persistent-path tests above do run the kernel they name)."""
    monkeypatch.setenv("SD_PERSISTENT", kind)
    run = get_preset(name)
    dec = sd.Decoder(run.model, _blob(run.model), stream=_stream())
    info = dec.info()
    assert info.persistent > 0 and info.kernels_per_step == 1
    if kind == "cluster":
        assert info.persistent_clusters > 0 and info.cluster_size > 1
        assert info.persistent == info.persistent_clusters * info.cluster_size
        print(f"[{name}] cluster step: {info.persistent_clusters} clusters x {info.cluster_size} CTAs")
    else:
        assert info.persistent_clusters == 0
    dec.close()


@pytest.mark.parametrize("name", ["gpt2m_q4", "llama_q4"])
def test_default_step_path_is_the_cluster_step(sd, monkeypatch, name):
    """One row (GPT-2-Medium) and two rows (Llama) decode on the cluster step by default."""
    monkeypatch.delenv("SD_PERSISTENT", raising=False)
    run = get_preset(name)
    dec = sd.Decoder(run.model, _blob(run.model), stream=_stream())
    assert dec.info().persistent_clusters > 0
    dec.close()


def test_decode_n_equals_step_chain_bitwise(sd, step_path):
    run = get_preset("tiny").with_model(quant=P.Q4_0)
    spec = run.model
    blob = _blob(spec)
    prompt = prompt_tokens(run)
    n = 20
    draws = uniform_draws(7, n + 1, 1)[..., 0]
    s = sd.Sampler(0.8, 1000, 0.95, 0)
    a = sd.Decoder(spec, blob, stream=_stream())
    t = a.prefill(prompt, s, draws[0])
    chain = [int(t[0])]
    for i in range(n):
        t = a.step(np.array([chain[-1]], np.int32), s, draws[i + 1])
        chain.append(int(t[0]))
    za = a.logits()
    a.reset()
    t = a.prefill(prompt, s, draws[0])
    assert int(t[0]) == chain[0]
    out = torch.zeros(n, 1, dtype=torch.int32, device="cuda")
    a.decode_n(n, s, torch.from_numpy(np.ascontiguousarray(draws[1:])).cuda(), out)
    assert [int(x) for x in out.cpu().numpy()[:, 0]] == chain[1:]
    assert np.array_equal(a.logits().view(np.uint32), za.view(np.uint32))
    a.close()


def test_errors_and_context_limit(sd):
    spec = P.ModelSpec(arch=P.ARCH_GPT2, n_layer=1, d_model=256, n_head=4, n_kv_head=4, head_dim=64,
                       d_ff=512, vocab=300, max_ctx=40, batch=1, quant=P.Q8_0)
    blob = _blob(spec)
    dec = sd.Decoder(spec, blob, stream=_stream())
    s = sd.Sampler(1.0, 1, 1.0, 1)
    u = np.zeros(1, np.float32)
    with pytest.raises(sd.SdError) as e:
        dec.step(np.array([1], np.int32), s, u)
    assert e.value.code == -2                                        # SD_ERR_STATE
    with pytest.raises(sd.SdError) as e:
        dec.prefill(np.array([[1, 300]], np.int32), s, u)
    assert e.value.code == -1                                        # token out of range
    with pytest.raises(sd.SdError) as e:
        dec.prefill(np.array([[1, 2]], np.int32), sd.Sampler(0.5, 0, 0.9, 0), u)
    assert e.value.code == -1                                        # top_k < 1
    with pytest.raises(sd.SdError) as e:
        dec.prefill(np.array([[1, 2]], np.int32), sd.Sampler(0.8, 50, 0.9, 0, 1.3), u)
    assert e.value.code == -7                                        # a repetition penalty: SD_ERR_UNSUPPORTED
    with pytest.raises(sd.SdError) as e:
        dec.prefill(np.array([[1, 2]], np.int32), sd.Sampler(0.8, 50, 0.9, 0, -1.0), u)
    assert e.value.code == -1                                        # a negative penalty
    t = dec.prefill(np.arange(38, dtype=np.int32)[None], s, u)
    first = int(t[0])
    t = dec.step(t, s, u)
    t = dec.step(t, s, u)                                            # position 39: the last slot
    with pytest.raises(sd.SdError) as e:
        dec.step(t, s, u)
    assert e.value.code == -3                                        # SD_ERR_CTX_FULL
    dec.reset()                                                      # recovers after the error
    assert int(dec.prefill(np.arange(38, dtype=np.int32)[None], s, u)[0]) == first
    dec.close()


@pytest.mark.parametrize("kind", ["flat", "cluster"])
def test_expired_exchange_wait_reports_timeout_and_recovers(sd, monkeypatch, kind):
    """A wait on an exchange word that runs out.  A test hook (SD_TEST_STALL_US)
    makes the first directly launched persistent step (sd_decode_n; captured
    graphs never take it) wait in CTA 0, for 1 ms, for an epoch that no CTA
    writes; every other wait keeps its budget, sees the recorded error and ends,
    and each CTA waits for its bulk copies in flight before it returns (no
    mbarrier or copy wait is made to expire).  The call reports SD_ERR_TIMEOUT;
    after sd_reset the same context decodes with oracle-equal logits and tokens."""
    monkeypatch.setenv("SD_PERSISTENT", kind)
    monkeypatch.setenv("SD_TEST_STALL_US", "1000")
    run = get_preset("tiny").with_model(quant=P.Q4_0)
    run = dataclasses.replace(run, sampler=SamplerSpec(0.8, 1000, 0.95, False))
    spec = run.model
    blob = _blob(spec)
    prompt = prompt_tokens(run)
    n = 4
    draws = uniform_draws(run.draw_seed, n + 1, 1)[..., 0]
    s = sd.Sampler.from_spec(run.sampler)
    dec = sd.Decoder(spec, blob, stream=_stream())
    info = dec.info()
    assert info.persistent > 0 and (info.persistent_clusters > 0) == (kind == "cluster")
    dec.prefill(prompt, s, draws[0])
    u_dev = torch.from_numpy(np.ascontiguousarray(draws[1:3])).cuda()
    out_dev = torch.zeros(2, 1, dtype=torch.int32, device="cuda")
    with pytest.raises(sd.SdError) as e:
        dec.decode_n(2, s, u_dev, out_dev)                          # the first direct launch takes the hook
    assert e.value.code == -6, e.value                              # SD_ERR_TIMEOUT
    dec.reset()
    ref = oracle.run_t3(oracle.Model(blob, THREADS), spec, prompt, draws, n, run.sampler)[0]
    got = dec.prefill(prompt, s, draws[0])
    for i in range(n + 1):
        z = dec.logits()[0]
        assert _rel(z, ref.logits[i]) <= REL_L2, i
        if ref.margins[i] >= MARGIN:
            assert int(got[0]) == ref.tokens[i], i
        if i < n:
            got = dec.step(np.array([ref.tokens[i]], np.int32), s, draws[i + 1])
    dec.close()


# ----------------------------------------------------------------------------- Talker + code predictor

def _check_qwen(sd, spec, prompt, n_frames, sampler, name, cp_sampler=None):
    """sampler drives the Talker (and the code predictor unless cp_sampler is
    given); a Talker repetition penalty acts on the codebook-0 tokens fed so far."""
    cp_sampler = cp_sampler or sampler
    blob = _blob(spec)
    B = spec.batch
    draws = uniform_draws(3, n_frames + 1, B, 16)
    ref = oracle.run_qwen(oracle.Model(blob, THREADS), spec, prompt, draws, n_frames, sampler, cp_sampler)
    dec = sd.Decoder(spec, blob, stream=_stream())
    s, scp = sd.Sampler.from_spec(sampler), sd.Sampler.from_spec(cp_sampler)
    pen = float(sampler.rep_penalty)
    sa = [dict(temperature=x.temperature, top_k=x.top_k, top_p=x.top_p, greedy=x.greedy) for x in (sampler, cp_sampler)]
    dec.force(np.array([ref[b].tokens[0] for b in range(B)], np.int32))
    codes = dec.prefill(prompt, s, draws[0])
    name = f"{name} rows {B} frames {n_frames + 1}"
    tally = _Tally(name, sampler)
    worst = 0.0
    seen0 = np.zeros((B, spec.vocab), np.uint8)
    for f in range(n_frames + 1):
        z = dec.logits()
        for b in range(B):
            for j in range(16):
                V = spec.vocab if j == 0 else spec.cp_vocab
                r = _rel(z[b, j, :V], ref[b].logits[f][j])
                worst = max(worst, r)
                assert r <= REL_L2, (f, b, j, r)
                # the device sampler decides like the oracle's sampler on the same (device) logits
                hist = dict(seen=seen0[b], rep_penalty=pen) if j == 0 else {}
                tg, mg = oracle.sample(z[b, j, :V], u=float(draws[f][b][j]), **sa[j > 0], **hist)
                if mg >= SAMPLER_MARGIN:
                    assert int(codes[b, j]) == tg, ("sampler", f, b, j, int(codes[b, j]), tg, mg)
                # a penalty scales a logit by at most its factor
                d = _logit_error(z[b, j, :V], ref[b].logits[f][j]) * (max(pen, 1.0) if j == 0 else 1.0)
                tally.add((f, b, j), int(codes[b, j]), ref[b].tokens[f][j], ref[b].margins[f][j], None, None, d=d)
        if f < n_frames:
            prev = np.array([ref[b].tokens[f] for b in range(B)], np.int32)
            seen0[np.arange(B), prev[:, 0]] = 1
            dec.force(np.array([ref[b].tokens[f + 1] for b in range(B)], np.int32))
            codes = dec.frame(prev, s, scp, draws[f + 1])
    dec.close()
    print(f"[{name}] worst logits rel L2 {worst:.2e}")
    tally.check()
    assert tally.strict > 0


@pytest.mark.parametrize("rows", [1, 16])
def test_qwen_talker_repetition_penalty(sd, rows):
    """The Talker's codebook-0 sampler with a repetition penalty over the codes fed
    so far, kept on the device ("Every Frame Is a Memory Read", section 2 decodes
    with a penalty; section 8 moves it to the device per row), against the oracle."""
    spec = P.ModelSpec(arch=P.ARCH_QWEN_TTS, n_layer=2, d_model=512, n_head=4, n_kv_head=2, head_dim=128,
                       d_ff=1024, vocab=300, max_ctx=64, batch=rows, quant=P.A8G64,
                       cp_layer=2, cp_d_model=256, cp_n_head=4, cp_n_kv_head=4, cp_head_dim=64,
                       cp_d_ff=512, cp_vocab=128, n_codebooks=16, cp_max_ctx=16)
    prompt = np.random.default_rng(7).integers(0, 300, size=(rows, 12)).astype(np.int32)
    talker = SamplerSpec(0.9, 50, 0.95, False, rep_penalty=1.3)
    _check_qwen(sd, spec, prompt, 8, talker, "qwen talker penalty", cp_sampler=P.QWEN_SAMPLED)


def test_qwen_small(sd, prefill_path):
    spec = P.ModelSpec(arch=P.ARCH_QWEN_TTS, n_layer=2, d_model=512, n_head=4, n_kv_head=2, head_dim=128,
                       d_ff=1024, vocab=300, max_ctx=64, batch=2, quant=P.A8G64,
                       cp_layer=2, cp_d_model=256, cp_n_head=4, cp_n_kv_head=4, cp_head_dim=64,
                       cp_d_ff=512, cp_vocab=128, n_codebooks=16, cp_max_ctx=16)
    prompt = np.random.default_rng(3).integers(0, 300, size=(2, 12)).astype(np.int32)
    _check_qwen(sd, spec, prompt, 4, SamplerSpec(0.9, 50, 0.95, False), "qwen small")


@pytest.mark.parametrize("cp_quant", [P.A4G32, P.A4G64])
@pytest.mark.parametrize("rows", [1, 16])
def test_qwen_code_predictor_4bit(sd, cp_quant, rows):
    """The Talker in 8-bit affine and the code predictor in 4-bit affine, group
    32 or 64 ("Every Frame Is a Memory Read", section 5.8), at one row and at
    sixteen rollout rows (matvecs over pairs of rows for the 4-bit matrices)."""
    spec = P.ModelSpec(arch=P.ARCH_QWEN_TTS, n_layer=2, d_model=512, n_head=4, n_kv_head=2, head_dim=128,
                       d_ff=1024, vocab=300, max_ctx=64, batch=rows, quant=P.A8G64,
                       cp_layer=2, cp_d_model=256, cp_n_head=4, cp_n_kv_head=4, cp_head_dim=64,
                       cp_d_ff=512, cp_vocab=128, n_codebooks=16, cp_max_ctx=16, cp_quant=cp_quant)
    prompt = np.random.default_rng(5).integers(0, 300, size=(rows, 12)).astype(np.int32)
    _check_qwen(sd, spec, prompt, 3, SamplerSpec(0.9, 50, 0.95, False),
                f"qwen cp {P.QUANT_NAMES[cp_quant]}")


def test_qwen_full_size(sd):
    """The Talker + code predictor at full size, G = 1: the configured 300-token
    prompt, then 16 frames (17 with the prompt's)."""
    run = get_preset("qwen_a8")
    _check_qwen(sd, run.model, prompt_tokens(run), 16, run.sampler, "qwen_a8")


@pytest.fixture(params=["skinny", "tc"])
def rows_gemm(request, monkeypatch):
    """The 3-16 row GEMM: mma.sync skinny (default) or tcgen05 (SD_ROWS_GEMM=tc)."""
    if request.param == "tc":
        monkeypatch.setenv("SD_ROWS_GEMM", "tc")
    else:
        monkeypatch.delenv("SD_ROWS_GEMM", raising=False)
    return request.param


def test_qwen_g16_small(sd, prefill_path, rows_gemm):
    """Sixteen rollout rows (the G=16 configuration's batch) through the
    norm-kernel + tensor-core GEMM path that replaces the 1-2 row GEMV."""
    spec = P.ModelSpec(arch=P.ARCH_QWEN_TTS, n_layer=2, d_model=512, n_head=4, n_kv_head=2, head_dim=128,
                       d_ff=1024, vocab=300, max_ctx=64, batch=16, quant=P.A8G64,
                       cp_layer=2, cp_d_model=256, cp_n_head=4, cp_n_kv_head=4, cp_head_dim=64,
                       cp_d_ff=512, cp_vocab=128, n_codebooks=16, cp_max_ctx=16)
    prompt = np.random.default_rng(4).integers(0, 300, size=(16, 12)).astype(np.int32)
    _check_qwen(sd, spec, prompt, 3, SamplerSpec(0.9, 50, 0.95, False), "qwen g16 small")


def test_qwen_g16_full_size(sd):
    """The G = 16 configuration at full size: 16 rollouts of one 64-token prompt
    (the configured prompt's first 64 tokens), then 4 frames after the prompt's."""
    run = get_preset("qwen_a8_g16")
    prompt = np.repeat(prompt_tokens(run)[:1, :64], 16, axis=0)
    _check_qwen(sd, run.model, prompt, 4, run.sampler, "qwen_a8_g16")


def test_gpt2_four_rows(sd):
    """Rows beyond two on the GPT-2 path (norm kernel + GEMM per matrix)."""
    run = get_preset("tiny").with_model(batch=4)
    prompt = np.random.default_rng(8).integers(0, 6561, size=(4, 20)).astype(np.int32)
    _check_t3(sd, run, 10, prompt=prompt)

