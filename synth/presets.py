"""Workload shapes for the speech-token decode step.

The five workloads are the ones the decode method is measured on:

* ``tiny``      — 2-layer GPT-2-style decoder (d=256) with Q8_0 weights; a
                  32-token prompt then 64 greedy steps.
* ``gpt2m_q8``  — GPT-2-Medium-shaped T3 (24 layers, d=1024, 16x64 heads,
                  GELU FFN 4096, learned positions, 6561 speech + 2 special
                  tokens), Q8_0 weights; 150-token prompt, 250 greedy steps.
                  T3 is described as a 24-layer GPT-2-Medium decoder in
                  "Chatterbox -> ggml Port: Development Journal", section 3.2.
* ``gpt2m_q4``  — the same shape with Q4_0 weights, sampled with
                  temperature 0.8, top-k 1000, top-p 0.95 (the T3 defaults of
                  the journal's section 3.9 table).
* ``llama_q4``  — Llama-style T3 (30 layers, RMSNorm, NEOX RoPE theta=1e4,
                  SwiGLU 4096, vocab 8194), Q4_0, batch 2 (two independent
                  rows decoded together, the journal's section 3.21 B=2 step).
* ``qwen_a8``   — Qwen3-style Talker (28 layers, d=2048, 16 q / 8 kv heads of
                  128, SwiGLU 6144, codebook-0 vocab 3072) plus a 5-layer code
                  predictor (d=1024, 16x64, FFN 3072, 15 heads of 2048) run as
                  15 sequential passes per frame ("Every Frame Is a Memory
                  Read", section 1), with 8-bit affine group-64 weights.

Where the pages leave a size open, the plainest reading is taken (cache
capacities, prompt-ID ranges); each such reading is listed in the design notes.
"""

from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field

# architecture ids (mirrored numerically by the C headers of both readers)
ARCH_GPT2 = 1
ARCH_LLAMA = 2
ARCH_QWEN_TTS = 3

# quantisation ids
Q8_0 = 1
Q4_0 = 2
A8G64 = 3
Q5_0 = 4
A4G32 = 5
A4G64 = 6

QUANT_NAMES = {Q8_0: "q8_0", Q4_0: "q4_0", A8G64: "a8g64", Q5_0: "q5_0", A4G32: "a4g32", A4G64: "a4g64"}
# bytes per weight of each stored format: Q8_0 = 34 B / 32, Q4_0 = 18 B / 32,
# Q5_0 = 22 B / 32, affine group 64 = (64 + 2 + 2) B / 64 -> 8.5 bits per weight,
# 4-bit affine = (16 + 4) B / 32 at group 32 and (32 + 4) B / 64 at group 64.
BYTES_PER_WEIGHT = {Q8_0: 34 / 32, Q4_0: 18 / 32, A8G64: 68 / 64, Q5_0: 22 / 32, A4G32: 20 / 32, A4G64: 36 / 64}


@dataclass(frozen=True)
class ModelSpec:
    arch: int
    n_layer: int
    d_model: int
    n_head: int
    n_kv_head: int
    head_dim: int
    d_ff: int
    vocab: int
    max_ctx: int
    batch: int
    quant: int
    rope_theta: float = 10000.0
    norm_eps: float = 1e-5
    # code predictor (ARCH_QWEN_TTS only)
    cp_layer: int = 0
    cp_d_model: int = 0
    cp_n_head: int = 0
    cp_n_kv_head: int = 0
    cp_head_dim: int = 0
    cp_d_ff: int = 0
    cp_vocab: int = 0
    n_codebooks: int = 0
    cp_max_ctx: int = 0
    # code predictor's weight format (0: the model's); the blob records each tensor's own format
    cp_quant: int = 0

    @property
    def q_dim(self) -> int:
        return self.n_head * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_head * self.head_dim

    @property
    def qkv_rows(self) -> int:
        return self.q_dim + 2 * self.kv_dim

    def quantised_params_per_step(self) -> int:
        """Quantised weights one decode step (or one frame) streams."""
        if self.arch == ARCH_GPT2:
            d, f = self.d_model, self.d_ff
            per_layer = self.qkv_rows * d + d * self.q_dim + f * d + d * f
            return self.n_layer * per_layer + self.vocab * d
        if self.arch == ARCH_LLAMA:
            d, f = self.d_model, self.d_ff
            per_layer = self.qkv_rows * d + d * self.q_dim + 2 * f * d + d * f
            return self.n_layer * per_layer + self.vocab * d
        # Talker step + 15 code-predictor passes + 15 reads of the projection Pr
        # (the first pass projects its two inputs with one read of Pr).
        n_pass = self.n_codebooks - 1
        return self.talker_params() + n_pass * self.cp_pass_params() \
            + n_pass * self.cp_d_model * self.d_model

    def talker_params(self) -> int:
        d, f = self.d_model, self.d_ff
        per_layer = self.qkv_rows * d + d * self.q_dim + 3 * f * d
        return self.n_layer * per_layer + self.vocab * d

    def cp_pass_params(self) -> int:
        d, f = self.cp_d_model, self.cp_d_ff
        qkv = (self.cp_n_head + 2 * self.cp_n_kv_head) * self.cp_head_dim
        per_layer = qkv * d + d * self.cp_n_head * self.cp_head_dim + 3 * f * d
        return self.cp_layer * per_layer + self.cp_vocab * d

    def kv_bytes_per_position(self) -> int:
        """fp16 K and V bytes written (and later read) per cached position, one row."""
        return 2 * self.n_layer * self.kv_dim * 2


@dataclass(frozen=True)
class SamplerSpec:
    temperature: float = 1.0
    top_k: int = 1
    top_p: float = 1.0
    greedy: bool = True
    rep_penalty: float = 1.0   # the Talker's penalty over its past codebook-0 tokens (1: none)


GREEDY = SamplerSpec()
T3_SAMPLED = SamplerSpec(temperature=0.8, top_k=1000, top_p=0.95, greedy=False)
# "Every Frame Is a Memory Read" section 2 decodes with T 0.9 / top-p 0.95 /
# top-k 50 (its repetition penalty is not part of this path).
QWEN_SAMPLED = SamplerSpec(temperature=0.9, top_k=50, top_p=0.95, greedy=False)


@dataclass(frozen=True)
class LadderSpec:
    """The multilingual T3's sampler ladder settings (CFG combine, repetition
    penalty, temperature, min_p, top-p, top-k)."""
    cfg_weight: float = 0.5
    rep_penalty: float = 2.0
    temperature: float = 0.8
    min_p: float = 0.05
    top_p: float = 1.0
    top_k: int = 1000


# The multilingual variant's sampling path names the stages but prints no
# values: a representative setting (guidance 0.5, penalty 2, T 0.8, min_p 0.05,
# top-p off, top-k 1000).
MTL_LADDER = LadderSpec()


@dataclass(frozen=True)
class RunSpec:
    name: str
    model: ModelSpec
    prompt_len: int
    n_steps: int            # decode steps (frames for the Talker+CP model)
    sampler: SamplerSpec
    prompt_vocab: int       # prompt token IDs are uniform in [0, prompt_vocab)
    weight_seed: int = 1
    prompt_seed: int = 2
    draw_seed: int = 3
    extra: dict = field(default_factory=dict)

    def with_model(self, **kw) -> "RunSpec":
        return dataclasses.replace(self, model=dataclasses.replace(self.model, **kw))


_TINY = ModelSpec(arch=ARCH_GPT2, n_layer=2, d_model=256, n_head=4, n_kv_head=4, head_dim=64,
                  d_ff=1024, vocab=6561, max_ctx=512, batch=1, quant=Q8_0)
_GPT2M = ModelSpec(arch=ARCH_GPT2, n_layer=24, d_model=1024, n_head=16, n_kv_head=16, head_dim=64,
                   d_ff=4096, vocab=6563, max_ctx=2048, batch=1, quant=Q8_0)
_LLAMA = ModelSpec(arch=ARCH_LLAMA, n_layer=30, d_model=1024, n_head=16, n_kv_head=16, head_dim=64,
                   d_ff=4096, vocab=8194, max_ctx=1024, batch=2, quant=Q4_0)
_QWEN = ModelSpec(arch=ARCH_QWEN_TTS, n_layer=28, d_model=2048, n_head=16, n_kv_head=8, head_dim=128,
                  d_ff=6144, vocab=3072, max_ctx=512, batch=1, quant=A8G64,
                  cp_layer=5, cp_d_model=1024, cp_n_head=16, cp_n_kv_head=16, cp_head_dim=64,
                  cp_d_ff=3072, cp_vocab=2048, n_codebooks=16, cp_max_ctx=16)

PRESETS: dict[str, RunSpec] = {
    "tiny": RunSpec("tiny", _TINY, prompt_len=32, n_steps=64, sampler=GREEDY, prompt_vocab=6561),
    "gpt2m_q8": RunSpec("gpt2m_q8", _GPT2M, prompt_len=150, n_steps=250, sampler=GREEDY,
                        prompt_vocab=6561),
    "gpt2m_q4": RunSpec("gpt2m_q4", dataclasses.replace(_GPT2M, quant=Q4_0), prompt_len=150,
                        n_steps=250, sampler=T3_SAMPLED, prompt_vocab=6561),
    "llama_q4": RunSpec("llama_q4", _LLAMA, prompt_len=200, n_steps=400, sampler=T3_SAMPLED,
                        prompt_vocab=8192),
    "qwen_a8": RunSpec("qwen_a8", _QWEN, prompt_len=300, n_steps=125, sampler=QWEN_SAMPLED,
                       prompt_vocab=3072),
    "qwen_a8_g16": RunSpec("qwen_a8_g16", dataclasses.replace(_QWEN, batch=16), prompt_len=300,
                           n_steps=125, sampler=QWEN_SAMPLED, prompt_vocab=3072,
                           extra={"shared_prompt": True}),
    # the other weight formats on the same shapes (journal A3: Q5_0 T3; the blog's section 5.8:
    # the code predictor in 4-bit affine, group 64, beside an 8-bit Talker)
    "gpt2m_q5": RunSpec("gpt2m_q5", dataclasses.replace(_GPT2M, quant=Q5_0), prompt_len=150,
                        n_steps=250, sampler=T3_SAMPLED, prompt_vocab=6561),
    "qwen_a8_cp4": RunSpec("qwen_a8_cp4", dataclasses.replace(_QWEN, cp_quant=A4G64), prompt_len=300,
                           n_steps=125, sampler=QWEN_SAMPLED, prompt_vocab=3072),
}


def get_preset(name: str) -> RunSpec:
    try:
        return PRESETS[name]
    except KeyError as e:
        raise KeyError(f"unknown preset {name!r}; known: {sorted(PRESETS)}") from e
