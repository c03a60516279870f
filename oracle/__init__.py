"""Oracle of the speech-token decode step -- TEST INFRASTRUCTURE ONLY.

A ctypes front end to ``sd_oracle.c`` (plain C, double-precision sums), plus
drivers that run a whole workload the way the method describes it: a prompt
processed position by position, then decode steps that each sample a token
(or, for the Talker + code predictor, frames of 16 codes).  The drivers record
every step's logits, sampled token and decision margin so that the CUDA
library can be checked against them with teacher forcing.

Only ``tests/``, the smoke entry and the benchmark's CPU-baseline leg import
this package.  It shares no code with the CUDA library.
"""

from __future__ import annotations

import contextlib
import ctypes as C
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

ARCH_GPT2, ARCH_LLAMA, ARCH_QWEN_TTS = 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "sd_oracle.h"))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_mutant(n: int) -> str:
    """The oracle compiled with planted mistake n (ORC_MUTANT, listed in
    sd_oracle.c) into oracle/_build/liboracle_m<n>.so, for the tests that check
    that the pins reject each mistake."""
    path = os.path.join(_HERE, "_build", f"liboracle_m{n}.so")
    os.makedirs(os.path.dirname(path), exist_ok=True)
    if os.path.exists(path) and os.path.getmtime(path) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "sd_oracle.h"))):
        return path
    tmp = path + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall", "-Wextra", f"-DORC_MUTANT={int(n)}",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


@contextlib.contextmanager
def using_library(path: str):
    """Route every oracle call to the library at `path` (a planted-mistake
    build) inside the block."""
    global _lib
    prev = lib()
    L = C.CDLL(path)
    _declare(L)
    _lib = L
    try:
        yield
    finally:
        _lib = prev


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _declare(_lib)
    return _lib


def _declare(L):
    f32p, i32p, u8p, u16p = (C.POINTER(C.c_float), C.POINTER(C.c_int32), C.POINTER(C.c_uint8),
                             C.POINTER(C.c_uint16))
    L.orc_half_to_float.argtypes = [C.c_uint16]; L.orc_half_to_float.restype = C.c_float
    L.orc_float_to_half.argtypes = [C.c_float]; L.orc_float_to_half.restype = C.c_uint16
    L.orc_dequant.argtypes = [C.c_int, u8p, C.c_int64, C.c_int64, f32p]
    L.orc_linear.argtypes = [C.c_int, u8p, C.c_int64, C.c_int64, f32p, f32p, f32p]
    L.orc_layernorm.argtypes = [f32p, C.c_int, f32p, f32p, C.c_float, f32p]; L.orc_layernorm.restype = None
    L.orc_rmsnorm.argtypes = [f32p, C.c_int, f32p, C.c_float, f32p]; L.orc_rmsnorm.restype = None
    L.orc_gelu_tanh.argtypes = [C.c_float]; L.orc_gelu_tanh.restype = C.c_float
    L.orc_silu.argtypes = [C.c_float]; L.orc_silu.restype = C.c_float
    L.orc_rope.argtypes = [f32p, C.c_int, C.c_int, C.c_float]; L.orc_rope.restype = None
    L.orc_attend.argtypes = [f32p, u16p, u16p, C.c_int, C.c_int, f32p]; L.orc_attend.restype = None
    L.orc_sample.argtypes = [f32p, C.c_int32, C.c_float, C.c_int32, C.c_float, C.c_int32, C.c_double,
                             C.POINTER(C.c_double)]
    L.orc_sample.restype = C.c_int32
    L.orc_sample_pen.argtypes = [f32p, C.c_int32, u8p, C.c_float, C.c_float, C.c_int32, C.c_float, C.c_int32,
                                 C.c_double, C.POINTER(C.c_double)]
    L.orc_sample_pen.restype = C.c_int32
    L.orc_sample_ladder.argtypes = [f32p, f32p, C.c_int32, C.c_float, u8p, C.c_float, C.c_float, C.c_float,
                                    C.c_float, C.c_int32, C.c_double, C.POINTER(C.c_double)]
    L.orc_sample_ladder.restype = C.c_int32
    L.orc_open.argtypes = [u8p, C.c_uint64, C.POINTER(C.c_void_p)]
    L.orc_close.argtypes = [C.c_void_p]; L.orc_close.restype = None
    L.orc_reset.argtypes = [C.c_void_p]; L.orc_reset.restype = None
    L.orc_set_threads.argtypes = [C.c_int]
    L.orc_pos.argtypes = [C.c_void_p, C.c_int]
    L.orc_copy_row.argtypes = [C.c_void_p, C.c_int, C.c_int]
    L.orc_token_forward.argtypes = [C.c_void_p, C.c_int, C.c_int32, f32p]
    L.orc_embed_forward.argtypes = [C.c_void_p, C.c_int, f32p, f32p]
    L.orc_talker_forward.argtypes = [C.c_void_p, C.c_int, f32p, f32p, f32p]
    L.orc_talker_embed.argtypes = [C.c_void_p, C.c_int32, f32p]
    L.orc_cp_forward.argtypes = [C.c_void_p, C.c_int, f32p, C.c_int, f32p]
    L.orc_cp_reset.argtypes = [C.c_void_p, C.c_int]; L.orc_cp_reset.restype = None
    L.orc_code_embed.argtypes = [C.c_void_p, C.c_int, C.c_int32, f32p]
    L.orc_code_embed_sum.argtypes = [C.c_void_p, i32p, f32p]


def _p(a, ct):
    return a.ctypes.data_as(C.POINTER(ct)) if a is not None else None


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


# ----------------------------------------------------------------------------- op-level

def half_to_float(h) -> np.ndarray:
    h = np.asarray(h, np.uint16).ravel()
    return np.array([lib().orc_half_to_float(int(v)) for v in h], np.float32)


def float_to_half(x) -> np.ndarray:
    x = np.asarray(x, np.float32).ravel()
    return np.array([lib().orc_float_to_half(float(v)) for v in x], np.uint16)


def dequant(kind: int, data: np.ndarray, rows: int, cols: int) -> np.ndarray:
    d = np.ascontiguousarray(data, np.uint8)
    out = np.empty((rows, cols), np.float32)
    rc = lib().orc_dequant(kind, _p(d, C.c_uint8), rows, cols, _p(out, C.c_float))
    if rc:
        raise ValueError("orc_dequant rejected its arguments")
    return out


def linear(kind: int, data: np.ndarray, rows: int, cols: int, x, bias=None) -> np.ndarray:
    d = np.ascontiguousarray(data, np.uint8 if kind else np.float32)
    xx = _f32(x)
    b = None if bias is None else _f32(bias)
    y = np.empty(rows, np.float32)
    rc = lib().orc_linear(kind, d.ctypes.data_as(C.POINTER(C.c_uint8)), rows, cols, _p(xx, C.c_float),
                          _p(b, C.c_float), _p(y, C.c_float))
    if rc:
        raise ValueError("orc_linear rejected its arguments")
    return y


def layernorm(x, g, b, eps=1e-5):
    x, g, b = _f32(x), _f32(g), _f32(b)
    out = np.empty_like(x)
    lib().orc_layernorm(_p(x, C.c_float), x.size, _p(g, C.c_float), _p(b, C.c_float), eps, _p(out, C.c_float))
    return out


def rmsnorm(x, g, eps=1e-5):
    x, g = _f32(x), _f32(g)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_p(x, C.c_float), x.size, _p(g, C.c_float), eps, _p(out, C.c_float))
    return out


def gelu_tanh(t):
    return np.array([lib().orc_gelu_tanh(float(v)) for v in np.ravel(t)], np.float32)


def silu(t):
    return np.array([lib().orc_silu(float(v)) for v in np.ravel(t)], np.float32)


def rope(x, pos: int, theta: float = 10000.0):
    x = _f32(x).copy()
    lib().orc_rope(_p(x, C.c_float), x.size, pos, theta)
    return x


def attend(q, k_half, v_half):
    q = _f32(q)
    k = np.ascontiguousarray(k_half, np.uint16)
    v = np.ascontiguousarray(v_half, np.uint16)
    n, hd = k.shape
    out = np.empty(hd, np.float32)
    lib().orc_attend(_p(q, C.c_float), _p(k, C.c_uint16), _p(v, C.c_uint16), n, hd, _p(out, C.c_float))
    return out


def sample(z, temperature=1.0, top_k=1, top_p=1.0, greedy=True, u=0.0, seen=None, rep_penalty=1.0):
    """Returns (token, margin); with seen and rep_penalty != 1 the logits of the
    seen tokens are penalised first."""
    z = _f32(z)
    m = C.c_double()
    if seen is not None and rep_penalty != 1.0:
        sn = np.ascontiguousarray(seen, np.uint8)
        tok = lib().orc_sample_pen(_p(z, C.c_float), z.size, _p(sn, C.c_uint8), float(rep_penalty),
                                   float(temperature), int(top_k), float(top_p), int(bool(greedy)), float(u),
                                   C.byref(m))
    else:
        tok = lib().orc_sample(_p(z, C.c_float), z.size, float(temperature), int(top_k), float(top_p),
                               int(bool(greedy)), float(u), C.byref(m))
    return int(tok), float(m.value)


def sample_ladder(z_cond, z_uncond=None, cfg_weight=0.0, seen=None, rep_penalty=1.0, temperature=1.0, min_p=0.0,
                  top_p=1.0, top_k=0, u=0.0, with_draw=False):
    """The multilingual T3's sampler ladder (CFG combine, repetition penalty,
    temperature, min_p, top-p, top-k, draw in vocabulary order).  Returns
    (token, margin), or (token, margin, draw distance) with with_draw."""
    zc = _f32(z_cond)
    zu = _f32(z_uncond) if z_uncond is not None else None
    sn = np.ascontiguousarray(seen, np.uint8) if seen is not None else None
    m, dd = C.c_double(), C.c_double()
    tok = lib().orc_sample_ladder(_p(zc, C.c_float), _p(zu, C.c_float), zc.size, float(cfg_weight),
                                  _p(sn, C.c_uint8), float(rep_penalty), float(temperature), float(min_p),
                                  float(top_p), int(top_k), float(u), C.byref(m), C.byref(dd))
    return (int(tok), float(m.value), float(dd.value)) if with_draw else (int(tok), float(m.value))


# ----------------------------------------------------------------------------- model-level

class Model:
    """One oracle model bound to a weight blob (kept alive by this object)."""

    def __init__(self, blob: np.ndarray, threads: int | None = None):
        self._blob = np.ascontiguousarray(blob, np.uint8)
        h = C.c_void_p()
        if lib().orc_open(_p(self._blob, C.c_uint8), self._blob.size, C.byref(h)):
            raise ValueError("oracle could not parse the weight blob")
        self._h = h
        self.threads = lib().orc_set_threads(threads if threads else 1)

    def close(self):
        if self._h:
            lib().orc_close(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self):
        lib().orc_reset(self._h)

    def pos(self, row=0):
        return lib().orc_pos(self._h, row)

    def token_forward(self, row: int, tok: int, vocab: int, want_logits=True):
        z = np.empty(vocab, np.float32) if want_logits else None
        if lib().orc_token_forward(self._h, row, int(tok), _p(z, C.c_float)):
            raise ValueError("orc_token_forward failed (bad token, row or full context)")
        return z

    def embed_forward(self, row: int, e, vocab: int, want_logits=True):
        """One position whose input is the vector e (a conditioning prefix row)."""
        e = _f32(e)
        z = np.empty(vocab, np.float32) if want_logits else None
        if lib().orc_embed_forward(self._h, row, _p(e, C.c_float), _p(z, C.c_float)):
            raise ValueError("orc_embed_forward failed (bad row or full context)")
        return z

    def talker_embed(self, tok: int, d: int):
        e = np.empty(d, np.float32)
        if lib().orc_talker_embed(self._h, int(tok), _p(e, C.c_float)):
            raise ValueError("bad talker token")
        return e

    def talker_forward(self, row: int, e, vocab: int, d: int):
        e = _f32(e)
        z = np.empty(vocab, np.float32)
        h = np.empty(d, np.float32)
        if lib().orc_talker_forward(self._h, row, _p(e, C.c_float), _p(z, C.c_float), _p(h, C.c_float)):
            raise ValueError("orc_talker_forward failed")
        return z, h

    def cp_forward(self, row: int, v, head: int, vocab: int):
        v = _f32(v)
        z = np.empty(vocab, np.float32) if head >= 1 else None
        if lib().orc_cp_forward(self._h, row, _p(v, C.c_float), head, _p(z, C.c_float)):
            raise ValueError("orc_cp_forward failed")
        return z

    def cp_reset(self, row: int):
        lib().orc_cp_reset(self._h, row)

    def copy_row(self, dst: int, src: int):
        """Row dst continues from row src's state (same inputs so far)."""
        if lib().orc_copy_row(self._h, dst, src):
            raise ValueError("bad row")

    def code_embed(self, j: int, code: int, d: int):
        e = np.empty(d, np.float32)
        if lib().orc_code_embed(self._h, j, int(code), _p(e, C.c_float)):
            raise ValueError("bad code")
        return e

    def code_embed_sum(self, codes, d: int):
        c = np.ascontiguousarray(codes, np.int32)
        e = np.empty(d, np.float32)
        if lib().orc_code_embed_sum(self._h, _p(c, C.c_int32), _p(e, C.c_float)):
            raise ValueError("bad codes")
        return e


@dataclass
class Trace:
    """What the oracle computed over one run of one row."""
    tokens: list = field(default_factory=list)     # sampled token (or [16] codes) per step
    logits: list = field(default_factory=list)     # logits per step (or [16][V] per frame)
    margins: list = field(default_factory=list)    # decision margin per sampled token


def _sampler_args(s):
    return dict(temperature=s.temperature, top_k=s.top_k, top_p=s.top_p, greedy=s.greedy)


def run_t3(model: Model, spec, prompt: np.ndarray, draws: np.ndarray, n_steps: int, sampler,
           keep_logits=True, forced=None, logit_steps=None, prompt_embeds=None) -> list:
    """GPT-2 / Llama: prompt then n_steps decode steps per row.

    prompt [B][P]; draws [n_steps+1][B] (draw 0 samples the prefill's token).
    Step i consumes the token sampled at step i-1 (the prefill's for i=0), or,
    with teacher forcing, forced[b][i-1] (the other implementation's token).
    Returns one Trace per row; trace.tokens[0] is the prefill's token and
    trace.logits[0] the logits of the last prompt position.  With logit_steps
    given, only those steps keep their logits (others hold None).  With
    prompt_embeds [B][P][d] the prompt positions take those vectors as their
    inputs instead of the prompt tokens' embedding rows (prompt then only gives
    the length)."""
    B = prompt.shape[0]
    V = spec.vocab
    traces = []
    sa = _sampler_args(sampler)
    for b in range(B):
        tr = Trace()
        z = None
        for i, tok in enumerate(prompt[b]):
            last = i == prompt.shape[1] - 1
            if prompt_embeds is not None:
                z = model.embed_forward(b, prompt_embeds[b][i], V, want_logits=last)
            else:
                z = model.token_forward(b, int(tok), V, want_logits=last)
        for i in range(n_steps + 1):
            tok, margin = sample(z, u=float(draws[i][b]), **sa)
            tr.tokens.append(tok)
            tr.margins.append(margin)
            if keep_logits:
                tr.logits.append(z if (logit_steps is None or i in logit_steps) else None)
            if i < n_steps:
                feed = tok if forced is None else int(forced[b][i])
                z = model.token_forward(b, feed, V)
        traces.append(tr)
    return traces


def run_t3_cfg(model: Model, spec, prompt: np.ndarray, draws: np.ndarray, n_steps: int, ladder,
               forced=None) -> Trace:
    """The multilingual T3 with classifier-free guidance: row 0 reads the
    conditional prompt, row 1 the unconditional one (same length), and both rows
    are fed the one token that the sampler ladder picks from the two rows' logits
    ("Multilingual (Llama-520M) variant", sampling path: the cond and uncond
    forwards are combined at the logit level).

    prompt [2][P]; draws [n_steps+1] (draw 0 samples the prefill's token);
    ladder holds cfg_weight, rep_penalty, temperature, min_p, top_p, top_k.  The
    repetition penalty's history is the tokens fed forward since the prompt (the
    prompt's own tokens are not in it): step i's ladder sees the tokens fed at
    steps 1..i.  With teacher forcing, forced[i-1] is fed at step i instead of
    the sampled token (and joins the history).  Returns one Trace whose logits
    are (conditional, unconditional) pairs."""
    V = spec.vocab
    assert prompt.shape[0] == 2
    zs = []
    for b in range(2):
        z = None
        for i, tok in enumerate(prompt[b]):
            z = model.token_forward(b, int(tok), V, want_logits=(i == prompt.shape[1] - 1))
        zs.append(z)
    seen = np.zeros(V, np.uint8)
    tr = Trace()
    for i in range(n_steps + 1):
        tok, margin = sample_ladder(zs[0], zs[1], ladder.cfg_weight, seen, ladder.rep_penalty,
                                    ladder.temperature, ladder.min_p, ladder.top_p, ladder.top_k,
                                    u=float(draws[i]))
        tr.tokens.append(tok)
        tr.margins.append(margin)
        tr.logits.append((zs[0], zs[1]))
        if i < n_steps:
            feed = tok if forced is None else int(forced[i])
            seen[feed] = 1
            zs = [model.token_forward(b, feed, V) for b in range(2)]
    return tr


def run_qwen(model: Model, spec, prompt: np.ndarray, draws: np.ndarray, n_frames: int, talker_sampler,
             cp_sampler, keep_logits=True, forced=None) -> list:
    """Talker + code predictor: prompt then frames per row.

    Frame 0 is produced by the prompt: the last prompt position's Talker logits
    give code 0 and its hidden state seeds the code predictor.  Frame f >= 1
    runs the Talker on the sum of frame f-1's 16 code embeddings.  Within a
    frame: code-predictor position 0 takes Pr*h_T, position 1 takes Pr*E_0[c0]
    and head 1 samples c1; position j takes Pr*E_{j-1}[c_{j-1}] and head j
    samples c_j.  draws [n_frames+1][B][16].  With teacher forcing the codes
    fed forward (inside the frame and into the next frame) are forced[b][f]
    instead of the sampled ones.  A Talker sampler with rep_penalty != 1
    penalises the codebook-0 tokens fed to the Talker so far (frames 0..f-1 at
    frame f; the prompt's tokens are not in the history).  Returns one Trace per
    row with tokens [16] per frame and logits as a list of 16 arrays per frame."""
    B = prompt.shape[0]
    d, V0, Vc, ncb = spec.d_model, spec.vocab, spec.cp_vocab, spec.n_codebooks
    ta, ca = _sampler_args(talker_sampler), _sampler_args(cp_sampler)
    # every row's prompt first; a row whose prompt equals an earlier row's takes a
    # copy of that row's state right after its prompt (the rows are independent)
    prompt_end = []
    for b in range(B):
        same = [a for a in range(b) if np.array_equal(prompt[a], prompt[b])]
        if same:
            model.copy_row(b, same[0])
            prompt_end.append(prompt_end[same[0]])
            continue
        z0 = h = None
        for tok in prompt[b]:
            z0, h = model.talker_forward(b, model.talker_embed(int(tok), d), V0, d)
        prompt_end.append((z0, h))
    pen = float(getattr(talker_sampler, "rep_penalty", 1.0))
    traces = []
    for b in range(B):
        tr = Trace()
        z0, h = prompt_end[b]
        seen0 = np.zeros(V0, np.uint8)
        for f in range(n_frames + 1):
            codes, zs, ms = [], [z0], []
            c0, m0 = sample(z0, u=float(draws[f][b][0]), seen=seen0, rep_penalty=pen, **ta)
            codes.append(c0); ms.append(m0)
            model.cp_reset(b)
            model.cp_forward(b, h, 0, Vc)
            feed = codes if forced is None else [int(c) for c in forced[b][f]]
            for j in range(1, ncb):
                z = model.cp_forward(b, model.code_embed(j - 1, feed[j - 1], d), j, Vc)
                cj, mj = sample(z, u=float(draws[f][b][j]), **ca)
                codes.append(cj); ms.append(mj); zs.append(z)
            tr.tokens.append(codes)
            tr.margins.append(ms)
            if keep_logits:
                tr.logits.append(zs)
            if f < n_frames:
                feed = codes if forced is None else [int(c) for c in forced[b][f]]
                seen0[feed[0]] = 1
                z0, h = model.talker_forward(b, model.code_embed_sum(feed, d), V0, d)
        traces.append(tr)
    return traces
