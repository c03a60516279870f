"""Seeded synthetic weights, their block quantisation, and seeded prompts.

Weights are drawn N(0, 0.02) per tensor from numpy's Philox bit generator keyed
by (seed, tensor index); norm gains are 1 + N(0, 0.02) and norm offsets and
biases N(0, 0.02), so that every fused term of the decode step is exercised.

Quantisers (they produce the stored inputs; the decode step only dequantises):

* Q8_0 -- blocks of 32 int8 codes with one fp16 scale d = max|w|/127; codes are
  round-half-away-from-zero of w/d (d taken in fp32), clamped to +-127.  The
  format is the ggml legacy block type named in "Chatterbox -> ggml Port:
  Development Journal", Tier A item A3.
* Q4_0 -- blocks of 32 unsigned 4-bit codes offset by 8 with one fp16 scale
  d = m/-8, where m is the signed element of largest magnitude (first on ties);
  code q = min(15, floor(w/d + 8.5)).  Element j < 16 of a block sits in the low
  nibble of byte j, element j+16 in its high nibble; a block is 2 + 16 = 18
  bytes and a row of K weights is K/32 blocks back to back (journal section
  3.23).
* A8G64 -- affine groups of 64: unsigned 8-bit q with fp16 scale and fp16 bias
  per group, w = scale*q + bias, scale = (max-min)/255, bias = min, q =
  round-half-even((w - bias)/scale) clamped to [0, 255] (about 8.5 bits per
  weight, "Every Frame Is a Memory Read", section 3).
* Q5_0 -- blocks of 32 unsigned 5-bit codes offset by 16 with one fp16 scale
  d = m/-16 (m as for Q4_0); code q = min(31, floor(w/d + 16.5)).  A block is the
  fp16 d, a little-endian u32 whose bit j is the fifth bit of element j, and the
  16 bytes of low nibbles laid out as in Q4_0: 22 bytes (the ggml legacy block
  type of the journal's Tier A item A3).
* A4G32 / A4G64 -- affine groups of 32 / 64: unsigned 4-bit q with fp16 scale and
  bias per group, scale = (max-min)/15, bias = min, q = round-half-even((w -
  bias)/scale) clamped to [0, 15]; two codes per byte, element 2i in the low
  nibble ("Every Frame Is a Memory Read", section 5.8: the 4-bit group-32 and
  group-64 code predictor).
"""

from __future__ import annotations

import numpy as np

from . import presets as P
from .blob import KIND_F32, KIND_Q4_0, KIND_Q8_0, KIND_A8G64, KIND_Q5_0, KIND_A4G32, KIND_A4G64, write_blob

_QKIND = {P.Q8_0: KIND_Q8_0, P.Q4_0: KIND_Q4_0, P.A8G64: KIND_A8G64, P.Q5_0: KIND_Q5_0, P.A4G32: KIND_A4G32,
          P.A4G64: KIND_A4G64}


# ----------------------------------------------------------------------------- quantisers

def _round_half_away(x: np.ndarray) -> np.ndarray:
    a = np.abs(x)
    fl = np.floor(a)
    r = fl + ((a - fl) >= 0.5)           # a - fl is exact in fp32
    return np.copysign(r, x)


def quantize_q8_0(w: np.ndarray) -> np.ndarray:
    """fp32 [rows, K] -> uint8 [rows, K/32, 34] (fp16 d, then 32 int8)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, k = w.shape
    assert k % 32 == 0
    b = w.reshape(rows, k // 32, 32)
    amax = np.max(np.abs(b), axis=-1)
    d = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        inv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    q = _round_half_away((b * inv[..., None]).astype(np.float32))
    q = np.clip(q, -127, 127).astype(np.int8)
    out = np.empty((rows, k // 32, 34), dtype=np.uint8)
    out[..., 0:2] = d.astype(np.float16).view(np.uint8).reshape(rows, k // 32, 2)
    out[..., 2:] = q.view(np.uint8)
    return out


def quantize_q4_0(w: np.ndarray) -> np.ndarray:
    """fp32 [rows, K] -> uint8 [rows, K/32, 18] (fp16 d, then 16 nibble bytes)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, k = w.shape
    assert k % 32 == 0
    b = w.reshape(rows, k // 32, 32)
    idx = np.argmax(np.abs(b), axis=-1)                      # first on ties
    m = np.take_along_axis(b, idx[..., None], axis=-1)[..., 0]
    d = (m / np.float32(-8.0)).astype(np.float32)
    d[d == 0] = np.float32(0.0)                              # an all-zero block stores +0, not -0
    with np.errstate(divide="ignore"):
        inv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    x = (b * inv[..., None] + np.float32(8.5)).astype(np.float32)
    q = np.minimum(np.float32(15), np.floor(x))
    q = np.clip(q, 0, 15).astype(np.uint8)
    q = np.where((d != 0)[..., None], q, np.uint8(8)).astype(np.uint8)
    out = np.empty((rows, k // 32, 18), dtype=np.uint8)
    out[..., 0:2] = d.astype(np.float16).view(np.uint8).reshape(rows, k // 32, 2)
    out[..., 2:] = q[..., :16] | (q[..., 16:] << 4)
    return out


def quantize_a8g64(w: np.ndarray):
    """fp32 [rows, K] -> (q uint8 [rows, K], scale fp16 [rows, K/64], bias fp16 [rows, K/64])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, k = w.shape
    assert k % 64 == 0
    g = w.reshape(rows, k // 64, 64)
    mn = g.min(axis=-1)
    mx = g.max(axis=-1)
    scale = ((mx - mn) / np.float32(255.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(scale[..., None] != 0, (g - mn[..., None]) / scale[..., None], 0).astype(np.float32)
    q = np.clip(np.rint(t), 0, 255).astype(np.uint8).reshape(rows, k)
    return q, scale.astype(np.float16), mn.astype(np.float16)


def quantize_q5_0(w: np.ndarray) -> np.ndarray:
    """fp32 [rows, K] -> uint8 [rows, K/32, 22] (fp16 d, u32 fifth bits, 16 nibble bytes)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, k = w.shape
    assert k % 32 == 0
    b = w.reshape(rows, k // 32, 32)
    idx = np.argmax(np.abs(b), axis=-1)                      # first on ties
    m = np.take_along_axis(b, idx[..., None], axis=-1)[..., 0]
    d = (m / np.float32(-16.0)).astype(np.float32)
    d[d == 0] = np.float32(0.0)
    with np.errstate(divide="ignore"):
        inv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    x = (b * inv[..., None] + np.float32(16.5)).astype(np.float32)
    q = np.clip(np.minimum(np.float32(31), np.floor(x)), 0, 31).astype(np.uint32)
    q = np.where((d != 0)[..., None], q, np.uint32(16)).astype(np.uint32)
    qh = ((q >> 4) << np.arange(32, dtype=np.uint32)).sum(axis=-1, dtype=np.uint64).astype(np.uint32)
    lo = (q & 0xF).astype(np.uint8)
    out = np.empty((rows, k // 32, 22), dtype=np.uint8)
    out[..., 0:2] = d.astype(np.float16).view(np.uint8).reshape(rows, k // 32, 2)
    out[..., 2:6] = qh.astype("<u4").view(np.uint8).reshape(rows, k // 32, 4)
    out[..., 6:] = lo[..., :16] | (lo[..., 16:] << 4)
    return out


def quantize_a4(w: np.ndarray, group: int):
    """fp32 [rows, K] -> (codes uint8 [rows, K/2], scale fp16 [rows, K/group], bias fp16 [rows, K/group])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, k = w.shape
    assert k % group == 0
    g = w.reshape(rows, k // group, group)
    mn = g.min(axis=-1)
    mx = g.max(axis=-1)
    scale = ((mx - mn) / np.float32(15.0)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(scale[..., None] != 0, (g - mn[..., None]) / scale[..., None], 0).astype(np.float32)
    q = np.clip(np.rint(t), 0, 15).astype(np.uint8).reshape(rows, k)
    packed = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return packed, scale.astype(np.float16), mn.astype(np.float16)


def quantize(w: np.ndarray, quant: int):
    if quant == P.Q8_0:
        return quantize_q8_0(w)
    if quant == P.Q4_0:
        return quantize_q4_0(w)
    if quant == P.A8G64:
        return quantize_a8g64(w)
    if quant == P.Q5_0:
        return quantize_q5_0(w)
    if quant == P.A4G32:
        return quantize_a4(w, 32)
    if quant == P.A4G64:
        return quantize_a4(w, 64)
    raise ValueError(f"unknown quant {quant}")


def tensor_quant(m: P.ModelSpec, name: str) -> int:
    """The weight format of matrix ``name``: the code predictor's tensors (``c<l>.*``,
    ``cp.*``) take ``cp_quant`` when it is set."""
    if m.cp_quant and (name.startswith("cp.") or (name.startswith("c") and name[1:2].isdigit())):
        return m.cp_quant
    return m.quant


# ----------------------------------------------------------------------------- tensor list

def tensor_list(m: P.ModelSpec):
    """Canonical (name, role, rows, cols) list.  role: emb | gain | bias | mat."""
    t = []
    if m.arch == P.ARCH_GPT2:
        d, f = m.d_model, m.d_ff
        t.append(("wte", "emb", m.vocab, d))
        t.append(("wpe", "emb", m.max_ctx, d))
        for l in range(m.n_layer):
            t += [(f"l{l}.ln1.g", "gain", 1, d), (f"l{l}.ln1.b", "bias", 1, d),
                  (f"l{l}.wqkv", "mat", m.qkv_rows, d), (f"l{l}.bqkv", "bias", 1, m.qkv_rows),
                  (f"l{l}.wo", "mat", d, m.q_dim), (f"l{l}.bo", "bias", 1, d),
                  (f"l{l}.ln2.g", "gain", 1, d), (f"l{l}.ln2.b", "bias", 1, d),
                  (f"l{l}.wfc", "mat", f, d), (f"l{l}.bfc", "bias", 1, f),
                  (f"l{l}.wproj", "mat", d, f), (f"l{l}.bproj", "bias", 1, d)]
        t += [("lnf.g", "gain", 1, d), ("lnf.b", "bias", 1, d), ("whead", "mat", m.vocab, d)]
    elif m.arch == P.ARCH_LLAMA:
        d, f = m.d_model, m.d_ff
        t.append(("wte", "emb", m.vocab, d))
        for l in range(m.n_layer):
            t += [(f"l{l}.rms1.g", "gain", 1, d), (f"l{l}.wqkv", "mat", m.qkv_rows, d),
                  (f"l{l}.wo", "mat", d, m.q_dim), (f"l{l}.rms2.g", "gain", 1, d),
                  (f"l{l}.wgu", "mat", 2 * f, d), (f"l{l}.wdown", "mat", d, f)]
        t += [("normf.g", "gain", 1, d), ("whead", "mat", m.vocab, d)]
    elif m.arch == P.ARCH_QWEN_TTS:
        d, f = m.d_model, m.d_ff
        t.append(("emb.0", "emb", m.vocab, d))
        for j in range(1, m.n_codebooks):
            t.append((f"emb.{j}", "emb", m.cp_vocab, d))
        for l in range(m.n_layer):
            t += [(f"t{l}.rms1.g", "gain", 1, d), (f"t{l}.wqkv", "mat", m.qkv_rows, d),
                  (f"t{l}.wo", "mat", d, m.q_dim), (f"t{l}.rms2.g", "gain", 1, d),
                  (f"t{l}.wgu", "mat", 2 * f, d), (f"t{l}.wdown", "mat", d, f)]
        t += [("t.normf.g", "gain", 1, d), ("t.head", "mat", m.vocab, d)]
        cd, cf = m.cp_d_model, m.cp_d_ff
        cqkv = (m.cp_n_head + 2 * m.cp_n_kv_head) * m.cp_head_dim
        t.append(("cp.proj", "mat", cd, d))
        for l in range(m.cp_layer):
            t += [(f"c{l}.rms1.g", "gain", 1, cd), (f"c{l}.wqkv", "mat", cqkv, cd),
                  (f"c{l}.wo", "mat", cd, m.cp_n_head * m.cp_head_dim), (f"c{l}.rms2.g", "gain", 1, cd),
                  (f"c{l}.wgu", "mat", 2 * cf, cd), (f"c{l}.wdown", "mat", cd, cf)]
        t.append(("cp.normf.g", "gain", 1, cd))
        for j in range(1, m.n_codebooks):
            t.append((f"cp.head.{j}", "mat", m.cp_vocab, cd))
    else:
        raise ValueError(f"unknown arch {m.arch}")
    return t


def _draw(seed: int, index: int, n: int) -> np.ndarray:
    rng = np.random.Generator(np.random.Philox(key=np.array([seed, index], dtype=np.uint64)))
    return rng.standard_normal(n, dtype=np.float32)


def generate_tensor(m: P.ModelSpec, seed: int, index: int, role: str, rows: int, cols: int) -> np.ndarray:
    """fp32 values of one tensor, drawn from its own Philox key (seed, index)."""
    z = _draw(seed, index, rows * cols).reshape(rows, cols)
    z *= np.float32(0.02)
    if role == "gain":
        z += np.float32(1.0)
    return z


def build_model_blob(m: P.ModelSpec, seed: int = 1, keep_fp32: bool = False):
    """Generate, quantise and serialise every tensor of model ``m``.

    Returns (blob: bytes-like numpy uint8 array, fp32: dict name -> fp32 array
    of the *unquantised* values when keep_fp32 else {}).
    """
    entries = []
    fp32 = {}
    for index, (name, role, rows, cols) in enumerate(tensor_list(m)):
        w = generate_tensor(m, seed, index, role, rows, cols)
        if keep_fp32:
            fp32[name] = w
        if role == "mat":
            q = tensor_quant(m, name)
            entries.append((name, _QKIND[q], rows, cols, quantize(w, q)))
        else:
            entries.append((name, KIND_F32, rows, cols, w))
    return write_blob(m, entries), fp32


def prompt_tokens(run: P.RunSpec, rows: int | None = None) -> np.ndarray:
    """Seeded prompt token IDs [rows][prompt_len], uniform in [0, prompt_vocab).

    When ``run.extra['shared_prompt']`` is set every row gets row 0's prompt
    (G rollouts of one prompt)."""
    rows = run.model.batch if rows is None else rows
    rng = np.random.Generator(np.random.Philox(key=np.array([run.prompt_seed, 0], dtype=np.uint64)))
    toks = rng.integers(0, run.prompt_vocab, size=(rows, run.prompt_len), dtype=np.int64)
    if run.extra.get("shared_prompt"):
        toks[:] = toks[0]
    return toks.astype(np.int32)
