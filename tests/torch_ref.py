"""A second, independent statement of the decode forward for pinning the oracle.

Written from the same model description with torch float64 library ops
(layer_norm, rms_norm, gelu, silu, scaled_dot_product_attention with a causal
mask) over the *whole* sequence at once -- full causal recompute rather than
the oracle's incremental KV-cache decode.  Activations are rounded to fp32 and
K/V to fp16 at the same points the method stores them, so the two statements
agree to within fp32 rounding noise.  Test helper only.
"""

from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from synth import presets as P
from synth.blob import read_table, KIND_F32


def r32(t):
    return t.float().double()


class Weights:
    def __init__(self, blob):
        self.blob = np.asarray(blob, np.uint8)
        self.table = read_table(self.blob)

    def get(self, name):
        kind, rows, cols, off, nb = self.table[name]
        raw = self.blob[off:off + nb]
        if kind == KIND_F32:
            a = raw.view(np.float32).reshape(rows, cols)
        else:
            a = oracle.dequant(kind, raw, rows, cols)
        return torch.tensor(a.astype(np.float64))

    def vec(self, name):
        return self.get(name)[0]


def _rope(x, theta):
    """x [T, H, hd]; NEOX half-split rotation as a complex product."""
    T, H, hd = x.shape
    half = hd // 2
    i = torch.arange(half, dtype=torch.float64)
    phi = torch.arange(T, dtype=torch.float64)[:, None] * theta ** (-2.0 * i / hd)
    z = torch.complex(x[..., :half], x[..., half:]) * torch.polar(torch.ones_like(phi), phi)[:, None, :]
    return torch.cat([z.real, z.imag], dim=-1)


def stack_forward(W: Weights, X, pfx, n_layer, d, H, Hk, hd, ff, gpt2, eps, theta, final_norm):
    """X [T, d] float64 inputs (already fp32-valued).  Returns final-normed hidden [T, d]."""
    T = X.shape[0]
    qd, kd = H * hd, Hk * hd
    for l in range(n_layer):
        g = lambda n: W.vec(f"{pfx}{l}.{n}")
        if gpt2:
            h = r32(F.layer_norm(X, (d,), g("ln1.g"), g("ln1.b"), eps=eps))
            qkv = r32(h @ W.get(f"{pfx}{l}.wqkv").T + g("bqkv"))
        else:
            h = r32(F.rms_norm(X, (d,), g("rms1.g"), eps=eps))
            qkv = r32(h @ W.get(f"{pfx}{l}.wqkv").T)
        q = qkv[:, :qd].reshape(T, H, hd)
        k = qkv[:, qd:qd + kd].reshape(T, Hk, hd)
        v = qkv[:, qd + kd:].reshape(T, Hk, hd)
        if not gpt2:
            q, k = r32(_rope(q, theta)), r32(_rope(k, theta))
        k16, v16 = k.half().double(), v.half().double()
        rep = H // Hk
        k16 = k16.repeat_interleave(rep, dim=1)
        v16 = v16.repeat_interleave(rep, dim=1)
        o = F.scaled_dot_product_attention(q.transpose(0, 1), k16.transpose(0, 1), v16.transpose(0, 1),
                                           is_causal=True)
        o = r32(o.transpose(0, 1).reshape(T, qd))
        y = o @ W.get(f"{pfx}{l}.wo").T
        if gpt2:
            y = y + g("bo")
        X = r32(X + r32(y))
        if gpt2:
            h = r32(F.layer_norm(X, (d,), g("ln2.g"), g("ln2.b"), eps=eps))
            t = r32(h @ W.get(f"{pfx}{l}.wfc").T + g("bfc"))
            u = r32(F.gelu(t, approximate="tanh"))
            y = r32(u @ W.get(f"{pfx}{l}.wproj").T + g("bproj"))
        else:
            h = r32(F.rms_norm(X, (d,), g("rms2.g"), eps=eps))
            gu = r32(h @ W.get(f"{pfx}{l}.wgu").T)
            u = r32(r32(F.silu(gu[:, :ff])) * gu[:, ff:])
            y = r32(u @ W.get(f"{pfx}{l}.wdown").T)
        X = r32(X + y)
    nf = final_norm
    if gpt2:
        return r32(F.layer_norm(X, (d,), W.vec(nf + ".g"), W.vec(nf + ".b"), eps=eps))
    return r32(F.rms_norm(X, (d,), W.vec(nf + ".g"), eps=eps))


def t3_logits(blob, m: P.ModelSpec, tokens, prefix=None):
    """Logits at every position of a token sequence [T] (GPT-2 or Llama); with
    prefix [P][d], positions 0..P-1 take those vectors in place of their tokens'
    embedding rows (tokens then starts with P placeholders)."""
    W = Weights(blob)
    toks = torch.tensor(np.asarray(tokens, np.int64))
    T = len(toks)
    X = W.get("wte")[toks]
    if prefix is not None:
        X = X.clone()
        X[: len(prefix)] = torch.from_numpy(np.asarray(prefix, np.float32)).to(X.dtype)
    gpt2 = m.arch == P.ARCH_GPT2
    if gpt2:
        X = r32(X + W.get("wpe")[:T])
    h = stack_forward(W, X, "l", m.n_layer, m.d_model, m.n_head, m.n_kv_head, m.head_dim, m.d_ff, gpt2,
                      m.norm_eps, m.rope_theta, "lnf" if gpt2 else "normf")
    return r32(h @ W.get("whead").T).numpy()


def qwen_frame_logits(blob, m: P.ModelSpec, prompt, frames):
    """Teacher-forced logits of every frame given the codes of all frames.

    prompt [P] tokens; frames [F][16] codes.  Returns [F][16][V] logits (pass 0
    on the codebook-0 vocab) computed by full causal recompute of the Talker
    over [prompt embeddings, code-embedding sums of frames 0..F-2] and of the
    code predictor over each frame's [Pr h_T, Pr E_0[c0], ..., Pr E_14[c14]]."""
    W = Weights(blob)
    d = m.d_model
    E = [W.get(f"emb.{j}") for j in range(m.n_codebooks)]
    frames = np.asarray(frames, np.int64)
    F_ = len(frames)
    X = [E[0][int(t)] for t in prompt]
    for f in range(F_ - 1):
        X.append(r32(sum(E[j][int(frames[f][j])] for j in range(m.n_codebooks))))
    X = torch.stack(X)
    hT = stack_forward(W, X, "t", m.n_layer, d, m.n_head, m.n_kv_head, m.head_dim, m.d_ff, False,
                       m.norm_eps, m.rope_theta, "t.normf")
    z0 = r32(hT @ W.get("t.head").T)
    Pr = W.get("cp.proj")
    out = []
    P_len = len(prompt)
    for f in range(F_):
        h = hT[P_len - 1 + f]
        vin = [h] + [E[j][int(frames[f][j])] for j in range(m.n_codebooks - 1)]
        Xc = r32(torch.stack(vin) @ Pr.T)
        hc = stack_forward(W, Xc, "c", m.cp_layer, m.cp_d_model, m.cp_n_head, m.cp_n_kv_head, m.cp_head_dim,
                           m.cp_d_ff, False, m.norm_eps, m.rope_theta, "cp.normf")
        zs = [z0[P_len - 1 + f].numpy()]
        for j in range(1, m.n_codebooks):
            zs.append(r32(hc[j] @ W.get(f"cp.head.{j}").T).numpy())
        out.append(zs)
    return out
