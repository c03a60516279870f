"""Thin ctypes binding of libsd.so (include/sd.h, include/sd_ops.h).

Argument marshalling only: every step of the decode path runs in the
library's CUDA kernels.  Functions keep the C names; a negative return code
raises SdError with the library's message.  Device pointers can be given as
integers or as objects with ``data_ptr()`` (torch tensors); host arrays are
numpy arrays.  If the library has not been built, importing works but the
first call raises: there is no fallback path.
"""

from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsd.so")

SD_OK = 0
ERRORS = {-1: "SD_ERR_INVALID_ARG", -2: "SD_ERR_STATE", -3: "SD_ERR_CTX_FULL", -4: "SD_ERR_OOM",
          -5: "SD_ERR_CUDA", -6: "SD_ERR_TIMEOUT", -7: "SD_ERR_UNSUPPORTED", -8: "SD_ERR_BLOB",
          -9: "SD_ERR_DEVICE"}
MAX_CODEBOOKS = 16

# every symbol the headers declare
EXPORTS = ["sd_create", "sd_load_weights", "sd_prefill", "sd_prefill_shared", "sd_prefill_embeds", "sd_step", "sd_frame", "sd_set_forced_codes", "sd_set_ladder",
           "sd_decode_n", "sd_get_logits", "sd_reset", "sd_destroy", "sd_last_error", "sd_get_info",
           "sd_qmat_create", "sd_qmat_destroy", "sd_qmat_dequant", "sd_qmat_gemv", "sd_qmat_gemm", "sd_qmat_gemm16", "sd_qmat_gemm_tc", "sd_sample_rows", "sd_sample_rows_ladder",
           "sd_attend_rows", "sd_attend_rows_static"]


class SdError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class ModelConfig(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("arch", "n_layer", "d_model", "n_head", "n_kv_head", "head_dim", "d_ff",
                                         "vocab", "max_ctx", "batch", "quant")] + \
               [("rope_theta", C.c_float), ("norm_eps", C.c_float)] + \
               [(n, C.c_int32) for n in ("cp_layer", "cp_d_model", "cp_n_head", "cp_n_kv_head", "cp_head_dim",
                                         "cp_d_ff", "cp_vocab", "n_codebooks", "cp_max_ctx")]

    @classmethod
    def from_spec(cls, m) -> "ModelConfig":
        return cls(**{f: getattr(m, f) for f, _ in cls._fields_})


class Sampler(C.Structure):
    """sd_sampler; rep_penalty 0 (the default) or 1 applies no penalty."""
    _fields_ = [("temperature", C.c_float), ("top_k", C.c_int32), ("top_p", C.c_float), ("greedy", C.c_int32),
                ("rep_penalty", C.c_float)]

    @classmethod
    def from_spec(cls, s) -> "Sampler":
        return cls(float(s.temperature), int(s.top_k), float(s.top_p), int(bool(s.greedy)),
                   float(getattr(s, "rep_penalty", 1.0)))


class SamplerLadder(C.Structure):
    """sd_sampler_ladder: CFG weight, repetition penalty, temperature, min_p, top_p, top_k."""
    _fields_ = [("cfg_weight", C.c_float), ("repetition_penalty", C.c_float), ("temperature", C.c_float),
                ("min_p", C.c_float), ("top_p", C.c_float), ("top_k", C.c_int32)]

    @classmethod
    def from_spec(cls, spec) -> "SamplerLadder":
        return cls(spec.cfg_weight, spec.rep_penalty, spec.temperature, spec.min_p, spec.top_p, spec.top_k)


class Info(C.Structure):
    _fields_ = [("pos", C.c_int32), ("sm_count", C.c_int32), ("kernels_per_step", C.c_int32),
                ("attn_splits", C.c_int32), ("weight_bytes", C.c_int64), ("kv_bytes", C.c_int64),
                ("step_h2d_bytes", C.c_int64), ("step_d2h_bytes", C.c_int64), ("persistent", C.c_int32),
                ("prefill", C.c_int32), ("persistent_clusters", C.c_int32), ("cluster_size", C.c_int32)]


_lib = None


def load_library(path: str | None = None):
    """Load libsd.so (raises if it is missing: the library must be built)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libsd.so not found at {p}: build it with __graft_entry__.build() "
                           "or python autoregressive_speech_token_gb300/build.py")
    L = C.CDLL(p)
    vp, i32, i64, f32p, i32p = C.c_void_p, C.c_int32, C.c_int64, C.POINTER(C.c_float), C.POINTER(C.c_int32)
    sig = {
        "sd_create": ([C.POINTER(ModelConfig), C.c_int, vp, C.POINTER(vp)], C.c_int),
        "sd_load_weights": ([vp, vp, C.c_size_t, C.c_int], C.c_int),
        "sd_prefill": ([vp, i32p, i32, C.POINTER(Sampler), f32p, i32p], C.c_int),
        "sd_prefill_shared": ([vp, i32p, i32, C.POINTER(Sampler), f32p, i32p], C.c_int),
        "sd_prefill_embeds": ([vp, f32p, i32, C.POINTER(Sampler), f32p, i32p], C.c_int),
        "sd_step": ([vp, i32p, C.POINTER(Sampler), f32p, i32p], C.c_int),
        "sd_frame": ([vp, i32p, C.POINTER(Sampler), C.POINTER(Sampler), f32p, i32p], C.c_int),
        "sd_set_forced_codes": ([vp, i32p], C.c_int),
        "sd_set_ladder": ([vp, C.POINTER(SamplerLadder)], C.c_int),
        "sd_decode_n": ([vp, i32, C.POINTER(Sampler), vp, vp], C.c_int),
        "sd_get_logits": ([vp, f32p, C.c_size_t], C.c_int),
        "sd_reset": ([vp], C.c_int),
        "sd_destroy": ([vp], None),
        "sd_last_error": ([vp], C.c_char_p),
        "sd_get_info": ([vp, C.POINTER(Info)], C.c_int),
        "sd_qmat_create": ([C.c_int, vp, i64, i64, C.c_int, C.c_int, C.POINTER(vp)], C.c_int),
        "sd_qmat_destroy": ([vp], None),
        "sd_qmat_dequant": ([vp, vp, vp], C.c_int),
        "sd_qmat_gemv": ([vp, vp, i32, vp, vp, vp], C.c_int),
        "sd_qmat_gemm": ([vp, vp, i32, i32, vp, vp, vp, vp], C.c_int),
        "sd_qmat_gemm16": ([vp, vp, i32, i32, vp, vp, vp, vp], C.c_int),
        "sd_qmat_gemm_tc": ([vp, vp, i32, i32, vp, vp, vp, vp], C.c_int),
        "sd_sample_rows": ([vp, i32, i32, C.POINTER(Sampler), vp, vp, vp], C.c_int),
        "sd_sample_rows_ladder": ([vp, vp, i32, i32, C.POINTER(SamplerLadder), vp, vp, vp, vp], C.c_int),
        "sd_attend_rows": ([vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp], C.c_int),
        "sd_attend_rows_static": ([vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp], C.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return L


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a device pointer, got {type(x)}")


def _check(rc: int, handle=None):
    if rc != SD_OK:
        msg = load_library().sd_last_error(handle)
        raise SdError(rc, msg.decode() if msg else "")


def _arr(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


def _p(a, ct):
    return a.ctypes.data_as(C.POINTER(ct))


# ------------------------------------------------------------------ model-level

def sd_create(cfg: ModelConfig, device: int = 0, stream=None) -> int:
    h = C.c_void_p()
    L = load_library()
    rc = L.sd_create(C.byref(cfg), device, stream if stream else None, C.byref(h))
    _check(rc, None)
    return h.value


def sd_load_weights(ctx: int, blob, blob_on_device: bool = False):
    L = load_library()
    if blob_on_device:
        rc = L.sd_load_weights(ctx, _ptr(blob), blob.numel() * blob.element_size(), 1)
    else:
        b = _arr(blob, np.uint8)
        rc = L.sd_load_weights(ctx, b.ctypes.data, b.nbytes, 0)
    _check(rc, ctx)


def sd_prefill(ctx: int, tokens: np.ndarray, sampler: Sampler, u: np.ndarray, out_width: int = 1) -> np.ndarray:
    t = _arr(tokens, np.int32)
    B, n = t.shape
    uu = _arr(u, np.float32)
    out = np.empty((B, out_width), np.int32)
    _check(load_library().sd_prefill(ctx, _p(t, C.c_int32), n, C.byref(sampler), _p(uu, C.c_float),
                                     _p(out, C.c_int32)), ctx)
    return out


def sd_prefill_shared(ctx: int, tokens: np.ndarray, batch: int, sampler: Sampler, u: np.ndarray,
                      out_width: int = 1) -> np.ndarray:
    """sd_prefill_shared: one prompt tokens [n] for every row."""
    t = _arr(tokens, np.int32).reshape(-1)
    uu = _arr(u, np.float32)
    out = np.empty((batch, out_width), np.int32)
    _check(load_library().sd_prefill_shared(ctx, _p(t, C.c_int32), t.size, C.byref(sampler), _p(uu, C.c_float),
                                            _p(out, C.c_int32)), ctx)
    return out


def sd_prefill_embeds(ctx: int, embeds: np.ndarray, sampler: Sampler, u: np.ndarray, out_width: int = 1) -> np.ndarray:
    """sd_prefill_embeds: embeds [batch][n][d_model] input vectors."""
    e = _arr(embeds, np.float32)
    B, n, _ = e.shape
    uu = _arr(u, np.float32)
    out = np.empty((B, out_width), np.int32)
    _check(load_library().sd_prefill_embeds(ctx, _p(e, C.c_float), n, C.byref(sampler), _p(uu, C.c_float),
                                            _p(out, C.c_int32)), ctx)
    return out


def sd_step(ctx: int, tok: np.ndarray, sampler: Sampler, u: np.ndarray) -> np.ndarray:
    t = _arr(tok, np.int32)
    uu = _arr(u, np.float32)
    out = np.empty_like(t)
    _check(load_library().sd_step(ctx, _p(t, C.c_int32), C.byref(sampler), _p(uu, C.c_float), _p(out, C.c_int32)),
           ctx)
    return out


def sd_frame(ctx: int, codes_in: np.ndarray, talker: Sampler, cp: Sampler, u: np.ndarray) -> np.ndarray:
    ci = _arr(codes_in, np.int32)
    uu = _arr(u, np.float32)
    out = np.empty_like(ci)
    _check(load_library().sd_frame(ctx, _p(ci, C.c_int32), C.byref(talker), C.byref(cp), _p(uu, C.c_float),
                                   _p(out, C.c_int32)), ctx)
    return out


def sd_set_forced_codes(ctx: int, codes) -> None:
    L = load_library()
    if codes is None:
        _check(L.sd_set_forced_codes(ctx, None), ctx)
        return
    c = _arr(codes, np.int32)
    B, ncb = c.shape
    full = np.zeros((B, MAX_CODEBOOKS), np.int32)
    full[:, :ncb] = c
    _check(L.sd_set_forced_codes(ctx, _p(full, C.c_int32)), ctx)


def sd_set_ladder(ctx: int, ladder) -> None:
    """sd_set_ladder: a SamplerLadder (one token per step for the cond / uncond row pair), or None."""
    L = load_library()
    _check(L.sd_set_ladder(ctx, C.byref(ladder) if ladder is not None else None), ctx)


def sd_decode_n(ctx: int, n_steps: int, sampler: Sampler, u_dev, out_dev) -> None:
    _check(load_library().sd_decode_n(ctx, n_steps, C.byref(sampler), _ptr(u_dev), _ptr(out_dev)), ctx)


def sd_get_logits(ctx: int, n_floats: int) -> np.ndarray:
    out = np.empty(n_floats, np.float32)
    _check(load_library().sd_get_logits(ctx, _p(out, C.c_float), n_floats), ctx)
    return out


def sd_reset(ctx: int) -> None:
    _check(load_library().sd_reset(ctx), ctx)


def sd_destroy(ctx: int) -> None:
    if ctx:
        load_library().sd_destroy(ctx)


def sd_last_error(ctx: int | None = None) -> str:
    m = load_library().sd_last_error(ctx)
    return m.decode() if m else ""


def sd_get_info(ctx: int) -> Info:
    info = Info()
    _check(load_library().sd_get_info(ctx, C.byref(info)), ctx)
    return info


# ------------------------------------------------------------------ op-level

def sd_qmat_create(quant: int, canon, rows: int, cols: int, on_device: bool = False, device: int = 0) -> int:
    h = C.c_void_p()
    L = load_library()
    if on_device:
        rc = L.sd_qmat_create(quant, _ptr(canon), rows, cols, 1, device, C.byref(h))
    else:
        c = _arr(canon, np.uint8)
        rc = L.sd_qmat_create(quant, c.ctypes.data, rows, cols, 0, device, C.byref(h))
    _check(rc, None)
    return h.value


def sd_qmat_destroy(m: int) -> None:
    if m:
        load_library().sd_qmat_destroy(m)


def sd_qmat_dequant(m: int, out_dev, stream=None) -> None:
    _check(load_library().sd_qmat_dequant(m, _ptr(out_dev), stream), None)


def sd_qmat_gemv(m: int, x_dev, nb: int, bias_dev, y_dev, stream=None) -> None:
    _check(load_library().sd_qmat_gemv(m, _ptr(x_dev), nb, _ptr(bias_dev), _ptr(y_dev), stream), None)


EPI_LINEAR, EPI_GELU, EPI_SWIGLU = 0, 1, 2


def sd_qmat_gemm(m: int, x_dev, M: int, epilogue: int, bias_dev, resid_dev, y_dev, stream=None) -> None:
    _check(load_library().sd_qmat_gemm(m, _ptr(x_dev), M, epilogue, _ptr(bias_dev), _ptr(resid_dev), _ptr(y_dev),
                                       stream), None)


def sd_qmat_gemm16(m: int, x_dev, M: int, epilogue: int, bias_dev, resid_dev, y_dev, stream=None) -> None:
    _check(load_library().sd_qmat_gemm16(m, _ptr(x_dev), M, epilogue, _ptr(bias_dev), _ptr(resid_dev),
                                         _ptr(y_dev), stream), None)


def sd_qmat_gemm_tc(m: int, x_dev, M: int, epilogue: int, bias_dev, resid_dev, y_dev, stream=None) -> None:
    _check(load_library().sd_qmat_gemm_tc(m, _ptr(x_dev), M, epilogue, _ptr(bias_dev), _ptr(resid_dev),
                                          _ptr(y_dev), stream), None)


def sd_sample_rows_ladder(logits_cond_dev, logits_uncond_dev, rows: int, V: int, sampler: SamplerLadder, seen_dev,
                          u_dev, out_dev, stream=None) -> None:
    _check(load_library().sd_sample_rows_ladder(_ptr(logits_cond_dev), _ptr(logits_uncond_dev), rows, V,
                                                C.byref(sampler), _ptr(seen_dev), _ptr(u_dev), _ptr(out_dev),
                                                stream), None)


def sd_sample_rows(logits_dev, rows: int, V: int, sampler: Sampler, u_dev, out_dev, stream=None) -> None:
    _check(load_library().sd_sample_rows(_ptr(logits_dev), rows, V, C.byref(sampler), _ptr(u_dev), _ptr(out_dev),
                                         stream), None)


def sd_attend_rows(q_dev, k_dev, v_dev, B, H, Hkv, hd, n_ctx, n, nsplit, out_dev, stream=None) -> None:
    _check(load_library().sd_attend_rows(_ptr(q_dev), _ptr(k_dev), _ptr(v_dev), B, H, Hkv, hd, n_ctx, n, nsplit,
                                         _ptr(out_dev), stream), None)


def sd_attend_rows_static(q_dev, k_dev, v_dev, B, H, Hkv, hd, n_ctx, n, nsplit, out_dev, stream=None) -> None:
    """sd_attend_rows without any device allocation (fixed scratch array)."""
    _check(load_library().sd_attend_rows_static(_ptr(q_dev), _ptr(k_dev), _ptr(v_dev), B, H, Hkv, hd, n_ctx, n,
                                                nsplit, _ptr(out_dev), stream), None)


# ------------------------------------------------------------------ convenience wrapper

class Decoder:
    """One decode context: weights, KV cache and captured step graphs."""

    def __init__(self, spec, blob, device: int = 0, stream=None, blob_on_device: bool = False):
        self.spec = spec
        self.cfg = ModelConfig.from_spec(spec)
        self.ctx = sd_create(self.cfg, device, stream)
        try:
            sd_load_weights(self.ctx, blob, blob_on_device)
        except Exception:
            sd_destroy(self.ctx)
            self.ctx = None
            raise
        self.qwen = spec.arch == 3
        self.n_logits = spec.batch * (MAX_CODEBOOKS * max(spec.vocab, spec.cp_vocab) if self.qwen else spec.vocab)

    def close(self):
        if self.ctx:
            sd_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, tokens, sampler, u):
        w = self.spec.n_codebooks if self.qwen else 1
        out = sd_prefill(self.ctx, tokens, sampler, u, out_width=w)
        return out if self.qwen else out[:, 0]

    def prefill_shared(self, tokens, sampler, u):
        """One prompt tokens [n] for every row (rollouts of one prompt)."""
        w = self.spec.n_codebooks if self.qwen else 1
        out = sd_prefill_shared(self.ctx, tokens, self.spec.batch, sampler, u, out_width=w)
        return out if self.qwen else out[:, 0]

    def prefill_embeds(self, embeds, sampler, u):
        """A prompt of input vectors embeds [batch][n][d_model]."""
        w = self.spec.n_codebooks if self.qwen else 1
        out = sd_prefill_embeds(self.ctx, embeds, sampler, u, out_width=w)
        return out if self.qwen else out[:, 0]

    def step(self, tok, sampler, u):
        return sd_step(self.ctx, tok, sampler, u)

    def frame(self, codes_in, talker, cp, u):
        return sd_frame(self.ctx, codes_in, talker, cp, u)

    def force(self, codes):
        sd_set_forced_codes(self.ctx, codes)

    def set_ladder(self, ladder):
        sd_set_ladder(self.ctx, ladder)

    def decode_n(self, n, sampler, u_dev, out_dev):
        sd_decode_n(self.ctx, n, sampler, u_dev, out_dev)

    def logits(self):
        z = sd_get_logits(self.ctx, self.n_logits)
        if self.qwen:
            return z.reshape(self.spec.batch, MAX_CODEBOOKS, -1)
        return z.reshape(self.spec.batch, self.spec.vocab)

    def reset(self):
        sd_reset(self.ctx)

    def info(self) -> Info:
        return sd_get_info(self.ctx)
