"""Flat little-endian weight blob shared by the two readers.

Layout::

    0    u32 magic 0x31574453 ("SDW1")      4  u32 version (1)
    8    u32 n_tensors                      12 u32 table offset (= 16 + 128)
    16   config echo: 32 x 4-byte fields (int32 unless noted)
         [arch, n_layer, d_model, n_head, n_kv_head, head_dim, d_ff, vocab,
          max_ctx, batch, quant, rope_theta (f32), norm_eps (f32), cp_layer,
          cp_d_model, cp_n_head, cp_n_kv_head, cp_head_dim, cp_d_ff, cp_vocab,
          n_codebooks, cp_max_ctx, 0 ...]
    144  tensor table, n_tensors x 96 bytes:
         char name[64] (NUL padded), u32 kind, u32 rows, u32 cols, u32 0,
         u64 offset (from blob start), u64 nbytes
    ...  tensor data, each tensor 256-byte aligned

Tensor kinds and canonical storage:

    0 F32    rows x cols fp32, row-major
    1 Q8_0   rows x (cols/32) blocks of 34 bytes: fp16 d, 32 x int8
    2 Q4_0   rows x (cols/32) blocks of 18 bytes: fp16 d, 16 bytes of nibbles
             (byte j: low nibble = element j, high nibble = element j+16)
    3 A8G64  rows x cols uint8 codes, then rows x cols/64 fp16 scales, then
             rows x cols/64 fp16 biases
    4 Q5_0   rows x (cols/32) blocks of 22 bytes: fp16 d, u32 of fifth bits
             (bit j = element j), 16 bytes of low nibbles as in Q4_0
    5 A4G32  rows x cols/2 bytes of 4-bit codes (byte i: low nibble = element
             2i, high nibble = element 2i+1), then rows x cols/32 fp16 scales,
             then rows x cols/32 fp16 biases
    6 A4G64  as A4G32 with groups of 64
"""

from __future__ import annotations

import struct

import numpy as np

MAGIC = 0x31574453
VERSION = 1
CONFIG_FIELDS = 32
HEADER_BYTES = 16 + 4 * CONFIG_FIELDS
ENTRY_BYTES = 96
ALIGN = 256

KIND_F32 = 0
KIND_Q8_0 = 1
KIND_Q4_0 = 2
KIND_A8G64 = 3
KIND_Q5_0 = 4
KIND_A4G32 = 5
KIND_A4G64 = 6
AFFINE_KINDS = (KIND_A8G64, KIND_A4G32, KIND_A4G64)


def config_words(m) -> bytes:
    ints = [m.arch, m.n_layer, m.d_model, m.n_head, m.n_kv_head, m.head_dim, m.d_ff, m.vocab,
            m.max_ctx, m.batch, m.quant]
    tail = [m.cp_layer, m.cp_d_model, m.cp_n_head, m.cp_n_kv_head, m.cp_head_dim, m.cp_d_ff,
            m.cp_vocab, m.n_codebooks, m.cp_max_ctx]
    raw = struct.pack("<11i2f9i", *ints, float(m.rope_theta), float(m.norm_eps), *tail)
    return raw + b"\0" * (4 * CONFIG_FIELDS - len(raw))


def with_batch(blob: np.ndarray, batch: int) -> np.ndarray:
    """A copy of ``blob`` whose header names ``batch`` rows (the tensors do not
    depend on the batch)."""
    magic, _ver, _n, _toff = struct.unpack_from("<4I", blob, 0)
    assert magic == MAGIC
    out = np.array(blob, dtype=np.uint8, copy=True)
    struct.pack_into("<i", out, 16 + 4 * 9, int(batch))
    return out


def _payload(kind: int, data) -> bytes:
    if kind in AFFINE_KINDS:
        q, s, b = data
        return (np.ascontiguousarray(q, np.uint8).tobytes() + np.ascontiguousarray(s, np.float16).tobytes()
                + np.ascontiguousarray(b, np.float16).tobytes())
    if kind == KIND_F32:
        return np.ascontiguousarray(data, np.float32).tobytes()
    return np.ascontiguousarray(data, np.uint8).tobytes()


def write_blob(m, entries) -> np.ndarray:
    """entries: list of (name, kind, rows, cols, data).  Returns a uint8 array."""
    n = len(entries)
    table_off = HEADER_BYTES
    data_off = table_off + n * ENTRY_BYTES
    data_off = (data_off + ALIGN - 1) // ALIGN * ALIGN
    payloads = [_payload(kind, data) for (_, kind, _, _, data) in entries]
    offsets = []
    cur = data_off
    for p in payloads:
        offsets.append(cur)
        cur = (cur + len(p) + ALIGN - 1) // ALIGN * ALIGN
    out = np.zeros(cur, dtype=np.uint8)
    hdr = struct.pack("<4I", MAGIC, VERSION, n, table_off) + config_words(m)
    out[:HEADER_BYTES] = np.frombuffer(hdr, np.uint8)
    for i, ((name, kind, rows, cols, _), p, off) in enumerate(zip(entries, payloads, offsets)):
        nb = name.encode("ascii")
        assert len(nb) < 64, name
        ent = nb + b"\0" * (64 - len(nb)) + struct.pack("<4I2Q", kind, rows, cols, 0, off, len(p))
        o = table_off + i * ENTRY_BYTES
        out[o:o + ENTRY_BYTES] = np.frombuffer(ent, np.uint8)
        out[off:off + len(p)] = np.frombuffer(p, np.uint8)
    return out


def read_table(blob: np.ndarray) -> dict:
    """Parse the tensor table (used by tests and tooling, not by either implementation)."""
    b = np.asarray(blob, np.uint8)
    magic, ver, n, toff = struct.unpack_from("<4I", b, 0)
    assert magic == MAGIC and ver == VERSION
    out = {}
    for i in range(n):
        o = toff + i * ENTRY_BYTES
        name = bytes(b[o:o + 64]).split(b"\0", 1)[0].decode()
        kind, rows, cols, _, off, nbytes = struct.unpack_from("<4I2Q", b, o + 64)
        out[name] = (kind, rows, cols, off, nbytes)
    return out
