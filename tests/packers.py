"""Test-side block packers: fields -> bytes.

Written independently of the oracle (which goes bytes -> weights), from the
same reading of the layouts, so that a round trip through the oracle checks
every field's bit position.  Layout readings (GGML K-quant super-blocks of
256 weights; fp16 fields little-endian):

  Q4_K (144 B): d @0, dmin @2, scales[12] @4, qs[128] @16; element 64c+l is
                the low nibble of qs[32c+l], element 64c+32+l its high nibble.
  Q5_K (176 B): d @0, dmin @2, scales[12] @4, qh[32] @16, qs[128] @48; the
                fifth bit of element 64c+l is bit 2c of qh[l], of element
                64c+32+l bit 2c+1 of qh[l].
  Q6_K (210 B): ql[128] @0, qh[64] @128, int8 scales[16] @192, d @208.
  NVFP4:        element 2i in the low nibble of byte i, 2i+1 in the high one.
  FP8:          e4m3 codes [M][K], bf16 scales [ceil(M/128)][K/128] (one per
                128 x 128 block), weight = e4m3 * scale.
"""
from __future__ import annotations

import numpy as np


def f16_bytes(v) -> np.ndarray:
    return np.array([v], dtype=np.float16).view(np.uint8)


def pack_scales_q4k(sc, m) -> np.ndarray:
    """Eight 6-bit scales and eight 6-bit mins -> 12 bytes."""
    sc = [int(v) for v in sc]
    m = [int(v) for v in m]
    assert all(0 <= v < 64 for v in sc + m)
    out = np.zeros(12, dtype=np.uint8)
    for s in range(4):
        out[s] = (sc[s] & 63) | ((sc[s + 4] >> 4) << 6)
        out[s + 4] = (m[s] & 63) | ((m[s + 4] >> 4) << 6)
        out[s + 8] = (sc[s + 4] & 15) | ((m[s + 4] & 15) << 4)
    return out


def pack_q4k_block(d, dmin, sc, m, q) -> np.ndarray:
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= 0 and q.max() < 16
    blk = np.zeros(144, dtype=np.uint8)
    blk[0:2] = f16_bytes(d)
    blk[2:4] = f16_bytes(dmin)
    blk[4:16] = pack_scales_q4k(sc, m)
    for c in range(4):
        for l in range(32):
            blk[16 + 32 * c + l] = q[64 * c + l] | (q[64 * c + 32 + l] << 4)
    return blk


def pack_q5k_block(d, dmin, sc, m, q5) -> np.ndarray:
    q5 = np.asarray(q5, dtype=np.int64)
    assert q5.shape == (256,) and q5.min() >= 0 and q5.max() < 32
    blk = np.zeros(176, dtype=np.uint8)
    blk[0:2] = f16_bytes(d)
    blk[2:4] = f16_bytes(dmin)
    blk[4:16] = pack_scales_q4k(sc, m)
    qh = np.zeros(32, dtype=np.int64)
    for c in range(4):
        for l in range(32):
            lo, hi = q5[64 * c + l], q5[64 * c + 32 + l]
            blk[48 + 32 * c + l] = (lo & 15) | ((hi & 15) << 4)
            qh[l] |= ((lo >> 4) & 1) << (2 * c)
            qh[l] |= ((hi >> 4) & 1) << (2 * c + 1)
    blk[16:48] = qh.astype(np.uint8)
    return blk


def pack_q6k_block(d, scales16, q) -> np.ndarray:
    """q: 256 signed values in [-32, 31]; scales16: 16 int8 values."""
    q = np.asarray(q, dtype=np.int64)
    assert q.shape == (256,) and q.min() >= -32 and q.max() <= 31
    v = q + 32
    blk = np.zeros(210, dtype=np.uint8)
    ql = np.zeros(128, dtype=np.int64)
    qh = np.zeros(64, dtype=np.int64)
    for h in range(2):
        for s in range(4):
            for l in range(32):
                e = v[128 * h + 32 * s + l]
                idx = 64 * h + 32 * (s & 1) + l
                ql[idx] |= (e & 15) << (4 * (s >> 1))
                qh[32 * h + l] |= (e >> 4) << (2 * s)
    blk[0:128] = ql.astype(np.uint8)
    blk[128:192] = qh.astype(np.uint8)
    blk[192:208] = np.asarray(scales16, dtype=np.int8).view(np.uint8)
    blk[208:210] = f16_bytes(d)
    return blk


def pack_nvfp4_row(codes) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.int64)
    assert codes.size % 2 == 0 and codes.min() >= 0 and codes.max() < 16
    return (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)


def e4m3_code(v: float) -> int:
    """The e4m3 ("fn": bias 7, no infinities) code of a value it represents
    exactly, by search over the finite codes written from the definition."""
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        val = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        if (-val if s else val) == v and not (v == 0 and s):
            return c
    raise ValueError(f"{v} is not an e4m3 value")


def bf16_bits(v: float) -> int:
    """bf16 bits of a value whose float32 form has a zero low half."""
    b = int(np.array([v], dtype=np.float32).view(np.uint32)[0])
    assert b & 0xFFFF == 0, v
    return b >> 16
