"""The canonical block layouts, written out by hand for building test blocks.

Byte layouts (little-endian), one block each:
  Q8_0  f16 d | int8 q[32]                                   34 B
  Q4_0  f16 d | u8 qs[16]  (element k in byte k/2, low nibble for even k)   18 B
  Q4_K  f16 d | f16 dmin | 12 B: sixteen 6-bit fields sc_0..7, m_0..7, LSB-first |
        u8 qs[128] (4-bit codes as Q4_0)                     144 B
  Q6_K  u8 ql[128] (low 4 bits, as Q4_0) | u8 qh[64] (high 2 bits of element k in
        byte k/4 at bits 2*(k%4)) | int8 sc[16] | f16 d       210 B
  Q5_K  f16 d | f16 dmin | 12 B scales as Q4_K | u8 qh[32] (fifth bit of element k
        in byte k/8 at bit k%8) | u8 qs[128] (low 4 bits, as Q4_0)   176 B
Used by tests to build blocks from chosen (d, q, ...) independently of the
oracle's own packing code.
"""
import struct

import numpy as np


def f16_bits(x: float) -> int:
    return int(np.array([x], np.float16).view(np.uint16)[0])


def nibbles(q) -> bytes:
    out = bytearray(len(q) // 2)
    for k, v in enumerate(q):
        assert 0 <= v < 16
        out[k // 2] |= (v << 4) if k % 2 else v
    return bytes(out)


def pack_q8_0(d: float, q) -> bytes:
    assert len(q) == 32
    return struct.pack("<H", f16_bits(d)) + bytes((v & 0xFF) for v in q)


def pack_q4_0(d: float, q) -> bytes:
    assert len(q) == 32
    return struct.pack("<H", f16_bits(d)) + nibbles(q)


def pack_q4_k(d: float, dmin: float, sc, m, q) -> bytes:
    assert len(sc) == 8 and len(m) == 8 and len(q) == 256
    bits = 0
    for f, v in enumerate(list(sc) + list(m)):
        assert 0 <= v < 64
        bits |= v << (6 * f)
    return struct.pack("<HH", f16_bits(d), f16_bits(dmin)) + bits.to_bytes(12, "little") + nibbles(q)


def pack_q6_k(d: float, sc, q) -> bytes:
    assert len(sc) == 16 and len(q) == 256
    ql = nibbles([v & 15 for v in q])
    qh = bytearray(64)
    for k, v in enumerate(q):
        assert 0 <= v < 64
        qh[k // 4] |= (v >> 4) << (2 * (k % 4))
    return ql + bytes(qh) + bytes((s & 0xFF) for s in sc) + struct.pack("<H", f16_bits(d))


def pack_q5_k(d: float, dmin: float, sc, m, q) -> bytes:
    assert len(sc) == 8 and len(m) == 8 and len(q) == 256
    bits = 0
    for f, v in enumerate(list(sc) + list(m)):
        assert 0 <= v < 64
        bits |= v << (6 * f)
    qh = bytearray(32)
    for k, v in enumerate(q):
        assert 0 <= v < 32
        qh[k // 8] |= (v >> 4) << (k % 8)
    return (struct.pack("<HH", f16_bits(d), f16_bits(dmin)) + bits.to_bytes(12, "little") + bytes(qh)
            + nibbles([v & 15 for v in q]))
