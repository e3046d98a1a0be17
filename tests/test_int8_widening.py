"""The INT8 cache's widening to f16 in the decode kernel, checked on the host for every
byte: with u = byte ^ 0x80 (= v + 128 for the signed value v), the f16 whose bits are
0x6400 | u is 1024 + u, and subtracting 1152 (f16 bits 0x6480) leaves v exactly.  The
byte permutes place byte i of a word under the high byte 0x64 in the order the kernel's
selectors 0x4140 and 0x4342 give: (byte 0, byte 1) and (byte 2, byte 3)."""
import numpy as np


def prmt(a: int, b: int, sel: int) -> int:
    """PTX prmt.b32 (default mode): result byte i = byte (sel >> 4i) & 7 of (b:a)."""
    src = a.to_bytes(4, "little") + b.to_bytes(4, "little")
    return int.from_bytes(bytes(src[(sel >> (4 * i)) & 7] for i in range(4)), "little")


def widen(word: int):
    u = word ^ 0x80808080
    lo, hi = prmt(u, 0x64646464, 0x4140), prmt(u, 0x64646464, 0x4342)
    out = []
    for w in (lo, hi):
        h = np.array([w & 0xFFFF, w >> 16], np.uint16).view(np.float16)
        out += list((h - np.float16(1152.0)).astype(np.float64))  # f16 arithmetic, exact
    return out


def test_every_byte_in_every_position():
    values = np.arange(256, dtype=np.uint8).view(np.int8).astype(np.float64)
    for pos in range(4):
        for b in range(256):
            word = (b << (8 * pos)) | (0x7F << (8 * ((pos + 1) % 4)))
            got = widen(word)
            assert got[pos] == values[b], (pos, b, got)


def test_offset_constant_is_1152():
    assert np.array([0x6480], np.uint16).view(np.float16)[0] == 1152.0
    assert np.array([0x6400], np.uint16).view(np.float16)[0] == 1024.0
    # unit spacing on [1024, 2048): 0x64ff is 1024 + 255
    assert np.array([0x64FF], np.uint16).view(np.float16)[0] == 1279.0
