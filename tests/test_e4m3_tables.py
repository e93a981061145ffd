"""The e4m3 lookup constants of the kind::f8f6f4 GEMM (csrc/qmm_e4m3.cuh),
checked on the CPU against an independent e4m3 decoder.

The weights-in-N GEMM's e4m3 form feeds the tensor cores small integers that
e4m3 holds exactly: the offset-binary weight nibbles u = q + 8 in [0, 15], and
the planes 16 * floor(a / 16) and a mod 16 of each int8 activation code a. The
device builds those bytes with byte permutes (prmt) over constant tables. This
test reads the tables from the header, emulates prmt (default mode: selector
nibble bits 0-2 pick one of eight bytes, bit 3 replicates that byte's sign),
and checks every nibble value and every int8 code through the same operation
sequence as the kernel: a wrong table byte, a swapped table or a selector
mistake turns it red.
"""

import os
import re

import numpy as np

HDR = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "bit_group_quantized_qmm_gb300", "csrc",
                   "qmm_e4m3.cuh")


def tables():
    src = open(HDR).read()
    return {k: int(v, 16) for k, v in re.findall(r"\b(k[UPN]\d)\s*=\s*(0x[0-9A-Fa-f]+)u", src)}


def prmt(a, b, c):
    src = [(a >> (8 * i)) & 0xFF for i in range(4)] + [(b >> (8 * i)) & 0xFF for i in range(4)]
    out = 0
    for i in range(4):
        s = (c >> (4 * i)) & 0xF
        byte = src[s & 7]
        if s & 8:
            byte = 0xFF if byte & 0x80 else 0x00
        out |= byte << (8 * i)
    return out


def e4m3_value(b):
    """The OCP e4m3 value of a byte: sign, 4 exponent bits (bias 7), 3 mantissa bits."""
    s = -1.0 if b & 0x80 else 1.0
    e, m = (b >> 3) & 15, b & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def u4(t, s, sx):
    return prmt(t["kU0"], t["kU1"], s) | prmt(t["kU2"], t["kU3"], sx)


def test_tables_present():
    t = tables()
    assert set(t) == {"kU0", "kU1", "kU2", "kU3", "kP0", "kP1", "kN0", "kN1"}


def test_weight_nibbles():
    """expand_word_e4m3: bytes [slot 0..3] from w, [slot 4..7] from w >> 16 -> e4m3(u)."""
    t = tables()
    rng = np.random.default_rng(3)
    words = [int(w) for w in rng.integers(0, 2**32, size=4000, dtype=np.uint64)]
    words += [sum(u << (4 * i) for i in range(8)) for u in range(16)]   # every nibble value in every slot
    for w in words:
        x = w ^ 0x88888888
        a = u4(t, w & 0xFFFF, x & 0xFFFF)
        b = u4(t, (w >> 16) & 0xFFFF, (x >> 16) & 0xFFFF)
        for i in range(4):
            assert e4m3_value((a >> (8 * i)) & 0xFF) == (w >> (4 * i)) & 15
            assert e4m3_value((b >> (8 * i)) & 0xFF) == (w >> (16 + 4 * i)) & 15


def split_codes(t, c):
    """split_codes: four int8 codes (bytes of c) -> hi plane e4m3(16 floor(a/16)), lo plane e4m3(a mod 16)."""
    def nibble_sel(v):
        tt = v & 0x0F0F0F0F
        return prmt((tt | (tt >> 4)) & 0xFFFFFFFF, 0, 0x0020) & 0xFFFF
    sl = nibble_sel(c)
    lo = u4(t, sl, sl ^ 0x8888)
    sh = nibble_sel(c >> 4)
    s7 = sh & 0x7777
    hi = prmt(prmt(t["kP0"], t["kP1"], s7), prmt(t["kN0"], t["kN1"], s7), ((sh >> 1) & 0x4444) | 0x3210)
    return hi, lo


def test_activation_planes_every_code():
    t = tables()
    codes = list(range(-128, 128))
    for base in range(0, 256, 4):
        four = [codes[(base + i) % 256] for i in range(4)]
        c = sum((v & 0xFF) << (8 * i) for i, v in enumerate(four))
        hi, lo = split_codes(t, c)
        for i, a in enumerate(four):
            h, l = e4m3_value((hi >> (8 * i)) & 0xFF), e4m3_value((lo >> (8 * i)) & 0xFF)
            assert h == 16 * (a >> 4) and l == (a & 15), (a, h, l)
            assert h + l == a


def test_plane_k_order_matches_weight_slots():
    """The kernel gathers the codes of an 8-k block as k = 0, 2, 4, 6 then 1, 3, 5, 7 (the nibble slot order
    of a packed word) from four fp16 pairs offset by 1536: check the byte gathering."""
    import struct
    rng = np.random.default_rng(4)
    for _ in range(500):
        a = [int(v) for v in rng.integers(-127, 128, size=8)]
        w4 = []
        for i in range(4):
            lo = struct.unpack("<H", struct.pack("<e", float(a[2 * i]) + 1536.0))[0]
            hi = struct.unpack("<H", struct.pack("<e", float(a[2 * i + 1]) + 1536.0))[0]
            w4.append(lo | (hi << 16))
        x, y = prmt(w4[0], w4[1], 0x6240), prmt(w4[2], w4[3], 0x6240)
        ca, cb = prmt(x, y, 0x5410), prmt(x, y, 0x7632)
        got = [((ca >> (8 * i)) & 0xFF) for i in range(4)] + [((cb >> (8 * i)) & 0xFF) for i in range(4)]
        got = [g - 256 if g > 127 else g for g in got]
        assert got == [a[k] for k in (0, 2, 4, 6, 1, 3, 5, 7)]


def test_a_planted_table_error_is_caught():
    """Control: one wrong byte in a table fails the weight check."""
    t = dict(tables())
    t["kU1"] ^= 0x00000100   # entry u = 5 off by one mantissa step
    w = sum(5 << (4 * i) for i in range(8))
    x = w ^ 0x88888888
    a = u4(t, w & 0xFFFF, x & 0xFFFF)
    assert e4m3_value(a & 0xFF) != 5
