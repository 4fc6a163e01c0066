"""Pins of the CPU oracle to what the formats and the mathematics fix.

Each pin is checked against something other than the oracle itself: bit-field
definitions of the element formats, exact rational brute force written here
with Python integers and Fractions, fixtures printed on the pages, library
routines (torch bf16 conversion, numpy integer matmul, scipy's logistic), and
invariants. The mutation tests at the end plant plausible mistakes in the
oracle (on the CPU) and check that at least one pin fails for each.
"""
import os
import re
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import oracle.qmv_oracle as O
import qmv_inputs as qi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Independent element-format definitions (bit fields, exact rationals)
# ---------------------------------------------------------------------------

def bf_e2m1(nib: int) -> Fraction:
    """E2M1: sign bit 3, 2-bit exponent (bias 1) in bits 2..1, 1-bit mantissa in bit 0."""
    s = (nib >> 3) & 1
    e = (nib >> 1) & 3
    m = nib & 1
    if e == 0:
        v = Fraction(m, 2)                        # subnormal: m * 2**(1-1) * 1/2
    else:
        v = Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return -v if s else v


def bf_e8m0(e: int) -> Fraction:
    return Fraction(2) ** (e - 127)


def bf_bf16(bits: int) -> Fraction:
    s = (bits >> 15) & 1
    ex = (bits >> 7) & 0xFF
    man = bits & 0x7F
    assert ex != 0xFF
    if ex == 0:
        v = Fraction(man, 128) * Fraction(2) ** (-126)
    else:
        v = (1 + Fraction(man, 128)) * Fraction(2) ** (ex - 127)
    return -v if s else v


def bf_fp16(bits: int) -> Fraction:
    s = (bits >> 15) & 1
    ex = (bits >> 10) & 0x1F
    man = bits & 0x3FF
    if ex == 0:
        v = Fraction(man, 1024) * Fraction(2) ** (-14)
    else:
        v = (1 + Fraction(man, 1024)) * Fraction(2) ** (ex - 15)
    return -v if s else v


def bf_e4m3(code: int):
    """E4M3: sign bit 7, 4-bit exponent (bias 7) in bits 6..3, 3-bit mantissa;
    exponent 0 subnormal; S.1111.111 NaN (returned as None); no infinity."""
    s = (code >> 7) & 1
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return None
    if e == 0:
        v = Fraction(m, 8) * Fraction(2) ** (-6)
    else:
        v = (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
    return -v if s else v


def fp16_round_bits(x) -> int:
    """Round an exact rational to fp16 (ties to even) by its definition; the
    bit pattern, with overflow to infinity."""
    v = Fraction(x)
    sign = 0x8000 if v < 0 else 0
    a = abs(v)
    if a == 0:
        return sign
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -14) - 10)
    n, rem = divmod(a, quantum)
    n = int(n)
    if rem > quantum / 2 or (rem == quantum / 2 and n % 2 == 1):
        n += 1
    r = n * quantum
    if r > 65504:                      # rounded past the largest finite fp16
        return sign | 0x7C00
    if r < Fraction(2) ** -14:
        return sign | int(r / Fraction(2) ** -24)
    ee = r.numerator.bit_length() - r.denominator.bit_length()
    if Fraction(2) ** ee > r:
        ee -= 1
    mant = int((r / Fraction(2) ** ee - 1) * 1024)
    return sign | ((ee + 15) << 10) | mant


def fp32_round(x) -> float:
    """Round an exact rational to the nearest fp32 (ties to even), no double rounding."""
    v = Fraction(x)
    if v == 0:
        return 0.0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    n, rem = divmod(a, quantum)
    n = int(n)
    if rem > quantum / 2 or (rem == quantum / 2 and n % 2 == 1):
        n += 1
    r = float(n * quantum)
    return -r if v < 0 else r


def codes_from_packed(fmt: str, row: bytes, K: int):
    """Canonical packed bytes of one row -> list of K codes, with Python ints."""
    out = []
    if fmt in ("mxfp4", "cb4"):
        for k in range(K):
            out.append((row[k // 2] >> (4 * (k % 2))) & 0xF)
    elif fmt == "cb2":
        for k in range(K):
            out.append((row[k // 4] >> (2 * (k % 4))) & 3)
    elif fmt == "cb3":
        for k in range(K):
            grp = k // 8
            word = int.from_bytes(row[3 * grp:3 * grp + 3], "little")
            out.append((word >> (3 * (k % 8))) & 7)
    return out


# ---------------------------------------------------------------------------
# Pins (functions, so the mutation tests can re-run them)
# ---------------------------------------------------------------------------

def pin_e2m1_table():
    got = O.e2m1_decode(np.arange(16))
    for n in range(16):
        assert Fraction(float(got[n])) == bf_e2m1(n), n
        # every value is exactly representable in fp16 and bf16
        assert float(np.float16(got[n])) == float(got[n])


def pin_e2m1_stated_values():
    # magnitudes {0,.5,1,1.5,2,3,4,6} for codes 0..7, negated for 8..15
    mags = sorted({abs(bf_e2m1(n)) for n in range(16)})
    assert mags == [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2),
                    Fraction(2), Fraction(3), Fraction(4), Fraction(6)]
    got = O.e2m1_decode(np.arange(16))
    assert all(got[8 + i] == -got[i] for i in range(8))


def pin_e8m0():
    e = np.arange(256)
    got = O.e8m0_decode(e)
    for i in range(1, 255):
        # fp32 with biased exponent field i and zero mantissa is exactly 2**(i-127)
        f = struct.unpack("<f", struct.pack("<I", i << 23))[0]
        assert got[i] == f, i
        assert Fraction(float(got[i])) == bf_e8m0(i)
    # e = 0: 2**-127, the fp32 subnormal with only mantissa bit 22 set
    assert got[0] == struct.unpack("<f", struct.pack("<I", 0x00400000))[0]
    assert np.isnan(got[255])


def pin_bf16_conversions():
    torch = pytest.importorskip("torch")
    g = qi.rng(11)
    bits = g.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    ex = (bits >> 7) & 0xFF
    bits = bits[ex != 0xFF]
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.bf16_bits_to_f64(bits), ref)
    # rounding: fp32 values round to bf16 exactly as torch does (single rounding)
    f = (g.standard_normal(4096) * np.exp2(g.integers(-20, 20, 4096))).astype(np.float32)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f64_to_bf16_bits(f.astype(np.float64)), want)
    # ties go to even: 1 + 2**-8 lies halfway between 1 and 1 + 2**-7
    assert O.f64_to_bf16_bits(np.array([1 + 2.0 ** -8]))[0] == 0x3F80
    assert O.f64_to_bf16_bits(np.array([1 + 3 * 2.0 ** -8]))[0] == 0x3F82
    assert O.f64_to_bf16_bits(np.array([-(1 + 2.0 ** -8)]))[0] == 0xBF80


def pin_packings():
    g = qi.rng(12)
    for fmt, bits in (("mxfp4", 4), ("cb4", 4), ("cb2", 2), ("cb3", 3)):
        c = qi.codes(g, (3, 64), bits)
        p = O.pack_codes(fmt, c)
        assert p.shape == (3, 64 * bits // 8)
        assert np.array_equal(O.unpack_codes(fmt, p), c)
        for r in range(3):
            assert codes_from_packed(fmt, bytes(p[r]), 64) == c[r].tolist()
    # MXFP4: a little-endian uint32 read at byte k/2 holds elements k..k+7 in nibbles 0..7
    c = qi.codes(g, (1, 64), 4)
    p = bytes(O.pack_codes("mxfp4", c)[0])
    for k in range(0, 64, 8):
        word = int.from_bytes(p[k // 2:k // 2 + 4], "little")
        assert [(word >> (4 * j)) & 0xF for j in range(8)] == c[0, k:k + 8].tolist()
    # CB3 fixture; a 16-weight half-block is one 48-bit window of 6 bytes
    with open(os.path.join(GOLDEN, "cb3_packing_example.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            lhs, rhs = line.split(":")
            codes = np.array([int(t) for t in lhs.split()], dtype=np.uint8)
            want = [int(t, 16) for t in rhs.split()]
            assert O.pack_cb3(codes[None])[0].tolist() == want
    c = qi.codes(g, (1, 64), 3)
    p = bytes(O.pack_cb3(c)[0])
    for h in range(4):
        window = int.from_bytes(p[6 * h:6 * h + 6], "little")
        assert [(window >> (3 * j)) & 7 for j in range(16)] == c[0, 16 * h:16 * h + 16].tolist()


def read_page_tables():
    tables = {}
    with open(os.path.join(GOLDEN, "rocmfpx_code_tables.txt")) as fh:
        for line in fh:
            if line.startswith("#") or not line.strip():
                continue
            name, *vals = line.split()
            tables[name] = [int(v) for v in vals]
    return tables


def pin_decode_contract():
    """Unpacked code -> value x half-block scale (e[i >= QK/2]) equals the dequantizer, bit-exact."""
    tables = read_page_tables()
    g = qi.rng(13)
    for fmt, name in (("cb3", "fp3"), ("cb2", "fp2")):
        lut = tables[name]
        bits = qi.FORMAT_BITS[fmt]
        c = qi.codes(g, (4, 64), bits)
        e = qi.e8m0(g, (4, 4))                      # 2 half-block scales per 32-block
        p = O.pack_codes(fmt, c)
        W = O.cb_dequant(O.unpack_codes(fmt, p), e, lut, 16)
        for r in range(4):
            codes_r = codes_from_packed(fmt, bytes(p[r]), 64)
            for i in range(64):
                blk, within = divmod(i, 32)
                half = 1 if within >= 16 else 0
                want = lut[codes_r[i]] * bf_e8m0(int(e[r, 2 * blk + half]))
                assert Fraction(float(W[r, i])) == want


def brute_mxfp4(packed_rows, scales, x_bits, K):
    out = []
    for r, row in enumerate(packed_rows):
        cs = codes_from_packed("mxfp4", bytes(row), K)
        acc = Fraction(0)
        for k in range(K):
            acc += bf_e2m1(cs[k]) * bf_e8m0(int(scales[r, k // 32])) * bf_bf16(int(x_bits[k]))
        out.append(acc)
    return out


def brute_cb(fmt, packed_rows, scales, lut, group, q, d_bits, K):
    out = []
    for r, row in enumerate(packed_rows):
        cs = codes_from_packed(fmt, bytes(row), K)
        acc = Fraction(0)
        for k in range(K):
            acc += (lut[cs[k]] * bf_e8m0(int(scales[r, k // group]))
                    * int(q[k]) * bf_fp16(int(d_bits[k // 32])))
        out.append(acc)
    return out


def pin_brute_force_mxfp4():
    g = qi.rng(14)
    for N, K in ((1, 32), (4, 64)):
        c = qi.codes(g, (N, K), 4)
        s = qi.e8m0(g, (N, K // 32))
        x = qi.normal_bf16_bits(g, (1, K))
        y = O.mxfp4_matvec(c, s, x)[0]
        want = brute_mxfp4(O.pack_nibbles(c), s, x[0], K)
        absum = O.mxfp4_abs_products(c, s, x)[0]
        for r in range(N):
            assert abs(Fraction(float(y[r])) - want[r]) <= Fraction(float(absum[r])) * Fraction(1, 10 ** 13)


def pin_brute_force_cb():
    g = qi.rng(15)
    for fmt, lut in (("cb2", qi.LUT_CB2), ("cb3", qi.LUT_CB3), ("cb4", qi.LUT_CB4)):
        group = qi.FORMAT_GROUP[fmt]
        for N, K in ((1, 32), (4, 64)):
            c = qi.codes(g, (N, K), qi.FORMAT_BITS[fmt])
            s = qi.e8m0(g, (N, K // group))
            q, d = O.q8_1_quantize(qi.normal_f32(g, (1, K)))
            y = O.cb_matvec(c, s, lut, group, q, d)[0]
            want = brute_cb(fmt, O.pack_codes(fmt, c), s, lut, group, q[0], d[0], K)
            absum = O.cb_abs_products(c, s, lut, group, q, d)[0]
            for r in range(N):
                assert abs(Fraction(float(y[r])) - want[r]) <= Fraction(float(absum[r])) * Fraction(1, 10 ** 13)


def pin_block_sums_exact():
    g = qi.rng(16)
    for fmt, lut in (("cb2", qi.LUT_CB2), ("cb3", qi.LUT_CB3), ("cb4", qi.LUT_CB4)):
        span = qi.FORMAT_GROUP[fmt]
        c = qi.codes(g, (4, 64), qi.FORMAT_BITS[fmt])
        q = g.integers(-127, 128, size=(2, 64)).astype(np.int8)
        got = O.cb_block_sums(c, lut, q, span)
        for v in range(2):
            for r in range(4):
                cs = codes_from_packed(fmt, bytes(O.pack_codes(fmt, c)[r]), 64)
                for h in range(64 // span):
                    want = sum(lut[cs[i]] * int(q[v, i]) for i in range(h * span, (h + 1) * span))
                    assert int(got[v, r, h]) == want


def pin_identity_special_case():
    """LUT = identity and all scales 2**0: the codebook matvec is an integer matmul."""
    g = qi.rng(17)
    for fmt in ("cb2", "cb3", "cb4"):
        bits = qi.FORMAT_BITS[fmt]
        group = qi.FORMAT_GROUP[fmt]
        lut = list(range(1 << bits))
        c = qi.codes(g, (8, 96), bits)
        s = np.full((8, 96 // group), 127, dtype=np.uint8)
        q = g.integers(-127, 128, size=(3, 96)).astype(np.int8)
        d = np.full((3, 3), 0x3C00, dtype=np.uint16)            # fp16 1.0
        want = q.astype(np.int64) @ c.astype(np.int64).T
        assert np.array_equal(O.cb_matvec(c, s, lut, group, q, d), want.astype(np.float64))
        sums = O.cb_block_sums(c, lut, q, group)
        blocks = np.einsum("vkb,nkb->vnk", q.astype(np.int64).reshape(3, -1, group),
                           c.astype(np.int64).reshape(8, -1, group))
        assert np.array_equal(sums, blocks)
    # MXFP4 with scale 2**0 and x = unit vectors picks single decoded weights
    c = qi.codes(g, (5, 64), 4)
    s = np.full((5, 2), 127, dtype=np.uint8)
    eye = np.zeros((64, 64), dtype=np.uint16)
    eye[np.arange(64), np.arange(64)] = 0x3F80                      # bf16 1.0
    got = O.mxfp4_matvec(c, s, eye)                                 # [64, 5]
    assert np.array_equal(got.T, O.e2m1_decode(c))


def pin_q8_quantizer():
    g = qi.rng(18)
    x = qi.normal_f32(g, (3, 256)) * np.float32(3.0)
    x[1, 32:64] = 0.0                                               # an all-zero block
    q, d = O.q8_1_quantize(x)
    qb = q.reshape(3, 8, 32).astype(np.int64)
    xb = x.reshape(3, 8, 32)
    assert np.all(np.abs(qb) <= 127)
    for t in range(3):
        for b in range(8):
            amax = float(np.max(np.abs(xb[t, b])))
            if amax == 0:
                assert np.all(qb[t, b] == 0) and d[t, b] == 0
                continue
            i = int(np.argmax(np.abs(xb[t, b])))
            assert abs(qb[t, b, i]) == 127
            dd = fp32_round(Fraction(amax) / 127)
            assert d[t, b] == np.float16(dd).view(np.uint16)
            inv = fp32_round(Fraction(1) / Fraction(dd))
            for k in range(32):
                v = Fraction(fp32_round(Fraction(float(xb[t, b, k])) * Fraction(inv)))
                mag = abs(v)
                r = int(mag) + (1 if mag - int(mag) >= Fraction(1, 2) else 0)
                r = min(r, 127)
                assert int(qb[t, b, k]) == (-r if v < 0 else r)
    # exact ties round away from zero: amax 127 gives d = 1, id = 1
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :6] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5]
    q, d = O.q8_1_quantize(x)
    assert q[0, :6].tolist() == [127, 3, -3, 1, -1, 2]
    assert d[0, 0] == 0x3C00


def pin_gather():
    g = qi.rng(19)
    E, N, K = 5, 8, 64
    c = qi.codes(g, (E, N, K), 4)
    s = qi.e8m0(g, (E, N, K // 32))
    x = qi.normal_bf16_bits(g, (2 * 3, K))
    ids = np.array([[4, 0, 7], [2, -1, 2]], dtype=np.int32)      # 7 and -1 are invalid
    for per_slot in (False, True):
        y = O.mxfp4_moe_gather(c, s, x, ids, per_slot)
        for t in range(2):
            for j in range(3):
                e = int(ids[t, j])
                v = t * 3 + j if per_slot else t
                if 0 <= e < E:
                    want = O.mxfp4_dequant(c[e], s[e]) @ O.bf16_bits_to_f64(x[v])
                    assert np.array_equal(y[t, j], want)
                else:
                    assert np.all(y[t, j] == 0)


def pin_silu():
    special = pytest.importorskip("scipy.special")
    z = np.linspace(-30, 30, 1201)
    assert np.allclose(O.silu(z), z * special.expit(z), rtol=1e-15, atol=1e-300)
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert np.allclose(O.silu(z) - O.silu(-z), z, rtol=1e-13, atol=1e-13)
    g = np.array([1.0, -2.0, 0.5])
    u = np.array([3.0, 0.25, -4.0])
    assert np.allclose(O.swiglu(g, u), u * g * special.expit(g), rtol=1e-15)


def pin_swiglu_tolerance():
    """The derivative bound used to propagate tolerances: max |silu'(z)| < 1.1,
    and the propagated bound covers actual perturbations of g and u."""
    special = pytest.importorskip("scipy.special")
    z = np.linspace(-40, 40, 200001)
    s = special.expit(z)
    assert np.max(np.abs(s * (1 + z * (1 - s)))) < 1.1
    g = qi.rng(20)
    gg, uu = g.standard_normal(1000) * 5, g.standard_normal(1000) * 5
    tg, tu = np.abs(g.standard_normal(1000)) * 0.1, np.abs(g.standard_normal(1000)) * 0.1
    for sg in (-1, 1):
        for su in (-1, 1):
            dh = np.abs(O.swiglu(gg + sg * tg, uu + su * tu) - O.swiglu(gg, uu))
            assert np.all(dh <= O.swiglu_tolerance(gg, uu, tg, tu) + 1e-12)


def pin_fused_gate_up():
    g = qi.rng(21)
    E, N, K = 4, 8, 64
    cg, cu = qi.codes(g, (E, N, K), 4), qi.codes(g, (E, N, K), 4)
    sg, su = qi.e8m0(g, (E, N, K // 32)), qi.e8m0(g, (E, N, K // 32))
    x = qi.normal_bf16_bits(g, (2, K))
    ids = np.array([[1, 3], [0, 9]], dtype=np.int32)
    h, gv, uv = O.moe_gate_up_swiglu(lambda e, t: O.mxfp4_matvec(cg[e], sg[e], x[t:t + 1])[0],
                                     lambda e, t: O.mxfp4_matvec(cu[e], su[e], x[t:t + 1])[0], E, ids, N)
    for t in range(2):
        for j in range(2):
            e = int(ids[t, j])
            if e >= E:
                assert np.all(h[t, j] == 0)
                continue
            xv = [bf_bf16(int(b)) for b in x[t]]
            for n in range(N):
                gx = sum(bf_e2m1(int(cg[e, n, k])) * bf_e8m0(int(sg[e, n, k // 32])) * xv[k] for k in range(K))
                ux = sum(bf_e2m1(int(cu[e, n, k])) * bf_e8m0(int(su[e, n, k // 32])) * xv[k] for k in range(K))
                assert abs(Fraction(float(gv[t, j, n])) - gx) <= abs(gx) * Fraction(1, 10 ** 12) + Fraction(1, 10 ** 300)
                assert abs(Fraction(float(uv[t, j, n])) - ux) <= abs(ux) * Fraction(1, 10 ** 12) + Fraction(1, 10 ** 300)
                want = float(gx) / (1 + np.exp(-float(gx))) * float(ux)
                assert abs(h[t, j, n] - want) <= 1e-12 * abs(want) + 1e-300


def pin_e4m3_table():
    torch = pytest.importorskip("torch")
    got = O.e4m3_decode(np.arange(256))
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        want = bf_e4m3(c)
        if want is None:
            assert np.isnan(got[c]) and np.isnan(lib[c]), c
            continue
        assert Fraction(float(got[c])) == want, c
        assert float(lib[c]) == float(got[c]), c
        # every finite E4M3 value is exact in fp16 (the device decodes to f16)
        assert float(np.float16(got[c])) == float(got[c]), c
    # OCP MX E4M3 landmarks: largest normal 448, smallest normal 2**-6,
    # smallest subnormal 2**-9, one, NaN only at S.1111.111
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0
    assert [c for c in range(256) if np.isnan(got[c])] == [0x7F, 0xFF]
    assert got[0x80] == 0 and np.signbit(got[0x80])


def pin_f16_rounding():
    g = qi.rng(16)
    vals = g.standard_normal(3000) * np.exp2(g.integers(-30, 18, 3000))
    got = O.f64_to_f16_bits(vals)
    for v, b in zip(vals, got):
        assert int(b) == fp16_round_bits(Fraction(float(v))), v
    for v, b in ((1 + 2.0 ** -11, 0x3C00), (1 + 3 * 2.0 ** -11, 0x3C02), (65504.0, 0x7BFF),
                 (65520.0, 0x7C00), (2.0 ** -25, 0x0000), (3 * 2.0 ** -26, 0x0001), (-(2.0 ** -24), 0x8001)):
        assert int(O.f64_to_f16_bits(np.array([v]))[0]) == b, v
    assert O.f16_bits_to_f64(np.array([0x3C00, 0x0001, 0xFBFF], dtype=np.uint16)).tolist() == [1.0, 2.0 ** -24, -65504.0]


def brute_mx(fmt, codes, scales, x_bits, x_dtype, K):
    elem = bf_e2m1 if fmt == "mxfp4" else bf_e4m3
    act = bf_bf16 if x_dtype == "bf16" else bf_fp16
    out = []
    for r in range(codes.shape[0]):
        acc = Fraction(0)
        for k in range(K):
            acc += elem(int(codes[r, k])) * bf_e8m0(int(scales[r, k // 32])) * act(int(x_bits[k]))
        out.append(acc)
    return out


def pin_brute_force_mx_variants():
    g = qi.rng(17)
    for fmt in ("mxfp8", "mxfp4"):
        for x_dtype in ("bf16", "f16"):
            for N, K in ((1, 32), (4, 64)):
                c = qi.format_codes(g, fmt, (N, K))
                s = qi.e8m0(g, (N, K // 32))
                x = qi.normal_bf16_bits(g, (1, K)) if x_dtype == "bf16" else qi.normal_f16_bits(g, (1, K))
                codes = O.unpack_codes(fmt, O.pack_codes(fmt, c))
                y = O.mx_matvec(fmt, codes, s, x, x_dtype)[0]
                absum = O.mx_abs_products(fmt, codes, s, x, x_dtype)[0]
                want = brute_mx(fmt, c, s, x[0], x_dtype, K)
                for r in range(N):
                    assert abs(Fraction(float(y[r])) - want[r]) <= Fraction(float(absum[r])) * Fraction(1, 10 ** 13)


def pin_mx_gather_f16():
    """mx_moe_gather: per-slot fp16 activations, an invalid id gives zeros, each
    valid slot equals the brute-force product of its expert and its vector."""
    g = qi.rng(18)
    E, N, K = 3, 2, 32
    c = qi.format_codes(g, "mxfp8", (E, N, K))
    s = qi.e8m0(g, (E, N, 1))
    ids = np.array([[2, 5], [0, 2]], dtype=np.int32)
    x = qi.normal_f16_bits(g, (4, K))
    y = O.mx_moe_gather("mxfp8", c, s, x, ids, True, "f16")
    assert np.all(y[0, 1] == 0)
    for t in range(2):
        for j in range(2):
            e = int(ids[t, j])
            if e >= E:
                continue
            want = brute_mx("mxfp8", c[e], s[e], x[t * 2 + j], "f16", K)
            for n in range(N):
                assert abs(Fraction(float(y[t, j, n])) - want[n]) <= abs(want[n]) * Fraction(1, 10 ** 12) + Fraction(1, 10 ** 300)


ALL_PINS = [pin_e2m1_table, pin_e2m1_stated_values, pin_e8m0, pin_bf16_conversions,
            pin_packings, pin_decode_contract, pin_brute_force_mxfp4, pin_brute_force_cb,
            pin_block_sums_exact, pin_identity_special_case, pin_q8_quantizer, pin_gather,
            pin_silu, pin_swiglu_tolerance, pin_fused_gate_up, pin_e4m3_table, pin_f16_rounding,
            pin_brute_force_mx_variants, pin_mx_gather_f16]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_page_tables_decode():
    """The page's fp3/fp2 tables, used as LUTs, decode codes to exactly those values."""
    tables = read_page_tables()
    assert tables["fp3"] == [0, 1, 2, 4, 0, -1, -2, -4]
    for name, bits in (("fp3", 3), ("fp2", 2)):
        c = np.arange(1 << bits, dtype=np.uint8)[None, :].repeat(1, 0)
        c = np.tile(c, (1, 32 // (1 << bits) * 2))[:, :32]
        s = np.full((1, 2), 127, dtype=np.uint8)
        W = O.cb_dequant(c, s, tables[name], 16)
        assert W[0].tolist() == [float(tables[name][int(k)]) for k in c[0]]


# ---------------------------------------------------------------------------
# Mutation tests: a planted oracle mistake must fail at least one pin
# ---------------------------------------------------------------------------

def _fails_some_pin(pins):
    for p in pins:
        try:
            p()
        except Exception:
            return True
    return False


def test_mutation_sign_bit_dropped(monkeypatch):
    real = O.e2m1_decode
    monkeypatch.setattr(O, "e2m1_decode", lambda c: np.abs(real(c)))
    assert _fails_some_pin([pin_e2m1_table, pin_brute_force_mxfp4])


def test_mutation_nibble_order(monkeypatch):
    monkeypatch.setattr(O, "pack_nibbles",
                        lambda c: (np.asarray(c)[..., 1::2] | (np.asarray(c)[..., 0::2] << 4)).astype(np.uint8))
    assert _fails_some_pin([pin_packings])


def test_mutation_e8m0_bias(monkeypatch):
    monkeypatch.setattr(O, "e8m0_decode", lambda e: np.ldexp(1.0, np.asarray(e).astype(np.int64) - 126))
    assert _fails_some_pin([pin_e8m0, pin_brute_force_mxfp4, pin_brute_force_cb])


def test_mutation_cb3_bit_order(monkeypatch):
    def bad_pack(codes):
        c = np.asarray(codes, dtype=np.uint32)
        lead = c.shape[:-1]
        gg = c.reshape(lead + (-1, 8))
        word = np.zeros(gg.shape[:-1], dtype=np.uint32)
        for j in range(8):
            word |= gg[..., j] << (21 - 3 * j)
        out = np.stack([(word >> (8 * b)) & 0xFF for b in range(3)], -1).astype(np.uint8)
        return out.reshape(lead + (-1,))
    monkeypatch.setattr(O, "pack_cb3", bad_pack)
    assert _fails_some_pin([pin_packings])


def test_mutation_q8_half_even(monkeypatch):
    real = O.q8_1_quantize

    def half_even(x):
        x = np.asarray(x, dtype=np.float32)
        lead, K = x.shape[:-1], x.shape[-1]
        xb = x.reshape(lead + (K // 32, 32))
        d = (np.max(np.abs(xb), -1) / np.float32(127)).astype(np.float32)
        with np.errstate(divide="ignore"):
            inv = np.where(d != 0, np.float32(1) / d, np.float32(0)).astype(np.float32)
        v = (xb * inv[..., None]).astype(np.float32)
        q = np.clip(np.rint(v), -127, 127).astype(np.int8).reshape(lead + (K,))
        return q, real(x)[1]
    monkeypatch.setattr(O, "q8_1_quantize", half_even)
    assert _fails_some_pin([pin_q8_quantizer])


def test_mutation_transposed_operand(monkeypatch):
    monkeypatch.setattr(O, "mxfp4_matvec",
                        lambda c, s, x: O.bf16_bits_to_f64(x) @ O.mxfp4_dequant(c, s))
    assert _fails_some_pin([pin_brute_force_mxfp4])


def test_mutation_mxfp4_group_16(monkeypatch):
    def bad(codes, scales):
        K = codes.shape[-1]
        gidx = np.minimum(np.arange(K) // 16, scales.shape[-1] - 1)
        return O.e2m1_decode(codes) * O.e8m0_decode(scales)[..., gidx]
    monkeypatch.setattr(O, "mxfp4_dequant", bad)
    assert _fails_some_pin([pin_brute_force_mxfp4])


def test_mutation_half_block_scale_ignored(monkeypatch):
    real = O.cb_dequant

    def bad(codes, scales, lut, group):
        s = np.asarray(scales).copy()
        if group == 16:
            s[..., 1::2] = s[..., 0::2]                # use the first half-block scale for both
        return real(codes, s, lut, group)
    monkeypatch.setattr(O, "cb_dequant", bad)
    assert _fails_some_pin([pin_decode_contract])


def test_mutation_block_sum_span(monkeypatch):
    real = O.cb_block_sums
    monkeypatch.setattr(O, "cb_block_sums",
                        lambda c, lut, q, span: real(c, lut, q, span) + (1 if span == 16 else 0))
    assert _fails_some_pin([pin_block_sums_exact, pin_brute_force_cb])


def test_mutation_fp16_d_ignored(monkeypatch):
    real = O.cb_matvec

    def bad(codes, scales, lut, group, q, d_bits):
        return real(codes, scales, lut, group, q, np.full_like(d_bits, 0x3C00))
    monkeypatch.setattr(O, "cb_matvec", bad)
    assert _fails_some_pin([pin_brute_force_cb])


def test_mutation_invalid_id_not_zeroed(monkeypatch):
    real = O.moe_gather

    def bad(matvec, n_experts, ids, per_slot, N):
        return real(matvec, n_experts, np.clip(ids, 0, n_experts - 1), per_slot, N)
    monkeypatch.setattr(O, "moe_gather", bad)
    assert _fails_some_pin([pin_gather])


# ---------------------------------------------------------------------------
# Router-weighted combine of per-slot outputs
# ---------------------------------------------------------------------------

def pin_combine():
    """Exact rational check of out[t] = sum of w * y over valid slots, on a
    small case with an invalid id (its slot must not contribute), plus the
    one-hot special case (it selects a slot)."""
    g = np.random.default_rng(5)
    ntok, top_k, N, E = 2, 3, 5, 4
    y = g.integers(-8, 9, size=(ntok, top_k, N)).astype(np.float64) / 4
    w = g.integers(1, 9, size=(ntok, top_k)).astype(np.float64) / 8
    ids = np.array([[0, 3, 1], [2, 7, 1]], dtype=np.int32)     # id 7 invalid
    got = O.moe_combine(y, w, ids, E)
    for t in range(ntok):
        for n in range(N):
            want = sum((Fraction(w[t, j]) * Fraction(y[t, j, n]) for j in range(top_k) if 0 <= ids[t, j] < E),
                       Fraction(0))
            assert Fraction(got[t, n]) == want
    onehot = np.zeros((ntok, top_k))
    onehot[:, 2] = 1.0
    assert np.array_equal(O.moe_combine(y, onehot, ids, E), y[:, 2])


def test_combine_pin():
    pin_combine()


def test_mutation_combine_ignores_invalid(monkeypatch):
    real = O.moe_combine

    def bad(y_slots, weights, ids, n_experts):
        return real(y_slots, weights, np.clip(ids, 0, n_experts - 1), n_experts)
    monkeypatch.setattr(O, "moe_combine", bad)
    assert _fails_some_pin([pin_combine])


def test_mutation_e4m3_bias(monkeypatch):
    real = O.e4m3_decode
    monkeypatch.setattr(O, "e4m3_decode", lambda c: real(c) * 2.0)     # bias 6 instead of 7
    assert _fails_some_pin([pin_e4m3_table, pin_brute_force_mx_variants])


def test_mutation_e4m3_subnormal_as_normal(monkeypatch):
    def bad(codes):
        c = np.asarray(codes).astype(np.int64)
        ex, man = (c >> 3) & 15, c & 7
        mag = np.ldexp(1.0 + man / 8.0, ex - 7)
        v = np.where((c >> 7) & 1, -mag, mag)
        return np.where((ex == 15) & (man == 7), np.nan, v)
    monkeypatch.setattr(O, "e4m3_decode", bad)
    assert _fails_some_pin([pin_e4m3_table])


def test_mutation_f16_read_as_bf16(monkeypatch):
    monkeypatch.setattr(O, "act_bits_to_f64", lambda b, d="bf16": O.bf16_bits_to_f64(b))
    assert _fails_some_pin([pin_brute_force_mx_variants, pin_mx_gather_f16])


def test_mutation_mxfp8_group_16(monkeypatch):
    def bad(codes, scales):
        K = codes.shape[-1]
        g = np.minimum(np.arange(K) // 16, scales.shape[-1] - 1)
        return O.e4m3_decode(codes) * O.e8m0_decode(scales)[..., g]
    monkeypatch.setattr(O, "mxfp8_dequant", bad)
    assert _fails_some_pin([pin_brute_force_mx_variants])


# ---------------------------------------------------------------------------
# Tolerance bases, gathered block sums and the MoE layer chain
# ---------------------------------------------------------------------------

def bf16_round_fraction(v: Fraction) -> int:
    """Bit pattern of the bf16 nearest to the exact rational v (ties to even),
    written from the bf16 bit layout (8 significant bits, exponent bias 127)."""
    if v == 0:
        return 0
    s = 0x8000 if v < 0 else 0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                       # subnormals share the smallest exponent
    ulp = Fraction(2) ** (e - 7)
    m, rem = divmod(a, ulp)
    m = int(m)
    if rem > ulp / 2 or (rem == ulp / 2 and m % 2 == 1):
        m += 1
    if e == -126 and m < 128:
        return s | m                       # subnormal (or rounds up into the normals: m == 128)
    if m == 256:
        m, e = 128, e + 1
    assert e <= 127, "bf16 overflow in a pin input"
    return s | ((e + 127) << 7) | (m - 128)


def pin_bf16_round_fraction_helper():
    """The helper above against torch's fp32 -> bf16 rounding on values that
    fp32 holds exactly (so no double rounding can occur)."""
    torch = pytest.importorskip("torch")
    g = qi.rng(40)
    f = (g.standard_normal(4000) * np.exp2(g.integers(-30, 30, 4000))).astype(np.float32)
    f[:4] = [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -130]   # ties and a subnormal
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    for x, w in zip(f.tolist(), want.tolist()):
        assert bf16_round_fraction(Fraction(x)) == w, x


def brute_abs(elem_values, scales_f, group, act_values):
    """sum_k |elem[k] * scale[k // group] * act[k]| for one row, exact."""
    return sum(abs(elem_values[k] * scales_f[k // group] * act_values[k]) for k in range(len(elem_values)))


def pin_abs_products():
    """The tolerance base of every float parity check, sum_k |w[n, k] * x[v, k]|,
    against an exact rational brute force over the decoded elements, for every
    format and activation type on 1x32 and 4x64 matrices with several vectors.
    Checked term by term: |w| and |x| are exact in float64, and a sum of 64
    non-negative float64 terms is within 64 * 2^-53 of the exact sum."""
    g = qi.rng(41)
    rel = Fraction(1, 10 ** 13)
    for N, K in ((1, 32), (4, 64)):
        V = 3
        for fmt in ("mxfp4", "mxfp8"):
            for x_dtype in ("bf16", "f16"):
                c = qi.format_codes(g, fmt, (N, K))
                s = qi.e8m0(g, (N, K // 32))
                x = qi.normal_bf16_bits(g, (V, K)) if x_dtype == "bf16" else qi.normal_f16_bits(g, (V, K))
                x[:, 0] ^= 0x8000                               # a negative activation in every vector
                elem = bf_e2m1 if fmt == "mxfp4" else bf_e4m3
                act = bf_bf16 if x_dtype == "bf16" else bf_fp16
                got_mx = O.mx_abs_products(fmt, c, s, x, x_dtype)
                got_fmt = (O.mxfp4_abs_products if fmt == "mxfp4" else O.mxfp8_abs_products)(c, s, x, x_dtype)
                assert got_mx.shape == (V, N) and np.array_equal(got_mx, got_fmt)
                for v in range(V):
                    av = [act(int(b)) for b in x[v]]
                    for n in range(N):
                        want = brute_abs([elem(int(k)) for k in c[n]], [bf_e8m0(int(e)) for e in s[n]], 32, av)
                        assert abs(Fraction(float(got_mx[v, n])) - want) <= want * rel
        for fmt, lut in (("cb2", qi.LUT_CB2), ("cb3", qi.LUT_CB3), ("cb4", qi.LUT_CB4)):
            group = qi.FORMAT_GROUP[fmt]
            c = qi.codes(g, (N, K), qi.FORMAT_BITS[fmt])
            s = qi.e8m0(g, (N, K // group))
            q, d = O.q8_1_quantize(qi.normal_f32(g, (V, K)))
            got = O.cb_abs_products(c, s, lut, group, q, d)
            assert got.shape == (V, N)
            for v in range(V):
                av = [int(q[v, k]) * bf_fp16(int(d[v, k // 32])) for k in range(K)]
                for n in range(N):
                    want = brute_abs([Fraction(lut[int(k)]) for k in c[n]],
                                     [bf_e8m0(int(e)) for e in s[n]], group, av)
                    assert abs(Fraction(float(got[v, n])) - want) <= want * rel


def pin_cb_moe_block_sums():
    """Gathered integer block sums and the gathered codebook matvec, shared and
    per-slot activations, with an invalid id: per (t, j) against Python-integer
    sums over the slot's expert and vector (x[t] shared, x[t * top_k + j]
    per-slot); an invalid slot is all zero."""
    g = qi.rng(42)
    E, N, K = 3, 4, 64
    ids = np.array([[2, 0], [1, 5], [0, 2]], dtype=np.int32)       # 5 is invalid
    ntok, top_k = ids.shape
    for fmt, lut in (("cb2", qi.LUT_CB2), ("cb3", qi.LUT_CB3), ("cb4", qi.LUT_CB4)):
        group = qi.FORMAT_GROUP[fmt]
        c = qi.codes(g, (E, N, K), qi.FORMAT_BITS[fmt])
        s = qi.e8m0(g, (E, N, K // group))
        q, d = O.q8_1_quantize(qi.normal_f32(g, (ntok * top_k, K)))
        for per_slot in (False, True):
            sums = O.cb_moe_block_sums(c, lut, group, q, ids, per_slot)
            y = O.cb_moe_gather(c, s, lut, group, q, d, ids, per_slot)
            assert sums.shape == (ntok, top_k, N, K // group)
            for t in range(ntok):
                for j in range(top_k):
                    e = int(ids[t, j])
                    v = t * top_k + j if per_slot else t
                    if not 0 <= e < E:
                        assert np.all(sums[t, j] == 0) and np.all(y[t, j] == 0)
                        continue
                    for n in range(N):
                        cs = codes_from_packed(fmt, bytes(O.pack_codes(fmt, c[e])[n]), K)
                        exact_y = Fraction(0)
                        for h in range(K // group):
                            want = sum(lut[cs[i]] * int(q[v, i]) for i in range(h * group, (h + 1) * group))
                            assert int(sums[t, j, n, h]) == want
                            exact_y += (want * bf_e8m0(int(s[e, n, h]))
                                        * bf_fp16(int(d[v, (h * group) // 32])))
                        absum = sum(abs(lut[cs[i]] * bf_e8m0(int(s[e, n, i // group])) * int(q[v, i])
                                        * bf_fp16(int(d[v, i // 32]))) for i in range(K))
                        assert abs(Fraction(float(y[t, j, n])) - exact_y) <= absum * Fraction(1, 10 ** 13)


def pin_mxfp4_moe_layer():
    """The MoE layer chain g, u -> h -> y on E = 3, N = K = 64 with an invalid
    id, stage by stage: g and u are the exact rational gate/up products rounded
    to bf16 (nearest even, by the bit-layout helper above); h is
    silu(g) * u of those bf16 values (Python float arithmetic, math.exp) and
    h_bits its bf16 rounding; y is the exact rational product of the down
    expert of each slot with that slot's own h_bits row."""
    import math
    g = qi.rng(43)
    E, N, K = 3, 64, 64
    mats = [(qi.codes(g, (E, N, K), 4), qi.e8m0(g, (E, N, K // 32))) for _ in range(3)]
    x = qi.normal_bf16_bits(g, (2, K))
    ids = np.array([[2, 0], [1, 4]], dtype=np.int32)                # 4 is invalid
    out = O.mxfp4_moe_layer(mats[0], mats[1], mats[2], x, ids)

    def exact_row(m, e, n, act_bits):
        cc, ss = m
        return sum(bf_e2m1(int(cc[e, n, k])) * bf_e8m0(int(ss[e, n, k // 32])) * bf_bf16(int(act_bits[k]))
                   for k in range(K))

    for t in range(2):
        for j in range(2):
            e = int(ids[t, j])
            row = out["h_rows_bits"][t * 2 + j]
            assert np.array_equal(row, out["h_bits"][t, j])
            if not 0 <= e < E:
                assert np.all(out["y"][t, j] == 0)
                continue
            for n in range(N):
                gb = bf16_round_fraction(exact_row(mats[0], e, n, x[t]))
                ub = bf16_round_fraction(exact_row(mats[1], e, n, x[t]))
                assert int(out["g_bits"][t, j, n]) == gb and int(out["u_bits"][t, j, n]) == ub
                gv, uv = float(bf_bf16(gb)), float(bf_bf16(ub))
                hv = gv / (1.0 + math.exp(-gv)) * uv
                assert abs(out["h"][t, j, n] - hv) <= 1e-15 * abs(hv) + 1e-300
                assert int(out["h_bits"][t, j, n]) == bf16_round_fraction(Fraction(float(out["h"][t, j, n])))
            for n in range(N):
                want = exact_row(mats[2], e, n, row)
                absum = sum(abs(bf_e2m1(int(mats[2][0][e, n, k])) * bf_e8m0(int(mats[2][1][e, n, k // 32]))
                                * bf_bf16(int(row[k]))) for k in range(K))
                assert abs(Fraction(float(out["y"][t, j, n])) - want) <= absum * Fraction(1, 10 ** 13)


NEW_PINS = [pin_bf16_round_fraction_helper, pin_abs_products, pin_cb_moe_block_sums, pin_mxfp4_moe_layer]


@pytest.mark.parametrize("pin", NEW_PINS, ids=lambda f: f.__name__)
def test_pin_chain(pin):
    pin()


def test_mutation_abs_dropped_from_x(monkeypatch):
    def bad(codes, scales, x_bits, x_dtype="bf16"):
        return O.act_bits_to_f64(x_bits, x_dtype) @ np.abs(O.mxfp4_dequant(codes, scales)).T
    monkeypatch.setattr(O, "mxfp4_abs_products", bad)
    assert _fails_some_pin([pin_abs_products])


def test_mutation_abs_of_sum(monkeypatch):
    def bad(codes, scales, lut, group, q, d_bits):
        return np.abs(O.cb_matvec(codes, scales, lut, group, q, d_bits))
    monkeypatch.setattr(O, "cb_abs_products", bad)
    assert _fails_some_pin([pin_abs_products])


def test_mutation_abs_d_not_repeated(monkeypatch):
    def bad(codes, scales, lut, group, q, d_bits):
        W = np.abs(O.cb_dequant(codes, scales, lut, group))
        d = O.f16_bits_to_f64(d_bits)
        K = codes.shape[-1]
        xq = np.abs(np.asarray(q).astype(np.float64) * np.tile(d, K // 32))     # block b's d on the wrong weights
        return xq @ W.T
    monkeypatch.setattr(O, "cb_abs_products", bad)
    assert _fails_some_pin([pin_abs_products])


def test_mutation_mxfp8_abs_scale_dropped(monkeypatch):
    def bad(codes, scales, x_bits, x_dtype="bf16"):
        W = np.abs(O.e4m3_decode(codes))
        return np.abs(O.act_bits_to_f64(x_bits, x_dtype)) @ W.T
    monkeypatch.setattr(O, "mxfp8_abs_products", bad)
    assert _fails_some_pin([pin_abs_products])


def test_mutation_block_sums_slot_index(monkeypatch):
    real = O.gather_vectors

    def bad(ids, per_slot):
        ntok, top_k = ids.shape
        return [[(j * ntok + t) if per_slot else t for j in range(top_k)] for t in range(ntok)]
    monkeypatch.setattr(O, "gather_vectors", bad)
    assert real is not bad
    assert _fails_some_pin([pin_cb_moe_block_sums])


def test_mutation_layer_h_unrounded(monkeypatch):
    real = O.f64_to_bf16_bits
    calls = {"n": 0}

    def bad(v):
        calls["n"] += 1
        if calls["n"] % 3 == 0:                     # the third rounding of each layer is h's
            return (np.asarray(v, dtype=np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        return real(v)
    monkeypatch.setattr(O, "f64_to_bf16_bits", bad)
    assert _fails_some_pin([pin_mxfp4_moe_layer])


def test_mutation_layer_down_shared_x(monkeypatch):
    real = O.mxfp4_moe_gather

    def bad(codes, scales, x_bits, ids, per_slot, x_dtype="bf16"):
        if per_slot:
            ntok, top_k = ids.shape
            x_bits = x_bits[::top_k]                  # one h row per token instead of per slot
        return real(codes, scales, x_bits, ids, False, x_dtype)
    monkeypatch.setattr(O, "mxfp4_moe_gather", bad)
    assert _fails_some_pin([pin_mxfp4_moe_layer])


def test_every_oracle_function_is_pinned():
    """Each public function of the oracle is exercised by some pin: named in
    a pin's source, or called (transitively) by a function a pin names."""
    import inspect
    pins = ALL_PINS + NEW_PINS + [pin_combine, test_page_tables_decode]
    text = "\n".join(inspect.getsource(p) for p in pins)
    funcs = {n: f for n, f in vars(O).items()
             if inspect.isfunction(f) and not n.startswith("_") and f.__module__ == O.__name__}
    covered = {n for n in funcs if f"O.{n}(" in text}
    frontier = list(covered)
    while frontier:
        body = inspect.getsource(funcs[frontier.pop()])
        for n in funcs:
            if n not in covered and re.search(rf"\b{n}\(", body):
                covered.add(n)
                frontier.append(n)
    assert sorted(set(funcs) - covered) == []
