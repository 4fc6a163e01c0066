"""Plain double-precision CPU oracle for the block-quantized decode matvec.

TEST INFRASTRUCTURE -- not part of the product. Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import it. It shares no code with the CUDA library in
``bit_quantized_moe_gb300`` and imports nothing from it; the library never
imports this module.

Every weight is decoded to a float64 and every dot product is taken in
float64. There is no blocking, fusion or reordering beyond what the formats
define: each function decodes, multiplies and sums in the plain order a reader
can check against the definitions cited in its docstring. Arrays are numpy;
matrix-vector products are numpy's float64 / int64 reductions.

Sources (web pages, cited by title and section):
  [mlxcel-2178]  "perf(rocm): add an mxfp4 arm to the warp-shared gather_qmv
                 kernel for gpt-oss decode" (mlxcel issue #2178)
  [lucebox-21]   "perf(ggml/hip): optimize ROCMFPX fp3/fp2 MMVQ on RDNA
                 (perm-LUT + VDR=4 + fp2)" (lucebox-hub PR #21)
  [lucebox-19]   "perf(ggml/hip): speed up fp3 ROCMFPX matvec (Q3_0_ROCMFPX)
                 on RDNA" (lucebox-hub PR #19)
  [geo-31]       "DS4 H200: rocmfp2_mix MoE matvec 3.31x + ROCmFP4 dense matvec
                 1.53x (+42.6% decode)" (geo-lucebox PR #31)
  [OCP-MX]       the OCP Microscaling Formats (MX) v1.0 specification, for the
                 E4M3 element of MXFP8, which the pages name but do not define

Readings taken where the pages are silent:
  * E2M1 value table {0,.5,1,1.5,2,3,4,6} with the sign in bit 3 and E8M0
    scale 2**(e-127), e = 255 -> NaN (OCP MX convention).
  * MXFP8: E4M3 elements (bias 7, subnormals, S.1111.111 = NaN, no
    infinities) with one E8M0 scale per 32 weights, one code per byte; the
    f16-activation variants take fp16 activations and store fp16 outputs.
  * q8_1: per 32-block, d = amax/127 in fp32, codes round(x/d) half away from
    zero, clamped to [-127, 127]; d stored as fp16 (RNE). The block-sum field
    of q8_1 is not stored because no dot product here reads it.
  * Canonical byte packings: MXFP4 and CB4 low nibble first; CB2 code j of a
    byte at bits [2j, 2j+2); CB3 code j of a 3-byte group at bits [3j, 3j+3)
    of the little-endian 24-bit word.
  * MoE layer: plain SwiGLU h = silu(g) * u between gate/up and down, no
    biases, no clamp, per-slot outputs; g, u, h and y are rounded to bf16
    where the GPU path stores bf16. The optional combine weights the per-slot
    outputs by the router's top-k weights and sums them (moe_combine).

Parity status: every function below is pinned by the not-gpu tests in
tests/test_oracle_pins.py except where a docstring says "parity unpinned".
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# Element formats
# ---------------------------------------------------------------------------

# E2M1 magnitudes indexed by the low three bits of the nibble; bit 3 is the
# sign. The MXFP4 arm decodes each nibble with fp4_e2m1_to_float
# [mlxcel-2178, "Current Behavior" and "Proposed Solution" item 1].
E2M1_MAGNITUDE = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)

MXFP4_GROUP = 32          # one E8M0 scale per 32 weights along K [mlxcel-2178, "Current Behavior"]
Q8_BLOCK = 32             # q8_1 activation block length


def e2m1_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each E2M1 nibble: (-1)**bit3 * E2M1_MAGNITUDE[nibble & 7]."""
    c = np.asarray(codes).astype(np.int64)
    mag = np.asarray(E2M1_MAGNITUDE, dtype=np.float64)[c & 7]
    return np.where((c >> 3) & 1, -mag, mag)


def e8m0_decode(e: np.ndarray) -> np.ndarray:
    """E8M0 scale byte -> 2**(e - 127); e = 255 encodes NaN.

    The E8M0 uint8 scale is the per-32-weight scale the MXFP4 arm must keep
    [mlxcel-2178, "Current Behavior", E8M0 uint8_t scale dispatch].
    """
    e = np.asarray(e).astype(np.int64)
    v = np.ldexp(1.0, e - 127)
    return np.where(e == 255, np.nan, v)


# E4M3 element of MXFP8 [OCP-MX]: sign bit 7, exponent bits 6..3 with bias 7,
# mantissa bits 2..0. Exponent field 0 is subnormal (m/8 * 2**-6); the two
# codes with every exponent and mantissa bit set are NaN; there is no
# infinity. The pages list f16 MXFP4 and MXFP8 gathers as the next scope
# beyond the bf16 MXFP4 arm [mlxcel-2178, "Scope": out of scope].
MXFP8_GROUP = 32


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each E4M3 byte, float64 (NaN for 0x7F and 0xFF)."""
    c = np.asarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    ex = (c >> 3) & 15
    man = c & 7
    normal = np.ldexp(1.0 + man / 8.0, ex - 7)
    subnormal = np.ldexp(man / 8.0, -6)
    mag = np.where(ex == 0, subnormal, normal)
    v = np.where(sign == 1, -mag, mag)
    return np.where((ex == 15) & (man == 7), np.nan, v)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns (the upper half of an fp32)."""
    u = np.asarray(bits).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16, nearest-even, returned as bit patterns.

    Rounds straight from float64 (no intermediate fp32 rounding). Finite
    values only; magnitudes at or above the bf16 overflow threshold become
    +-inf.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    flat_v = v.reshape(-1)
    flat_o = out.reshape(-1)
    for i, x in enumerate(flat_v):
        flat_o[i] = _f64_to_bf16_scalar(float(x))
    return out


def _f64_to_bf16_scalar(x: float) -> int:
    if x != x:
        return 0x7FC0
    sign = 0x8000 if (x < 0 or (x == 0 and np.signbit(x))) else 0
    a = abs(x)
    if a == 0:
        return sign
    m, e = np.frexp(a)                   # a = m * 2**e, m in [0.5, 1)
    # bf16 keeps 8 significant bits for normals; below 2**-126 the quantum is
    # fixed at 2**-133 (subnormals).
    if e - 1 >= -126:
        q = np.ldexp(1.0, int(e) - 8)
    else:
        q = np.ldexp(1.0, -133)
    r = np.rint(a / q) * q               # rint: round half to even
    if r >= np.ldexp(1.0, 128):
        return sign | 0x7F80
    f32 = np.float32(r)                  # exact: r has at most 8 significant bits
    return sign | int(np.array(f32).view(np.uint32) >> 16)


# ---------------------------------------------------------------------------
# Canonical byte packings (the formats' storage order)
# ---------------------------------------------------------------------------

def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """4-bit codes [..., K] -> bytes [..., K/2], element k in byte k//2, low nibble for even k.

    This is the order in which a little-endian uint32 read at byte k/2 holds
    eight consecutive nibbles of one group [mlxcel-2178, "Proposed Solution"
    item 1].
    """
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def pack_cb2(codes: np.ndarray) -> np.ndarray:
    """2-bit codes [..., K] -> bytes [..., K/4]; code j of each byte at bits [2j, 2j+2)."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::4] | (c[..., 1::4] << 2) | (c[..., 2::4] << 4) | (c[..., 3::4] << 6)).astype(np.uint8)


def unpack_cb2(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 4,), dtype=np.uint8)
    for j in range(4):
        out[..., j::4] = (p >> (2 * j)) & 3
    return out


def pack_cb3(codes: np.ndarray) -> np.ndarray:
    """3-bit codes [..., K] -> bytes [..., 3K/8]: 8 codes per 3 bytes, little-endian.

    Code j of a group of eight sits at bits [3j, 3j+3) of the 24-bit
    little-endian word formed by the group's three bytes. A 16-weight
    half-block is therefore one 48-bit window [lucebox-21, "Changes" item 2].
    """
    c = np.asarray(codes, dtype=np.uint32)
    lead = c.shape[:-1]
    g = c.reshape(lead + (-1, 8))
    word = np.zeros(g.shape[:-1], dtype=np.uint32)
    for j in range(8):
        word |= g[..., j] << (3 * j)
    out = np.empty(g.shape[:-1] + (3,), dtype=np.uint8)
    for b in range(3):
        out[..., b] = (word >> (8 * b)) & 0xFF
    return out.reshape(lead + (-1,))


def unpack_cb3(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint32)
    lead = p.shape[:-1]
    g = p.reshape(lead + (-1, 3))
    word = g[..., 0] | (g[..., 1] << 8) | (g[..., 2] << 16)
    out = np.empty(g.shape[:-1] + (8,), dtype=np.uint8)
    for j in range(8):
        out[..., j] = (word >> (3 * j)) & 7
    return out.reshape(lead + (-1,))


def pack_codes(fmt: str, codes: np.ndarray) -> np.ndarray:
    if fmt == "mxfp8":
        return np.array(codes, dtype=np.uint8)         # one code per byte
    if fmt in ("mxfp4", "cb4"):
        return pack_nibbles(codes)
    if fmt == "cb2":
        return pack_cb2(codes)
    if fmt == "cb3":
        return pack_cb3(codes)
    raise ValueError(fmt)


def unpack_codes(fmt: str, packed: np.ndarray) -> np.ndarray:
    if fmt == "mxfp8":
        return np.array(packed, dtype=np.uint8)
    if fmt in ("mxfp4", "cb4"):
        return unpack_nibbles(packed)
    if fmt == "cb2":
        return unpack_cb2(packed)
    if fmt == "cb3":
        return unpack_cb3(packed)
    raise ValueError(fmt)


# ---------------------------------------------------------------------------
# Dequantisation
# ---------------------------------------------------------------------------

def mxfp4_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W[n, k] = e2m1(code[n, k]) * 2**(scale[n, k // 32] - 127), float64.

    All eight nibbles of a word belong to one group g = k // 32
    [mlxcel-2178, "Proposed Solution" item 1].
    """
    K = codes.shape[-1]
    g = np.arange(K) // MXFP4_GROUP
    return e2m1_decode(codes) * e8m0_decode(scales)[..., g]


def mxfp8_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W[n, k] = e4m3(code[n, k]) * 2**(scale[n, k // 32] - 127), float64."""
    K = codes.shape[-1]
    g = np.arange(K) // MXFP8_GROUP
    return e4m3_decode(codes) * e8m0_decode(scales)[..., g]


def cb_dequant(codes: np.ndarray, scales: np.ndarray, lut, group: int) -> np.ndarray:
    """W[n, k] = lut[code[n, k]] * 2**(scale[n, k // group] - 127), float64.

    Code -> value through the format's table, times the block scale; for the
    fp3/fp2 formats the scale is per 16-weight half-block, chosen by
    e[i >= QK/2] within each 32-block [lucebox-21, review reply, "decode
    contract"].
    """
    K = codes.shape[-1]
    g = np.arange(K) // group
    vals = np.asarray(lut, dtype=np.float64)[np.asarray(codes).astype(np.int64)]
    return vals * e8m0_decode(scales)[..., g]


# ---------------------------------------------------------------------------
# q8_1 activation quantiser
# ---------------------------------------------------------------------------

def q8_1_quantize(x: np.ndarray):
    """Quantise fp32 activations [..., K] to q8_1 blocks of 32.

    Returns (q int8 [..., K], d_bits uint16 fp16 [..., K/32]). Per block, in
    fp32 arithmetic: amax = max|x|, d = amax / 127, id = 1/d (0 if d == 0),
    q = clamp(round_half_away(x * id), -127, 127); d is stored as fp16 (RNE).
    The kernels consume int8 blocks of 32 with an fp16 scale d_b
    [lucebox-21, review reply, "dot structure"; geo-31, "Caveats",
    quantize_q8_1]. The exact rounding rule is a reading (module header).
    """
    x = np.asarray(x, dtype=np.float32)
    lead = x.shape[:-1]
    K = x.shape[-1]
    xb = x.reshape(lead + (K // Q8_BLOCK, Q8_BLOCK))
    amax = np.max(np.abs(xb), axis=-1)                     # exact in fp32
    d = (amax / np.float32(127.0)).astype(np.float32)      # IEEE fp32 division
    with np.errstate(divide="ignore"):
        inv = np.where(d != 0, np.float32(1.0) / d, np.float32(0.0)).astype(np.float32)
    v = (xb * inv[..., None]).astype(np.float32)           # fp32 product, no FMA
    v64 = v.astype(np.float64)                             # exact
    r = np.sign(v64) * np.floor(np.abs(v64) + 0.5)         # half away from zero, exact in f64
    q = np.clip(r, -127, 127).astype(np.int8).reshape(lead + (K,))
    d16 = d.astype(np.float16).view(np.uint16)
    return q, d16


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def f64_to_f16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 values to fp16 (nearest-even, straight from float64: numpy's
    float64 -> float16 conversion), returned as bit patterns."""
    with np.errstate(over="ignore"):
        return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------------------
# Dot products
# ---------------------------------------------------------------------------

def cb_block_sums(codes: np.ndarray, lut, q: np.ndarray, span: int) -> np.ndarray:
    """Exact integer block sums isum[..., v, n, h] = sum_{i in h} lut[code[n, i]] * q[v, i].

    h runs over consecutive spans of `span` weights along K (16 for the
    half-block formats, 32 otherwise). These are the dp4a chains of the
    codebook vec-dot [lucebox-21, "Changes" items 2 and 4; review reply,
    "dot structure"]. codes: [N, K]; q: [V, K] int8. Result int64 [V, N, K/span].
    """
    N, K = codes.shape
    w = np.asarray(lut, dtype=np.int64)[np.asarray(codes).astype(np.int64)]   # [N, K]
    qq = np.asarray(q).astype(np.int64)                                        # [V, K]
    prod = w[None, :, :] * qq[:, None, :]                                      # [V, N, K]
    return prod.reshape(qq.shape[0], N, K // span, span).sum(axis=-1)


def cb_matvec(codes, scales, lut, group: int, q, d_bits) -> np.ndarray:
    """Codebook matvec y[v, n] = sum_b d_b * sum_{h in b} scale(e_{n,h}) * isum[v, n, h].

    The dot structure db * sum_half(e_half * sum_i code * q8) of the
    ROCMFPX vec-dot [lucebox-21, review reply, "dot structure"], in float64
    with exact integer block sums. codes [N, K], scales [N, K/group],
    q [V, K] int8, d_bits [V, K/32] fp16. Returns float64 [V, N].
    """
    isum = cb_block_sums(codes, lut, q, group).astype(np.float64)   # [V, N, K/group]
    es = e8m0_decode(scales)                                          # [N, K/group]
    per_group = isum * es[None, :, :]
    per_block = per_group.reshape(per_group.shape[0], per_group.shape[1], -1, Q8_BLOCK // group).sum(-1)
    d = f16_bits_to_f64(d_bits)                                       # [V, K/32]
    return (per_block * d[:, None, :]).sum(axis=-1)


def cb_abs_products(codes, scales, lut, group: int, q, d_bits) -> np.ndarray:
    """sum_k |w[n, k] * x~[v, k]| with x~ = d * q, the tolerance base for cb_matvec."""
    W = np.abs(cb_dequant(codes, scales, lut, group))                 # [N, K]
    d = f16_bits_to_f64(d_bits)
    K = codes.shape[-1]
    xq = np.abs(np.asarray(q).astype(np.float64) * np.repeat(d, Q8_BLOCK, axis=-1)[..., :K])
    return xq @ W.T


def act_bits_to_f64(bits: np.ndarray, x_dtype: str = "bf16") -> np.ndarray:
    """Exact value of bf16 or fp16 activation bit patterns."""
    if x_dtype == "bf16":
        return bf16_bits_to_f64(bits)
    if x_dtype == "f16":
        return f16_bits_to_f64(bits)
    raise ValueError(x_dtype)


def mxfp4_matvec(codes, scales, x_bits, x_dtype: str = "bf16") -> np.ndarray:
    """MXFP4 x bf16 matvec y[v, n] = sum_k W[n, k] * x[v, k] in float64.

    W decoded per mxfp4_dequant; x are bf16 activations [mlxcel-2178,
    "Current Behavior": bf16 activations, group size 32, no biases], or fp16
    ones for the f16 variant ("Scope"). codes [N, K], scales [N, K/32],
    x_bits [V, K] uint16. Returns [V, N].
    """
    W = mxfp4_dequant(codes, scales)
    x = act_bits_to_f64(x_bits, x_dtype)
    return x @ W.T


def mxfp4_abs_products(codes, scales, x_bits, x_dtype: str = "bf16") -> np.ndarray:
    W = np.abs(mxfp4_dequant(codes, scales))
    x = np.abs(act_bits_to_f64(x_bits, x_dtype))
    return x @ W.T


def mxfp8_matvec(codes, scales, x_bits, x_dtype: str = "bf16") -> np.ndarray:
    """MXFP8 matvec y[v, n] = sum_k W[n, k] * x[v, k] in float64, W decoded per
    mxfp8_dequant. codes [N, K] (one E4M3 byte each), scales [N, K/32],
    x_bits [V, K] bf16 or fp16. Returns [V, N]."""
    W = mxfp8_dequant(codes, scales)
    x = act_bits_to_f64(x_bits, x_dtype)
    return x @ W.T


def mxfp8_abs_products(codes, scales, x_bits, x_dtype: str = "bf16") -> np.ndarray:
    W = np.abs(mxfp8_dequant(codes, scales))
    x = np.abs(act_bits_to_f64(x_bits, x_dtype))
    return x @ W.T


def mx_matvec(fmt: str, codes, scales, x_bits, x_dtype: str = "bf16") -> np.ndarray:
    if fmt == "mxfp4":
        return mxfp4_matvec(codes, scales, x_bits, x_dtype)
    if fmt == "mxfp8":
        return mxfp8_matvec(codes, scales, x_bits, x_dtype)
    raise ValueError(fmt)


def mx_abs_products(fmt: str, codes, scales, x_bits, x_dtype: str = "bf16") -> np.ndarray:
    if fmt == "mxfp4":
        return mxfp4_abs_products(codes, scales, x_bits, x_dtype)
    if fmt == "mxfp8":
        return mxfp8_abs_products(codes, scales, x_bits, x_dtype)
    raise ValueError(fmt)


# ---------------------------------------------------------------------------
# Expert gather
# ---------------------------------------------------------------------------

def gather_vectors(ids: np.ndarray, per_slot: bool):
    """(t, j) -> activation row index: x[t] when shared, x[t * top_k + j] when per-slot."""
    ntok, top_k = ids.shape
    return [[(t * top_k + j) if per_slot else t for j in range(top_k)] for t in range(ntok)]


def moe_gather(matvec, n_experts: int, ids: np.ndarray, per_slot: bool, N: int) -> np.ndarray:
    """y[t, j, :] = W[ids[t, j]] . x(t, j); an id outside [0, E) gives a zero row.

    `matvec(e, v)` returns expert e applied to activation row v (float64 [N]).
    The unsorted decode gather launches one column block per (token, slot)
    and writes 0 when rhs_idx >= E [mlxcel-2178, "Current Behavior" and
    "Implementation Notes", edge cases].
    """
    ntok, top_k = ids.shape
    vidx = gather_vectors(ids, per_slot)
    y = np.zeros((ntok, top_k, N), dtype=np.float64)
    for t in range(ntok):
        for j in range(top_k):
            e = int(ids[t, j])
            if 0 <= e < n_experts:
                y[t, j] = matvec(e, vidx[t][j])
    return y


def mxfp4_moe_gather(codes, scales, x_bits, ids, per_slot: bool, x_dtype: str = "bf16"):
    """MXFP4 expert gather. codes [E, N, K], scales [E, N, K/32], x_bits [V, K]."""
    E, N, _ = codes.shape
    return moe_gather(lambda e, v: mxfp4_matvec(codes[e], scales[e], x_bits[v:v + 1], x_dtype)[0],
                      E, ids, per_slot, N)


def mx_moe_gather(fmt: str, codes, scales, x_bits, ids, per_slot: bool, x_dtype: str = "bf16"):
    """MXFP4 or MXFP8 expert gather. codes [E, N, K], scales [E, N, K/32], x_bits [V, K]."""
    E, N, _ = codes.shape
    return moe_gather(lambda e, v: mx_matvec(fmt, codes[e], scales[e], x_bits[v:v + 1], x_dtype)[0],
                      E, ids, per_slot, N)


def cb_moe_gather(codes, scales, lut, group, q, d_bits, ids, per_slot: bool):
    """Codebook expert gather. codes [E, N, K], q [V, K], d_bits [V, K/32]."""
    E, N, _ = codes.shape
    return moe_gather(lambda e, v: cb_matvec(codes[e], scales[e], lut, group,
                                             q[v:v + 1], d_bits[v:v + 1])[0],
                      E, ids, per_slot, N)


def cb_moe_block_sums(codes, lut, group, q, ids, per_slot: bool):
    """Integer block sums of every gathered (token, slot): int64 [ntok, top_k, N, K/group]."""
    E, N, K = codes.shape
    ntok, top_k = ids.shape
    vidx = gather_vectors(ids, per_slot)
    out = np.zeros((ntok, top_k, N, K // group), dtype=np.int64)
    for t in range(ntok):
        for j in range(top_k):
            e = int(ids[t, j])
            if 0 <= e < E:
                v = vidx[t][j]
                out[t, j] = cb_block_sums(codes[e], lut, q[v:v + 1], group)[0]
    return out


# ---------------------------------------------------------------------------
# SwiGLU and one gpt-oss-style MoE layer
# ---------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)), float64."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """h = silu(g) * u, float64, between the gate/up and down gathers.

    The gpt-oss decode layer runs gate, up and down gather matvecs per layer
    [mlxcel-2178, "Problem / Background": 24 layers times gate, up and down;
    "Current Behavior": GptOssSwitchGLU]. The activation between them is
    taken to be plain SwiGLU (a reading; parity unpinned against gpt-oss
    itself, pinned to the closed form of silu).
    """
    return silu(g) * np.asarray(u, dtype=np.float64)


def mxfp4_moe_layer(gate, up, down, x_bits, ids):
    """One MoE decode layer: g, u = gather(gate/up, x); h = swiglu(g, u); y = gather(down, h).

    gate/up/down are (codes [E, N, K], scales [E, N, K/32]) pairs; x_bits
    [ntok, K] bf16. The GPU path stores g, u and h as bf16, so the chain
    rounds them to bf16 (RNE) before they feed the next step. Returns a dict
    of float64 arrays g, u, h (as bf16 values) and y (unrounded).
    """
    g = mxfp4_moe_gather(gate[0], gate[1], x_bits, ids, per_slot=False)
    u = mxfp4_moe_gather(up[0], up[1], x_bits, ids, per_slot=False)
    g_b = f64_to_bf16_bits(g)
    u_b = f64_to_bf16_bits(u)
    h = swiglu(bf16_bits_to_f64(g_b), bf16_bits_to_f64(u_b))
    h_b = f64_to_bf16_bits(h)
    ntok, top_k = ids.shape
    h_rows = h_b.reshape(ntok * top_k, -1)
    y = mxfp4_moe_gather(down[0], down[1], h_rows, ids, per_slot=True)
    return {"g_bits": g_b, "u_bits": u_b, "h_bits": h_b, "h": h, "y": y, "h_rows_bits": h_rows}


def moe_gate_up_swiglu(gate_matvec, up_matvec, n_experts: int, ids: np.ndarray, N: int):
    """Fused gate/up/SwiGLU of one MoE layer: h[t, j] = silu(g) * u with
    g = W_gate[ids[t, j]] . x[t] and u = W_up[ids[t, j]] . x[t] taken exactly
    (float64, no intermediate rounding). `gate_matvec(e, t)` / `up_matvec(e, t)`
    return one expert applied to token t's activation. An invalid id gives a
    zero row. Returns (h, g, u), float64 [ntok, top_k, N].

    The gate and up gathers share the token's activation and the SwiGLU sits
    between them and the down gather [mlxcel-2178, "Problem / Background";
    "Current Behavior": GptOssSwitchGLU]; fusing them changes no definition,
    only where g and u live (registers instead of bf16 buffers).
    """
    g = moe_gather(gate_matvec, n_experts, ids, False, N)
    u = moe_gather(up_matvec, n_experts, ids, False, N)
    return swiglu(g, u), g, u


def swiglu_tolerance(g, u, tol_g, tol_u):
    """Propagate absolute bounds on g and u through h = silu(g) * u.

    |d silu / dz| = |s(z) (1 + z (1 - s(z)))| <= 1.1 for all z (s the logistic
    function), so |dh| <= 1.1 |u| tol_g + |silu(g)| tol_u + 1.1 tol_g tol_u.
    """
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    return 1.1 * np.abs(u) * tol_g + np.abs(silu(g)) * tol_u + 1.1 * tol_g * tol_u



def moe_combine(y_slots, weights, ids, n_experts: int):
    """Router-weighted combine of a MoE layer's per-slot expert outputs:
    out[t] = sum_j weights[t, j] * y_slots[t, j] over the slots j whose id is
    in [0, n_experts) (an invalid id contributes nothing), in float64.

    y_slots [ntok, top_k, N], weights and ids [ntok, top_k]. The pages print
    the switch-GLU part of the gpt-oss layer (per-slot outputs of the top-k
    experts) [mlxcel-2178, "Current Behavior": GptOssSwitchGLU]; weighting
    those outputs by the router's top-k weights and summing them is the MoE
    block's combine (a reading: the pages do not print it).
    """
    y_slots = np.asarray(y_slots, dtype=np.float64)
    weights = np.asarray(weights, dtype=np.float64)
    ntok, top_k, N = y_slots.shape
    out = np.zeros((ntok, N), dtype=np.float64)
    for t in range(ntok):
        for j in range(top_k):
            if 0 <= int(ids[t, j]) < n_experts:
                out[t] += weights[t, j] * y_slots[t, j]
    return out
