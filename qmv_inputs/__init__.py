"""Seeded synthetic inputs for the block-quantized decode matvec.

This module is shared by the oracle's tests, the GPU parity tests and the
benchmark. It holds random draws and workload recipes only -- none of the
arithmetic of the method (no decoding, no scaling, no dot products, no
quantisation of activations). Everything is drawn from numpy's PCG64
``Generator`` with an explicit seed, so a (recipe, seed) pair names one input.

Value distributions follow the workloads the pages describe:

* weight codes: uniform over all ``2**bits`` codes (E2M1 nibbles for MXFP4,
  LUT indices for the codebook formats);
* E8M0 block scales: uniform integers in ``[120, 130]``;
* activations: N(0, 1), rounded to bf16 (MXFP4 path) or kept as fp32
  (codebook paths, which quantise them to q8_1 themselves);
* router ids: ``top_k`` distinct expert ids per token, uniform.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# Bits per code and E8M0 group length (weights per scale along K) per format.
FORMAT_BITS = {"mxfp4": 4, "cb2": 2, "cb3": 3, "cb4": 4, "mxfp8": 8}
FORMAT_GROUP = {"mxfp4": 32, "cb2": 16, "cb3": 16, "cb4": 32, "mxfp8": 32}

# MXFP8 codes that are NaN (never drawn: every synthetic weight is finite).
E4M3_NAN_CODES = (0x7F, 0xFF)

# Codebooks of the synthetic workloads (int8 values indexed by code).
LUT_CB2 = (-3, -1, 1, 3)
LUT_CB3 = (-8, -5, -3, -1, 1, 3, 5, 8)
LUT_CB4 = (-12, -9, -7, -5, -4, -3, -2, -1, 1, 2, 3, 4, 5, 7, 9, 12)


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def codes(g: np.random.Generator, shape, bits: int) -> np.ndarray:
    """Uniform codes in [0, 2**bits), one code per uint8."""
    return g.integers(0, 1 << bits, size=shape, dtype=np.uint8)


def finite_e4m3_codes(g: np.random.Generator, shape) -> np.ndarray:
    """Uniform over the 254 E4M3 codes that are not NaN, one per uint8."""
    c = g.integers(0, 254, size=shape, dtype=np.int32)
    c = c + (c >= 0x7F)          # skip 0x7F; 0xFF lies beyond the drawn range
    return c.astype(np.uint8)


def format_codes(g: np.random.Generator, fmt: str, shape) -> np.ndarray:
    """Synthetic codes of a format, one per uint8: uniform over every code,
    except MXFP8, whose NaN codes are left out."""
    if fmt == "mxfp8":
        return finite_e4m3_codes(g, shape)
    return codes(g, shape, FORMAT_BITS[fmt])


def canonical_uniform_codes(g: np.random.Generator, lead_shape, K: int, bits: int) -> np.ndarray:
    """Canonical packed code bytes of uniform codes: [..., K * bits / 8] uniform bytes.

    Every canonical packing used here (two nibbles per byte, four 2-bit codes
    per byte, eight 3-bit codes per three bytes) maps uniform random bytes to
    independent uniform codes, so no packing step is needed to draw them.
    8-bit codes are MXFP8 bytes and leave out its NaN codes.
    """
    if bits == 8:
        return finite_e4m3_codes(g, tuple(lead_shape) + (K,))
    return g.integers(0, 256, size=tuple(lead_shape) + (K * bits // 8,), dtype=np.uint8)


def e8m0(g: np.random.Generator, shape, lo: int = 120, hi: int = 130) -> np.ndarray:
    """Uniform E8M0 exponent bytes in [lo, hi] (inclusive)."""
    return g.integers(lo, hi + 1, size=shape, dtype=np.uint8)


def normal_f32(g: np.random.Generator, shape) -> np.ndarray:
    return g.standard_normal(size=shape, dtype=np.float64).astype(np.float32)


def normal_f16_bits(g: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) samples as fp16 bit patterns (uint16): the fp32 draw converted by
    numpy (nearest-even)."""
    return normal_f32(g, shape).astype(np.float16).view(np.uint16)


def normal_bf16_bits(g: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) samples as bf16 bit patterns (uint16), round-to-nearest-even.

    The draw is made in fp32 and its upper half kept with RNE; the samples are
    finite, so no NaN handling is needed here.
    """
    f = normal_f32(g, shape)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def scaled_normal_bf16_bits(g: np.random.Generator, shape, exp_shifts) -> np.ndarray:
    """N(0,1) samples times 2**s as bf16 bit patterns, s = exp_shifts[i] for
    row i of the leading axis: the fp32 draw scaled exactly by a power of two
    (np.ldexp), then its upper half kept with round-to-nearest-even."""
    f = normal_f32(g, shape)
    s = np.asarray(exp_shifts, dtype=np.int64).reshape((-1,) + (1,) * (f.ndim - 1))
    f = np.ldexp(f.astype(np.float64), s).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def e8m0_choice(g: np.random.Generator, shape, values) -> np.ndarray:
    """E8M0 bytes drawn uniformly from the given values."""
    return np.asarray(values, dtype=np.uint8)[g.integers(0, len(values), size=shape)]


def e4m3_subnormal_codes(g: np.random.Generator, shape) -> np.ndarray:
    """E4M3 codes with a zero exponent field (zero and the subnormals), either sign."""
    return (g.integers(0, 8, size=shape) | (g.integers(0, 2, size=shape) << 7)).astype(np.uint8)


def topk_ids(g: np.random.Generator, ntok: int, top_k: int, n_experts: int) -> np.ndarray:
    """[ntok][top_k] int32: distinct expert ids per token, uniform."""
    out = np.empty((ntok, top_k), dtype=np.int32)
    for t in range(ntok):
        out[t] = g.choice(n_experts, size=top_k, replace=False)
    return out


def router_weights(g: np.random.Generator, ntok: int, top_k: int) -> np.ndarray:
    """[ntok][top_k] fp32 positive top-k router weights, each token's summing
    to about 1 (a flat Dirichlet draw)."""
    return g.dirichlet(np.ones(top_k), size=ntok).astype(np.float32)


@dataclasses.dataclass(frozen=True)
class Recipe:
    """One synthetic workload: matrix shape, format and routing."""
    name: str
    fmt: str
    N: int
    K: int
    n_experts: int = 1          # 1 = dense
    top_k: int = 0              # 0 = dense
    ntok: int = 1
    per_slot_x: bool = False    # down projection: one activation per (token, slot)
    lut: Optional[tuple] = None
    seed: int = 0

    @property
    def bits(self) -> int:
        return FORMAT_BITS[self.fmt]

    @property
    def group(self) -> int:
        return FORMAT_GROUP[self.fmt]

    def matrix_bytes(self) -> int:
        """Code bytes plus E8M0 bytes of one N x K matrix (no padding)."""
        return self.N * self.K * self.bits // 8 + self.N * (self.K // self.group)


@dataclasses.dataclass
class Weights:
    codes: np.ndarray    # [E][N][K] uint8, one code per byte
    scales: np.ndarray   # [E][N][K/group] uint8 E8M0


def draw_weights(g: np.random.Generator, r: Recipe, n_experts: Optional[int] = None) -> Weights:
    E = r.n_experts if n_experts is None else n_experts
    c = codes(g, (E, r.N, r.K), r.bits)
    s = e8m0(g, (E, r.N, r.K // r.group))
    return Weights(c, s)


# The five workloads. Config 1 is one gpt-oss MoE layer: gate, up and down are
# three separate 2880 x 2880 expert sets; a step sweeps 24 such layers.
CONFIG0 = Recipe("dense_mxfp4_2880x2880", "mxfp4", 2880, 2880, seed=0)
CONFIG1_GATE = Recipe("moe_mxfp4_gate", "mxfp4", 2880, 2880, n_experts=32, top_k=4, seed=1)
CONFIG1_UP = Recipe("moe_mxfp4_up", "mxfp4", 2880, 2880, n_experts=32, top_k=4, seed=1)
CONFIG1_DOWN = Recipe("moe_mxfp4_down", "mxfp4", 2880, 2880, n_experts=32, top_k=4,
                      per_slot_x=True, seed=1)
CONFIG1_LAYERS = 24
CONFIG2 = Recipe("moe_cb2_gate_up_7168to2048", "cb2", 2048, 7168, n_experts=256, top_k=4,
                 lut=LUT_CB2, seed=2)
CONFIG3 = Recipe("moe_cb3_down_2048to7168_ntok4", "cb3", 7168, 2048, n_experts=256, top_k=4,
                 ntok=4, per_slot_x=True, lut=LUT_CB3, seed=3)
CONFIG4_SHAPES = ((7168, 7168), (2048, 7168))
CONFIG4_NTOKS = (1, 2, 3, 4)


def config4(N: int, K: int, ntok: int) -> Recipe:
    return Recipe(f"dense_cb4_{N}x{K}_ntok{ntok}", "cb4", N, K, ntok=ntok, lut=LUT_CB4, seed=4)
