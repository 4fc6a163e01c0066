"""Shared helpers for the GPU parity tests: upload seeded inputs, run the CUDA
path through the C ABI binding, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import bit_quantized_moe_gb300 as qmv
import oracle
import qmv_inputs as qi

DEV = "cuda:0"


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(a).to(DEV)


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


# E8M0 ranges of the synthetic weights of the MX-variant tests, chosen so that
# the rms weight is about 0.03 (rms E2M1 value 2.9, rms E4M3 value ~92): a
# K = 2880 layer's g, u, h and y then stay O(1-10), far inside fp16's range
# (65504), for fp16 and bf16 activations alike.
MX_SCALES = {"mxfp4": (112, 122), "mxfp8": (107, 117)}


def act_bits(g, x_dtype: str, shape) -> np.ndarray:
    """N(0,1) activations as bf16 or fp16 bit patterns."""
    return qi.normal_bf16_bits(g, shape) if x_dtype == "bf16" else qi.normal_f16_bits(g, shape)


def act_to_dev(bits: np.ndarray, x_dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV)
    return t.view(torch.bfloat16 if x_dtype == "bf16" else torch.float16)


def mx_flags(x_dtype: str) -> int:
    return qmv.QMV_FLAG_X_F16 if x_dtype == "f16" else 0


class Matrices:
    """E expert matrices of one format; only `experts` hold drawn data, the
    rest of the device buffer is zero (the kernels never read them)."""

    def __init__(self, fmt, N, K, E, experts, seed, lut=None, scale_lo=120, scale_hi=130):
        self.fmt, self.N, self.K, self.E = fmt, N, K, E
        self.lut = list(lut) if lut is not None else None
        self.desc = qmv.wdesc(fmt, N, K, E, lut)
        self.one = qmv.wdesc(fmt, N, K, 1, lut)
        self.eb = qmv.qmv_packed_expert_bytes(self.desc)
        g = qi.rng(seed)
        self.codes, self.scales = {}, {}
        self.w = torch.zeros(self.eb * E, dtype=torch.uint8, device=DEV)
        for e in sorted(set(int(v) for v in experts if 0 <= int(v) < E)):
            c = qi.format_codes(g, fmt, (N, K))
            s = qi.e8m0(g, (N, K // qi.FORMAT_GROUP[fmt]), scale_lo, scale_hi)
            self.set_expert(e, c, s)

    def set_expert(self, e, codes, scales):
        self.codes[e], self.scales[e] = codes, scales
        packed = qmv.qmv_pack_weights(self.one, oracle.pack_codes(self.fmt, codes[None]), scales[None])
        self.w[e * self.eb:(e + 1) * self.eb] = torch.from_numpy(packed).to(DEV)


def round_out(v, out: str) -> np.ndarray:
    """float64 values rounded to nearest (ties to even) in the output type
    `out` ("bf16" or "f16"), returned as float64; "f32" returns v unchanged.
    bf16 rounds straight from the float64 bits (no intermediate fp32), with
    its subnormals on the 2^-133 grid and overflow to +-inf; fp16 uses numpy's
    float64 -> float16 conversion (round to nearest even)."""
    v = np.asarray(v, dtype=np.float64)
    if out == "f32":
        return v
    if out == "f16":
        with np.errstate(over="ignore"):
            return v.astype(np.float16).astype(np.float64)
    assert out == "bf16", out
    c = np.ascontiguousarray(v)
    b = c.view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    r = ((b + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)).view(np.float64)
    r = np.where(np.abs(r) > 3.3895313892515355e38, np.copysign(np.inf, c), r)
    sub = np.rint(c * 2.0 ** 133) * 2.0 ** -133
    r = np.where(np.abs(c) < 2.0 ** -126, sub, r)
    return np.where(np.isfinite(c), r, c)


def close_mask(got, ref, bound, out: str) -> np.ndarray:
    """True where a stored output is consistent with the exact value `ref`:
    the kernel's fp32 result lies within `bound` of ref, and a bf16 or fp16
    output is that fp32 result rounded to nearest. Rounding is monotone, so
    the stored value must lie between round(ref - bound) and
    round(ref + bound); an fp32 output must lie within bound of ref."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    if out == "f32":
        return np.abs(got - ref) <= bound
    return (round_out(ref - bound, out) <= got) & (got <= round_out(ref + bound, out))


def _out_name(out) -> str:
    if out is True:
        return "bf16"
    if out is False:
        return "f32"
    return out


def out_of(fmt: str, x_dtype: str = "bf16") -> str:
    """Stored output type of a call: the activation type for the MX formats,
    fp32 for the codebook formats."""
    return x_dtype if fmt in ("mxfp4", "mxfp8") else "f32"


def stored_err(v, bound, out: str) -> np.ndarray:
    """Bound on |stored - v| when the kernel's fp32 result lies within `bound`
    of v and is stored in `out`, rounded to nearest: bound plus half an ulp at
    |v| + bound (bf16, 8 significant bits: 2^-8 relative, subnormal
    half-quantum 2^-134; fp16, 11 bits: 2^-11, 2^-25)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    b = np.asarray(bound, dtype=np.float64)
    if out == "bf16":
        return b + (a + b) * 2.0 ** -8 + 2.0 ** -134
    if out == "f16":
        return b + (a + b) * 2.0 ** -11 + 2.0 ** -25
    return b


def assert_within(got, ref, bound, out, what=""):
    """Every stored output consistent with ref within the fp32 bound (close_mask)."""
    out = _out_name(out)
    got = np.asarray(got, dtype=np.float64)
    bound = np.broadcast_to(np.asarray(bound, dtype=np.float64), got.shape)
    bad = ~close_mask(got, ref, bound, out)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} outputs outside tolerance; first {i}: "
                             f"got {got[i]!r} want {np.asarray(ref)[i]!r} bound {bound[i]!r} ({out})")


def assert_close(got, ref, absum, out, what=""):
    """Per output element: max|gpu - oracle| <= 1e-3 * sum|w x| for the
    kernel's fp32 result, checked on the stored value as close_mask does.
    out: "bf16", "f16" or "f32" (True / False mean bf16 / fp32)."""
    assert_within(got, ref, 1e-3 * np.asarray(absum, dtype=np.float64), out, what)


def quantize_on_gpu(x_f32: np.ndarray):
    """x [nvec][K] fp32 -> (device q8 buffer, q int8, d fp16 bits) via qmv_quantize_act_q8."""
    nvec, K = x_f32.shape
    xq = torch.empty(qmv.qmv_act_q8_bytes(nvec, K), dtype=torch.uint8, device=DEV)
    qmv.qmv_quantize_act_q8(to_dev(x_f32.astype(np.float32)), nvec, K, xq)
    torch.cuda.synchronize()
    q, d = qmv.qmv_act_q8_unpack(xq.cpu().numpy(), nvec, K)
    return xq, q, d


def status_clean():
    return qmv.qmv_device_status(clear=True) == 0
