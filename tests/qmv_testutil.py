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


def tolerance(absum: np.ndarray, ref: np.ndarray, bf16_out: bool) -> np.ndarray:
    """1e-3 * sum|w x| per output, plus one bf16 ulp of the result when the
    output is stored as bf16 (its rounding alone can exceed the first term
    when |y| is close to sum|w x|)."""
    tol = 1e-3 * absum
    if bf16_out:
        tol = tol + np.abs(ref) * 2.0 ** -8
    return tol + 1e-30


def assert_close(got, ref, absum, bf16_out, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    tol = tolerance(absum, ref, bf16_out)
    bad = ~(err <= tol)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} outputs outside tolerance; first {tuple(i)}: "
                             f"got {got[tuple(i)]!r} want {ref[tuple(i)]!r} tol {tol[tuple(i)]!r}")


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
