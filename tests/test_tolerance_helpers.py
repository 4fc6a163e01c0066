"""CPU checks of the comparison helpers the GPU parity tests use: the
float64 -> bf16 / fp16 rounding of the stored-output check against the
oracle's pinned roundings, and the rounding-interval rule itself."""
import numpy as np
import pytest

import oracle
import qmv_inputs as qi

pytest.importorskip("bit_quantized_moe_gb300")
from qmv_testutil import close_mask, round_out, stored_err  # noqa: E402


def _sample():
    g = qi.rng(77)
    v = g.standard_normal(20000) * np.exp2(g.integers(-140, 130, 20000).astype(np.float64))
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 2.0 ** -133 * 1.5, 2.0 ** -133 * 2.5,
                     3.3895313892515355e38, 3.3961775292304e38, 3.4e38, -3.4e38, 0.0, -0.0, 2.0 ** -126,
                     2.0 ** -126 * (1 - 2.0 ** -9)])
    return np.concatenate([ties, v, np.nextafter(v, np.inf)])


def test_round_out_bf16_matches_oracle():
    v = _sample()
    with np.errstate(over="ignore"):
        want = oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(v))
    got = round_out(v, "bf16")
    same = (got == want) | (np.isinf(got) & np.isinf(want) & (np.sign(got) == np.sign(want)))
    assert same.all(), v[~same][:5]


def test_round_out_f16_matches_oracle():
    v = _sample() * 2.0 ** -100
    want = oracle.f16_bits_to_f64(oracle.f64_to_f16_bits(v))
    got = round_out(v, "f16")
    assert np.array_equal(got, want)


def test_close_mask_is_the_rounding_interval():
    """A stored value passes exactly when some fp32 result within the bound
    rounds to it: the neighbours just outside round(ref -+ bound) fail."""
    ref = np.array([1.0, 1.0, -3.0, 1e-3])
    bound = np.array([2.0 ** -10, 2.0 ** -7, 2.0 ** -6, 0.0])
    lo, hi = round_out(ref - bound, "bf16"), round_out(ref + bound, "bf16")
    assert close_mask(lo, ref, bound, "bf16").all() and close_mask(hi, ref, bound, "bf16").all()
    # the bf16 neighbours just outside [lo, hi]
    lb, hb = oracle.f64_to_bf16_bits(lo).astype(np.int64), oracle.f64_to_bf16_bits(hi).astype(np.int64)
    below = oracle.bf16_bits_to_f64(np.where(lo > 0, lb - 1, lb + 1).astype(np.uint16))
    above = oracle.bf16_bits_to_f64(np.where(hi > 0, hb + 1, hb - 1).astype(np.uint16))
    assert not close_mask(below, ref, bound, "bf16").any()
    assert not close_mask(above, ref, bound, "bf16").any()
    assert close_mask(ref + bound, ref, bound, "f32").all()
    assert not close_mask(ref + bound * 1.01 + 1e-12, ref, bound, "f32").any()


def test_stored_err_covers_rounding():
    g = qi.rng(78)
    v = g.standard_normal(5000) * 10.0
    b = np.abs(g.standard_normal(5000)) * 1e-3
    for out in ("bf16", "f16"):
        for s in (-1.0, 1.0):
            stored = round_out(v + s * b, out)
            assert np.all(np.abs(stored - v) <= stored_err(v, b, out))
