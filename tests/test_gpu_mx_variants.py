"""GPU parity of the MX variants: MXFP8 weights (E4M3 elements, E8M0 per 32)
and fp16 activations and outputs (QMV_FLAG_X_F16) for MXFP4 and MXFP8, dense,
gathered, fused gate/up, whole layers and the router-weighted combine -- the
f16 MXFP4 and MXFP8 gathers that "perf(rocm): add an mxfp4 arm to the
warp-shared gather_qmv kernel for gpt-oss decode" ("Scope") lists beyond the
bf16 MXFP4 arm. Same bar as the MXFP4 tests: decoded weights bit-exact,
max|gpu - oracle| <= 1e-3 * sum|w x| plus one output ulp for the products."""
import numpy as np
import pytest
import torch

import oracle
import qmv_inputs as qi

pytestmark = pytest.mark.gpu

qmv = pytest.importorskip("bit_quantized_moe_gb300")
from qmv_testutil import (DEV, MX_SCALES, Matrices, act_bits, act_to_dev, assert_close,  # noqa: E402
                          assert_within, mx_flags, status_clean, stored_err, to_dev)
from test_gpu_parity import GateUp, _combine_tol, _layer_expected, check_gate_up  # noqa: E402

# (weight format, activation type) pairs beyond the bf16 MXFP4 path
VARIANTS = [("mxfp8", "bf16"), ("mxfp8", "f16"), ("mxfp4", "f16")]


def _np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def _out_dtype(x_dtype):
    return torch.bfloat16 if x_dtype == "bf16" else torch.float16


def _mats(fmt, N, K, E, experts, seed):
    lo, hi = MX_SCALES[fmt]
    return Matrices(fmt, N, K, E, experts, seed=seed, scale_lo=lo, scale_hi=hi)


def test_mxfp8_dequant_every_code():
    """All 256 E4M3 codes (NaN ones included) under several scales decode
    bit-exactly through the device path."""
    N, K = 16, 256
    m = Matrices("mxfp8", N, K, 1, [], seed=1)
    codes = np.tile(np.arange(256, dtype=np.uint8), (N, 1))
    scales = np.repeat(np.array([127, 100, 140, 1, 254, 127, 120, 133], dtype=np.uint8)[None, :], N, 0)
    m.set_expert(0, codes, scales)
    out = torch.empty(N, K, dtype=torch.float32, device=DEV)
    qmv.qmv_debug_dequant(m.desc, m.w, 0, out)
    got = out.cpu().numpy()
    ref = oracle.mxfp8_dequant(codes, scales).astype(np.float32)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), f"{(~same).sum()} decoded weights differ"
    assert status_clean()


@pytest.mark.parametrize("fmt,x_dtype", VARIANTS)
@pytest.mark.parametrize("N,K", [(1, 32), (17, 96), (516, 2880), (2880, 2880), (48, 4096)])
@pytest.mark.parametrize("ntok", [1, 2, 4])
def test_mx_dense(fmt, x_dtype, N, K, ntok):
    m = _mats(fmt, N, K, 1, [0], seed=11 * N + K)
    x = act_bits(qi.rng(ntok + N + K), x_dtype, (ntok, K))
    y = torch.empty(ntok, N, dtype=_out_dtype(x_dtype), device=DEV)
    qmv.qmv_dense_ex(m.desc, m.w, act_to_dev(x, x_dtype), ntok, y, mx_flags(x_dtype))
    ref = oracle.mx_matvec(fmt, m.codes[0], m.scales[0], x, x_dtype)
    absum = oracle.mx_abs_products(fmt, m.codes[0], m.scales[0], x, x_dtype)
    assert_close(_np(y), ref, absum, x_dtype, f"{fmt}/{x_dtype} dense {N}x{K} ntok={ntok}")
    assert status_clean()


@pytest.mark.parametrize("fmt,x_dtype", VARIANTS)
@pytest.mark.parametrize("ntok,top_k,per_slot", [(1, 4, False), (1, 4, True), (4, 4, False), (4, 4, True),
                                                 (2, 8, True), (3, 1, False)])
def test_mx_gather(fmt, x_dtype, ntok, top_k, per_slot):
    E, N, K = 32, 2880, 2880
    g = qi.rng(N + 10 * ntok + top_k + (7 if per_slot else 0))
    ids = qi.topk_ids(g, ntok, top_k, E)
    if ntok > 1:
        ids[1, 0] = ids[0, 0]          # an expert shared by two tokens
        ids[-1, -1] = E + 1            # an invalid id: zero row
    m = _mats(fmt, N, K, E, ids.reshape(-1), seed=N + top_k)
    nvec = ntok * top_k if per_slot else ntok
    x = act_bits(g, x_dtype, (nvec, K))
    y = torch.full((ntok, top_k, N), 5.0, dtype=_out_dtype(x_dtype), device=DEV)
    qmv.qmv_moe_gather_ex(m.desc, m.w, act_to_dev(x, x_dtype), int(per_slot), to_dev(ids), ntok, top_k, y,
                          mx_flags(x_dtype))
    got = _np(y)
    for t in range(ntok):
        for j in range(top_k):
            e = int(ids[t, j])
            if not (0 <= e < E):
                assert np.all(got[t, j] == 0)
                continue
            v = t * top_k + j if per_slot else t
            ref = oracle.mx_matvec(fmt, m.codes[e], m.scales[e], x[v:v + 1], x_dtype)[0]
            absum = oracle.mx_abs_products(fmt, m.codes[e], m.scales[e], x[v:v + 1], x_dtype)[0]
            assert_close(got[t, j], ref, absum, x_dtype, f"slot ({t},{j}) expert {e}")
    assert status_clean()


@pytest.mark.parametrize("fmt,x_dtype", [("mxfp8", "bf16"), ("mxfp4", "bf16"), ("mxfp4", "f16")])
def test_per_slot_gather_stages_only_its_vectors(fmt, x_dtype):
    """32 per-slot vectors of K = 4096 (256 KB of staged f16, more than a
    CTA's shared memory): each CTA stages only the vectors of its own items,
    at consecutive positions."""
    E, N, K, ntok, top_k = 16, 1032, 4096, 4, 8
    g = qi.rng(900)
    ids = np.stack([g.permutation(E)[:top_k] for _ in range(ntok)]).astype(np.int32)
    ids[2, 3] = -1
    m = _mats(fmt, N, K, E, ids.reshape(-1), seed=901)
    x = act_bits(g, x_dtype, (ntok * top_k, K))
    y = torch.full((ntok, top_k, N), 5.0, dtype=_out_dtype(x_dtype), device=DEV)
    qmv.qmv_moe_gather_ex(m.desc, m.w, act_to_dev(x, x_dtype), 1, to_dev(ids), ntok, top_k, y, mx_flags(x_dtype))
    got = _np(y)
    for t in range(ntok):
        for j in range(top_k):
            e, v = int(ids[t, j]), t * top_k + j
            if e < 0:
                assert np.all(got[t, j] == 0)
                continue
            ref = oracle.mx_matvec(fmt, m.codes[e], m.scales[e], x[v:v + 1], x_dtype)[0]
            absum = oracle.mx_abs_products(fmt, m.codes[e], m.scales[e], x[v:v + 1], x_dtype)[0]
            assert_close(got[t, j], ref, absum, x_dtype, f"slot ({t},{j}) expert {e}")
    assert status_clean()


@pytest.mark.parametrize("fmt,x_dtype", VARIANTS)
@pytest.mark.parametrize("N,ntok,top_k", [(2880, 1, 4), (516, 2, 4), (515, 1, 3)])
def test_mx_gate_up_swiglu(fmt, x_dtype, N, ntok, top_k):
    E, K = 32, 2880
    g = qi.rng(N + ntok + 40)
    ids = qi.topk_ids(g, ntok, top_k, E)
    if ntok > 1:
        ids[1, 0] = ids[0, 0]
        ids[-1, -1] = 77
    lo, hi = MX_SCALES[fmt]
    m = GateUp(fmt, N, K, E, ids.reshape(-1), seed=N + 41, scale_lo=lo, scale_hi=hi)
    x = act_bits(g, x_dtype, (ntok, K))
    h = torch.full((ntok, top_k, N), 3.0, dtype=_out_dtype(x_dtype), device=DEV)
    qmv.qmv_moe_gate_up_swiglu(m.desc, m.w, act_to_dev(x, x_dtype), to_dev(ids), ntok, top_k, h, mx_flags(x_dtype))
    check_gate_up(m, ids, _np(h), x, x_dtype=x_dtype)
    assert status_clean()


MX_PAIRS = [("mxfp8", "mxfp8"), ("mxfp4", "mxfp8"), ("mxfp4", "mxfp4")]


def _mx_layer_case(fmt_gu, fmt_dn, x_dtype, ntok, top_k, seed, N=2880, K=2880, E=32):
    g = qi.rng(seed)
    ids = qi.topk_ids(g, ntok, top_k, E)
    if ntok > 1:
        ids[1, 0] = ids[0, 0]
        ids[-1, -1] = -1
    lo, hi = MX_SCALES[fmt_gu]
    gu = GateUp(fmt_gu, N, K, E, ids.reshape(-1), seed=seed + 1, scale_lo=lo, scale_hi=hi)
    lo, hi = MX_SCALES[fmt_dn]
    down = Matrices(fmt_dn, K, N, E, ids.reshape(-1), seed=seed + 2, scale_lo=lo, scale_hi=hi)
    x = act_bits(g, x_dtype, (ntok, K))
    return ids, gu, down, x


@pytest.mark.parametrize("pair", MX_PAIRS, ids=lambda p: f"{p[0]}-{p[1]}")
@pytest.mark.parametrize("x_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("ntok,top_k", [(1, 4), (4, 2)])
def test_mx_layer(pair, x_dtype, ntok, top_k):
    if pair == ("mxfp4", "mxfp4") and x_dtype == "bf16":
        pytest.skip("the bf16 MXFP4 layer is covered by test_layer_format_pairs")
    ids, gu, down, x = _mx_layer_case(*pair, x_dtype, ntok, top_k, 700 + ntok * 10 + top_k)
    ws = torch.empty(qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k), dtype=torch.uint8, device=DEV)
    y = torch.full((ntok, top_k, gu.K), 7.0, dtype=_out_dtype(x_dtype), device=DEV)
    qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, act_to_dev(x, x_dtype), to_dev(ids), ntok, top_k, ws, y,
                      mx_flags(x_dtype))
    want, tol = _layer_expected(gu, down, ids, x=x, x_dtype=x_dtype)
    assert_within(_np(y), want, tol, x_dtype, "layer")
    assert status_clean()


@pytest.mark.parametrize("x_dtype", ["bf16", "f16"])
def test_mx_layer_combine(x_dtype):
    """MXFP8 layer + router-weighted combine against the oracle chain, and bit
    for bit against the layer followed by qmv_moe_combine_ex."""
    ntok, top_k = 2, 4
    ids, gu, down, x = _mx_layer_case("mxfp8", "mxfp8", x_dtype, ntok, top_k, 760)
    E, K = gu.E, gu.K
    w = qi.router_weights(qi.rng(761), ntok, top_k)
    ids_d, w_d, x_d = to_dev(ids), to_dev(w), act_to_dev(x, x_dtype)
    flags = mx_flags(x_dtype)
    ws = torch.empty(qmv.qmv_moe_layer_combine_workspace_bytes(gu.desc, down.desc, ntok, top_k), dtype=torch.uint8,
                     device=DEV)
    y = torch.full((ntok, K), 7.0, dtype=_out_dtype(x_dtype), device=DEV)
    qmv.qmv_moe_layer_combine(gu.desc, gu.w, down.desc, down.w, x_d, ids_d, w_d, ntok, top_k, ws, y, flags)
    slots, slot_tol = _layer_expected(gu, down, ids, x=x, x_dtype=x_dtype)
    want = oracle.moe_combine(slots, w, ids, E)
    tol = _combine_tol(slots, w, ids, E, stored_err(slots, slot_tol, x_dtype))
    assert_within(_np(y), want, tol, x_dtype, "combined layer")
    ws2 = torch.empty(qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k), dtype=torch.uint8, device=DEV)
    ys = torch.empty(ntok, top_k, K, dtype=_out_dtype(x_dtype), device=DEV)
    qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, x_d, ids_d, ntok, top_k, ws2, ys, flags)
    y2 = torch.full_like(y, -7.0)
    qmv.qmv_moe_combine_ex(down.desc, ys, w_d, ids_d, ntok, top_k, y2, flags)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert status_clean()
