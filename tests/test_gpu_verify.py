"""GPU parity of verify-batch calls: dense matvecs of 5 to 16 tokens (one
weight stream per group of 4 tokens, groups dealt side by side) and gathers /
layers with up to 32 routed (token, slot) pairs -- the speculative-decoding
verify batch that "perf(ggml/hip): optimize ROCMFPX fp3/fp2 MMVQ on RDNA ..."
("Depends on": the batched ROCmFPX MMQ) runs beside the single-token path.
Same bar as the decode tests."""
import numpy as np
import pytest
import torch

import oracle
import qmv_inputs as qi

pytestmark = pytest.mark.gpu

qmv = pytest.importorskip("bit_quantized_moe_gb300")
from qmv_testutil import (DEV, MX_SCALES, Matrices, assert_close, assert_within, bf16_to_np,  # noqa: E402
                          out_of, quantize_on_gpu, status_clean, stored_err, to_dev)
from test_gpu_parity import LUTS, GateUp, _combine_tol, _layer_expected  # noqa: E402


@pytest.mark.parametrize("fmt,N,K", [("mxfp4", 2880, 2880), ("mxfp4", 516, 4096), ("mxfp8", 2880, 2880),
                                     ("cb4", 2048, 7168), ("cb4", 7168, 7168), ("cb3", 1032, 2048)])
@pytest.mark.parametrize("ntok", [5, 8, 13, 16])
def test_verify_dense(fmt, N, K, ntok):
    lo, hi = MX_SCALES.get(fmt, (120, 130))
    m = Matrices(fmt, N, K, 1, [0], seed=N + K + ntok, lut=LUTS.get(fmt), scale_lo=lo, scale_hi=hi)
    g = qi.rng(ntok * 31 + N)
    if fmt in ("mxfp4", "mxfp8"):
        x = qi.normal_bf16_bits(g, (ntok, K))
        y = torch.empty(ntok, N, dtype=torch.bfloat16, device=DEV)
        qmv.qmv_dense(m.desc, m.w, to_dev(x), ntok, y)
        ref = oracle.mx_matvec(fmt, m.codes[0], m.scales[0], x)
        absum = oracle.mx_abs_products(fmt, m.codes[0], m.scales[0], x)
        assert_close(bf16_to_np(y), ref, absum, True, f"{fmt} dense {N}x{K} ntok={ntok}")
    else:
        xq, q, d = quantize_on_gpu(qi.normal_f32(g, (ntok, K)))
        y = torch.empty(ntok, N, dtype=torch.float32, device=DEV)
        qmv.qmv_dense(m.desc, m.w, xq, ntok, y)
        grp = qi.FORMAT_GROUP[fmt]
        ref = oracle.cb_matvec(m.codes[0], m.scales[0], m.lut, grp, q, d)
        absum = oracle.cb_abs_products(m.codes[0], m.scales[0], m.lut, grp, q, d)
        assert_close(y.cpu().numpy(), ref, absum, False, f"{fmt} dense {N}x{K} ntok={ntok}")
    assert status_clean()


@pytest.mark.parametrize("fmt", ["mxfp4", "cb3"])
@pytest.mark.parametrize("ntok,top_k,per_slot", [(8, 4, True), (8, 4, False), (16, 2, True), (6, 5, False)])
def test_verify_gather(fmt, ntok, top_k, per_slot):
    E, N, K = 32, (2880 if fmt == "mxfp4" else 7168), (2880 if fmt == "mxfp4" else 2048)
    g = qi.rng(ntok * 100 + top_k + per_slot)
    ids = qi.topk_ids(g, ntok, top_k, E)
    ids[1, 0] = ids[0, 0]
    ids[-1, -1] = -1
    m = Matrices(fmt, N, K, E, ids.reshape(-1), seed=ntok + top_k, lut=LUTS.get(fmt))
    nvec = ntok * top_k if per_slot else ntok
    if fmt == "mxfp4":
        x = qi.normal_bf16_bits(g, (nvec, K))
        y = torch.full((ntok, top_k, N), 5.0, dtype=torch.bfloat16, device=DEV)
        qmv.qmv_moe_gather(m.desc, m.w, to_dev(x), int(per_slot), to_dev(ids), ntok, top_k, y)
        got = bf16_to_np(y)
    else:
        xq, q, d = quantize_on_gpu(qi.normal_f32(g, (nvec, K)))
        y = torch.full((ntok, top_k, N), 5.0, dtype=torch.float32, device=DEV)
        qmv.qmv_moe_gather(m.desc, m.w, xq, int(per_slot), to_dev(ids), ntok, top_k, y)
        got = y.cpu().numpy().astype(np.float64)
    for t in range(ntok):
        for j in range(top_k):
            e = int(ids[t, j])
            if e < 0:
                assert np.all(got[t, j] == 0)
                continue
            v = t * top_k + j if per_slot else t
            if fmt == "mxfp4":
                ref = oracle.mxfp4_matvec(m.codes[e], m.scales[e], x[v:v + 1])[0]
                absum = oracle.mxfp4_abs_products(m.codes[e], m.scales[e], x[v:v + 1])[0]
            else:
                ref = oracle.cb_matvec(m.codes[e], m.scales[e], m.lut, 16, q[v:v + 1], d[v:v + 1])[0]
                absum = oracle.cb_abs_products(m.codes[e], m.scales[e], m.lut, 16, q[v:v + 1], d[v:v + 1])[0]
            assert_close(got[t, j], ref, absum, out_of(fmt), f"slot ({t},{j}) expert {e}")
    assert status_clean()


@pytest.mark.parametrize("pair", [("mxfp4", "mxfp4", 2880, 2880, 32), ("cb2", "cb3", 2048, 7168, 64)],
                         ids=lambda p: f"{p[0]}-{p[1]}")
def test_verify_layer_combine(pair):
    """An 8-token verify batch through the layer (32 routed slots) and the
    router-weighted combine, against the oracle chain."""
    fmt_gu, fmt_dn, N, K, E = pair
    ntok, top_k = 8, 4
    g = qi.rng(880)
    ids = qi.topk_ids(g, ntok, top_k, E)
    ids[2, 1] = ids[0, 0]
    ids[5, 3] = E + 4
    gu = GateUp(fmt_gu, N, K, E, ids.reshape(-1), seed=881, lut=LUTS.get(fmt_gu))
    down = Matrices(fmt_dn, K, N, E, ids.reshape(-1), seed=882, lut=LUTS.get(fmt_dn))
    w = qi.router_weights(g, ntok, top_k)
    if fmt_gu == "mxfp4":
        x = qi.normal_bf16_bits(g, (ntok, K))
        xin, q, d, dt = to_dev(x), None, None, torch.bfloat16
    else:
        x = None
        xin, q, d = quantize_on_gpu(qi.normal_f32(g, (ntok, K)))
        dt = torch.float32
    ws = torch.empty(qmv.qmv_moe_layer_combine_workspace_bytes(gu.desc, down.desc, ntok, top_k), dtype=torch.uint8,
                     device=DEV)
    y = torch.full((ntok, K), 7.0, dtype=dt, device=DEV)
    qmv.qmv_moe_layer_combine(gu.desc, gu.w, down.desc, down.w, xin, to_dev(ids), to_dev(w), ntok, top_k, ws, y)
    slots, slot_tol = _layer_expected(gu, down, ids, x=x, q=q, d=d)
    want = oracle.moe_combine(slots, w, ids, E)
    out = out_of(fmt_dn)
    tol = _combine_tol(slots, w, ids, E, stored_err(slots, slot_tol, out))
    got = bf16_to_np(y) if dt == torch.bfloat16 else y.cpu().numpy().astype(np.float64)
    assert_within(got, want, tol, out, "combined layer")
    assert status_clean()


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
@pytest.mark.parametrize("N,K", [(1, 32), (17, 96), (130, 1056), (1032, 2048), (4099, 1024), (300, 7168)])
@pytest.mark.parametrize("ntok", [5, 16])
def test_verify_tensor_core_shapes(fmt, N, K, ntok):
    """The tensor-core verify path over ragged row blocks (N not a multiple of
    128), ragged K chunks, K ranges split across cluster ranks, and 5 tokens
    (11 padding columns of the MMA)."""
    lo, hi = MX_SCALES[fmt]
    m = Matrices(fmt, N, K, 1, [0], seed=3 * N + K, scale_lo=lo, scale_hi=hi)
    x = qi.normal_bf16_bits(qi.rng(N + K + ntok), (ntok, K))
    y = torch.full((ntok, N), 9.0, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_dense(m.desc, m.w, to_dev(x), ntok, y)
    ref = oracle.mx_matvec(fmt, m.codes[0], m.scales[0], x)
    absum = oracle.mx_abs_products(fmt, m.codes[0], m.scales[0], x)
    assert_close(bf16_to_np(y), ref, absum, True, f"{fmt} verify {N}x{K} ntok={ntok}")
    assert status_clean()


def test_verify_tensor_core_deterministic_and_chained():
    """Two launches give identical bits; a launch on a side stream after
    another kernel (programmatic dependent launch) and inside a CUDA graph
    gives the same bits as the eager call."""
    N, K, T = 2880, 2880, 12
    m = Matrices("mxfp4", N, K, 1, [0], seed=77)
    x = to_dev(qi.normal_bf16_bits(qi.rng(78), (T, K)))
    y1 = torch.empty(T, N, dtype=torch.bfloat16, device=DEV)
    y2 = torch.empty_like(y1)
    qmv.qmv_dense(m.desc, m.w, x, T, y1)
    qmv.qmv_dense(m.desc, m.w, x, T, y2)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    x2 = torch.empty_like(x)
    y3 = torch.empty_like(y1)
    with torch.cuda.stream(s):
        x2.copy_(x)                      # the verify launch depends on this kernel's output
        qmv.qmv_dense(m.desc, m.w, x2, T, y3, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y3.view(torch.int16))
    g = torch.cuda.CUDAGraph()
    y4 = torch.zeros_like(y1)
    with torch.cuda.graph(g, stream=s):
        qmv.qmv_dense(m.desc, m.w, x2, T, y4, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y4.view(torch.int16))
    assert status_clean()


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
@pytest.mark.parametrize("ntok,top_k,per_slot", [(16, 8, True), (16, 8, False), (8, 8, True), (12, 3, False)])
def test_sorted_gather(fmt, ntok, top_k, per_slot):
    """33..128 routed slots: the sorted tensor-core gather, against the oracle
    per slot. Expert 5 takes 20 slots (two work items of <= 16), ids repeat
    within a token, and invalid ids give zero rows."""
    E, N, K = 32, 520, 2880
    g = qi.rng(ntok * 1000 + top_k * 10 + per_slot)
    ids = qi.topk_ids(g, ntok, top_k, E)
    ids[:, 0] = 5
    if top_k > 1:
        ids[:4, 1] = 5
        ids[-1, -1] = -3
        ids[0, -1] = E
    lo, hi = MX_SCALES[fmt]
    m = Matrices(fmt, N, K, E, ids.reshape(-1), seed=ntok + top_k + 7, scale_lo=lo, scale_hi=hi)
    nvec = ntok * top_k if per_slot else ntok
    x = qi.normal_bf16_bits(g, (nvec, K))
    y = torch.full((ntok, top_k, N), 5.0, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_moe_gather_ex(m.desc, m.w, to_dev(x), int(per_slot), to_dev(ids), ntok, top_k, y, qmv.QMV_FLAG_PATH_TENSOR)
    got = bf16_to_np(y)
    cache = {}
    for t in range(ntok):
        for j in range(top_k):
            e = int(ids[t, j])
            if not (0 <= e < E):
                assert np.all(got[t, j] == 0), (t, j)
                continue
            v = t * top_k + j if per_slot else t
            if (e, v) not in cache:
                cache[(e, v)] = (oracle.mx_matvec(fmt, m.codes[e], m.scales[e], x[v:v + 1])[0],
                                 oracle.mx_abs_products(fmt, m.codes[e], m.scales[e], x[v:v + 1])[0])
            ref, absum = cache[(e, v)]
            assert_close(got[t, j], ref, absum, True, f"slot ({t},{j}) expert {e}")
    assert status_clean()


def test_sorted_gather_prefetch_chain():
    """The sorted gather with QMV_FLAG_PREFETCH_INPUTS after a kernel that
    writes its activations, on a side stream (dependent launch): same bits as
    the plain call; invalid ids still give zero rows."""
    E, N, K, ntok, top_k = 16, 264, 1024, 8, 8
    g = qi.rng(990)
    ids = np.stack([g.permutation(E)[:top_k] for _ in range(ntok)]).astype(np.int32)
    ids[3, 2] = -1
    m = Matrices("mxfp4", N, K, E, ids.reshape(-1), seed=991)
    x = to_dev(qi.normal_bf16_bits(g, (ntok, K)))
    ids_d = to_dev(ids)
    y1 = torch.full((ntok, top_k, N), 3.0, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_moe_gather_ex(m.desc, m.w, x, 0, ids_d, ntok, top_k, y1, qmv.QMV_FLAG_PATH_TENSOR)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    x2 = torch.empty_like(x)
    y2 = torch.full_like(y1, 4.0)
    with torch.cuda.stream(s):
        x2.copy_(x)
        qmv.qmv_moe_gather_ex(m.desc, m.w, x2, 0, ids_d, ntok, top_k, y2,
                              qmv.QMV_FLAG_PREFETCH_INPUTS | qmv.QMV_FLAG_PATH_TENSOR, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.count_nonzero(y2[3, 2].float()).item() == 0
    assert status_clean()


# ---------------------------------------------------------------------------
# Every legal E8M0 byte on the tensor-core path (and the CUDA-core path at 4
# tokens): the scales are applied in fp32 outside the f16 operands
# ---------------------------------------------------------------------------

EXTREME_E8M0 = (0, 1, 2, 3, 127, 253, 254)
# per-token power-of-two magnitudes of the activations, so that rows of the
# largest and the smallest scales both meet tokens that keep their products
# inside fp32's finite range
TOKEN_SHIFTS = (-100, -60, -30, -8, 0, 8, 30, 60, -80, -40, -20, 20, 40, 80, 100, 0)
FP32_TINY = 2.0 ** -140     # fp32 subnormal arithmetic: a few quanta of 2^-149


def _extreme_matrix(fmt, N, K, g):
    """Rows with one scale byte each from EXTREME_E8M0, and rows mixing them
    along K; MXFP8 also gets rows of subnormal E4M3 codes only."""
    codes = qi.format_codes(g, fmt, (N, K))
    scales = np.empty((N, K // 32), np.uint8)
    for r in range(N):
        kind = r % 9
        scales[r] = EXTREME_E8M0[kind] if kind < len(EXTREME_E8M0) else qi.e8m0_choice(g, (K // 32,), EXTREME_E8M0)
    if fmt == "mxfp8":
        sub = np.arange(N) % 4 == 3
        codes[sub] = qi.e4m3_subnormal_codes(g, (int(sub.sum()), K))
    return codes, scales


def _in_range(fmt, codes, scales, x):
    """(token, row) pairs the fp32 kernels can represent: every 32-group's
    sum|w x| and the whole row's stay below 2^120 (the float64 oracle has no
    such limit). Returns the mask [T, N] and sum|w x| [T, N]."""
    Wabs = np.abs(oracle.mxfp4_dequant(codes, scales) if fmt == "mxfp4" else oracle.mxfp8_dequant(codes, scales))
    xa = np.abs(oracle.bf16_bits_to_f64(x))
    N, K = codes.shape
    per_group = np.einsum("ngk,tgk->tng", Wabs.reshape(N, K // 32, 32), xa.reshape(-1, K // 32, 32))
    absum = per_group.sum(-1)
    return (per_group.max(-1) < 2.0 ** 120) & (absum < 2.0 ** 120), absum


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
@pytest.mark.parametrize("ntok", [4, 8, 16])
def test_extreme_scales_dense(fmt, ntok):
    N, K = 264, 1024
    g = qi.rng(2000 + ntok + (7 if fmt == "mxfp8" else 0))
    codes, scales = _extreme_matrix(fmt, N, K, g)
    m = Matrices(fmt, N, K, 1, [], seed=1)
    m.set_expert(0, codes, scales)
    x = qi.scaled_normal_bf16_bits(g, (ntok, K), TOKEN_SHIFTS[:ntok])
    y = torch.full((ntok, N), 3.0, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_dense(m.desc, m.w, to_dev(x), ntok, y)
    ref = oracle.mx_matvec(fmt, codes, scales, x)
    mask, absum = _in_range(fmt, codes, scales, x)
    got = bf16_to_np(y)
    assert_within(got[mask], ref[mask], 1e-3 * absum[mask] + FP32_TINY, "bf16", f"{fmt} ntok={ntok}")
    # every scale byte is checked somewhere
    for e in EXTREME_E8M0:
        rows = np.arange(N)[(np.arange(N) % 9) == EXTREME_E8M0.index(e)]
        assert mask[:, rows].any(), e
    assert status_clean()


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
def test_extreme_scales_sorted_gather(fmt):
    """40 routed slots (8 tokens x top-5) over 4 experts of extreme scales:
    the sorted tensor-core gather, per slot against the oracle."""
    E, N, K, ntok, top_k = 4, 136, 512, 8, 5
    g = qi.rng(2100 + (7 if fmt == "mxfp8" else 0))
    ids = np.stack([np.concatenate([g.permutation(E), [int(g.integers(0, E))]]) for _ in range(ntok)]).astype(np.int32)
    m = Matrices(fmt, N, K, E, [], seed=2)
    mats = {}
    for e in range(E):
        mats[e] = _extreme_matrix(fmt, N, K, g)
        m.set_expert(e, *mats[e])
    x = qi.scaled_normal_bf16_bits(g, (ntok, K), TOKEN_SHIFTS[:ntok])
    y = torch.full((ntok, top_k, N), 3.0, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_moe_gather_ex(m.desc, m.w, to_dev(x), 0, to_dev(ids), ntok, top_k, y, qmv.QMV_FLAG_PATH_TENSOR)
    got = bf16_to_np(y)
    for t in range(ntok):
        for j in range(top_k):
            c, s = mats[int(ids[t, j])]
            ref = oracle.mx_matvec(fmt, c, s, x[t:t + 1])[0]
            mask, absum = _in_range(fmt, c, s, x[t:t + 1])
            assert_within(got[t, j][mask[0]], ref[mask[0]], 1e-3 * absum[0][mask[0]] + FP32_TINY, "bf16",
                          f"slot ({t},{j})")
    assert status_clean()


SPREAD_SETS = (
    (100, 124),        # 24 octaves: 2^-24, f16's smallest subnormal, as the factor of the smaller scale
    (110, 118, 125),   # factors 2^-15 (subnormal) and 2^-7
    (99, 124),         # 25 octaves: recomputed on the CUDA cores
    (230, 254),        # the largest legal scales, 24 octaves apart
    (0, 1, 20),        # the smallest legal scales
    (112, 122),        # the usual range
)


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8"])
@pytest.mark.parametrize("ntok", [8, 16])
def test_verify_scale_spread(fmt, ntok):
    """Rows whose scale bytes span up to 24 octaves take the tensor cores with
    factors 2^(e - e_ref) down to 2^-24; wider rows and rows holding the NaN
    byte 255 are recomputed on the CUDA cores. Per (token, row) against the
    oracle wherever the products stay inside fp32's range."""
    N, K = 264, 2048
    g = qi.rng(2200 + ntok + (7 if fmt == "mxfp8" else 0))
    codes = qi.format_codes(g, fmt, (N, K))
    scales = np.empty((N, K // 32), np.uint8)
    kinds = len(SPREAD_SETS) + 1
    for r in range(N):
        kind = r % kinds
        if kind < len(SPREAD_SETS):
            scales[r] = qi.e8m0_choice(g, (K // 32,), SPREAD_SETS[kind])
        else:
            scales[r] = qi.e8m0_choice(g, (K // 32,), (118, 120))
            scales[r, int(g.integers(0, K // 32))] = 255
    m = Matrices(fmt, N, K, 1, [], seed=3)
    m.set_expert(0, codes, scales)
    x = qi.scaled_normal_bf16_bits(g, (ntok, K), TOKEN_SHIFTS[:ntok])
    y = torch.full((ntok, N), 3.0, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_dense(m.desc, m.w, to_dev(x), ntok, y)
    got = bf16_to_np(y)
    nan_rows = np.arange(N) % kinds == len(SPREAD_SETS)
    assert np.isnan(got[:, nan_rows]).all()
    keep = ~nan_rows
    ref = oracle.mx_matvec(fmt, codes[keep], scales[keep], x)
    mask, absum = _in_range(fmt, codes[keep], scales[keep], x)
    sub = got[:, keep]
    assert_within(sub[mask], ref[mask], 1e-3 * absum[mask] + FP32_TINY, "bf16", f"{fmt} ntok={ntok}")
    for kind in range(len(SPREAD_SETS)):
        rows = (np.arange(N)[keep] % kinds) == kind
        assert mask[:, rows].any(), SPREAD_SETS[kind]
    assert status_clean()


# ---------------------------------------------------------------------------
# Codebook formats on the tensor cores: exact integer block sums per
# (half-)block, the d * 2^(e-127) epilogue in fp32
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt,N,K", [("cb2", 1032, 2048), ("cb3", 7168, 2048), ("cb4", 520, 7168),
                                     ("cb3", 136, 96)])
@pytest.mark.parametrize("ntok", [5, 8, 16])
def test_verify_codebook_block_sums(fmt, N, K, ntok):
    """Dense verify batches of the codebook formats: every integer block sum
    bit-exact against the oracle, y within the tolerance; fp32 activations
    (quantized in the launch) give the same bits as the q8_1 input."""
    grp = qi.FORMAT_GROUP[fmt]
    m = Matrices(fmt, N, K, 1, [0], seed=N + K + ntok, lut=LUTS[fmt])
    g = qi.rng(3000 + ntok + N)
    xf = qi.normal_f32(g, (ntok, K))
    xq, q, d = quantize_on_gpu(xf)
    y = torch.full((ntok, N), 3.0, dtype=torch.float32, device=DEV)
    sums = torch.full((ntok, N, K // grp), -7, dtype=torch.int32, device=DEV)
    qmv.qmv_debug_block_sums(m.desc, m.w, xq, 0, None, ntok, 1, y, sums, flags=qmv.QMV_FLAG_PATH_TENSOR)
    want = oracle.cb_block_sums(m.codes[0], m.lut, q, grp)
    assert np.array_equal(sums.cpu().numpy(), want), "block sums differ from the oracle"
    ref = oracle.cb_matvec(m.codes[0], m.scales[0], m.lut, grp, q, d)
    absum = oracle.cb_abs_products(m.codes[0], m.scales[0], m.lut, grp, q, d)
    assert_close(y.cpu().numpy(), ref, absum, "f32", f"{fmt} {N}x{K} ntok={ntok}")
    y2 = torch.full_like(y, -3.0)
    qmv.qmv_dense_ex(m.desc, m.w, to_dev(xf), ntok, y2, qmv.QMV_FLAG_X_F32 | qmv.QMV_FLAG_PATH_TENSOR)
    y3 = torch.full_like(y, -4.0)
    qmv.qmv_dense_ex(m.desc, m.w, xq, ntok, y3, qmv.QMV_FLAG_PATH_TENSOR)
    # the CUDA-core path (one weight stream per 4 tokens): the same block sums
    y4 = torch.full_like(y, -5.0)
    sums4 = torch.full_like(sums, -8)
    qmv.qmv_debug_block_sums(m.desc, m.w, xq, 0, None, ntok, 1, y4, sums4, flags=qmv.QMV_FLAG_PATH_CUDA_CORES)
    torch.cuda.synchronize()
    assert torch.equal(sums4, sums)
    assert_close(y4.cpu().numpy(), ref, absum, "f32", f"{fmt} {N}x{K} ntok={ntok} CUDA cores")
    assert torch.equal(y2.view(torch.int32), y3.view(torch.int32))
    assert torch.equal(y.view(torch.int32), y3.view(torch.int32))
    assert status_clean()


@pytest.mark.parametrize("fmt,N,K,E,ntok,top_k,per_slot", [
    ("cb3", 7168, 2048, 64, 16, 4, True),     # a DS4 down projection over a 16-token verify batch
    ("cb2", 2048, 7168, 64, 16, 4, False),    # its gate (shared activations)
    ("cb4", 1032, 1024, 16, 16, 8, True),     # 128 slots, experts of up to 16 slots
    ("cb3", 264, 512, 8, 12, 3, False),
])
def test_sorted_gather_codebook(fmt, N, K, E, ntok, top_k, per_slot):
    """33..128 routed slots of a codebook format: the sorted tensor-core
    gather, block sums bit-exact per slot and y within the tolerance;
    repeated experts, an expert of more than 16 slots and invalid ids."""
    grp = qi.FORMAT_GROUP[fmt]
    g = qi.rng(4000 + N + ntok * 10 + top_k)
    ids = np.stack([g.permutation(E)[:top_k] for _ in range(ntok)]).astype(np.int32)
    ids[:, 0] = 1
    ids[:3, 1] = 1 if top_k > 1 else ids[:3, 0]
    ids[-1, -1] = -2
    ids[2, -1] = E + 5
    m = Matrices(fmt, N, K, E, ids.reshape(-1), seed=4001 + N, lut=LUTS[fmt])
    nvec = ntok * top_k if per_slot else ntok
    xf = qi.normal_f32(g, (nvec, K))
    xq, q, d = quantize_on_gpu(xf)
    y = torch.full((ntok, top_k, N), 5.0, dtype=torch.float32, device=DEV)
    sums = torch.full((ntok, top_k, N, K // grp), -7, dtype=torch.int32, device=DEV)
    ids_d = to_dev(ids)
    qmv.qmv_debug_block_sums(m.desc, m.w, xq, int(per_slot), ids_d, ntok, top_k, y, sums, flags=qmv.QMV_FLAG_PATH_TENSOR)
    got_sums, got = sums.cpu().numpy(), y.cpu().numpy()
    for t in range(ntok):
        for j in range(top_k):
            e = int(ids[t, j])
            if not (0 <= e < E):
                assert np.all(got[t, j] == 0) and np.all(got_sums[t, j] == -7), (t, j)
                continue
            v = t * top_k + j if per_slot else t
            assert np.array_equal(got_sums[t, j], oracle.cb_block_sums(m.codes[e], m.lut, q[v:v + 1], grp)[0]), (t, j)
            ref = oracle.cb_matvec(m.codes[e], m.scales[e], m.lut, grp, q[v:v + 1], d[v:v + 1])[0]
            absum = oracle.cb_abs_products(m.codes[e], m.scales[e], m.lut, grp, q[v:v + 1], d[v:v + 1])[0]
            assert_close(got[t, j], ref, absum, "f32", f"slot ({t},{j}) expert {e}")
    y2 = torch.full_like(y, -5.0)
    qmv.qmv_moe_gather_ex(m.desc, m.w, to_dev(xf), int(per_slot), ids_d, ntok, top_k, y2,
                          qmv.QMV_FLAG_X_F32 | qmv.QMV_FLAG_PATH_TENSOR)
    y3 = torch.full_like(y, -6.0)
    qmv.qmv_moe_gather_ex(m.desc, m.w, xq, int(per_slot), ids_d, ntok, top_k, y3, qmv.QMV_FLAG_PATH_TENSOR)
    torch.cuda.synchronize()
    assert torch.equal(y2.view(torch.int32), y3.view(torch.int32))
    assert torch.equal(y.view(torch.int32), y3.view(torch.int32))
    assert status_clean()
