"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bar: bit-exact for the decoded weights, q8_1 codes and scales, and every
integer block sum; max|gpu - oracle| <= 1e-3 * sum|w x| per output element for
the floating-point outputs (plus one bf16 ulp of the result where the output
is bf16). Shapes span several row tiles, ragged row tiles (N = 516, 17, 1) and
ragged K chunks (K = 2880, 96, 32)."""
import numpy as np
import pytest
import torch

import oracle
import qmv_inputs as qi

pytestmark = pytest.mark.gpu

qmv = pytest.importorskip("bit_quantized_moe_gb300")
from qmv_testutil import (DEV, MX_SCALES, Matrices, act_bits, act_to_dev, assert_close,  # noqa: E402
                          assert_within, bf16_to_np, mx_flags, out_of, quantize_on_gpu, status_clean,
                          stored_err, to_dev)

LUTS = {"cb2": qi.LUT_CB2, "cb3": qi.LUT_CB3, "cb4": qi.LUT_CB4}


# ---------------------------------------------------------------------------
# Decode of the packed layout and the activation quantizer (bit-exact)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt", ["mxfp4", "cb2", "cb3", "cb4", "mxfp8"])
@pytest.mark.parametrize("N,K", [(17, 96), (516, 2880), (16, 2048)])
def test_dequant_bit_exact(fmt, N, K):
    m = Matrices(fmt, N, K, 1, [0], seed=N + K, lut=LUTS.get(fmt), scale_lo=0, scale_hi=255)
    out = torch.empty(N, K, dtype=torch.float32, device=DEV)
    qmv.qmv_debug_dequant(m.desc, m.w, 0, out)
    got = out.cpu().numpy()
    if fmt == "mxfp4":
        ref = oracle.mxfp4_dequant(m.codes[0], m.scales[0])
    elif fmt == "mxfp8":
        ref = oracle.mxfp8_dequant(m.codes[0], m.scales[0])
    else:
        ref = oracle.cb_dequant(m.codes[0], m.scales[0], m.lut, qi.FORMAT_GROUP[fmt])
    with np.errstate(over="ignore"):
        ref32 = ref.astype(np.float32)        # fp32 overflow of 6 * 2^127 matches the kernel's fp32 product
    same = (got == ref32) | (np.isnan(got) & np.isnan(ref32))
    assert same.all(), f"{(~same).sum()} decoded weights differ"
    assert status_clean()


def test_dequant_page_tables():
    """The fp3/fp2 code tables printed on the ROCMFPX PR decode exactly through the device LUT path."""
    tables = {"cb3": [0, 1, 2, 4, 0, -1, -2, -4], "cb2": [-1, 0, 1, 2]}
    for fmt, lut in tables.items():
        m = Matrices(fmt, 16, 64, 1, [], seed=1, lut=lut)
        codes = np.tile(np.arange(1 << qi.FORMAT_BITS[fmt], dtype=np.uint8), (16, 64 // (1 << qi.FORMAT_BITS[fmt])))
        m.set_expert(0, codes, np.full((16, 4), 127, dtype=np.uint8))
        out = torch.empty(16, 64, dtype=torch.float32, device=DEV)
        qmv.qmv_debug_dequant(m.desc, m.w, 0, out)
        assert out.cpu().numpy().tolist() == [[float(lut[c]) for c in row] for row in codes]


@pytest.mark.parametrize("nvec,K", [(1, 32), (4, 2048), (16, 2048), (3, 7168)])
def test_q8_quantizer_bit_exact(nvec, K):
    g = qi.rng(nvec * K)
    x = qi.normal_f32(g, (nvec, K)) * np.float32(2.0) ** g.integers(-8, 8, size=(nvec, 1)).astype(np.float32)
    x[0, :32] = 0.0                                   # all-zero block
    if K >= 64:
        x[0, 32:64] = 0.0
        x[0, 32:38] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5]   # exact ties after scaling by 1
        x[0, 64 % K:64 % K + 4] = [1e-40, -3e-39, 2e-38, 5e-39] if K > 64 else x[0, 0:4]
    _, q, d = quantize_on_gpu(x)
    q_ref, d_ref = oracle.q8_1_quantize(x)
    assert np.array_equal(q, q_ref)
    assert np.array_equal(d, d_ref)
    if K >= 64:
        assert q[0, 32:38].tolist() == [127, 3, -3, 1, -1, 2]


# ---------------------------------------------------------------------------
# MXFP4 x bf16
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K", [(1, 32), (17, 96), (516, 2880), (2880, 2880), (48, 4096)])
@pytest.mark.parametrize("ntok", [1, 2, 3, 4])
def test_mxfp4_dense(N, K, ntok):
    m = Matrices("mxfp4", N, K, 1, [0], seed=7 * N + K)
    x = qi.normal_bf16_bits(qi.rng(ntok + N), (ntok, K))
    y = torch.empty(ntok, N, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_dense(m.desc, m.w, to_dev(x), ntok, y)
    ref = oracle.mxfp4_matvec(m.codes[0], m.scales[0], x)
    absum = oracle.mxfp4_abs_products(m.codes[0], m.scales[0], x)
    assert_close(bf16_to_np(y), ref, absum, True, f"mxfp4 dense {N}x{K} ntok={ntok}")
    assert status_clean()


@pytest.mark.parametrize("N,K", [(516, 2880), (2880, 2880)])
@pytest.mark.parametrize("ntok,top_k,per_slot", [(1, 4, False), (1, 4, True), (4, 4, False), (4, 4, True),
                                                 (2, 8, True), (3, 1, False)])
def test_mxfp4_gather(N, K, ntok, top_k, per_slot):
    E = 32
    g = qi.rng(N + 10 * ntok + top_k)
    ids = qi.topk_ids(g, ntok, top_k, E)
    m = Matrices("mxfp4", N, K, E, ids.reshape(-1), seed=N + top_k)
    nvec = ntok * top_k if per_slot else ntok
    x = qi.normal_bf16_bits(g, (nvec, K))
    y = torch.empty(ntok, top_k, N, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_moe_gather(m.desc, m.w, to_dev(x), int(per_slot), to_dev(ids), ntok, top_k, y)
    got = bf16_to_np(y)
    for t in range(ntok):
        for j in range(top_k):
            e = int(ids[t, j])
            v = t * top_k + j if per_slot else t
            ref = oracle.mxfp4_matvec(m.codes[e], m.scales[e], x[v:v + 1])[0]
            absum = oracle.mxfp4_abs_products(m.codes[e], m.scales[e], x[v:v + 1])[0]
            assert_close(got[t, j], ref, absum, True, f"slot ({t},{j}) expert {e}")
    assert status_clean()


def test_mxfp4_gather_invalid_and_repeated_ids():
    """Invalid ids give zero rows; an expert repeated across slots or tokens is still right."""
    E, N, K = 8, 516, 2880
    ids = np.array([[3, 3, -1, 8], [3, 5, 7, 100]], dtype=np.int32)
    m = Matrices("mxfp4", N, K, E, ids.reshape(-1), seed=5)
    x = qi.normal_bf16_bits(qi.rng(9), (8, K))
    for per_slot in (0, 1):
        y = torch.full((2, 4, N), 7.0, dtype=torch.bfloat16, device=DEV)
        qmv.qmv_moe_gather(m.desc, m.w, to_dev(x), per_slot, to_dev(ids), 2, 4, y)
        ref = oracle.mxfp4_moe_gather(np.stack([m.codes.get(e, np.zeros((N, K), np.uint8)) for e in range(E)]),
                                      np.stack([m.scales.get(e, np.zeros((N, K // 32), np.uint8)) for e in range(E)]),
                                      x, ids, bool(per_slot))
        got = bf16_to_np(y)
        for t in range(2):
            for j in range(4):
                e = int(ids[t, j])
                if 0 <= e < E:
                    v = t * 4 + j if per_slot else t
                    absum = oracle.mxfp4_abs_products(m.codes[e], m.scales[e], x[v:v + 1])[0]
                    assert_close(got[t, j], ref[t, j], absum, True, f"({t},{j})")
                else:
                    assert np.all(got[t, j] == 0.0)
    assert status_clean()


def test_mxfp4_special_scales():
    """E8M0 255 decodes to NaN; 0 to 2^-127 (kept, not flushed)."""
    N, K = 16, 64
    m = Matrices("mxfp4", N, K, 1, [], seed=3)
    codes = np.full((N, K), 2, dtype=np.uint8)          # every weight 1.0
    scales = np.full((N, 2), 127, dtype=np.uint8)
    scales[3, :] = 255
    scales[5, :] = 0
    m.set_expert(0, codes, scales)
    x = np.full((1, K), 0x3F80, dtype=np.uint16)         # all ones
    y = torch.empty(1, N, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_dense(m.one, m.w, to_dev(x), 1, y)
    got = bf16_to_np(y)[0]
    assert np.isnan(got[3])
    assert got[0] == 64.0
    ref5 = 64.0 * 2.0 ** -127
    assert abs(got[5] - ref5) <= ref5 * 2 ** -8


# ---------------------------------------------------------------------------
# Codebook formats x q8_1 (integer block sums bit-exact)
# ---------------------------------------------------------------------------

def _cb_check(fmt, m, x, ids, per_slot, ntok, top_k, what):
    group = qi.FORMAT_GROUP[fmt]
    xq, q, d = quantize_on_gpu(x)
    q_ref, d_ref = oracle.q8_1_quantize(x)
    assert np.array_equal(q, q_ref) and np.array_equal(d, d_ref)
    N, K = m.N, m.K
    slots = ntok * top_k if ids is not None else ntok
    y = torch.empty(slots, N, dtype=torch.float32, device=DEV)
    sums = torch.full((slots, N, K // group), -7, dtype=torch.int32, device=DEV)
    y2 = torch.empty_like(y)
    if ids is None:
        qmv.qmv_dense(m.desc, m.w, xq, ntok, y2)
        qmv.qmv_debug_block_sums(m.desc, m.w, xq, 0, None, ntok, 1, y, sums)
    else:
        qmv.qmv_moe_gather(m.desc, m.w, xq, int(per_slot), to_dev(ids), ntok, top_k, y2)
        qmv.qmv_debug_block_sums(m.desc, m.w, xq, int(per_slot), to_dev(ids), ntok, top_k, y, sums)
    got_y, got_y2, got_s = y.cpu().numpy(), y2.cpu().numpy(), sums.cpu().numpy()
    assert np.array_equal(got_y, got_y2), "debug and production kernels disagree"
    for s in range(slots):
        if ids is None:
            e, v = 0, s
        else:
            t, j = divmod(s, top_k)
            e = int(ids[t, j])
            v = s if per_slot else t
            if not (0 <= e < m.E):
                assert np.all(got_y2[s] == 0.0)
                continue
        ref_s = oracle.cb_block_sums(m.codes[e], m.lut, q_ref[v:v + 1], group)[0]
        assert np.array_equal(got_s[s], ref_s), f"{what}: block sums differ for slot {s}"
        ref = oracle.cb_matvec(m.codes[e], m.scales[e], m.lut, group, q_ref[v:v + 1], d_ref[v:v + 1])[0]
        absum = oracle.cb_abs_products(m.codes[e], m.scales[e], m.lut, group, q_ref[v:v + 1], d_ref[v:v + 1])[0]
        assert_close(got_y2[s], ref, absum, False, f"{what} slot {s}")


@pytest.mark.parametrize("fmt", ["cb2", "cb3", "cb4"])
@pytest.mark.parametrize("N,K", [(1, 32), (17, 96), (516, 2880), (64, 7168)])
@pytest.mark.parametrize("ntok", [1, 4])
def test_cb_dense(fmt, N, K, ntok):
    m = Matrices(fmt, N, K, 1, [0], seed=N + K + ntok, lut=LUTS[fmt])
    x = qi.normal_f32(qi.rng(N * ntok), (ntok, K))
    _cb_check(fmt, m, x, None, False, ntok, 1, f"{fmt} dense {N}x{K}")
    assert status_clean()


@pytest.mark.parametrize("fmt", ["cb2", "cb3", "cb4"])
@pytest.mark.parametrize("ntok,top_k,per_slot", [(1, 4, False), (4, 4, True), (2, 3, False)])
def test_cb_gather(fmt, ntok, top_k, per_slot):
    E, N, K = 64, 272, 2048
    g = qi.rng(ntok * 10 + top_k)
    ids = qi.topk_ids(g, ntok, top_k, E)
    if ntok == 4:
        ids[2, 1] = ids[0, 0]           # an expert shared by two tokens
        ids[3, 0] = -5                  # an invalid id
    m = Matrices(fmt, N, K, E, ids.reshape(-1), seed=E + ntok, lut=LUTS[fmt])
    nvec = ntok * top_k if per_slot else ntok
    x = qi.normal_f32(g, (nvec, K))
    _cb_check(fmt, m, x, ids, per_slot, ntok, top_k, f"{fmt} gather")
    assert status_clean()


@pytest.mark.parametrize("fmt,lut", [("cb3", [0, 1, 2, 4, 0, -1, -2, -4]), ("cb2", [-1, 0, 1, 2]),
                                     ("cb4", [-128, -100, -7, -5, -4, -3, -2, -1, 0, 2, 3, 4, 5, 7, 99, 127])])
def test_cb_other_codebooks(fmt, lut):
    """The page's fp3/fp2 tables and a full-range int8 16-entry table."""
    m = Matrices(fmt, 48, 1024, 1, [0], seed=11, lut=lut)
    x = qi.normal_f32(qi.rng(12), (2, 1024))
    _cb_check(fmt, m, x, None, False, 2, 1, f"{fmt} lut {lut}")


# ---------------------------------------------------------------------------
# SwiGLU and one MXFP4 MoE layer
# ---------------------------------------------------------------------------

# Absolute error of fp32 SwiGLU arithmetic whose result is an fp32 subnormal:
# exp(z) for z < -87 is subnormal (quantum 2^-149) and z * exp(z) scales its
# rounding by |z| <= 104 before fp32 underflows entirely.
FP32_TINY = 2.0 ** -140


@pytest.mark.parametrize("n", [1, 8, 11520, 11527])
def test_swiglu(n):
    g = qi.rng(n)
    gb = qi.normal_bf16_bits(g, (n,))
    ub = qi.normal_bf16_bits(g, (n,))
    if n > 8:
        # gate values where exp(-g) overflows fp32 while silu(g) * u is still a normal value
        gb[:16] = oracle.f64_to_bf16_bits(-np.linspace(86.0, 100.0, 16))
    h = torch.empty(n, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_swiglu_bf16(to_dev(gb), to_dev(ub), h, n)
    ref = oracle.swiglu(oracle.bf16_bits_to_f64(gb), oracle.bf16_bits_to_f64(ub))
    got = bf16_to_np(h)
    # fp32 arithmetic (exp, add, divide, multiply: a few ulp, or a few
    # subnormal quanta at the bottom of fp32's range), then bf16 rounding
    assert_within(got, ref, 1e-6 * np.abs(ref) + FP32_TINY, "bf16", "swiglu")


def test_mxfp4_moe_layer_chain():
    """gate, up (gather, shared x) -> SwiGLU -> down (gather, per-slot h): a full layer at 2880."""
    E, N, K, top_k = 32, 2880, 2880, 4
    g = qi.rng(21)
    ids = qi.topk_ids(g, 1, top_k, E)
    gate = Matrices("mxfp4", N, K, E, ids[0], seed=22)
    up = Matrices("mxfp4", N, K, E, ids[0], seed=23)
    down = Matrices("mxfp4", N, K, E, ids[0], seed=24)
    x = qi.normal_bf16_bits(g, (1, K))
    ids_d, x_d = to_dev(ids), to_dev(x)
    yg = torch.empty(1, top_k, N, dtype=torch.bfloat16, device=DEV)
    yu = torch.empty_like(yg)
    h = torch.empty_like(yg)
    y = torch.empty_like(yg)
    qmv.qmv_moe_gather(gate.desc, gate.w, x_d, 0, ids_d, 1, top_k, yg)
    qmv.qmv_moe_gather(up.desc, up.w, x_d, 0, ids_d, 1, top_k, yu)
    qmv.qmv_swiglu_bf16(yg, yu, h, top_k * N)
    qmv.qmv_moe_gather(down.desc, down.w, h, 1, ids_d, 1, top_k, y)

    def full(mm):
        cs = np.zeros((E, N, K), np.uint8)
        ss = np.zeros((E, N, K // 32), np.uint8)
        for e in mm.codes:
            cs[e], ss[e] = mm.codes[e], mm.scales[e]
        return cs, ss
    ref = oracle.mxfp4_moe_layer(full(gate), full(up), full(down), x, ids)
    # gate/up: per-output tolerance
    for name, got, refv, mm in (("gate", yg, ref["g_bits"], gate), ("up", yu, ref["u_bits"], up)):
        for j in range(top_k):
            e = int(ids[0, j])
            r = oracle.mxfp4_matvec(mm.codes[e], mm.scales[e], x)[0]
            absum = oracle.mxfp4_abs_products(mm.codes[e], mm.scales[e], x)[0]
            assert_close(bf16_to_np(got)[0, j], r, absum, True, f"{name} slot {j}")
    # h, stage-wise: the SwiGLU kernel on the GPU's own bf16 g and u (fp32
    # arithmetic, then one bf16 rounding), every element
    hg = bf16_to_np(h)[0]
    stage = oracle.swiglu(bf16_to_np(yg)[0], bf16_to_np(yu)[0])
    assert_within(hg, stage, 1e-6 * np.abs(stage) + FP32_TINY, "bf16", "h stage-wise")
    # h, chain-wise: against silu(g) * u of the exact g and u, their matvec
    # bounds and bf16 storage propagated through SwiGLU, every element
    gx = np.stack([oracle.mxfp4_matvec(gate.codes[int(e)], gate.scales[int(e)], x)[0] for e in ids[0]])
    ux = np.stack([oracle.mxfp4_matvec(up.codes[int(e)], up.scales[int(e)], x)[0] for e in ids[0]])
    eg = stored_err(gx, 1e-3 * np.stack([oracle.mxfp4_abs_products(gate.codes[int(e)], gate.scales[int(e)], x)[0]
                                         for e in ids[0]]), "bf16")
    eu = stored_err(ux, 1e-3 * np.stack([oracle.mxfp4_abs_products(up.codes[int(e)], up.scales[int(e)], x)[0]
                                         for e in ids[0]]), "bf16")
    hx = oracle.swiglu(gx, ux)
    assert_within(hg, hx, oracle.swiglu_tolerance(gx, ux, eg, eu) + 1e-6 * np.abs(hx) + FP32_TINY, "bf16", "h chain-wise")
    # down: against the oracle chain (its own h)
    for j in range(top_k):
        e = int(ids[0, j])
        absum = oracle.mxfp4_abs_products(down.codes[e], down.scales[e], ref["h_rows_bits"][j:j + 1])[0]
        assert_close(bf16_to_np(y)[0, j], ref["y"][0, j], absum, True, f"down slot {j}")
    assert status_clean()


# ---------------------------------------------------------------------------
# Determinism and full-size configurations (sampled outputs)
# ---------------------------------------------------------------------------

def test_two_runs_bit_identical():
    E, N, K = 32, 2880, 2880
    ids = qi.topk_ids(qi.rng(31), 1, 4, E)
    m = Matrices("mxfp4", N, K, E, ids[0], seed=32)
    x = to_dev(qi.normal_bf16_bits(qi.rng(33), (4, K)))
    outs = []
    for _ in range(2):
        y = torch.empty(1, 4, N, dtype=torch.bfloat16, device=DEV)
        qmv.qmv_moe_gather(m.desc, m.w, x, 1, to_dev(ids), 1, 4, y)
        outs.append(y.view(torch.int16).cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    c = Matrices("cb3", 7168, 2048, 1, [0], seed=34, lut=qi.LUT_CB3)
    xq, _, _ = quantize_on_gpu(qi.normal_f32(qi.rng(35), (4, 2048)))
    outs = []
    for _ in range(2):
        y = torch.empty(4, 7168, dtype=torch.float32, device=DEV)
        qmv.qmv_dense(c.desc, c.w, xq, 4, y)
        outs.append(y.cpu().numpy())
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_config2_full_size():
    """256 experts x 2048 x 7168 CB2 gate and up, 4 ids, ntok = 1 (full shapes)."""
    r = qi.CONFIG2
    g = qi.rng(r.seed)
    ids = qi.topk_ids(g, 1, r.top_k, r.n_experts)
    x = qi.normal_f32(g, (1, r.K))
    for proj in ("gate", "up"):
        m = Matrices("cb2", r.N, r.K, r.n_experts, ids[0], seed=r.seed + (proj == "up"), lut=r.lut)
        _cb_check("cb2", m, x, ids, False, 1, r.top_k, f"config2 {proj}")
    assert status_clean()


def test_config3_full_size():
    """256 experts x 7168 x 2048 CB3 down, ntok = 4 tokens x top-4 independent ids, per-slot q8."""
    r = qi.CONFIG3
    g = qi.rng(r.seed)
    ids = qi.topk_ids(g, r.ntok, r.top_k, r.n_experts)
    m = Matrices("cb3", r.N, r.K, r.n_experts, ids.reshape(-1), seed=r.seed, lut=r.lut)
    x = qi.normal_f32(g, (r.ntok * r.top_k, r.K))
    _cb_check("cb3", m, x, ids, True, r.ntok, r.top_k, "config3")
    assert status_clean()


@pytest.mark.parametrize("N,K", qi.CONFIG4_SHAPES)
def test_config4_full_size_sampled_rows(N, K):
    """Dense CB4 7168x7168 and 2048x7168 at ntok 1..4: every output compared on sampled rows,
    block sums on the same rows bit-exact."""
    r = qi.config4(N, K, 4)
    m = Matrices("cb4", N, K, 1, [0], seed=r.seed + N, lut=r.lut)
    g = qi.rng(N)
    rows = np.unique(np.concatenate([g.choice(N, 256, replace=False), [0, 15, 16, N - 1]]))
    for ntok in qi.CONFIG4_NTOKS:
        x = qi.normal_f32(g, (ntok, K))
        xq, q, d = quantize_on_gpu(x)
        y = torch.empty(ntok, N, dtype=torch.float32, device=DEV)
        sums = torch.empty(ntok, N, K // 32, dtype=torch.int32, device=DEV)
        qmv.qmv_debug_block_sums(m.desc, m.w, xq, 0, None, ntok, 1, y, sums)
        got_s = sums.cpu().numpy()[:, rows]
        got_y = y.cpu().numpy()[:, rows]
        cs, ss = m.codes[0][rows], m.scales[0][rows]
        assert np.array_equal(got_s, oracle.cb_block_sums(cs, m.lut, q, 32))
        ref = oracle.cb_matvec(cs, ss, m.lut, 32, q, d)
        absum = oracle.cb_abs_products(cs, ss, m.lut, 32, q, d)
        assert_close(got_y, ref, absum, False, f"config4 {N}x{K} ntok={ntok}")
    assert status_clean()


# ---------------------------------------------------------------------------
# Failure detection without a fault: a bounded wait runs out
# ---------------------------------------------------------------------------

def test_bounded_wait_times_out_and_context_survives():
    assert qmv.qmv_device_status(clear=True) == 0
    qmv.qmv_debug_wait_probe(20_000_000)          # 20 ms on a barrier nothing completes
    torch.cuda.synchronize()
    assert qmv.qmv_device_status(clear=True) == 8
    assert qmv.qmv_device_status() == 0
    # the context is still usable
    m = Matrices("mxfp4", 16, 64, 1, [0], seed=1)
    x = qi.normal_bf16_bits(qi.rng(2), (1, 64))
    y = torch.empty(1, 16, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_dense(m.desc, m.w, to_dev(x), 1, y)
    ref = oracle.mxfp4_matvec(m.codes[0], m.scales[0], x)
    assert_close(bf16_to_np(y), ref, oracle.mxfp4_abs_products(m.codes[0], m.scales[0], x), True, "after probe")


# ---------------------------------------------------------------------------
# Launch flags: prefetching weights/ids before the dependent-launch wait
# ---------------------------------------------------------------------------

def test_prefetch_flag_matches_plain_path_in_a_dependent_chain():
    """gate, up (prefetch), SwiGLU, down (prefetch, reads the SwiGLU output) on
    one stream: results bit-identical to the same chain without the flag."""
    E, N, K, N_down, top_k = 16, 2880, 2880, 516, 4
    g = qi.rng(41)
    ids = to_dev(qi.topk_ids(g, 1, top_k, E))
    mats = [Matrices("mxfp4", N, K, E, range(E), seed=42 + i) for i in range(2)]
    mats.append(Matrices("mxfp4", N_down, N, E, range(E), seed=44))
    x = to_dev(qi.normal_bf16_bits(g, (1, K)))
    outs = []
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for flags in (0, qmv.QMV_FLAG_PREFETCH_INPUTS, 0, qmv.QMV_FLAG_PREFETCH_INPUTS):
            yg = torch.empty(1, top_k, N, dtype=torch.bfloat16, device=DEV)
            yu, h = torch.empty_like(yg), torch.empty_like(yg)
            y = torch.empty(1, top_k, N_down, dtype=torch.bfloat16, device=DEV)
            qmv.qmv_moe_gather(mats[0].desc, mats[0].w, x, 0, ids, 1, top_k, yg)
            qmv.qmv_moe_gather_ex(mats[1].desc, mats[1].w, x, 0, ids, 1, top_k, yu, flags)
            qmv.qmv_swiglu_bf16(yg, yu, h, top_k * N)
            qmv.qmv_moe_gather_ex(mats[2].desc, mats[2].w, h, 1, ids, 1, top_k, y, flags)
            outs.append(y.view(torch.int16).clone())
    s.synchronize()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    assert status_clean()


def test_dense_ex_prefetch_matches():
    m = Matrices("cb4", 520, 7168, 1, [0], seed=43, lut=qi.LUT_CB4)
    xq, _, _ = quantize_on_gpu(qi.normal_f32(qi.rng(44), (3, 7168)))
    y0 = torch.empty(3, 520, dtype=torch.float32, device=DEV)
    y1 = torch.empty_like(y0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qmv.qmv_dense(m.desc, m.w, xq, 3, y0)
        qmv.qmv_dense_ex(m.desc, m.w, xq, 3, y1, qmv.QMV_FLAG_PREFETCH_INPUTS)
    s.synchronize()
    assert torch.equal(y0.view(torch.int32), y1.view(torch.int32))


# ---------------------------------------------------------------------------
# Gate/up/SwiGLU fusion
# ---------------------------------------------------------------------------

class GateUp:
    """Gate and up expert sets packed together; only `experts` hold data."""

    def __init__(self, fmt, N, K, E, experts, seed, lut=None, scale_lo=120, scale_hi=130):
        self.fmt, self.N, self.K, self.E, self.lut = fmt, N, K, E, (list(lut) if lut else None)
        self.desc = qmv.wdesc(fmt, N, K, E, lut)
        one = qmv.wdesc(fmt, N, K, 1, lut)
        eb = qmv.qmv_packed_gate_up_expert_bytes(self.desc)
        self.w = torch.zeros(E * eb, dtype=torch.uint8, device=DEV)
        g = qi.rng(seed)
        bits, grp = qi.FORMAT_BITS[fmt], qi.FORMAT_GROUP[fmt]
        self.cg, self.sg, self.cu, self.su = {}, {}, {}, {}
        for e in sorted(set(int(v) for v in experts if 0 <= int(v) < E)):
            self.cg[e], self.cu[e] = qi.format_codes(g, fmt, (N, K)), qi.format_codes(g, fmt, (N, K))
            self.sg[e] = qi.e8m0(g, (N, K // grp), scale_lo, scale_hi)
            self.su[e] = qi.e8m0(g, (N, K // grp), scale_lo, scale_hi)
            p = qmv.qmv_pack_gate_up(one, oracle.pack_codes(fmt, self.cg[e][None]), self.sg[e][None],
                                     oracle.pack_codes(fmt, self.cu[e][None]), self.su[e][None])
            self.w[e * eb:(e + 1) * eb] = torch.from_numpy(p).to(DEV)

    def matvecs(self, xin, q=None, d=None, x_dtype="bf16"):
        """(gate, up, gate |w x|, up |w x|) callables of (expert, token) for the oracle."""
        if self.fmt in ("mxfp4", "mxfp8"):
            f = self.fmt
            mv = lambda c, s: (lambda e, t: oracle.mx_matvec(f, c[e], s[e], xin[t:t + 1], x_dtype)[0])
            ab = lambda c, s: (lambda e, t: oracle.mx_abs_products(f, c[e], s[e], xin[t:t + 1], x_dtype)[0])
        else:
            grp = qi.FORMAT_GROUP[self.fmt]
            mv = lambda c, s: (lambda e, t: oracle.cb_matvec(c[e], s[e], self.lut, grp, q[t:t + 1], d[t:t + 1])[0])
            ab = lambda c, s: (lambda e, t: oracle.cb_abs_products(c[e], s[e], self.lut, grp, q[t:t + 1],
                                                                   d[t:t + 1])[0])
        return mv(self.cg, self.sg), mv(self.cu, self.su), ab(self.cg, self.sg), ab(self.cu, self.su)


def check_gate_up(m, ids, h_gpu, xin, q=None, d=None, x_dtype="bf16"):
    gm, um, ga, ua = m.matvecs(xin, q, d, x_dtype)
    h, gv, uv = oracle.moe_gate_up_swiglu(gm, um, m.E, ids, m.N)
    tg = oracle.moe_gather(ga, m.E, ids, False, m.N) * 1e-3
    tu = oracle.moe_gather(ua, m.E, ids, False, m.N) * 1e-3
    # the matvec bounds propagated through SwiGLU, plus its fp32 arithmetic;
    # the stored h (bf16 / fp16 for the MX formats) is that result rounded
    tol = oracle.swiglu_tolerance(gv, uv, tg, tu) + 1e-6 * np.abs(h) + FP32_TINY
    assert_within(h_gpu, h, tol, out_of(m.fmt, x_dtype), "fused gate/up")


@pytest.mark.parametrize("N,ntok,top_k", [(2880, 1, 4), (516, 2, 4), (515, 1, 3), (64, 4, 2)])
def test_mxfp4_gate_up_swiglu(N, ntok, top_k):
    E, K = 32, 2880
    g = qi.rng(N + ntok)
    ids = qi.topk_ids(g, ntok, top_k, E)
    if ntok > 1:
        ids[1, 0] = ids[0, 0]           # shared expert
        ids[-1, -1] = 77                # invalid id
    m = GateUp("mxfp4", N, K, E, ids.reshape(-1), seed=N)
    x = qi.normal_bf16_bits(g, (ntok, K))
    h = torch.full((ntok, top_k, N), 3.0, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_moe_gate_up_swiglu(m.desc, m.w, to_dev(x), to_dev(ids), ntok, top_k, h)
    check_gate_up(m, ids, bf16_to_np(h), x)
    assert status_clean()


@pytest.mark.parametrize("fmt", ["cb2", "cb3", "cb4"])
def test_cb_gate_up_swiglu(fmt):
    E, N, K, ntok, top_k = 64, 2048, 7168 if fmt == "cb2" else 2048, 1, 4
    g = qi.rng(7)
    ids = qi.topk_ids(g, ntok, top_k, E)
    m = GateUp(fmt, N, K, E, ids.reshape(-1), seed=8, lut=LUTS[fmt])
    xq, q, d = quantize_on_gpu(qi.normal_f32(g, (ntok, K)))
    h = torch.empty(ntok, top_k, N, dtype=torch.float32, device=DEV)
    qmv.qmv_moe_gate_up_swiglu(m.desc, m.w, xq, to_dev(ids), ntok, top_k, h)
    check_gate_up(m, ids, h.cpu().numpy().astype(np.float64), None, q, d)
    assert status_clean()


# ---------------------------------------------------------------------------
# One MoE layer: fused gate/up/SwiGLU, then down on the per-slot h
# ---------------------------------------------------------------------------

MX = ("mxfp4", "mxfp8")


def _mx_dequant(fmt, codes, scales):
    return oracle.mxfp4_dequant(codes, scales) if fmt == "mxfp4" else oracle.mxfp8_dequant(codes, scales)


def _layer_expected(gu, down, ids, x=None, q=None, d=None, x_dtype="bf16"):
    """Oracle chain and the per-output bound on the kernel's fp32 y (before
    its storage rounding, which the callers check with the stored type). h
    differs from the GPU's by the propagated SwiGLU bound plus its storage
    rounding (a bf16 ulp, or an fp16 one, for the MX formats; one q8_1
    quantum of its block for the codebooks)."""
    gm, um, ga, ua = gu.matvecs(x, q, d, x_dtype)
    h, gv, uv = oracle.moe_gate_up_swiglu(gm, um, gu.E, ids, gu.N)
    tol_h = oracle.swiglu_tolerance(gv, uv, oracle.moe_gather(ga, gu.E, ids, False, gu.N) * 1e-3,
                                    oracle.moe_gather(ua, gu.E, ids, False, gu.N) * 1e-3)
    ntok, top_k = ids.shape
    rows = h.reshape(ntok * top_k, gu.N)
    if gu.fmt in MX:
        hb = oracle.f64_to_bf16_bits(rows) if x_dtype == "bf16" else oracle.f64_to_f16_bits(rows)
        # |GPU h - h| (its fp32 bound, stored rounded) + |hb - h| (the oracle's rounding)
        dh = (stored_err(rows, tol_h.reshape(rows.shape) + 1e-6 * np.abs(rows) + FP32_TINY, x_dtype)
              + stored_err(rows, 0.0, x_dtype))
        y = oracle.mx_moe_gather(down.fmt,
                                 np.stack([down.codes.get(e, np.zeros((down.N, down.K), np.uint8)) for e in range(down.E)]),
                                 np.stack([down.scales.get(e, np.zeros((down.N, down.K // 32), np.uint8)) for e in range(down.E)]),
                                 hb, ids, True, x_dtype)
    else:
        hq, hd = oracle.q8_1_quantize(rows.astype(np.float32))
        dq = oracle.f16_bits_to_f64(hd)
        dh = tol_h.reshape(rows.shape) + np.repeat(dq, 32, axis=1) * 1.01
        grp = qi.FORMAT_GROUP[down.fmt]
        y = oracle.cb_moe_gather(np.stack([down.codes.get(e, np.zeros((down.N, down.K), np.uint8)) for e in range(down.E)]),
                                 np.stack([down.scales.get(e, np.zeros((down.N, down.K // grp), np.uint8)) for e in range(down.E)]),
                                 down.lut, grp, hq, hd, ids, True)
    tol = np.zeros_like(y)
    for t in range(ntok):
        for j in range(top_k):
            e, s = int(ids[t, j]), t * top_k + j
            if not (0 <= e < down.E):
                continue
            if down.fmt in MX:
                Wabs = np.abs(_mx_dequant(down.fmt, down.codes[e], down.scales[e]))
                base = Wabs @ np.abs(oracle.act_bits_to_f64(hb[s], x_dtype))
            else:
                Wabs = np.abs(oracle.cb_dequant(down.codes[e], down.scales[e], down.lut, grp))
                base = Wabs @ np.abs(hq[s].astype(np.float64) * np.repeat(dq[s], 32))
            tol[t, j] = 1e-3 * base + Wabs @ dh[s]
    return y, tol


def test_mxfp4_moe_layer():
    E, N, K, top_k = 32, 2880, 2880, 4
    for ntok in (1, 2):
        g = qi.rng(60 + ntok)
        ids = qi.topk_ids(g, ntok, top_k, E)
        gu = GateUp("mxfp4", N, K, E, ids.reshape(-1), seed=61)
        down = Matrices("mxfp4", K, N, E, ids.reshape(-1), seed=62)
        x = qi.normal_bf16_bits(g, (ntok, K))
        ws = torch.empty(qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k), dtype=torch.uint8, device=DEV)
        y = torch.empty(ntok, top_k, K, dtype=torch.bfloat16, device=DEV)
        qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, to_dev(x), to_dev(ids), ntok, top_k, ws, y)
        want, tol = _layer_expected(gu, down, ids, x=x)
        assert_within(bf16_to_np(y), want, tol, "bf16", "layer")
    assert status_clean()


def test_cb_moe_layer_ds4_shapes():
    """CB2 gate/up 2048 x 7168, q8_1 of h, CB3 down 7168 x 2048 (the DS4 expert shapes)."""
    E, top_k, ntok = 64, 4, 1
    g = qi.rng(70)
    ids = qi.topk_ids(g, ntok, top_k, E)
    gu = GateUp("cb2", 2048, 7168, E, ids.reshape(-1), seed=71, lut=qi.LUT_CB2)
    down = Matrices("cb3", 7168, 2048, E, ids.reshape(-1), seed=72, lut=qi.LUT_CB3)
    xq, q, d = quantize_on_gpu(qi.normal_f32(g, (ntok, 7168)))
    ws = torch.empty(qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k), dtype=torch.uint8, device=DEV)
    y = torch.empty(ntok, top_k, 7168, dtype=torch.float32, device=DEV)
    qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, xq, to_dev(ids), ntok, top_k, ws, y)
    want, tol = _layer_expected(gu, down, ids, q=q, d=d)
    assert_within(y.cpu().numpy(), want, tol, "f32", "layer")
    assert status_clean()


# ---------------------------------------------------------------------------
# Layers across format pairs, token counts and routing edge cases
# ---------------------------------------------------------------------------

LAYER_PAIRS = [("mxfp4", "mxfp4", 2880, 2880, 32), ("cb2", "cb3", 2048, 7168, 64), ("cb4", "cb4", 1024, 2048, 16)]


def _layer_case(fmt_gu, fmt_dn, N, K, E, ntok, top_k, seed):
    g = qi.rng(seed)
    ids = qi.topk_ids(g, ntok, top_k, E)
    if ntok > 1:
        ids[1, 0] = ids[0, 0]       # an expert shared by two tokens
        ids[-1, -1] = -1            # an invalid id: zero output row
    gu = GateUp(fmt_gu, N, K, E, ids.reshape(-1), seed=seed + 1, lut=LUTS.get(fmt_gu))
    down = Matrices(fmt_dn, K, N, E, ids.reshape(-1), seed=seed + 2, lut=LUTS.get(fmt_dn))
    if fmt_gu == "mxfp4":
        x = qi.normal_bf16_bits(g, (ntok, K))
        return ids, gu, down, x, to_dev(x), None, None, None, torch.bfloat16
    xf = qi.normal_f32(g, (ntok, K))
    xin, q, d = quantize_on_gpu(xf)
    return ids, gu, down, None, xin, q, d, to_dev(xf), torch.float32


@pytest.mark.parametrize("pair", LAYER_PAIRS, ids=lambda p: f"{p[0]}-{p[1]}")
@pytest.mark.parametrize("ntok,top_k", [(1, 4), (2, 4), (4, 2)])
def test_layer_format_pairs(pair, ntok, top_k):
    """qmv_moe_layer against the oracle chain; codebook layers also from fp32
    x (QMV_FLAG_X_F32), which must equal the q8_1 input bit for bit."""
    fmt_gu, fmt_dn, N, K, E = pair
    ids, gu, down, x, xin, q, d, xf, dt = _layer_case(fmt_gu, fmt_dn, N, K, E, ntok, top_k, 300 + ntok * 10 + top_k)
    ids_d = to_dev(ids)
    ws = torch.empty(qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k), dtype=torch.uint8, device=DEV)
    y = torch.full((ntok, top_k, K), 7.0, dtype=dt, device=DEV)
    qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, xin, ids_d, ntok, top_k, ws, y)
    want, tol = _layer_expected(gu, down, ids, x=x, q=q, d=d)
    got = bf16_to_np(y) if dt == torch.bfloat16 else y.cpu().numpy().astype(np.float64)
    assert_within(got, want, tol, out_of(fmt_dn), "layer")
    if xf is not None:
        y2 = torch.full_like(y, -7.0)
        qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, xf, ids_d, ntok, top_k, ws, y2, qmv.QMV_FLAG_X_F32)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
    assert status_clean()


def test_layer_many_slots():
    """32 routed slots (4 tokens x top-8), repeated experts and invalid ids."""
    E, N, K, ntok, top_k = 16, 512, 1024, 4, 8
    g = qi.rng(420)
    ids = np.stack([g.permutation(E)[:top_k] for _ in range(ntok)]).astype(np.int32)
    ids[3, 7] = E          # invalid
    ids[2, 0] = -5         # invalid
    gu = GateUp("mxfp4", N, K, E, ids.reshape(-1), seed=421)
    down = Matrices("mxfp4", K, N, E, ids.reshape(-1), seed=422)
    x = qi.normal_bf16_bits(g, (ntok, K))
    ws = torch.empty(qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k), dtype=torch.uint8, device=DEV)
    y = torch.full((ntok, top_k, K), 5.0, dtype=torch.bfloat16, device=DEV)
    qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, to_dev(x), to_dev(ids), ntok, top_k, ws, y)
    want, tol = _layer_expected(gu, down, ids, x=x)
    got = bf16_to_np(y)
    assert np.all(got[3, 7] == 0) and np.all(got[2, 0] == 0)
    assert_within(got, want, tol, "bf16", "layer")
    assert status_clean()


def test_layer_chain_graph_stream_prefetch():
    """Consecutive layers sharing one workspace, launched on a side stream
    (programmatic dependent launch) with QMV_FLAG_PREFETCH_INPUTS and replayed
    from a CUDA graph, as a decode step runs them, each layer's x the previous
    layer's output: every replay gives exactly the eager legacy-stream chain
    (no dependent launch, no prefetch)."""
    E, N, K, top_k, L = 8, 1024, 1024, 4, 4
    g = qi.rng(430)
    layers = []
    for l in range(L):
        ids = qi.topk_ids(g, 1, top_k, E)
        # scales around 2^-7 keep every layer's output O(1) through the chain
        gu = GateUp("mxfp4", N, K, E, range(E), seed=431 + l, scale_lo=118, scale_hi=122)
        down = Matrices("mxfp4", K, N, E, range(E), seed=441 + l, scale_lo=118, scale_hi=122)
        layers.append((gu, down, to_dev(ids)))
    x = to_dev(qi.normal_bf16_bits(g, (1, K)))
    nbytes = qmv.qmv_moe_layer_workspace_bytes(layers[0][0].desc, 1, top_k)

    def chain(y, ws, flags, stream):
        for l, (gu, down, ids_d) in enumerate(layers):
            xin = x if l == 0 else y[l - 1, 0, 0].view(1, K)
            qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, xin, ids_d, 1, top_k, ws, y[l], flags, stream=stream)

    y_ref = torch.empty(L, 1, top_k, K, dtype=torch.bfloat16, device=DEV)
    chain(y_ref, torch.empty(nbytes, dtype=torch.uint8, device=DEV), 0, 0)
    torch.cuda.synchronize()
    assert torch.isfinite(y_ref.float()).all()
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    y = torch.empty_like(y_ref)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain(y, ws, qmv.QMV_FLAG_PREFETCH_INPUTS, s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        chain(y, ws, qmv.QMV_FLAG_PREFETCH_INPUTS, s)
    for _ in range(3):
        y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    assert status_clean()


# ---------------------------------------------------------------------------
# QMV_FLAG_X_F32: fp32 activations quantized to q8_1 inside the matvec launch
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt,N,K", [("cb2", 2048, 7168), ("cb3", 515, 2080), ("cb4", 1024, 7168)])
@pytest.mark.parametrize("ntok", [1, 3, 4])
def test_x_f32_dense_equals_quantize_then_call(fmt, N, K, ntok):
    g = qi.rng(500 + ntok)
    m = Matrices(fmt, N, K, 1, [0], seed=501, lut=LUTS[fmt])
    xf = qi.normal_f32(g, (ntok, K))
    xf[0, :32] = 0.0                      # an all-zero block: d = 0
    xf[-1, 64] = 1e4                      # a block dominated by one value
    xq, _, _ = quantize_on_gpu(xf)
    y1 = torch.empty(ntok, N, dtype=torch.float32, device=DEV)
    y2 = torch.full_like(y1, 3.0)
    qmv.qmv_dense(m.desc, m.w, xq, ntok, y1)
    qmv.qmv_dense_ex(m.desc, m.w, to_dev(xf), ntok, y2, qmv.QMV_FLAG_X_F32)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    assert status_clean()


@pytest.mark.parametrize("per_slot", [0, 1])
def test_x_f32_gather_equals_quantize_then_call(per_slot):
    E, N, K, ntok, top_k = 64, 7168, 2048, 4, 4
    g = qi.rng(510 + per_slot)
    ids = qi.topk_ids(g, ntok, top_k, E)
    ids[2, 1] = 99
    m = Matrices("cb3", N, K, E, ids.reshape(-1), seed=511, lut=LUTS["cb3"])
    nvec = ntok * top_k if per_slot else ntok
    xf = qi.normal_f32(g, (nvec, K))
    xq, _, _ = quantize_on_gpu(xf)
    y1 = torch.empty(ntok, top_k, N, dtype=torch.float32, device=DEV)
    y2 = torch.full_like(y1, 3.0)
    ids_d = to_dev(ids)
    qmv.qmv_moe_gather(m.desc, m.w, xq, per_slot, ids_d, ntok, top_k, y1)
    qmv.qmv_moe_gather_ex(m.desc, m.w, to_dev(xf), per_slot, ids_d, ntok, top_k, y2, qmv.QMV_FLAG_X_F32)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    assert torch.all(y2[2, 1] == 0)
    assert status_clean()


# ---------------------------------------------------------------------------
# Split-K inside a CTA: uneven K ranges, sampled rows, run-to-run identity
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("ntok", [1, 2, 3])
def test_mxfp4_dense_split_k_uneven_ranges(ntok):
    """6400 x 7168 MXFP4 (800 row tiles of 7 chunks): the one-vector kernel
    cuts each row tile into 3 K ranges (3, 3, 1 chunks), the 2- and
    3-vector kernels into 2 (4, 3). Sampled rows against the oracle; two runs
    bit-identical."""
    N, K = 6400, 7168
    m = Matrices("mxfp4", N, K, 1, [0], seed=600)
    g = qi.rng(601 + ntok)
    x = qi.normal_bf16_bits(g, (ntok, K))
    rows = np.unique(np.concatenate([g.choice(N, 96, replace=False), [0, 7, 8, N - 1]]))
    outs = []
    for _ in range(2):
        y = torch.empty(ntok, N, dtype=torch.bfloat16, device=DEV)
        qmv.qmv_dense(m.desc, m.w, to_dev(x), ntok, y)
        outs.append(y.view(torch.int16).cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    got = bf16_to_np(torch.from_numpy(outs[0]).view(torch.bfloat16))[:, rows]
    cs, ss = m.codes[0][rows], m.scales[0][rows]
    ref = oracle.mxfp4_matvec(cs, ss, x)
    absum = oracle.mxfp4_abs_products(cs, ss, x)
    assert_close(got, ref, absum, True, f"mxfp4 dense split-K {N}x{K} ntok={ntok}")
    assert status_clean()


# ---------------------------------------------------------------------------
# Router-weighted combine of the per-slot outputs
# ---------------------------------------------------------------------------

def _combine_tol(ys, w, ids, E, slot_err=None):
    """Bound on the combine's fp32 result: the fma chain over top_k slots
    rounds once per step (2^-24 relative of the running magnitude, bounded by
    sum|w y|); slot_err bounds each stored per-slot input, weighted. The
    stored result (bf16, fp16 or fp32) is checked against it by rounding
    interval."""
    ntok, top_k, N = ys.shape
    valid = ((ids >= 0) & (ids < E)).astype(np.float64)[..., None]
    aw = np.abs(w.astype(np.float64))[..., None] * valid
    mag = (aw * np.abs(ys)).sum(axis=1)
    tol = mag * (top_k + 1) * 2.0 ** -24
    if slot_err is not None:
        tol = tol + (aw * slot_err).sum(axis=1)
    return tol


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("ntok,top_k,N", [(1, 4, 2880), (4, 8, 7168), (3, 1, 17), (2, 8, 4096)])
def test_combine(dtype, ntok, top_k, N):
    """qmv_moe_combine on given per-slot outputs against the oracle's float64
    combine; invalid ids (negative and >= E) contribute nothing."""
    E = 64
    g = qi.rng(500 + ntok * 37 + top_k + N)
    ids = np.stack([g.permutation(E)[:top_k] for _ in range(ntok)]).astype(np.int32)
    if top_k > 1:
        ids[0, 1] = -1
        ids[-1, 0] = E + 3
    w = qi.router_weights(g, ntok, top_k)
    fmt = "mxfp4" if dtype == "bf16" else "cb3"
    desc = qmv.wdesc(fmt, N, 64, E, lut=LUTS.get(fmt))
    if dtype == "bf16":
        bits = qi.normal_bf16_bits(g, (ntok, top_k, N))
        ys_np = oracle.bf16_bits_to_f64(bits)
        ys = to_dev(bits).view(torch.bfloat16)
        y = torch.full((ntok, N), 3.0, dtype=torch.bfloat16, device=DEV)
    else:
        f = qi.normal_f32(g, (ntok, top_k, N))
        ys_np = f.astype(np.float64)
        ys = to_dev(f)
        y = torch.full((ntok, N), 3.0, dtype=torch.float32, device=DEV)
    qmv.qmv_moe_combine(desc, ys, to_dev(w), to_dev(ids), ntok, top_k, y)
    want = oracle.moe_combine(ys_np, w, ids, E)
    got = bf16_to_np(y) if dtype == "bf16" else y.cpu().numpy().astype(np.float64)
    assert_within(got, want, _combine_tol(ys_np, w, ids, E), dtype, "combine")
    assert status_clean()


def test_combine_all_invalid_gives_zero():
    E, ntok, top_k, N = 8, 2, 4, 256
    g = qi.rng(520)
    ids = np.full((ntok, top_k), -1, dtype=np.int32)
    ids[1] = [E, E + 1, -7, 2 ** 31 - 1]
    w = qi.router_weights(g, ntok, top_k)
    ys = to_dev(qi.normal_f32(g, (ntok, top_k, N)))
    y = torch.full((ntok, N), 9.0, dtype=torch.float32, device=DEV)
    qmv.qmv_moe_combine(qmv.wdesc("cb4", N, 64, E, lut=qi.LUT_CB4), ys, to_dev(w), to_dev(ids), ntok, top_k, y)
    torch.cuda.synchronize()
    assert torch.count_nonzero(y).item() == 0
    assert status_clean()


@pytest.mark.parametrize("pair", LAYER_PAIRS, ids=lambda p: f"{p[0]}-{p[1]}")
@pytest.mark.parametrize("ntok,top_k", [(1, 4), (4, 2)])
def test_layer_combine(pair, ntok, top_k):
    """qmv_moe_layer_combine against the oracle chain (gate/up, SwiGLU, down,
    combine), and bit for bit against qmv_moe_layer followed by
    qmv_moe_combine."""
    fmt_gu, fmt_dn, N, K, E = pair
    ids, gu, down, x, xin, q, d, xf, dt = _layer_case(fmt_gu, fmt_dn, N, K, E, ntok, top_k, 600 + ntok * 10 + top_k)
    g = qi.rng(650 + ntok + top_k)
    w = qi.router_weights(g, ntok, top_k)
    ids_d, w_d = to_dev(ids), to_dev(w)
    nbytes = qmv.qmv_moe_layer_combine_workspace_bytes(gu.desc, down.desc, ntok, top_k)
    assert nbytes >= qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k) + ntok * top_k * K * (2 if dt == torch.bfloat16 else 4)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    y = torch.full((ntok, K), 7.0, dtype=dt, device=DEV)
    qmv.qmv_moe_layer_combine(gu.desc, gu.w, down.desc, down.w, xin, ids_d, w_d, ntok, top_k, ws, y)
    slots, slot_tol = _layer_expected(gu, down, ids, x=x, q=q, d=d)
    want = oracle.moe_combine(slots, w, ids, E)
    out = out_of(fmt_dn)
    tol = _combine_tol(slots, w, ids, E, stored_err(slots, slot_tol, out))
    got = bf16_to_np(y) if dt == torch.bfloat16 else y.cpu().numpy().astype(np.float64)
    assert_within(got, want, tol, out, "combined layer")
    ws2 = torch.empty(qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k), dtype=torch.uint8, device=DEV)
    ys = torch.empty(ntok, top_k, K, dtype=dt, device=DEV)
    qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, xin, ids_d, ntok, top_k, ws2, ys)
    y2 = torch.full_like(y, -7.0)
    qmv.qmv_moe_combine(down.desc, ys, w_d, ids_d, ntok, top_k, y2)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16 if dt == torch.bfloat16 else torch.int32),
                       y2.view(torch.int16 if dt == torch.bfloat16 else torch.int32))
    assert status_clean()
