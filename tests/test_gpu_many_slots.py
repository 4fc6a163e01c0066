"""GPU parity of gathers, gate/up fusions and layers of 33..128 routed
(token, slot) pairs -- a verify or prefill batch through a MoE projection
("perf(ggml/hip): optimize ROCMFPX fp3/fp2 MMVQ on RDNA ...", "Depends on":
the batched MMQ path; "perf(rocm): add an mxfp4 arm ...", "Implementation
Notes": sorted calls for larger batches). When the experts carry few slots
each, or the call has no tensor-core form (fp16 activations, the gate/up
fusion), it runs as CUDA-core gathers of whole tokens, 32 slots at a time:
those must give the bits of the same calls made by hand on token halves.
Otherwise it is the sorted tensor-core gather, checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import qmv_inputs as qi

pytestmark = pytest.mark.gpu

qmv = pytest.importorskip("bit_quantized_moe_gb300")
from qmv_testutil import (DEV, Matrices, assert_close, assert_within, bf16_to_np, out_of,  # noqa: E402
                          quantize_on_gpu, status_clean, to_dev)
from test_gpu_parity import LUTS, GateUp, _layer_case, _layer_expected  # noqa: E402


def _ids(g, ntok, top_k, E):
    ids = qi.topk_ids(g, ntok, top_k, E)
    ids[1, 0] = ids[0, 0]        # an expert shared across the token halves
    ids[ntok - 1, 0] = ids[0, 0]
    ids[3, top_k - 1] = -1       # invalid ids: zero rows
    ids[ntok - 2, 1] = E + 2
    return ids


@pytest.mark.parametrize("fmt,act,per_slot", [("mxfp4", "bf16", False), ("mxfp4", "f16", True),
                                              ("mxfp8", "bf16", True), ("cb3", "q8", True), ("cb2", "f32", False)])
def test_split_gather_equals_token_halves(fmt, act, per_slot):
    """64 slots over 256 experts (about one slot per expert): CUDA-core
    gathers of 8 tokens each, bit-identical to two calls on the token halves;
    sampled slots against the oracle."""
    E, N, K, ntok, top_k = 256, 264, 1024, 16, 4
    g = qi.rng(5000 + len(fmt) + per_slot)
    ids = _ids(g, ntok, top_k, E)
    m = Matrices(fmt, N, K, E, ids.reshape(-1), seed=5001, lut=LUTS.get(fmt))
    nvec = ntok * top_k if per_slot else ntok
    flags = {"f16": qmv.QMV_FLAG_X_F16, "f32": qmv.QMV_FLAG_X_F32}.get(act, 0)
    if act in ("bf16", "f16"):
        xb = qi.normal_bf16_bits(g, (nvec, K)) if act == "bf16" else qi.normal_f16_bits(g, (nvec, K))
        xin, ydt = to_dev(xb), (torch.bfloat16 if act == "bf16" else torch.float16)
    elif act == "q8":
        xin, q, d = quantize_on_gpu(qi.normal_f32(g, (nvec, K)))
        ydt = torch.float32
    else:
        xf = qi.normal_f32(g, (nvec, K))
        xin, ydt = to_dev(xf), torch.float32
        _, q, d = quantize_on_gpu(xf)
    ids_d = to_dev(ids)
    y = torch.full((ntok, top_k, N), 5.0, dtype=ydt, device=DEV)
    qmv.qmv_moe_gather_ex(m.desc, m.w, xin, int(per_slot), ids_d, ntok, top_k, y, flags)
    yh = torch.full_like(y, -5.0)
    half = ntok // 2
    vb = qmv.qmv_act_q8_vec_bytes(K) if act == "q8" else 1   # q8_1: a flat byte buffer
    for t0 in (0, half):
        v0 = t0 * top_k if per_slot else t0
        xv = xin[v0 * vb:]
        qmv.qmv_moe_gather_ex(m.desc, m.w, xv, int(per_slot), ids_d[t0:], half, top_k, yh[t0:], flags)
    torch.cuda.synchronize()
    bits = torch.int16 if ydt != torch.float32 else torch.int32
    assert torch.equal(y.view(bits), yh.view(bits))
    got = y.float().cpu().numpy().astype(np.float64) if ydt != torch.bfloat16 else bf16_to_np(y)
    for t, j in ((0, 0), (1, 0), (5, 2), (9, 1), (15, 3), (3, top_k - 1), (ntok - 2, 1)):
        e = int(ids[t, j])
        if not (0 <= e < E):
            assert np.all(got[t, j] == 0), (t, j)
            continue
        v = t * top_k + j if per_slot else t
        if fmt.startswith("mx"):
            xd = "bf16" if act == "bf16" else "f16"
            ref = oracle.mx_matvec(fmt, m.codes[e], m.scales[e], xb[v:v + 1], xd)[0]
            absum = oracle.mx_abs_products(fmt, m.codes[e], m.scales[e], xb[v:v + 1], xd)[0]
            assert_close(got[t, j], ref, absum, act, f"slot ({t},{j})")
        else:
            grp = qi.FORMAT_GROUP[fmt]
            ref = oracle.cb_matvec(m.codes[e], m.scales[e], m.lut, grp, q[v:v + 1], d[v:v + 1])[0]
            absum = oracle.cb_abs_products(m.codes[e], m.scales[e], m.lut, grp, q[v:v + 1], d[v:v + 1])[0]
            assert_close(got[t, j], ref, absum, "f32", f"slot ({t},{j})")
    assert status_clean()


@pytest.mark.parametrize("fmt", ["mxfp4", "cb2"])
def test_gate_up_many_slots(fmt):
    """The fused gate/up/SwiGLU over 64 slots (no tensor-core form): two
    CUDA-core launches, bit-identical to the calls on the token halves."""
    E, N, K, ntok, top_k = 32, 520, 1024, 16, 4
    g = qi.rng(5100 + len(fmt))
    ids = _ids(g, ntok, top_k, E)
    gu = GateUp(fmt, N, K, E, ids.reshape(-1), seed=5101, lut=LUTS.get(fmt))
    if fmt == "mxfp4":
        xin, hdt = to_dev(qi.normal_bf16_bits(g, (ntok, K))), torch.bfloat16
    else:
        xin, _, _ = quantize_on_gpu(qi.normal_f32(g, (ntok, K)))
        hdt = torch.float32
    ids_d = to_dev(ids)
    h = torch.full((ntok, top_k, N), 3.0, dtype=hdt, device=DEV)
    qmv.qmv_moe_gate_up_swiglu(gu.desc, gu.w, xin, ids_d, ntok, top_k, h)
    hh = torch.full_like(h, -3.0)
    vb = 1 if fmt == "mxfp4" else qmv.qmv_act_q8_vec_bytes(K)   # q8_1: a flat byte buffer
    for t0 in (0, ntok // 2):
        qmv.qmv_moe_gate_up_swiglu(gu.desc, gu.w, xin[t0 * vb:], ids_d[t0:], ntok // 2, top_k, hh[t0:])
    torch.cuda.synchronize()
    bits = torch.int16 if hdt == torch.bfloat16 else torch.int32
    assert torch.equal(h.view(bits), hh.view(bits))
    assert torch.count_nonzero(h[3, top_k - 1].float()).item() == 0
    assert status_clean()


@pytest.mark.parametrize("pair,E,path", [
    (("mxfp4", "mxfp4", 512, 1024), 8, 0),           # 8 slots per expert: down on the tensor cores
    (("mxfp4", "mxfp4", 512, 1024), 8, 16),          # the same, forced onto the CUDA cores
    (("mxfp4", "mxfp4", 512, 1024), 64, 0),          # one slot per expert: CUDA-core gathers
    (("cb2", "cb3", 512, 1024), 8, 8),               # codebook down forced onto the tensor cores
    (("cb4", "cb4", 512, 1024), 64, 0),
], ids=["mxfp4-E8", "mxfp4-E8-cuda", "mxfp4-E64", "cb2-cb3-E8-tensor", "cb4-E64"])
def test_layer_64_slots(pair, E, path):
    """A 16-token batch through a MoE layer (64 routed slots): gate/up on the
    CUDA cores, the down projection sorted on the tensor cores or as CUDA-core
    gathers of 8 tokens, against the oracle chain."""
    fmt_gu, fmt_dn, N, K = pair
    ntok, top_k = 16, 4
    ids, gu, down, x, xin, q, d, xf, dt = _layer_case(fmt_gu, fmt_dn, N, K, E, ntok, top_k, 5200 + E)
    ids_d = to_dev(ids)
    ws = torch.empty(qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k), dtype=torch.uint8, device=DEV)
    y = torch.full((ntok, top_k, K), 7.0, dtype=dt, device=DEV)
    qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, xin, ids_d, ntok, top_k, ws, y, path)
    want, tol = _layer_expected(gu, down, ids, x=x, q=q, d=d)
    got = bf16_to_np(y) if dt == torch.bfloat16 else y.cpu().numpy().astype(np.float64)
    assert_within(got, want, tol, out_of(fmt_dn), "layer")
    assert np.all(got[ntok - 1, top_k - 1] == 0)
    assert status_clean()
