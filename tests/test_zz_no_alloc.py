"""qmv_moe_layer_noalloc: the MoE layer for callers that cannot allocate GPU
memory (an inference server that pre-assigns the whole device to its own
pool, a plugin under another application's fixed budget, code running during
stream capture). Its scratch is a static array inside the library; it must
give exactly what qmv_moe_layer gives with a caller workspace.

This file is collected last on purpose, and its tests run both alone in a
fresh process and after the rest of the suite.
"""
import numpy as np
import pytest

qmv = pytest.importorskip("bit_quantized_moe_gb300")
import qmv_inputs as qi  # noqa: E402


def _raw_noalloc(gu, dn, ntok, top_k):
    """Calls the entry point with fake (aligned) device addresses: only the
    host-side argument checks can run on them."""
    return qmv.lib.qmv_moe_layer_noalloc(qmv.ctypes.byref(gu), 1 << 40, qmv.ctypes.byref(dn), 1 << 40, 1 << 40,
                                         1 << 40, ntok, top_k, 1 << 40, 0, 0)


def test_noalloc_rejects_layers_larger_than_its_scratch():
    """A layer whose scratch exceeds the static array is refused before any GPU work."""
    gu = qmv.wdesc("mxfp4", 65536, 64, 8)      # 4 tokens x 8 slots x 65536 bf16 = 4 MiB of h
    dn = qmv.wdesc("mxfp4", 64, 65536, 8)
    assert qmv.qmv_moe_layer_workspace_bytes(gu, 4, 8) > qmv.QMV_NOALLOC_SCRATCH_BYTES
    assert _raw_noalloc(gu, dn, 4, 8) == qmv.QMV_ESIZE
    assert "static scratch" in qmv.qmv_last_error()


@pytest.mark.parametrize("fmt,N", [("mxfp4", 16384), ("cb2", 8192)])
def test_noalloc_size_boundary(fmt, N):
    """32 routed slots of h: exactly the array's size passes the size check
    (it then fails later, here for want of a GPU or on the fake pointers,
    never with QMV_ESIZE); one row tile more is refused with QMV_ESIZE."""
    lut = qi.LUT_CB2 if fmt == "cb2" else None
    dn_fmt = "cb3" if fmt == "cb2" else fmt
    for n, fits in ((N, True), (N + 32, False)):
        gu = qmv.wdesc(fmt, n, 64, 4, lut)
        dn = qmv.wdesc(dn_fmt, 64, n, 4, qi.LUT_CB3 if fmt == "cb2" else None)
        need = qmv.qmv_moe_layer_workspace_bytes(gu, 4, 8)
        assert (need == qmv.QMV_NOALLOC_SCRATCH_BYTES) == fits or need > qmv.QMV_NOALLOC_SCRATCH_BYTES
        rc = _raw_noalloc(gu, dn, 4, 8)
        if fits:
            assert need == qmv.QMV_NOALLOC_SCRATCH_BYTES
            assert rc != qmv.QMV_ESIZE, qmv.qmv_last_error()
        else:
            assert rc == qmv.QMV_ESIZE and "static scratch" in qmv.qmv_last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("pair", ["mxfp4", "cb2-cb3"])
def test_noalloc_layer_matches_workspace_layer_on_two_calls(pair):
    """Two calls in a row (different ids and activations): each is bit for bit
    qmv_moe_layer with a caller workspace, and within the suite's bound of the
    oracle chain (gate/up, SwiGLU, down). The codebook layer takes fp32 x
    (QMV_FLAG_X_F32) and keeps its fp32 h in the static array."""
    import torch
    from qmv_testutil import DEV, Matrices, assert_within, bf16_to_np, quantize_on_gpu, to_dev
    from test_gpu_parity import GateUp, _layer_expected

    E, ntok, top_k = 8, 2, 4
    if pair == "mxfp4":
        N, K = 512, 512
        gu = GateUp("mxfp4", N, K, E, range(E), seed=901)
        down = Matrices("mxfp4", 516, N, E, range(E), seed=902)
        dt, flags = torch.bfloat16, 0
    else:
        N, K = 1024, 2048
        gu = GateUp("cb2", N, K, E, range(E), seed=911, lut=qi.LUT_CB2)
        down = Matrices("cb3", 1032, N, E, range(E), seed=912, lut=qi.LUT_CB3)
        dt, flags = torch.float32, qmv.QMV_FLAG_X_F32
    for call in range(2):
        g = qi.rng(903 + call)
        ids = qi.topk_ids(g, ntok, top_k, E)
        if pair == "mxfp4":
            x = qi.normal_bf16_bits(g, (ntok, K))
            x_d, q, d = to_dev(x), None, None
        else:
            x = None
            xf = qi.normal_f32(g, (ntok, K))
            _, q, d = quantize_on_gpu(xf)
            x_d = to_dev(xf)
        ids_d = to_dev(ids)
        ws = torch.empty(qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k), dtype=torch.uint8, device=DEV)
        y_ref = torch.empty(ntok, top_k, down.N, dtype=dt, device=DEV)
        y = torch.full_like(y_ref, 5.0)
        qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, x_d, ids_d, ntok, top_k, ws, y_ref, flags)
        qmv.qmv_moe_layer_noalloc(gu.desc, gu.w, down.desc, down.w, x_d, ids_d, ntok, top_k, y, flags)
        torch.cuda.synchronize()
        iv = torch.int16 if dt == torch.bfloat16 else torch.int32
        assert torch.equal(y.view(iv), y_ref.view(iv)), f"call {call}: differs from qmv_moe_layer"
        want, tol = _layer_expected(gu, down, ids, x=x, q=q, d=d)
        got = bf16_to_np(y) if dt == torch.bfloat16 else y.cpu().numpy()
        assert_within(got, want, tol, "bf16" if dt == torch.bfloat16 else "f32", f"call {call} vs oracle")
    assert qmv.qmv_device_status(clear=True) == 0
