"""qmv_moe_layer_noalloc: the MoE layer for callers that cannot allocate GPU
memory (an inference server that pre-assigns the whole device to its own
pool, a plugin under another application's fixed budget, code running during
stream capture). It must give what qmv_moe_layer gives with a workspace.

This file is collected last on purpose, and its tests run both alone in a
fresh process and after the rest of the suite.
"""
import numpy as np
import pytest

qmv = pytest.importorskip("bit_quantized_moe_gb300")
import oracle  # noqa: E402
import qmv_inputs as qi  # noqa: E402


def test_noalloc_rejects_layers_larger_than_its_scratch():
    """A layer whose scratch exceeds the static array is refused before any GPU work."""
    gu = qmv.wdesc("mxfp4", 65536, 64, 8)      # 4 tokens x 8 slots x 65536 bf16 = 4 MiB of h
    dn = qmv.wdesc("mxfp4", 64, 65536, 8)
    assert qmv.qmv_moe_layer_workspace_bytes(gu, 4, 8) > qmv.QMV_NOALLOC_SCRATCH_BYTES
    rc = qmv.lib.qmv_moe_layer_noalloc(qmv.ctypes.byref(gu), 1 << 40, qmv.ctypes.byref(dn), 1 << 40, 1 << 40,
                                       1 << 40, 4, 8, 1 << 40, 0, 0)
    assert rc == qmv.QMV_ESIZE
    assert "static scratch" in qmv.qmv_last_error()


@pytest.mark.gpu
def test_noalloc_layer_matches_workspace_layer_on_two_calls():
    """Two calls in a row (different ids and activations): each matches
    qmv_moe_layer with a caller workspace within the suite's float tolerance."""
    import torch
    from qmv_testutil import DEV, Matrices, bf16_to_np, to_dev
    from test_gpu_parity import GateUp, _layer_expected

    E, N, K, N_down, ntok, top_k = 8, 512, 512, 516, 2, 4
    gu = GateUp("mxfp4", N, K, E, range(E), seed=901)
    down = Matrices("mxfp4", N_down, N, E, range(E), seed=902)
    for call in range(2):
        g = qi.rng(903 + call)
        ids = qi.topk_ids(g, ntok, top_k, E)
        x = qi.normal_bf16_bits(g, (ntok, K))
        x_d, ids_d = to_dev(x), to_dev(ids)
        ws = torch.empty(qmv.qmv_moe_layer_workspace_bytes(gu.desc, ntok, top_k), dtype=torch.uint8, device=DEV)
        y_ref = torch.empty(ntok, top_k, N_down, dtype=torch.bfloat16, device=DEV)
        y = torch.full_like(y_ref, 5.0)
        qmv.qmv_moe_layer(gu.desc, gu.w, down.desc, down.w, x_d, ids_d, ntok, top_k, ws, y_ref)
        qmv.qmv_moe_layer_noalloc(gu.desc, gu.w, down.desc, down.w, x_d, ids_d, ntok, top_k, y)
        torch.cuda.synchronize()
        # the tolerance the suite uses for this layer (oracle-derived bound)
        _, tol = _layer_expected(gu, down, ids, x=x)
        diff = np.abs(bf16_to_np(y) - bf16_to_np(y_ref))
        assert np.all(diff <= tol + 1e-30), f"call {call}: {(diff > tol).sum()} outputs differ beyond tolerance"
    assert qmv.qmv_device_status(clear=True) == 0
