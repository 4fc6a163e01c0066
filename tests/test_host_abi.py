"""Host-side tests of the C ABI: the library loads, exports every declared
symbol, packs and unpacks every format bit-exactly, and rejects bad arguments
with the documented error codes before touching a GPU."""
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
import qmv_inputs as qi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmv.h")

qmv = pytest.importorskip("bit_quantized_moe_gb300", reason="libqmv not built")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qmv_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(qmv.EXPORTS)


def test_library_exports_every_declared_symbol():
    out = subprocess.run(["nm", "-D", "--defined-only", qmv.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\sT\s+(qmv_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(qmv.lib, name)


def test_version_and_format_constants():
    assert "sm_103a" in qmv.qmv_version()
    assert [qmv.qmv_scale_group(f) for f in ("mxfp4", "cb2", "cb3", "cb4", "mxfp8")] == [32, 16, 16, 32, 32]
    assert [qmv.qmv_code_bits(f) for f in ("mxfp4", "cb2", "cb3", "cb4", "mxfp8")] == [4, 2, 3, 4, 8]
    assert qmv.qmv_code_bits(5) == 0
    assert qmv.qmv_scale_group(7) == 0


SHAPES = [(1, 32), (5, 96), (16, 1024), (17, 1056), (40, 2048), (516, 2880)]


@pytest.mark.parametrize("fmt", ["mxfp4", "cb2", "cb3", "cb4", "mxfp8"])
@pytest.mark.parametrize("N,K", SHAPES)
def test_pack_roundtrip_bit_exact(fmt, N, K):
    E = 2
    g = qi.rng(100 + N + K)
    codes = qi.codes(g, (E, N, K), qi.FORMAT_BITS[fmt])   # every byte value, NaN codes included
    scales = qi.e8m0(g, (E, N, K // qi.FORMAT_GROUP[fmt]), 0, 255)
    canon = oracle.pack_codes(fmt, codes)
    d = qmv.wdesc(fmt, N, K, E)
    assert qmv.qmv_canonical_code_bytes(d) == canon[0].nbytes
    assert qmv.qmv_canonical_scale_bytes(d) == scales[0].nbytes
    packed = qmv.qmv_pack_weights(d, canon, scales)
    assert packed.nbytes == qmv.qmv_packed_bytes(d) == E * qmv.qmv_packed_expert_bytes(d)
    assert qmv.qmv_packed_expert_bytes(d) % 256 == 0
    c2, s2 = qmv.qmv_unpack_weights(d, packed)
    assert np.array_equal(c2.reshape(canon.shape), canon)
    assert np.array_equal(s2.reshape(scales.shape), scales)
    assert np.array_equal(oracle.unpack_codes(fmt, c2.reshape(canon.shape)), codes)


def test_pack_changes_with_every_code():
    """Every canonical code bit lands somewhere in the GPU layout (no dropped bits)."""
    for fmt in ("mxfp4", "cb2", "cb3", "cb4", "mxfp8"):
        N, K = 3, 64
        d = qmv.wdesc(fmt, N, K)
        codes = np.zeros((1, N, K), dtype=np.uint8)
        scales = np.zeros((1, N, K // qi.FORMAT_GROUP[fmt]), dtype=np.uint8)
        base = qmv.qmv_pack_weights(d, oracle.pack_codes(fmt, codes), scales)
        seen = set()
        for n in range(N):
            for k in range(K):
                for b in range(qi.FORMAT_BITS[fmt]):
                    c = codes.copy()
                    c[0, n, k] = 1 << b
                    p = qmv.qmv_pack_weights(d, oracle.pack_codes(fmt, c), scales)
                    diff = np.nonzero(p != base)[0]
                    assert len(diff) == 1
                    bit = (int(diff[0]), int(p[diff[0]] ^ base[diff[0]]))
                    assert bit not in seen
                    seen.add(bit)


def test_packed_bytes_match_algorithmic_bytes():
    # 2880 x 2880 MXFP4: 1440 code bytes + 90 scale bytes per row, no padding
    # besides rounding the expert stride to 256 bytes.
    d = qmv.wdesc("mxfp4", 2880, 2880)
    alg = 2880 * 1440 + 2880 * 90
    assert alg == 4406400
    assert alg <= qmv.qmv_packed_expert_bytes(d) < alg + 256
    d = qmv.wdesc("cb3", 7168, 2048)
    alg = 7168 * 2048 * 3 // 8 + 7168 * 128
    assert alg == 6422528
    assert alg <= qmv.qmv_packed_expert_bytes(d) < alg + 256
    d = qmv.wdesc("cb2", 2048, 7168)
    assert 2048 * 7168 // 4 + 2048 * 448 == 4587520
    assert qmv.qmv_packed_expert_bytes(d) == 4587520
    d = qmv.wdesc("cb4", 7168, 7168)
    assert qmv.qmv_packed_expert_bytes(d) == 27295744
    # MXFP8 2880 x 2880: 2880 code bytes + 90 scale bytes per row
    d = qmv.wdesc("mxfp8", 2880, 2880)
    alg = 2880 * 2880 + 2880 * 90
    assert alg <= qmv.qmv_packed_expert_bytes(d) < alg + 256


def test_q8_sizes_and_unpack():
    assert qmv.qmv_act_q8_vec_bytes(32) == 48           # 32 + 2 -> 48
    assert qmv.qmv_act_q8_vec_bytes(7168) == 7168 + 448
    assert qmv.qmv_act_q8_vec_bytes(33) == 0
    assert qmv.qmv_act_q8_bytes(3, 2048) == 3 * (2048 + 128)
    vb = qmv.qmv_act_q8_vec_bytes(64)
    buf = np.arange(2 * vb, dtype=np.uint8)
    q, d = qmv.qmv_act_q8_unpack(buf, 2, 64)
    assert np.array_equal(q[1].view(np.uint8), buf[vb:vb + 64])
    assert np.array_equal(d[1], buf[vb + 64:vb + 68].view(np.uint16))


FAKE = 1 << 40          # 16-byte aligned address that is never dereferenced


@pytest.mark.parametrize("case,code", [
    ("K not multiple of 32", qmv.QMV_ESHAPE),
    ("N zero", qmv.QMV_ESHAPE),
    ("bad format", qmv.QMV_EINVAL),
    ("ntok 17", qmv.QMV_EINVAL),
    ("ntok 0", qmv.QMV_EINVAL),
    ("misaligned x", qmv.QMV_EALIGN),
    ("null y", qmv.QMV_EINVAL),
    ("dense with experts", qmv.QMV_EINVAL),
])
def test_dense_argument_errors(case, code):
    d = qmv.wdesc("cb4", 64, 64)
    w, x, y, ntok = FAKE, FAKE, FAKE, 1
    if case == "K not multiple of 32":
        d.K = 48
    elif case == "N zero":
        d.N = 0
    elif case == "bad format":
        d.fmt = 9
    elif case == "ntok 17":
        ntok = 17
    elif case == "ntok 0":
        ntok = 0
    elif case == "misaligned x":
        x = FAKE + 4
    elif case == "null y":
        y = None
    elif case == "dense with experts":
        d.n_experts = 3
    with pytest.raises(qmv.QmvError) as ei:
        qmv.qmv_dense(d, w, x, ntok, y, stream=0)
    assert ei.value.code == code
    assert qmv.qmv_last_error()


@pytest.mark.parametrize("top_k,ids,code", [(9, FAKE, qmv.QMV_EINVAL), (0, FAKE, qmv.QMV_EINVAL),
                                            (4, None, qmv.QMV_EINVAL), (4, FAKE + 8, qmv.QMV_EALIGN)])
def test_gather_argument_errors(top_k, ids, code):
    d = qmv.wdesc("mxfp4", 64, 64, 8)
    with pytest.raises(qmv.QmvError) as ei:
        qmv.qmv_moe_gather(d, FAKE, FAKE, 0, ids, 1, top_k, FAKE, stream=0)
    assert ei.value.code == code


def test_routed_slot_limit():
    """Gathers and layers route at most QMV_MAX_SLOTS (128) (token, slot)
    pairs, any format and activation type (beyond QMV_MAX_LAYER_SLOTS (32)
    they run as the sorted tensor-core gather or as CUDA-core gathers of 32
    slots each); 16 tokens and top-8 are the limits. (No call here reaches a
    launch: every one fails validation, or, for the accepted calls, the
    device query of a machine without a GPU.)"""
    assert qmv.MAX_SLOTS == 128 and qmv.MAX_LAYER_SLOTS == 32 and qmv.MAX_NTOK == 16
    B = qmv.ctypes.byref
    G = qmv.lib.qmv_moe_gather_ex
    cb = qmv.wdesc("cb3", 64, 64, 8, qi.LUT_CB3)
    assert G(B(cb), FAKE, FAKE, 0, FAKE, 8, 8, FAKE, 0, 0) != qmv.QMV_EINVAL      # 64 codebook slots
    assert G(B(cb), FAKE, FAKE, 0, FAKE, 16, 9, FAKE, 0, 0) == qmv.QMV_EINVAL     # 144 slots
    mx = qmv.wdesc("mxfp4", 64, 64, 8)
    assert G(B(mx), FAKE, FAKE, 0, FAKE, 8, 8, FAKE, qmv.QMV_FLAG_X_F16, 0) != qmv.QMV_EINVAL   # fp16, 64 slots
    assert G(B(mx), FAKE, FAKE, 0, FAKE, 17, 1, FAKE, 0, 0) == qmv.QMV_EINVAL     # 17 tokens
    assert G(B(mx), FAKE, FAKE, 0, FAKE, 16, 9, FAKE, 0, 0) == qmv.QMV_EINVAL     # top_k 9
    gu = qmv.wdesc("mxfp4", 64, 64, 8)
    assert qmv.qmv_moe_layer_workspace_bytes(gu, 8, 4) == (32 * 64 * 2 + 255) // 256 * 256
    assert qmv.qmv_moe_layer_workspace_bytes(gu, 16, 8) == (128 * 64 * 2 + 255) // 256 * 256
    assert qmv.qmv_moe_layer_workspace_bytes(gu, 16, 9) == 0                        # 144 slots
    L = qmv.lib.qmv_moe_layer
    assert L(B(gu), FAKE, B(gu), FAKE, FAKE, FAKE, 16, 4, FAKE, 1 << 20, FAKE, 0, 0) != qmv.QMV_EINVAL
    assert L(B(gu), FAKE, B(gu), FAKE, FAKE, FAKE, 16, 9, FAKE, 1 << 20, FAKE, 0, 0) == qmv.QMV_EINVAL
    assert qmv.lib.qmv_quantize_act_q8(FAKE, 129, 64, FAKE, 1 << 22, 0) == qmv.QMV_EINVAL


def test_debug_sums_size_error():
    d = qmv.wdesc("cb2", 64, 64)
    small = np.zeros(4, dtype=np.int32)
    rc = qmv.lib.qmv_debug_block_sums(qmv.ctypes.byref(d), FAKE, FAKE, 0, None, 1, 1, FAKE, FAKE, small.nbytes, 0)
    assert rc == qmv.QMV_ESIZE
    d = qmv.wdesc("mxfp4", 64, 64)
    rc = qmv.lib.qmv_debug_block_sums(qmv.ctypes.byref(d), FAKE, FAKE, 0, None, 1, 1, FAKE, FAKE, 1 << 20, 0)
    assert rc == qmv.QMV_EINVAL


def test_pack_size_errors():
    d = qmv.wdesc("cb3", 16, 64)
    codes = np.zeros(qmv.qmv_canonical_code_bytes(d), dtype=np.uint8)
    scales = np.zeros(qmv.qmv_canonical_scale_bytes(d), dtype=np.uint8)
    out = np.zeros(qmv.qmv_packed_bytes(d) - 16, dtype=np.uint8)
    rc = qmv.lib.qmv_pack_weights(qmv.ctypes.byref(d), codes.ctypes.data, scales.ctypes.data, out.ctypes.data,
                                  out.nbytes)
    assert rc == qmv.QMV_ESIZE
    rc = qmv.lib.qmv_pack_weights(qmv.ctypes.byref(d), None, scales.ctypes.data, out.ctypes.data, out.nbytes)
    assert rc == qmv.QMV_EINVAL


def test_quantize_and_swiglu_argument_errors():
    assert qmv.lib.qmv_quantize_act_q8(FAKE, 1, 33, FAKE, 1 << 20, 0) == qmv.QMV_ESHAPE
    assert qmv.lib.qmv_quantize_act_q8(FAKE, 1, 64, FAKE, 8, 0) == qmv.QMV_ESIZE
    assert qmv.lib.qmv_quantize_act_q8(FAKE + 4, 1, 64, FAKE, 1 << 20, 0) == qmv.QMV_EALIGN
    assert qmv.lib.qmv_swiglu_bf16(FAKE, FAKE, None, 16, 0) == qmv.QMV_EINVAL
    assert qmv.lib.qmv_swiglu_bf16(FAKE, FAKE + 2, FAKE, 16, 0) == qmv.QMV_EALIGN


def test_wait_probe_argument_errors():
    assert qmv.lib.qmv_debug_wait_probe(0, 0) == qmv.QMV_EINVAL
    assert qmv.lib.qmv_debug_wait_probe(2_000_000_000, 0) == qmv.QMV_EINVAL


def test_unknown_launch_flags_rejected():
    d = qmv.wdesc("mxfp4", 64, 64, 4)
    rc = qmv.lib.qmv_moe_gather_ex(qmv.ctypes.byref(d), FAKE, FAKE, 0, FAKE, 1, 4, FAKE, 6, 0)
    assert rc == qmv.QMV_EINVAL
    d = qmv.wdesc("cb2", 64, 64)
    assert qmv.lib.qmv_dense_ex(qmv.ctypes.byref(d), FAKE, FAKE, 1, FAKE, 32, 0) == qmv.QMV_EINVAL
    # the two path overrides are exclusive; block sums take only prefetch and path flags
    both = qmv.QMV_FLAG_PATH_TENSOR | qmv.QMV_FLAG_PATH_CUDA_CORES
    assert qmv.lib.qmv_dense_ex(qmv.ctypes.byref(d), FAKE, FAKE, 8, FAKE, both, 0) == qmv.QMV_EINVAL
    S = qmv.lib.qmv_debug_block_sums_ex
    assert S(qmv.ctypes.byref(d), FAKE, FAKE, 0, None, 1, 1, FAKE, FAKE, 1 << 20, qmv.QMV_FLAG_X_F32, 0) == qmv.QMV_EINVAL
    assert S(qmv.ctypes.byref(d), FAKE, FAKE, 0, None, 1, 1, FAKE, FAKE, 1 << 20, both, 0) == qmv.QMV_EINVAL
    # fp16 activations exist only for the MX formats, fp32 ones only for the codebooks
    assert qmv.lib.qmv_dense_ex(qmv.ctypes.byref(d), FAKE, FAKE, 1, FAKE, qmv.QMV_FLAG_X_F16, 0) == qmv.QMV_EINVAL
    m8 = qmv.wdesc("mxfp8", 64, 64)
    assert qmv.lib.qmv_dense_ex(qmv.ctypes.byref(m8), FAKE, FAKE, 1, FAKE, qmv.QMV_FLAG_X_F32, 0) == qmv.QMV_EINVAL
    assert qmv.lib.qmv_dense_ex(qmv.ctypes.byref(m8), FAKE, FAKE, 1, FAKE, 64, 0) == qmv.QMV_EINVAL
    C = qmv.lib.qmv_moe_combine_ex
    cb = qmv.wdesc("cb3", 64, 64, 4)
    assert C(qmv.ctypes.byref(cb), FAKE, FAKE, FAKE, 1, 4, FAKE, qmv.QMV_FLAG_X_F16, 0) == qmv.QMV_EINVAL
    assert C(qmv.ctypes.byref(m8), FAKE, FAKE, FAKE, 1, 4, FAKE, 1, 0) == qmv.QMV_EINVAL


@pytest.mark.parametrize("fmt", ["mxfp4", "cb3"])
@pytest.mark.parametrize("N", [1, 8, 515, 516])
def test_pack_gate_up_interleaves_rows(fmt, N):
    """The fused gate/up layout is the plain layout of a 2*round_up(N,4)-row
    matrix whose 8-row tile i holds gate rows 4i..4i+3 then up rows 4i..4i+3."""
    E, K = 2, 96
    g = qi.rng(N)
    bits, grp = qi.FORMAT_BITS[fmt], qi.FORMAT_GROUP[fmt]
    cg, cu = qi.codes(g, (E, N, K), bits), qi.codes(g, (E, N, K), bits)
    sg, su = qi.e8m0(g, (E, N, K // grp)), qi.e8m0(g, (E, N, K // grp))
    d = qmv.wdesc(fmt, N, K, E)
    packed = qmv.qmv_pack_gate_up(d, oracle.pack_codes(fmt, cg), sg, oracle.pack_codes(fmt, cu), su)
    R = 2 * ((N + 3) // 4 * 4)
    dm = qmv.wdesc(fmt, R, K, E)
    assert packed.nbytes == qmv.qmv_packed_bytes(dm) == E * qmv.qmv_packed_gate_up_expert_bytes(d)
    c2, s2 = qmv.qmv_unpack_weights(dm, packed)
    codes = oracle.unpack_codes(fmt, c2.reshape(E, R, -1))
    scales = s2.reshape(E, R, -1)
    for row in range(R):
        tile, r = divmod(row, 8)
        src = 4 * tile + r % 4
        if src >= N:
            assert not codes[:, row].any() and not scales[:, row].any()
            continue
        want_c, want_s = (cu, su) if r >= 4 else (cg, sg)
        assert np.array_equal(codes[:, row], want_c[:, src])
        assert np.array_equal(scales[:, row], want_s[:, src])


def test_moe_layer_argument_errors():
    gu = qmv.wdesc("mxfp4", 2880, 2880, 32)
    dn = qmv.wdesc("mxfp4", 2880, 2880, 32)
    need = qmv.qmv_moe_layer_workspace_bytes(gu, 1, 4)
    assert need == (4 * 2880 * 2 + 255) // 256 * 256
    cbd = qmv.wdesc("cb2", 2048, 7168, 64)
    assert qmv.qmv_moe_layer_workspace_bytes(cbd, 1, 4) == 4 * 2048 * 4
    L = qmv.lib.qmv_moe_layer
    B = qmv.ctypes.byref
    assert L(B(gu), FAKE, B(dn), FAKE, FAKE, FAKE, 1, 4, FAKE, need - 16, FAKE, 0, 0) == qmv.QMV_ESIZE
    bad = qmv.wdesc("mxfp4", 2880, 1024, 32)
    assert L(B(gu), FAKE, B(bad), FAKE, FAKE, FAKE, 1, 4, FAKE, need, FAKE, 0, 0) == qmv.QMV_ESHAPE
    cb = qmv.wdesc("cb3", 2880, 2880, 32)
    assert L(B(gu), FAKE, B(cb), FAKE, FAKE, FAKE, 1, 4, FAKE, need, FAKE, 0, 0) == qmv.QMV_EINVAL
    assert L(B(gu), FAKE, B(dn), FAKE, FAKE, None, 1, 4, FAKE, need, FAKE, 0, 0) == qmv.QMV_EINVAL
    assert L(B(gu), FAKE, B(dn), FAKE, FAKE, FAKE, 1, 4, FAKE, need, FAKE, 32, 0) == qmv.QMV_EINVAL   # unknown flag
    # fp32 activations exist only for the codebook formats
    assert L(B(gu), FAKE, B(dn), FAKE, FAKE, FAKE, 1, 4, FAKE, need, FAKE, qmv.QMV_FLAG_X_F32, 0) == qmv.QMV_EINVAL
    d = qmv.wdesc("mxfp4", 64, 64)
    assert qmv.lib.qmv_dense_ex(B(d), FAKE, FAKE, 1, FAKE, qmv.QMV_FLAG_X_F32, 0) == qmv.QMV_EINVAL


def test_combine_argument_errors():
    B = qmv.ctypes.byref
    dn = qmv.wdesc("mxfp4", 2880, 2880, 32)
    C = qmv.lib.qmv_moe_combine
    assert C(B(dn), None, FAKE, FAKE, 1, 4, FAKE, 0) == qmv.QMV_EINVAL
    assert C(B(dn), FAKE, None, FAKE, 1, 4, FAKE, 0) == qmv.QMV_EINVAL
    assert C(B(dn), FAKE, FAKE, FAKE, 0, 4, FAKE, 0) == qmv.QMV_EINVAL
    assert C(B(dn), FAKE, FAKE, FAKE, 1, 9, FAKE, 0) == qmv.QMV_EINVAL
    assert C(B(dn), FAKE, FAKE + 4, FAKE, 1, 4, FAKE, 0) == qmv.QMV_EALIGN
    assert C(None, FAKE, FAKE, FAKE, 1, 4, FAKE, 0) == qmv.QMV_EINVAL
    gu = qmv.wdesc("mxfp4", 2880, 2880, 32)
    layer = qmv.qmv_moe_layer_workspace_bytes(gu, 2, 4)
    need = qmv.qmv_moe_layer_combine_workspace_bytes(gu, dn, 2, 4)
    assert need == layer + (2 * 4 * 2880 * 2 + 255) // 256 * 256
    cg = qmv.wdesc("cb2", 2048, 7168, 64)
    cd = qmv.wdesc("cb3", 7168, 2048, 64)
    assert qmv.qmv_moe_layer_combine_workspace_bytes(cg, cd, 1, 4) == 4 * 2048 * 4 + 4 * 7168 * 4
    assert qmv.qmv_moe_layer_combine_workspace_bytes(cg, cd, 0, 4) == 0
    L = qmv.lib.qmv_moe_layer_combine
    assert L(B(gu), FAKE, B(dn), FAKE, FAKE, FAKE, FAKE, 2, 4, FAKE, need - 16, FAKE, 0, 0) == qmv.QMV_ESIZE
    assert L(B(gu), FAKE, B(dn), FAKE, FAKE, FAKE, None, 2, 4, FAKE, need, FAKE, 0, 0) == qmv.QMV_EINVAL
    assert L(B(gu), FAKE, B(dn), FAKE, FAKE, FAKE, FAKE, 2, 4, None, need, FAKE, 0, 0) == qmv.QMV_ESIZE
    assert L(B(gu), FAKE, B(dn), FAKE, FAKE, FAKE, FAKE, 2, 4, FAKE, need, FAKE, 32, 0) == qmv.QMV_EINVAL
