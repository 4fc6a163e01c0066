"""Python binding of libqmv (include/qmv.h): GB300 block-quantized decode matvec.

Argument marshalling only -- every step of the computation runs in the CUDA
library. Device buffers are torch CUDA tensors (or raw device addresses);
host buffers are numpy arrays. Each function has the name of the C entry
point it calls and raises QmvError when that entry point returns an error.

The library is built in-tree by ``python bit_quantized_moe_gb300/build.py``
(or ``__graft_entry__.build()``). Importing this package without the built
library raises ImportError: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np
import torch  # noqa: F401  (load PyTorch's CUDA runtime first; libqmv binds to the same one)

_PKG = os.path.dirname(os.path.abspath(__file__))
# QMV_LIB selects another build of the same library (the phase-probe variant
# that bench.py --phase-probe builds); the default is the in-tree product build.
LIB_PATH = os.environ.get("QMV_LIB") or os.path.join(_PKG, "_build", "libqmv.so")

QMV_OK = 0
QMV_EINVAL = -1
QMV_ESHAPE = -2
QMV_EALIGN = -3
QMV_ESIZE = -4
QMV_ECUDA = -5
QMV_FLAG_PREFETCH_INPUTS = 1
QMV_FLAG_X_F32 = 2
QMV_FLAG_X_F16 = 4
QMV_FLAG_PATH_TENSOR = 8
QMV_FLAG_PATH_CUDA_CORES = 16
QMV_NOALLOC_SCRATCH_BYTES = 1 << 20

MXFP4, CB2, CB3, CB4, MXFP8 = 0, 1, 2, 3, 4
FORMATS = {"mxfp4": MXFP4, "cb2": CB2, "cb3": CB3, "cb4": CB4, "mxfp8": MXFP8}
MAX_NTOK = 16
MAX_SLOTS = 128
MAX_LAYER_SLOTS = 32
MAX_TOPK = 8

# Every symbol include/qmv.h declares.
EXPORTS = (
    "qmv_scale_group", "qmv_code_bits", "qmv_canonical_code_bytes", "qmv_canonical_scale_bytes",
    "qmv_packed_expert_bytes", "qmv_packed_bytes", "qmv_pack_weights", "qmv_unpack_weights",
    "qmv_act_q8_vec_bytes", "qmv_act_q8_bytes", "qmv_quantize_act_q8", "qmv_act_q8_unpack",
    "qmv_dense", "qmv_moe_gather", "qmv_dense_ex", "qmv_moe_gather_ex", "qmv_packed_gate_up_expert_bytes",
    "qmv_pack_gate_up", "qmv_moe_gate_up_swiglu", "qmv_moe_layer_workspace_bytes", "qmv_moe_layer",
    "qmv_moe_layer_noalloc", "qmv_moe_combine", "qmv_moe_combine_ex", "qmv_moe_layer_combine_workspace_bytes", "qmv_moe_layer_combine",
    "qmv_swiglu_bf16", "qmv_debug_block_sums", "qmv_debug_block_sums_ex", "qmv_debug_path", "qmv_debug_dequant", "qmv_debug_plan",
    "qmv_device_status", "qmv_debug_wait_probe", "qmv_debug_chunk_rate", "qmv_debug_phase_entries",
    "qmv_debug_phase_probe",
    "qmv_debug_phase_read", "qmv_last_error", "qmv_version",
)


class QmvError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"qmv error {code}: {message}")
        self.code = code


class WDesc(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("lut", ctypes.c_int8 * 16)]


def wdesc(fmt, N: int, K: int, n_experts: int = 1, lut: Optional[Sequence[int]] = None) -> WDesc:
    d = WDesc()
    d.fmt = FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
    d.N, d.K, d.n_experts = int(N), int(K), int(n_experts)
    if lut is not None:
        for i, v in enumerate(lut):
            d.lut[i] = int(v)
    return d


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libqmv is not built ({LIB_PATH} missing); run "
                          "`python bit_quantized_moe_gb300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    D = ctypes.POINTER(WDesc)
    sig = {
        "qmv_scale_group": (I32, [I32]),
        "qmv_code_bits": (I32, [I32]),
        "qmv_canonical_code_bytes": (SZ, [D]),
        "qmv_canonical_scale_bytes": (SZ, [D]),
        "qmv_packed_expert_bytes": (SZ, [D]),
        "qmv_packed_bytes": (SZ, [D]),
        "qmv_pack_weights": (ctypes.c_int, [D, P, P, P, SZ]),
        "qmv_unpack_weights": (ctypes.c_int, [D, P, SZ, P, P]),
        "qmv_act_q8_vec_bytes": (SZ, [I32]),
        "qmv_act_q8_bytes": (SZ, [I32, I32]),
        "qmv_quantize_act_q8": (ctypes.c_int, [P, I32, I32, P, SZ, P]),
        "qmv_act_q8_unpack": (ctypes.c_int, [P, I32, I32, P, P]),
        "qmv_dense": (ctypes.c_int, [D, P, P, I32, P, P]),
        "qmv_moe_gather": (ctypes.c_int, [D, P, P, I32, P, I32, I32, P, P]),
        "qmv_dense_ex": (ctypes.c_int, [D, P, P, I32, P, ctypes.c_uint32, P]),
        "qmv_packed_gate_up_expert_bytes": (SZ, [D]),
        "qmv_pack_gate_up": (ctypes.c_int, [D, P, P, P, P, P, SZ]),
        "qmv_moe_gate_up_swiglu": (ctypes.c_int, [D, P, P, P, I32, I32, P, ctypes.c_uint32, P]),
        "qmv_moe_layer_workspace_bytes": (SZ, [D, I32, I32]),
        "qmv_moe_layer": (ctypes.c_int, [D, P, D, P, P, P, I32, I32, P, SZ, P, ctypes.c_uint32, P]),
        "qmv_moe_layer_noalloc": (ctypes.c_int, [D, P, D, P, P, P, I32, I32, P, ctypes.c_uint32, P]),
        "qmv_moe_combine": (ctypes.c_int, [D, P, P, P, I32, I32, P, P]),
        "qmv_moe_combine_ex": (ctypes.c_int, [D, P, P, P, I32, I32, P, ctypes.c_uint32, P]),
        "qmv_moe_layer_combine_workspace_bytes": (SZ, [D, D, I32, I32]),
        "qmv_moe_layer_combine": (ctypes.c_int, [D, P, D, P, P, P, P, I32, I32, P, SZ, P, ctypes.c_uint32, P]),
        "qmv_moe_gather_ex": (ctypes.c_int, [D, P, P, I32, P, I32, I32, P, ctypes.c_uint32, P]),
        "qmv_swiglu_bf16": (ctypes.c_int, [P, P, P, I64, P]),
        "qmv_debug_block_sums": (ctypes.c_int, [D, P, P, I32, P, I32, I32, P, P, SZ, P]),
        "qmv_debug_block_sums_ex": (ctypes.c_int, [D, P, P, I32, P, I32, I32, P, P, SZ, ctypes.c_uint32, P]),
        "qmv_debug_path": (ctypes.c_int, [D, I32, I32, I32, I32, ctypes.c_uint32, P, I32]),
        "qmv_debug_dequant": (ctypes.c_int, [D, P, I32, P, SZ, P]),
        "qmv_debug_plan": (ctypes.c_int, [D, I32, I32, I32, I32, ctypes.c_uint32, I32, I32, I64,
                                          ctypes.POINTER(I64), I32]),
        "qmv_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), I32]),
        "qmv_debug_wait_probe": (ctypes.c_int, [ctypes.c_uint64, P]),
        "qmv_debug_chunk_rate": (ctypes.c_int, [I32, I32, I32, I32, P, SZ, ctypes.POINTER(I64),
                                                ctypes.POINTER(I64), P]),
        "qmv_debug_phase_entries": (SZ, []),
        "qmv_debug_phase_probe": (ctypes.c_int, [I32]),
        "qmv_debug_phase_read": (ctypes.c_int, [I32, P, SZ, I32]),
        "qmv_last_error": (ctypes.c_char_p, []),
        "qmv_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def _check(rc: int) -> None:
    if rc != QMV_OK:
        raise QmvError(rc, lib.qmv_last_error().decode())


def _ptr(t) -> Optional[int]:
    """Device/host address of a torch tensor, numpy array or int (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _nbytes(t) -> int:
    if isinstance(t, np.ndarray):
        return t.nbytes
    return t.numel() * t.element_size()


# --- sizes -----------------------------------------------------------------

def qmv_scale_group(fmt) -> int:
    return lib.qmv_scale_group(FORMATS.get(fmt, fmt) if isinstance(fmt, str) else fmt)


def qmv_code_bits(fmt) -> int:
    return lib.qmv_code_bits(FORMATS.get(fmt, fmt) if isinstance(fmt, str) else fmt)


def qmv_canonical_code_bytes(desc: WDesc) -> int:
    return lib.qmv_canonical_code_bytes(ctypes.byref(desc))


def qmv_canonical_scale_bytes(desc: WDesc) -> int:
    return lib.qmv_canonical_scale_bytes(ctypes.byref(desc))


def qmv_packed_expert_bytes(desc: WDesc) -> int:
    return lib.qmv_packed_expert_bytes(ctypes.byref(desc))


def qmv_packed_bytes(desc: WDesc) -> int:
    return lib.qmv_packed_bytes(ctypes.byref(desc))


def qmv_act_q8_vec_bytes(K: int) -> int:
    return lib.qmv_act_q8_vec_bytes(K)


def qmv_act_q8_bytes(nvec: int, K: int) -> int:
    return lib.qmv_act_q8_bytes(nvec, K)


# --- host packer -------------------------------------------------------------

def qmv_pack_weights(desc: WDesc, codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Canonical packed codes [E][...] and E8M0 scales [E][N][K/group] -> GPU layout bytes."""
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    E = desc.n_experts
    if codes.nbytes != E * qmv_canonical_code_bytes(desc) or scales.nbytes != E * qmv_canonical_scale_bytes(desc):
        raise ValueError("codes/scales do not match the descriptor's canonical sizes")
    out = np.empty(qmv_packed_bytes(desc), dtype=np.uint8)
    _check(lib.qmv_pack_weights(ctypes.byref(desc), codes.ctypes.data, scales.ctypes.data,
                                out.ctypes.data, out.nbytes))
    return out


def qmv_packed_gate_up_expert_bytes(desc: WDesc) -> int:
    return lib.qmv_packed_gate_up_expert_bytes(ctypes.byref(desc))


def qmv_pack_gate_up(desc: WDesc, gate_codes, gate_scales, up_codes, up_scales) -> np.ndarray:
    """Canonical gate and up codes/scales (each as for qmv_pack_weights) -> fused GPU layout bytes."""
    arrs = [np.ascontiguousarray(a, dtype=np.uint8) for a in (gate_codes, gate_scales, up_codes, up_scales)]
    E = desc.n_experts
    if (arrs[0].nbytes != E * qmv_canonical_code_bytes(desc) or arrs[2].nbytes != arrs[0].nbytes
            or arrs[1].nbytes != E * qmv_canonical_scale_bytes(desc) or arrs[3].nbytes != arrs[1].nbytes):
        raise ValueError("gate/up codes or scales do not match the descriptor's canonical sizes")
    out = np.empty(E * qmv_packed_gate_up_expert_bytes(desc), dtype=np.uint8)
    _check(lib.qmv_pack_gate_up(ctypes.byref(desc), *[a.ctypes.data for a in arrs], out.ctypes.data, out.nbytes))
    return out


def qmv_unpack_weights(desc: WDesc, packed: np.ndarray):
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    E = desc.n_experts
    codes = np.empty(E * qmv_canonical_code_bytes(desc), dtype=np.uint8)
    scales = np.empty(E * qmv_canonical_scale_bytes(desc), dtype=np.uint8)
    _check(lib.qmv_unpack_weights(ctypes.byref(desc), packed.ctypes.data, packed.nbytes,
                                  codes.ctypes.data, scales.ctypes.data))
    return codes, scales


def qmv_act_q8_unpack(xq_host: np.ndarray, nvec: int, K: int):
    q = np.empty((nvec, K), dtype=np.int8)
    d = np.empty((nvec, K // 32), dtype=np.uint16)
    xq_host = np.ascontiguousarray(xq_host, dtype=np.uint8)
    _check(lib.qmv_act_q8_unpack(xq_host.ctypes.data, nvec, K, q.ctypes.data, d.ctypes.data))
    return q, d


# --- GPU entry points ----------------------------------------------------------

def qmv_quantize_act_q8(x, nvec: int, K: int, xq, stream=None) -> None:
    _check(lib.qmv_quantize_act_q8(_ptr(x), nvec, K, _ptr(xq), _nbytes(xq), _stream(stream)))


def qmv_dense(desc: WDesc, w, x, ntok: int, y, stream=None) -> None:
    _check(lib.qmv_dense(ctypes.byref(desc), _ptr(w), _ptr(x), ntok, _ptr(y), _stream(stream)))


def qmv_moe_gather(desc: WDesc, w, x, per_slot_x: int, ids, ntok: int, top_k: int, y, stream=None) -> None:
    _check(lib.qmv_moe_gather(ctypes.byref(desc), _ptr(w), _ptr(x), int(per_slot_x), _ptr(ids), ntok,
                              top_k, _ptr(y), _stream(stream)))


def qmv_dense_ex(desc: WDesc, w, x, ntok: int, y, flags: int, stream=None) -> None:
    _check(lib.qmv_dense_ex(ctypes.byref(desc), _ptr(w), _ptr(x), ntok, _ptr(y), int(flags), _stream(stream)))


def qmv_moe_gather_ex(desc: WDesc, w, x, per_slot_x: int, ids, ntok: int, top_k: int, y, flags: int,
                      stream=None) -> None:
    _check(lib.qmv_moe_gather_ex(ctypes.byref(desc), _ptr(w), _ptr(x), int(per_slot_x), _ptr(ids), ntok, top_k,
                                 _ptr(y), int(flags), _stream(stream)))


def qmv_moe_gate_up_swiglu(desc: WDesc, w, x, ids, ntok: int, top_k: int, h, flags: int = 0,
                           stream=None) -> None:
    _check(lib.qmv_moe_gate_up_swiglu(ctypes.byref(desc), _ptr(w), _ptr(x), _ptr(ids), ntok, top_k, _ptr(h),
                                      int(flags), _stream(stream)))


def qmv_moe_layer_workspace_bytes(gate_up_desc: WDesc, ntok: int, top_k: int) -> int:
    return lib.qmv_moe_layer_workspace_bytes(ctypes.byref(gate_up_desc), ntok, top_k)


def qmv_moe_layer(gate_up_desc: WDesc, w_gate_up, down_desc: WDesc, w_down, x, ids, ntok: int, top_k: int,
                  workspace, y, flags: int = 0, stream=None) -> None:
    _check(lib.qmv_moe_layer(ctypes.byref(gate_up_desc), _ptr(w_gate_up), ctypes.byref(down_desc), _ptr(w_down),
                             _ptr(x), _ptr(ids), ntok, top_k, _ptr(workspace), _nbytes(workspace), _ptr(y),
                             int(flags), _stream(stream)))


def qmv_moe_layer_noalloc(gate_up_desc: WDesc, w_gate_up, down_desc: WDesc, w_down, x, ids, ntok: int, top_k: int,
                          y, flags: int = 0, stream=None) -> None:
    """qmv_moe_layer without a workspace, for callers that may not allocate
    device memory: the scratch is a static array inside the library (see
    include/qmv.h for its size, sharing and first-call rules)."""
    _check(lib.qmv_moe_layer_noalloc(ctypes.byref(gate_up_desc), _ptr(w_gate_up), ctypes.byref(down_desc),
                                     _ptr(w_down), _ptr(x), _ptr(ids), ntok, top_k, _ptr(y), int(flags),
                                     _stream(stream)))


def qmv_moe_combine(down_desc: WDesc, ys, weights, ids, ntok: int, top_k: int, y, stream=None) -> None:
    _check(lib.qmv_moe_combine(ctypes.byref(down_desc), _ptr(ys), _ptr(weights), _ptr(ids), ntok, top_k, _ptr(y),
                               _stream(stream)))


def qmv_moe_combine_ex(down_desc: WDesc, ys, weights, ids, ntok: int, top_k: int, y, flags: int,
                       stream=None) -> None:
    _check(lib.qmv_moe_combine_ex(ctypes.byref(down_desc), _ptr(ys), _ptr(weights), _ptr(ids), ntok, top_k,
                                  _ptr(y), int(flags), _stream(stream)))


def qmv_moe_layer_combine_workspace_bytes(gate_up_desc: WDesc, down_desc: WDesc, ntok: int, top_k: int) -> int:
    return lib.qmv_moe_layer_combine_workspace_bytes(ctypes.byref(gate_up_desc), ctypes.byref(down_desc), ntok,
                                                     top_k)


def qmv_moe_layer_combine(gate_up_desc: WDesc, w_gate_up, down_desc: WDesc, w_down, x, ids, weights, ntok: int,
                          top_k: int, workspace, y, flags: int = 0, stream=None) -> None:
    _check(lib.qmv_moe_layer_combine(ctypes.byref(gate_up_desc), _ptr(w_gate_up), ctypes.byref(down_desc),
                                     _ptr(w_down), _ptr(x), _ptr(ids), _ptr(weights), ntok, top_k,
                                     _ptr(workspace), _nbytes(workspace), _ptr(y), int(flags), _stream(stream)))


def qmv_swiglu_bf16(g, u, h, n: int, stream=None) -> None:
    _check(lib.qmv_swiglu_bf16(_ptr(g), _ptr(u), _ptr(h), int(n), _stream(stream)))


def qmv_debug_block_sums(desc: WDesc, w, x, per_slot_x: int, ids, ntok: int, top_k: int, y, sums,
                         stream=None, flags: int = 0) -> None:
    _check(lib.qmv_debug_block_sums_ex(ctypes.byref(desc), _ptr(w), _ptr(x), int(per_slot_x), _ptr(ids), ntok,
                                       top_k, _ptr(y), _ptr(sums), _nbytes(sums), int(flags), _stream(stream)))


def qmv_debug_path(desc: WDesc, ntok: int, top_k: int = 1, gather: bool = False, glu: bool = False,
                   flags: int = 0):
    """(tensor cores?, tokens per CUDA-core launch) of a call (host only)."""
    out = (ctypes.c_int64 * 2)()
    _check(lib.qmv_debug_path(ctypes.byref(desc), int(ntok), int(top_k), int(bool(gather)), int(bool(glu)),
                              int(flags), out, 2))
    return bool(out[0]), int(out[1])


def qmv_debug_dequant(desc: WDesc, w, expert: int, out, stream=None) -> None:
    _check(lib.qmv_debug_dequant(ctypes.byref(desc), _ptr(w), expert, _ptr(out), _nbytes(out),
                                 _stream(stream)))


PLAN_FIELDS = ("nv", "warps", "stages", "items", "grid", "splits", "split_chunks", "items_per_cta", "x_slots",
               "contig", "smem", "row_tiles")


def qmv_debug_plan(desc: WDesc, ntok: int, top_k: int, gather: bool, per_slot_x: bool, flags: int = 0,
                   sm_count: int = 152, ctas_per_sm: int = 2, smem_per_sm: int = 233472) -> dict:
    """The CUDA-core matvec's launch plan for a call and device shape (host only)."""
    out = (ctypes.c_int64 * 12)()
    _check(lib.qmv_debug_plan(ctypes.byref(desc), ntok, top_k, int(gather), int(per_slot_x), int(flags), sm_count,
                              ctas_per_sm, smem_per_sm, out, 12))
    return dict(zip(PLAN_FIELDS, list(out)))


def qmv_device_status(clear: bool = False) -> int:
    v = ctypes.c_uint32(0)
    _check(lib.qmv_device_status(ctypes.byref(v), 1 if clear else 0))
    return v.value


def qmv_debug_wait_probe(limit_ns: int, stream=None) -> None:
    _check(lib.qmv_debug_wait_probe(int(limit_ns), _stream(stream)))


def qmv_debug_chunk_rate(fmt, nv: int, ctas_per_sm: int, iters: int, sink=None, stream=None):
    """Launches the compute-rate probe (or, with sink None, only sizes it);
    returns (matrix weights per launch, threads = sink entries)."""
    w, t = ctypes.c_int64(0), ctypes.c_int64(0)
    f = FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
    _check(lib.qmv_debug_chunk_rate(f, nv, ctas_per_sm, iters, _ptr(sink), _nbytes(sink) if sink is not None else 0,
                                    ctypes.byref(w), ctypes.byref(t), _stream(stream)))
    return w.value, t.value


PHASES = ("start", "work_list", "early_tiles", "dep_wait", "act_loads", "ring_issued", "act_staged",
          "tile0_ready", "tile0_done", "tile1_ready", "tile2_ready", "last_done", "end")


def qmv_debug_phase_probe(enable: bool) -> None:
    """Record the phases of the matvec launches made from now on (phase-probe
    build only; raises QmvError in the product build)."""
    _check(lib.qmv_debug_phase_probe(1 if enable else 0))


def qmv_debug_phase_read(fmt, clear: bool = True) -> np.ndarray:
    """The format's phase stamps, uint64 ns [slot][cta][warp][phase] (0 = not
    recorded). Synchronizes the device."""
    n = lib.qmv_debug_phase_entries()
    out = np.zeros(n, dtype=np.uint64)
    f = FORMATS[fmt] if isinstance(fmt, str) else int(fmt)
    _check(lib.qmv_debug_phase_read(f, out.ctypes.data, n, 1 if clear else 0))
    return out.reshape(8, 512, 16, 16)


def qmv_last_error() -> str:
    return lib.qmv_last_error().decode()


def qmv_version() -> str:
    return lib.qmv_version().decode()
