"""The CUDA-core matvec's launch planner, checked on the host against a
simulation of the kernel's work dealing (no GPU): for every call the library
accepts (validation rejects a call whose two-CTA plan does not fit the
per-block shared-memory limit) and every entry count the call can produce,
each CTA's items fit the split-K partial slots, a CTA of a contiguously
dealt call touches no more activation vectors than its staged region holds
(else the kernel records a planning error), and the plan the launcher may
use -- two CTAs per SM, or one when two do not fit -- fits the device."""
import itertools

import pytest

qmv = pytest.importorskip("bit_quantized_moe_gb300")

SMS, SMEM_SM, OPTIN = 152, 233472, 232448


def deal(n_items, grid, contig, b):
    """Items of CTA b: (first, stride, count), as the kernel deals them."""
    if contig:
        per, rem = divmod(n_items, grid)
        return b * per + min(b, rem), 1, per + (1 if b < rem else 0)
    return b, grid, (n_items - b + grid - 1) // grid if b < n_items else 0


def accepted(desc, ntok, top_k, gather, per_slot):
    """The library's validation: the two-CTA plan plus the kernel's static
    shared memory (256 bytes allowed) within the per-block limit."""
    p2 = qmv.qmv_debug_plan(desc, ntok, top_k, gather, per_slot, sm_count=SMS, ctas_per_sm=2, smem_per_sm=SMEM_SM)
    return p2["smem"] + 256 <= OPTIN


def check_plan(desc, ntok, top_k, gather, per_slot, ctas):
    p = qmv.qmv_debug_plan(desc, ntok, top_k, gather, per_slot, sm_count=SMS, ctas_per_sm=ctas,
                           smem_per_sm=SMEM_SM)
    if not accepted(desc, ntok, top_k, gather, per_slot):
        return None
    rt, nv = p["row_tiles"], p["nv"]
    nvec = ntok * top_k if (gather and per_slot) else ntok
    max_entries = p["items"] // rt
    assert p["grid"] <= SMS * ctas and p["grid"] <= p["items"]
    assert p["smem"] + 1024 <= OPTIN
    if not p["contig"]:
        assert p["x_slots"] == nvec
    for n_ent in range(1, max_entries + 1):
        n_items = n_ent * rt
        for b in range(p["grid"]):
            first, stride, count = deal(n_items, p["grid"], p["contig"], b)
            assert count <= p["items_per_cta"], (n_ent, b)
            if p["contig"] and count > 0:
                e0, e1 = first // rt, (first + count - 1) // rt
                assert (e1 - e0 + 1) * nv <= p["x_slots"] or p["x_slots"] == nvec, (n_ent, b, p)
    return p


FMTS = ["mxfp4", "mxfp8", "cb2", "cb3", "cb4"]
SHAPES = [(1, 32), (17, 1056), (516, 2880), (2880, 2880), (7168, 2048), (2048, 7168)]


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ctas", [1, 2])
def test_gather_plans(fmt, ctas):
    for (N, K), (ntok, top_k), per_slot in itertools.product(SHAPES, [(1, 4), (4, 4), (4, 8), (8, 4), (16, 2)],
                                                           [False, True]):
        if fmt in ("cb2", "cb3") and K % 32:
            continue
        check_plan(qmv.wdesc(fmt, N, K, 64), ntok, top_k, True, per_slot, ctas)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("ctas", [1, 2])
def test_dense_plans(fmt, ctas):
    for (N, K), ntok in itertools.product(SHAPES, [1, 3, 4, 5, 8, 13, 16]):
        p = check_plan(qmv.wdesc(fmt, N, K, 1), ntok, 1, False, False, ctas)
        if p is None:
            continue
        assert p["contig"] == (1 if ntok > 4 else 0)
        assert p["nv"] == min(ntok, 4)


def test_decode_shapes_are_accepted():
    """Every decode-path configuration of the workloads passes validation."""
    cases = [("mxfp4", 2880, 2880, 32, 1, 4, True, False), ("mxfp4", 2880, 2880, 32, 1, 4, True, True),
             ("cb2", 4096, 7168, 256, 1, 4, True, False), ("cb3", 7168, 2048, 256, 4, 4, True, True),
             ("cb4", 7168, 7168, 1, 4, 1, False, False), ("mxfp8", 5760, 2880, 32, 4, 8, True, False),
             ("mxfp4", 5760, 2880, 32, 8, 4, True, False), ("cb2", 4096, 7168, 64, 8, 4, True, False)]
    for fmt, N, K, E, ntok, top_k, gather, per_slot in cases:
        assert accepted(qmv.wdesc(fmt, N, K, E), ntok, top_k, gather, per_slot), (fmt, N, K, ntok, top_k)


def test_compact_region_only_when_needed():
    # the MXFP4 down gather of the decode layer keeps every vector at its own index
    p = qmv.qmv_debug_plan(qmv.wdesc("mxfp4", 2880, 2880, 32), 1, 4, True, True)
    assert p["x_slots"] == 4 and p["contig"] == 1
    # 32 per-slot vectors of K = 4096 cannot all sit beside the ring: compact
    p = qmv.qmv_debug_plan(qmv.wdesc("mxfp4", 1032, 4096, 16), 4, 8, True, True)
    assert p["x_slots"] < 32


def test_plan_argument_errors():
    d = qmv.wdesc("mxfp4", 64, 64, 8)
    with pytest.raises(qmv.QmvError):
        qmv.qmv_debug_plan(d, 8, 8, True, True)          # 64 slots: not a CUDA-core gather
    with pytest.raises(qmv.QmvError):
        qmv.qmv_debug_plan(d, 1, 4, True, True, sm_count=0)


def sorted_gather_items(ids, n_experts, group=16):
    """The sorted gather's work items in the kernel's order: experts by first
    slot, each expert's slots (in slot order) cut into groups of <= 16."""
    flat = [int(e) for e in ids.reshape(-1)]
    items = []
    for s, e in enumerate(flat):
        if not (0 <= e < n_experts) or e in flat[:s]:
            continue
        slots = [q for q, eq in enumerate(flat) if eq == e]
        for g0 in range(0, len(slots), group):
            items.append((e, slots[g0:g0 + group]))
    return items


def test_sorted_gather_items_cover_slots_within_grid_bound():
    import numpy as np
    rng = np.random.default_rng(5)
    for trial in range(300):
        ntok = int(rng.integers(1, 17))
        top_k = int(rng.integers(1, 9))
        E = int(rng.choice([1, 2, 8, 32, 256]))
        ids = rng.integers(-2, E + 2, size=(ntok, top_k))
        if trial % 3 == 0:
            ids[:, 0] = 0                       # one expert in every token
        n = ntok * top_k
        items = sorted_gather_items(ids, E)
        cap = (n + 15) // 16 + min(E, n)       # the launcher's grid.y
        assert len(items) <= cap
        covered = sorted(s for _, group in items for s in group)
        valid = [s for s, e in enumerate(ids.reshape(-1)) if 0 <= e < E]
        assert covered == valid                 # every valid slot exactly once
        assert all(1 <= len(g) <= 16 for _, g in items)


# ---------------------------------------------------------------------------
# Tensor cores or CUDA cores: the cost model of the verify batch and of
# gathers beyond 32 routed slots, and the QMV_FLAG_PATH_* overrides
# ---------------------------------------------------------------------------

def test_path_dense_verify_batches():
    """MX dense calls of 5..16 bf16 tokens take the tensor cores (not 1..4
    tokens, not fp16 activations); codebook ones only when their CUDA-core
    weight streams (one per 4 tokens) exceed 64 MB."""
    P = qmv.qmv_debug_path
    mx = qmv.wdesc("mxfp4", 2880, 2880)
    assert [P(mx, n)[0] for n in range(1, 17)] == [False] * 4 + [True] * 12
    assert P(mx, 16, flags=qmv.QMV_FLAG_X_F16) == (False, 16)
    assert P(mx, 16, flags=qmv.QMV_FLAG_PATH_CUDA_CORES) == (False, 16)
    assert P(mx, 4, flags=qmv.QMV_FLAG_PATH_TENSOR) == (False, 4)   # no tensor-core form at 4 tokens
    cb4 = qmv.wdesc("cb4", 7168, 7168)                                # 27.3 MB per stream
    assert P(cb4, 16)[0] and P(cb4, 9)[0] and not P(cb4, 8)[0] and not P(cb4, 5)[0]   # 3 streams: 82 MB
    cb3 = qmv.wdesc("cb3", 7168, 2048)
    assert not P(cb3, 16)[0]
    assert P(cb3, 16, flags=qmv.QMV_FLAG_PATH_TENSOR)[0]
    assert P(cb3, 16, flags=qmv.QMV_FLAG_PATH_TENSOR | qmv.QMV_FLAG_X_F32)[0]


@pytest.mark.parametrize("fmt,E,ntok,top_k,tensor", [
    ("mxfp4", 32, 16, 8, True),     # 128 slots, 4 per expert
    ("mxfp4", 32, 16, 4, False),    # 64 slots, 2 per expert
    ("mxfp4", 16, 16, 4, True),     # 64 slots, 4 per expert
    ("mxfp4", 256, 16, 8, False),   # 128 slots, 1 per expert
    ("mxfp8", 8, 9, 4, True),       # 36 slots, 4.5 per expert
    ("cb3", 8, 16, 8, True),        # 128 slots, 16 per expert
    ("cb3", 16, 16, 8, False),      # 128 slots, 8 per expert
    ("cb4", 16, 16, 8, True),       # 128 slots, 8 per expert (A in tensor memory: cheaper per item)
    ("cb4", 32, 16, 8, False),      # 128 slots, 4 per expert
    ("cb2", 8, 16, 8, True),        # 128 slots, 16 per expert
    ("cb2", 2, 16, 2, True),        # 32 slots: the decode gather
])
def test_path_gathers(fmt, E, ntok, top_k, tensor):
    """Gathers of 33..128 routed slots: the sorted tensor-core gather at >= 4
    (MX), >= 8 (CB4) or >= 12 (CB2, CB3) slots per expert that can occur, else CUDA-core
    gathers of 32-slot token ranges; 32 slots or fewer are always the decode
    gather in one launch."""
    lut = {"cb2": [0] * 4, "cb3": [0] * 8, "cb4": [0] * 16}.get(fmt)
    d = qmv.wdesc(fmt, 1024, 2048, E, lut)
    slots = ntok * top_k
    if slots <= 32:
        assert qmv.qmv_debug_path(d, ntok, top_k, gather=True) == (False, ntok)
        return
    assert qmv.qmv_debug_path(d, ntok, top_k, gather=True) == (tensor, 32 // top_k)
    assert qmv.qmv_debug_path(d, ntok, top_k, gather=True, flags=qmv.QMV_FLAG_PATH_TENSOR)[0]
    assert qmv.qmv_debug_path(d, ntok, top_k, gather=True, flags=qmv.QMV_FLAG_PATH_CUDA_CORES) == (False,
                                                                                                  32 // top_k)


def test_path_gate_up_and_fp16_have_no_tensor_form():
    """The fused gate/up and fp16 activations run on the CUDA cores at any slot
    count, split into launches of at most 32 slots; the overrides are
    exclusive."""
    d = qmv.wdesc("mxfp4", 2880, 2880, 32)
    assert qmv.qmv_debug_path(d, 16, 8, gather=True, glu=True) == (False, 4)
    assert qmv.qmv_debug_path(d, 16, 8, gather=True, glu=True, flags=qmv.QMV_FLAG_PATH_TENSOR) == (False, 4)
    assert qmv.qmv_debug_path(d, 16, 8, gather=True, flags=qmv.QMV_FLAG_X_F16) == (False, 4)
    assert qmv.qmv_debug_path(d, 5, 7, gather=True) == (False, 4)   # 35 slots, top-7: 4 tokens per launch
    with pytest.raises(qmv.QmvError):
        qmv.qmv_debug_path(d, 16, 8, gather=True,
                           flags=qmv.QMV_FLAG_PATH_TENSOR | qmv.QMV_FLAG_PATH_CUDA_CORES)
    with pytest.raises(qmv.QmvError):
        qmv.qmv_debug_path(d, 16, 9, gather=True)
