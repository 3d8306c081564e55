"""Every entry of the forward dispatch table against the fp64 oracle.

``attn_dispatch`` names the table entry a call runs (tile mode, unit order,
O store, per D and dtype).  Each 16-bit one-pass entry is exercised here on
a small shape chosen to land on it, every output element compared with the
oracle, and the list is checked to cover the whole table.
"""
import itertools

import pytest
import torch

import attention_attn_fwd_gb300 as attn
from attention_attn_fwd_gb300.inputs import Workload
from tests.gpu_parity import check_full

# (Hq, Hkv, Sq, Skv, causal, input_pos): shapes for each tile mode x order.
SHAPES = {
    # two query heads per unit (even group), causal from position 0:
    # heaviest row block first
    ("paired-heads", "lpt"): (4, 2, 300, 300, True, 0),
    # ... no mask: the row blocks of a head in turn
    ("paired-heads", "head-major"): (4, 2, 300, 400, False, 0),
    # 256 rows of one head per unit (odd group)
    ("256-rows", "lpt"): (3, 3, 520, 520, True, 0),
    ("256-rows", "head-major"): (3, 1, 300, 257, False, 0),
    # few query rows: the heads of a K/V group packed into one tile
    ("gqa-packed", "lpt"): (8, 2, 3, 700, True, 697),
}


def entry_cases():
    for D, dt in itertools.product((64, 128), ("f16", "bf16")):
        for (mode, order), shp in SHAPES.items():
            Hq, Hkv, Sq, Skv, causal, pos = shp
            yield Workload("%s_%s_d%d_%s" % (mode, order, D, dt), 1, Hq, Hkv,
                           Sq, Skv, D, dt, causal, pos)


CASES = list(entry_cases())


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build()


def entry(w):
    dt = attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_F16
    return attn.attn_dispatch(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D,
                              int(w.causal), w.input_pos, dt)


def test_cases_cover_the_table():
    """Host only: the shapes above reach every 16-bit one-pass entry but
    the plan entries (test_plan_entries_named)."""
    names = {entry(w)["name"] for w in CASES}
    want = set()
    for D, dt in itertools.product(("64", "128"), ("f16", "bf16")):
        for mode in ("paired-heads", "256-rows"):
            for order in ("lpt", "head-major"):
                want.add("d%s.%s.%s.%s.tma" % (D, dt, mode, order))
        want.add("d%s.%s.gqa-packed.lpt.rows" % (D, dt))
    assert names == want, sorted(want - names)


def test_plan_entries_named():
    """Host only: causal one-pass launches of more units than SMs (and at
    most 1024) run the plan entries, one per tile mode and D among the
    planned launches whose every element test_parity_gpu.py compares with
    the oracle (the plan decision uses 152 SMs without a device)."""
    from tests.test_parity_gpu import PLANNED
    names = {entry(w)["name"] for w in PLANNED}
    want = {"d128.bf16.256-rows.plan.tma", "d64.f16.paired-heads.plan.tma",
            "d64.bf16.256-rows.plan.tma", "d128.f16.paired-heads.plan.tma"}
    assert names == want


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_entry_against_oracle(w):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    name = entry(w)["name"]
    mode = w.name.split("_")[0]
    assert mode in name
    check_full(w, seed=71)
