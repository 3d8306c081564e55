"""Host-side unit plan of causal two-tile forward launches (attn_unit_plan).

A planned launch walks the units its plan gives each persistent CTA
instead of the zigzag rounds; the plan must give every unit to exactly one
CTA, and its busiest CTA must carry no more work than under the rounds.
The work of a unit is recomputed here from the causal extents of its rows
(independently of the library's arithmetic) and the reported figures are
checked against it.
"""
import pytest

import attention_attn_fwd_gb300 as attn


def unit_work(B, Hq, Hkv, Sq, Skv, causal, input_pos):
    """Half K/V steps of each unit: 2 per key tile its later Q tile sees
    (from key 0), plus 3; units numbered heaviest row block first, the
    heads of a row block in turn."""
    group = Hq // Hkv
    paired = group % 2 == 0
    rows = 128 if paired else 256
    m_blocks = (Sq + rows - 1) // rows
    per_m = B * (Hq // 2) if paired else B * Hq
    work = []
    for u in range(m_blocks * per_m):
        mb = m_blocks - 1 - u // per_m
        last_row = min(mb * rows + rows, Sq) - 1
        if not paired and mb * rows + 128 >= Sq:
            last_row = min(mb * rows + 128, Sq) - 1
        keys = min(input_pos + last_row + 1, Skv) if causal else Skv
        work.append(2 * ((keys + 127) // 128) + 3)
    return work


def zigzag_max(work, grid):
    load = [0] * grid
    for u, w in enumerate(work):
        k, r = divmod(u, grid)
        load[grid - 1 - r if k & 1 else r] += w
    return max(load)


SHAPES = [
    (1, 32, 4, 8192, 8192, 0),      # GQA 8k (paired heads)
    (1, 32, 32, 4096, 4096, 0),     # MHA 4k (256-row units)
    (8, 32, 8, 512, 4096, 3584),    # prefill chunk (causal offset)
    (2, 20, 4, 1800, 1800, 0),      # group 5, ragged rows, batch 2
    (1, 32, 8, 2560, 3000, 400),    # causal offset: rounds 16 % over the plan
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_plan_assigns_every_unit_once(shape):
    B, Hq, Hkv, Sq, Skv, pos = shape
    r = attn.attn_unit_plan(B, Hq, Hkv, Sq, Skv, 128, True, pos, grid=152)
    work = unit_work(B, Hq, Hkv, Sq, Skv, True, pos)
    assert r["units"] == len(work)
    rounds = zigzag_max(work, min(152, len(work)))
    assert r["work_rounds"] == rounds
    assert r["planned"] == 1
    cta_units = r["cta_units"]
    assert len(cta_units) == 152
    assert sorted(u for units in cta_units for u in units) == \
        list(range(len(work)))
    loads = [sum(work[u] for u in units) for units in cta_units]
    assert max(loads) == r["work_max"] < rounds
    # Within one unit of the mean (the list-scheduling bound).
    mean = sum(work) / 152
    assert max(loads) <= mean + max(work)
    # Each CTA walks its units heaviest first.
    for units in cta_units:
        w = [work[u] for u in units]
        assert w == sorted(w, reverse=True)


@pytest.mark.parametrize("args", [
    (4, 16, 16, 8192, 8192, False, 0),   # non-causal: equal units
    (1, 4, 2, 512, 512, True, 0),        # 8 units on 8 CTAs
    (4, 32, 8, 8, 4096, True, 4088),     # few rows: packed GQA tiles
    (1, 32, 4, 32768, 32768, True, 0),   # 4096 units: more than a plan holds
])
def test_launches_without_plan(args):
    B, Hq, Hkv, Sq, Skv, causal, pos = args
    r = attn.attn_unit_plan(B, Hq, Hkv, Sq, Skv, 128, causal, pos, grid=152)
    assert r["planned"] == 0 and "cta_units" not in r


def test_plan_rejects_bad_arguments():
    with pytest.raises(attn.AttnError):
        attn.attn_unit_plan(1, 3, 2, 128, 128, 128, True, 0, grid=152)
    with pytest.raises(attn.AttnError):
        attn.attn_unit_plan(1, 32, 4, 8192, 8192, 128, True, 0, grid=0)
