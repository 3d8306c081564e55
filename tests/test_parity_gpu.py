"""GPU parity: the sm_103a kernel (through the C ABI) against the fp64 CPU
oracle, element by element, with max-abs tolerances of 2e-3 (fp16) and
1.5e-2 (bf16) on O and 1e-3 on LSE."""
import numpy as np
import pytest
import torch

import attention_attn_fwd_gb300 as attn
from attention_attn_fwd_gb300.inputs import (GQA_8K, MHA_4K, PREFILL_CHUNK,
                                             SMALL, Workload, make_qkv, sweep)
from tests.gpu_parity import TOL_O, check_full, check_sampled, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_small_workload(seed):
    check_full(SMALL, seed)


def W(name, B, Hq, Hkv, Sq, Skv, D, dt, causal, pos=0):
    return Workload(name, B, Hq, Hkv, Sq, Skv, D, dt, causal, pos)


EDGE = [
    W("one_by_one", 1, 1, 1, 1, 1, 64, "f16", False),
    W("one_query_many_keys", 1, 2, 1, 1, 1000, 128, "bf16", False),
    W("decode_offset", 2, 4, 2, 1, 1000, 128, "f16", True, 999),
    W("decode_offset_mid", 1, 8, 1, 3, 515, 64, "bf16", True, 300),
    W("tiny_causal", 1, 2, 2, 77, 77, 64, "f16", True),
    W("ragged_causal_300", 1, 2, 2, 300, 300, 128, "f16", True),
    W("key_tail_noncausal", 1, 2, 2, 129, 383, 64, "f16", False),
    W("offset_ragged", 1, 2, 1, 200, 330, 128, "bf16", True, 130),
    W("two_tiles_d64_bf16", 1, 2, 2, 256, 256, 64, "bf16", True),
    W("gqa8_offset_ragged", 1, 16, 2, 513, 700, 128, "bf16", True, 187),
    W("mqa_causal", 1, 32, 1, 130, 260, 128, "f16", True),
    W("gqa4_noncausal", 2, 8, 2, 384, 640, 64, "f16", False),
    W("batch3_causal", 3, 4, 4, 384, 384, 128, "f16", True),
    W("offset_beyond_keys", 1, 2, 2, 64, 128, 64, "bf16", True, 5000),
    W("skv_tile_plus_one", 1, 2, 2, 257, 257, 128, "bf16", False),
    W("skv_tile_plus_one_causal", 1, 2, 2, 129, 257, 64, "f16", True, 128),
    W("long_keys_short_q", 1, 4, 4, 40, 2049, 128, "f16", False),
    W("sq_gt_skv_causal", 1, 2, 2, 600, 200, 64, "bf16", True),
    # Head counts that are not powers of two: the unit decode divides by
    # the group (3, 5, 6), by Hq or Hq / 2 and by the units per row block.
    W("gqa3_causal_batch2", 2, 6, 2, 333, 333, 128, "bf16", True),
    W("gqa6_paired_offset", 1, 12, 2, 300, 700, 64, "f16", True, 400),
    W("gqa5_noncausal_batch3", 3, 10, 2, 200, 450, 64, "bf16", False),
    # Few query rows with grouped K/V heads: all heads of a group in one tile.
    W("packed_full_tile", 1, 32, 4, 16, 900, 128, "bf16", True, 884),
    W("packed_ragged", 2, 8, 2, 30, 333, 64, "f16", True, 303),
    W("packed_noncausal", 1, 8, 2, 5, 700, 128, "bf16", False),
    W("packed_one_row", 3, 4, 2, 1, 130, 64, "f16", True, 129),
]


@pytest.mark.parametrize("w", EDGE, ids=lambda w: w.name)
def test_edge_shapes(w):
    check_full(w, seed=3)


@pytest.mark.parametrize("scale", [0.0, -0.0883883, 0.5, 1.0])
def test_scale_values(scale):
    # Peaked softmax (large scale) exercises the rescale path hard; bf16
    # keeps the comparison inside its documented bound.
    w = W("scale", 1, 4, 2, 384, 520, 128, "bf16", True, 7)
    check_full(w, seed=4, scale=scale)


def test_growing_scores_force_rescales():
    """Keys whose scores grow along the sequence move the running maximum
    tile after tile, so O and l are corrected many times."""
    w = W("growing", 1, 2, 2, 256, 1024, 64, "bf16", False)
    q, k, v = make_qkv(w, seed=5)
    ramp = torch.linspace(0.0, 6.0, w.Skv).to(torch.float32)
    k = (k.float() * 0.2 + ramp[None, None, :, None]).to(w.torch_dtype)
    q = (q.float().abs() * 0.3).to(w.torch_dtype)
    check_full(w, q=q, k=k, v=v)


@pytest.mark.parametrize("w", [MHA_4K, GQA_8K, PREFILL_CHUNK],
                         ids=lambda w: w.name)
def test_full_size_workloads(w):
    check_sampled(w, seed=0)


@pytest.mark.parametrize("w", sweep(), ids=lambda w: w.name)
def test_full_size_sweep(w):
    check_sampled(w, seed=1, n_rows=96)


# Causal launches whose units the host packs onto the CTAs (attn_unit_plan):
# every element against the oracle on two that are small enough, and on the
# full-size ones every row written (the plan must give each unit to one CTA).
PLANNED = [
    W("planned_group5_batch2", 2, 20, 4, 1800, 1800, 128, "bf16", True),
    W("planned_offset_d64", 1, 32, 8, 2560, 3000, 64, "f16", True, 400),
    # the other two (tile mode, D) pairs of the plan entries
    W("planned_group5_d64", 4, 20, 4, 1024, 1024, 64, "bf16", True),
    W("planned_paired_d128", 4, 16, 4, 1280, 1280, 128, "f16", True),
]


def planned(w):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return attn.attn_unit_plan(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.causal,
                               w.input_pos, grid=sms)["planned"] == 1


@pytest.mark.parametrize("w", PLANNED, ids=lambda w: w.name)
def test_planned_launches(w):
    assert planned(w)
    check_full(w, seed=9)


@pytest.mark.parametrize("w", [MHA_4K, GQA_8K, PREFILL_CHUNK],
                         ids=lambda w: w.name)
def test_planned_full_size_writes_every_row(w):
    assert planned(w)
    q, k, v = (t.cuda() for t in make_qkv(w, seed=10))
    o = torch.full(q.shape, float("nan"), dtype=w.out_dtype, device="cuda")
    lse = torch.full((w.B, w.Hq, w.Sq), float("nan"), dtype=torch.float32,
                     device="cuda")
    attn.fwd(q, k, v, scale=w.scale, causal=w.causal, input_pos=w.input_pos,
             out=o, lse=lse)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == (0, 0)
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())


def test_bitwise_reproducible():
    w = W("repro", 1, 8, 2, 1000, 1000, 128, "bf16", True, 0)
    q, k, v = make_qkv(w, 6)
    o1, l1 = run_gpu(w, q, k, v)
    o2, l2 = run_gpu(w, q, k, v)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_guard_bands_untouched():
    """Writes stay inside O and LSE: sentinels around both survive."""
    w = W("guard", 1, 2, 1, 300, 300, 128, "f16", True)
    q, k, v = make_qkv(w, 7)
    guard = 4096
    n_o = w.B * w.Hq * w.Sq * w.D
    n_l = w.B * w.Hq * w.Sq
    o_buf = torch.full((n_o + 2 * guard,), 7.0, dtype=torch.float16,
                       device="cuda")
    l_buf = torch.full((n_l + 2 * guard,), -3.0, dtype=torch.float32,
                       device="cuda")
    o = o_buf[guard:guard + n_o].view(w.B, w.Hq, w.Sq, w.D)
    lse = l_buf[guard:guard + n_l].view(w.B, w.Hq, w.Sq)
    attn.fwd(q.cuda(), k.cuda(), v.cuda(), scale=w.scale, causal=True,
             out=o, lse=lse)
    torch.cuda.synchronize()
    assert bool((o_buf[:guard] == 7.0).all())
    assert bool((o_buf[guard + n_o:] == 7.0).all())
    assert bool((l_buf[:guard] == -3.0).all())
    assert bool((l_buf[guard + n_l:] == -3.0).all())
    check_full(w, q=q, k=k, v=v)


def test_lse_optional():
    w = W("nolse", 1, 4, 4, 256, 256, 64, "f16", True)
    q, k, v = make_qkv(w, 8)
    o1, _ = attn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    o2, none = attn.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True,
                        need_lse=False)
    torch.cuda.synchronize()
    assert none is None
    assert torch.equal(o1, o2)


def test_side_stream():
    w = W("stream", 1, 4, 2, 512, 512, 128, "bf16", True)
    q, k, v = (t.cuda() for t in make_qkv(w, 9))
    ref, _ = attn.fwd(q, k, v, causal=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, _ = attn.fwd(q, k, v, causal=True)
    s.synchronize()
    assert torch.equal(o, ref)


def test_raw_c_abi_call():
    """The C entry point with plain pointers and sizes."""
    w = SMALL
    q, k, v = (t.cuda() for t in make_qkv(w, 10))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device="cuda")
    st = attn.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                       lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D,
                       w.scale, 0, 0, attn.ATTN_F16,
                       torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK
    ref, ref_lse = attn.fwd(q, k, v, scale=w.scale, causal=False)
    torch.cuda.synchronize()
    assert torch.equal(o, ref) and torch.equal(lse, ref_lse)


def test_host_pointers_rejected():
    """Host memory is refused before any launch."""
    w = SMALL
    q, k, v = make_qkv(w, 11)
    o = torch.empty_like(q)
    st = attn.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                       0, w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.scale, 0, 0,
                       attn.ATTN_F16, 0)
    assert st == attn.ATTN_ERR_INVALID_ARG


def test_device_status_clean():
    assert attn.attn_device_status() == (0, 0)
