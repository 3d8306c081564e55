"""The allocation-free split-KV entry point.

Some callers cannot allocate device memory: code that runs where the
allocator must not be entered (a real-time loop, a callback inside another
runtime) or a plugin whose host owns every allocation.  For them
``attn_fwd_splitkv_noalloc`` keeps its partial results in a fixed scratch
array inside the library.  These tests call it through the C ABI and check,
on consecutive calls, that it gives bit for bit the result of the
workspace-taking ``attn_fwd_splitkv`` at the same split count (the same
kernel on the same inputs) and matches the fp64 oracle element by element.

The name sorts this file after every other test file, so pytest collects it
last: the scratch array is shared by every call in the process, and a run
that stops at the first failure has then already run every other test
before this one touches it.  The tests also pass when run alone.
"""
import numpy as np
import pytest
import torch

import attention_attn_fwd_gb300 as attn
import oracle
from attention_attn_fwd_gb300.inputs import Workload, make_qkv
from tests.gpu_parity import TOL_LSE, TOL_O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _dtype(w):
    return attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_F16


def call_noalloc(w, q, k, v, o, lse, splits):
    return attn.attn_fwd_splitkv_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
        lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.scale,
        int(w.causal), w.input_pos, _dtype(w), splits,
        torch.cuda.current_stream().cuda_stream)


def planned(w, splits):
    ns, _ = attn.attn_splitkv_plan(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D,
                                   int(w.causal), w.input_pos, _dtype(w),
                                   splits)
    return ns


DECODE = Workload("noalloc_decode", 4, 32, 8, 1, 3000, 128, "bf16", True,
                  2999)
CHUNK = Workload("noalloc_chunk", 1, 8, 2, 96, 1500, 64, "f16", True, 1404)


def test_consecutive_calls_match_workspace_call_and_oracle():
    assert attn.attn_noalloc_scratch_bytes() >= 1 << 20
    # The same shape twice with new inputs (the second call finds the
    # first call's partials in the scratch), then another shape and split
    # count.
    calls = [(DECODE, 0, 40), (DECODE, 0, 41), (CHUNK, planned(CHUNK, 5), 42)]
    for w, splits, seed in calls:
        ns = planned(w, splits)
        q, k, v = make_qkv(w, seed=seed)
        qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
        o = torch.full_like(qd, float("nan"))
        lse = torch.full((w.B, w.Hq, w.Sq), float("nan"),
                         dtype=torch.float32, device="cuda")
        assert call_noalloc(w, qd, kd, vd, o, lse, splits) == attn.ATTN_OK
        ref, ref_lse = attn.fwd_splitkv(qd, kd, vd, scale=w.scale,
                                        causal=w.causal,
                                        input_pos=w.input_pos,
                                        num_splits=ns)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == (0, 0)
        assert torch.equal(o, ref), (w.name, seed)
        assert torch.equal(lse, ref_lse), (w.name, seed)
        o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.causal,
                                          w.input_pos)
        err_o = float(np.max(np.abs(o.double().cpu().numpy() - o_ref)))
        err_l = float(np.max(np.abs(lse.double().cpu().numpy() - lse_ref)))
        assert err_o <= TOL_O[w.dtype], (w.name, seed, err_o)
        assert err_l <= TOL_LSE, (w.name, seed, err_l)


def test_rejects_unplanned_split_count():
    # 12 key tiles: a request of 5 ranges plans as 4 (3 tiles each); the
    # workspace-taking call rejects 5 and so does this one.
    w = CHUNK
    assert planned(w, 5) != 5
    q = torch.zeros((w.B, w.Hq, w.Sq, w.D), dtype=torch.float16,
                    device="cuda")
    k = torch.zeros((w.B, w.Hkv, w.Skv, w.D), dtype=torch.float16,
                    device="cuda")
    o = torch.empty_like(q)
    assert call_noalloc(w, q, k, k, o, torch.empty(
        (w.B, w.Hq, w.Sq), dtype=torch.float32, device="cuda"), 5) == \
        attn.ATTN_ERR_INVALID_ARG


def test_rejects_results_larger_than_scratch():
    # 64 query rows x 128 heads x D=128 in 8 splits: 32 MiB of partials.
    w = Workload("too_big", 1, 128, 128, 64, 1024, 128, "bf16", False)
    dt = attn.ATTN_BF16
    ns, need = attn.attn_splitkv_plan(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, 0,
                                      0, dt, 8)
    assert ns == 8
    assert need > attn.attn_noalloc_scratch_bytes()
    q = torch.zeros((w.B, w.Hq, w.Sq, w.D), dtype=torch.bfloat16,
                    device="cuda")
    k = torch.zeros((w.B, w.Hkv, w.Skv, w.D), dtype=torch.bfloat16,
                    device="cuda")
    o = torch.empty_like(q)
    st = attn.attn_fwd_splitkv_noalloc(
        q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(), 0, w.B, w.Hq,
        w.Hkv, w.Sq, w.Skv, w.D, w.scale, 0, 0, dt, ns, 0)
    assert st == attn.ATTN_ERR_UNSUPPORTED
