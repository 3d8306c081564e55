"""The allocation-free split-KV entry point.

Some callers cannot allocate device memory (the allocator is off limits
where they run, or their host owns every allocation), so
``attn_fwd_splitkv_noalloc`` keeps its partial results in a fixed scratch
array inside the library.  This checks, through the C ABI, that two calls
in a row give the same results as the workspace-taking entry point.  The
file name makes pytest collect it last.
"""
import pytest
import torch

import attention_attn_fwd_gb300 as attn
from attention_attn_fwd_gb300.inputs import Workload, make_qkv
from tests.gpu_parity import TOL_LSE, TOL_O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def call_noalloc(w, q, k, v, o, lse, splits):
    dt = attn.ATTN_BF16 if w.dtype == "bf16" else attn.ATTN_F16
    return attn.attn_fwd_splitkv_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
        lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.scale,
        int(w.causal), w.input_pos, dt, splits,
        torch.cuda.current_stream().cuda_stream)


def test_two_calls_match_workspace_entry_point():
    cases = [
        (Workload("noalloc_decode", 4, 32, 8, 1, 3000, 128, "bf16", True,
                  2999), 0),
        (Workload("noalloc_chunk", 1, 8, 2, 96, 1500, 64, "f16", True, 1404),
         5),
    ]
    assert attn.attn_noalloc_scratch_bytes() >= 1 << 20
    for seed, (w, splits) in enumerate(cases):   # two calls in a row
        q, k, v = (t.cuda() for t in make_qkv(w, seed=40 + seed))
        o = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.Hq, w.Sq), float("nan"),
                         dtype=torch.float32, device="cuda")
        assert call_noalloc(w, q, k, v, o, lse, splits) == attn.ATTN_OK
        ref, ref_lse = attn.fwd_splitkv(q, k, v, scale=w.scale,
                                        causal=w.causal,
                                        input_pos=w.input_pos,
                                        num_splits=splits)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == (0, 0)
        assert float((o.float() - ref.float()).abs().max()) <= TOL_O[w.dtype]
        assert float((lse - ref_lse).abs().max()) <= TOL_LSE


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
