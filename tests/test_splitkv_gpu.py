"""GPU parity of the split-KV forward (key range cut into pieces, merged by
log-sum-exp) against the fp64 CPU oracle and against the one-pass kernel."""
import numpy as np
import pytest
import torch

import attention_attn_fwd_gb300 as attn
import oracle
from attention_attn_fwd_gb300.inputs import PREFILL_CHUNK, Workload, make_qkv
from tests.gpu_parity import TOL_LSE, TOL_O, sample_rows
from tests.test_abi import PLAN_PICKS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def W(name, B, Hq, Hkv, Sq, Skv, D, dt, causal, pos=0):
    return Workload(name, B, Hq, Hkv, Sq, Skv, D, dt, causal, pos)


def run_split(w, q, k, v, splits):
    o, lse = attn.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), scale=w.scale,
                              causal=w.causal, input_pos=w.input_pos,
                              num_splits=splits)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == (0, 0)
    return o, lse


CASES = [
    W("decode_gqa4", 2, 8, 2, 1, 1000, 128, "bf16", True, 999),
    W("decode_noncausal", 2, 8, 2, 1, 1000, 128, "f16", False),
    W("decode_d64_mqa", 1, 16, 1, 3, 777, 64, "f16", True, 774),
    W("chunk_ragged", 1, 4, 2, 200, 700, 128, "bf16", True, 300),
    W("chunk_rows_mode", 1, 3, 1, 130, 513, 64, "bf16", True, 383),
    W("short_keys", 1, 2, 2, 5, 129, 128, "f16", True, 124),
    # the remaining D = 64 variants: packed bf16, one head per tile f16
    W("decode_d64_bf16", 2, 8, 2, 1, 900, 64, "bf16", True, 899),
    W("chunk_d64_f16", 1, 4, 2, 200, 700, 64, "f16", True, 300),
]


@pytest.mark.parametrize("splits", [0, 1, 3, 8])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_against_oracle(w, splits):
    q, k, v = make_qkv(w, seed=21)
    o, lse = run_split(w, q, k, v, splits)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.causal, w.input_pos)
    err_o = float(np.max(np.abs(o.double().cpu().numpy() - o_ref)))
    err_l = float(np.max(np.abs(lse.double().cpu().numpy() - lse_ref)))
    assert err_o <= TOL_O[w.dtype], (w.name, splits, err_o)
    assert err_l <= TOL_LSE, (w.name, splits, err_l)


def test_matches_one_pass_kernel():
    w = W("cmp", 1, 8, 4, 64, 2048, 128, "bf16", True, 1984)
    q, k, v = (t.cuda() for t in make_qkv(w, seed=22))
    o1, l1 = attn.fwd(q, k, v, causal=True, input_pos=w.input_pos)
    o2, l2 = attn.fwd_splitkv(q, k, v, causal=True, input_pos=w.input_pos,
                              num_splits=6)
    torch.cuda.synchronize()
    assert float((o1.float() - o2.float()).abs().max()) <= TOL_O["bf16"]
    assert float((l1 - l2).abs().max()) <= TOL_LSE


def test_plan_clamps_and_reports_workspace():
    ns, ws = attn.attn_splitkv_plan(1, 4, 2, 1, 300, 128, 1, 299,
                                    attn.ATTN_BF16, 64)
    assert ns == 3          # 300 keys = 3 tiles of 128
    rows = 1 * 4 * 1
    assert ws >= ns * rows * 128 * 4 + ns * rows * 4
    ns_auto, _ = attn.attn_splitkv_plan(8, 32, 8, 1, 4096, 128, 1, 4095,
                                        attn.ATTN_BF16, 0)
    assert 1 <= ns_auto <= 32


def test_rejects_unplanned_split_count_and_small_workspace():
    w = W("rej", 1, 4, 2, 1, 300, 128, "bf16", True, 299)
    q, k, v = (t.cuda() for t in make_qkv(w, seed=23))
    o = torch.empty_like(q)
    ns, ws = attn.attn_splitkv_plan(1, 4, 2, 1, 300, 128, 1, 299,
                                    attn.ATTN_BF16, 3)
    buf = torch.empty(ws, dtype=torch.uint8, device="cuda")
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), 0,
            1, 4, 2, 1, 300, 128, w.scale, 1, 299, attn.ATTN_BF16]
    assert attn.attn_fwd_splitkv(*args, 5, buf.data_ptr(), ws, 0) == \
        attn.ATTN_ERR_INVALID_ARG          # 5 is not a planned count (3)
    assert attn.attn_fwd_splitkv(*args, ns, buf.data_ptr(), ws - 4, 0) == \
        attn.ATTN_ERR_INVALID_ARG          # workspace too small
    assert attn.attn_fwd_splitkv(*args, ns, buf.data_ptr() + 16, ws - 16, 0) \
        == attn.ATTN_ERR_ALIGNMENT
    assert attn.attn_fwd_splitkv(*args, ns, buf.data_ptr(), ws, 0) == \
        attn.ATTN_OK
    torch.cuda.synchronize()


def test_prefill_chunk_workload_full_size():
    """The KV-cache prefill-chunk workload, split 4 ways, sampled rows."""
    w = PREFILL_CHUNK
    q, k, v = make_qkv(w, seed=0)
    o, lse = run_split(w, q, k, v, 4)
    rows = sample_rows(w, 128, seed=3)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, w.scale, w.causal,
                                           w.input_pos, rows)
    idx = torch.from_numpy(rows).cuda()
    o_rows = o[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    l_rows = lse[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    assert float(np.max(np.abs(o_rows - o_ref))) <= TOL_O[w.dtype]
    assert float(np.max(np.abs(l_rows - lse_ref))) <= TOL_LSE


def test_decode_workload_full():
    """One new token per sequence against a 4096-key cache (decode)."""
    w = PREFILL_CHUNK.with_(name="decode", Sq=1, input_pos=4095)
    q, k, v = make_qkv(w, seed=5)
    o, lse = run_split(w, q, k, v, 0)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, w.causal, w.input_pos)
    assert float(np.max(np.abs(o.double().cpu().numpy() - o_ref))) <= \
        TOL_O[w.dtype]
    assert float(np.max(np.abs(lse.double().cpu().numpy() - lse_ref))) <= \
        TOL_LSE


@pytest.mark.parametrize("fill", [0x00, 0xA5, 0xFF])
def test_workspace_contents_and_reuse(fill):
    """The workspace needs no clearing: it starts as arbitrary bytes and is
    reused by calls of different shapes and split counts in a row."""
    a = W("reuse_a", 2, 8, 2, 1, 1500, 128, "bf16", True, 1499)
    b = W("reuse_b", 1, 4, 2, 40, 900, 64, "f16", True, 860)
    c = W("reuse_c", 1, 3, 1, 130, 513, 64, "bf16", True, 383)  # not packed
    plans = [(a, 4), (b, 3), (c, 2), (a, 6), (a, 4), (c, 2)]
    need = max(attn.attn_splitkv_plan(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, 1,
                                      w.input_pos,
                                      attn.ATTN_BF16 if w.dtype == "bf16"
                                      else attn.ATTN_F16, s)[1]
               for w, s in plans)
    buf = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
    for w, s in plans:
        q, k, v = make_qkv(w, seed=24)
        o, lse = attn.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), scale=w.scale,
                                  causal=True, input_pos=w.input_pos,
                                  num_splits=s, workspace=buf)
        torch.cuda.synchronize()
        assert attn.attn_device_status() == (0, 0)
        o_ref, lse_ref = oracle.attention(q, k, v, w.scale, True, w.input_pos)
        assert float(np.max(np.abs(o.double().cpu().numpy() - o_ref))) <= \
            TOL_O[w.dtype], (w.name, s)
        assert float(np.max(np.abs(lse.double().cpu().numpy() - lse_ref))) <= \
            TOL_LSE, (w.name, s)


@pytest.mark.parametrize("w, splits", [
    # 40 x 8 (batch, K/V head) groups x 2 ranges: more units than SMs, so
    # the key ranges merge through the workspace in the merge launch.
    (W("many_groups", 40, 32, 8, 1, 700, 128, "bf16", True, 699), 2),
    # 2 groups x 8 ranges: every unit runs at once, each group's 8 ranges
    # form one thread-block cluster and merge over its shared memory.
    (W("cluster_of_8", 1, 8, 2, 1, 4000, 128, "f16", True, 3999), 8),
    (W("cluster_window", 2, 8, 2, 3, 3000, 64, "bf16", True, 2997), 4),
], ids=["merge_launch", "cluster_merge_8", "cluster_merge_window"])
def test_merge_paths_against_oracle(w, splits):
    """Both ways of merging the key ranges of packed split-KV tiles."""
    q, k, v = make_qkv(w, seed=31)
    window = 1500 if "window" in w.name else 0
    o, lse = attn.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), scale=w.scale,
                              causal=True, input_pos=w.input_pos,
                              num_splits=splits, window=window)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == (0, 0)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, True, w.input_pos,
                                      window)
    assert float(np.max(np.abs(o.double().cpu().numpy() - o_ref))) <= \
        TOL_O[w.dtype]
    assert float(np.max(np.abs(lse.double().cpu().numpy() - lse_ref))) <= \
        TOL_LSE


@pytest.mark.parametrize("w, splits, window", [
    # 2 x 8 heads x 2 row blocks of 256 x 16 ranges = 512 units: four waves
    # of units on 152 SMs, each row merged from 16 ranges.
    (W("merge_waves", 2, 8, 8, 300, 4096, 128, "bf16", True, 3796), 16, 0),
    # paired heads, D = 64, f16, a window: rows skip the ranges before it.
    (W("merge_window_d64", 1, 4, 2, 200, 3000, 64, "f16", True, 2800), 6,
     1000),
    # one head, 32 ranges of one tile each, rows of a ragged last block.
    (W("merge_32_ranges", 1, 1, 1, 70, 4000, 128, "f16", True, 3930), 32, 0),
], ids=lambda x: x.name if isinstance(x, Workload) else str(x))
def test_merge_launch_against_oracle(w, splits, window):
    """The merge launch (split-KV launches not merged in a cluster): many
    waves, many ranges, windows; sampled rows against the oracle."""
    q, k, v = make_qkv(w, seed=33)
    o, lse = attn.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), scale=w.scale,
                              causal=True, input_pos=w.input_pos,
                              num_splits=splits, window=window)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == (0, 0)
    rows = sample_rows(w, min(96, w.B * w.Hq * w.Sq), seed=4)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, w.scale, True,
                                           w.input_pos, rows, window)
    idx = torch.from_numpy(rows).cuda()
    o_rows = o[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    l_rows = lse[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    assert float(np.max(np.abs(o_rows - o_ref))) <= TOL_O[w.dtype]
    assert float(np.max(np.abs(l_rows - lse_ref))) <= TOL_LSE


@pytest.mark.parametrize("shape, expect", PLAN_PICKS)
def test_plan_picks_on_gb300(shape, expect):
    """The automatic split count on a 152-SM GB300 for shapes whose timings
    over 1-32 ranges fitted the planner's costs (best or within 5 % of the
    best measured count)."""
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("planner picks are stated for 152 SMs")
    ns, _ = attn.attn_splitkv_plan(*shape, attn.ATTN_BF16, 0)
    assert ns == expect
