"""GPU parity of the causal sliding window (query at position p sees keys
p - window + 1 .. p) against the fp64 oracle: one-pass and split-KV paths,
every tile mode, window edges on and off tile boundaries."""
import numpy as np
import pytest
import torch

import attention_attn_fwd_gb300 as attn
import oracle
from attention_attn_fwd_gb300.inputs import WINDOW_32K, Workload, make_qkv
from tests.gpu_parity import TOL_LSE, TOL_O, check_full, check_sampled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def W(name, B, Hq, Hkv, Sq, Skv, D, dt, pos, window):
    return Workload(name, B, Hq, Hkv, Sq, Skv, D, dt, True, pos, window)


CASES = [
    # packed GQA tiles (few query rows)
    W("decode_w1", 2, 8, 2, 1, 1000, 128, "bf16", 999, 1),
    W("decode_w256", 2, 8, 2, 1, 1000, 128, "f16", 999, 256),
    W("packed_rows_w50", 1, 16, 4, 20, 500, 128, "f16", 480, 50),
    W("packed_d64_w129", 3, 4, 2, 7, 700, 64, "bf16", 690, 129),
    W("packed_d64_f16_w90", 2, 8, 2, 5, 600, 64, "f16", 595, 90),
    # two heads per CTA (even group), same rows
    W("pair_w129", 1, 8, 2, 700, 700, 128, "bf16", 0, 129),
    W("pair_offset_w384", 1, 4, 2, 300, 1100, 128, "bf16", 800, 384),
    W("pair_d64_w200", 1, 8, 2, 600, 900, 64, "bf16", 300, 200),
    # 256 rows of one head per CTA
    W("rows_w200", 1, 4, 4, 600, 600, 64, "f16", 0, 200),
    W("rows_odd_group_w333", 1, 3, 1, 260, 900, 64, "f16", 500, 333),
    W("rows_w128_aligned", 1, 2, 2, 512, 512, 64, "bf16", 0, 128),
    W("rows_w1", 1, 2, 2, 300, 300, 128, "f16", 0, 1),
    # key tail and a window wider than every prefix
    W("key_tail_w64", 1, 2, 2, 100, 333, 128, "bf16", 233, 64),
    W("window_covers_all", 1, 2, 2, 256, 256, 64, "f16", 0, 100000),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_window_against_oracle(w):
    check_full(w, seed=31)


def test_window_zero_and_wide_match_plain_causal():
    w = W("cmp", 1, 4, 2, 384, 384, 128, "bf16", 0, 0)
    q, k, v = (t.cuda() for t in make_qkv(w, seed=32))
    o0, l0 = attn.fwd(q, k, v, causal=True)
    o1, l1 = attn.fwd(q, k, v, causal=True, window=0)
    o2, l2 = attn.fwd(q, k, v, causal=True, window=384)
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    assert torch.equal(o0, o2) and torch.equal(l0, l2)


SPLIT_CASES = [
    W("split_decode_w300", 2, 8, 2, 1, 2000, 128, "bf16", 1999, 300),
    W("split_decode_w1", 1, 4, 2, 1, 777, 64, "f16", 776, 1),
    W("split_chunk_w500", 1, 4, 2, 200, 1500, 128, "bf16", 1300, 500),
    W("split_rows_w257", 1, 3, 1, 130, 900, 64, "f16", 770, 257),
    # every remaining (D, dtype, packed) combination with split and window
    W("split_decode_d64_bf16_w200", 2, 8, 2, 1, 1500, 64, "bf16", 1499, 200),
    W("split_rows_d64_bf16_w300", 1, 3, 1, 130, 900, 64, "bf16", 770, 300),
    W("split_chunk_f16_w400", 1, 4, 2, 200, 1500, 128, "f16", 1300, 400),
    W("split_decode_f16_w300", 2, 8, 2, 1, 2000, 128, "f16", 1999, 300),
]


@pytest.mark.parametrize("splits", [0, 3, 8])
@pytest.mark.parametrize("w", SPLIT_CASES, ids=lambda w: w.name)
def test_window_splitkv_against_oracle(w, splits):
    q, k, v = make_qkv(w, seed=33)
    o, lse = attn.fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), scale=w.scale,
                              causal=True, input_pos=w.input_pos,
                              num_splits=splits, window=w.window)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == (0, 0)
    o_ref, lse_ref = oracle.attention(q, k, v, w.scale, True, w.input_pos,
                                      w.window)
    err_o = float(np.max(np.abs(o.double().cpu().numpy() - o_ref)))
    err_l = float(np.max(np.abs(lse.double().cpu().numpy() - lse_ref)))
    assert err_o <= TOL_O[w.dtype], (w.name, splits, err_o)
    assert err_l <= TOL_LSE, (w.name, splits, err_l)


def test_window_full_size_workload():
    """GQA 32k causal with a 4096-key window, sampled rows."""
    check_sampled(WINDOW_32K, seed=0, n_rows=96)


def test_window_argument_checks():
    w = W("args", 1, 2, 2, 4, 64, 64, "f16", 0, 8)
    q, k, v = (t.cuda() for t in make_qkv(w, seed=34))
    o = torch.empty_like(q)
    a = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), 0, 1, 2, 2,
         4, 64, 64, w.scale]
    # causal, input_pos, window
    assert attn.attn_fwd_window(*a, 0, 0, 8, attn.ATTN_F16, 0) == \
        attn.ATTN_ERR_INVALID_ARG          # window needs causal
    assert attn.attn_fwd_window(*a, 1, 0, -1, attn.ATTN_F16, 0) == \
        attn.ATTN_ERR_INVALID_ARG          # negative window
    assert attn.attn_fwd_window(*a, 1, 62, 1, attn.ATTN_F16, 0) == \
        attn.ATTN_ERR_INVALID_ARG          # last row (position 65) sees no key
    assert attn.attn_fwd_window(*a, 1, 60, 1, attn.ATTN_F16, 0) == \
        attn.ATTN_OK                       # positions 60..63: own key each
    torch.cuda.synchronize()
    assert attn.attn_device_status() == (0, 0)
