"""The bounded-wait abort path of the forward kernel, through the C ABI.

Every mbarrier wait in the kernel gives up after a time limit: the waiting
role raises the CTA's abort flag and ORs a code into the device status word,
every role of that CTA stops issuing work, drains what it has in flight
(again bounded) and the CTA frees its TMEM and exits.  Nothing traps and the
context stays usable.  ``attn_selftest_wait_timeout`` makes one wait run out
on purpose -- the first CTA never loads its first K tile, so its MMA issuer
waits for a tile that cannot arrive -- with a 10 ms limit.  These tests check
that the launch returns, the status word reports the timeout and the roles
that gave up, the other CTAs' rows are correct, and the next normal call
matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

import attention_attn_fwd_gb300 as attn
import oracle
from attention_attn_fwd_gb300.inputs import Workload, make_qkv
from tests.gpu_parity import TOL_LSE, TOL_O, check_full

pytestmark = pytest.mark.gpu

LIMIT_NS = 10_000_000  # 10 ms


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


# Two query heads per K/V head at the same rows form a unit of two 128-row
# tiles: 2 head pairs x 4 row blocks = 8 units on 8 CTAs.  Units are issued
# heaviest causal row block first, so the first CTA owns rows 384-511 of
# query heads 0 and 1.
W = Workload("timeout_case", 1, 4, 2, 512, 512, 128, "bf16", True)


def selftest(w, q, k, v, o, lse, stream):
    return attn.attn_selftest_wait_timeout(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
        lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.scale,
        int(w.causal), w.input_pos, attn.ATTN_BF16, LIMIT_NS, stream)


def check_timeout_code(st, code):
    assert st == attn.ATTN_ERR_TIMEOUT, (st, code)
    assert code & 0xFF == 1, hex(code)
    # Producer (1), MMA issuer (2), softmax (3) and output store (4) all
    # wait on the missing tile's consequences; whichever run out first OR
    # their numbers in.
    assert 1 <= (code >> 8) & 0xFF <= 7, hex(code)


def test_wait_runs_out_and_context_stays_usable():
    assert attn.attn_device_status() == (0, 0)
    q, k, v = make_qkv(W, seed=61)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((W.B, W.Hq, W.Sq), float("nan"), dtype=torch.float32,
                     device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.perf_counter()
    assert selftest(W, qd, kd, vd, o, lse, stream) == attn.ATTN_OK
    check_timeout_code(*attn.attn_device_status())
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0, elapsed  # the limit is 10 ms, not the default 2 s
    # Read and cleared: the next query is clean.
    assert attn.attn_device_status() == (0, 0)

    # Every row outside the first CTA's unit was computed normally.
    o_ref, lse_ref = oracle.attention(q, k, v, W.scale, W.causal,
                                      W.input_pos)
    o_gpu = o.double().cpu().numpy()
    lse_gpu = lse.double().cpu().numpy()
    keep = np.ones((W.B, W.Hq, W.Sq), dtype=bool)
    keep[:, 0:2, 384:512] = False
    err_o = float(np.max(np.abs(o_gpu - o_ref)[keep]))
    err_l = float(np.max(np.abs(lse_gpu - lse_ref)[keep]))
    assert err_o <= TOL_O[W.dtype], err_o
    assert err_l <= TOL_LSE, err_l

    # A normal call right after matches the oracle everywhere.
    check_full(W, seed=61)
    assert attn.attn_device_status() == (0, 0)


def test_stream_status_on_a_side_stream():
    q, k, v = (t.cuda() for t in make_qkv(W, seed=62))
    o = torch.empty_like(q)
    lse = torch.empty((W.B, W.Hq, W.Sq), dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    assert attn.attn_stream_status(side.cuda_stream) == (0, 0)
    with torch.cuda.stream(side):
        assert selftest(W, q, k, v, o, lse, side.cuda_stream) == attn.ATTN_OK
    check_timeout_code(*attn.attn_stream_status(side.cuda_stream))
    # The clearing was enqueued on the side stream; after it, all is clean.
    side.synchronize()
    assert attn.attn_stream_status(side.cuda_stream) == (0, 0)
    assert attn.attn_device_status() == (0, 0)
    check_full(W, seed=62)


def test_rejects_zero_limit():
    q = torch.zeros((W.B, W.Hq, W.Sq, W.D), dtype=torch.bfloat16,
                    device="cuda")
    k = torch.zeros((W.B, W.Hkv, W.Skv, W.D), dtype=torch.bfloat16,
                    device="cuda")
    o = torch.empty_like(q)
    st = attn.attn_selftest_wait_timeout(
        q.data_ptr(), k.data_ptr(), k.data_ptr(), o.data_ptr(), 0, W.B, W.Hq,
        W.Hkv, W.Sq, W.Skv, W.D, W.scale, 1, 0, attn.ATTN_BF16, 0, 0)
    assert st == attn.ATTN_ERR_INVALID_ARG
