"""GPU parity of the backward pass (dQ, dK, dV through the C ABI) against
the fp64 oracle's chain rule, and exact invariants of the gradients at the
full GQA 8k size."""
import numpy as np
import pytest
import torch

import attention_attn_fwd_gb300 as attn
import oracle
from attention_attn_fwd_gb300.inputs import (GQA_8K, Workload, make_do,
                                             make_qkv)
from tests.gpu_parity import sample_rows

pytestmark = pytest.mark.gpu

# max |gradient - oracle| / max |oracle| per gradient tensor.  The 16-bit
# P^T / dS operands and outputs carry 2^-9 (bf16) or 2^-12 (fp16) relative
# error each; signed sums grow like sqrt(N) as their values do, so the
# normalised error stays near a few units of that: 2e-2 and 5e-3 leave a
# factor of about four.
TOL_REL = {"f16": 5e-3, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def W(name, B, Hq, Hkv, Sq, Skv, D, dt, causal, pos=0, window=0):
    return Workload(name, B, Hq, Hkv, Sq, Skv, D, dt, causal, pos, window)


def run_bwd(w, q, k, v, do, scale):
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = attn.fwd(qd, kd, vd, scale=scale, causal=w.causal,
                      input_pos=w.input_pos, window=w.window)
    dq, dk, dv = attn.bwd(qd, kd, vd, o, lse, dod, scale=scale,
                          causal=w.causal, input_pos=w.input_pos,
                          window=w.window)
    torch.cuda.synchronize()
    st, code = attn.attn_device_status()
    assert st == 0, "device status %d code %#x" % (st, code)
    return dq, dk, dv


def rel_err(got, ref):
    g = got.double().cpu().numpy()
    assert np.all(np.isfinite(g))
    denom = float(np.max(np.abs(ref)))
    return float(np.max(np.abs(g - ref))) / max(denom, 1e-30)


def row_err(got, ref):
    """Per sampled row: max |got - ref| over the row, divided by the row's
    largest oracle value, or by 1 % of the largest over all sampled rows
    when the row's own is smaller (a row whose exact gradient is near zero,
    such as dQ of the first causal query, which sees one key, carries the
    rounding of terms as large as its neighbours')."""
    row_max = np.max(np.abs(ref), axis=1)
    floor = 0.01 * float(row_max.max())
    return np.max(np.abs(got - ref), axis=1) / np.maximum(row_max, floor)


CASES = [
    W("small_noncausal", 1, 2, 2, 128, 128, 64, "f16", False),
    W("causal_gqa_ragged", 1, 8, 2, 300, 300, 128, "bf16", True),
    W("offset_chunk", 1, 4, 2, 200, 500, 128, "bf16", True, 300),
    W("noncausal_rect", 2, 2, 1, 129, 383, 64, "f16", False),
    W("decode_rows", 1, 8, 2, 5, 700, 128, "f16", True, 695),
    W("mha_d64", 2, 4, 4, 256, 256, 64, "bf16", True),
    W("unseen_keys", 1, 2, 2, 100, 600, 64, "f16", True, 0),
    W("window", 1, 4, 2, 400, 400, 128, "bf16", True, 0, 130),
    W("window_offset", 1, 2, 1, 150, 900, 64, "f16", True, 700, 257),
    W("odd_group", 1, 3, 1, 200, 260, 128, "f16", True, 60),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_bwd_against_oracle(w):
    q, k, v = make_qkv(w, seed=41)
    do = make_do(w, seed=41)
    dq, dk, dv = run_bwd(w, q, k, v, do, w.scale)
    ref = oracle.backward(q, k, v, do, w.scale, w.causal, w.input_pos,
                          w.window)
    for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        e = rel_err(got, r)
        assert e <= TOL_REL[w.dtype], (w.name, name, e)


def test_bwd_unseen_keys_are_zero():
    """Keys past every query's causal horizon get exactly zero dK, dV."""
    w = W("unseen", 1, 2, 2, 100, 600, 64, "bf16", True, 0)
    q, k, v = make_qkv(w, seed=42)
    _, dk, dv = run_bwd(w, q, k, v, make_do(w, seed=42), w.scale)
    assert bool((dk[:, :, 100:] == 0).all()) and bool((dv[:, :, 100:] == 0).all())


@pytest.mark.parametrize("scale", [-0.125, 0.0])
def test_bwd_scale_values(scale):
    w = W("scale", 1, 4, 2, 200, 300, 128, "f16", True, 100)
    q, k, v = make_qkv(w, seed=43)
    do = make_do(w, seed=43)
    dq, dk, dv = run_bwd(w, q, k, v, do, scale)
    ref = oracle.backward(q, k, v, do, scale, True, 100)
    for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        if not np.any(r):
            assert bool((got == 0).all()), name
            continue
        assert rel_err(got, r) <= TOL_REL["f16"], (name, scale)


def test_bwd_deterministic():
    w = W("repro", 1, 8, 2, 384, 384, 128, "bf16", True)
    q, k, v = make_qkv(w, seed=44)
    do = make_do(w, seed=44)
    a = run_bwd(w, q, k, v, do, w.scale)
    b = run_bwd(w, q, k, v, do, w.scale)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_bwd_side_stream_and_graph():
    """The dQ kernel runs on an internal stream forked from the caller's:
    a call on a user stream, and a replay of the call captured into a CUDA
    graph, give the bit-identical gradients of a default-stream call."""
    w = W("streams", 1, 8, 2, 384, 640, 128, "bf16", True, 256)
    q, k, v = (t.cuda() for t in make_qkv(w, seed=45))
    do = make_do(w, seed=45).cuda()
    o, lse = attn.fwd(q, k, v, scale=w.scale, causal=True,
                      input_pos=w.input_pos)
    ref = attn.bwd(q, k, v, o, lse, do, scale=w.scale, causal=True,
                   input_pos=w.input_pos)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    outs = tuple(torch.full_like(t, 7.0) for t in ref)
    ws = torch.empty(attn.attn_bwd_workspace_bytes(w.B, w.Hq, w.Sq),
                     dtype=torch.uint8, device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        got = attn.bwd(q, k, v, o, lse, do, scale=w.scale, causal=True,
                       input_pos=w.input_pos, dq=outs[0], dk=outs[1],
                       dv=outs[2], workspace=ws)
    s.synchronize()
    for x, y in zip(ref, got):
        assert torch.equal(x, y)
    for t in outs:
        t.fill_(7.0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        attn.bwd(q, k, v, o, lse, do, scale=w.scale, causal=True,
                 input_pos=w.input_pos, dq=outs[0], dk=outs[1], dv=outs[2],
                 workspace=ws)
    for t in outs:
        t.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_device_status() == (0, 0)
    for x, y in zip(ref, outs):
        assert torch.equal(x, y)


def test_bwd_full_size_gqa8k():
    """GQA 8k causal: dQ on sampled query rows and dK, dV on sampled key
    rows of one K/V head against the oracle, each row's largest error
    normalised by that row's largest oracle value; dK and dV at every
    element through exact identities -- each row of dS sums to zero, so
    sum_j dK_j = 0, and each row of P sums to one, so sum_j dV_j equals the
    sum of dO over the group's query heads and rows."""
    w = GQA_8K
    q, k, v = make_qkv(w, seed=0)
    do = make_do(w, seed=0)
    dq, dk, dv = run_bwd(w, q, k, v, do, w.scale)
    rows = sample_rows(w, 64, seed=5)
    ref = oracle.backward_dq_rows(q, k, v, do, w.scale, True, 0, rows)
    idx = torch.from_numpy(rows).cuda()
    got = dq[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    e = float(np.max(np.abs(got - ref))) / float(np.max(np.abs(ref)))
    assert e <= TOL_REL["bf16"], ("dQ rows", e)
    assert float(row_err(got, ref).max()) <= TOL_REL["bf16"], "dQ per row"
    # Key rows of the last K/V head: tile edges (128-key tiles), the last
    # key (seen by one query row per head) and random keys.
    rng = np.random.default_rng(6)
    kvh = w.Hkv - 1
    js = {0, 1, 127, 128, 129, 4095, 4096, w.Skv - 129, w.Skv - 128,
          w.Skv - 2, w.Skv - 1}
    js |= set(int(x) for x in rng.integers(0, w.Skv, 21))
    keys = np.array([(0, kvh, j) for j in sorted(js)], dtype=np.int64)
    ref_dk, ref_dv = oracle.backward_dkdv_rows(q, k, v, do, w.scale, True, 0,
                                               keys)
    kidx = torch.from_numpy(keys).cuda()
    for name, g, r in (("dK", dk, ref_dk), ("dV", dv, ref_dv)):
        got = g[kidx[:, 0], kidx[:, 1], kidx[:, 2]].double().cpu().numpy()
        assert np.all(np.isfinite(got))
        e_row = row_err(got, r)
        assert float(e_row.max()) <= TOL_REL["bf16"], (name, e_row.max(),
                                                       keys[e_row.argmax()])
    g = w.Hq // w.Hkv
    dk64, dv64 = dk.double(), dv.double()
    s_dk = dk64.sum(dim=2)
    assert float(s_dk.abs().max()) <= 1e-2 * float(dk64.abs().sum(dim=2).max())
    want = do.cuda().double().reshape(w.B, w.Hkv, g, w.Sq, w.D).sum(dim=(2, 3))
    s_dv = dv64.sum(dim=2)
    assert float((s_dv - want).abs().max()) <= \
        1e-2 * float(dv64.abs().sum(dim=2).max())
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())


def test_bwd_argument_checks():
    w = W("args", 1, 2, 2, 64, 64, 64, "f16", True)
    q, k, v = (t.cuda() for t in make_qkv(w, seed=45))
    o, lse = attn.fwd(q, k, v, causal=True)
    do = make_do(w, seed=45).cuda()
    dq, dk, dv = (torch.empty_like(t) for t in (q, k, v))
    ws_bytes = attn.attn_bwd_workspace_bytes(1, 2, 64)
    assert ws_bytes >= 2 * 2 * 128 * 4
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    base = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
            lse.data_ptr(), do.data_ptr()]
    shp = [1, 2, 2, 64, 64, 64, w.scale, 1, 0, 0, attn.ATTN_F16]
    ok = attn.attn_bwd(*base, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                       *shp, ws.data_ptr(), ws_bytes, 0)
    assert ok == attn.ATTN_OK
    # dQ aliasing Q, missing LSE, small workspace, window without causal
    assert attn.attn_bwd(*base, q.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                         *shp, ws.data_ptr(), ws_bytes, 0) == \
        attn.ATTN_ERR_INVALID_ARG
    bad = list(base)
    bad[4] = 0
    assert attn.attn_bwd(*bad, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                         *shp, ws.data_ptr(), ws_bytes, 0) == \
        attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_bwd(*base, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                         *shp, ws.data_ptr(), ws_bytes - 4, 0) == \
        attn.ATTN_ERR_INVALID_ARG
    shp_nc = [1, 2, 2, 64, 64, 64, w.scale, 0, 0, 8, attn.ATTN_F16]
    assert attn.attn_bwd(*base, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                         *shp_nc, ws.data_ptr(), ws_bytes, 0) == \
        attn.ATTN_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert attn.attn_device_status() == (0, 0)
