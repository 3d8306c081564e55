"""GPU parity of the FP8 (E4M3) forward against the fp64 CPU oracle.

The oracle decodes the E4M3 codes with its own decoder, multiplies by the
descale factors and computes exact attention.  The kernel rounds the
softmax weights to E4M3 for the P.V product, so O is compared against a
per-element bound derived from that rounding (below); LSE, which uses the
unrounded weights, keeps the 16-bit paths' 1e-3.

Bound on O (one row, oracle probabilities P_j, P_max = max_j P_j = 1/L):
the kernel's weights are p_j = P_j * l with l >= L (its reference maximum
is at most the true one), E4M3 round-to-nearest moves a weight by at most
2^-4 of itself (normal range) or 2^-10 (subnormal range, below 2^-6), and
the bf16 output adds half an ulp (2^-9 relative):

    |dO_d| <= sum_j max(2^-4 P_j, 2^-10 P_max) |v_jd| + 2^-9 |O_d| + 1e-5.

That bound assumes every rounding error points the same way.  Independent
round-to-nearest errors are far smaller: their RMS is compared with the
bound's RMS-combination sqrt(sum_j (max(...) v_jd)^2 / 3) (uniform rounding
error, variance h^2 / 3 at half-spacing h), which round-to-nearest keeps
below 1 (about 0.75 for uniformly spread mantissas) and truncation would
not.
"""
import math

import numpy as np
import pytest
import torch

import attention_attn_fwd_gb300 as attn
import oracle
from attention_attn_fwd_gb300.inputs import GQA_8K_FP8, Workload, make_qkv
from tests.gpu_parity import TOL_LSE, sample_rows

pytestmark = pytest.mark.gpu

U8 = 2.0 ** -4          # E4M3 unit roundoff (3 mantissa bits)
SUB = 2.0 ** -10        # half the E4M3 subnormal spacing
U_BF16 = 2.0 ** -9


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def W(name, B, Hq, Hkv, Sq, Skv, causal, pos=0, window=0):
    return Workload(name, B, Hq, Hkv, Sq, Skv, 128, "e4m3", causal, pos,
                    window)


def decoded(w, q8, k8, v8, qd, kd, vd):
    return (oracle.decode_e4m3(q8, qd), oracle.decode_e4m3(k8, kd),
            oracle.decode_e4m3(v8, vd))


def run_fp8(w, q8, k8, v8, qd=1.0, kd=1.0, vd=1.0, scale=None, splits=0):
    scale = w.scale if scale is None else scale
    o, lse = attn.fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), scale=scale,
                          q_descale=qd, k_descale=kd, v_descale=vd,
                          causal=w.causal, input_pos=w.input_pos,
                          window=w.window, num_splits=splits)
    torch.cuda.synchronize()
    assert attn.attn_device_status() == (0, 0)
    assert o.dtype == torch.bfloat16
    return o, lse


def bounds(w, q, k, v, scale, rows, o_ref):
    """(worst-case bound, RMS-combined bound) for each row in ``rows``."""
    g = w.Hq // w.Hkv
    worst = np.zeros((len(rows), w.D))
    rms = np.zeros((len(rows), w.D))
    for n, (b, h, i) in enumerate(rows):
        p = oracle.prob_row(q, k, v, scale, w.causal, w.input_pos, int(b),
                            int(h), int(i), w.window)
        wgt = np.maximum(U8 * p, SUB * p.max())
        av = np.abs(v[b, h // g])
        worst[n] = wgt @ av + U_BF16 * np.abs(o_ref[n]) + 1e-5
        rms[n] = np.sqrt(((wgt[:, None] * av) ** 2).sum(axis=0) / 3.0 +
                         (U_BF16 * o_ref[n]) ** 2 / 3.0)
    return worst, rms


def compare(w, o, lse, q, k, v, scale, rows=None):
    """O within the per-element bound and with rounding-noise RMS; LSE to
    1e-3.  ``rows`` None: every row."""
    if rows is None:
        rows = np.array([(b, h, i) for b in range(w.B) for h in range(w.Hq)
                         for i in range(w.Sq)], dtype=np.int64)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, scale, w.causal,
                                           w.input_pos, rows, w.window)
    idx = torch.from_numpy(rows).cuda()
    o_g = o[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    l_g = lse[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    assert np.all(np.isfinite(o_g)) and np.all(np.isfinite(l_g))
    worst, rms = bounds(w, q, k, v, scale, rows, o_ref)
    err = np.abs(o_g - o_ref)
    ratio = float(np.max(err / worst))
    noise = float(np.sqrt(np.mean(err ** 2)) / np.sqrt(np.mean(rms ** 2)))
    err_l = float(np.max(np.abs(l_g - lse_ref)))
    assert ratio <= 1.0, (w.name, "O over its bound", ratio)
    assert noise <= 1.0, (w.name, "O error RMS over rounding noise", noise)
    assert err_l <= TOL_LSE, (w.name, "LSE", err_l)
    return ratio, noise, err_l


CASES = [
    (W("noncausal_ragged", 1, 4, 2, 300, 383, False), (1.0, 1.0, 1.0)),
    (W("causal_gqa8_offset", 1, 16, 2, 513, 700, True, 187), (0.5, 2.0, 0.75)),
    (W("causal_square", 2, 4, 4, 384, 384, True), (1.25, 0.8, 1.5)),
    (W("rows_mode_odd_group", 1, 3, 1, 260, 260, True), (1.0, 1.0, 2.0)),
    (W("window_offset", 1, 8, 2, 400, 900, True, 500, 300), (0.9, 1.1, 1.0)),
    (W("packed_decode_rows", 2, 32, 4, 4, 777, True, 773), (1.0, 0.5, 1.0)),
    (W("packed_noncausal", 1, 8, 2, 5, 700, False), (2.0, 1.0, 0.25)),
    (W("packed_window", 2, 8, 2, 6, 900, True, 894, 200), (1.0, 1.0, 1.0)),
    (W("one_key", 1, 2, 1, 3, 1, False), (1.0, 1.0, 1.0)),
]


@pytest.mark.parametrize("w,ds", CASES, ids=lambda c: getattr(c, "name", ""))
def test_against_oracle(w, ds):
    q8, k8, v8 = make_qkv(w, seed=51)
    qd, kd, vd = ds
    o, lse = run_fp8(w, q8, k8, v8, qd, kd, vd)
    q, k, v = decoded(w, q8, k8, v8, qd, kd, vd)
    compare(w, o, lse, q, k, v, w.scale)


@pytest.mark.parametrize("splits", [-1, 3])
def test_splitkv_decode(splits):
    w = W("splitkv_decode", 2, 32, 8, 1, 4096, True, 4095)
    q8, k8, v8 = make_qkv(w, seed=52)
    o, lse = run_fp8(w, q8, k8, v8, 1.0, 1.0, 0.5, splits=splits)
    q, k, v = decoded(w, q8, k8, v8, 1.0, 1.0, 0.5)
    compare(w, o, lse, q, k, v, w.scale)


@pytest.mark.parametrize("w,splits", [
    (W("splitkv_chunk_rows", 1, 4, 2, 100, 2000, True, 1900), 3),
    (W("splitkv_decode_window", 2, 8, 2, 1, 3000, True, 2999, 500), 4),
], ids=["chunk_rows", "decode_window"])
def test_splitkv_remaining_variants(w, splits):
    """Split-KV with one head per tile (no window) and packed with a window:
    with the cases above, every FP8 variant has a parity case."""
    q8, k8, v8 = make_qkv(w, seed=55)
    o, lse = run_fp8(w, q8, k8, v8, splits=splits)
    q, k, v = decoded(w, q8, k8, v8, 1.0, 1.0, 1.0)
    compare(w, o, lse, q, k, v, w.scale)


def test_splitkv_window_chunk():
    w = W("splitkv_window", 1, 8, 2, 64, 3000, True, 2936, 1000)
    q8, k8, v8 = make_qkv(w, seed=53)
    o, lse = run_fp8(w, q8, k8, v8, splits=4)
    q, k, v = decoded(w, q8, k8, v8, 1.0, 1.0, 1.0)
    compare(w, o, lse, q, k, v, w.scale)


@pytest.mark.parametrize("scale", [-0.0883883, 0.0, 0.4])
def test_scale_values(scale):
    w = W("scale", 1, 4, 2, 256, 520, True, 7)
    q8, k8, v8 = make_qkv(w, seed=54)
    o, lse = run_fp8(w, q8, k8, v8, 0.75, 1.0, 1.0, scale=scale)
    q, k, v = decoded(w, q8, k8, v8, 0.75, 1.0, 1.0)
    compare(w, o, lse, q, k, v, scale)


def test_full_size_sampled():
    """The FP8 bench workload at full size: sampled rows against the
    oracle; every element finite and inside its head's V range."""
    w = GQA_8K_FP8
    q8, k8, v8 = make_qkv(w, seed=0)
    o, lse = run_fp8(w, q8, k8, v8)
    q, k, v = decoded(w, q8, k8, v8, 1.0, 1.0, 1.0)
    rows = sample_rows(w, 64, seed=0)
    compare(w, o, lse, q, k, v, w.scale, rows)
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    g = w.Hq // w.Hkv
    vg = v8.cuda().float()
    vmax = vg.amax(dim=2).repeat_interleave(g, dim=1)[:, :, None, :]
    vmin = vg.amin(dim=2).repeat_interleave(g, dim=1)[:, :, None, :]
    slack = U8 * float(vg.abs().max()) + 1e-2
    of = o.float()
    assert bool((of <= vmax + slack).all()) and bool((of >= vmin - slack).all())


def test_uint8_codes_accepted():
    """Raw uint8 codes give the bit-identical result of float8 tensors."""
    w = W("u8", 1, 4, 2, 130, 260, True)
    q8, k8, v8 = (t.cuda() for t in make_qkv(w, seed=55))
    o1, l1 = attn.fwd_fp8(q8, k8, v8, causal=True)
    o2, l2 = attn.fwd_fp8(q8.view(torch.uint8), k8.view(torch.uint8),
                          v8.view(torch.uint8), causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_bitwise_reproducible():
    w = W("repro", 1, 8, 2, 1000, 1000, True)
    q8, k8, v8 = (t.cuda() for t in make_qkv(w, seed=56))
    o1, l1 = attn.fwd_fp8(q8, k8, v8, causal=True)
    o2, l2 = attn.fwd_fp8(q8, k8, v8, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_rejected_forms():
    w = W("rej", 1, 2, 2, 128, 128, False)
    q8, k8, v8 = (t.cuda() for t in make_qkv(w, seed=57))
    o = torch.empty(1, 2, 128, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 2, 128, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    args = (q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), o.data_ptr(),
            lse.data_ptr(), 1, 2, 2, 128, 128)
    # E4M3 through a 16-bit entry point (no descales): invalid.
    assert attn.attn_fwd(*args, 128, 0.1, 0, 0, attn.ATTN_E4M3,
                         stream) == attn.ATTN_ERR_INVALID_ARG
    # Head dimension 64 in FP8: not implemented.
    assert attn.attn_fwd_fp8(*args, 64, 0.1, 1.0, 1.0, 1.0, 0, 0, 0, 0, 0, 0,
                             stream) == attn.ATTN_ERR_UNSUPPORTED
    # Non-finite descale, or a score factor that overflows fp32.
    assert attn.attn_fwd_fp8(*args, 128, 0.1, math.inf, 1.0, 1.0, 0, 0, 0,
                             0, 0, 0, stream) == attn.ATTN_ERR_INVALID_ARG
    assert attn.attn_fwd_fp8(*args, 128, 1e30, 1e30, 1.0, 1.0, 0, 0, 0, 0, 0,
                             0, stream) == attn.ATTN_ERR_INVALID_ARG
    # Split-KV without a workspace.
    assert attn.attn_fwd_fp8(*args, 128, 0.1, 1.0, 1.0, 1.0, 0, 0, 0, 1, 0,
                             0, stream) == attn.ATTN_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert attn.attn_device_status() == (0, 0)
