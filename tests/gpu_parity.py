"""Shared helpers of the GPU parity tests: run the CUDA path through the C
ABI and compare with the fp64 oracle element by element."""
import numpy as np
import torch

import attention_attn_fwd_gb300 as attn
import oracle
from attention_attn_fwd_gb300.inputs import make_qkv

# Max-abs tolerances on O per dtype and on LSE (natural log).
TOL_O = {"f16": 2e-3, "bf16": 1.5e-2}
TOL_LSE = 1e-3


def run_gpu(w, q, k, v, scale=None):
    scale = w.scale if scale is None else scale
    o, lse = attn.fwd(q.cuda(), k.cuda(), v.cuda(), scale=scale,
                      causal=w.causal, input_pos=w.input_pos, window=w.window)
    torch.cuda.synchronize()
    st, code = attn.attn_device_status()
    assert st == 0, "device status %d code %#x" % (st, code)
    return o, lse


def check_full(w, seed=0, scale=None, q=None, k=None, v=None):
    """Every output element against the oracle; returns the max errors."""
    if q is None:
        q, k, v = make_qkv(w, seed)
    scale = w.scale if scale is None else scale
    o, lse = run_gpu(w, q, k, v, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, scale, w.causal, w.input_pos,
                                      w.window)
    o_gpu = o.double().cpu().numpy()
    lse_gpu = lse.double().cpu().numpy()
    assert np.all(np.isfinite(o_gpu)) and np.all(np.isfinite(lse_gpu))
    err_o = float(np.max(np.abs(o_gpu - o_ref))) if o_ref.size else 0.0
    err_l = float(np.max(np.abs(lse_gpu - lse_ref))) if lse_ref.size else 0.0
    assert err_o <= TOL_O[w.dtype], (w, "O", err_o)
    assert err_l <= TOL_LSE, (w, "LSE", err_l)
    return err_o, err_l


def sample_rows(w, n, seed=0):
    """(b, h, i) rows: tile edges of the first/last heads plus random rows."""
    rng = np.random.default_rng(seed)
    rows = set()
    edges = [0, 1, 127, 128, 129, 255, 256, w.Sq // 2, w.Sq - 2, w.Sq - 1]
    edges = [i for i in edges if 0 <= i < w.Sq]
    for b in sorted({0, w.B - 1}):
        for h in sorted({0, w.Hq - 1, int(rng.integers(w.Hq))}):
            for i in edges:
                rows.add((b, h, i))
    while len(rows) < n:
        rows.add((int(rng.integers(w.B)), int(rng.integers(w.Hq)),
                  int(rng.integers(w.Sq))))
    return np.array(sorted(rows), dtype=np.int64)


def check_sampled(w, seed=0, n_rows=192):
    """Full-size run; sampled rows against the oracle, global properties on
    every element."""
    q, k, v = make_qkv(w, seed)
    o, lse = run_gpu(w, q, k, v)
    rows = sample_rows(w, n_rows, seed)
    o_ref, lse_ref = oracle.attention_rows(q, k, v, w.scale, w.causal,
                                           w.input_pos, rows, w.window)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    idx = torch.from_numpy(rows).cuda()
    o_rows = o[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    lse_rows = lse[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    err_o = float(np.max(np.abs(o_rows - o_ref)))
    err_l = float(np.max(np.abs(lse_rows - lse_ref)))
    assert err_o <= TOL_O[w.dtype], (w.name, "O", err_o)
    assert err_l <= TOL_LSE, (w.name, "LSE", err_l)
    # Properties at every element: finite, and each output lies within the
    # range of its K/V head's value rows (a convex combination of them).
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
    g = w.Hq // w.Hkv
    vg = v.cuda().float()
    vmax = vg.amax(dim=2).repeat_interleave(g, dim=1)[:, :, None, :]
    vmin = vg.amin(dim=2).repeat_interleave(g, dim=1)[:, :, None, :]
    of = o.float()
    tol = TOL_O[w.dtype]
    assert bool((of <= vmax + tol).all()) and bool((of >= vmin - tol).all())
    return err_o, err_l
