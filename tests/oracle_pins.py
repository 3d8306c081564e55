"""Checks that pin the CPU oracle to facts that do not come from its own code.

Each check takes an ``oracle.Oracle`` instance so the same checks can run
against the real oracle and against deliberately broken copies of it (see
test_oracle_mutants.py).  Every check raises AssertionError on failure.
"""
import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "hand_cases.json")

_MATH = {"log": math.log, "exp": math.exp, "e": math.e}


def _val(x):
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, _MATH))
    return float(x)


def _arr(nested):
    def conv(n):
        return [conv(t) for t in n] if isinstance(n, list) else _val(n)
    return np.array(conv(nested), dtype=np.float64)


def _rand(shape, rng):
    return rng.standard_normal(shape)


def pin_hand_cases(orc):
    """Hand-derived small cases stored under tests/golden/."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q, k, v = _arr(c["q"]), _arr(c["k"]), _arr(c["v"])
        o, lse = orc.attention(q, k, v, _val(c["scale"]), c["causal"],
                               c["input_pos"])
        np.testing.assert_allclose(o, _arr(c["o"]), rtol=0, atol=1e-12,
                                   err_msg=c["name"])
        np.testing.assert_allclose(lse, _arr(c["lse"]), rtol=0, atol=1e-12,
                                   err_msg=c["name"])


def pin_single_key(orc):
    """Skv = 1: the only weight is 1, so O = V_0 and LSE = scale * q.k_0."""
    rng = np.random.default_rng(1)
    B, Hq, Hkv, Sq, D = 2, 4, 2, 5, 8
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, 1, D), rng)
    v = _rand((B, Hkv, 1, D), rng)
    for causal, pos in ((False, 0), (True, 0), (True, 3)):
        o, lse = orc.attention(q, k, v, 0.3, causal, pos)
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            np.testing.assert_allclose(
                o[:, h], np.broadcast_to(v[:, kvh, 0][:, None, :], (B, Sq, D)),
                rtol=0, atol=1e-13)
            dots = np.einsum("bsd,bd->bs", q[:, h], k[:, kvh, 0])
            np.testing.assert_allclose(lse[:, h], 0.3 * dots, rtol=0,
                                       atol=1e-12)


def _visible_counts(Sq, Skv, causal, pos):
    if not causal:
        return np.full(Sq, Skv)
    return np.array([min(Skv, pos + i + 1) for i in range(Sq)])


def pin_uniform_scores(orc):
    """scale = 0 (or Q = 0): O_i = mean of the visible V rows, LSE = ln(#visible)."""
    rng = np.random.default_rng(2)
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 7, 11, 6
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    for causal, pos in ((False, 0), (True, 0), (True, 2), (True, 9)):
        cnt = _visible_counts(Sq, Skv, causal, pos)
        for qq, sc in ((q, 0.0), (np.zeros_like(q), 1.7)):
            o, lse = orc.attention(qq, k, v, sc, causal, pos)
            for h in range(Hq):
                kvh = h // (Hq // Hkv)
                for i in range(Sq):
                    mean = v[0, kvh, :cnt[i]].mean(axis=0)
                    np.testing.assert_allclose(o[0, h, i], mean, rtol=0,
                                               atol=1e-12)
                    assert abs(lse[0, h, i] - math.log(cnt[i])) < 1e-12


def pin_prob_rows(orc):
    """Softmax weights are >= 0, zero where masked, and sum to 1."""
    rng = np.random.default_rng(3)
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 6, 9, 4
    q = _rand((B, Hq, Sq, D), rng) * 3
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    for causal, pos in ((False, 0), (True, 0), (True, 2)):
        for h in range(Hq):
            for i in range(Sq):
                p = orc.prob_row(q, k, v, 0.5, causal, pos, 0, h, i)
                assert np.all(p >= 0)
                assert abs(p.sum() - 1.0) < 1e-12
                if causal:
                    assert np.all(p[pos + i + 1:] == 0)
                    assert np.all(p[:min(Skv, pos + i + 1)] > 0)


def pin_gqa_equivalence(orc):
    """GQA equals MHA on K/V whose heads are repeated group-size times."""
    rng = np.random.default_rng(4)
    B, Hq, Hkv, Sq, Skv, D = 2, 8, 2, 5, 7, 4
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    g = Hq // Hkv
    k_rep, v_rep = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    for causal, pos in ((False, 0), (True, 1)):
        o1, l1 = orc.attention(q, k, v, 0.4, causal, pos)
        o2, l2 = orc.attention(q, k_rep, v_rep, 0.4, causal, pos)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def pin_causal_first_row(orc):
    """Causal with input_pos = 0: query 0 sees only key 0, so O = V_0."""
    rng = np.random.default_rng(5)
    B, Hq, Hkv, Sq, Skv, D = 2, 4, 4, 3, 6, 5
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    o, _ = orc.attention(q, k, v, 0.7, True, 0)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=1e-13)


def pin_permutation_invariance(orc):
    """Non-causal: permuting K and V rows together changes nothing."""
    rng = np.random.default_rng(6)
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 2, 4, 9, 3
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    perm = rng.permutation(Skv)
    o1, l1 = orc.attention(q, k, v, 0.9, False, 0)
    o2, l2 = orc.attention(q, k[:, :, perm], v[:, :, perm], 0.9, False, 0)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def pin_causal_prefix(orc):
    """Causal row i equals non-causal attention over the keys [0, pos+i]."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 4, 10, 3
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    # Future keys with huge scores must not leak in: with a maximum taken over
    # masked keys too, every visible weight would underflow to zero.
    k = k.copy()
    k[:, :, 7:] = 1000.0 * np.sign(q[0, 0, 0])[None, None, None, :]
    for pos in (0, 3, 6, 20):
        o, lse = orc.attention(q, k, v, 0.8, True, pos)
        for i in range(Sq):
            n = min(Skv, pos + i + 1)
            o2, l2 = orc.attention(q[:, :, i:i + 1], k[:, :, :n], v[:, :, :n],
                                   0.8, False, 0)
            np.testing.assert_allclose(o[:, :, i], o2[:, :, 0], rtol=0,
                                       atol=1e-13)
            np.testing.assert_allclose(lse[:, :, i], l2[:, :, 0], rtol=0,
                                       atol=1e-13)


def pin_shift_invariance(orc):
    """Adding c to every key shifts row i's scores by scale*q_i.c: O is
    unchanged and LSE moves by exactly that amount, even when the shift is
    far beyond exp's range (a softmax without the max subtraction fails)."""
    rng = np.random.default_rng(12)
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 4, 6, 3
    q = np.abs(_rand((B, Hq, Sq, D), rng)) + 1.0
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    c = np.full(D, 400.0)
    for causal in (False, True):
        o1, l1 = orc.attention(q, k, v, 1.0, causal, 0)
        o2, l2 = orc.attention(q, k + c, v, 1.0, causal, 0)
        shift = np.einsum("bhsd,d->bhs", q, c)
        assert np.all(np.isfinite(o2)) and np.all(np.isfinite(l2))
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-9)
        np.testing.assert_allclose(l2 - shift, l1, rtol=0, atol=1e-9)


def pin_negated_scale(orc):
    """scale -> -scale with K -> -K is the same computation."""
    rng = np.random.default_rng(8)
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 3, 5, 4
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    o1, l1 = orc.attention(q, k, v, -0.6, True, 1)
    o2, l2 = orc.attention(q, -k, v, 0.6, True, 1)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def pin_torch_sdpa(orc):
    """Library pin: torch's softmax-attention and logsumexp in float64 on CPU."""
    F = torch.nn.functional
    rng = np.random.default_rng(9)
    for (B, Hq, Hkv, Sq, Skv, D, causal, pos) in (
            (2, 4, 4, 9, 13, 16, False, 0),
            (1, 4, 4, 12, 12, 8, True, 0),
            (1, 2, 2, 5, 11, 8, True, 4)):
        q = _rand((B, Hq, Sq, D), rng)
        k = _rand((B, Hkv, Skv, D), rng)
        v = _rand((B, Hkv, Skv, D), rng)
        scale = 0.35
        o, lse = orc.attention(q, k, v, scale, causal, pos)
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        if causal and pos == 0 and Sq == Skv:
            ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True,
                                                 scale=scale)
            mask = torch.ones(Sq, Skv, dtype=torch.bool).tril()
        elif causal:
            rows = torch.arange(Sq)[:, None] + pos
            mask = torch.arange(Skv)[None, :] <= rows
            ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                                 scale=scale)
        else:
            mask = torch.ones(Sq, Skv, dtype=torch.bool)
            ref = F.scaled_dot_product_attention(tq, tk, tv, scale=scale)
        np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
        s = torch.matmul(tq, tk.transpose(-1, -2)) * scale
        s = s.masked_fill(~mask, float("-inf"))
        np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(),
                                   rtol=0, atol=1e-12)


def pin_window_single_key(orc):
    """Window W = 1: each query sees only its own position, so O = V at that
    position and LSE = scale * q . k there (a one-term softmax)."""
    rng = np.random.default_rng(21)
    B, Hq, Hkv, Sq, Skv, D, pos = 2, 4, 2, 5, 12, 8, 6
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    o, lse = orc.attention(q, k, v, 0.4, True, pos, window=1)
    for b in range(B):
        for h in range(Hq):
            kvh = h // (Hq // Hkv)
            for i in range(Sq):
                j = min(pos + i, Skv - 1)
                if pos + i > Skv - 1:
                    continue
                np.testing.assert_allclose(o[b, h, i], v[b, kvh, j],
                                           rtol=0, atol=1e-12)
                np.testing.assert_allclose(
                    lse[b, h, i], 0.4 * float(q[b, h, i] @ k[b, kvh, j]),
                    rtol=0, atol=1e-12)


def pin_window_uniform_scores(orc):
    """scale = 0 with a window: O is the mean of V over the window's keys
    (positions pos-W+1 .. pos, clipped to the cache) and LSE = ln(count)."""
    rng = np.random.default_rng(22)
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 6, 20, 4
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    for pos, W in ((0, 3), (4, 5), (13, 2), (10, 30)):
        o, lse = orc.attention(q, k, v, 0.0, True, pos, window=W)
        for i in range(Sq):
            lo, hi = max(0, pos + i - W + 1), min(pos + i, Skv - 1)
            np.testing.assert_allclose(o[0, :, i],
                                       np.broadcast_to(v[0, 0, lo:hi + 1]
                                                       .mean(axis=0), (Hq, D)),
                                       rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[0, :, i], math.log(hi - lo + 1),
                                       rtol=0, atol=1e-12)


def pin_window_wide_is_causal(orc):
    """A window at least as long as every query's prefix changes nothing."""
    rng = np.random.default_rng(23)
    q = _rand((1, 2, 7, 8), rng)
    k = _rand((1, 2, 15, 8), rng)
    v = _rand((1, 2, 15, 8), rng)
    o, lse = orc.attention(q, k, v, 0.5, True, 3)
    for W in (10, 11, 40):
        ow, lw = orc.attention(q, k, v, 0.5, True, 3, window=W)
        np.testing.assert_array_equal(ow, o)
        np.testing.assert_array_equal(lw, lse)


def pin_window_decode_slice(orc):
    """Library pin: one query at position pos with window W equals torch's
    float64 softmax attention (no mask) over the contiguous key slice
    [pos-W+1, pos] -- the window as a slice of the cache, not a predicate."""
    F = torch.nn.functional
    rng = np.random.default_rng(24)
    B, Hq, Hkv, Skv, D = 2, 4, 2, 40, 16
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    for pos, W in ((39, 7), (25, 1), (30, 31), (12, 5)):
        q = _rand((B, Hq, 1, D), rng)
        o, lse = orc.attention(q, k, v, 0.3, True, pos, window=W)
        lo = max(0, pos - W + 1)
        g = Hq // Hkv
        tq = torch.from_numpy(q)
        tk = torch.from_numpy(k[:, :, lo:pos + 1]).repeat_interleave(g, dim=1)
        tv = torch.from_numpy(v[:, :, lo:pos + 1]).repeat_interleave(g, dim=1)
        ref = F.scaled_dot_product_attention(tq, tk, tv, scale=0.3)
        np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
        s = torch.matmul(tq, tk.transpose(-1, -2)) * 0.3
        np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(),
                                   rtol=0, atol=1e-12)


def _sdpa_grads(q, k, v, do, scale, causal, pos, window):
    """torch float64 autograd through scaled_dot_product_attention with the
    visibility written as an explicit boolean mask."""
    F = torch.nn.functional
    g = q.shape[1] // k.shape[1]
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    Sq, Skv = q.shape[2], k.shape[2]
    rows = torch.arange(Sq)[:, None] + pos
    cols = torch.arange(Skv)[None, :]
    mask = torch.ones(Sq, Skv, dtype=torch.bool)
    if causal:
        mask = cols <= rows
        if window:
            mask = mask & (cols > rows - window)
    o = F.scaled_dot_product_attention(tq, tk.repeat_interleave(g, dim=1),
                                       tv.repeat_interleave(g, dim=1),
                                       attn_mask=mask, scale=scale)
    o.backward(torch.from_numpy(do))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def pin_bwd_torch_autograd(orc):
    """Library pin of the backward: torch autograd in float64 (GQA heads
    expanded by repeat_interleave, whose gradient sums the group)."""
    rng = np.random.default_rng(31)
    for (B, Hq, Hkv, Sq, Skv, D, causal, pos, W) in (
            (2, 4, 2, 6, 9, 8, False, 0, 0),
            (1, 2, 2, 7, 7, 4, True, 0, 0),
            (1, 4, 1, 5, 12, 8, True, 6, 0),
            (2, 2, 1, 6, 14, 8, True, 5, 4)):
        q = _rand((B, Hq, Sq, D), rng)
        k = _rand((B, Hkv, Skv, D), rng)
        v = _rand((B, Hkv, Skv, D), rng)
        do = _rand((B, Hq, Sq, D), rng)
        got = orc.backward(q, k, v, do, 0.45, causal, pos, W)
        ref = _sdpa_grads(q, k, v, do, 0.45, causal, pos, W)
        for name, a_, b_ in zip(("dQ", "dK", "dV"), got, ref):
            np.testing.assert_allclose(a_, b_, rtol=0, atol=1e-12,
                                       err_msg=name)
        # The row-sampled dQ against the same library gradient.
        rows = np.array([(bb, h, i) for bb in range(B) for h in range(Hq)
                         for i in range(0, Sq, 2)])
        dq_rows = orc.backward_dq_rows(q, k, v, do, 0.45, causal, pos, rows, W)
        np.testing.assert_allclose(dq_rows, ref[0][rows[:, 0], rows[:, 1],
                                                   rows[:, 2]],
                                   rtol=0, atol=1e-12, err_msg="dQ rows")
        # The key-sampled dK / dV (every key of the last K/V head, every
        # third key of the others, in shuffled order) against the same
        # library gradients.
        keys = [(bb, kh, j) for bb in range(B) for kh in range(Hkv)
                for j in range(Skv) if kh == Hkv - 1 or j % 3 == 0]
        keys = np.array(keys)[rng.permutation(len(keys))]
        dk_rows, dv_rows = orc.backward_dkdv_rows(q, k, v, do, 0.45, causal,
                                                  pos, keys, W)
        sel = (keys[:, 0], keys[:, 1], keys[:, 2])
        np.testing.assert_allclose(dk_rows, ref[1][sel], rtol=0, atol=1e-12,
                                   err_msg="dK rows")
        np.testing.assert_allclose(dv_rows, ref[2][sel], rtol=0, atol=1e-12,
                                   err_msg="dV rows")


def pin_bwd_finite_differences(orc):
    """The backward is the derivative of the forward: central differences
    of L = sum(O * dO) through the oracle's forward pass, every input
    element of a tiny causal GQA case with an offset and a window."""
    rng = np.random.default_rng(32)
    B, Hq, Hkv, Sq, Skv, D, pos, W = 1, 2, 1, 3, 5, 3, 2, 3
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, Skv, D), rng)
    v = _rand((B, Hkv, Skv, D), rng)
    do = _rand((B, Hq, Sq, D), rng)
    grads = orc.backward(q, k, v, do, 0.7, True, pos, W)
    h = 1e-5
    for x, gx in zip((q, k, v), grads):
        for idx in np.ndindex(x.shape):
            old = x[idx]
            x[idx] = old + h
            lp = float(np.sum(orc.attention(q, k, v, 0.7, True, pos, W)[0] * do))
            x[idx] = old - h
            lm = float(np.sum(orc.attention(q, k, v, 0.7, True, pos, W)[0] * do))
            x[idx] = old
            assert abs((lp - lm) / (2 * h) - gx[idx]) < 1e-7, idx


def pin_bwd_single_key(orc):
    """Skv = 1: O = V_0 whatever Q and K are, so dQ = dK = 0 and dV_0 is
    the sum of dO over the group's query heads and rows."""
    rng = np.random.default_rng(33)
    B, Hq, Hkv, Sq, D = 2, 4, 2, 3, 5
    q = _rand((B, Hq, Sq, D), rng)
    k = _rand((B, Hkv, 1, D), rng)
    v = _rand((B, Hkv, 1, D), rng)
    do = _rand((B, Hq, Sq, D), rng)
    dq, dk, dv = orc.backward(q, k, v, do, 0.9, True, 0)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    want = do.reshape(B, Hkv, Hq // Hkv, Sq, D).sum(axis=(2, 3))
    np.testing.assert_allclose(dv[:, :, 0], want, rtol=0, atol=1e-12)
    keys = np.array([(bb, kh, 0) for bb in range(B) for kh in range(Hkv)])
    dk_rows, dv_rows = orc.backward_dkdv_rows(q, k, v, do, 0.9, True, 0, keys)
    assert np.all(dk_rows == 0.0)
    np.testing.assert_allclose(dv_rows, want.reshape(-1, D), rtol=0,
                               atol=1e-12)


# FP8 (E4M3) inputs: the oracle's own decoder, then the definition above.

# Codes and values fixed by the E4M3 bit layout (sign | 4-bit exponent,
# bias 7 | 3-bit mantissa; exponent 0 subnormal; S.1111.111 NaN).
_E4M3_HAND = {
    0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
    0x30: 0.5, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x44: 3.0, 0x77: 240.0,
    0x78: 256.0, 0x7E: 448.0, 0x81: -(2.0 ** -9), 0xB8: -1.0, 0xFE: -448.0,
}


def pin_e4m3_closed_forms(orc):
    """Values of hand-picked codes, signed zero, the two NaN codes, and
    the ordering of the positive codes."""
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.decode_e4m3(codes)
    for c, want in _E4M3_HAND.items():
        assert vals[c] == want, (hex(c), vals[c], want)
    assert vals[0x80] == 0.0 and math.copysign(1.0, vals[0x80]) < 0
    assert math.isnan(vals[0x7F]) and math.isnan(vals[0xFF])
    assert int(np.isnan(vals).sum()) == 2
    assert np.all(np.diff(vals[:0x7F]) > 0)          # 0x00 .. 0x7E ascend
    np.testing.assert_array_equal(vals[0x80:0xFF], -vals[:0x7F])
    half = orc.decode_e4m3(np.array([0x38, 0x40, 0x01], np.uint8), 0.375)
    np.testing.assert_array_equal(half, [0.375, 0.75, 0.375 * 2.0 ** -9])


def pin_e4m3_torch(orc):
    """Every code against torch's float8_e4m3fn conversion (library)."""
    codes = torch.arange(256, dtype=torch.uint8)
    want = codes.view(torch.float8_e4m3fn).double().numpy()
    got = orc.decode_e4m3(codes.numpy())
    np.testing.assert_array_equal(got, want)


def _e4m3(shape, rng):
    """Random E4M3 codes of N(0, 1) draws (torch's rounding), uint8."""
    x = torch.from_numpy(_rand(shape, rng).astype(np.float32))
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_fp8_attention_sdpa(orc):
    """Decoded E4M3 inputs with descale factors, through the oracle, against
    torch float64 scaled_dot_product_attention on torch-decoded inputs times
    the same factors; the V factor scales O and leaves LSE alone."""
    rng = np.random.default_rng(41)
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 9, 13, 16
    q8, k8, v8 = (_e4m3((B, Hq, Sq, D), rng), _e4m3((B, Hkv, Skv, D), rng),
                  _e4m3((B, Hkv, Skv, D), rng))
    qd, kd, vd, scale = 0.75, 1.25, 0.5, 0.3
    for causal, pos, window in ((False, 0, 0), (True, 3, 0), (True, 4, 5)):
        o, lse = orc.attention(orc.decode_e4m3(q8, qd),
                               orc.decode_e4m3(k8, kd),
                               orc.decode_e4m3(v8, vd), scale, causal, pos,
                               window)

        def lib(c, f):
            return (torch.from_numpy(c).view(torch.float8_e4m3fn).double()
                    * f)
        q, k, v = lib(q8, qd), lib(k8, kd), lib(v8, vd)
        k = k.repeat_interleave(Hq // Hkv, dim=1)
        v = v.repeat_interleave(Hq // Hkv, dim=1)
        s = scale * q @ k.transpose(-1, -2)
        mask = torch.ones(Sq, Skv, dtype=torch.bool)
        if causal:
            i = torch.arange(Sq)[:, None] + pos
            j = torch.arange(Skv)[None, :]
            mask = j <= i
            if window:
                mask &= j > i - window
        s = s.masked_fill(~mask, float("-inf"))
        want_o = torch.softmax(s, dim=-1) @ v
        want_lse = torch.logsumexp(s, dim=-1)
        np.testing.assert_allclose(o, want_o.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, want_lse.numpy(), rtol=0, atol=1e-12)
        o1, lse1 = orc.attention(orc.decode_e4m3(q8, qd),
                                 orc.decode_e4m3(k8, kd),
                                 orc.decode_e4m3(v8, 1.0), scale, causal,
                                 pos, window)
        np.testing.assert_allclose(o, vd * o1, rtol=0, atol=1e-12)
        np.testing.assert_array_equal(lse, lse1)


ALL_PINS = [
    pin_hand_cases, pin_single_key, pin_uniform_scores, pin_prob_rows,
    pin_gqa_equivalence, pin_causal_first_row, pin_permutation_invariance,
    pin_causal_prefix, pin_shift_invariance, pin_negated_scale,
    pin_torch_sdpa, pin_window_single_key, pin_window_uniform_scores,
    pin_window_wide_is_causal, pin_window_decode_slice,
    pin_bwd_torch_autograd, pin_bwd_finite_differences, pin_bwd_single_key,
    pin_e4m3_closed_forms, pin_e4m3_torch, pin_fp8_attention_sdpa,
]
