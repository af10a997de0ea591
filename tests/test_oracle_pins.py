"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Every check here is independent of the oracle's own code: closed forms derived
by hand, invariants the mathematics fixes, an independent blockwise
online-softmax recomputation (the FlashAttention-2 loop with deferred
normalisation from the tiny_flash_attn.py page, and the normalise-every-step
loop of the Modular recipe's FlashAttention kernel listing), and torch's fp64
scaled_dot_product_attention as a library special case.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape) * scale


def _visible_count(i, S, causal, window):
    lo = 0
    hi = i if causal else S - 1
    if window > 0:
        lo = max(0, i - window + 1)
        if not causal:
            hi = min(S - 1, i + window - 1)
    return hi - lo + 1


MASKS = [(False, -1), (True, -1), (True, 1), (True, 2), (True, 5), (True, 64), (False, 1),
         (False, 3), (False, 64)]


# --- closed forms -----------------------------------------------------------

@pytest.mark.parametrize("causal,window", MASKS)
def test_constant_values_give_ones(oracle_mod, causal, window):
    """V == 1 gives O == 1 exactly when every softmax row sums to one."""
    B, S, H, D = 2, 37, 3, 8
    q, k = _rand((B, S, H, D), 1), _rand((B, S, H, D), 2)
    v = np.ones((B, S, H, D))
    out, _ = oracle_mod.mha_forward(q, k, v, 0.7, causal, window)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal,window", MASKS)
def test_identical_keys_average_visible_values(oracle_mod, causal, window):
    """All keys equal: every visible score is the same, O[i] = mean of the
    visible V rows and lse = scale*q.k + ln(#visible). Pins the mask/window
    boundary convention (window W = the W keys ending at the query)."""
    B, S, H, D = 1, 23, 2, 4
    scale = 0.37
    q = _rand((B, S, H, D), 3)
    krow = _rand((1, 1, H, D), 4)
    k = np.broadcast_to(krow, (B, S, H, D)).copy()
    v = _rand((B, S, H, D), 5)
    out, lse = oracle_mod.mha_forward(q, k, v, scale, causal, window)
    for i in range(S):
        lo = max(0, i - window + 1) if window > 0 else 0
        hi = i + 1 if causal else (min(S, i + window) if window > 0 else S)
        n = _visible_count(i, S, causal, window)
        assert hi - lo == n
        for h in range(H):
            np.testing.assert_allclose(out[0, i, h], v[0, lo:hi, h].mean(axis=0), atol=1e-13)
            expect = scale * float(q[0, i, h] @ krow[0, 0, h]) + math.log(n)
            assert abs(lse[0, h, i] - expect) < 1e-12


def test_scale_zero_is_uniform(oracle_mod):
    B, S, H, D = 1, 19, 1, 3
    q, k, v = _rand((B, S, H, D), 6), _rand((B, S, H, D), 7), _rand((B, S, H, D), 8)
    out, lse = oracle_mod.mha_forward(q, k, v, 0.0, True, 4)
    for i in range(S):
        lo = max(0, i - 3)
        np.testing.assert_allclose(out[0, i, 0], v[0, lo:i + 1, 0].mean(axis=0), atol=1e-14)
        assert abs(lse[0, 0, i] - math.log(i + 1 - lo)) < 1e-14


def test_single_visible_key_returns_its_value(oracle_mod):
    """Window 1 leaves each query only itself: O[i] = V[i], lse = scale*q_i.k_i."""
    B, S, H, D = 2, 11, 2, 5
    q, k, v = _rand((B, S, H, D), 9), _rand((B, S, H, D), 10), _rand((B, S, H, D), 11)
    out, lse = oracle_mod.mha_forward(q, k, v, 0.5, True, 1)
    np.testing.assert_array_equal(out, v)
    expect = 0.5 * np.einsum("bshd,bshd->bhs", q, k)
    np.testing.assert_allclose(lse, expect, atol=1e-13)


def test_causal_row_zero_returns_first_value(oracle_mod):
    B, S, H, D = 1, 9, 3, 4
    q, k, v = _rand((B, S, H, D), 12), _rand((B, S, H, D), 13), _rand((B, S, H, D), 14)
    out, _ = oracle_mod.mha_forward(q, k, v, 1.3, True, -1)
    np.testing.assert_array_equal(out[:, 0], v[:, 0])


def test_two_key_sigmoid(oracle_mod):
    """D=1, S=2, no mask: O = sigmoid(s0-s1) v0 + sigmoid(s1-s0) v1."""
    rng = np.random.default_rng(15)
    for _ in range(20):
        q = rng.standard_normal((1, 2, 1, 1)) * 3
        k = rng.standard_normal((1, 2, 1, 1)) * 3
        v = rng.standard_normal((1, 2, 1, 1))
        scale = float(rng.uniform(0.1, 2.0))
        out, lse = oracle_mod.mha_forward(q, k, v, scale, False, -1)
        for i in range(2):
            s0 = scale * q[0, i, 0, 0] * k[0, 0, 0, 0]
            s1 = scale * q[0, i, 0, 0] * k[0, 1, 0, 0]
            w0 = 1.0 / (1.0 + math.exp(s1 - s0))
            w1 = 1.0 / (1.0 + math.exp(s0 - s1))
            assert abs(out[0, i, 0, 0] - (w0 * v[0, 0, 0, 0] + w1 * v[0, 1, 0, 0])) < 1e-13
            assert abs(lse[0, 0, i] - (max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))))) < 1e-13


def _golden_value(x):
    if isinstance(x, str):
        return eval(x, {"__builtins__": {}}, {"ln": math.log, "exp": math.exp})
    return float(x)


def _golden_array(nested):
    if isinstance(nested, list):
        return np.array([_golden_array(e) for e in nested], dtype=np.float64)
    return _golden_value(nested)


def test_golden_closed_form_cases(oracle_mod):
    with open(os.path.join(HERE, "golden", "closed_form_cases.json")) as f:
        cases = json.load(f)["cases"]
    assert len(cases) >= 5
    for c in cases:
        q, k, v = _golden_array(c["q"]), _golden_array(c["k"]), _golden_array(c["v"])
        assert q.shape == (c["B"], c["S"], c["H"], c["D"]), c["name"]
        assert k.shape == (c["B"], c["S"], c["Hkv"], c["D"]), c["name"]
        out, lse = oracle_mod.mha_forward(q, k, v, _golden_value(c["scale"]),
                                          c["causal"], c["window"])
        np.testing.assert_allclose(out, _golden_array(c["out"]), atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(lse, _golden_array(c["lse"]), atol=1e-12, err_msg=c["name"])


# --- invariants ---------------------------------------------------------------

@pytest.mark.parametrize("causal,window", MASKS)
def test_grouped_equals_explicit_repeat(oracle_mod, causal, window):
    """Grouped attention equals ordinary attention with each KV head repeated
    G times consecutively (query head h reads KV head h // G)."""
    B, S, H, Hkv, D = 2, 21, 6, 2, 8
    q = _rand((B, S, H, D), 16)
    k, v = _rand((B, S, Hkv, D), 17), _rand((B, S, Hkv, D), 18)
    out, lse = oracle_mod.mha_forward(q, k, v, 0.3, causal, window)
    G = H // Hkv
    kr, vr = np.repeat(k, G, axis=2), np.repeat(v, G, axis=2)
    out2, lse2 = oracle_mod.mha_forward(q, kr, vr, 0.3, causal, window)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)
    # The repeated form is not what a tiled head map (h % Hkv) computes.
    out3, _ = oracle_mod.mha_forward(q, k, v, 0.3, causal, window,
                                     head_map=oracle_mod.HEAD_MAP_TILED)
    assert np.abs(out3 - out).max() > 1e-3


def test_tiled_head_map_is_a_head_permutation(oracle_mod):
    """The two readings of the grouped head map differ only by a permutation
    of the query-head axis: tiled(q) == perm^-1(grouped(perm(q)))."""
    B, S, H, Hkv, D = 1, 13, 6, 3, 4
    G = H // Hkv
    q = _rand((B, S, H, D), 19)
    k, v = _rand((B, S, Hkv, D), 20), _rand((B, S, Hkv, D), 21)
    tiled, _ = oracle_mod.mha_forward(q, k, v, 0.8, True, -1,
                                      head_map=oracle_mod.HEAD_MAP_TILED)
    # grouped head g*G + r reads KV head g; tiled head r*Hkv + g reads KV head g.
    perm = np.array([(h % G) * Hkv + h // G for h in range(H)])  # grouped slot -> tiled head
    grouped, _ = oracle_mod.mha_forward(q[:, :, perm], k, v, 0.8, True, -1)
    back = np.empty_like(grouped)
    back[:, :, perm] = grouped
    np.testing.assert_allclose(back, tiled, atol=1e-14)


@pytest.mark.parametrize("causal,window", MASKS)
def test_key_shift_invariance(oracle_mod, causal, window):
    """Adding one vector c to every key row shifts every score of a query row
    by scale*q.c, which softmax removes: O is unchanged, lse shifts."""
    B, S, H, D = 1, 17, 2, 6
    q, k, v = _rand((B, S, H, D), 22), _rand((B, S, H, D), 23), _rand((B, S, H, D), 24)
    c = _rand((1, 1, H, D), 25)
    out, lse = oracle_mod.mha_forward(q, k, v, 0.6, causal, window)
    out2, lse2 = oracle_mod.mha_forward(q, k + c, v, 0.6, causal, window)
    np.testing.assert_allclose(out2, out, atol=1e-12)
    shift = 0.6 * np.einsum("bshd,hd->bhs", q, c[0, 0])
    np.testing.assert_allclose(lse2, lse + shift, atol=1e-12)


def test_key_permutation_invariance_without_mask(oracle_mod):
    B, S, H, D = 2, 15, 2, 4
    q, k, v = _rand((B, S, H, D), 26), _rand((B, S, H, D), 27), _rand((B, S, H, D), 28)
    perm = np.random.default_rng(29).permutation(S)
    out, lse = oracle_mod.mha_forward(q, k, v, 0.9, False, -1)
    out2, lse2 = oracle_mod.mha_forward(q, k[:, perm], v[:, perm], 0.9, False, -1)
    np.testing.assert_allclose(out2, out, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, atol=1e-13)


def test_rows_subset_matches_full(oracle_mod):
    B, S, H, Hkv, D = 2, 40, 4, 2, 8
    q = _rand((B, S, H, D), 30)
    k, v = _rand((B, S, Hkv, D), 31), _rand((B, S, Hkv, D), 32)
    out, lse = oracle_mod.mha_forward(q, k, v, 0.4, True, 7)
    rows = [0, 5, 6, 39, 17]
    o2, l2 = oracle_mod.mha_forward(q[:, rows], k, v, 0.4, True, 7, rows=rows)
    np.testing.assert_array_equal(o2, out[:, rows])
    np.testing.assert_array_equal(l2, lse[:, :, rows])


def test_thread_count_does_not_change_results(oracle_mod):
    B, S, H, D = 1, 33, 4, 8
    q, k, v = _rand((B, S, H, D), 33), _rand((B, S, H, D), 34), _rand((B, S, H, D), 35)
    a = oracle_mod.mha_forward(q, k, v, 0.5, True, -1, nthreads=1)
    b = oracle_mod.mha_forward(q, k, v, 0.5, True, -1, nthreads=7)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_rejects_bad_arguments(oracle_mod):
    q = np.zeros((1, 4, 3, 2))
    k = np.zeros((1, 4, 2, 2))
    with pytest.raises(ValueError):  # H % Hkv != 0
        oracle_mod.mha_forward(q, k, k, 1.0)
    with pytest.raises(ValueError):  # row out of range
        oracle_mod.mha_forward(q[:, :1], q, q, 1.0, rows=[4])


# --- independent blockwise online-softmax recomputation ------------------------

def _visible_matrix(S, causal, window):
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    vis = np.ones((S, S), dtype=bool)
    if causal:
        vis &= j <= i
    if window > 0:
        vis &= (i - j) < window
        if not causal:
            vis &= (j - i) < window
    return vis


def _blockwise_fa2(q, k, v, scale, vis, block_q, block_k):
    """FlashAttention-2 ordering (Q blocks outer, KV blocks inner) with a running
    max m, running sum l, unnormalised O rescaled by exp(m_old - m_new), and a
    single division by l at the end, as in the flash_attn_v2 loop of the
    tiny_flash_attn.py page (here with the scale and a mask added)."""
    S, D = q.shape
    out = np.zeros((S, D))
    lse = np.zeros(S)
    for q0 in range(0, S, block_q):
        qb = q[q0:q0 + block_q]
        n = qb.shape[0]
        m = np.full(n, -np.inf)
        l = np.zeros(n)
        o = np.zeros((n, D))
        for k0 in range(0, S, block_k):
            s = scale * (qb @ k[k0:k0 + block_k].T)
            s = np.where(vis[q0:q0 + n, k0:k0 + block_k], s, -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            base = np.where(np.isneginf(m_new), 0.0, m_new)  # fully hidden rows so far
            p = np.exp(s - base[:, None])
            alpha = np.exp(np.where(np.isneginf(m), -np.inf, m - base))
            l = alpha * l + p.sum(axis=1)
            o = alpha[:, None] * o + p @ v[k0:k0 + block_k]
            m = m_new
        out[q0:q0 + n] = o / l[:, None]
        lse[q0:q0 + n] = m + np.log(l)
    return out, lse


def _blockwise_normalise_each_step(q, k, v, scale, vis, block_q, block_k):
    """Normalise-every-step variant of the Modular recipe's kernel listing:
    O <- O * (l_old / l_new) * exp(m_old - m_new) + (P / l_new) V each KV tile."""
    S, D = q.shape
    out = np.zeros((S, D))
    for q0 in range(0, S, block_q):
        qb = q[q0:q0 + block_q]
        n = qb.shape[0]
        m = np.full(n, -np.inf)
        l = np.zeros(n)
        o = np.zeros((n, D))
        for k0 in range(0, S, block_k):
            s = scale * (qb @ k[k0:k0 + block_k].T)
            s = np.where(vis[q0:q0 + n, k0:k0 + block_k], s, -np.inf)
            m_new = np.maximum(m, s.max(axis=1))
            live = ~np.isneginf(m_new)
            base = np.where(live, m_new, 0.0)
            e = np.exp(s - base[:, None])
            decay = np.exp(np.where(np.isneginf(m), -np.inf, m - base))
            l_new = decay * l + e.sum(axis=1)
            safe = np.where(l_new > 0, l_new, 1.0)
            o = np.where(live[:, None],
                         o * (l / safe * decay)[:, None] + (e / safe[:, None]) @ v[k0:k0 + block_k],
                         o)
            m, l = m_new, l_new
        out[q0:q0 + n] = o
    return out


@pytest.mark.parametrize("block", [1, 3, 4, 16])
@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (True, 3), (True, 10),
                                           (False, 4)])
def test_blockwise_online_softmax_agrees(oracle_mod, block, causal, window):
    B, S, H, Hkv, D = 1, 29, 4, 2, 8
    q = _rand((B, S, H, D), 40, 2.0)
    k, v = _rand((B, S, Hkv, D), 41, 2.0), _rand((B, S, Hkv, D), 42)
    scale = 1 / math.sqrt(D)
    out, lse = oracle_mod.mha_forward(q, k, v, scale, causal, window)
    vis = _visible_matrix(S, causal, window)
    for h in range(H):
        hk = h // (H // Hkv)
        o1, l1 = _blockwise_fa2(q[0, :, h], k[0, :, hk], v[0, :, hk], scale, vis, block, block + 2)
        o2 = _blockwise_normalise_each_step(q[0, :, h], k[0, :, hk], v[0, :, hk], scale, vis,
                                            block + 1, block)
        np.testing.assert_allclose(o1, out[0, :, h], atol=1e-12)
        np.testing.assert_allclose(l1, lse[0, h], atol=1e-12)
        np.testing.assert_allclose(o2, out[0, :, h], atol=1e-12)


# --- library special case --------------------------------------------------------

@pytest.mark.parametrize("causal,window", [(False, -1), (True, -1), (True, 1), (True, 6),
                                           (False, 5)])
@pytest.mark.parametrize("Hkv", [4, 2, 1])
def test_matches_torch_sdpa_fp64(oracle_mod, causal, window, Hkv):
    B, S, H, D = 2, 31, 4, 16
    q = _rand((B, S, H, D), 50)
    k, v = _rand((B, S, Hkv, D), 51), _rand((B, S, Hkv, D), 52)
    scale = 0.2
    out, lse = oracle_mod.mha_forward(q, k, v, scale, causal, window)
    G = H // Hkv
    tq = torch.from_numpy(q).permute(0, 2, 1, 3)  # BHSD
    tk = torch.from_numpy(np.repeat(k, G, axis=2)).permute(0, 2, 1, 3)
    tv = torch.from_numpy(np.repeat(v, G, axis=2)).permute(0, 2, 1, 3)
    if window > 0:
        mask = torch.from_numpy(_visible_matrix(S, causal, window))
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                                               scale=scale)
    else:
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                               scale=scale)
    np.testing.assert_allclose(out, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12)
    scores = scale * (tq @ tk.transpose(-1, -2))
    scores = scores.masked_fill(~torch.from_numpy(_visible_matrix(S, causal, window)), -math.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(scores, dim=-1).numpy(), atol=1e-12)
