"""Pins for the KV-cache form of the fp64 oracle (``mha_forward_kvcache``).

The pages define only the no-cache operator; the cached form read here is the
same operator with the Sq queries being the last tokens of a sequence whose
L_b keys and values sit at the start of a cache (query row r at position
L_b - Sq + r). Each check is independent of the oracle's code: torch's fp64
scaled_dot_product_attention on the sliced cache with an end-aligned mask
built from ``torch.tril`` diagonals, closed-form window means, values planted
past the cache length that must never be read, a hand-written split-KV
recombination (partial softmax per key chunk, merged by log-sum-exp weights),
and the already-pinned no-cache form on the full sequence.
"""
import math

import numpy as np
import pytest
import torch

MASKS = [(False, -1), (True, -1), (True, 1), (True, 4), (True, 9), (False, 2), (False, 7)]


def _rand(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal(shape) * scale


def _end_aligned_mask(Sq, L, causal, window):
    """Boolean [Sq, L] mask for queries at positions L - Sq .. L - 1, built
    from lower-triangular bands (torch.tril with a diagonal offset)."""
    ones = torch.ones(Sq, L, dtype=torch.bool)
    shift = L - Sq  # query row r sits at position shift + r
    if causal:
        vis = ones.tril(shift)
        if window > 0:
            vis = vis & ~ones.tril(shift - window)
    else:
        vis = ones.clone()
        if window > 0:
            vis = ones.tril(shift + window - 1) & ~ones.tril(shift - window)
    return vis


def _sdpa_reference(q, k, v, lens, scale, causal, window):
    """fp64 torch SDPA per batch on k[:L], v[:L] with the explicit mask; rows
    with no visible key are defined as out 0, lse -inf."""
    B, Sq, H, D = q.shape
    Hkv = k.shape[2]
    G = H // Hkv
    out = np.zeros((B, Sq, H, D))
    lse = np.full((B, H, Sq), -np.inf)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        qb = torch.from_numpy(q[b]).permute(1, 0, 2)  # [H, Sq, D]
        kb = torch.from_numpy(k[b, :L]).permute(1, 0, 2).repeat_interleave(G, dim=0)
        vb = torch.from_numpy(v[b, :L]).permute(1, 0, 2).repeat_interleave(G, dim=0)
        mask = _end_aligned_mask(Sq, L, causal, window)
        live = mask.any(dim=1)
        if live.any():
            o = torch.nn.functional.scaled_dot_product_attention(
                qb[:, live], kb, vb, attn_mask=mask[live], scale=scale)
            out[b][live.numpy()] = o.permute(1, 0, 2).numpy()
            s = (qb[:, live] @ kb.transpose(1, 2)) * scale
            s = s.masked_fill(~mask[live], float("-inf"))
            lse[b][:, live.numpy()] = torch.logsumexp(s, dim=-1).numpy()
    return out, lse


@pytest.mark.parametrize("causal,window", MASKS)
@pytest.mark.parametrize("Sq", [1, 3, 12])
def test_matches_torch_sdpa_on_sliced_cache(oracle_mod, causal, window, Sq):
    B, S_cache, H, Hkv, D = 3, 40, 4, 2, 8
    lens = [40, 17, 12 if Sq <= 12 else Sq]
    q = _rand((B, Sq, H, D), 11)
    k = _rand((B, S_cache, Hkv, D), 12)
    v = _rand((B, S_cache, Hkv, D), 13)
    out, lse = oracle_mod.mha_forward_kvcache(q, k, v, 0.41, lens, causal, window)
    ref_out, ref_lse = _sdpa_reference(q, k, v, lens, 0.41, causal, window)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal,window", MASKS)
def test_identical_keys_average_visible_values(oracle_mod, causal, window):
    """All keys equal: O = mean of the V rows visible at the query's position
    (keys max(0, p - W + 1) .. p for a causal window, .. min(p + W - 1, L - 1)
    for a two-sided one), lse = scale*q.k + ln(count)."""
    B, Sq, S_cache, H, D = 2, 4, 30, 2, 4
    lens = [30, 9]
    scale = 0.53
    q = _rand((B, Sq, H, D), 21)
    krow = _rand((1, 1, H, D), 22)
    k = np.broadcast_to(krow, (B, S_cache, H, D)).copy()
    v = _rand((B, S_cache, H, D), 23)
    out, lse = oracle_mod.mha_forward_kvcache(q, k, v, scale, lens, causal, window)
    for b in range(B):
        L = lens[b]
        for r in range(Sq):
            p = L - Sq + r
            lo, hi = 0, (p if causal else L - 1)
            if window > 0:
                lo = max(0, p - window + 1)
                if not causal:
                    hi = min(L - 1, p + window - 1)
            n = hi - lo + 1
            for h in range(H):
                np.testing.assert_allclose(out[b, r, h], v[b, lo:hi + 1, h].mean(axis=0),
                                           rtol=0, atol=1e-13)
                s = scale * float(q[b, r, h] @ krow[0, 0, h])
                assert abs(lse[b, h, r] - (s + math.log(n))) < 1e-12


def test_last_query_of_full_cache_sees_every_key(oracle_mod):
    """Sq = 1 at the end of a full cache with the causal mask: every key is
    visible, so the result is the unmasked softmax average (hand-written)."""
    S, D = 11, 5
    q = _rand((1, 1, 1, D), 31)
    k = _rand((1, S, 1, D), 32)
    v = _rand((1, S, 1, D), 33)
    out, lse = oracle_mod.mha_forward_kvcache(q, k, v, 0.8, None, True, -1)
    s = 0.8 * (k[0, :, 0] @ q[0, 0, 0])
    w = np.exp(s - s.max())
    np.testing.assert_allclose(out[0, 0, 0], (w[:, None] * v[0, :, 0]).sum(0) / w.sum(),
                               rtol=0, atol=1e-14)
    assert abs(lse[0, 0, 0] - (s.max() + math.log(w.sum()))) < 1e-13


@pytest.mark.parametrize("causal,window", MASKS)
def test_never_reads_past_the_cache_length(oracle_mod, causal, window):
    """Rows at or beyond L_b are not part of the sequence: NaN planted there
    changes nothing."""
    B, Sq, S_cache, H, D = 2, 3, 25, 2, 4
    lens = [14, 25]
    q = _rand((B, Sq, H, D), 41)
    k = _rand((B, S_cache, H, D), 42)
    v = _rand((B, S_cache, H, D), 43)
    kn, vn = k.copy(), v.copy()
    kn[0, 14:] = np.nan
    vn[0, 14:] = np.nan
    a = oracle_mod.mha_forward_kvcache(q, k, v, 0.6, lens, causal, window)
    b = oracle_mod.mha_forward_kvcache(q, kn, vn, 0.6, lens, causal, window)
    for x, y in zip(a, b):
        assert np.isfinite(y).all()
        np.testing.assert_array_equal(x, y)


def test_queries_before_the_sequence_start_see_nothing(oracle_mod):
    """Causal, L_b < Sq: rows at negative positions have no visible key
    (out 0, lse -inf); the others see keys 0 .. p. L_b = 0 hides everything
    under every mask."""
    B, Sq, S_cache, H, D = 2, 5, 8, 2, 4
    q = _rand((B, Sq, H, D), 51)
    k = _rand((B, S_cache, H, D), 52)
    v = _rand((B, S_cache, H, D), 53)
    out, lse = oracle_mod.mha_forward_kvcache(q, k, v, 0.5, [3, 0], True, -1)
    # batch 0: positions -2, -1, 0, 1, 2
    assert np.all(out[0, :2] == 0) and np.all(lse[0, :, :2] == -np.inf)
    np.testing.assert_allclose(out[0, 2], v[0, 0], rtol=0, atol=1e-15)
    assert np.all(out[1] == 0) and np.all(lse[1] == -np.inf)
    for causal, window in [(False, -1), (False, 3)]:
        o2, l2 = oracle_mod.mha_forward_kvcache(q, k, v, 0.5, [3, 0], causal, window)
        assert np.all(o2[1] == 0) and np.all(l2[1] == -np.inf)
        assert np.isfinite(o2[0]).all()


@pytest.mark.parametrize("causal,window", [(True, -1), (False, -1), (True, 5), (False, 4)])
def test_full_cache_equals_last_rows_of_no_cache(oracle_mod, causal, window):
    """With L_b = S_cache the cached form is the no-cache operator's last Sq
    rows on the whole sequence (the no-cache form is pinned on its own)."""
    B, S, Sq, H, Hkv, D = 2, 19, 6, 4, 2, 8
    q_full = _rand((B, S, H, D), 61)
    k = _rand((B, S, Hkv, D), 62)
    v = _rand((B, S, Hkv, D), 63)
    full_out, full_lse = oracle_mod.mha_forward(q_full, k, v, 0.35, causal, window)
    out, lse = oracle_mod.mha_forward_kvcache(q_full[:, S - Sq:], k, v, 0.35, None, causal,
                                              window)
    np.testing.assert_allclose(out, full_out[:, S - Sq:], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, full_lse[:, :, S - Sq:], rtol=0, atol=1e-15)


def _split_kv_recombined(q, k, v, L, scale, vis, chunk):
    """One (b, h) slice: partial softmax over each chunk of keys, then the
    chunks merged with weights exp(lse_c - lse). q [Sq, D], k/v [L, D]."""
    Sq = q.shape[0]
    parts = []
    for a in range(0, L, chunk):
        e = min(L, a + chunk)
        s = scale * (q @ k[a:e].T)
        s = np.where(vis[:, a:e], s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        m_safe = np.where(np.isfinite(m), m, 0.0)
        w = np.exp(s - m_safe)
        den = w.sum(axis=1, keepdims=True)
        o = np.where(den > 0, (w @ v[a:e]) / np.where(den > 0, den, 1.0), 0.0)
        lse_c = np.where(den[:, 0] > 0, m_safe[:, 0] + np.log(np.where(den[:, 0] > 0,
                                                                      den[:, 0], 1.0)), -np.inf)
        parts.append((o, lse_c))
    lses = np.stack([p[1] for p in parts])  # [chunks, Sq]
    top = lses.max(axis=0)
    top_safe = np.where(np.isfinite(top), top, 0.0)
    wts = np.exp(lses - top_safe)
    tot = wts.sum(axis=0)
    out = sum(wts[c][:, None] * parts[c][0] for c in range(len(parts)))
    out = np.where(tot[:, None] > 0, out / np.where(tot > 0, tot, 1.0)[:, None], 0.0)
    lse = np.where(tot > 0, top_safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    return out, lse


@pytest.mark.parametrize("chunk", [1, 4, 7, 64])
@pytest.mark.parametrize("causal,window", [(True, -1), (True, 6), (False, -1), (False, 5)])
def test_split_kv_recombination_agrees(oracle_mod, chunk, causal, window):
    B, Sq, S_cache, H, D = 2, 3, 33, 2, 6
    lens = [33, 20]
    q = _rand((B, Sq, H, D), 71)
    k = _rand((B, S_cache, H, D), 72)
    v = _rand((B, S_cache, H, D), 73)
    out, lse = oracle_mod.mha_forward_kvcache(q, k, v, 0.45, lens, causal, window)
    for b in range(B):
        L = lens[b]
        vis = _end_aligned_mask(Sq, L, causal, window).numpy()
        for h in range(H):
            o, l = _split_kv_recombined(q[b, :, h], k[b, :L, h], v[b, :L, h], L, 0.45, vis, chunk)
            np.testing.assert_allclose(out[b, :, h], o, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b, h], l, rtol=0, atol=1e-12)


def test_rejects_bad_lengths(oracle_mod):
    q = np.zeros((2, 1, 2, 4))
    k = np.zeros((2, 8, 2, 4))
    with pytest.raises(ValueError):
        oracle_mod.mha_forward_kvcache(q, k, k, 1.0, [9, 1])
    with pytest.raises(ValueError):
        oracle_mod.mha_forward_kvcache(q, k, k, 1.0, [-1, 1])
    with pytest.raises(ValueError):
        oracle_mod.mha_forward_kvcache(q, k, k, 1.0, [1])
