"""Host logic of the KV-cache entry points, without a GPU: the work plan
(split count, workspace size) and the argument checks that run before any
CUDA call."""
import ctypes

import pytest

import attention_fa2_forward_gb300 as fa


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load_library()


def _plan(*a, **kw):
    kw.setdefault("num_sms", 152)
    return fa.kv_cache_plan(*a, **kw)


def _tiles(S):
    return (S + 127) // 128


def _expected_splits(req, tiles):
    """Splits after evening out: every split takes ceil(tiles / req) tiles."""
    req = min(req, 128, tiles)
    per = -(-tiles // req)
    return -(-tiles // per)


def _ws(slots, R, d_pad=128):
    """Workspace of `slots` partial slots of R rows: fp32 O rows, then LSEs."""
    return ((slots * R * d_pad * 4 + 255) // 256 * 256) + ((slots * R * 4 + 255) // 256 * 256)


def _auto(units, tiles, R, Hkv, sms=152):
    """The automatic plan: units that fill half the SMs (or caches of at most
    two tiles) run whole; fewer are shared out stream-K fashion over groups of
    Hkv CTAs (27/32 x SMs CTAs in all), a unit cut into at most one piece per
    CTA group; one partial slot per unit plus one per CTA."""
    if 2 * units >= sms or tiles <= 2:
        return 1, 0
    ctas = max(Hkv, 27 * sms // 32 // Hkv * Hkv)
    return max(2, min(ctas // Hkv, tiles)), _ws(units + ctas, R)


def test_auto_plan_of_the_decode_workloads():
    # one 131072-key sequence x 8 KV heads (G = 4, one position: R = 4 rows);
    # a ragged batch of 8 x 8 KV heads, 4 positions (R = 16): both stream-K
    # over 128 CTAs in 16 groups of 8 (one per KV head)
    assert _plan(1, 1, 131072, 32, 8, 128) == (16, _ws(8 + 128, 4))
    assert _plan(8, 4, 32768, 32, 8, 128) == (16, _ws(64 + 128, 16))
    assert _plan(1, 1, 131072, 32, 8, 128, num_sms=76) == (8, _ws(8 + 64, 4))
    assert _plan(1, 1, 131072, 24, 3, 128) == _auto(3, 1024, 8, 3)  # 126 CTAs


def test_enough_units_take_one_split():
    # 16 batches x 8 KV heads = 128 units: one split, no workspace; 76 units
    # (half of 152 SMs) still one.
    assert _plan(16, 1, 8192, 32, 8, 128) == (1, 0)
    assert _plan(19, 1, 8192, 16, 4, 128) == (1, 0)
    assert _plan(37, 1, 8192, 8, 2, 128)[0] > 1
    # caches of two tiles or fewer are not shared out
    assert _plan(1, 1, 256, 8, 2, 128) == (1, 0)


@pytest.mark.parametrize("B,Hkv,S", [(1, 8, 131072), (2, 8, 32768), (1, 1, 65536), (4, 4, 8192),
                                     (8, 8, 32768)])
def test_few_units_are_shared_out(B, Hkv, S):
    assert _plan(B, 1, S, 8 * Hkv, Hkv, 128) == _auto(B * Hkv, _tiles(S), 8, Hkv)


@pytest.mark.parametrize("req", [1, 2, 3, 7, 64, 200])
def test_requested_splits_are_capped_and_cover_every_tile(req):
    S = 5000
    splits, ws = _plan(1, 1, S, 8, 2, 128, num_splits=req)
    tiles = _tiles(S)
    assert 1 <= splits <= min(req, 128, tiles)
    assert splits == _expected_splits(req, tiles)  # no trailing split without tiles
    # one slot of R = 4 rows per (unit, split)
    assert ws == (0 if splits == 1 else _ws(2 * splits, 4))


def test_window_bounds_the_tiles_to_split():
    # A causal window of 4096 keys spans at most 33 tiles of 128 keys.
    splits, _ = _plan(1, 1, 131072, 32, 8, 128, "causal", 4096)
    assert splits <= 33
    splits_none, _ = _plan(1, 1, 131072, 32, 8, 128, "none", 4096)
    assert splits_none <= 65


def test_more_groups_than_an_item_list_holds_take_fixed_splits():
    # 100 batches x 1 KV head on a 400-SM device: 100 units, fewer than half
    # the SMs, but 100 position-tile groups exceed the 80 items a CTA's list
    # holds, so the plan falls back to even splits (about two CTAs per SM:
    # ceil(800 / 100) = 8)
    splits, ws = _plan(100, 1, 8192, 8, 1, 128, num_sms=400)
    assert splits == _expected_splits(8, 64)
    assert ws == _ws(100 * splits, 8)


def test_position_tiles_count_as_units():
    # Sq = 64 with 4 heads per KV head: 2 position tiles of 32 positions
    # (R = 128 rows); Sq = 32: one.
    assert _plan(1, 64, 16384, 8, 2, 128) == _auto(4, 128, 128, 2)
    assert _plan(1, 32, 16384, 8, 2, 128) == _auto(2, 128, 128, 2)
    # 40 batches x 2 KV heads x 2 position tiles fill half of 152 SMs
    assert _plan(40, 64, 16384, 8, 2, 128) == (1, 0)


P = 0x10000  # a non-null, 16-byte aligned fake address: never dereferenced


def _call(lib, out=P, q=P, k=P, v=P, lens=None, B=1, Sq=1, S=256, H=8, Hkv=2, D=128,
          scale=0.1, mask=1, window=-1, splits=0, ws=None, ws_bytes=0, dtype=0, lse=None):
    return lib.fa_mha_kv_cache(out, lse, q, k, v, lens, B, Sq, S, H, Hkv, D, scale, mask, window,
                               splits, ws, ws_bytes, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(k=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Sq=0), fa.FA_ERR_INVALID_ARG),
    (dict(S=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=6, Hkv=4), fa.FA_ERR_INVALID_ARG),
    (dict(mask=3), fa.FA_ERR_INVALID_ARG),
    (dict(window=0), fa.FA_ERR_INVALID_ARG),
    (dict(splits=-1), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-0.5), fa.FA_ERR_UNSUPPORTED),
    (dict(D=100), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=1), fa.FA_ERR_UNSUPPORTED),
    (dict(H=258, Hkv=1), fa.FA_ERR_UNSUPPORTED),  # more than 128 query heads per KV head
    (dict(q=P + 8), fa.FA_ERR_UNSUPPORTED),
    (dict(lens=P + 2), fa.FA_ERR_UNSUPPORTED),
    (dict(S=1 << 30, Hkv=64, H=64), fa.FA_ERR_UNSUPPORTED),
])
def test_kv_cache_argument_validation_happens_before_cuda(lib, kw, code):
    assert _call(lib, **kw) == code
    assert lib.fa_last_error_message()


def test_plan_rejects_bad_arguments(lib):
    s, w = ctypes.c_int(0), ctypes.c_ulonglong(0)
    assert lib.fa_mha_kv_cache_plan(1, 1, 256, 8, 2, 128, 1, -1, 0, 152, None,
                                    ctypes.byref(w)) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_mha_kv_cache_plan(1, 1, 256, 8, 2, 128, 1, -1, 0, -1, ctypes.byref(s),
                                    ctypes.byref(w)) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_mha_kv_cache_plan(1, 1, 256, 8, 2, 64, 1, -1, 0, 152, ctypes.byref(s),
                                    ctypes.byref(w)) == fa.FA_OK
    assert s.value == 1 and w.value == 0 or s.value > 1
