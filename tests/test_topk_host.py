"""Host logic of the top-K entry points, without a GPU: the work plan and the
argument checks that run before any CUDA call."""
import ctypes

import pytest

import attention_fa2_forward_gb300 as fa


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load_library()


@pytest.mark.parametrize("B,V,K", [(64, 131072, 50), (1, 131072, 50), (1, 1000, 1000),
                                   (300, 32000, 8), (2, 5, 3), (7, 1 << 20, 1024)])
def test_plan_bounds(lib, B, V, K):
    chunks, ws = fa.topk_plan(B, V, K, num_sms=152)
    assert chunks >= 1
    chunk = -(-V // chunks)
    assert chunks * K <= max(4096, K)          # the merge's candidates
    # one chunk, or a cluster of 2, 4 or 8 (K <= 128): no candidates kept
    clustered = chunks == 1 or (chunks in (2, 4, 8) and K <= 128)
    assert ws == (0 if clustered else B * chunks * K * 8)
    # every chunk but the last is a whole number of 2048-element steps
    step_chunk = -(-(-(-V // chunks)) // 2048) * 2048
    assert -(-V // step_chunk) == chunks
    assert chunk <= step_chunk


@pytest.mark.parametrize("B", [1, 7, 64, 100, 152, 256, 303, 304, 305, 4096])
def test_plan_stays_within_one_wave(lib, B):
    """Chunk CTAs (two resident per SM) fit one wave whenever the rows do."""
    chunks, _ = fa.topk_plan(B, 1 << 18, 50, num_sms=152)
    if B <= 304:
        # at most the requested count (whole 2048-element steps can leave fewer)
        assert chunks <= min(304 // B, 4096 // 50)
        assert chunks >= min(304 // B, 4096 // 50) // 2
    else:
        assert chunks == 1


def test_plan_fills_the_gpu_for_small_batches(lib):
    chunks, _ = fa.topk_plan(8, 1 << 20, 16, num_sms=152)
    assert chunks >= 34  # about two CTAs per SM over 8 rows (chunks round up to 2048)


P = 0x10000  # a non-null fake address: never dereferenced


def _call(lib, values=P, indices=P, scores=P, B=2, V=100, stride=100, K=5, ws=P, ws_bytes=1 << 20):
    return lib.fa_topk(values, indices, scores, B, V, stride, K, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(values=None), fa.FA_ERR_INVALID_ARG),
    (dict(scores=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(V=0), fa.FA_ERR_INVALID_ARG),
    (dict(K=0), fa.FA_ERR_INVALID_ARG),
    (dict(K=101), fa.FA_ERR_INVALID_ARG),
    (dict(V=5000, stride=5000, K=1025), fa.FA_ERR_UNSUPPORTED),
    (dict(stride=99), fa.FA_ERR_INVALID_ARG),
    (dict(B=70000), fa.FA_ERR_UNSUPPORTED),
    (dict(scores=P + 2), fa.FA_ERR_UNSUPPORTED),
    (dict(ws=P + 4), fa.FA_ERR_UNSUPPORTED),
])
def test_topk_argument_validation_happens_before_cuda(lib, kw, code):
    assert _call(lib, **kw) == code
    assert lib.fa_last_error_message()


def test_topk_plan_rejects_bad_arguments(lib):
    c, w = ctypes.c_int(0), ctypes.c_ulonglong(0)
    assert lib.fa_topk_plan(1, 10, 11, 152, ctypes.byref(c), ctypes.byref(w)) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_topk_plan(1, 10, 3, -1, ctypes.byref(c), ctypes.byref(w)) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_topk_plan(1, 10, 3, 152, None, ctypes.byref(w)) == fa.FA_ERR_INVALID_ARG
