"""The allocation-free entry point, fa_mha_no_cache_noalloc.

Some callers cannot call cudaMalloc (their allocator belongs to a framework
or to a pool sized in advance, or they must not allocate on a hot path). For
them the library offers an entry point whose only scratch memory is a fixed
array inside the library. This test calls it through the C ABI and checks its
output against fa_mha_no_cache on the same inputs, within the parity
tolerances of the GPU tests, on two calls in a row (the second call must see
a cleared status word, not the first call's leftovers). Both entry points run
the same kernel, so the outputs must also be equal bit for bit.

The file name makes pytest collect it last.
"""
import ctypes
import math

import pytest
import torch

import attention_fa2_forward_gb300 as fa
from attention_fa2_forward_gb300.inputs import make_qkv


def _noalloc_fn():
    lib = fa.load_library()
    fn = lib.fa_mha_no_cache_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.restype = i
    fn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float, i, i, vp, i]
    return fn


@pytest.mark.gpu
@pytest.mark.parametrize("S,H,Hkv,D,mask,window", [
    (1000, 8, 2, 128, fa.MASK_CAUSAL, -1),
    (777, 4, 4, 64, fa.MASK_NONE, -1),
    (1500, 4, 1, 128, fa.MASK_CAUSAL, 300),
])
def test_noalloc_matches_allocating_entry_point(oracle_mod, S, H, Hkv, D, mask, window):
    """Both entry points run the same kernel on the same inputs, so their
    outputs must agree bit for bit; the oracle then checks the values."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    fn = _noalloc_fn()
    dev = torch.device("cuda:0")
    B = 2
    q_h, k_h, v_h = make_qkv(B, S, H, Hkv, D, torch.bfloat16, seed=S + D)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    scale = 1.0 / math.sqrt(D)
    ref, ref_lse = fa.mha_no_cache(q, k, v, scale, mask, window, return_lse=True)
    stream = torch.cuda.current_stream(dev).cuda_stream
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device=dev)
        rc = fn(out.data_ptr(), lse.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                B, S, H, Hkv, D, scale, mask, window, stream, 1)
        assert rc == fa.FA_OK, (call, rc, fa.load_library().fa_last_error_message())
        torch.cuda.synchronize()
        assert torch.equal(out, ref), call
        assert torch.equal(lse, ref_lse), call
    o_ref, l_ref = oracle_mod.mha_forward(q_h, k_h, v_h, scale, mask == fa.MASK_CAUSAL, window)
    err = (out.double().cpu() - torch.from_numpy(o_ref)).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
    assert (lse.double().cpu() - torch.from_numpy(l_ref)).abs().max().item() <= 2e-3
    assert fa.device_status() == fa.FA_OK


@pytest.mark.gpu
def test_noalloc_without_status_check_or_lse():
    """check_status = 0 returns right after the launch; lse may be NULL."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    fn = _noalloc_fn()
    dev = torch.device("cuda:0")
    B, S, H, Hkv, D = 1, 900, 4, 2, 128
    q, k, v = (t.to(dev) for t in make_qkv(B, S, H, Hkv, D, torch.bfloat16, seed=5))
    scale = 1.0 / math.sqrt(D)
    ref = fa.mha_no_cache(q, k, v, scale, "causal")
    stream = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        rc = fn(out.data_ptr(), None, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                B, S, H, Hkv, D, scale, fa.MASK_CAUSAL, -1, stream, 0)
        assert rc == fa.FA_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref)


def test_noalloc_rejects_arguments_before_launch():
    fa.build()
    fn = _noalloc_fn()
    P = 0x10000
    assert fn(P, None, P, P, P, 1, 8, 3, 2, 64, 0.1, 1, -1, None, 0) == fa.FA_ERR_INVALID_ARG
    assert fn(P, None, P, P, P, 1, 8, 2, 2, 100, 0.1, 1, -1, None, 0) == fa.FA_ERR_UNSUPPORTED
    assert fa.load_library().fa_last_error_message()
