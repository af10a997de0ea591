"""The C-ABI library loads without a GPU, exports every symbol the header
declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import attention_fa2_forward_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_mha.h")


@pytest.fixture(scope="module")
def lib():
    fa.build()
    return fa.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert _declared_functions() == sorted(fa.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_status_strings(lib):
    assert fa.version() == 100
    assert lib.fa_status_string(0) == b"FA_OK"
    assert lib.fa_status_string(4) == b"FA_ERR_TIMEOUT"
    assert lib.fa_status_string(99) == b"FA_ERR_UNKNOWN"


def test_wait_timeout_setting_roundtrip(lib):
    old = fa.set_wait_timeout_ns(12345)
    assert fa.set_wait_timeout_ns(0) == 12345
    assert fa.set_wait_timeout_ns(old) == 2_000_000_000


P = 0x10000  # a non-null, 16-byte aligned fake address: never dereferenced


def _call(lib, out=P, lse=None, q=P, k=P, v=P, B=1, S=8, H=2, Hkv=2, D=64, scale=0.125,
          mask=1, window=-1, dtype=0):
    return lib.fa_mha_no_cache(out, lse, q, k, v, B, S, H, Hkv, D, scale, mask, window, dtype,
                               None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(out=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(S=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=3, Hkv=2), fa.FA_ERR_INVALID_ARG),
    (dict(Hkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(mask=2), fa.FA_ERR_INVALID_ARG),
    (dict(window=0), fa.FA_ERR_INVALID_ARG),
    (dict(window=-2), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_UNSUPPORTED),
    (dict(D=100), fa.FA_ERR_UNSUPPORTED),
    (dict(D=264), fa.FA_ERR_UNSUPPORTED),
    (dict(D=256, H=258, Hkv=1), fa.FA_ERR_UNSUPPORTED),  # D > 128 needs H / Hkv <= 128
    (dict(D=80, dtype=1), fa.FA_ERR_UNSUPPORTED),  # fp32: D in {32, 64, 96, 128}
    (dict(dtype=7), fa.FA_ERR_UNSUPPORTED),
    (dict(q=P + 8), fa.FA_ERR_UNSUPPORTED),  # bf16 tensors need 16-byte alignment
    (dict(S=1 << 30, H=1 << 10), fa.FA_ERR_UNSUPPORTED),
])
def test_argument_validation_happens_before_cuda(lib, kw, code):
    assert _call(lib, **kw) == code
    assert lib.fa_last_error_message()  # a reason is recorded


def test_python_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 4, 2, 64)
    with pytest.raises(ValueError):
        fa.mha_no_cache(q, q, q)


def _call_strided(lib, strides=((64, 32, 16),) * 4, q=P, dtype=0, null=None):
    arr = ctypes.c_longlong * 3
    st = [arr(*s) for s in strides]
    if null is not None:
        st[null] = None
    return lib.fa_mha_no_cache_strided(P, None, q, P, P, 1, 8, 2, 2, 64, st[0], st[1], st[2],
                                       st[3], 0.125, 1, -1, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(null=0), fa.FA_ERR_INVALID_ARG),
    (dict(null=3), fa.FA_ERR_INVALID_ARG),
    (dict(strides=((64, 32, 16),) * 3 + ((64, 0, 16),)), fa.FA_ERR_INVALID_ARG),
    (dict(strides=((64, 32, -16),) + ((64, 32, 16),) * 3), fa.FA_ERR_INVALID_ARG),
    (dict(strides=((64, 36, 16),) + ((64, 32, 16),) * 3), fa.FA_ERR_UNSUPPORTED),  # bf16: 16 B
    (dict(strides=((1 << 40, 32, 16),) * 4), fa.FA_ERR_UNSUPPORTED),
])
def test_strided_validation_happens_before_cuda(lib, kw, code):
    assert _call_strided(lib, **kw) == code
    assert lib.fa_last_error_message()


def _call_f32tc(lib, out=P, q=P, k=P, v=P, B=1, S=8, H=2, Hkv=2, D=64, scale=0.125, mask=1,
                window=-1, ws=P, ws_bytes=1 << 30):
    return lib.fa_mha_no_cache_f32_tc(out, None, q, k, v, B, S, H, Hkv, D, scale, mask, window, ws,
                                      ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(H=3, Hkv=2), fa.FA_ERR_INVALID_ARG),
    (dict(window=0), fa.FA_ERR_INVALID_ARG),
    (dict(D=96), fa.FA_ERR_UNSUPPORTED),
    (dict(q=P + 4), fa.FA_ERR_UNSUPPORTED),
    (dict(ws=P + 16), fa.FA_ERR_UNSUPPORTED),
    (dict(ws_bytes=16), fa.FA_ERR_INVALID_ARG),
    (dict(ws=None), fa.FA_ERR_INVALID_ARG),
])
def test_f32_tensor_core_validation_happens_before_cuda(lib, kw, code):
    assert _call_f32tc(lib, **kw) == code
    assert lib.fa_last_error_message()


def test_f32_tensor_core_workspace_size(lib):
    # six bf16 planes of [B, S, Hkv, D] (K's and V's three parts), 256-byte rounded
    plane = 2 * 100 * 4 * 128 * 2
    assert lib.fa_mha_no_cache_f32_tc_workspace(2, 100, 4, 128) == 6 * (-(-plane // 256) * 256)
    assert lib.fa_mha_no_cache_f32_tc_workspace(2, 100, 4, 96) == 0


def test_status_string_names_the_bounds_status(lib):
    assert lib.fa_status_string(fa.FA_ERR_BOUNDS) == b"FA_ERR_BOUNDS"


def test_trace_and_guard_knobs_are_debug_only(lib):
    # The default build has no trace and no guards; turning tracing off is
    # always accepted. None of these calls touches CUDA.
    assert lib.fa_trace_bytes_per_cta() == 0
    assert lib.fa_trace_set_buffer(None, 0) == fa.FA_OK
    assert lib.fa_trace_set_buffer(P, 1 << 20) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_debug_set_lse_limit(10) == fa.FA_ERR_UNSUPPORTED


def test_trace_cta_count_follows_the_prefill_grid(lib):
    # one CTA per (query block, head, batch): blocks of 128 queries (one Q
    # tile) for head dims up to 64, else of 256 (two tiles); head dims above
    # 128 run another kernel and have no trace
    assert lib.fa_trace_ctas(4, 1024, 16, 64) == 8 * 16 * 4
    assert lib.fa_trace_ctas(4, 1025, 16, 64) == 9 * 16 * 4
    assert lib.fa_trace_ctas(1, 4096, 2, 40) == 32 * 2
    assert lib.fa_trace_ctas(4, 1024, 16, 72) == 4 * 16 * 4
    assert lib.fa_trace_ctas(2, 4097, 32, 128) == 17 * 32 * 2
    assert lib.fa_trace_ctas(1, 1, 1, 8) == 1
    assert lib.fa_trace_ctas(1, 100, 2, 256) == 0
    assert lib.fa_trace_ctas(0, 100, 2, 64) == 0


def test_debug_build_exports_the_same_symbols_and_traces():
    dbg = fa.load_debug_library()
    for name in _declared_functions():
        assert hasattr(dbg, name), name
    assert dbg.fa_trace_bytes_per_cta() == 10 * 256 * 16
    assert dbg.fa_trace_set_buffer(P + 8, 1 << 20) == fa.FA_ERR_INVALID_ARG  # 16-byte aligned
    assert dbg.fa_debug_set_lse_limit(-1) == fa.FA_ERR_INVALID_ARG
    assert dbg.fa_debug_set_lse_limit(0) == fa.FA_OK
    assert dbg.fa_trace_set_buffer(None, 0) == fa.FA_OK


def _call_host(lib, out=P, q=P, k=P, v=P, B=1, S=8, H=2, Hkv=2, D=64, ws=P, ws_bytes=1 << 30,
               dtype=0, window=-1):
    return lib.fa_mha_no_cache_host(out, None, q, k, v, B, S, H, Hkv, D, 0.125, 1, window, dtype,
                                    ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), fa.FA_ERR_INVALID_ARG),
    (dict(ws=None), fa.FA_ERR_INVALID_ARG),
    (dict(ws=P + 16), fa.FA_ERR_INVALID_ARG),       # 256-byte aligned workspace
    (dict(ws_bytes=1024), fa.FA_ERR_INVALID_ARG),   # too small
    (dict(H=3, Hkv=2), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(window=0), fa.FA_ERR_INVALID_ARG),
    (dict(D=100), fa.FA_ERR_UNSUPPORTED),
    (dict(dtype=5), fa.FA_ERR_UNSUPPORTED),
])
def test_host_entry_point_checks_everything_before_copying(lib, kw, code):
    assert _call_host(lib, **kw) == code
    assert lib.fa_last_error_message()


def test_host_entry_point_workspace_size(lib):
    def a(x):
        return -(-x // 256) * 256
    B, S, H, Hkv, D = 2, 100, 4, 2, 64
    q, kv, lse = B * S * H * D * 2, B * S * Hkv * D * 2, B * H * S * 4
    assert lib.fa_mha_no_cache_host_workspace(B, S, H, Hkv, D, 0) == \
        a(a(a(a(q) + kv) + kv) + q) + a(lse)
    # fp32 at D 64 / 128 also holds the six bf16 planes of K and V
    q4, kv4 = 2 * q, 2 * kv
    base = a(a(a(a(q4) + kv4) + kv4) + q4) + a(lse)
    assert lib.fa_mha_no_cache_host_workspace(B, S, H, Hkv, D, 1) == \
        base + lib.fa_mha_no_cache_f32_tc_workspace(B, S, Hkv, D)
    assert lib.fa_mha_no_cache_host_workspace(B, S, H, Hkv, 32, 1) == \
        a(a(a(a(q4 // 2) + kv4 // 2) + kv4 // 2) + q4 // 2) + a(lse)
    assert lib.fa_mha_no_cache_host_workspace(0, S, H, Hkv, D, 0) == 0
