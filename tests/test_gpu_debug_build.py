"""The debug build (FA_TRACE=1): event trace and bounds guards of the prefill
kernel.

The trace must describe the launch the kernel actually made: every CTA
starts on a valid SM, each role's events are in time order, every Q tile sees
exactly the KV tiles its mask needs (each S MMA issued before the softmax
reads it), and the traced launch computes the same bits as the default
build. The bounds guard is exercised without an out-of-range access: a debug
knob lowers the LSE limit, the guard skips the elements past it (they keep
their poison) and the stream status reports FA_ERR_BOUNDS.
"""
import math

import pytest
import torch

import attention_fa2_forward_gb300 as fa
from attention_fa2_forward_gb300 import trace
from attention_fa2_forward_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    fa.load_debug_library()


def _kv_tiles(q0, S, causal, window):
    """KV tiles [lo, hi) a 128-row Q tile starting at q0 needs (the mask's
    visible keys, rounded out to 128-key tiles)."""
    if q0 >= S:
        return 0, 0
    if causal:
        kv_end = min(S, q0 + 128)
    elif window > 0:
        kv_end = min(S, q0 + 127 + window)
    else:
        kv_end = S
    kv_begin = max(0, q0 - window + 1) if window > 0 else 0
    return kv_begin // 128, (kv_end + 127) // 128


@pytest.mark.parametrize("B,S,H,Hkv,D,causal,window", [
    (2, 1000, 4, 2, 128, True, -1),
    (1, 1500, 4, 4, 64, False, -1),
    (2, 900, 4, 2, 64, True, -1),
    (1, 2100, 2, 1, 128, True, 300),
    (1, 700, 2, 2, 64, False, 200),
])
def test_trace_matches_the_launch(B, S, H, Hkv, D, causal, window):
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(B, S, H, Hkv, D, torch.bfloat16, seed=5 + S))
    scale = 1.0 / math.sqrt(D)
    mask = "causal" if causal else "none"
    out, lse, status, events = trace.run_traced(q, k, v, scale, mask, window)
    torch.cuda.synchronize()
    assert status == fa.FA_OK
    ref, ref_lse = fa.mha_no_cache(q, k, v, scale, mask, window, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    tiles = 1 if D <= 64 else 2  # Q tiles of 128 rows per CTA
    nqb = (S + 128 * tiles - 1) // (128 * tiles)
    assert len(events) == nqb * H * B
    eff_window = window if 0 < window < S else -1
    for e in events:
        c = e["cta"]
        assert e["sm"] is not None and 0 <= e["sm"] < sms
        for name, ev in e["roles"].items():
            times = [t for t, _, _, _ in ev]
            assert times == sorted(times), (c, name)
        qb = nqb - 1 - c // (H * B)
        s_issued = {}
        for t_ns, _, code, arg in e["roles"]["mma"]:
            if code == "s_issued":
                s_issued[(arg >> 16, arg & 0xFFFF)] = t_ns
        for t in range(tiles):
            lo, hi = _kv_tiles(qb * 128 * tiles + t * 128, S, causal, eff_window)
            ready = [(t_ns, arg) for t_ns, _, code, arg in e["roles"][f"softmax{t}"]
                     if code == "s_ready"]
            assert [a for _, a in ready] == list(range(lo, hi)), (c, t)
            for t_ns, j in ready:
                assert s_issued[(t, j)] <= t_ns, (c, t, j)
            codes = [code for _, _, code, _ in e["roles"][f"softmax{t}"]]
            if hi > lo:
                assert codes[-2:] == ["epilogue_start", "epilogue_end"], (c, t)
        assert e["roles"]["mma"][-1][2] == "mma_drained"
    summary = trace.summarize(events)
    assert summary["span_ns"] > 0 and summary["kv_step_ns_median"] > 0
    print(f"trace B{B} S{S} H{H}/{Hkv} D{D}: {summary}")


def test_bounds_guard_skips_and_reports():
    dev = torch.device("cuda:0")
    B, S, H, Hkv, D = 1, 600, 4, 2, 128
    q, k, v = (t.to(dev) for t in make_qkv(B, S, H, Hkv, D, torch.bfloat16, seed=77))
    scale = 1.0 / math.sqrt(D)
    limit = (B * H * S) // 2
    out, lse, status, _ = trace.run_traced(q, k, v, scale, "causal", -1, lse_limit=limit)
    torch.cuda.synchronize()
    assert status == fa.FA_ERR_BOUNDS
    ref, ref_lse = fa.mha_no_cache(q, k, v, scale, "causal", return_lse=True)
    torch.cuda.synchronize()
    flat, ref_flat = lse.reshape(-1), ref_lse.reshape(-1)
    assert torch.equal(flat[:limit], ref_flat[:limit])
    assert torch.isnan(flat[limit:]).all()
    assert torch.equal(out, ref)
    # The next launch without the lowered limit is clean again.
    _, _, status, _ = trace.run_traced(q, k, v, scale, "causal", -1)
    assert status == fa.FA_OK
