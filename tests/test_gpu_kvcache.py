"""GPU parity of the KV-cache entry point (fa_mha_kv_cache, through the C ABI)
against the fp64 oracle's KV-cache form on the same seeded bf16 inputs.

Tolerances are those of the bf16 no-cache path: max-abs 2e-2 and mean-abs
2e-3 on the output, max-abs 2e-3 on finite LSE rows; rows that see no key
must be exactly 0 with LSE = -inf.
"""
import math

import numpy as np
import pytest
import torch

import attention_fa2_forward_gb300 as fa
from attention_fa2_forward_gb300.inputs import KV_WORKLOADS, kv_workload_inputs, make_kv_cache

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN, BF16_LSE = 2e-2, 2e-3, 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    fa.load_library()
    yield
    assert fa.device_status() == fa.FA_OK


def _run_gpu(q, k, v, lens, scale, causal, window, num_splits=0, pass_lens=True):
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    ld = lens.to(dev) if pass_lens else None
    B, Sq, H, _ = q.shape
    out = torch.full_like(qd, float("nan"))
    lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32, device=dev)
    fa.mha_kv_cache(qd, kd, vd, ld, scale, "causal" if causal else "none", window,
                    num_splits=num_splits, out=out, lse=lse)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def _compare(out, lse, ref_out, ref_lse, label):
    assert np.isfinite(out).all(), f"{label}: non-finite output"
    dead = ~np.isfinite(ref_lse)  # rows that see no key
    assert np.all(lse[dead] == -np.inf), f"{label}: lse of rows without keys"
    assert np.isfinite(lse[~dead]).all(), f"{label}: non-finite lse"
    err = np.abs(out - ref_out)
    lerr = np.abs(lse[~dead] - ref_lse[~dead])
    assert err.max() <= BF16_MAX, f"{label}: max-abs {err.max():.3e}"
    assert err.mean() <= BF16_MEAN, f"{label}: mean-abs {err.mean():.3e}"
    if lerr.size:
        assert lerr.max() <= BF16_LSE, f"{label}: lse max-abs {lerr.max():.3e}"
    return float(err.max())


def _case(oracle_mod, B, Sq, S_cache, H, Hkv, D, lens, causal, window, num_splits=0, seed=7,
          scale=None, nan_tail=False, pass_lens=True):
    q, k, v, ln = make_kv_cache(B, Sq, S_cache, H, Hkv, D, seed, lens=lens)
    if nan_tail:  # rows past the lengths are not part of the sequences
        for b in range(B):
            k[b, int(ln[b]):] = float("nan")
            v[b, int(ln[b]):] = float("nan")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out, lse = _run_gpu(q, k, v, ln, scale, causal, window, num_splits, pass_lens)
    ref_out, ref_lse = oracle_mod.mha_forward_kvcache(q, k, v, scale,
                                                      ln.numpy() if pass_lens else None,
                                                      causal, window)
    label = (f"B{B} Sq{Sq} S_cache{S_cache} lens{list(ln.numpy())} H{H}/{Hkv} D{D} "
             f"causal={causal} W={window} splits={num_splits}")
    return _compare(out, lse, ref_out, ref_lse, label)


CASES = [
    # B, Sq, S_cache, H, Hkv, D, lens, causal, window
    (3, 1, 1000, 8, 2, 128, [1000, 517, 1], True, -1),       # decode, ragged, partial tiles
    (2, 1, 777, 8, 2, 64, [777, 300], True, -1),
    (2, 1, 1024, 8, 8, 128, [1024, 896], True, -1),          # lengths on tile boundaries
    (2, 4, 2048, 32, 8, 128, [2048, 1500], True, 300),       # speculative step, causal window
    (2, 40, 1000, 8, 2, 64, [1000, 640], True, -1),          # two position tiles, ragged
    (1, 8, 700, 16, 1, 128, [700], True, -1),                # 16 heads x 8 positions = 128 rows
    (2, 5, 500, 12, 2, 128, [500, 129], True, -1),           # G = 6 (rows 30)
    (2, 3, 600, 4, 4, 64, [600, 256], False, -1),            # MHA, no mask
    (2, 3, 600, 8, 2, 128, [600, 256], False, 100),          # two-sided window
    (2, 2, 3000, 8, 2, 128, [3000, 2500], True, 1),          # window of one key
]


@pytest.mark.parametrize("num_splits", [0, 1, 3])
@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_kv_cache_matches_oracle(oracle_mod, case, num_splits):
    _case(oracle_mod, *case, num_splits=num_splits, seed=11 + CASES.index(case))


@pytest.mark.parametrize("D", [16, 32, 80, 96, 112, 136, 256])
@pytest.mark.parametrize("num_splits", [1, 3])
def test_kv_cache_other_head_dims(oracle_mod, D, num_splits):
    _case(oracle_mod, 2, 3, 700, 8, 2, D, [700, 333], True, -1, num_splits=num_splits,
          seed=50 + D)


@pytest.mark.parametrize("num_splits", [2, 5, 8, 64])
def test_many_splits_on_a_long_cache(oracle_mod, num_splits):
    _case(oracle_mod, 2, 1, 5000, 8, 2, 128, [5000, 3333], True, -1, num_splits=num_splits)


def test_queries_before_the_sequence_start(oracle_mod):
    """Causal rows at negative positions (L_b < Sq) and an empty cache
    (L_b = 0) see no key: out 0, lse -inf."""
    for splits in (0, 1, 2):
        _case(oracle_mod, 2, 6, 300, 4, 2, 64, [3, 0], True, -1, num_splits=splits)
        _case(oracle_mod, 2, 6, 300, 4, 2, 64, [3, 0], False, -1, num_splits=splits)


def test_cache_rows_past_the_length_are_never_used(oracle_mod):
    """NaN planted in every cache row past L_b must not reach the output."""
    _case(oracle_mod, 3, 2, 1000, 8, 2, 128, [1000, 517, 130], True, -1, nan_tail=True)
    _case(oracle_mod, 2, 1, 700, 8, 2, 64, [700, 5], False, -1, nan_tail=True, num_splits=3)


def test_stream_k_quotas_spanning_many_sequences(oracle_mod):
    """The automatic plan on 60 short sequences of one KV head (60 units,
    fewer than half the SMs, 60 position-tile groups): CTA quotas of key tiles
    cover pieces of several sequences, some with no keys (whose rows must come
    out 0 / -inf), some cut at a quota boundary; NaN planted past every
    length."""
    rng = np.random.default_rng(61)
    lens = [int(x) for x in rng.integers(0, 700, size=60)]
    lens[3] = 0
    lens[17] = 0
    lens[40] = 699
    _case(oracle_mod, 60, 1, 700, 4, 1, 128, lens, True, -1, nan_tail=True, seed=61)
    _case(oracle_mod, 60, 2, 700, 8, 1, 64, lens, True, 100, seed=62)


def test_full_caches_without_lengths(oracle_mod):
    _case(oracle_mod, 2, 3, 900, 8, 2, 128, [900, 900], True, -1, pass_lens=False)


def test_zero_scale_averages_visible_values(oracle_mod):
    _case(oracle_mod, 2, 2, 400, 4, 2, 128, [400, 150], True, 64, scale=0.0)


@pytest.mark.parametrize("name", sorted(KV_WORKLOADS))
def test_kv_workload_full_size(oracle_mod, name):
    """The decode workloads at their full sizes, every query row checked."""
    w = KV_WORKLOADS[name]
    q, k, v, ln = kv_workload_inputs(w)
    out, lse = _run_gpu(q, k, v, ln, w.scale, w.causal, w.window)
    ref_out, ref_lse = oracle_mod.mha_forward_kvcache(q, k, v, w.scale, ln.numpy(), w.causal,
                                                      w.window)
    _compare(out, lse, ref_out, ref_lse, name)


def test_stall_probe_reports_timeout_on_the_kv_cache_path():
    """The bounded waits of the KV-cache kernel expire under the stall probe:
    the call completes, the status reports FA_ERR_TIMEOUT, and the next call
    on the same context is correct again."""
    q, k, v, ln = make_kv_cache(2, 1, 600, 8, 2, 128, 5, lens=[600, 300])
    dev = torch.device("cuda:0")
    qd, kd, vd, ld = q.to(dev), k.to(dev), v.to(dev), ln.to(dev)
    assert fa.device_status() == fa.FA_OK
    old_limit = fa.set_wait_timeout_ns(20_000_000)
    fa.set_stall_probe(True)
    try:
        fa.mha_kv_cache(qd, kd, vd, ld, num_splits=2)
        assert fa.device_status(clear=True) == fa.FA_ERR_TIMEOUT
    finally:
        fa.set_stall_probe(False)
        fa.set_wait_timeout_ns(old_limit)
    out = fa.mha_kv_cache(qd, kd, vd, ld, num_splits=2)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FA_OK
    assert torch.isfinite(out).all()


def test_workspace_too_small_is_rejected():
    lib = fa.load_library()
    dev = torch.device("cuda:0")
    q = torch.zeros(1, 1, 8, 128, dtype=torch.bfloat16, device=dev)
    kc = torch.zeros(1, 4096, 2, 128, dtype=torch.bfloat16, device=dev)
    splits, ws = fa.kv_cache_plan(1, 1, 4096, 8, 2, 128, num_splits=4)
    assert splits == 4 and ws > 0
    buf = torch.empty(ws, dtype=torch.uint8, device=dev)
    rc = lib.fa_mha_kv_cache(q.data_ptr(), None, q.data_ptr(), kc.data_ptr(), kc.data_ptr(), None,
                             1, 1, 4096, 8, 2, 128, 0.1, 1, -1, 4, buf.data_ptr(), ws - 16, 0,
                             None)
    assert rc == fa.FA_ERR_INVALID_ARG
    rc = lib.fa_mha_kv_cache(q.data_ptr(), None, q.data_ptr(), kc.data_ptr(), kc.data_ptr(), None,
                             1, 1, 4096, 8, 2, 128, 0.1, 1, -1, 4, None, 0, 0, None)
    assert rc == fa.FA_ERR_INVALID_ARG
