"""Failure detection without a GPU fault: the kernels' spin-waits are bounded.

The stall probe makes the MMA-issuing thread of each CTA wait on a barrier
that nothing signals. With a 20 ms wait limit that wait expires; every CTA
must then record the time-out in the device status word, stop issuing, drain
its own TMA copies and MMAs, free its tensor memory and return. The call
completes, fa_device_status reports FA_ERR_TIMEOUT, and the context stays
usable: a following call without the probe is correct.
"""
import math

import pytest
import torch

import attention_fa2_forward_gb300 as fa
from attention_fa2_forward_gb300.inputs import make_qkv

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_is_reported_and_recoverable(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    dev = torch.device("cuda:0")
    q, k, v = make_qkv(1, 1024, 8, 2, 128, torch.bfloat16, seed=21)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    scale = 1.0 / math.sqrt(128)
    fa.mha_no_cache(qd, kd, vd, scale, "causal")
    assert fa.device_status(clear=True) == fa.FA_OK
    old = fa.set_wait_timeout_ns(20_000_000)
    fa.set_stall_probe(True)
    try:
        fa.mha_no_cache(qd, kd, vd, scale, "causal")
        assert fa.device_status(clear=True) == fa.FA_ERR_TIMEOUT
    finally:
        fa.set_stall_probe(False)
        fa.set_wait_timeout_ns(old)
    assert fa.device_status(clear=True) == fa.FA_OK
    out = fa.mha_no_cache(qd, kd, vd, scale, "causal")
    torch.cuda.synchronize()
    ref, _ = oracle_mod.mha_forward(q, k, v, scale, True, -1)
    err = (out.double().cpu() - torch.from_numpy(ref)).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
    assert fa.device_status() == fa.FA_OK


def test_bounded_wait_timeout_on_the_persistent_schedule(oracle_mod):
    """The same stall probe on the persistent one-tile kernel (head dim 64,
    S 1024, more query tiles than resident CTAs): the MMA thread gives up,
    the softmax warps' waits expire and they leave their item loop together,
    the producer drains its copies; the next call is correct."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    dev = torch.device("cuda:0")
    q, k, v = make_qkv(4, 1024, 16, 16, 64, torch.bfloat16, seed=23)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    scale = 1.0 / math.sqrt(64)
    assert fa.device_status(clear=True) == fa.FA_OK
    old = fa.set_wait_timeout_ns(20_000_000)
    fa.set_stall_probe(True)
    try:
        fa.mha_no_cache(qd, kd, vd, scale, "causal")
        assert fa.device_status(clear=True) == fa.FA_ERR_TIMEOUT
    finally:
        fa.set_stall_probe(False)
        fa.set_wait_timeout_ns(old)
    assert fa.device_status(clear=True) == fa.FA_OK
    out = fa.mha_no_cache(qd, kd, vd, scale, "causal")
    torch.cuda.synchronize()
    ref, _ = oracle_mod.mha_forward(q, k, v, scale, True, -1)
    err = (out.double().cpu() - torch.from_numpy(ref)).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
    assert fa.device_status() == fa.FA_OK


def test_timeout_is_reported_on_its_own_stream_only(oracle_mod):
    """fa_stream_status reads the status word of one stream, ordered on that
    stream: a time-out on stream A shows on A and not on B, and reading it
    waits for A's work only."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    dev = torch.device("cuda:0")
    q, k, v = make_qkv(1, 1024, 8, 2, 128, torch.bfloat16, seed=22)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    scale = 1.0 / math.sqrt(128)
    a, b = torch.cuda.Stream(), torch.cuda.Stream()
    for s in (a, b):
        with torch.cuda.stream(s):
            fa.mha_no_cache(qd, kd, vd, scale, "causal")
        assert fa.stream_status(s) == fa.FA_OK
    old = fa.set_wait_timeout_ns(20_000_000)
    fa.set_stall_probe(True)
    try:
        with torch.cuda.stream(a):
            fa.mha_no_cache(qd, kd, vd, scale, "causal")
    finally:
        fa.set_stall_probe(False)
        fa.set_wait_timeout_ns(old)
    with torch.cuda.stream(b):
        out_b = fa.mha_no_cache(qd, kd, vd, scale, "causal")
    assert fa.stream_status(b) == fa.FA_OK
    assert fa.stream_status(a, clear=False) == fa.FA_ERR_TIMEOUT  # sticky until cleared
    assert fa.stream_status(a, clear=True) == fa.FA_ERR_TIMEOUT
    assert fa.stream_status(a) == fa.FA_OK
    assert fa.device_status(clear=True) == fa.FA_OK
    ref, _ = oracle_mod.mha_forward(q, k, v, scale, True, -1)
    err = (out_b.double().cpu() - torch.from_numpy(ref)).abs()
    assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3


def test_device_status_sees_every_stream():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    dev = torch.device("cuda:0")
    q, k, v = (t.to(dev) for t in make_qkv(1, 512, 4, 4, 64, torch.bfloat16, seed=23))
    s = torch.cuda.Stream()
    old = fa.set_wait_timeout_ns(20_000_000)
    fa.set_stall_probe(True)
    try:
        with torch.cuda.stream(s):
            fa.mha_no_cache(q, k, v, 0.125, "none")
    finally:
        fa.set_stall_probe(False)
        fa.set_wait_timeout_ns(old)
    assert fa.device_status(clear=False) == fa.FA_ERR_TIMEOUT
    assert fa.device_status(clear=True) == fa.FA_ERR_TIMEOUT
    assert fa.stream_status(s) == fa.FA_OK
