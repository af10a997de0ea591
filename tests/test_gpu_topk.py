"""GPU parity of fa_topk (through the C ABI) against the CPU top-K oracle:
values and indices must match bit for bit (the order is total, so the answer
is unique)."""
import struct

import numpy as np
import pytest
import torch

import attention_fa2_forward_gb300 as fa
from attention_fa2_forward_gb300.inputs import TOPK_WORKLOADS, make_scores
from oracle import topk as topk_oracle

pytestmark = pytest.mark.gpu

NEG_NAN = struct.unpack("<f", struct.pack("<I", 0xffc00000))[0]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    fa.build()
    fa.load_library()
    yield
    assert fa.device_status() == fa.FA_OK


def _check(scores_cpu, k, scores_dev=None):
    x = scores_cpu.numpy()
    dev = scores_dev if scores_dev is not None else scores_cpu.cuda()
    vals, idx = fa.topk(dev, k)
    torch.cuda.synchronize()
    ref_v, ref_i = topk_oracle.topk(x, k)
    got_i = idx.cpu().numpy()
    got_v = vals.cpu().numpy()
    np.testing.assert_array_equal(got_i, ref_i)
    assert got_v.tobytes() == ref_v.tobytes(), "values differ bit-wise"


@pytest.mark.parametrize("k", [1, 7, 50, 128, 1000, 1024])
@pytest.mark.parametrize("V", [1024, 5000, 40003])
def test_random_rows(k, V):
    if k > V:
        pytest.skip("k > V")
    _check(make_scores(5, V, 100 + V + k), k)


@pytest.mark.parametrize("k", [1, 3, 64, 500])
def test_many_ties(k):
    g = torch.Generator().manual_seed(7)
    x = torch.randint(-3, 4, (4, 9000), generator=g).float()
    _check(x, k)


def test_all_equal_rows_take_the_lowest_indices():
    _check(torch.full((3, 7000), 2.5), 100)


def test_specials_signed_zeros_infinities_nans():
    g = torch.Generator().manual_seed(8)
    x = torch.randn((4, 3000), generator=g)
    x[0, 10] = float("inf")
    x[0, 20] = float("-inf")
    x[1, 5] = float("nan")
    x[1, 6] = NEG_NAN
    x[2, :] = 0.0
    x[2, ::3] = -0.0
    x[3, 100:200] = float("inf")
    _check(x, 150)


@pytest.mark.parametrize("order", ["ascending", "descending"])
def test_sorted_rows(order):
    """Ascending rows make every element beat the running threshold (a prune
    every step); descending rows settle the threshold at once."""
    v = torch.arange(20000, dtype=torch.float32) * 0.01
    if order == "descending":
        v = v.flip(0)
    _check(torch.stack([v, -v]), 333)


def test_short_rows_and_k_equal_v():
    for V in (1, 2, 5, 17, 1023):
        x = make_scores(3, V, V)
        _check(x, V)
        _check(x, 1)


def test_strided_rows():
    wide = make_scores(6, 9000, 9)
    x = wide[:, 100:8100]
    dev = wide.cuda()[:, 100:8100]
    assert dev.stride(0) == 9000
    _check(x.contiguous(), 77, dev)


def test_more_rows_than_one_wave_of_ctas():
    """More rows than resident CTAs: one chunk per row, several waves, each
    chunk CTA sorting its own row."""
    _check(make_scores(700, 3000, 21), 20)
    _check(make_scores(400, 2500, 22), 200)


def test_single_chunk_rows_take_no_workspace():
    """A plan of one chunk per row needs no workspace: the C ABI accepts NULL."""
    B, V, K = 256, 8192, 10
    chunks, ws = fa.topk_plan(B, V, K)
    assert chunks == 1 and ws == 0
    x = make_scores(B, V, 23)
    dev = x.cuda()
    vals = torch.empty((B, K), dtype=torch.float32, device="cuda")
    idx = torch.empty((B, K), dtype=torch.int32, device="cuda")
    lib = fa.load_library()
    rc = lib.fa_topk(vals.data_ptr(), idx.data_ptr(), dev.data_ptr(), B, V, V, K, None, 0,
                     torch.cuda.current_stream().cuda_stream)
    assert rc == fa.FA_OK
    torch.cuda.synchronize()
    ref_v, ref_i = topk_oracle.topk(x.numpy(), K)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_i)
    assert vals.cpu().numpy().tobytes() == ref_v.tobytes()


@pytest.mark.parametrize("B,V,K", [(1, 262144, 50), (1, 262144, 1024), (3, 100000, 1000),
                                   (2, 300000, 7), (9, 65536, 333)])
def test_rows_split_over_many_chunks(B, V, K):
    """Rows spread over several chunk CTAs: each chunk's candidates, merged per
    row by the merge kernel or inside a cluster (up to 147 chunks of a row, K
    up to 1024)."""
    chunks, ws = fa.topk_plan(B, V, K)
    assert chunks > 1
    # clusters of 2, 4, 8 (K <= 128) merge in shared memory
    assert (ws == 0) == (chunks in (2, 4, 8) and K <= 128)
    _check(make_scores(B, V, 30 + K), K)


@pytest.mark.parametrize("B,V,K,chunks", [(152, 8192, 10, 2), (64, 131072, 100, 4),
                                          (38, 65536, 64, 8), (38, 65536, 128, 8)])
def test_rows_merged_inside_a_cluster(B, V, K, chunks):
    """Rows of 2, 4 or 8 chunks with K <= 128: the chunk CTAs of a row form one
    cluster whose first CTA merges the others' candidates from their shared
    memory."""
    got_chunks, ws = fa.topk_plan(B, V, K)
    assert got_chunks == chunks and ws == 0
    _check(make_scores(B, V, 60 + chunks + K), K)


def test_special_values_inside_a_cluster():
    """NaNs of both signs, infinities, signed zeros and all-negative rows on the
    cluster path (8 chunks per row, K <= 128): bit-exact against the oracle."""
    B, V, K = 38, 65536, 64
    assert fa.topk_plan(B, V, K)[0] == 8
    g = torch.Generator().manual_seed(70)
    x = torch.randn((B, V), generator=g)
    x[0, ::97] = float("nan")
    x[1, 5:300] = NEG_NAN
    x[2, 1000:1100] = float("inf")
    x[3, :] = -x[3, :].abs() - 1.0                     # every score negative
    x[4, :] = float("-inf")                            # every score -inf
    x[5, ::2] = 0.0
    x[5, 1::2] = -0.0
    x[6, 60000:] = float("inf")                        # the top K all in the last chunk
    _check(x, K)


def test_negative_thresholds_and_unaligned_rows():
    """Rows whose K-th score is negative (the total-order test on the scan's
    common path) and rows that are not 16-byte aligned (4-byte copies)."""
    g = torch.Generator().manual_seed(71)
    x = -torch.rand((6, 20001), generator=g) - 0.5
    _check(x, 40)
    wide = torch.randn((5, 30003), generator=g)
    dev = wide.cuda()[:, 1:30001]
    assert dev.stride(0) == 30003 and dev.data_ptr() % 16 != 0
    _check(wide[:, 1:30001].contiguous(), 33, dev)


def test_workspace_reused_across_calls():
    """Whatever the workspace held before, every call writes the candidates it
    reads."""
    B, V, K = 4, 70000, 64
    _, ws_bytes = fa.topk_plan(B, V, K)
    ws = torch.full((ws_bytes,), 0xAB, dtype=torch.uint8, device="cuda")
    for seed in (41, 42, 43):
        x = make_scores(B, V, seed)
        vals, idx = fa.topk(x.cuda(), K, workspace=ws)
        torch.cuda.synchronize()
        ref_v, ref_i = topk_oracle.topk(x.numpy(), K)
        np.testing.assert_array_equal(idx.cpu().numpy(), ref_i)
        assert vals.cpu().numpy().tobytes() == ref_v.tobytes()


@pytest.mark.parametrize("name", sorted(TOPK_WORKLOADS))
def test_topk_workload_full_size(name):
    w = TOPK_WORKLOADS[name]
    _check(make_scores(w.B, w.V, w.seed), w.K)
