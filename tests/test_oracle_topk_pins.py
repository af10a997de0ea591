"""Pins for the CPU top-K oracle (oracle/topk.py), each independent of its
code: numpy's sort on distinct finite values (library special case), a
property check that characterises the unique answer under the stated order
(written with Python's own float comparisons, not the oracle's bit keys),
hand-derived fixtures in tests/golden/topk_cases.json, and planted mistakes
that must each fail one of these pins."""
import json
import math
import os
import struct

import numpy as np
import pytest

from oracle import topk as topk_mod

HERE = os.path.dirname(os.path.abspath(__file__))


def _f(v):
    return float(v) if not isinstance(v, str) else {
        "inf": math.inf, "-inf": -math.inf, "nan": math.nan,
        "-nan": struct.unpack("<f", struct.pack("<I", 0xffc00000))[0]}[v]


def _order(x):
    """Total-order position of a fp32 value as a tuple, from Python float
    comparisons and the sign bit (canonical NaNs only)."""
    neg = math.copysign(1.0, x) < 0
    if math.isnan(x):
        return (-2,) if neg else (2,)
    if x == 0.0:
        return (0, 0.0, -1 if neg else 1)
    return (0, x, 0)


def _check_valid(x, k, values, indices):
    """The output is the unique top-k: values match their indices, indices are
    distinct, the order is descending with ties by ascending index, and no
    left-out element beats (or ties with a lower index than) the last one."""
    V = x.shape[0]
    idx = [int(i) for i in indices]
    assert len(set(idx)) == k and all(0 <= i < V for i in idx)
    for j in range(k):
        assert np.float32(x[idx[j]]).tobytes() == np.float32(values[j]).tobytes()
    keys = [(_order(float(x[i])), -i) for i in idx]
    assert all(keys[j] > keys[j + 1] for j in range(k - 1)), "not descending"
    last = keys[-1]
    chosen = set(idx)
    for i in range(V):
        if i not in chosen:
            assert (_order(float(x[i])), -i) < last, f"element {i} should be in the top-{k}"


def _topk(mod, scores, k):
    return mod.topk(scores, k)


@pytest.mark.parametrize("k", [1, 5, 64, 300])
def test_distinct_finite_values_match_numpy_sort(k):
    rng = np.random.default_rng(1)
    x = rng.permutation(np.arange(1, 1001, dtype=np.float32) * 0.37).reshape(2, 500)
    x[1] *= -1.0
    vals, idx = topk_mod.topk(x, k)
    for b in range(2):
        order = np.argsort(-x[b].astype(np.float64), kind="stable")[:k]
        np.testing.assert_array_equal(idx[b], order)
        np.testing.assert_array_equal(vals[b], np.sort(x[b])[::-1][:k])


@pytest.mark.parametrize("k", [1, 3, 17, 40])
def test_ties_and_specials_satisfy_the_selection_properties(k):
    rng = np.random.default_rng(2)
    x = rng.integers(-4, 5, size=(6, 40)).astype(np.float32)  # many ties
    x[0, 5] = -0.0
    x[0, 7] = 0.0
    x[1, 3] = np.inf
    x[2, 9] = -np.inf
    x[3, 4] = np.nan
    x[4, 11] = struct.unpack("<f", struct.pack("<I", 0xffc00000))[0]
    vals, idx = topk_mod.topk(x, k)
    for b in range(x.shape[0]):
        _check_valid(x[b], k, vals[b], idx[b])


def test_golden_cases():
    data = json.load(open(os.path.join(HERE, "golden", "topk_cases.json")))
    for case in data["cases"]:
        x = np.array([[_f(v) for v in row] for row in case["scores"]], dtype=np.float32)
        vals, idx = topk_mod.topk(x, case["k"])
        exp_v = np.array([[_f(v) for v in row] for row in case["values"]], dtype=np.float32)
        np.testing.assert_array_equal(idx, np.array(case["indices"]), err_msg=case["name"])
        assert vals.tobytes() == exp_v.tobytes() or np.array_equal(vals, exp_v, equal_nan=True), \
            case["name"]
        # NaN sign must match too (total order distinguishes it)
        assert (np.signbit(vals) == np.signbit(exp_v)).all(), case["name"]


def test_k_equal_v_orders_the_whole_row():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((3, 33)).astype(np.float32)
    vals, idx = topk_mod.topk(x, 33)
    for b in range(3):
        assert sorted(idx[b].tolist()) == list(range(33))
        _check_valid(x[b], 33, vals[b], idx[b])


def test_rejects_bad_k():
    with pytest.raises(ValueError):
        topk_mod.topk(np.zeros((1, 4)), 0)
    with pytest.raises(ValueError):
        topk_mod.topk(np.zeros((1, 4)), 5)


# --- planted mistakes ---------------------------------------------------------------
MUTANTS = {
    "ties_highest_index_first": ("np.lexsort((idx, -keys))", "np.lexsort((-idx, -keys))"),
    "raw_bits_order": ("np.where(neg, ~bits, bits | np.uint32(0x80000000))", "bits"),
    "negatives_not_inverted": ("np.where(neg, ~bits, bits | np.uint32(0x80000000))",
                               "np.where(neg, bits & np.uint32(0x7fffffff), bits | np.uint32(0x80000000))"),
    "ascending": ("np.lexsort((idx, -keys))", "np.lexsort((idx, keys))"),
    "off_by_one": ("np.lexsort((idx, -keys))[:k]", "np.lexsort((idx, -keys))[1:k + 1]"),
}


def _mutant(name):
    src = open(topk_mod.__file__).read()
    before, after = MUTANTS[name]
    assert src.count(before) == 1
    ns = {"__name__": f"topk_mutant_{name}"}
    exec(compile(src.replace(before, after), f"<{name}>", "exec"), ns)

    class M:
        topk = staticmethod(ns["topk"])
    return M


def _pins_fail(mod):
    checks = []
    rng = np.random.default_rng(4)

    def distinct():
        x = rng.permutation(np.arange(1, 201, dtype=np.float32)).reshape(1, 200) - 100.5
        v, i = mod.topk(x, 7)
        np.testing.assert_array_equal(i[0], np.argsort(-x[0], kind="stable")[:7])

    def props():
        x = rng.integers(-3, 4, size=(3, 25)).astype(np.float32)
        x[0, 2] = -0.0
        v, i = mod.topk(x, 9)
        for b in range(3):
            _check_valid(x[b], 9, v[b], i[b])

    def golden():
        data = json.load(open(os.path.join(HERE, "golden", "topk_cases.json")))
        for case in data["cases"]:
            x = np.array([[_f(t) for t in row] for row in case["scores"]], dtype=np.float32)
            v, i = mod.topk(x, case["k"])
            np.testing.assert_array_equal(i, np.array(case["indices"]))

    checks = [distinct, props, golden]
    for c in checks:
        try:
            c()
        except (AssertionError, ValueError, IndexError):
            return True
    return False


def test_real_oracle_passes_the_mutant_pins():
    assert not _pins_fail(topk_mod)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    with np.errstate(all="ignore"):
        assert _pins_fail(_mutant(name)), f"mutant {name} passed every pin"
