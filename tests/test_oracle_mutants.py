"""Planted mistakes: each mutant is a copy of the oracle's C source with one
plausible error (an off-by-one mask, a dropped term, a swapped operand, a wrong
head index...). It is compiled on the CPU and the independent pins are run on
it; every mutant must fail at least one of them. This shows the pins would
catch such a mistake in the real oracle.
"""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import test_oracle_pins as pins

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "fa_oracle.c")

MUTANTS = {
    "causal_includes_future": ("if (causal && j > i) return 0;", "if (causal && j > i + 1) return 0;"),
    "causal_hides_diagonal": ("if (causal && j > i) return 0;", "if (causal && j >= i) return 0;"),
    "window_one_too_wide": ("if (window > 0 && i - j >= window) return 0;",
                            "if (window > 0 && i - j > window) return 0;"),
    "two_sided_window_open_right": ("if (!causal && window > 0 && j - i >= window) return 0;",
                                    "if (!causal && window > 0 && j - i > window) return 0;"),
    "tiled_head_map": ("job->head_map == 0 ? h / G : h % Hkv", "job->head_map == 0 ? h % Hkv : h % Hkv"),
    "scale_dropped": ("score[j] = job->scale * dot;", "score[j] = dot;"),
    "scale_squared": ("score[j] = job->scale * dot;", "score[j] = job->scale * job->scale * dot;"),
    "no_max_subtraction": ("const double e = exp(score[j] - m);", "const double e = exp(score[j]);"),
    "values_from_keys": ("const double *vrow = job->v + ", "const double *vrow = job->k + "),
    "no_normalisation": ("orow[d] = acc[d] / denom;", "orow[d] = acc[d];"),
    "lse_drops_max": ("m + log(denom)", "log(denom)"),
    "lse_log2": ("m + log(denom)", "m + log2(denom)"),
    "query_row_offset": ("const double *qrow = job->q + ((b * job->nrows + r) * H + h) * D;",
                         "const double *qrow = job->q + ((b * job->nrows + r) * H + (h + 1) % H) * D;"),
}


# Mistakes specific to the KV-cache form (lengths, end alignment, empty rows).
KVCACHE_MUTANTS = {
    "cache_ignores_lengths": ("const long L = job->lens ? job->lens[b] : S;", "const long L = S;"),
    "cache_position_one_late": ("L - job->nrows + r :", "L - job->nrows + r + 1 :"),
    "cache_position_from_start": ("job->from_end ? L - job->nrows + r :", "job->from_end ? r :"),
    "cache_sum_reads_to_capacity": ("for (long j = 0; j < L; ++j) {\n      if (!seen[j]) continue;",
                                    "for (long j = 0; j < S; ++j) {\n      if (!seen[j]) continue;"),
    "cache_empty_row_divides_by_zero": ("if (denom > 0.0) {", "if (1) {"),
}


def _build_mutant(name, tmp_path):
    before, after = {**MUTANTS, **KVCACHE_MUTANTS}[name]
    src = open(SRC).read()
    assert src.count(before) == 1, f"mutation site for {name} not unique"
    mpath = tmp_path / f"{name}.c"
    mpath.write_text(src.replace(before, after))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(mpath),
                    "-lm", "-lpthread"], check=True)
    return str(so)


def _pins_fail(oracle_mod, lib):
    """Run a compact set of the independent pins; True if any fails."""
    def run(fn):
        try:
            fn()
            return False
        except (AssertionError, ValueError, FloatingPointError):
            return True

    class Bound:  # the oracle module, redirected to the mutant library
        HEAD_MAP_GROUPED = oracle_mod.HEAD_MAP_GROUPED
        HEAD_MAP_TILED = oracle_mod.HEAD_MAP_TILED

        @staticmethod
        def mha_forward(*a, **kw):
            out, lse = oracle_mod.mha_forward(*a, lib=lib, **kw)
            if not (np.isfinite(out).all() and np.isfinite(lse).all()):
                raise AssertionError("non-finite output")
            return out, lse

    checks = [
        lambda: pins.test_golden_closed_form_cases(Bound),
        lambda: pins.test_identical_keys_average_visible_values(Bound, True, 5),
        lambda: pins.test_single_visible_key_returns_its_value(Bound),
        lambda: pins.test_grouped_equals_explicit_repeat(Bound, True, -1),
    ]
    checks.append(lambda: pins.test_identical_keys_average_visible_values(Bound, False, 3))
    for causal, window in [(False, -1), (True, -1), (True, 6), (False, 5)]:
        checks.append(lambda c=causal, w=window: pins.test_matches_torch_sdpa_fp64(Bound, c, w, 2))
    return any(run(c) for c in checks)


def test_real_oracle_passes_compact_pins(oracle_mod):
    assert not _pins_fail(oracle_mod, None)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(oracle_mod, tmp_path, name):
    lib = oracle_mod.load_library(_build_mutant(name, tmp_path))
    with np.errstate(all="ignore"):
        assert _pins_fail(oracle_mod, lib), f"mutant {name} passed every pin"


def _kvcache_pins_fail(oracle_mod, lib):
    """Run a compact set of the KV-cache pins against a (mutant) library."""
    import test_oracle_kvcache_pins as kv

    def run(fn):
        try:
            fn()
            return False
        except (AssertionError, ValueError, FloatingPointError):
            return True

    class Bound:
        @staticmethod
        def mha_forward(*a, **kw):
            return oracle_mod.mha_forward(*a, lib=lib, **kw)

        @staticmethod
        def mha_forward_kvcache(*a, **kw):
            return oracle_mod.mha_forward_kvcache(*a, lib=lib, **kw)

    checks = [
        lambda: kv.test_matches_torch_sdpa_on_sliced_cache(Bound, True, -1, 3),
        lambda: kv.test_matches_torch_sdpa_on_sliced_cache(Bound, False, 2, 3),
        lambda: kv.test_identical_keys_average_visible_values(Bound, True, 4),
        lambda: kv.test_never_reads_past_the_cache_length(Bound, True, -1),
        lambda: kv.test_queries_before_the_sequence_start_see_nothing(Bound),
    ]
    return any(run(c) for c in checks)


def test_real_oracle_passes_compact_kvcache_pins(oracle_mod):
    assert not _kvcache_pins_fail(oracle_mod, None)


@pytest.mark.parametrize("name", sorted(KVCACHE_MUTANTS))
def test_planted_kvcache_mistake_is_caught(oracle_mod, tmp_path, name):
    lib = oracle_mod.load_library(_build_mutant(name, tmp_path))
    with np.errstate(all="ignore"):
        assert _kvcache_pins_fail(oracle_mod, lib), f"mutant {name} passed every pin"
