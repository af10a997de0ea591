"""fp64 CPU oracle for the multi-head attention forward, without KV cache
(``mha_forward``) and with one (``mha_forward_kvcache``).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
CPU-baseline / reference leg may import this package; the product path never
does. The arithmetic lives in ``fa_oracle.c`` (plain C, fp64, one query row at
a time, see its header for the step-by-step definition and the page passages
it follows). This module only compiles that file with gcc and marshals numpy
arrays through ctypes.

Parity status: pinned. ``tests/test_oracle_pins.py`` checks it against closed
forms (uniform keys give the mean of the visible values, one visible key
returns its value row, the two-key sigmoid mix), invariants (key shift, key
permutation, rows summing to one), hand-derived fixtures in ``tests/golden/``,
an independent blockwise online-softmax recomputation (the FlashAttention-2
loop of the tiny_flash_attn.py page and the normalise-every-step loop of the
Modular recipe's kernel listing), and torch's fp64 scaled_dot_product_attention.
``tests/test_oracle_kvcache_pins.py`` pins the KV-cache form the same way
(torch SDPA on the sliced cache with an explicit end-aligned mask, closed-form
window means, never reading past the cache length, split-KV recombination).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libfa_oracle.so")

_lib = None
_lock = threading.Lock()

HEAD_MAP_GROUPED = 0  # query head h reads KV head h // (H // Hkv)
HEAD_MAP_TILED = 1  # query head h reads KV head h % Hkv


def build(force: bool = False) -> str:
    """Compile fa_oracle.c into a shared library (gcc, -O2, IEEE arithmetic)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """Open a compiled oracle library and declare its C signature."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    lp = ctypes.POINTER(ctypes.c_long)
    lib.fa_oracle_forward.restype = ctypes.c_int
    lib.fa_oracle_forward.argtypes = [
        dp, dp, dp, dp, dp,
        ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long, ctypes.c_long,
        ctypes.c_double, ctypes.c_int, ctypes.c_long, ctypes.c_int,
        lp, ctypes.c_long, ctypes.c_int,
    ]
    if hasattr(lib, "fa_oracle_forward_kvcache"):
        lib.fa_oracle_forward_kvcache.restype = ctypes.c_int
        lib.fa_oracle_forward_kvcache.argtypes = [
            dp, dp, dp, dp, dp,
            ctypes.c_long, ctypes.c_long, ctypes.c_long, lp, ctypes.c_long, ctypes.c_long,
            ctypes.c_long, ctypes.c_double, ctypes.c_int, ctypes.c_long, ctypes.c_int,
        ]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _as_f64(x) -> np.ndarray:
    """Widen a numpy array or a CPU torch tensor (any float dtype) to fp64."""
    if hasattr(x, "detach"):  # torch tensor: bf16 has no numpy dtype
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def mha_forward(q, k, v, scale: float, causal: bool = False, window: int = -1,
                rows=None, head_map: int = HEAD_MAP_GROUPED, nthreads: int | None = None,
                lib=None):
    """Attention forward in fp64.

    q: [B, S, H, D], or [B, len(rows), H, D] when ``rows`` lists the query
    positions to evaluate. k, v: [B, S, Hkv, D]. Returns (out [B, nq, H, D],
    lse [B, H, nq]) as fp64 numpy arrays, nq = S or len(rows). ``lib`` selects
    another compiled copy of the oracle (used by the planted-mistake tests).
    """
    qd, kd, vd = _as_f64(q), _as_f64(k), _as_f64(v)
    B, S, Hkv, D = kd.shape
    H = qd.shape[2]
    if vd.shape != kd.shape or qd.shape[0] != B or qd.shape[3] != D:
        raise ValueError(f"shape mismatch q{qd.shape} k{kd.shape} v{vd.shape}")
    if rows is None:
        if qd.shape[1] != S:
            raise ValueError("q must hold all S rows when rows is None")
        nrows, rows_arr, rows_ptr = S, None, None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
        if qd.shape[1] != nrows:
            raise ValueError("q must hold exactly the requested rows")
        rows_ptr = rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
    out = np.empty((B, nrows, H, D), dtype=np.float64)
    lse = np.empty((B, H, nrows), dtype=np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    rc = (lib or _load()).fa_oracle_forward(
        qd.ctypes.data_as(dp), kd.ctypes.data_as(dp), vd.ctypes.data_as(dp),
        out.ctypes.data_as(dp), lse.ctypes.data_as(dp),
        B, S, H, Hkv, D, float(scale), int(bool(causal)), int(window), int(head_map),
        rows_ptr, nrows, int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"fa_oracle_forward failed with status {rc}")
    return out, lse


def mha_forward_kvcache(q, k_cache, v_cache, scale: float, cache_lens=None,
                        causal: bool = False, window: int = -1,
                        nthreads: int | None = None, lib=None):
    """KV-cache attention forward in fp64: batch b holds cache_lens[b] keys
    (the first rows of k_cache / v_cache, [B, S_cache, Hkv, D]) and its Sq
    queries q[b] ([B, Sq, H, D]) are the last Sq tokens of that sequence, so
    query row r sits at position cache_lens[b] - Sq + r. cache_lens = None
    means S_cache keys everywhere. A query that sees no key gets out = 0 and
    lse = -inf. Returns (out [B, Sq, H, D], lse [B, H, Sq]) fp64 arrays.
    """
    qd, kd, vd = _as_f64(q), _as_f64(k_cache), _as_f64(v_cache)
    B, S, Hkv, D = kd.shape
    Sq, H = qd.shape[1], qd.shape[2]
    if vd.shape != kd.shape or qd.shape[0] != B or qd.shape[3] != D:
        raise ValueError(f"shape mismatch q{qd.shape} k{kd.shape} v{vd.shape}")
    lens_ptr, lens_arr = None, None
    if cache_lens is not None:
        lens_arr = np.ascontiguousarray(np.asarray(cache_lens, dtype=np.int64).reshape(-1))
        if lens_arr.size != B:
            raise ValueError("cache_lens needs one entry per batch")
        lens_ptr = lens_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_long))
    out = np.empty((B, Sq, H, D), dtype=np.float64)
    lse = np.empty((B, H, Sq), dtype=np.float64)
    dp = ctypes.POINTER(ctypes.c_double)
    rc = (lib or _load()).fa_oracle_forward_kvcache(
        qd.ctypes.data_as(dp), kd.ctypes.data_as(dp), vd.ctypes.data_as(dp),
        out.ctypes.data_as(dp), lse.ctypes.data_as(dp),
        B, Sq, S, lens_ptr, H, Hkv, D, float(scale), int(bool(causal)), int(window),
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"fa_oracle_forward_kvcache failed with status {rc}")
    return out, lse
