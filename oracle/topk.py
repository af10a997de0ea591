"""Plain CPU top-K selection: the second workload of the Modular recipe
"Custom Operations: Applications in AI Models" (section "Optimizing top-K
token sampling for GPUs in MAX"). TEST INFRASTRUCTURE ONLY: called by the
tests, the smoke check and the benchmark's CPU legs, never by the product
path; it shares no code with the CUDA library.

What the section says the op does: it takes a batch of rows of scores (in the
demo, how often each candidate next word appears, as percentages) and returns
two arrays that order each row by highest value — the values and their
indices. Readings where the prose stops:

* K: the op returns the K highest entries of each row (1 <= K <= V); K = V
  orders the whole row, as in the demo.
* Order: descending by value under IEEE-754 total order
  (-NaN < -inf < ... < -0 < +0 < ... < +inf < +NaN), so every input,
  NaN and signed zeros included, has one place. Equal values (identical bit
  patterns) keep ascending index order. With these two rules the output is
  unique, so a GPU result can be compared bit for bit.
* Drawing one token from the K survivors (the "sampling" in the section's
  title) is not described; the op stops at the ordered selection.

The implementation maps each fp32 value to a 32-bit key that orders like the
total order (sign bit clear: set it; sign bit set: invert every bit) and
sorts (key descending, index ascending) with numpy's lexsort — a library sort
as the one step, nothing fused or reordered.

Parity status: pinned by ``tests/test_oracle_topk_pins.py``.
"""
from __future__ import annotations

import numpy as np


def total_order_keys(x: np.ndarray) -> np.ndarray:
    """uint32 keys whose unsigned order is the IEEE-754 total order of fp32 x."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    neg = (bits & np.uint32(0x80000000)) != 0
    return np.where(neg, ~bits, bits | np.uint32(0x80000000)).astype(np.uint32)


def topk(scores, k: int):
    """scores: [B, V] (anything numpy turns into fp32). Returns (values [B, k]
    fp32, indices [B, k] int32): per row the k highest entries, descending in
    total order, equal values by ascending index."""
    x = np.asarray(scores, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("scores must be [B, V]")
    B, V = x.shape
    if not 1 <= k <= V:
        raise ValueError(f"k must be in [1, {V}]")
    values = np.empty((B, k), dtype=np.float32)
    indices = np.empty((B, k), dtype=np.int32)
    idx = np.arange(V, dtype=np.int64)
    for b in range(B):
        keys = total_order_keys(x[b]).astype(np.int64)
        # lexsort sorts by the last key first: -key (descending), then index.
        order = np.lexsort((idx, -keys))[:k]
        indices[b] = order.astype(np.int32)
        values[b] = x[b][order]
    return values, indices
