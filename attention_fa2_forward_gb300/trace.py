"""Event traces of the bf16 prefill kernel, recorded by the debug build.

The debug build (``libfa_mha_debug.so``, compiled with FA_TRACE=1) lets each
CTA of the prefill kernel append time-stamped events per warp role into a
device buffer (layout: ``include/fa_mha.h``, ``fa_trace_set_buffer``).
:func:`run_traced` runs one forward through that build and returns the
decoded events; :func:`summarize` turns them into per-CTA phase times.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _mask_code, load_debug_library

# "softmax0" / "softmax1": warp 0 / 4, the first warp of Q tile 0 / 1; the
# other softmax warps follow ("softmax0_w1" = warp 1, ...).
ROLES = ("producer", "mma", "softmax0", "softmax1", "softmax0_w1", "softmax0_w2",
         "softmax0_w3", "softmax1_w1", "softmax1_w2", "softmax1_w3")
CODES = {1: "cta_start", 2: "q_load_issued", 3: "k_load_issued", 4: "v_load_issued",
         5: "q_ready", 6: "s_issued", 7: "pv_issued", 8: "mma_drained", 9: "s_ready",
         10: "p_ready", 11: "epilogue_start", 12: "epilogue_end", 13: "s_loaded",
         14: "max_done", 15: "exp_done", 16: "p_seen"}
EVENTS_PER_ROLE = 256


def run_traced(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float, mask="causal",
               window: int = -1, lse_limit: int = 0):
    """One bf16 forward (dense BSHD, D <= 128) through the debug build with the
    event trace on. Returns (out, lse, status, events): status is the
    stream's status after the call (FA_OK, or FA_ERR_BOUNDS when a bounds
    guard fired; ``lse_limit`` > 0 makes the LSE guard fire past that many
    elements), events the list :func:`decode` returns."""
    lib = load_debug_library()
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    ctas = int(lib.fa_trace_ctas(B, S, H, D))
    if ctas <= 0:
        raise ValueError("the trace covers the bf16 prefill kernel (D <= 128)")
    per_cta = int(lib.fa_trace_bytes_per_cta())
    buf = torch.zeros(ctas * per_cta, dtype=torch.uint8, device=q.device)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        lib.fa_stream_status(stream.cuda_stream, 1)
        if lib.fa_trace_set_buffer(buf.data_ptr(), buf.numel()) != 0:
            raise RuntimeError(lib.fa_last_error_message().decode())
        lib.fa_debug_set_lse_limit(int(lse_limit))
        try:
            rc = lib.fa_mha_no_cache(out.data_ptr(), lse.data_ptr(), q.data_ptr(), k.data_ptr(),
                                     v.data_ptr(), B, S, H, Hkv, D, float(scale),
                                     _mask_code(mask), int(window), 0, stream.cuda_stream)
            if rc != 0:
                raise RuntimeError(lib.fa_last_error_message().decode())
            status = int(lib.fa_stream_status(stream.cuda_stream, 1))
        finally:
            lib.fa_trace_set_buffer(None, 0)
            lib.fa_debug_set_lse_limit(0)
    return out, lse, status, decode(buf.cpu().numpy(), ctas)


def decode(raw: np.ndarray, ctas: int) -> list[dict]:
    """Per CTA: {"cta", "sm", "roles": {role: [(t_ns, clock, code, arg), ...]}}
    with events in recording order; t_ns is the global timer, clock the SM's
    32-bit cycle counter."""
    rec = np.ascontiguousarray(raw).view(np.uint32).reshape(ctas, len(ROLES), EVENTS_PER_ROLE, 4)
    result = []
    for c in range(ctas):
        roles = {}
        sm = None
        for r, name in enumerate(ROLES):
            ev = []
            for x, y, z, w in rec[c, r]:
                code = int(w) >> 24
                if code == 0:
                    break
                arg = int(w) & 0xFFFFFF
                ev.append((int(x) | (int(y) << 32), int(z), CODES.get(code, str(code)), arg))
                if code == 1:
                    sm = arg
            roles[name] = ev
        result.append({"cta": c, "sm": sm, "roles": roles})
    return result


def summarize(events: list[dict]) -> dict:
    """Kernel-wide phase times from decoded events: span of the launch, and
    per CTA the time from its start to its first S MMA, from there to its last
    PV MMA, and its epilogue, plus the median time between consecutive S(j)
    arrivals of one Q tile (the KV-step period), all in ns."""
    t0 = min(e["roles"]["producer"][0][0] for e in events if e["roles"]["producer"])
    t1 = 0
    setup, main, epi, periods = [], [], [], []
    for e in events:
        roles = e["roles"]
        if not roles["producer"] or not roles["mma"]:
            continue
        start = roles["producer"][0][0]
        s_iss = [t for t, _, c, _ in roles["mma"] if c == "s_issued"]
        pv_iss = [t for t, _, c, _ in roles["mma"] if c == "pv_issued"]
        ends = [t for name in ("softmax0", "softmax1") for t, _, c, _ in roles[name]
                if c == "epilogue_end"]
        starts = [t for name in ("softmax0", "softmax1") for t, _, c, _ in roles[name]
                  if c == "epilogue_start"]
        if s_iss:
            setup.append(s_iss[0] - start)
        if s_iss and pv_iss:
            main.append(pv_iss[-1] - s_iss[0])
        if starts and ends:
            epi.append(max(ends) - min(starts))
        if ends:
            t1 = max(t1, max(ends))
        for name in ("softmax0", "softmax1"):
            ready = [t for t, _, c, _ in roles[name] if c == "s_ready"]
            periods += [b - a for a, b in zip(ready, ready[1:])]

    def med(x):
        return float(np.median(x)) if x else None

    return {"span_ns": t1 - t0, "ctas": len(events), "setup_ns_median": med(setup),
            "main_ns_median": med(main), "epilogue_ns_median": med(epi),
            "kv_step_ns_median": med(periods)}
