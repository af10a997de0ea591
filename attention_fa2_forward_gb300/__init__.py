"""GB300-native fused multi-head attention forward, without KV cache
(:func:`mha_no_cache`) and over a KV cache (:func:`mha_kv_cache`).

Python binding of the C ABI in ``include/fa_mha.h`` (library
``_build/libfa_mha.so``, built by :func:`build`). The binding only marshals
arguments: it checks tensor placement/shape/dtype, allocates the outputs with
torch and passes raw device pointers and the current CUDA stream to the
library. Every step of the computation runs in the library's CUDA kernels;
there is no fallback: if the library is missing or the GPU is not sm_103a the
call raises.

The operation is MAX's ``mo.mha.no_cache`` (API page "FlashAttentionGPU",
method ``execute``): q in BSHD, k/v in BSHD or BShD (grouped-query attention,
query head h reads KV head h // (H // Hkv)), output with q's shape and dtype,
mask "none", "causal", or causal with a sliding window of W keys.
"""
from __future__ import annotations

import ctypes
import functools
import os
import threading

import torch

from .build import DEBUG_LIB_PATH, LIB_PATH, build  # noqa: F401  (re-exported)

MASK_NONE = 0
MASK_CAUSAL = 1
DTYPE_BF16 = 0
DTYPE_F32 = 1

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_BOUNDS = 5

# Every symbol the header declares (checked by the tests).
EXPORTS = ("fa_mha_no_cache", "fa_mha_no_cache_strided", "fa_mha_no_cache_noalloc",
           "fa_mha_no_cache_host", "fa_mha_no_cache_host_workspace",
           "fa_mha_no_cache_f32_tc", "fa_mha_no_cache_f32_tc_workspace",
           "fa_mha_kv_cache", "fa_mha_kv_cache_plan", "fa_topk", "fa_topk_plan",
           "fa_stream_status", "fa_device_status",
           "fa_set_wait_timeout_ns", "fa_set_stall_probe", "fa_status_string",
           "fa_last_error_message", "fa_version", "fa_trace_set_buffer",
           "fa_trace_bytes_per_cta", "fa_trace_ctas", "fa_debug_set_lse_limit", "fa_shutdown")

_lib = None
_debug_lib = None
_lock = threading.Lock()


class FAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


def load_library(path: str | None = None):
    """Open libfa_mha.so and declare the C signatures. Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        lib = _open(path or LIB_PATH)
        if path is None:
            _lib = lib
        return lib


def load_debug_library():
    """Open the debug build libfa_mha_debug.so (event trace, bounds guards),
    building it first if needed."""
    global _debug_lib
    build(variant="debug")
    with _lock:
        if _debug_lib is None:
            _debug_lib = _open(DEBUG_LIB_PATH)
        return _debug_lib


def _open(p: str):
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library {p} is not built; call attention_fa2_forward_gb300.build() "
            "(nvcc, sm_103a) first")
    lib = ctypes.CDLL(p)
    _declare(lib)
    return lib


def _declare(lib):
    """Declare the C signatures of include/fa_mha.h on a loaded library."""
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.fa_mha_no_cache.restype = i
    lib.fa_mha_no_cache.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float,
                                    i, i, i, vp]
    lp = ctypes.POINTER(ctypes.c_longlong)
    lib.fa_mha_no_cache_strided.restype = i
    lib.fa_mha_no_cache_strided.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, lp, lp, lp, lp,
                                            ctypes.c_float, i, i, i, vp]
    ull = ctypes.c_ulonglong
    lib.fa_mha_kv_cache.restype = i
    lib.fa_mha_kv_cache.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float,
                                    i, i, i, vp, ull, i, vp]
    lib.fa_mha_kv_cache_plan.restype = i
    lib.fa_mha_kv_cache_plan.argtypes = [i, i, i, i, i, i, i, i, i, i,
                                         ctypes.POINTER(i), ctypes.POINTER(ull)]
    lib.fa_mha_no_cache_f32_tc.restype = i
    lib.fa_mha_no_cache_f32_tc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float,
                                           i, i, vp, ull, vp]
    lib.fa_mha_no_cache_host.restype = i
    lib.fa_mha_no_cache_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.c_float,
                                         i, i, i, vp, ull, vp]
    lib.fa_mha_no_cache_host_workspace.restype = ull
    lib.fa_mha_no_cache_host_workspace.argtypes = [i, i, i, i, i, i]
    lib.fa_mha_no_cache_f32_tc_workspace.restype = ull
    lib.fa_mha_no_cache_f32_tc_workspace.argtypes = [i, i, i, i]
    lib.fa_topk.restype = i
    lib.fa_topk.argtypes = [vp, vp, vp, i, i, ctypes.c_longlong, i, vp, ull, vp]
    lib.fa_topk_plan.restype = i
    lib.fa_topk_plan.argtypes = [i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(ull)]
    lib.fa_device_status.restype = i
    lib.fa_device_status.argtypes = [i, i]
    lib.fa_stream_status.restype = i
    lib.fa_stream_status.argtypes = [vp, i]
    lib.fa_trace_set_buffer.restype = i
    lib.fa_trace_set_buffer.argtypes = [vp, ull]
    lib.fa_trace_bytes_per_cta.restype = ull
    lib.fa_trace_bytes_per_cta.argtypes = []
    lib.fa_trace_ctas.restype = ctypes.c_longlong
    lib.fa_trace_ctas.argtypes = [i, i, i, i]
    lib.fa_debug_set_lse_limit.restype = i
    lib.fa_debug_set_lse_limit.argtypes = [ctypes.c_longlong]
    lib.fa_set_wait_timeout_ns.restype = ctypes.c_ulonglong
    lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_ulonglong]
    lib.fa_set_stall_probe.restype = i
    lib.fa_set_stall_probe.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_status_string.argtypes = [i]
    lib.fa_last_error_message.restype = ctypes.c_char_p
    lib.fa_last_error_message.argtypes = []
    lib.fa_version.restype = i
    lib.fa_version.argtypes = []
    lib.fa_shutdown.restype = None
    lib.fa_shutdown.argtypes = []


def status_string(status: int) -> str:
    try:
        return load_library().fa_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _check(status: int):
    if status != FA_OK:
        msg = load_library().fa_last_error_message().decode()
        raise FAError(status, msg)


def _mask_code(mask) -> int:
    if mask in (None, "none", MASK_NONE, False):
        return MASK_NONE
    if mask in ("causal", MASK_CAUSAL, True):
        return MASK_CAUSAL
    raise ValueError(f"unknown mask {mask!r} (use 'none' or 'causal')")


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return DTYPE_BF16
    if dt == torch.float32:
        return DTYPE_F32
    raise TypeError(f"unsupported dtype {dt} (bf16 or fp32)")


def mha_no_cache(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
                 mask="causal", window: int = -1, *, out: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None, return_lse: bool = False,
                 stream: torch.cuda.Stream | None = None, fp32_tensor_cores: bool = True,
                 workspace: torch.Tensor | None = None):
    """Fused attention forward (``mo.mha.no_cache``) on the current CUDA device.

    q: [B, S, H, D]; k, v: [B, S, Hkv, D]; CUDA tensors of one dtype (bf16 or
    fp32) whose last dimension is contiguous (any other strides are passed to
    the strided entry point). ``scale`` defaults to 1/sqrt(D). ``mask`` is
    "none" or "causal"; ``window`` > 0 adds a sliding window (causal: the W
    keys ending at the query; none: keys within W - 1 on either side).
    Returns out [B, S, H, D] (q's dtype), and lse [B, H, S] fp32 if
    ``return_lse``; a given ``out`` may also be a strided view. fp32 tensors
    run on the tensor cores (three bf16 parts per value, fp32 accuracy) when
    they are dense with D in {64, 128} and ``fp32_tensor_cores``; otherwise on
    the CUDA-core fp32 kernel.
    """
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D (BSHD)")
    B, S, H, D = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != S or k.shape[3] != D:
        raise ValueError(f"k/v shape {tuple(k.shape)}/{tuple(v.shape)} does not match q "
                         f"{tuple(q.shape)} (expected [B, S, Hkv, D])")
    Hkv = k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.stride(-1) != 1:
            raise ValueError(f"{name} must have a contiguous last (D) dimension")
        if t.dtype != q.dtype:
            raise TypeError("q, k, v must share one dtype")
        if t.device != q.device:
            raise ValueError("q, k, v must be on one device")
    dtype = _dtype_code(q.dtype)
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or out.stride(-1) != 1 \
            or out.device != q.device:
        raise ValueError("out must have q's shape, dtype and device and a contiguous last dim")
    if lse is None and return_lse:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    elif lse is not None and (lse.shape != (B, H, S) or lse.dtype != torch.float32
                              or not lse.is_contiguous() or lse.device != q.device):
        raise ValueError("lse must be a contiguous fp32 [B, H, S] tensor on q's device")
    lib = load_library()
    with torch.cuda.device(q.device):
        st = stream if stream is not None else torch.cuda.current_stream(q.device)
        lse_ptr = lse.data_ptr() if lse is not None else None
        dense = all(t.is_contiguous() for t in (q, k, v, out))
        if dtype == DTYPE_F32 and fp32_tensor_cores and dense and D in (64, 128):
            ws_bytes = int(lib.fa_mha_no_cache_f32_tc_workspace(B, S, Hkv, D))
            if workspace is None or workspace.numel() * workspace.element_size() < ws_bytes:
                workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
            rc = lib.fa_mha_no_cache_f32_tc(
                out.data_ptr(), lse_ptr, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                B, S, H, Hkv, D, float(scale), _mask_code(mask), int(window),
                workspace.data_ptr(), ws_bytes, st.cuda_stream)
        elif dense:
            rc = lib.fa_mha_no_cache(
                out.data_ptr(), lse_ptr, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                B, S, H, Hkv, D, float(scale), _mask_code(mask), int(window), dtype,
                st.cuda_stream)
        else:
            arr = ctypes.c_longlong * 3
            sq, sk, sv, so = (arr(*t.stride()[:3]) for t in (q, k, v, out))
            rc = lib.fa_mha_no_cache_strided(
                out.data_ptr(), lse_ptr, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                B, S, H, Hkv, D, sq, sk, sv, so, float(scale), _mask_code(mask), int(window),
                dtype, st.cuda_stream)
    _check(rc)
    return (out, lse) if return_lse else out


def host_workspace_bytes(B: int, S: int, H: int, Hkv: int, D: int, dtype: torch.dtype) -> int:
    """Device bytes :func:`mha_no_cache_host` needs for these sizes."""
    return int(load_library().fa_mha_no_cache_host_workspace(
        int(B), int(S), int(H), int(Hkv), int(D), _dtype_code(dtype)))


def mha_no_cache_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
                      workspace: torch.Tensor, scale: float | None = None, mask="causal",
                      window: int = -1, *, lse: torch.Tensor | None = None,
                      stream: torch.cuda.Stream | None = None):
    """The forward on HOST tensors (q, k, v, out, lse: contiguous CPU tensors,
    pinned for asynchronous copies): one C call enqueues the copies in, the
    kernel and the copies out on ``stream`` (default: the current stream of
    the workspace's device). ``workspace`` is a CUDA tensor of at least
    :func:`host_workspace_bytes` bytes. Returns after enqueueing; synchronise
    the stream before reading ``out``."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D (BSHD)")
    B, S, H, D = q.shape
    Hkv = k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != S or k.shape[3] != D:
        raise ValueError("k/v shape does not match q (expected [B, S, Hkv, D])")
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous host tensor of q's dtype")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    if lse is not None and (lse.is_cuda or lse.shape != (B, H, S) or lse.dtype != torch.float32
                            or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 [B, H, S] host tensor")
    if not workspace.is_cuda:
        raise ValueError("workspace must be a CUDA tensor")
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    lib = load_library()
    with torch.cuda.device(workspace.device):
        st = stream if stream is not None else torch.cuda.current_stream(workspace.device)
        rc = lib.fa_mha_no_cache_host(
            out.data_ptr(), lse.data_ptr() if lse is not None else None, q.data_ptr(),
            k.data_ptr(), v.data_ptr(), B, S, H, Hkv, D, float(scale), _mask_code(mask),
            int(window), _dtype_code(q.dtype), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), st.cuda_stream)
    _check(rc)
    return out


def kv_cache_plan(B: int, Sq: int, S_cache: int, H: int, Hkv: int, D: int, mask="causal",
                  window: int = -1, num_splits: int = 0, num_sms: int = 0) -> tuple[int, int]:
    """(splits, workspace bytes) that :func:`mha_kv_cache` uses for these sizes:
    splits = 1 when every unit runs whole, else the most pieces one unit can
    be cut into. ``num_sms`` = 0 plans for the current device; n > 0 for an
    n-SM device (no CUDA call)."""
    if num_sms == 0:
        num_sms = _sm_count(torch.cuda.current_device())
    return _kv_cache_plan(int(B), int(Sq), int(S_cache), int(H), int(Hkv), int(D),
                          _mask_code(mask), int(window), int(num_splits), int(num_sms))


@functools.lru_cache(maxsize=None)
def _sm_count(device: int) -> int:
    return torch.cuda.get_device_properties(device).multi_processor_count


@functools.lru_cache(maxsize=256)
def _kv_cache_plan(B, Sq, S_cache, H, Hkv, D, mask_code, window, num_splits, num_sms):
    lib = load_library()
    splits = ctypes.c_int(0)
    ws = ctypes.c_ulonglong(0)
    _check(lib.fa_mha_kv_cache_plan(B, Sq, S_cache, H, Hkv, D, mask_code, window, num_splits,
                                    num_sms, ctypes.byref(splits), ctypes.byref(ws)))
    return int(splits.value), int(ws.value)


def mha_kv_cache(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 cache_lens: torch.Tensor | None = None, scale: float | None = None,
                 mask="causal", window: int = -1, *, num_splits: int = 0,
                 out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                 return_lse: bool = False, workspace: torch.Tensor | None = None,
                 stream: torch.cuda.Stream | None = None):
    """Attention over a KV cache (bf16, tensor cores) on the current CUDA device.

    q: [B, Sq, H, D], the last Sq tokens of each sequence; k_cache, v_cache:
    [B, S_cache, Hkv, D] whose first cache_lens[b] rows hold batch b's keys and
    values (cache_lens: int32 CUDA tensor [B], or None for full caches). Query
    row s of batch b sits at position cache_lens[b] - Sq + s; the mask is
    evaluated there. All tensors contiguous bf16. ``num_splits`` = 0 lets the
    library share out the work (few (batch, KV head, position tile) units:
    equal quotas of all units' key tiles per persistent CTA, found from
    cache_lens on the device); n >= 1 cuts every unit into n even key ranges.
    The workspace it needs is allocated here unless given. Returns out
    [B, Sq, H, D] (and lse [B, H, Sq] fp32 if ``return_lse``).
    """
    if q.dim() != 4 or k_cache.dim() != 4 or v_cache.dim() != 4:
        raise ValueError("q, k_cache, v_cache must be 4-D (BSHD)")
    B, Sq, H, D = q.shape
    if k_cache.shape != v_cache.shape or k_cache.shape[0] != B or k_cache.shape[3] != D:
        raise ValueError(f"cache shapes {tuple(k_cache.shape)}/{tuple(v_cache.shape)} do not "
                         f"match q {tuple(q.shape)} (expected [B, S_cache, Hkv, D])")
    S_cache, Hkv = k_cache.shape[1], k_cache.shape[2]
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bf16")
        if t.device != q.device:
            raise ValueError("q and the caches must be on one device")
    if cache_lens is not None and (cache_lens.dtype != torch.int32 or cache_lens.numel() != B
                                   or not cache_lens.is_contiguous()
                                   or cache_lens.device != q.device):
        raise ValueError("cache_lens must be a contiguous int32 [B] tensor on q's device")
    if scale is None:
        scale = 1.0 / (D ** 0.5)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() \
            or out.device != q.device:
        raise ValueError("out must be a contiguous tensor with q's shape, dtype and device")
    if lse is None and return_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    elif lse is not None and (lse.shape != (B, H, Sq) or lse.dtype != torch.float32
                              or not lse.is_contiguous() or lse.device != q.device):
        raise ValueError("lse must be a contiguous fp32 [B, H, Sq] tensor on q's device")
    lib = load_library()
    with torch.cuda.device(q.device):
        _, ws_bytes = kv_cache_plan(B, Sq, S_cache, H, Hkv, D, mask, window, num_splits)
        if ws_bytes > 0 and (workspace is None or workspace.numel() * workspace.element_size()
                             < ws_bytes):
            workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
        st = stream if stream is not None else torch.cuda.current_stream(q.device)
        rc = lib.fa_mha_kv_cache(
            out.data_ptr(), lse.data_ptr() if lse is not None else None, q.data_ptr(),
            k_cache.data_ptr(), v_cache.data_ptr(),
            cache_lens.data_ptr() if cache_lens is not None else None,
            B, Sq, S_cache, H, Hkv, D, float(scale), _mask_code(mask), int(window),
            int(num_splits), workspace.data_ptr() if ws_bytes > 0 else None,
            int(ws_bytes), DTYPE_BF16, st.cuda_stream)
    _check(rc)
    return (out, lse) if return_lse else out


def topk_plan(B: int, V: int, K: int, num_sms: int = 0) -> tuple[int, int]:
    """(chunks per row, workspace bytes) that :func:`topk` uses; ``num_sms`` = 0
    plans for the current device, n > 0 for an n-SM device (no CUDA call)."""
    if num_sms == 0:
        num_sms = _sm_count(torch.cuda.current_device())
    return _topk_plan(int(B), int(V), int(K), int(num_sms))


@functools.lru_cache(maxsize=256)
def _topk_plan(B, V, K, num_sms):
    lib = load_library()
    chunks = ctypes.c_int(0)
    ws = ctypes.c_ulonglong(0)
    _check(lib.fa_topk_plan(B, V, K, num_sms, ctypes.byref(chunks), ctypes.byref(ws)))
    return int(chunks.value), int(ws.value)


def topk(scores: torch.Tensor, k: int, *, values: torch.Tensor | None = None,
         indices: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
         stream: torch.cuda.Stream | None = None):
    """Exact top-k of each row of a [B, V] fp32 CUDA tensor (last dim
    contiguous): (values [B, k] fp32 descending in IEEE total order, indices
    [B, k] int32), equal values by ascending index."""
    if scores.dim() != 2 or not scores.is_cuda or scores.dtype != torch.float32:
        raise ValueError("scores must be a 2-D fp32 CUDA tensor")
    if scores.stride(1) != 1:
        raise ValueError("scores must have a contiguous last dimension")
    B, V = scores.shape
    if values is None:
        values = torch.empty((B, k), dtype=torch.float32, device=scores.device)
    if indices is None:
        indices = torch.empty((B, k), dtype=torch.int32, device=scores.device)
    for name, t, dt in (("values", values, torch.float32), ("indices", indices, torch.int32)):
        if t.shape != (B, k) or t.dtype != dt or not t.is_contiguous() or t.device != scores.device:
            raise ValueError(f"{name} must be a contiguous {dt} [B, k] tensor on scores' device")
    lib = load_library()
    with torch.cuda.device(scores.device):
        _, ws_bytes = topk_plan(B, V, k)
        if workspace is None or workspace.numel() * workspace.element_size() < ws_bytes:
            workspace = torch.empty(max(ws_bytes, 8), dtype=torch.uint8, device=scores.device)
        st = stream if stream is not None else torch.cuda.current_stream(scores.device)
        rc = lib.fa_topk(values.data_ptr(), indices.data_ptr(), scores.data_ptr(), B, V,
                         scores.stride(0), int(k), workspace.data_ptr(), int(ws_bytes),
                         st.cuda_stream)
    _check(rc)
    return values, indices


def device_status(device: int | None = None, clear: bool = True) -> int:
    """Synchronise the device and return the sticky status of all its streams
    (FA_OK, FA_ERR_TIMEOUT, or FA_ERR_BOUNDS from the debug build)."""
    if device is None:
        device = torch.cuda.current_device()
    return int(load_library().fa_device_status(int(device), int(bool(clear))))


def stream_status(stream: torch.cuda.Stream | None = None, clear: bool = True, lib=None) -> int:
    """Synchronise one stream (default: the current one) and return the sticky
    status of the work enqueued on it (FA_OK, FA_ERR_TIMEOUT, FA_ERR_BOUNDS)."""
    st = stream if stream is not None else torch.cuda.current_stream()
    with torch.cuda.device(st.device):
        return int((lib or load_library()).fa_stream_status(st.cuda_stream, int(bool(clear))))


def set_wait_timeout_ns(ns: int) -> int:
    """Set the kernels' bounded-wait limit (0 restores the default); returns the old one."""
    return int(load_library().fa_set_wait_timeout_ns(int(ns)))


def set_stall_probe(enable: bool) -> bool:
    """Test hook: make subsequent bf16 launches take their time-out path."""
    return bool(load_library().fa_set_stall_probe(int(bool(enable))))


def version() -> int:
    return int(load_library().fa_version())
