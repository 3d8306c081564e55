"""GB300 (sm_103a) FlashAttention-style attention forward.

Python binding of the C ABI declared in ``include/attn.h``: argument
marshalling only.  Every step of the computation runs in the CUDA library
``_build/libattn_fwd_gb300.so`` (built by ``attention_attn_fwd_gb300.build``);
there is no fallback, and every entry point raises ``AttnError`` when the
library is missing.

Layouts follow the host launcher of "Flash Attention in CUDA Tile (cuTile)":
Q, O are [B, Hq, Sq, D] and K, V are [B, Hkv, Skv, D], contiguous.
"""
import ctypes
import math
import os
import threading

__all__ = [
    "ATTN_F16", "ATTN_BF16", "ATTN_E4M3", "AttnError", "attn_fwd",
    "attn_fwd_window", "attn_fwd_fp8",
    "attn_fwd_splitkv", "attn_fwd_splitkv_window",
    "attn_splitkv_plan", "attn_fwd_splitkv_noalloc",
    "attn_noalloc_scratch_bytes", "attn_status_string", "attn_device_status",
    "attn_stream_status", "attn_selftest_wait_timeout", "attn_dispatch",
    "attn_tile_config", "attn_unit_plan", "attn_version", "attn_bwd",
    "attn_bwd_workspace_bytes",
    "fwd", "fwd_splitkv", "fwd_fp8", "bwd",
    "library_path", "load_library",
]

ATTN_F16 = 0
ATTN_BF16 = 1
ATTN_E4M3 = 2

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_ALIGNMENT = 3
ATTN_ERR_CUDA = 4
ATTN_ERR_TIMEOUT = 5

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libattn_fwd_gb300.so")
_lib = None
_lock = threading.Lock()


class AttnError(RuntimeError):
    """A non-OK status from the C ABI, or the library is not available."""

    def __init__(self, msg, status=None):
        super().__init__(msg)
        self.status = status


class _Dispatch(ctypes.Structure):
    """attn_dispatch_t of include/attn.h."""
    _fields_ = [(n, ctypes.c_int) for n in (
        "block_m", "block_n", "q_tiles", "paired", "s_buffers", "stages",
        "order", "o_store", "hold_scores", "num_splits", "units",
        "smem_bytes", "merge")] + [("name", ctypes.c_char_p)]


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load the CUDA library (once).  Raises AttnError if it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise AttnError(
                "CUDA library not built (%s); run "
                "`python -m attention_attn_fwd_gb300.build`" % _LIB_PATH)
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i = ctypes.c_void_p, ctypes.c_int
        ip = ctypes.POINTER(ctypes.c_int)
        lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                 ctypes.c_float, i, i, i, vp]
        lib.attn_fwd.restype = i
        lib.attn_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                        ctypes.c_float, i, i, i, i, vp]
        lib.attn_fwd_window.restype = i
        lib.attn_status_string.argtypes = [i]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint)]
        lib.attn_device_status.restype = i
        lib.attn_tile_config.argtypes = [i, i, i, i, i, i, i, i, i,
                                         ip, ip, ip, ip, ip]
        lib.attn_tile_config.restype = i
        lib.attn_version.argtypes = []
        lib.attn_version.restype = i
        sz = ctypes.c_size_t
        lib.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                         ctypes.c_float, i, i, i, i, vp, sz,
                                         vp]
        lib.attn_fwd_splitkv.restype = i
        lib.attn_fwd_splitkv_window.argtypes = [vp, vp, vp, vp, vp, i, i, i,
                                                i, i, i, ctypes.c_float, i, i,
                                                i, i, i, vp, sz, vp]
        lib.attn_fwd_splitkv_window.restype = i
        lib.attn_splitkv_plan.argtypes = [i, i, i, i, i, i, i, i, i, ip,
                                          ctypes.POINTER(sz)]
        lib.attn_splitkv_plan.restype = i
        lib.attn_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i,
                                                 i, i, i, ctypes.c_float, i,
                                                 i, i, i, vp]
        lib.attn_fwd_splitkv_noalloc.restype = i
        lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i,
                                 i, i, i, ctypes.c_float, i, i, i, i, vp, sz,
                                 vp]
        lib.attn_bwd.restype = i
        lib.attn_bwd_workspace_bytes.argtypes = [i, i, i]
        lib.attn_bwd_workspace_bytes.restype = sz
        f = ctypes.c_float
        lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i,
                                     f, f, f, f, i, i, i, i, vp, sz, vp]
        lib.attn_fwd_fp8.restype = i
        lib.attn_noalloc_scratch_bytes.argtypes = []
        lib.attn_noalloc_scratch_bytes.restype = sz
        lib.attn_dispatch.argtypes = [i, i, i, i, i, i, i, i, i, i, i,
                                      ctypes.POINTER(_Dispatch)]
        lib.attn_dispatch.restype = i
        lp = ctypes.POINTER(ctypes.c_longlong)
        lib.attn_unit_plan.argtypes = [i] * 10 + [ip, lp, lp, ip, ip]
        lib.attn_unit_plan.restype = i
        lib.attn_stream_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
        lib.attn_stream_status.restype = i
        lib.attn_selftest_wait_timeout.argtypes = [
            vp, vp, vp, vp, vp, i, i, i, i, i, i, ctypes.c_float, i, i, i,
            ctypes.c_ulonglong, vp]
        lib.attn_selftest_wait_timeout.restype = i
        _lib = lib
        return lib


def attn_fwd(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, scale, causal,
             input_pos, dtype, stream) -> int:
    """Raw C-ABI call; pointers and the stream are integers (0 = NULL)."""
    return int(load_library().attn_fwd(
        Q or None, K or None, V or None, O or None, LSE or None, B, Hq, Hkv,
        Sq, Skv, D, float(scale), int(causal), int(input_pos), int(dtype),
        stream or None))


def attn_fwd_window(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, scale, causal,
                    input_pos, window, dtype, stream) -> int:
    """Raw C-ABI call with a causal sliding window of ``window`` keys."""
    return int(load_library().attn_fwd_window(
        Q or None, K or None, V or None, O or None, LSE or None, B, Hq, Hkv,
        Sq, Skv, D, float(scale), int(causal), int(input_pos), int(window),
        int(dtype), stream or None))


def attn_fwd_fp8(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, scale, q_descale,
                 k_descale, v_descale, causal, input_pos, window, num_splits,
                 workspace, workspace_bytes, stream) -> int:
    """Raw C-ABI call with E4M3 inputs and a bfloat16 O."""
    return int(load_library().attn_fwd_fp8(
        Q or None, K or None, V or None, O or None, LSE or None, B, Hq, Hkv,
        Sq, Skv, D, float(scale), float(q_descale), float(k_descale),
        float(v_descale), int(causal), int(input_pos), int(window),
        int(num_splits), workspace or None, int(workspace_bytes),
        stream or None))


def attn_fwd_splitkv_window(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, scale,
                            causal, input_pos, window, dtype, num_splits,
                            workspace, workspace_bytes, stream) -> int:
    """Raw C-ABI call of the split-KV forward with a sliding window."""
    return int(load_library().attn_fwd_splitkv_window(
        Q or None, K or None, V or None, O or None, LSE or None, B, Hq, Hkv,
        Sq, Skv, D, float(scale), int(causal), int(input_pos), int(window),
        int(dtype), int(num_splits), workspace or None, int(workspace_bytes),
        stream or None))


def attn_fwd_splitkv(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, scale, causal,
                     input_pos, dtype, num_splits, workspace, workspace_bytes,
                     stream) -> int:
    """Raw C-ABI call of the split-KV forward; pointers are integers."""
    return int(load_library().attn_fwd_splitkv(
        Q or None, K or None, V or None, O or None, LSE or None, B, Hq, Hkv,
        Sq, Skv, D, float(scale), int(causal), int(input_pos), int(dtype),
        int(num_splits), workspace or None, int(workspace_bytes),
        stream or None))


def attn_fwd_splitkv_noalloc(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, scale,
                             causal, input_pos, dtype, num_splits,
                             stream) -> int:
    """Raw C-ABI call of the split-KV forward that uses the library's fixed
    scratch array instead of a workspace (for callers that cannot allocate
    device memory); pointers are integers."""
    return int(load_library().attn_fwd_splitkv_noalloc(
        Q or None, K or None, V or None, O or None, LSE or None, B, Hq, Hkv,
        Sq, Skv, D, float(scale), int(causal), int(input_pos), int(dtype),
        int(num_splits), stream or None))


def attn_bwd(Q, K, V, O, LSE, dO, dQ, dK, dV, B, Hq, Hkv, Sq, Skv, D, scale,
             causal, input_pos, window, dtype, workspace, workspace_bytes,
             stream) -> int:
    """Raw C-ABI call of the backward pass; pointers are integers."""
    return int(load_library().attn_bwd(
        Q or None, K or None, V or None, O or None, LSE or None, dO or None,
        dQ or None, dK or None, dV or None, B, Hq, Hkv, Sq, Skv, D,
        float(scale), int(causal), int(input_pos), int(window), int(dtype),
        workspace or None, int(workspace_bytes), stream or None))


def attn_bwd_workspace_bytes(B, Hq, Sq) -> int:
    return int(load_library().attn_bwd_workspace_bytes(B, Hq, Sq))


def attn_noalloc_scratch_bytes() -> int:
    return int(load_library().attn_noalloc_scratch_bytes())


def attn_splitkv_plan(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, dtype,
                      num_splits=0):
    """(num_splits, workspace_bytes) attn_fwd_splitkv accepts."""
    ns = ctypes.c_int(int(num_splits))
    ws = ctypes.c_size_t(0)
    st = int(load_library().attn_splitkv_plan(
        B, Hq, Hkv, Sq, Skv, D, int(causal), int(input_pos), int(dtype),
        ctypes.byref(ns), ctypes.byref(ws)))
    if st != ATTN_OK:
        raise AttnError("attn_splitkv_plan: " + attn_status_string(st), st)
    return ns.value, ws.value


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def attn_device_status():
    """(status, code): synchronises the device and clears the status word."""
    code = ctypes.c_uint(0)
    st = int(load_library().attn_device_status(ctypes.byref(code)))
    return st, int(code.value)


def attn_stream_status(stream=0):
    """(status, code) of the device status word, read after the work on
    ``stream`` (an integer handle, 0 = the legacy default stream) and
    cleared of the bits it reports."""
    code = ctypes.c_uint(0)
    st = int(load_library().attn_stream_status(stream or None,
                                                ctypes.byref(code)))
    return st, int(code.value)


def attn_selftest_wait_timeout(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D,
                               scale, causal, input_pos, dtype, timeout_ns,
                               stream) -> int:
    """Raw C-ABI call of the bounded-wait self-test launch (a forward whose
    first CTA withholds its first K tile; waits give up after
    ``timeout_ns``)."""
    return int(load_library().attn_selftest_wait_timeout(
        Q or None, K or None, V or None, O or None, LSE or None, B, Hq, Hkv,
        Sq, Skv, D, float(scale), int(causal), int(input_pos), int(dtype),
        int(timeout_ns), stream or None))


def attn_tile_config(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, dtype):
    """Tile configuration attn_fwd would launch, as a dict (host only)."""
    out = [ctypes.c_int(0) for _ in range(5)]
    st = int(load_library().attn_tile_config(
        B, Hq, Hkv, Sq, Skv, D, int(causal), int(input_pos), int(dtype),
        *[ctypes.byref(o) for o in out]))
    if st != ATTN_OK:
        raise AttnError("attn_tile_config: " + attn_status_string(st), st)
    keys = ("block_m", "block_n", "stages", "grid", "smem_bytes")
    return {k: o.value for k, o in zip(keys, out)}


def attn_dispatch(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, dtype,
                  window=0, num_splits=0):
    """The forward dispatch-table entry for these arguments, as a dict
    (host only)."""
    d = _Dispatch()
    st = int(load_library().attn_dispatch(
        B, Hq, Hkv, Sq, Skv, D, int(causal), int(input_pos), int(window),
        int(dtype), int(num_splits), ctypes.byref(d)))
    if st != ATTN_OK:
        raise AttnError("attn_dispatch: " + attn_status_string(st), st)
    out = {n: getattr(d, n) for n, _ in _Dispatch._fields_}
    out["name"] = d.name.decode()
    return out


def attn_unit_plan(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, grid,
                   window=0):
    """How a one-pass forward call assigns its units to `grid` CTAs (host
    only): dict with planned, work_max, work_rounds (half K/V steps) and,
    when planned, cta_units (one list of unit indices per CTA)."""
    lib = load_library()
    planned = ctypes.c_int(0)
    wmax, wrounds = ctypes.c_longlong(0), ctypes.c_longlong(0)
    d = attn_dispatch(B, Hq, Hkv, Sq, Skv, D, causal, input_pos, ATTN_BF16,
                      window=window)
    n = d["units"]
    g = max(1, min(n, grid))
    order = (ctypes.c_int * max(1, n))()
    start = (ctypes.c_int * (g + 1))()
    st = int(lib.attn_unit_plan(
        B, Hq, Hkv, Sq, Skv, D, int(causal), int(input_pos), int(window),
        int(grid), ctypes.byref(planned), ctypes.byref(wmax),
        ctypes.byref(wrounds), order, start))
    if st != ATTN_OK:
        raise AttnError("attn_unit_plan: " + attn_status_string(st), st)
    out = {"planned": planned.value, "work_max": wmax.value,
           "work_rounds": wrounds.value, "units": n}
    if planned.value:
        out["cta_units"] = [list(order[start[c]:start[c + 1]])
                            for c in range(g)]
    return out


def attn_version() -> int:
    return int(load_library().attn_version())


def _dtype_code(t):
    import torch
    if t.dtype == torch.float16:
        return ATTN_F16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise AttnError("dtype must be float16 or bfloat16, got %s" % t.dtype,
                    ATTN_ERR_INVALID_ARG)


def fwd(q, k, v, scale=None, causal=True, input_pos=0, out=None, lse=None,
        need_lse=True, stream=None, window=0):
    """Attention forward on CUDA tensors.

    q [B, Hq, Sq, D], k and v [B, Hkv, Skv, D] (contiguous, same dtype,
    float16 or bfloat16).  ``scale`` defaults to 1/sqrt(D).  Returns
    (O, LSE) with LSE float32 [B, Hq, Sq] (None if ``need_lse`` is False).
    ``window`` > 0 (causal only): the query at position p sees keys
    p - window + 1 .. p.  The kernel is enqueued on ``stream`` (default:
    torch's current stream).
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dim() != 4:
            raise AttnError("%s must be 4-D [B, H, S, D]" % name,
                            ATTN_ERR_INVALID_ARG)
        if not t.is_cuda:
            raise AttnError("%s must be a CUDA tensor" % name,
                            ATTN_ERR_INVALID_ARG)
        if not t.is_contiguous():
            raise AttnError("%s must be contiguous" % name,
                            ATTN_ERR_INVALID_ARG)
    if not (q.dtype == k.dtype == v.dtype):
        raise AttnError("q, k, v must share a dtype", ATTN_ERR_INVALID_ARG)
    dt = _dtype_code(q)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Skv, Dk = k.shape
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape):
        raise AttnError("inconsistent q/k/v shapes", ATTN_ERR_INVALID_ARG)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if need_lse and lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        if window:
            st = attn_fwd_window(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                lse.data_ptr() if need_lse else 0, B, Hq, Hkv, Sq, Skv, D,
                scale, causal, input_pos, window, dt, stream.cuda_stream)
        else:
            st = attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                          out.data_ptr(), lse.data_ptr() if need_lse else 0,
                          B, Hq, Hkv, Sq, Skv, D, scale, causal, input_pos, dt,
                          stream.cuda_stream)
    if st != ATTN_OK:
        raise AttnError("attn_fwd: " + attn_status_string(st), st)
    return out, (lse if need_lse else None)


def fwd_splitkv(q, k, v, scale=None, causal=True, input_pos=0, num_splits=0,
                workspace=None, out=None, lse=None, need_lse=True,
                stream=None, window=0):
    """Split-KV attention forward (few query rows over a long key range).

    Same tensors and result as ``fwd`` (``window`` included).
    ``num_splits`` <= 0 lets the library choose; ``workspace`` (a CUDA
    tensor of at least the planned size, 256-byte aligned) is allocated
    with torch when not given.
    """
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise AttnError("q, k, v must be 4-D [B, H, S, D]",
                        ATTN_ERR_INVALID_ARG)
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise AttnError("q, k, v must be contiguous CUDA tensors",
                            ATTN_ERR_INVALID_ARG)
    dt = _dtype_code(q)
    B, Hq, Sq, D = q.shape
    _, Hkv, Skv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        splits, ws_bytes = attn_splitkv_plan(B, Hq, Hkv, Sq, Skv, D, causal,
                                             input_pos, dt, num_splits)
        if workspace is None:
            workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8,
                                    device=q.device)
        if out is None:
            out = torch.empty_like(q)
        if need_lse and lse is None:
            lse = torch.empty((B, Hq, Sq), dtype=torch.float32,
                              device=q.device)
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        ws_args = (splits, workspace.data_ptr(),
                   workspace.numel() * workspace.element_size(),
                   stream.cuda_stream)
        if window:
            st = attn_fwd_splitkv_window(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                lse.data_ptr() if need_lse else 0, B, Hq, Hkv, Sq, Skv, D,
                scale, causal, input_pos, window, dt, *ws_args)
        else:
            st = attn_fwd_splitkv(
                q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                lse.data_ptr() if need_lse else 0, B, Hq, Hkv, Sq, Skv, D,
                scale, causal, input_pos, dt, *ws_args)
    if st != ATTN_OK:
        raise AttnError("attn_fwd_splitkv: " + attn_status_string(st), st)
    return out, (lse if need_lse else None)


def fwd_fp8(q, k, v, scale=None, q_descale=1.0, k_descale=1.0,
            v_descale=1.0, causal=True, input_pos=0, window=0, num_splits=0,
            workspace=None, out=None, lse=None, need_lse=True, stream=None):
    """Attention forward on E4M3 CUDA tensors (torch.float8_e4m3fn, or
    uint8 holding the codes): q [B, Hq, Sq, 128], k and v [B, Hkv, Skv,
    128].  The real inputs are the codes times the per-tensor descale
    factors.  Returns (O bfloat16, LSE float32 or None).  ``num_splits``
    0: one pass; > 0 (or -1 to let the library choose): split-KV with a
    ``workspace`` allocated with torch when not given.
    """
    import torch
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dim() != 4 or not t.is_cuda or not t.is_contiguous():
            raise AttnError("%s must be a contiguous 4-D CUDA tensor" % name,
                            ATTN_ERR_INVALID_ARG)
        if t.element_size() != 1 or t.dtype not in (
                getattr(torch, "float8_e4m3fn", None), torch.uint8):
            raise AttnError("%s must hold E4M3 codes (float8_e4m3fn or "
                            "uint8), got %s" % (name, t.dtype),
                            ATTN_ERR_INVALID_ARG)
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Skv, Dk = k.shape
    if (Bk, Dk) != (B, D) or tuple(v.shape) != tuple(k.shape):
        raise AttnError("inconsistent q/k/v shapes", ATTN_ERR_INVALID_ARG)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        splits, ws_bytes = 0, 0
        if num_splits:
            splits, ws_bytes = attn_splitkv_plan(
                B, Hq, Hkv, Sq, Skv, D, causal, input_pos, ATTN_E4M3,
                max(num_splits, 0))
            if workspace is None:
                workspace = torch.empty(max(ws_bytes, 1), dtype=torch.uint8,
                                        device=q.device)
        if out is None:
            out = torch.empty((B, Hq, Sq, D), dtype=torch.bfloat16,
                              device=q.device)
        if need_lse and lse is None:
            lse = torch.empty((B, Hq, Sq), dtype=torch.float32,
                              device=q.device)
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        ws_ptr = workspace.data_ptr() if workspace is not None else 0
        ws_len = (workspace.numel() * workspace.element_size()
                  if workspace is not None else 0)
        st = attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                          out.data_ptr(), lse.data_ptr() if need_lse else 0,
                          B, Hq, Hkv, Sq, Skv, D, scale, q_descale, k_descale,
                          v_descale, causal, input_pos, window, splits,
                          ws_ptr, ws_len, stream.cuda_stream)
    if st != ATTN_OK:
        raise AttnError("attn_fwd_fp8: " + attn_status_string(st), st)
    return out, (lse if need_lse else None)


def bwd(q, k, v, o, lse, do, scale=None, causal=True, input_pos=0, window=0,
        dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward pass on CUDA tensors: (dQ, dK, dV) for upstream gradient
    ``do``, given the forward's ``o`` and ``lse`` for the same arguments."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do),
                    ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise AttnError("%s must be a contiguous CUDA tensor" % name,
                            ATTN_ERR_INVALID_ARG)
    dt = _dtype_code(q)
    B, Hq, Sq, D = q.shape
    _, Hkv, Skv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    with torch.cuda.device(q.device):
        if dq is None:
            dq = torch.empty_like(q)
        if dk is None:
            dk = torch.empty_like(k)
        if dv is None:
            dv = torch.empty_like(v)
        if workspace is None:
            workspace = torch.empty(max(attn_bwd_workspace_bytes(B, Hq, Sq), 1),
                                    dtype=torch.uint8, device=q.device)
        if stream is None:
            stream = torch.cuda.current_stream(q.device)
        st = attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                      lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
                      dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Sq, Skv, D,
                      scale, causal, input_pos, window, dt,
                      workspace.data_ptr(),
                      workspace.numel() * workspace.element_size(),
                      stream.cuda_stream)
    if st != ATTN_OK:
        raise AttnError("attn_bwd: " + attn_status_string(st), st)
    return dq, dk, dv
