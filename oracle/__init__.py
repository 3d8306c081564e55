"""fp64 CPU oracle for attention forward — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports it, and it imports nothing from the product.

The arithmetic lives in ``attn_oracle.c`` (plain loops in double); this file
only widens inputs to float64 and marshals arrays through ctypes.
"""
import ctypes

import numpy as np

from .build import LIB, build_oracle


def _f64(x):
    """Exact widening of a torch tensor / numpy array to contiguous float64.

    FP8 tensors are refused: they are widened by ``decode_e4m3`` (the
    oracle's own decoder), never by a library conversion."""
    if hasattr(x, "detach"):  # torch tensor, any 16/32/64-bit float dtype
        if x.element_size() == 1:
            raise TypeError("8-bit tensor: widen it with decode_e4m3")
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def torch_uint8():
    import torch
    return torch.uint8


def _ptr(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("expected 4-D [B, H, S, D] arrays")
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Skv, Dk = k.shape
    if (Bk, Dk) != (B, D) or v.shape != k.shape:
        raise ValueError("inconsistent q/k/v shapes")
    return B, Hq, Hkv, Sq, Skv, D


class Oracle:
    """ctypes view of one build of ``attn_oracle.c``."""

    def __init__(self, lib_path):
        lib = ctypes.CDLL(lib_path)
        dp = ctypes.POINTER(ctypes.c_double)
        L = ctypes.c_long
        lib.attn_oracle_fwd.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L, L,
                                        ctypes.c_double, ctypes.c_int, L, L]
        lib.attn_oracle_fwd.restype = ctypes.c_int
        lib.attn_oracle_rows.argtypes = [dp, dp, dp, L, L, L, L, L, L,
                                         ctypes.c_double, ctypes.c_int, L, L,
                                         ctypes.POINTER(ctypes.c_int64), L,
                                         dp, dp]
        lib.attn_oracle_rows.restype = ctypes.c_int
        lib.attn_oracle_prob_row.argtypes = [dp, dp, dp, L, L, L, L, L, L,
                                             ctypes.c_double, ctypes.c_int, L,
                                             L, L, L, L, dp]
        lib.attn_oracle_prob_row.restype = ctypes.c_int
        lib.attn_oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, L, L, L,
                                        L, L, L, ctypes.c_double,
                                        ctypes.c_int, L, L]
        lib.attn_oracle_bwd.restype = ctypes.c_int
        lib.attn_oracle_bwd_dq_rows.argtypes = [
            dp, dp, dp, dp, L, L, L, L, L, L, ctypes.c_double, ctypes.c_int,
            L, L, ctypes.POINTER(ctypes.c_int64), L, dp]
        lib.attn_oracle_bwd_dq_rows.restype = ctypes.c_int
        lib.attn_oracle_bwd_dkdv_rows.argtypes = [
            dp, dp, dp, dp, L, L, L, L, L, L, ctypes.c_double, ctypes.c_int,
            L, L, ctypes.POINTER(ctypes.c_int64), L, dp, dp]
        lib.attn_oracle_bwd_dkdv_rows.restype = ctypes.c_int
        lib.attn_oracle_decode_e4m3.argtypes = [
            ctypes.POINTER(ctypes.c_uint8), L, ctypes.c_double, dp]
        lib.attn_oracle_decode_e4m3.restype = ctypes.c_int
        lib.attn_oracle_threads.argtypes = []
        lib.attn_oracle_threads.restype = ctypes.c_int
        self._lib = lib

    def attention(self, q, k, v, scale, causal=False, input_pos=0, window=0):
        """Full forward: (O [B,Hq,Sq,D], LSE [B,Hq,Sq]) in float64.

        ``window`` > 0 (causal only): each query sees its last ``window``
        positions."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
        o = np.zeros((B, Hq, Sq, D), np.float64)
        lse = np.zeros((B, Hq, Sq), np.float64)
        rc = self._lib.attn_oracle_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq,
            Skv, D, float(scale), int(bool(causal)), int(input_pos),
            int(window))
        if rc != 0:
            raise ValueError("oracle rejected the arguments (code %d)" % rc)
        return o, lse

    def attention_rows(self, q, k, v, scale, causal, input_pos, rows,
                       window=0):
        """Rows (b, h, i) given as an (n, 3) int array: (O [n,D], LSE [n])."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
        rows = np.ascontiguousarray(
            np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        n = rows.shape[0]
        o = np.zeros((n, D), np.float64)
        lse = np.zeros((n,), np.float64)
        rc = self._lib.attn_oracle_rows(
            _ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Skv, D, float(scale),
            int(bool(causal)), int(input_pos), int(window),
            rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n, _ptr(o),
            _ptr(lse))
        if rc != 0:
            raise ValueError("oracle rejected the arguments (code %d)" % rc)
        return o, lse

    def prob_row(self, q, k, v, scale, causal, input_pos, b, h, i, window=0):
        """Softmax weights of query (b, h, i) over all keys, float64 [Skv]."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
        p = np.zeros((Skv,), np.float64)
        rc = self._lib.attn_oracle_prob_row(
            _ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Sq, Skv, D, float(scale),
            int(bool(causal)), int(input_pos), int(window), b, h, i, _ptr(p))
        if rc != 0:
            raise ValueError("oracle rejected the arguments (code %d)" % rc)
        return p

    def backward(self, q, k, v, do, scale, causal=False, input_pos=0,
                 window=0):
        """Gradients (dQ, dK, dV) in float64 for upstream gradient ``do``
        (same shape as the output)."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
        B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
        if do.shape != q.shape:
            raise ValueError("do must have the shape of q")
        dq = np.zeros(q.shape, np.float64)
        dk = np.zeros(k.shape, np.float64)
        dv = np.zeros(v.shape, np.float64)
        rc = self._lib.attn_oracle_bwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
            B, Hq, Hkv, Sq, Skv, D, float(scale), int(bool(causal)),
            int(input_pos), int(window))
        if rc != 0:
            raise ValueError("oracle rejected the arguments (code %d)" % rc)
        return dq, dk, dv

    def backward_dq_rows(self, q, k, v, do, scale, causal, input_pos, rows,
                         window=0):
        """dQ of rows (b, h, i) given as an (n, 3) int array: [n, D]."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
        B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
        rows = np.ascontiguousarray(
            np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        n = rows.shape[0]
        dq = np.zeros((n, D), np.float64)
        rc = self._lib.attn_oracle_bwd_dq_rows(
            _ptr(q), _ptr(k), _ptr(v), _ptr(do), B, Hq, Hkv, Sq, Skv, D,
            float(scale), int(bool(causal)), int(input_pos), int(window),
            rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n, _ptr(dq))
        if rc != 0:
            raise ValueError("oracle rejected the arguments (code %d)" % rc)
        return dq

    def backward_dkdv_rows(self, q, k, v, do, scale, causal, input_pos, keys,
                           window=0):
        """(dK, dV) of key rows (b, kvh, j) given as an (n, 3) int array:
        two [n, D] arrays."""
        q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
        B, Hq, Hkv, Sq, Skv, D = _shapes(q, k, v)
        if do.shape != q.shape:
            raise ValueError("do must have the shape of q")
        keys = np.ascontiguousarray(
            np.asarray(keys, dtype=np.int64).reshape(-1, 3))
        n = keys.shape[0]
        dk = np.zeros((n, D), np.float64)
        dv = np.zeros((n, D), np.float64)
        rc = self._lib.attn_oracle_bwd_dkdv_rows(
            _ptr(q), _ptr(k), _ptr(v), _ptr(do), B, Hq, Hkv, Sq, Skv, D,
            float(scale), int(bool(causal)), int(input_pos), int(window),
            keys.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n, _ptr(dk),
            _ptr(dv))
        if rc != 0:
            raise ValueError("oracle rejected the arguments (code %d)" % rc)
        return dk, dv

    def decode_e4m3(self, x8, descale=1.0):
        """E4M3 codes (a torch float8_e4m3fn / uint8 tensor or a uint8
        array) times ``descale``, as a float64 array of the same shape."""
        if hasattr(x8, "detach"):
            if x8.element_size() != 1:
                raise TypeError("expected an 8-bit tensor")
            x8 = x8.detach().to("cpu").contiguous().view(torch_uint8()).numpy()
        codes = np.ascontiguousarray(np.asarray(x8, dtype=np.uint8))
        out = np.zeros(codes.shape, np.float64)
        rc = self._lib.attn_oracle_decode_e4m3(
            codes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), codes.size,
            float(descale), _ptr(out))
        if rc != 0:
            raise ValueError("oracle rejected the arguments (code %d)" % rc)
        return out

    def threads(self) -> int:
        """Number of OpenMP threads the oracle's loops use."""
        return int(self._lib.attn_oracle_threads())


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build_oracle())
    return _default


def attention(q, k, v, scale, causal=False, input_pos=0, window=0):
    return default().attention(q, k, v, scale, causal, input_pos, window)


def attention_rows(q, k, v, scale, causal, input_pos, rows, window=0):
    return default().attention_rows(q, k, v, scale, causal, input_pos, rows,
                                    window)


def prob_row(q, k, v, scale, causal, input_pos, b, h, i, window=0):
    return default().prob_row(q, k, v, scale, causal, input_pos, b, h, i,
                              window)


def backward(q, k, v, do, scale, causal=False, input_pos=0, window=0):
    return default().backward(q, k, v, do, scale, causal, input_pos, window)


def backward_dq_rows(q, k, v, do, scale, causal, input_pos, rows, window=0):
    return default().backward_dq_rows(q, k, v, do, scale, causal, input_pos,
                                      rows, window)


def backward_dkdv_rows(q, k, v, do, scale, causal, input_pos, keys,
                       window=0):
    return default().backward_dkdv_rows(q, k, v, do, scale, causal,
                                        input_pos, keys, window)


def decode_e4m3(x8, descale=1.0):
    return default().decode_e4m3(x8, descale)


def threads() -> int:
    return default().threads()
